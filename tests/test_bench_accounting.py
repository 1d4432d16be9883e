"""The benchmark's algorithmic byte counts, pinned to the shapes they come
from (Qwen3-0.6B decode set: 28 layers of q 2048x1024, k/v 1024x1024,
o 1024x2048, gate/up 3072x1024, down 1024x3072; q4_K 144 bytes and q8_K 292
bytes per 256 values), computed here by hand rather than through bench.py's
own helpers."""
import bench


def test_decode_set_weight_bytes():
    mats, total = bench.mat_list()
    assert len(mats) == 196
    per_layer = (2048 * 4 + 1024 * 4 + 1024 * 4 + 1024 * 8 + 3072 * 4 + 3072 * 4 + 1024 * 12) * 144
    assert per_layer == 8_847_360
    assert total == 28 * per_layer == 247_726_080
    # storage order and offsets: contiguous, layer by layer
    off = 0
    for idx, (layer, j, n, k, o) in enumerate(mats):
        assert (layer, j) == divmod(idx, 7) and o == off
        off += n * (k // 256) * 144
    assert off == total


def test_grouped_gemv_bytes_per_launch():
    mats, total = bench.mat_list()
    blocks_per_layer = 4 + 4 + 4 + 8 + 4 + 4 + 12          # activation q8_K blocks (one row per matrix)
    rows_per_layer = 2048 + 1024 + 1024 + 1024 + 3072 + 3072 + 1024
    expect = total + 28 * blocks_per_layer * 292 + 28 * rows_per_layer * 4
    assert expect == 249_429_376
    assert sum(bench.gemv_bytes(n, k) for _, _, n, k, _ in mats) == expect


def test_step_bytes_add_the_quantizer():
    mats, _ = bench.mat_list()
    k_sum = 28 * (1024 + 1024 + 1024 + 2048 + 1024 + 1024 + 3072)   # activation values, one row per matrix
    assert k_sum == 286_720
    quant = k_sum * 4 + (k_sum // 256) * 292                      # f32 read + q8_K written
    assert bench.step_bytes(mats) == 249_429_376 + quant


def test_fused_step_bytes_are_weights_f32_activations_and_y():
    # the headline step reads the weights and the f32 activations once and
    # writes y once; the q8_K codes stay on the chip
    mats, weights = bench.mat_list()
    assert weights == 247_726_080
    x_f32 = 4 * 28 * (1024 + 1024 + 1024 + 2048 + 1024 + 1024 + 3072)
    y = 4 * 28 * (2048 + 1024 + 1024 + 1024 + 3072 + 3072 + 1024)
    assert bench.fused_step_bytes(mats) == weights + x_f32 + y == 250_249_216


def test_ncu_records_match_the_kernel_sources():
    """Every committed ncu traffic record still describes the kernel sources as they are:
    the bench reports `traffic` only while the sources' hash matches the capture's, so
    a source edit without a new capture would turn the bench line's traffic to null."""
    import json
    import os
    recs = json.load(open(os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")))
    assert set(recs) >= {"gemv_q4K_fused_grouped_m1", "gemv_q4K_grouped_m1", "gemm_q4K_12288x4096_m2048"}
    for key, rec in recs.items():
        assert bench.recorded_counters(key) is not None, "%s: stale (sources changed since the capture)" % key
        assert rec["dram_bytes_per_launch"] == rec["dram_read_bytes"] + rec["dram_write_bytes"]
        assert os.path.exists(os.path.join(bench.ROOT, rec["capture"]))
