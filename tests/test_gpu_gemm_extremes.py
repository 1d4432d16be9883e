"""GEMM parity at the extremes of every format's integer ranges.

The tensor-core GEMM contracts exact integer-valued f16 operands (q4_K/q5_K:
sc*q, q6_K: the int8 scale split as 16*hi + lo times q6 - 32) and sums them
in f32 per 256-weight block.  Uniform random codes keep those sums far below
2^24; the blocks here drive them to the format's largest magnitudes (a whole
q4_K block of code 15 at scale 63 against activation code -128 sums to about
3.1e7, past 2^24), so the f32 rounding inside a block, the q6_K scale split
and the min term are exercised where they are tightest.  The PocketLLM pages
(Korean README, "Current status" table, row "src/") state the matching
integer fact for the CPU path: q4_K sub-block sums fit int16, q6_K's do not.

Weight rows cycle through extreme blocks and one seeded random block; the
activation rows cycle through all -1 (codes -128), +1 (codes -128 with a
negative d), alternating +-1 (codes -128 / 127) and N(0,1).  Every case runs
through the plain entry point and the caller-workspace form with the minimal
(unsplit) and the split-K workspace, at m = 9, 130 and 512.  Tolerance: 1e-4
of sum_k |w_hat * x_hat| per output element, as in every parity test.
"""
import numpy as np
import pytest

import gen
import oracle
from tests.packers import pack_q2K, pack_q3K, pack_q4K, pack_q5K, pack_q6K

FMTS = ["q2K", "q3K", "q4K", "q5K", "q6K"]
BPB = {"q2K": 84, "q3K": 110, "q4K": 144, "q5K": 176, "q6K": 210}


def extreme_blocks(fmt):
    """The extreme block constructions of one format (each one block)."""
    alt = np.tile([0, 1], 128)
    if fmt == "q4K":
        return [pack_q4K(2e-3, 2e-3, [63] * 8, [63] * 8, np.full(256, 15)),     # largest isum
                pack_q4K(2e-3, 2e-3, [63] * 8, [63] * 8, np.zeros(256)),        # min term only
                pack_q4K(1e-4, 2e-3, [63, 0] * 4, [0, 63] * 4, 15 * alt),      # mixed table
                pack_q4K(2e-3, 0.0, [63] * 8, [0] * 8, np.full(256, 15))]
    if fmt == "q5K":
        return [pack_q5K(2e-3, 2e-3, [63] * 8, [63] * 8, np.full(256, 31)),     # sc*q = 1953
                pack_q5K(2e-3, 2e-3, [63] * 8, [63] * 8, np.zeros(256)),
                pack_q5K(2e-3, 1e-4, [63] * 8, [63, 0] * 4, 31 * alt),
                pack_q5K(2e-3, 2e-3, [1] * 8, [63] * 8, np.full(256, 16))]      # only the fifth bit
    if fmt == "q6K":
        return [pack_q6K(2e-3, [-64] * 16, np.zeros(256)),                     # scale -64, q6 = 0
                pack_q6K(2e-3, [-64] * 16, np.full(256, 63)),                  # scale -64, q6 = 63
                pack_q6K(2e-3, [-128] * 16, np.zeros(256)),                    # int8 minimum scale
                pack_q6K(2e-3, [127] * 16, np.full(256, 63)),
                pack_q6K(2e-3, [-1, 15, 16, -17] * 4, 63 * alt)]               # hi/lo split edges
    if fmt == "q3K":
        return [pack_q3K(2e-3, [0] * 16, np.full(256, -4)),                    # scale -32, code -4
                pack_q3K(2e-3, [63] * 16, np.full(256, 3)),
                pack_q3K(2e-3, [0, 63] * 8, np.full(256, -4) + 7 * alt)]
    return [pack_q2K(2e-3, 2e-3, [15] * 16, [15] * 16, np.full(256, 3)),
            pack_q2K(2e-3, 2e-3, [15] * 16, [15] * 16, np.zeros(256)),
            pack_q2K(2e-3, 2e-3, [15, 0] * 8, [0, 15] * 8, 3 * alt)]


def extreme_weights(fmt, n, k):
    """n rows of k/256 blocks: row r takes construction (r + b) mod (count + 1)
    at block b, the last choice being a seeded random block."""
    blocks = extreme_blocks(fmt)
    rand = getattr(gen, "%s_blocks" % fmt)(60, 0, n, k)
    nb = k // 256
    w = np.empty((n, nb * BPB[fmt]), dtype=np.uint8)
    for r in range(n):
        for b in range(nb):
            c = (r + b) % (len(blocks) + 1)
            src = blocks[c] if c < len(blocks) else rand[r, b * BPB[fmt]:(b + 1) * BPB[fmt]]
            w[r, b * BPB[fmt]:(b + 1) * BPB[fmt]] = src
    return w


def extreme_acts(m, k):
    x = gen.normal_f32(61, m, m, k)
    for i in range(m):
        kind = i % 4
        if kind == 0:
            x[i] = -1.0                       # every code -128
        elif kind == 1:
            x[i] = 1.0                        # every code -128, d negative
        elif kind == 2:
            x[i] = -1.0
            x[i, ::2] = 1.0                   # first element +1: codes -128 and 127
    return x


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [9, 130, 512])
def test_gemm_adversarial_extremes(fmt, m):
    import torch
    import quant_packed_gemv_gb300 as q
    from tests.gpu_helpers import assert_close, dev, host, oracle_ref
    n, k = 136, 2048                          # two weight-row tiles (ragged), 8 blocks: K splits in two
    w = extreme_weights(fmt, n, k)
    xq = oracle.quantize_q8K(extreme_acts(m, k))
    assert (xq.reshape(m, -1, 292)[0::4, :, 4:260].view(np.int8) == -128).all()
    ref, S = oracle_ref(fmt, w, xq, m, n, k)
    wd, xd = dev(w), dev(xq)
    unsplit = q.plm_gemm_workspace_size(fmt, m, k)
    split = q.plm_gemm_workspace_size_split(fmt, m, n, k)
    assert split > unsplit > 0                # the tensor-core path (k = 2048 qualifies q2_K, q3_K too), both K layouts
    outs = []
    for need in sorted({unsplit, split}):
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
        y = torch.full((m, n), float("nan"), device="cuda")
        getattr(q, "plm_gemm_%s_ws" % fmt)(wd, xd, y, m, n, k, ws if need else None, need)
        outs.append(host(y))
    y = torch.full((m, n), float("nan"), device="cuda")
    getattr(q, "plm_gemm_%s" % fmt)(wd, xd, y, m, n, k)
    outs.append(host(y))
    for out in outs:
        assert not np.isnan(out).any()
        assert_close(out, ref, S)
    assert q.plm_device_fault() == 0


def test_extreme_block_sums_pass_2_24():
    """The q4_K construction really drives a block's integer sum past 2^24
    (where f32 stops being exact), as the test above intends."""
    blk = extreme_blocks("q4K")[0]
    x = np.full((1, 256), -1.0, dtype=np.float32)
    xq = oracle.quantize_q8K(x)
    sub = oracle.subdots_q4K(blk.reshape(1, -1), xq, 1, 1, 256)
    isum = int((63 * sub.astype(np.int64)).sum())
    assert abs(isum) > 2 ** 24
