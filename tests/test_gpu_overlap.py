"""Early launch (plm_set_overlap): a kernel of the library may be scheduled
while the kernel before it on the stream still runs, and in PREFETCH mode a
GEMV may copy weights before that kernel ends.  Results must not depend on
the mode, also when every kernel consumes what the kernel just before it
wrote, as in a decoder: the y of one GEMV is quantized and becomes the next
GEMV's activation row.  Intermediate buffers start as NaN (f32) or 0xFF
bytes (q8_K, whose d then reads as NaN), so a kernel that read its input
before the producer had finished would leave NaNs or different bits."""
import numpy as np
import pytest
import torch

import gen
import oracle
import quant_packed_gemv_gb300 as q
from tests.gpu_helpers import TOL, dev, host

pytestmark = pytest.mark.gpu

MODES = (q.PLM_OVERLAP_OFF, q.PLM_OVERLAP_LAUNCH, q.PLM_OVERLAP_PREFETCH)


class Chain:
    """One decoder-shaped layer at m = 1 plus a small prefill pair at m = 64:
    x(1024) -q4_K-> 2048 -fused q4_K-> 1024 -SwiGLU q4_K pair-> 3072 -q6_K-> 1024 -q5_K-> 1024;
    X(64x1024) -q4_K GEMM-> 64x2048 -q6_K GEMM (split K)-> 64x1024."""

    def __init__(self, seed):
        s = seed
        self.w1 = dev(gen.q4K_blocks(s, 1, 2048, 1024))
        self.w2 = dev(gen.q4K_blocks(s, 2, 1024, 2048))
        self.wg = dev(gen.q4K_blocks(s, 3, 3072, 1024))
        self.wu = dev(gen.q4K_blocks(s, 4, 3072, 1024))
        self.w4 = dev(gen.q6K_blocks(s, 5, 1024, 3072))
        self.w5 = dev(gen.q5K_blocks(s, 6, 1024, 1024))
        self.g1 = dev(gen.q4K_blocks(s, 7, 2048, 1024))
        self.g2 = dev(gen.q6K_blocks(s, 8, 1024, 2048))
        self.x = dev(gen.normal_f32(s, 9, 1, 1024))
        self.X = dev(gen.normal_f32(s, 10, 64, 1024))
        f32 = lambda *shape: torch.empty(shape, dtype=torch.float32, device="cuda")
        u8 = lambda nbytes: torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        self.xq = u8(4 * 292)
        self.y1, self.y2, self.h, self.y4, self.y5 = f32(2048), f32(1024), f32(3072), f32(1024), f32(1024)
        self.q2, self.q3, self.q4 = u8(4 * 292), u8(12 * 292), u8(4 * 292)
        self.Xq, self.Y1, self.Y1q, self.Y2 = u8(64 * 4 * 292), f32(64, 2048), u8(64 * 8 * 292), f32(64, 1024)
        self.ws = torch.empty(q.plm_gemm_workspace_size_split(6, 64, 1024, 2048), dtype=torch.uint8,
                              device="cuda")

    def poison(self):
        for t in (self.y1, self.y2, self.h, self.y4, self.y5, self.Y1, self.Y2):
            t.fill_(float("nan"))
        for t in (self.xq, self.q2, self.q3, self.q4, self.Xq, self.Y1q):
            t.fill_(0xFF)
        torch.cuda.synchronize()   # the fills ran on the current stream, the chain runs on its own

    def run(self, stream, sync=False):
        st = stream.cuda_stream
        step = (lambda: torch.cuda.synchronize()) if sync else (lambda: None)
        q.plm_quantize_q8K(self.x, self.xq, 1, 1024, stream=st); step()
        q.plm_gemv_q4K(self.w1, self.xq, self.y1, 1, 2048, 1024, stream=st); step()
        q.plm_quantize_gemv_q4K(self.w2, self.y1, self.y2, 1, 1024, 2048, stream=st); step()
        q.plm_quantize_q8K(self.y2, self.q2, 1, 1024, stream=st); step()
        q.plm_gemv_q4K_swiglu(self.wg, self.wu, self.q2, self.h, 1, 3072, 1024, stream=st); step()
        q.plm_quantize_q8K(self.h, self.q3, 1, 3072, stream=st); step()
        q.plm_gemv_q6K(self.w4, self.q3, self.y4, 1, 1024, 3072, stream=st); step()
        q.plm_quantize_q8K(self.y4, self.q4, 1, 1024, stream=st); step()
        q.plm_gemv_q5K(self.w5, self.q4, self.y5, 1, 1024, 1024, stream=st); step()
        q.plm_quantize_q8K(self.X, self.Xq, 64, 1024, stream=st); step()
        q.plm_gemm_q4K(self.g1, self.Xq, self.Y1, 64, 2048, 1024, stream=st); step()
        q.plm_quantize_q8K(self.Y1, self.Y1q, 64, 2048, stream=st); step()
        q.plm_gemm_q6K_ws(self.g2, self.Y1q, self.Y2, 64, 1024, 2048, self.ws, self.ws.numel(), stream=st)
        step()

    def outputs(self):
        torch.cuda.synchronize()
        return {k: getattr(self, k).cpu().numpy().copy() for k in ("y1", "y2", "h", "y4", "y5", "Y1", "Y2")}


@pytest.fixture
def restore_mode():
    prev = q.plm_set_overlap(q.PLM_OVERLAP_LAUNCH)
    yield
    q.plm_set_overlap(prev)


def check_equal(ref, got, what):
    for k in ref:
        assert not np.isnan(got[k]).any(), "%s: %s has unwritten or stale-input elements" % (what, k)
        assert np.array_equal(ref[k], got[k]), "%s: %s differs from the serialized run" % (what, k)


def test_chain_same_bits_in_every_mode(restore_mode):
    c = Chain(21)
    s = torch.cuda.Stream()
    q.plm_set_overlap(q.PLM_OVERLAP_OFF)
    c.poison()
    c.run(s, sync=True)
    ref = c.outputs()
    # the first stage against the oracle (the rest are pinned by the per-op tests)
    x = gen.normal_f32(21, 9, 1, 1024)
    xq = oracle.quantize_q8K(x)
    w1 = gen.q4K_blocks(21, 1, 2048, 1024)
    err = np.abs(ref["y1"].astype(np.float64) - oracle.gemm_q4K_f64(w1, xq, 1, 2048, 1024)[0])
    assert np.all(err <= TOL * oracle.absscale_q4K(w1, xq, 1, 2048, 1024)[0])
    for mode in MODES:
        q.plm_set_overlap(mode)
        for rep in range(3):
            c.poison()
            c.run(s)
            check_equal(ref, c.outputs(), "mode %d eager, pass %d" % (mode, rep))


@pytest.mark.parametrize("mode", [q.PLM_OVERLAP_LAUNCH, q.PLM_OVERLAP_PREFETCH])
def test_chain_same_bits_in_a_cuda_graph(mode, restore_mode):
    c = Chain(22)
    s = torch.cuda.Stream()
    q.plm_set_overlap(q.PLM_OVERLAP_OFF)
    c.poison()
    c.run(s, sync=True)
    ref = c.outputs()
    q.plm_set_overlap(mode)
    with torch.cuda.stream(s):
        c.run(s)   # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):   # the same layer three times in one graph: each pass waits for the previous
            c.run(s)
    for rep in range(3):
        c.poison()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.replay()
        check_equal(ref, c.outputs(), "mode %d graph, replay %d" % (mode, rep))
    assert q.plm_device_fault() == 0
