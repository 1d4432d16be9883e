"""Pins of the x16 row-interleaved q4_K layout on the host.

The oracle reads the x16 layout with its own inverse walk (plm_ref.c,
dequant_q4K_x16); the test-side packer builds the layout from its definition
in the packing direction (tests/packers.py).  A round trip through both must
give back exactly the weights the plain q4_K decoder reads from the original
blocks, for ragged row counts (a padded last tile) and several k."""
import numpy as np
import pytest

import gen
import oracle
from tests.packers import pack_q4K_x16, pack_q6K_x16


@pytest.mark.parametrize("n,k", [(1, 256), (16, 512), (37, 1024), (130, 768)])
def test_x16_round_trip_equals_plain_decode(n, k):
    w = gen.q4K_blocks(70, n, n, k)
    wx = pack_q4K_x16(w, n, k)
    assert wx.size == -(-n // 16) * (k // 256) * 2304
    np.testing.assert_array_equal(oracle.dequant_q4K_x16(wx, n, k), oracle.dequant_q4K(w, n, k))


def test_x16_every_qs_byte_lands_once():
    # each qs byte of a tile-block, marked with its own index, is found by
    # the oracle's walk at exactly one weight pair: a permutation, no overlap
    n, k = 16, 256
    w = np.zeros((n, 144), dtype=np.uint8)
    w[:, 0:2] = np.array([1.0], dtype=np.float16).view(np.uint8)      # d = 1, dmin = 0
    w[:, 4:8] = 1                                                     # sc_0..3 = 1 (m = 0)
    w[:, 12:16] = 1                                                   # sc_4..7 = 1
    seen = set()
    for r in range(n):
        for c in range(128):
            ww = w.copy()
            ww[r, 16 + c] = 0x21                      # low nibble 1, high nibble 2
            deq = oracle.dequant_q4K_x16(pack_q4K_x16(ww, n, k), n, k)
            nz = np.argwhere(deq != 0)
            assert len(nz) == 2 and (nz[:, 0] == r).all()
            lo, hi = sorted(nz[:, 1])
            chunk = c // 32
            assert (lo, hi) == (64 * chunk + c % 32, 64 * chunk + 32 + c % 32)
            assert deq[r, lo] == 1.0 and deq[r, hi] == 2.0
            seen.add((r, c))
    assert len(seen) == n * 128


def test_x16_padding_rows_are_zero_blocks():
    n, k = 21, 512
    w = gen.q4K_blocks(71, 0, n, k)
    wx = pack_q4K_x16(w, n, k).reshape(2, 2, 2304)
    # tile 1 holds rows 16..20, then eleven zero rows whose headers are zero
    for b in range(2):
        hdr = wx[1, b, :256].reshape(16, 16)
        assert (hdr[5:] == 0).all() and (hdr[:5] != 0).any()


@pytest.mark.parametrize("n,k", [(1, 256), (16, 512), (37, 1024), (130, 768)])
def test_q6K_x16_round_trip_equals_plain_decode(n, k):
    w = gen.q6K_blocks(72, n, n, k)
    wx = pack_q6K_x16(w, n, k)
    assert wx.size == -(-n // 16) * (k // 256) * 3360
    np.testing.assert_array_equal(oracle.dequant_q6K_x16(wx, n, k), oracle.dequant_q6K(w, n, k))


def test_q6K_x16_every_code_bit_lands_once():
    # a block of q6 = 32 (weight 0) with scale 1; set one code bit at a time
    # (each ql nibble bit and each qh bit): exactly one weight moves, by the
    # bit's value, at the position the q6_K format gives it
    from tests.packers import pack_q6K
    n, k = 16, 256
    base = np.full(256, 32)
    for r in (0, 9):
        for wgt in range(0, 256, 7):
            for bit in range(6):
                q = base.copy()
                q[wgt] ^= 1 << bit
                blk = pack_q6K(1.0, [1] * 16, q)
                w = np.tile(pack_q6K(1.0, [1] * 16, base), (n, 1))
                w[r] = blk
                deq = oracle.dequant_q6K_x16(pack_q6K_x16(w, n, k), n, k)
                nz = np.argwhere(deq != 0)
                assert len(nz) == 1 and tuple(nz[0]) == (r, wgt)
                assert deq[r, wgt] == q[wgt] - 32
