"""Pins for the oracle's f16 decode, q4_K / q6_K block decode, integer
sub-block dots and block combine (host only).

Formats: the GGML K-quant blocks the PocketLLM pages name ("What it runs":
q4_k / q6_k decoded inside the kernel, never widened), with the byte layouts
of the public GGML format.  The int16 statement comes from the "Current
status" table, row "src/ -- the C++ engine": q4_K sub-block sums may be held
in int16, q6_K ones may not.
"""
import numpy as np
import pytest

import gen
import oracle
from tests.packers import pack_q2K, pack_q3K, pack_q4K, pack_q5K, pack_q6K, pack_q8K


def test_f16_exhaustive_against_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.f16_to_f32(bits)
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_splitmix64_published_sequence():
    # SplitMix64 (Steele, Lea, Flood 2014) started at state 1234567: the
    # widely published first outputs of the reference implementation.
    r = gen.raw_draws(1234567, 0, 0, 3)
    assert [int(v) for v in r] == [6457827717110365317, 3203168211198807973, 9817491932198370423]


# ---------------------------------------------------------------- q4_K

def test_q4K_scale_table_roundtrip_all_values():
    for j in range(8):
        for sc in range(64):
            for mn in range(64):
                scs = [(j * 7 + 5 * t) % 64 for t in range(8)]
                mns = [(j * 11 + 3 * t) % 64 for t in range(8)]
                scs[j], mns[j] = sc, mn
                blk = pack_q4K(1.0, 0.0, scs, mns, np.zeros(256))
                for jj in range(8):
                    assert oracle.q4K_scale_min(blk[4:16], jj) == (scs[jj], mns[jj])


def test_q4K_single_nibble_position_map():
    seen = set()
    for byte in range(128):
        for hi in (0, 1):
            blk = np.zeros(144, dtype=np.uint8)
            blk[0:2] = np.array([1.0], dtype=np.float16).view(np.uint8)
            blk[4:8] = 1  # scales 0..3 = 1, mins 0..3 = 0
            blk[12:16] = 1  # scales 4..7 low nibble = 1, mins 4..7 = 0
            blk[16 + byte] = 0x10 if hi else 0x01
            w = oracle.dequant_q4K(blk, 1, 256)[0]
            nz = np.nonzero(w)[0]
            assert len(nz) == 1 and w[nz[0]] == 1.0
            chunk, l = divmod(byte, 32)
            assert nz[0] == 64 * chunk + 32 * hi + l
            seen.add(int(nz[0]))
    assert seen == set(range(256))


def _rand_q4K(rng):
    d = float(np.float16(rng.uniform(1e-4, 2e-3)))
    dmin = float(np.float16(rng.uniform(1e-4, 2e-3)))
    sc = rng.integers(0, 64, 8)
    mn = rng.integers(0, 64, 8)
    q = rng.integers(0, 16, 256)
    return d, dmin, sc, mn, q


def test_q4K_dequant_from_fields():
    rng = np.random.default_rng(1)
    for _ in range(50):
        d, dmin, sc, mn, q = _rand_q4K(rng)
        w = oracle.dequant_q4K(pack_q4K(d, dmin, sc, mn, q), 1, 256)[0]
        j = np.arange(256) // 32
        expect = np.float64(d) * sc[j] * q - np.float64(dmin) * mn[j]
        np.testing.assert_array_equal(w, expect)


def test_q4K_subdots_and_combine_from_fields():
    rng = np.random.default_rng(2)
    for _ in range(30):
        d, dmin, sc, mn, q = _rand_q4K(rng)
        wblk = pack_q4K(d, dmin, sc, mn, q)
        dx = np.float32(rng.uniform(-0.05, 0.05))
        q8 = rng.integers(-128, 128, 256)
        xblk = pack_q8K(dx, q8)
        dots = oracle.subdots_q4K(wblk, xblk, 1, 1, 256)[0, 0]
        np.testing.assert_array_equal(dots, (q * q8).reshape(8, 32).sum(axis=1))
        # block combine: d*dx*sum_j sc_j dot_j - dmin*dx*sum_j m_j (sum of codes in j)
        isum = int((sc * dots).sum())
        msum = int((mn * q8.reshape(8, 32).sum(axis=1)).sum())
        y = oracle.gemm_q4K_f64(wblk, xblk, 1, 1, 256)[0, 0]
        expect = float(np.float64(d) * np.float64(dx) * isum - np.float64(dmin) * np.float64(dx) * msum)
        assert y == pytest.approx(expect, rel=1e-15, abs=1e-300)


def test_q4K_all_zero_nibbles_closed_form():
    # zero nibbles, every min = M: every weight is -dmin*M, so
    # y = -dmin*M*dx*(sum of all codes), independent of the scales
    rng = np.random.default_rng(3)
    for M in (0, 1, 17, 63):
        dmin = 0.0009765625  # 2^-10, exact in f16
        blk = pack_q4K(0.5, dmin, rng.integers(0, 64, 8), [M] * 8, np.zeros(256))
        q8 = rng.integers(-128, 128, 256)
        xblk = pack_q8K(0.25, q8)
        y = oracle.gemm_q4K_f64(blk, xblk, 1, 1, 256)[0, 0]
        assert y == -dmin * M * 0.25 * q8.sum()


def test_q4K_int16_partial_sums_statement():
    # all nibbles 15, all codes -128: the adversarial corner
    blk = pack_q4K(1.0, 0.0, [63] * 8, [0] * 8, np.full(256, 15))
    xblk = pack_q8K(1.0, np.full(256, -128))
    dots = oracle.subdots_q4K(blk, xblk, 1, 1, 256)[0, 0]
    assert np.all(dots == 32 * 15 * -128)  # -61440: a full sub-block leaves int16
    half = 16 * 15 * -128                  # -30720: a 16-term partial stays in int16
    assert np.int16(half) == half
    assert np.int16(np.int32(dots[0])) != dots[0]


def test_q6K_int16_overflow_statement():
    blk = pack_q6K(1.0, [1] * 16, np.zeros(256, dtype=np.int64))  # q6 = 0 -> -32
    xblk = pack_q8K(1.0, np.full(256, -128))
    dots = oracle.subdots_q6K(blk, xblk, 1, 1, 256)[0, 0]
    assert np.all(dots == 16 * 32 * 128)  # 65536 per 16-group: does not fit int16
    assert 8 * 32 * 128 > np.iinfo(np.int16).max  # even 8 terms overflow


# ---------------------------------------------------------------- q6_K

def test_q6K_all_32_gives_zero():
    rng = np.random.default_rng(4)
    blk = pack_q6K(1.5, rng.integers(-64, 64, 16), np.full(256, 32))
    assert blk[0:128].max() == 0 and np.all(blk[128:192] == 0xAA)
    xblk = pack_q8K(0.1, rng.integers(-128, 128, 256))
    assert oracle.gemm_q6K_f64(blk, xblk, 1, 1, 256)[0, 0] == 0.0
    assert not oracle.dequant_q6K(blk, 1, 256).any()


def test_q6K_single_code_position_map():
    for pos in range(256):
        q = np.full(256, 32)
        q[pos] = 33 + (pos % 31)
        blk = pack_q6K(1.0, [1] * 16, q)
        w = oracle.dequant_q6K(blk, 1, 256)[0]
        nz = np.nonzero(w)[0]
        assert list(nz) == [pos] and w[pos] == q[pos] - 32


def test_q6K_dequant_and_dots_from_fields():
    rng = np.random.default_rng(5)
    for _ in range(30):
        d = float(np.float16(rng.uniform(1e-4, 2e-3)))
        scales = rng.integers(-64, 64, 16)
        scales[0] = -64
        q = rng.integers(0, 64, 256)
        blk = pack_q6K(d, scales, q)
        w = oracle.dequant_q6K(blk, 1, 256)[0]
        np.testing.assert_array_equal(w, np.float64(d) * scales[np.arange(256) // 16] * (q - 32))
        q8 = rng.integers(-128, 128, 256)
        dx = np.float32(rng.uniform(-0.05, 0.05))
        xblk = pack_q8K(dx, q8)
        dots = oracle.subdots_q6K(blk, xblk, 1, 1, 256)[0, 0]
        np.testing.assert_array_equal(dots, ((q - 32) * q8).reshape(16, 16).sum(axis=1))
        y = oracle.gemm_q6K_f64(blk, xblk, 1, 1, 256)[0, 0]
        expect = np.float64(d) * np.float64(dx) * int((scales * dots).sum())
        assert y == pytest.approx(expect, rel=1e-15, abs=1e-300)


# ------------------------------------------------ whole matmul, f64 check

@pytest.mark.parametrize("fmt", ["q2K", "q3K", "q4K", "q5K", "q6K"])
@pytest.mark.parametrize("seed,m,n,k", [(s, 3, 5, 256) for s in range(8)] + [(0, 4, 33, 1024), (7, 2, 9, 2048)])
def test_integer_path_equals_f64_dequant_matmul(fmt, seed, m, n, k):
    x = gen.normal_f32(seed, 100, m, k)
    xq = oracle.quantize_q8K(x)
    if fmt in ("q2K", "q3K"):
        w = getattr(gen, "%s_blocks" % fmt)(seed, 0, n, k)
        wd = getattr(oracle, "dequant_%s" % fmt)(w, n, k)
        y = getattr(oracle, "gemm_%s_f64" % fmt)(w, xq, m, n, k)
        S = getattr(oracle, "absscale_%s" % fmt)(w, xq, m, n, k)
        y32 = getattr(oracle, "gemm_%s_f32" % fmt)(w, xq, m, n, k)
    elif fmt == "q5K":
        w = gen.q5K_blocks(seed, 0, n, k)
        wd = oracle.dequant_q5K(w, n, k)
        y, S = oracle.gemm_q5K_f64(w, xq, m, n, k), oracle.absscale_q5K(w, xq, m, n, k)
        y32 = oracle.gemm_q5K_f32(w, xq, m, n, k)
    elif fmt == "q4K":
        w = gen.q4K_blocks(seed, 0, n, k)
        wd = oracle.dequant_q4K(w, n, k)
        y, S = oracle.gemm_q4K_f64(w, xq, m, n, k), oracle.absscale_q4K(w, xq, m, n, k)
        y32 = oracle.gemm_q4K_f32(w, xq, m, n, k)
    else:
        w = gen.q6K_blocks(seed, 0, n, k)
        wd = oracle.dequant_q6K(w, n, k)
        y, S = oracle.gemm_q6K_f64(w, xq, m, n, k), oracle.absscale_q6K(w, xq, m, n, k)
        y32 = oracle.gemm_q6K_f32(w, xq, m, n, k)
    ref = oracle.dequant_q8K(xq, m, k) @ wd.T
    assert np.all(np.abs(y - ref) <= 1e-12 * S)
    np.testing.assert_allclose(S, np.abs(oracle.dequant_q8K(xq, m, k)) @ np.abs(wd).T, rtol=1e-12)
    # the f32 block-order combine stays far inside the 1e-4 tolerance
    assert np.all(np.abs(y32 - y) <= 1e-6 * S)


def test_generated_fields_have_stated_ranges():
    w = gen.q4K_blocks(0, 0, 64, 1024).reshape(-1, 144)
    d = w[:, 0:4].copy().view(np.float16).astype(np.float64)
    assert d.min() >= 1e-4 * (1 - 1e-3) and d.max() <= 2e-3 * (1 + 1e-3)
    w6 = gen.q6K_blocks(3, 0, 64, 1024).reshape(-1, 210)
    sc = w6[:, 192:208].view(np.int8)
    assert sc.min() == -64 and sc.max() == 63
    d6 = w6[:, 208:210].copy().view(np.float16).astype(np.float64)
    assert d6.min() >= 1e-4 * (1 - 1e-3) and d6.max() <= 2e-3 * (1 + 1e-3)


def test_swiglu_epilogue_closed_forms():
    """silu(g) * u against identities that do not restate the formula:
    silu(0) = 0; silu(x) - silu(-x) = x; silu(ln 3) = (3/4) ln 3 (sigmoid(ln 3) = 3/4);
    silu(x) -> x for large x and -> 0 for very negative x; u scales h linearly."""
    x = np.linspace(-30.0, 30.0, 601)
    one = np.ones_like(x)
    h = oracle.swiglu_f64(x, one)
    hm = oracle.swiglu_f64(-x, one)
    np.testing.assert_allclose(h - hm, x, rtol=0, atol=1e-12)
    assert oracle.swiglu_f64(np.array([0.0]), np.array([5.0]))[0] == 0.0
    ln3 = np.log(3.0)
    np.testing.assert_allclose(oracle.swiglu_f64(np.array([ln3]), np.array([1.0])), [0.75 * ln3], rtol=1e-15)
    assert abs(oracle.swiglu_f64(np.array([40.0]), np.array([1.0]))[0] - 40.0) < 1e-12
    assert abs(oracle.swiglu_f64(np.array([-40.0]), np.array([1.0]))[0]) < 1e-12
    np.testing.assert_allclose(oracle.swiglu_f64(x, 3.0 * one), 3.0 * h, rtol=1e-15)


# ------------------------------------------------------------------ q5_K


def test_q5K_single_bit_position_map():
    """One set bit -- a low or high nibble bit, or a qh bit -- identifies
    exactly one weight, at the position the format text gives."""
    seen = {}
    for where in range(128 + 32):
        for bit in ((0, 3) if where < 128 else range(8)):
            blk = np.zeros(176, dtype=np.uint8)
            blk[0:2] = np.array([1.0], dtype=np.float16).view(np.uint8)
            blk[4:8] = 1    # scales 0..3 = 1, mins 0..3 = 0
            blk[12:16] = 1  # scales 4..7 = 1, mins 4..7 = 0
            if where < 128:        # qs byte: bit 0 (low nibble) or 4 (high nibble)
                blk[48 + where] = 1 << (4 * (bit // 3))
            else:
                blk[16 + where - 128] = 1 << bit
            w = oracle.dequant_q5K(blk, 1, 256)[0]
            nz = np.nonzero(w)[0]
            assert len(nz) == 1
            if where < 128:
                chunk, l = divmod(where, 32)
                hi = bit // 3
                assert nz[0] == 64 * chunk + 32 * hi + l and w[nz[0]] == 1.0
            else:
                l = where - 128
                chunk, hi = divmod(bit, 2)
                assert nz[0] == 64 * chunk + 32 * hi + l and w[nz[0]] == 16.0
                seen[int(nz[0])] = True
    assert len(seen) == 256


def test_q5K_dequant_dots_and_combine_from_fields():
    rng = np.random.default_rng(11)
    for _ in range(30):
        d = float(np.float16(rng.uniform(1e-4, 2e-3)))
        dmin = float(np.float16(rng.uniform(1e-4, 2e-3)))
        sc, mn, q = rng.integers(0, 64, 8), rng.integers(0, 64, 8), rng.integers(0, 32, 256)
        wblk = pack_q5K(d, dmin, sc, mn, q)
        j = np.arange(256) // 32
        np.testing.assert_array_equal(oracle.dequant_q5K(wblk, 1, 256)[0],
                                      np.float64(d) * sc[j] * q - np.float64(dmin) * mn[j])
        dx = np.float32(rng.uniform(-0.05, 0.05))
        q8 = rng.integers(-128, 128, 256)
        xblk = pack_q8K(dx, q8)
        dots = oracle.subdots_q5K(wblk, xblk, 1, 1, 256)[0, 0]
        np.testing.assert_array_equal(dots, (q * q8).reshape(8, 32).sum(axis=1))
        isum = int((sc * dots).sum())
        msum = int((mn * q8.reshape(8, 32).sum(axis=1)).sum())
        y = oracle.gemm_q5K_f64(wblk, xblk, 1, 1, 256)[0, 0]
        expect = float(np.float64(d) * np.float64(dx) * isum - np.float64(dmin) * np.float64(dx) * msum)
        assert y == pytest.approx(expect, rel=1e-15, abs=1e-300)


def test_q5K_reduces_to_q4K_without_fifth_bits():
    """With qh all zero a q5_K block is the q4_K block of the same fields."""
    rng = np.random.default_rng(12)
    d, dmin = 0.001, 0.0005
    sc, mn, q = rng.integers(0, 64, 8), rng.integers(0, 64, 8), rng.integers(0, 16, 256)
    np.testing.assert_array_equal(oracle.dequant_q5K(pack_q5K(d, dmin, sc, mn, q), 1, 256),
                                  oracle.dequant_q4K(pack_q4K(d, dmin, sc, mn, q), 1, 256))


def test_q5K_generated_fields():
    w = gen.q5K_blocks(5, 0, 64, 1024).reshape(-1, 176)
    d = w[:, 0:4].copy().view(np.float16).astype(np.float64)
    assert d.min() >= 1e-4 * (1 - 1e-3) and d.max() <= 2e-3 * (1 + 1e-3)
    # fifth bits are uniform: about half set
    bits = np.unpackbits(w[:, 16:48])
    assert abs(bits.mean() - 0.5) < 0.01


# ------------------------------------------------------------ q2_K, q3_K


def test_q3K_scale_table_roundtrip_all_values():
    for g in range(16):
        for v in range(64):
            s6 = [(5 * g + 7 * t) % 64 for t in range(16)]
            s6[g] = v
            blk = pack_q3K(1.0, s6, np.zeros(256, dtype=np.int64))
            for gg in range(16):
                assert oracle.q3K_scale(blk[96:108], gg) == s6[gg]


def test_q2K_single_bit_position_map():
    seen = set()
    for byte in range(64):
        for bit in range(8):
            blk = np.zeros(84, dtype=np.uint8)
            blk[0:16] = 1                      # scales 1, mins 0
            blk[16 + byte] = 1 << bit
            blk[80:82] = np.array([1.0], dtype=np.float16).view(np.uint8)
            w = oracle.dequant_q2K(blk, 1, 256)[0]
            nz = np.nonzero(w)[0]
            assert len(nz) == 1 and w[nz[0]] == float(1 << (bit % 2))
            h, rest = divmod(byte, 32)
            p, l = divmod(rest, 16)
            j = bit // 2
            assert nz[0] == 16 * (8 * h + 2 * j + p) + l
            seen.add(int(nz[0]))
    assert seen == set(range(256))


def test_q3K_single_bit_position_maps():
    """qs bits with every third bit set (codes = the low bits), and hmask bits
    over all-zero low bits (codes -4 except where the bit is set: 0)."""
    base = np.zeros(110, dtype=np.uint8)
    base[96:108] = pack_q3K(1.0, [33] * 16, np.zeros(256, dtype=np.int64))[96:108]   # s6 = 33: scale 1
    base[108:110] = np.array([1.0], dtype=np.float16).view(np.uint8)
    seen = set()
    for byte in range(64):
        for bit in range(8):
            blk = base.copy()
            blk[0:32] = 0xFF
            blk[32 + byte] = 1 << bit
            w = oracle.dequant_q3K(blk, 1, 256)[0]
            nz = np.nonzero(w)[0]
            assert len(nz) == 1 and w[nz[0]] == float(1 << (bit % 2))
            h, rest = divmod(byte, 32)
            p, l = divmod(rest, 16)
            assert nz[0] == 16 * (8 * h + 2 * (bit // 2) + p) + l
            seen.add(int(nz[0]))
    assert seen == set(range(256))
    seen = set()
    for byte in range(32):
        for bit in range(8):
            blk = base.copy()
            blk[byte] = 1 << bit
            w = oracle.dequant_q3K(blk, 1, 256)[0]
            z = np.nonzero(w == 0.0)[0]
            assert len(z) == 1 and np.all(np.delete(w, z) == -4.0)
            p, l = divmod(byte, 16)
            h, j = divmod(bit, 4)
            assert z[0] == 16 * (8 * h + 2 * j + p) + l
            seen.add(int(z[0]))
    assert seen == set(range(256))


def test_q2K_q3K_dequant_dots_and_combine_from_fields():
    rng = np.random.default_rng(21)
    for _ in range(20):
        d = float(np.float16(rng.uniform(1e-4, 2e-3)))
        dmin = float(np.float16(rng.uniform(1e-4, 2e-3)))
        dx = np.float32(rng.uniform(-0.05, 0.05))
        q8 = rng.integers(-128, 128, 256)
        xblk = pack_q8K(dx, q8)
        g = np.arange(256) // 16
        # q2_K
        sc, mn, q = rng.integers(0, 16, 16), rng.integers(0, 16, 16), rng.integers(0, 4, 256)
        wblk = pack_q2K(d, dmin, sc, mn, q)
        np.testing.assert_array_equal(oracle.dequant_q2K(wblk, 1, 256)[0],
                                      np.float64(d) * sc[g] * q - np.float64(dmin) * mn[g])
        dots = oracle.subdots_q2K(wblk, xblk, 1, 1, 256)[0, 0]
        np.testing.assert_array_equal(dots, (q * q8).reshape(16, 16).sum(axis=1))
        isum = int((sc * dots).sum())
        msum = int((mn * q8.reshape(16, 16).sum(axis=1)).sum())
        expect = float(np.float64(d) * np.float64(dx) * isum - np.float64(dmin) * np.float64(dx) * msum)
        assert oracle.gemm_q2K_f64(wblk, xblk, 1, 1, 256)[0, 0] == pytest.approx(expect, rel=1e-15, abs=1e-300)
        # q3_K
        s6, q3 = rng.integers(0, 64, 16), rng.integers(-4, 4, 256)
        wblk = pack_q3K(d, s6, q3)
        np.testing.assert_array_equal(oracle.dequant_q3K(wblk, 1, 256)[0], np.float64(d) * (s6[g] - 32) * q3)
        dots = oracle.subdots_q3K(wblk, xblk, 1, 1, 256)[0, 0]
        np.testing.assert_array_equal(dots, (q3 * q8).reshape(16, 16).sum(axis=1))
        expect = float(np.float64(d) * np.float64(dx) * int(((s6 - 32) * dots).sum()))
        assert oracle.gemm_q3K_f64(wblk, xblk, 1, 1, 256)[0, 0] == pytest.approx(expect, rel=1e-15, abs=1e-300)


def test_q2K_zero_codes_and_q3K_zero_codes_closed_forms():
    """q2_K with all codes 0: every weight is -dmin*m_g, so y = -dmin*dx*sum_g m_g*bsum_g;
    q3_K with all codes 0 (low bits 0, third bits set): y = 0."""
    rng = np.random.default_rng(22)
    q8 = rng.integers(-128, 128, 256)
    xblk = pack_q8K(0.01, q8)
    mn = rng.integers(0, 16, 16)
    dmin = 0.0009765625
    y = oracle.gemm_q2K_f64(pack_q2K(0.5, dmin, rng.integers(0, 16, 16), mn, np.zeros(256)), xblk, 1, 1, 256)
    expect = -dmin * np.float64(np.float32(0.01)) * float((mn * q8.reshape(16, 16).sum(axis=1)).sum())
    assert y[0, 0] == pytest.approx(expect, rel=1e-15)
    assert oracle.gemm_q3K_f64(pack_q3K(0.5, rng.integers(0, 64, 16), np.zeros(256)), xblk, 1, 1, 256)[0, 0] == 0.0
