"""Host model of the one-lane q2_K / q3_K decode's code assembly (the GPU's
`lane_block_q23`, codes kept in place).  Bit plane j of a qs word is masked,
not shifted, so each byte holds 4^e times its code (e = j; q3_K: e = min(j, 2),
plane 3 moved down one plane so that the third bit still fits in the byte),
and the hmask bit 4h + j lands on bit 2e + 2.  Every byte must equal 4^e times
the code the shifted form assembles, for every plane and half; and the scaled
group-pair sums must stay inside int32 at the formats' extremes."""
import random


def shifted(w, hm, h, j, q3):
    c = (w >> (2 * j)) & 0x03030303
    if q3:
        c |= ((hm >> (4 * h + j)) & 0x01010101) << 2
    return c


def in_place(w, hm, h, j, q3):
    e = 2 if (q3 and j == 3) else j
    c = (w if e == j else w >> 2) & (0x03030303 << (2 * e))
    if q3:
        hb = hm & (0x01010101 << (4 * h + j))
        sh = 2 * e + 2 - (4 * h + j)
        c |= (hb << sh) if sh >= 0 else (hb >> -sh)
    return c & 0xFFFFFFFF, e


def test_in_place_bytes_are_scaled_codes():
    rng = random.Random(7)
    words = [0, 0xFFFFFFFF, 0xAAAAAAAA, 0x55555555] + [rng.getrandbits(32) for _ in range(3000)]
    for q3 in (False, True):
        for w in words:
            hm = rng.getrandbits(32) if q3 else 0
            for h in range(2):
                for j in range(4):
                    c, e = in_place(w, hm, h, j, q3)
                    s = shifted(w, hm, h, j, q3)
                    for b in range(4):
                        assert (c >> (8 * b)) & 0xFF == ((s >> (8 * b)) & 0xFF) * 4 ** e, (q3, w, hm, h, j, b)


def test_scaled_sums_fit_int32():
    # per group pair: (s0 dot0 + s1 dot1) * 4^(3 - e), dots of 16 codes against q8 in [-128, 127],
    # eight pairs a block
    q2_pair = 2 * 15 * (3 * 4 ** 3) * 128 * 16          # plane 3: codes 3 * 64, scales <= 15
    q3_pair = 2 * 32 * (7 * 4 ** 2) * 128 * 16 * 4      # planes 2, 3: codes 7 * 16, |scale| <= 32
    assert 8 * q2_pair < 2 ** 31 and 8 * q3_pair < 2 ** 31
