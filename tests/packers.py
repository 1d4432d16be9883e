"""Block packers for the host tests, written from the public GGML K-quant
format text (the formats the PocketLLM pages name), in the opposite direction
to the oracle's decoders: fields in, bytes out.  A round trip through an
oracle decoder therefore pins that decoder against the format text, not
against itself.
"""
import numpy as np


def f16_bits(v):
    return np.array([v], dtype=np.float16).view(np.uint16)[0]


def pack_q4K(d, dmin, sc, mn, q):
    """d, dmin: floats (stored as f16); sc, mn: 8 ints in 0..63; q: 256 ints in 0..15."""
    sc = [int(v) for v in sc]
    mn = [int(v) for v in mn]
    blk = np.zeros(144, dtype=np.uint8)
    blk[0:2] = np.array([d], dtype=np.float16).view(np.uint8)
    blk[2:4] = np.array([dmin], dtype=np.float16).view(np.uint8)
    t = np.zeros(12, dtype=np.int64)
    # pairs 0..3: low six bits of bytes 0..3 (scales) and 4..7 (mins)
    for j in range(4):
        t[j] |= sc[j] & 63
        t[j + 4] |= mn[j] & 63
    # pairs 4..7: low four bits in bytes 8..11 (scale low nibble, min high
    # nibble); the two top bits go into bits 6-7 of bytes j-4 (scale) and j (min)
    for j in range(4, 8):
        t[j + 4] |= (sc[j] & 15) | ((mn[j] & 15) << 4)
        t[j - 4] |= (sc[j] >> 4) << 6
        t[j] |= (mn[j] >> 4) << 6
    blk[4:16] = t.astype(np.uint8)
    q = np.asarray(q, dtype=np.int64)
    w = np.arange(256)
    chunk, within = w // 64, w % 64
    byte = 32 * chunk + within % 32
    qs = np.zeros(128, dtype=np.int64)
    lo = within < 32
    qs[byte[lo]] |= q[lo]
    qs[byte[~lo]] |= q[~lo] << 4
    blk[16:144] = qs.astype(np.uint8)
    return blk


def pack_q5K(d, dmin, sc, mn, q):
    """q5_K: q4_K's header and scale table, then qh[32] holding the fifth bit of
    every weight, then qs[128].  q: 256 ints in 0..31.  Weight 64c + l (l < 32)
    keeps its low four bits in the low nibble of qs[32c + l] and its fifth bit
    in bit 2c of qh[l]; weight 64c + 32 + l uses the high nibble and bit 2c+1."""
    q = np.asarray(q, dtype=np.int64)
    q4 = pack_q4K(d, dmin, sc, mn, q & 15)
    blk = np.zeros(176, dtype=np.uint8)
    blk[0:16] = q4[0:16]
    blk[48:176] = q4[16:144]
    qh = np.zeros(32, dtype=np.int64)
    for w in range(256):
        chunk, within = divmod(w, 64)
        l, upper = within % 32, int(within >= 32)
        qh[l] |= ((q[w] >> 4) & 1) << (2 * chunk + upper)
    blk[16:48] = qh.astype(np.uint8)
    return blk


def _k2_positions():
    """Weight w of a q2_K/q3_K block: group g = w // 16 (h = g // 8, j = (g % 8) // 2,
    p = g % 2), lane l = w % 16; its two low bits are bits 2j, 2j+1 of
    qs[32h + 16p + l]; q3_K's third bit is bit 4h + j of hmask[16p + l]."""
    w = np.arange(256)
    g, l = w // 16, w % 16
    h, j, p = g // 8, (g % 8) // 2, g % 2
    return 32 * h + 16 * p + l, 2 * j, 16 * p + l, 4 * h + j


def pack_q2K(d, dmin, sc, mn, q):
    """d, dmin: floats (f16); sc, mn: 16 ints in 0..15; q: 256 two-bit codes."""
    q = np.asarray(q, dtype=np.int64)
    byte, shift, _, _ = _k2_positions()
    qs = np.zeros(64, dtype=np.int64)
    for w in range(256):
        qs[byte[w]] |= (q[w] & 3) << shift[w]
    blk = np.zeros(84, dtype=np.uint8)
    blk[0:16] = (np.asarray(sc, dtype=np.int64) & 15) | ((np.asarray(mn, dtype=np.int64) & 15) << 4)
    blk[16:80] = qs.astype(np.uint8)
    blk[80:82] = np.array([d], dtype=np.float16).view(np.uint8)
    blk[82:84] = np.array([dmin], dtype=np.float16).view(np.uint8)
    return blk


def pack_q3K(d, s6, q3):
    """d: float (f16); s6: 16 six-bit scales 0..63 (the weight uses s6 - 32);
    q3: 256 codes in -4..3 (stored as two low bits plus a third bit that is set
    when the code is >= 0)."""
    q3 = np.asarray(q3, dtype=np.int64)
    s6 = [int(v) for v in s6]
    byte, shift, hbyte, hbit = _k2_positions()
    qs = np.zeros(64, dtype=np.int64)
    hm = np.zeros(32, dtype=np.int64)
    for w in range(256):
        high = 1 if q3[w] >= 0 else 0
        low = q3[w] if high else q3[w] + 4
        qs[byte[w]] |= low << shift[w]
        hm[hbyte[w]] |= high << hbit[w]
    t = np.zeros(12, dtype=np.int64)
    for g in range(16):
        t[g % 8] |= (s6[g] & 15) << (4 * (g // 8))
        t[8 + g % 4] |= ((s6[g] >> 4) & 3) << (2 * (g // 4))
    blk = np.zeros(110, dtype=np.uint8)
    blk[0:32] = hm.astype(np.uint8)
    blk[32:96] = qs.astype(np.uint8)
    blk[96:108] = t.astype(np.uint8)
    blk[108:110] = np.array([d], dtype=np.float16).view(np.uint8)
    return blk


def pack_q6K(d, scales, q):
    """d: float (f16); scales: 16 ints in -128..127; q: 256 six-bit codes 0..63."""
    q = np.asarray(q, dtype=np.int64)
    blk = np.zeros(210, dtype=np.uint8)
    ql = np.zeros(128, dtype=np.int64)
    qh = np.zeros(64, dtype=np.int64)
    for w in range(256):
        half, r = divmod(w, 128)
        quarter, l = divmod(r, 32)
        ql_idx = 64 * half + 32 * (quarter % 2) + l
        shift = 4 if quarter >= 2 else 0
        ql[ql_idx] |= (q[w] & 15) << shift
        qh[32 * half + l] |= (q[w] >> 4) << (2 * quarter)
    blk[0:128] = ql.astype(np.uint8)
    blk[128:192] = qh.astype(np.uint8)
    blk[192:208] = np.asarray(scales, dtype=np.int64).astype(np.int8).view(np.uint8)
    blk[208:210] = np.array([d], dtype=np.float16).view(np.uint8)
    return blk


def pack_q8K(d, qs):
    """A q8_K block from its scale and codes; bsums are the 16-element sums."""
    qs = np.asarray(qs, dtype=np.int64)
    blk = np.zeros(292, dtype=np.uint8)
    blk[0:4] = np.array([d], dtype=np.float32).view(np.uint8)
    blk[4:260] = qs.astype(np.int8).view(np.uint8)
    blk[260:292] = qs.reshape(16, 16).sum(axis=1).astype(np.int16).view(np.uint8)
    return blk


def pack_q4K_x16(w, n, k):
    """The row-interleaved x16 form of q4_K weights w [n][k/256 * 144], built
    from the layout text in the packing direction: for every tile T (rows
    16T..16T+15, zero blocks past n) and block b, a 2304-byte tile-block made
    of the 16 headers (bytes 0..15 of each row's block) and, for j = 0..3 and
    L = 0..31, the 16-byte piece qs[32(L%4) + 16(j%2) ..] of row L//4 (+8 when
    j >= 2)."""
    nb = k // 256
    ntiles = -(-n // 16)
    src = np.zeros((ntiles * 16, nb, 144), dtype=np.uint8)
    src[:n] = np.asarray(w, dtype=np.uint8).reshape(n, nb, 144)
    out = np.zeros((ntiles, nb, 2304), dtype=np.uint8)
    for T in range(ntiles):
        for b in range(nb):
            tb = out[T, b]
            for i in range(16):
                tb[16 * i:16 * i + 16] = src[16 * T + i, b, 0:16]
            for j in range(4):
                for L in range(32):
                    row = 16 * T + L // 4 + (8 if j >= 2 else 0)
                    q0 = 16 + 32 * (L % 4) + 16 * (j % 2)     # qs starts at byte 16 of the block
                    off = 256 + 512 * j + 16 * L
                    tb[off:off + 16] = src[row, b, q0:q0 + 16]
    return out.reshape(-1)


def pack_q6K_x16(w, n, k):
    """The x16 form of q6_K weights w [n][k/256 * 210], built from the layout
    text in the packing direction: per tile T and block b, 3360 bytes: the 16
    rows' int8 scales (16 bytes each), their f16 d (2 bytes each), then for
    j = 0..3 and L = 0..31 the 16 bytes ql[64(j%2) + 16w + 4(L%4) ..+4] for
    w = 0..3 of row L//4 (+8 when j >= 2), then for j = 0..1 the 16 bytes
    qh[32h + 16s + 4(L%4) ..+4] for (h, s) = (0,0), (0,1), (1,0), (1,1) of row
    L//4 + 8j."""
    nb = k // 256
    ntiles = -(-n // 16)
    src = np.zeros((ntiles * 16, nb, 210), dtype=np.uint8)
    src[:n] = np.asarray(w, dtype=np.uint8).reshape(n, nb, 210)
    out = np.zeros((ntiles, nb, 3360), dtype=np.uint8)
    for T in range(ntiles):
        for b in range(nb):
            tb = out[T, b]
            blk = src[16 * T:16 * T + 16, b]
            for i in range(16):
                tb[16 * i:16 * i + 16] = blk[i, 192:208]
                tb[256 + 2 * i:258 + 2 * i] = blk[i, 208:210]
            for j in range(4):
                for L in range(32):
                    row = L // 4 + (8 if j >= 2 else 0)
                    base = 288 + 512 * j + 16 * L
                    for w4 in range(4):
                        q = 64 * (j % 2) + 16 * w4 + 4 * (L % 4)
                        tb[base + 4 * w4:base + 4 * w4 + 4] = blk[row, q:q + 4]
            for j in range(2):
                for L in range(32):
                    row = L // 4 + 8 * j
                    base = 2336 + 512 * j + 16 * L
                    for p, (h, s) in enumerate([(0, 0), (0, 1), (1, 0), (1, 1)]):
                        q = 128 + 32 * h + 16 * s + 4 * (L % 4)
                        tb[base + 4 * p:base + 4 * p + 4] = blk[row, q:q + 4]
    return out.reshape(-1)
