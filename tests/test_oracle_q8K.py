"""Pins for the oracle's q8_K activation quantizer (host only).

The rule comes from the q8_K description of the packed matmul's activation
path ("Current status" table of the PocketLLM pages, row "src/ -- the C++
engine"; activations quantized to int8 one 256-element block at a time).
"""
import os

import numpy as np
import pytest

import gen
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q8K_hand_cases.txt")


def _parse_cases(path):
    cases, cur = [], None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(" ")
        if key == "case":
            cur = {"name": rest, "x": {}, "qs": {}, "bsums": {}}
            cases.append(cur)
        elif key == "d":
            cur["d"] = float(rest)
        else:
            for tok in rest.split():
                i, v = tok.split(":")
                cur[key][int(i)] = float(v) if key == "x" else int(v)
    return cases


CASES = _parse_cases(GOLDEN)


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_hand_cases(case):
    x = np.zeros((1, 256), dtype=np.float32)
    for i, v in case["x"].items():
        x[0, i] = v
    f = oracle.q8K_fields(oracle.quantize_q8K(x), 1, 256)[0, 0]
    exp_qs = np.zeros(256, dtype=np.int64)
    for i, c in case["qs"].items():
        exp_qs[i] = c
    exp_bs = np.zeros(16, dtype=np.int64)
    for g, s in case["bsums"].items():
        exp_bs[g] = s
    assert f["d"] == np.float32(case["d"])
    np.testing.assert_array_equal(f["qs"].astype(np.int64), exp_qs)
    np.testing.assert_array_equal(f["bsums"].astype(np.int64), exp_bs)


def _numpy_q8K(x):
    """The same rule through numpy primitives: argmax (first occurrence),
    f32 divide and multiply, np.rint (ties to even)."""
    m, k = x.shape
    blocks = x.reshape(m, k // 256, 256)
    idx = np.argmax(np.abs(blocks), axis=2)
    mx = np.take_along_axis(blocks, idx[..., None], axis=2)[..., 0]
    zero = mx == 0
    safe = np.where(zero, np.float32(1), mx).astype(np.float32)
    iscale = (np.float32(-128.0) / safe).astype(np.float32)
    prod = (iscale[..., None] * blocks).astype(np.float32)
    q = np.minimum(np.rint(prod), 127).astype(np.int64)
    q[zero] = 0
    d = (np.float32(1.0) / iscale).astype(np.float32)
    d[zero] = 0
    return d, q, q.reshape(m, k // 256, 16, 16).sum(axis=3)


@pytest.mark.parametrize("seed,m,k", [(0, 1, 1024), (2, 7, 2048), (5, 3, 256)])
def test_matches_numpy_restatement(seed, m, k):
    x = gen.normal_f32(seed, 11, m, k)
    x[0, :256:7] = 0.0  # zeros and a few exact ties on magnitude
    x[0, 300 % k] = -x[0, 301 % k]
    f = oracle.q8K_fields(oracle.quantize_q8K(x), m, k)
    d, q, bs = _numpy_q8K(x)
    np.testing.assert_array_equal(f["d"], d)
    np.testing.assert_array_equal(f["qs"].astype(np.int64), q)
    np.testing.assert_array_equal(f["bsums"].astype(np.int64), bs)


def test_invariants_random():
    m, k = 16, 4096
    x = gen.normal_f32(9, 3, m, k) * np.float32(3.0)
    f = oracle.q8K_fields(oracle.quantize_q8K(x), m, k)
    xb = x.reshape(m, k // 256, 256)
    qs = f["qs"].astype(np.int64)
    # the largest-magnitude element (first occurrence) maps to exactly -128
    idx = np.argmax(np.abs(xb), axis=2)
    np.testing.assert_array_equal(np.take_along_axis(qs, idx[..., None], axis=2), -128)
    # every code is within half a step of its input, except the clamp at +128
    d = f["d"].astype(np.float64)[..., None]
    err = np.abs(qs * d - xb.astype(np.float64))
    clamped = (qs == 127) & (np.abs(xb.astype(np.float64) / d - 127) > 0.5)
    assert np.all(err[~clamped] <= 0.5 * np.abs(d).repeat(256, axis=2)[~clamped] * (1 + 1e-6))
    # bsums are the 16-element sums
    np.testing.assert_array_equal(f["bsums"], qs.reshape(m, k // 256, 16, 16).sum(axis=3))
    assert qs.min() >= -128 and qs.max() <= 127


def test_all_zero_chunk_between_nonzero():
    x = gen.normal_f32(1, 1, 1, 768)
    x[0, 256:512] = 0.0
    f = oracle.q8K_fields(oracle.quantize_q8K(x), 1, 768)[0]
    assert f[1]["d"] == 0 and not f[1]["qs"].any() and not f[1]["bsums"].any()
    assert f[0]["d"] != 0 and f[2]["d"] != 0
