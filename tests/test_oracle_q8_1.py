"""Pins for the oracle's fp16 conversion and Q8_1 activation quantiser.

fp16: checked against numpy's IEEE binary16 conversion (a library routine),
exhaustively for decode and on edge + random values for encode.

Q8_1 ("Strata" PR #2340 "int4 activation loads": 32 int8 quants behind a
4-byte header; PR #1774: block value d * ds * sumi): closed forms and
invariants that a plausible slip (a wrong rounding rule, d from the wrong
amax, s from the rounded d, a sign error) would break.
"""
import numpy as np
import pytest

import oracle
from tests._formats import q8_1_fields


def test_f16_decode_all_patterns_match_numpy():
    h = np.arange(65536, dtype=np.uint16)
    got = oracle.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f16_encode_matches_numpy_on_edges_and_random():
    rng = np.random.default_rng(7)
    # every fp16 value, the midpoints between neighbours (ties), and +-1 ulp around them
    h = np.arange(0, 0x7C00, dtype=np.uint16)
    v = h.view(np.float16).astype(np.float64)
    mids = (v[:-1] + v[1:]) / 2
    mids32 = mids.astype(np.float32)
    near = np.concatenate([mids32, np.nextafter(mids32, np.float32(np.inf)),
                           np.nextafter(mids32, np.float32(0))])
    rand = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 200000).astype(np.float32),
        rng.uniform(-70000, 70000, 50000).astype(np.float32),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, np.inf, -np.inf,
                  2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -14, 6e-8], np.float32),
    ])
    x = np.concatenate([v.astype(np.float32), near, -near, rand]).astype(np.float32)
    got = oracle.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):  # values past the fp16 range map to infinity on purpose
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def _q(x):
    xq = oracle.quantize_q8_1(np.asarray(x, np.float32)[None, :])
    d, s, q = q8_1_fields(xq[0, 0])
    return d, s, q, xq[0, 0]


def test_q8_1_all_zero_block():
    d, s, q, raw = _q(np.zeros(32))
    assert d == 0.0 and s == 0.0 and not q.any()
    assert not raw.any()


@pytest.mark.parametrize("pos,val", [(0, 1.0), (31, -3.7), (17, 1e-3), (5, -250.5)])
def test_q8_1_single_nonzero(pos, val):
    x = np.zeros(32, np.float32)
    x[pos] = val
    d, s, q, _ = _q(x)
    d32 = np.float32(abs(np.float32(val))) / np.float32(127)
    assert d == float(np.float16(d32))
    assert q[pos] == (127 if val > 0 else -127)
    assert np.count_nonzero(q) == 1
    assert s == float(np.float16(d32 * np.float32(q[pos])))


def test_q8_1_ties_round_half_away_from_zero():
    # amax = 127 makes d exactly 1, so x/d = x and every k + 0.5 is an exact tie.
    x = np.array([127.0, 0.5, -0.5, 1.5, -1.5, 2.5, -2.5, 3.5, 100.5, -100.5, 126.5, -126.5,
                  0.49999997, 2.4999998] + [0.0] * 18, np.float32)
    d, _, q, _ = _q(x)
    assert d == 1.0
    want = [127, 1, -1, 2, -2, 3, -3, 4, 101, -101, 127, -127, 0, 2]
    assert list(q[:14]) == want


def test_q8_1_sign_symmetry_and_power_of_two_scaling():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((64, 32)).astype(np.float32)
    a = oracle.quantize_q8_1(x.reshape(1, -1))
    b = oracle.quantize_q8_1(-x.reshape(1, -1))
    c = oracle.quantize_q8_1((x * np.float32(4)).reshape(1, -1))
    da, sa, qa = q8_1_fields(a)
    db, sb, qb = q8_1_fields(b)
    dc, sc, qc = q8_1_fields(c)
    assert np.array_equal(qa, -qb) and np.array_equal(da, db) and np.array_equal(sa, -sb)
    assert np.array_equal(qa, qc) and np.array_equal(dc, 4 * da) and np.array_equal(sc, 4 * sa)


def test_q8_1_bounds_and_reconstruction_error():
    rng = np.random.default_rng(12)
    K = 32 * 200
    x = (rng.standard_normal(K) * rng.uniform(0.01, 100, K)).astype(np.float32)
    d, s, q = q8_1_fields(oracle.quantize_q8_1(x[None, :])[0])
    xb = x.reshape(-1, 32).astype(np.float64)
    assert np.abs(q).max() <= 127
    # the element of largest magnitude maps to +-127
    idx = np.abs(xb).argmax(axis=1)
    assert np.all(np.abs(q[np.arange(q.shape[0]), idx]) == 127)
    # |x - q*d| <= d/2 up to the fp16 rounding of d (relative 2^-11, times |q| <= 127)
    err = np.abs(xb - q * d[:, None])
    assert np.all(err <= d[:, None] * (0.5 + 127 * 2.0 ** -11) + 1e-30)
    # s is d*sum(q) rounded once to fp16 (relative 2^-11 plus d's own rounding)
    ssum = q.sum(axis=1) * d
    assert np.all(np.abs(s - ssum) <= np.abs(ssum) * 2 * 2.0 ** -11 + 1e-12)


def test_q8_1_respects_ldx_and_columns():
    rng = np.random.default_rng(13)
    x = rng.standard_normal((3, 160)).astype(np.float32)
    full = oracle.quantize_q8_1(x, K=128)
    for c in range(3):
        one = oracle.quantize_q8_1(np.ascontiguousarray(x[c, :128])[None, :])
        assert np.array_equal(full[c], one[0])
