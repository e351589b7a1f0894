"""Pins for the oracle's Q6_K / Q4_K decodes, per-32-block integer sums and
FP32 block products.

* Decodes: brute force over every weight position and every code value, and
  over every (scale, min) pair of every Q4_K sub-block, through independently
  written encoders (tests/_formats.py).  A transposed index, a swapped nibble
  or a misplaced 2-bit field fails here.
* Block sums: exact integers from the ORIGINAL fields (before encoding), so
  the check does not go through the oracle's decode.
* Products: an fp64 dot product of the original fields against the Q8_1
  activations, within |dy| <= 1e-5 * sum|t_b| + 1e-6 ("Strata" PR #1774:
  sub-block order only moves the last bits); closed forms (zero
  activations; all codes 32; one nonzero weight gives
  d*scale*(q-32)*d_a*q_a); column linearity.
"""
import numpy as np
import pytest

import oracle
from block_quantized_matvec_gb300 import synth
from tests._formats import encode_q4_k, encode_q6_k, q8_1_fields

Q6, Q4 = oracle.TYPE_Q6_K, oracle.TYPE_Q4_K


def test_q6_k_decode_every_position_every_code():
    rng = np.random.default_rng(21)
    sc = rng.integers(-32, 32, 16).astype(np.int8)
    for n in range(256):
        for v in range(64):
            q = np.full(256, 32, np.int64)
            q[n] = v
            got, gsc, gd = oracle.decode_q6_k(encode_q6_k(q, sc, 0.5))
            assert got[n] == v, (n, v)
            assert np.count_nonzero(got != 32) == (v != 32)
        assert np.array_equal(gsc, sc) and gd == 0.5


def test_q6_k_decode_random_round_trip():
    rng = np.random.default_rng(22)
    for _ in range(200):
        q = rng.integers(0, 64, 256)
        sc = rng.integers(-32, 32, 16).astype(np.int8)
        d = float(np.float16(rng.uniform(1e-3, 1e-2)))
        got, gsc, gd = oracle.decode_q6_k(encode_q6_k(q, sc, d))
        assert np.array_equal(got, q) and np.array_equal(gsc, sc) and gd == d


def test_q4_k_decode_every_scale_min_pair_every_subblock():
    rng = np.random.default_rng(23)
    pairs = np.array([(a, b) for a in range(64) for b in range(64)])
    for j in range(8):
        for a, b in pairs:
            sc = rng.integers(0, 64, 8)
            m = rng.integers(0, 64, 8)
            sc[j], m[j] = a, b
            q = rng.integers(0, 16, 256)
            blk = encode_q4_k(q, sc, m, 0.25, 0.125)
            gq, gsc, gm, gd, gdm = oracle.decode_q4_k(blk)
            assert gsc[j] == a and gm[j] == b
            assert np.array_equal(gsc, sc) and np.array_equal(gm, m)
        assert np.array_equal(gq, q) and gd == 0.25 and gdm == 0.125


def test_q4_k_decode_every_nibble_position():
    for n in range(256):
        for v in range(16):
            q = np.zeros(256, np.int64)
            q[n] = v
            gq, *_ = oracle.decode_q4_k(encode_q4_k(q, np.zeros(8), np.zeros(8), 1.0, 1.0))
            assert gq[n] == v and np.count_nonzero(gq) == (v != 0)


# ---------------------------------------------------------------- products --

def _random_q6_k(rows, K, rng):
    nb = K // 256
    fields = []
    W = np.empty((rows, nb, 210), np.uint8)
    for r in range(rows):
        for b in range(nb):
            q = rng.integers(0, 64, 256)
            sc = rng.integers(-32, 32, 16).astype(np.int8)
            d = float(np.float16(rng.uniform(1e-3, 1e-2)))
            W[r, b] = encode_q6_k(q, sc, d)
            fields.append((r, b, q, sc.astype(np.int64), d))
    return W, fields


def _random_q4_k(rows, K, rng):
    nb = K // 256
    fields = []
    W = np.empty((rows, nb, 144), np.uint8)
    for r in range(rows):
        for b in range(nb):
            q = rng.integers(0, 16, 256)
            sc = rng.integers(0, 64, 8)
            m = rng.integers(0, 64, 8)
            d = float(np.float16(rng.uniform(1e-3, 1e-2)))
            dm = float(np.float16(rng.uniform(1e-3, 1e-2)))
            W[r, b] = encode_q4_k(q, sc, m, d, dm)
            fields.append((r, b, q, sc, m, d, dm))
    return W, fields


def _ref_q6_k(fields, rows, K, xq, ncols):
    """fp64 reference and exact integer block sums from the original fields."""
    da, _, qa = q8_1_fields(xq)            # [ncols, K/32], [ncols, K/32, 32]
    y = np.zeros((ncols, rows))
    mag = np.zeros((ncols, rows))
    sumi = np.zeros((ncols, rows, K // 32), np.int64)
    for (r, b, q, sc, d) in fields:
        w = (q - 32) * np.repeat(sc, 16)                      # sc * (q-32), per weight
        for c in range(ncols):
            a = qa[c, 8 * b:8 * b + 8].reshape(256)
            prod = (w * a).reshape(8, 32).sum(axis=1)         # integer per 32-block
            sumi[c, r, 8 * b:8 * b + 8] = prod
            t = d * da[c, 8 * b:8 * b + 8] * prod
            y[c, r] += t.sum()
            mag[c, r] += np.abs(t).sum()
    return y, mag, sumi


def _ref_q4_k(fields, rows, K, xq, ncols):
    da, sa, qa = q8_1_fields(xq)
    y = np.zeros((ncols, rows))
    mag = np.zeros((ncols, rows))
    sumi = np.zeros((ncols, rows, K // 32), np.int64)
    for (r, b, q, sc, m, d, dm) in fields:
        for c in range(ncols):
            a = qa[c, 8 * b:8 * b + 8]                        # [8, 32]
            prod = sc * (q.reshape(8, 32) * a).sum(axis=1)
            sumi[c, r, 8 * b:8 * b + 8] = prod
            tq = d * da[c, 8 * b:8 * b + 8] * prod
            tm = dm * m * sa[c, 8 * b:8 * b + 8]
            y[c, r] += (tq - tm).sum()
            mag[c, r] += (np.abs(tq) + np.abs(tm)).sum()
    return y, mag, sumi


@pytest.mark.parametrize("rows,K,ncols", [(1, 256, 1), (3, 512, 2), (4, 256, 8), (2, 768, 5)])
@pytest.mark.parametrize("kind", ["q6_k", "q4_k"])
def test_products_match_fp64_dot_of_original_fields(kind, rows, K, ncols):
    rng = np.random.default_rng(hash((kind, rows, K, ncols)) % 2**32)
    x = rng.standard_normal((ncols, K)).astype(np.float32)
    xq = oracle.quantize_q8_1(x)
    if kind == "q6_k":
        W, f = _random_q6_k(rows, K, rng)
        yr, mag, sref = _ref_q6_k(f, rows, K, xq, ncols)
        t = Q6
    else:
        W, f = _random_q4_k(rows, K, rng)
        yr, mag, sref = _ref_q4_k(f, rows, K, xq, ncols)
        t = Q4
    y, bound = oracle.gemv(t, W, rows, K, xq, ncols, with_bound=True)
    assert np.all(np.abs(y - yr) <= 1e-5 * mag + 1e-6)
    assert np.allclose(bound, mag, rtol=1e-5, atol=1e-9)
    s = oracle.block_sums(t, W, rows, K, xq, ncols)
    assert np.array_equal(s, sref)


@pytest.mark.parametrize("kind", ["q6_k", "q4_k"])
def test_zero_activations_give_exact_zero(kind):
    rows, K = 5, 512
    W = synth.q6_k_weights(rows, K) if kind == "q6_k" else synth.q4_k_weights(rows, K)
    xq = oracle.quantize_q8_1(np.zeros((3, K), np.float32))
    y = oracle.gemv(Q6 if kind == "q6_k" else Q4, W, rows, K, xq, 3)
    assert np.all(y == 0.0) and not np.signbit(y).any()


def test_q6_k_all_codes_32_give_exact_zero():
    rng = np.random.default_rng(31)
    K = 512
    W = np.stack([encode_q6_k(np.full(256, 32), rng.integers(-32, 32, 16).astype(np.int8), 0.01)
                  for _ in range(2 * 2)]).reshape(2, 2, 210)
    xq = oracle.quantize_q8_1(rng.standard_normal((2, K)).astype(np.float32))
    assert np.all(oracle.gemv(Q6, W, 2, K, xq, 2) == 0.0)


@pytest.mark.parametrize("n,code", [(0, 0), (77, 63), (200, 5), (255, 40)])
def test_q6_k_single_nonzero_weight_closed_form(n, code):
    rng = np.random.default_rng(n)
    K = 256
    sc = rng.integers(-32, 32, 16).astype(np.int8)
    q = np.full(256, 32)
    q[n] = code
    d = float(np.float16(0.0061))
    W = encode_q6_k(q, sc, d).reshape(1, 1, 210)
    xq = oracle.quantize_q8_1(rng.standard_normal((1, K)).astype(np.float32))
    da, _, qa = q8_1_fields(xq[0, n // 32])
    want = (np.float32(d) * np.float32(da)) * np.float32(int(sc[n // 16]) * (code - 32) * int(qa[n % 32]))
    assert oracle.gemv(Q6, W, 1, K, xq, 1)[0, 0] == want


@pytest.mark.parametrize("n,code", [(3, 15), (130, 1)])
def test_q4_k_single_nonzero_weight_closed_form(n, code):
    rng = np.random.default_rng(n)
    sc = rng.integers(1, 64, 8)
    m = np.zeros(8, np.int64)
    q = np.zeros(256)
    q[n] = code
    W = encode_q4_k(q, sc, m, 0.0078125, 0.003).reshape(1, 1, 144)
    xq = oracle.quantize_q8_1(rng.standard_normal((1, 256)).astype(np.float32))
    da, _, qa = q8_1_fields(xq[0, n // 32])
    want = (np.float32(0.0078125) * np.float32(da)) * np.float32(int(sc[n // 32]) * code * int(qa[n % 32]))
    assert oracle.gemv(Q4, W, 1, 256, xq, 1)[0, 0] == want


@pytest.mark.parametrize("kind", ["q6_k", "q4_k"])
def test_columns_are_independent(kind):
    rows, K, ncols = 7, 768, 6
    W = synth.q6_k_weights(rows, K, salt=3) if kind == "q6_k" else synth.q4_k_weights(rows, K, salt=3)
    t = Q6 if kind == "q6_k" else Q4
    xq = oracle.quantize_q8_1(synth.activations(K, ncols))
    y = oracle.gemv(t, W, rows, K, xq, ncols)
    for c in range(ncols):
        one = oracle.gemv(t, W, rows, K, np.ascontiguousarray(xq[c:c + 1]), 1)
        assert np.array_equal(y[c], one[0])
