"""Pins for the oracle's Q5_K decode, products and planar tiles.  The pages
run Q5_K matrices through the wide kernels (PR #2340 "ld_i4_a4"; the A770
dense_bench table) without giving the block; the reading is the GGUF Q5_K
arrangement (tests/_formats.py restates it independently of the oracle).

* Decode: every weight position x every 5-bit code, every (scale, min) pair
  of every sub-block, random round trips, through the test-side encoder.
* Products: exact integer block sums and an fp64 dot product of the ORIGINAL
  fields; a single nonzero weight (codes below and above 16) in closed form;
  zero activations; column independence.
* Planar tiles: round trip, size, marker bytes where the tile specification
  puts them, zero pad rows, products unchanged.
"""
import numpy as np
import pytest

import oracle
from block_quantized_matvec_gb300 import synth
from tests._formats import encode_q5_k, q8_1_fields

Q5, Q5P = oracle.TYPE_Q5_K, oracle.TYPE_Q5_K_PLANAR


def test_decode_every_position_every_code():
    for n in range(256):
        for v in range(32):
            q = np.zeros(256, np.int64)
            q[n] = v
            gq, *_ = oracle.decode_q5_k(encode_q5_k(q, np.zeros(8), np.zeros(8), 1.0, 1.0))
            assert gq[n] == v and np.count_nonzero(gq) == (v != 0), (n, v)


def test_decode_every_scale_min_pair_every_subblock():
    rng = np.random.default_rng(51)
    for j in range(8):
        for a in range(64):
            for b in range(64):
                sc = rng.integers(0, 64, 8)
                m = rng.integers(0, 64, 8)
                sc[j], m[j] = a, b
                gq, gsc, gm, gd, gdm = oracle.decode_q5_k(
                    encode_q5_k(np.zeros(256), sc, m, 0.25, 0.125))
                assert np.array_equal(gsc, sc) and np.array_equal(gm, m)
        assert gd == 0.25 and gdm == 0.125


def test_decode_random_round_trip():
    rng = np.random.default_rng(52)
    for _ in range(200):
        q = rng.integers(0, 32, 256)
        sc = rng.integers(0, 64, 8)
        m = rng.integers(0, 64, 8)
        d = float(np.float16(rng.uniform(1e-3, 1e-2)))
        dm = float(np.float16(rng.uniform(1e-3, 1e-2)))
        gq, gsc, gm, gd, gdm = oracle.decode_q5_k(encode_q5_k(q, sc, m, d, dm))
        assert np.array_equal(gq, q) and np.array_equal(gsc, sc) and np.array_equal(gm, m)
        assert gd == d and gdm == dm


def _random_q5_k(rows, K, rng):
    nb = K // 256
    fields = []
    W = np.empty((rows, nb, 176), np.uint8)
    for r in range(rows):
        for b in range(nb):
            q = rng.integers(0, 32, 256)
            sc = rng.integers(0, 64, 8)
            m = rng.integers(0, 64, 8)
            d = float(np.float16(rng.uniform(1e-3, 1e-2)))
            dm = float(np.float16(rng.uniform(1e-3, 1e-2)))
            W[r, b] = encode_q5_k(q, sc, m, d, dm)
            fields.append((r, b, q, sc, m, d, dm))
    return W, fields


@pytest.mark.parametrize("rows,K,ncols", [(1, 256, 1), (3, 512, 2), (4, 256, 8), (2, 768, 5)])
def test_products_match_fp64_dot_of_original_fields(rows, K, ncols):
    rng = np.random.default_rng(rows * 1000 + K + ncols)
    x = rng.standard_normal((ncols, K)).astype(np.float32)
    xq = oracle.quantize_q8_1(x)
    W, fields = _random_q5_k(rows, K, rng)
    da, sa, qa = q8_1_fields(xq)
    yr = np.zeros((ncols, rows))
    mag = np.zeros((ncols, rows))
    sref = np.zeros((ncols, rows, K // 32), np.int64)
    for (r, b, q, sc, m, d, dm) in fields:
        for c in range(ncols):
            a = qa[c, 8 * b:8 * b + 8]
            prod = sc * (q.reshape(8, 32) * a).sum(axis=1)
            sref[c, r, 8 * b:8 * b + 8] = prod
            tq = d * da[c, 8 * b:8 * b + 8] * prod
            tm = dm * m * sa[c, 8 * b:8 * b + 8]
            yr[c, r] += (tq - tm).sum()
            mag[c, r] += (np.abs(tq) + np.abs(tm)).sum()
    y, bound = oracle.gemv(Q5, W, rows, K, xq, ncols, with_bound=True)
    assert np.all(np.abs(y - yr) <= 1e-5 * mag + 1e-6)
    assert np.allclose(bound, mag, rtol=1e-5, atol=1e-9)
    assert np.array_equal(oracle.block_sums(Q5, W, rows, K, xq, ncols), sref)


@pytest.mark.parametrize("n,code", [(3, 15), (130, 16), (255, 31), (64, 1)])
def test_single_nonzero_weight_closed_form(n, code):
    rng = np.random.default_rng(n)
    sc = rng.integers(1, 64, 8)
    q = np.zeros(256)
    q[n] = code
    W = encode_q5_k(q, sc, np.zeros(8), 0.0078125, 0.003).reshape(1, 1, 176)
    xq = oracle.quantize_q8_1(rng.standard_normal((1, 256)).astype(np.float32))
    da, _, qa = q8_1_fields(xq[0, n // 32])
    want = (np.float32(0.0078125) * np.float32(da)) * np.float32(int(sc[n // 32]) * code * int(qa[n % 32]))
    assert oracle.gemv(Q5, W, 1, 256, xq, 1)[0, 0] == want


def test_zero_activations_and_independent_columns():
    rows, K, ncols = 7, 768, 6
    W = synth.q5_k_weights(rows, K, salt=3)
    xq0 = oracle.quantize_q8_1(np.zeros((2, K), np.float32))
    y0 = oracle.gemv(Q5, W, rows, K, xq0, 2)
    assert np.all(y0 == 0.0) and not np.signbit(y0).any()
    xq = oracle.quantize_q8_1(synth.activations(K, ncols))
    y = oracle.gemv(Q5, W, rows, K, xq, ncols)
    for c in range(ncols):
        assert np.array_equal(y[c], oracle.gemv(Q5, W, rows, K, np.ascontiguousarray(xq[c:c + 1]), 1)[0])


@pytest.mark.parametrize("rows,K", [(16, 256), (37, 512), (5, 2560)])
def test_planar_round_trip_size_and_product(rows, K):
    W = synth.q5_k_weights(rows, K, salt=rows)
    P = oracle.repack_planar(W, rows, K, Q5)
    assert P.size == -(-rows // 16) * (K // 256) * 2816 == oracle.planar_bytes(rows, K, Q5)
    assert np.array_equal(oracle.unpack_planar(P, rows, K, Q5), W)
    xq = oracle.quantize_q8_1(synth.activations(K, 2, salt=rows))
    assert np.array_equal(oracle.gemv(Q5, W, rows, K, xq, 2), oracle.gemv(Q5P, P, rows, K, xq, 2))
    if rows % 16:
        nb = K // 256
        g = rows // 16
        for b in range(nb):
            t = P[(g * nb + b) * 2816:(g * nb + b + 1) * 2816]
            for i in range(rows % 16, 16):
                assert not t[2048 + 16 * i:2064 + 16 * i].any() and not t[2304 + 32 * i:2336 + 32 * i].any()


def test_planar_marker_bytes_land_per_spec():
    rows, K = 40, 512
    nb = K // 256
    W = np.zeros((rows, nb, 176), np.uint8)
    cases = [(0, 0, 0), (1, 1, 15), (17, 0, 16), (39, 1, 47), (5, 1, 48), (22, 0, 111),
             (31, 1, 112), (8, 0, 175)]
    for k, (r, b, off) in enumerate(cases):
        W[r, b, off] = 1 + k
    P = oracle.repack_planar(W, rows, K, Q5)
    for k, (r, b, off) in enumerate(cases):
        g, i = divmod(r, 16)
        base = (g * nb + b) * 2816
        if off < 16:                                   # header: d, dmin, scales
            pos = base + 2048 + 16 * i + off
        elif off < 48:                                 # qh
            pos = base + 2304 + 32 * i + (off - 16)
        else:                                          # qs[64u + 16j + e]
            u, rem = divmod(off - 48, 64)
            j, e = divmod(rem, 16)
            pos = base + 512 * j + 16 * (16 * u + i) + e
        assert P[pos] == 1 + k, (r, b, off)
    assert np.count_nonzero(P) == len(cases)
