"""Pins for the oracle's planar Q6_K tiles, draft-row gather, expert grouping
and SiLU(gate)*up requantisation.

* Planar ("Strata" PR #2340 "STRATA_Q6_PLANAR": the same bytes as ql / qh /
  scales / d planes; the draft head's subset is gathered from the planar
  head): round trip, marker bytes placed where the library's tile
  specification (include/mmvq.h) says, padding rows zero, products unchanged.
* Grouping (PR #2746 "B70 validation": per-expert token groups, empty groups
  allowed): every routing slot appears exactly once, offsets are monotone,
  positions inside a group follow token order, and each grouped output row
  equals the dense product of that expert with that token's column.
* SiLU*up: against scipy's logistic function in fp64 (a library routine),
  closed forms at 0, then bit-exact Q8_1 of the oracle's own h.
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle
from block_quantized_matvec_gb300 import synth


@pytest.mark.parametrize("rows,K", [(16, 256), (37, 512), (5, 2560), (48, 768)])
def test_planar_round_trip_and_size(rows, K):
    W = synth.q6_k_weights(rows, K, salt=rows)
    P = oracle.repack_planar(W, rows, K)
    groups = -(-rows // 16)
    assert P.size == groups * (K // 256) * 3360 == oracle.planar_bytes(rows, K)
    assert np.array_equal(oracle.unpack_planar(P, rows, K), W)
    if rows % 16:
        # the pad rows of the last group hold zero bytes
        nb = K // 256
        for b in range(nb):
            tile = P[((groups - 1) * nb + b) * 3360:((groups - 1) * nb + b + 1) * 3360]
            for i in range(rows % 16, 16):
                for h in range(2):
                    L = 16 * h + i
                    for j in range(4):
                        assert not tile[512 * j + 16 * L:512 * j + 16 * L + 16].any()
                assert not tile[3328 + 2 * i:3330 + 2 * i].any()


def test_planar_marker_bytes_land_per_spec():
    rows, K = 40, 768
    nb = K // 256
    W = np.zeros((rows, nb, 210), np.uint8)
    cases = [(0, 0, 0), (1, 0, 63), (17, 2, 64), (39, 1, 127), (5, 1, 128), (22, 2, 191),
             (9, 0, 192), (33, 2, 207), (15, 1, 208), (31, 0, 209)]
    for k, (r, b, off) in enumerate(cases):
        W[r, b, off] = 1 + k
    P = oracle.repack_planar(W, rows, K)
    for k, (r, b, off) in enumerate(cases):
        g, i = divmod(r, 16)
        base = (g * nb + b) * 3360
        if off < 128:                       # ql[64h + 16j + e]
            h, rem = divmod(off, 64)
            j, e = divmod(rem, 16)
            pos = base + 512 * j + 16 * (16 * h + i) + e
        elif off < 192:                     # qh[32h + 16j + e]
            h, rem = divmod(off - 128, 32)
            j, e = divmod(rem, 16)
            pos = base + 2048 + 512 * j + 16 * (16 * h + i) + e
        elif off < 208:                     # scales[8h + e]
            h, e = divmod(off - 192, 8)
            pos = base + 3072 + 8 * (16 * h + i) + e
        else:                               # d
            pos = base + 3328 + 2 * i + (off - 208)
        assert P[pos] == 1 + k, (r, b, off)
    assert np.count_nonzero(P) == len(cases)


def test_planar_product_equals_gguf_product():
    rows, K, ncols = 45, 1024, 3
    W = synth.q6_k_weights(rows, K, salt=9)
    P = oracle.repack_planar(W, rows, K)
    xq = oracle.quantize_q8_1(synth.activations(K, ncols, salt=9))
    a = oracle.gemv(oracle.TYPE_Q6_K, W, rows, K, xq, ncols)
    b = oracle.gemv(oracle.TYPE_Q6_K_PLANAR, P, rows, K, xq, ncols)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("rows,K", [(16, 256), (37, 512), (5, 2560)])
def test_planar_q4_round_trip_size_and_product(rows, K):
    W = synth.q4_k_weights(rows, K, salt=rows)
    P = oracle.repack_planar(W, rows, K, oracle.TYPE_Q4_K)
    assert P.size == -(-rows // 16) * (K // 256) * 2304 == oracle.planar_bytes(rows, K, oracle.TYPE_Q4_K)
    assert np.array_equal(oracle.unpack_planar(P, rows, K, oracle.TYPE_Q4_K), W)
    xq = oracle.quantize_q8_1(synth.activations(K, 2, salt=rows))
    assert np.array_equal(oracle.gemv(oracle.TYPE_Q4_K, W, rows, K, xq, 2),
                          oracle.gemv(oracle.TYPE_Q4_K_PLANAR, P, rows, K, xq, 2))


def test_planar_q4_marker_bytes_land_per_spec():
    rows, K = 40, 512
    nb = K // 256
    W = np.zeros((rows, nb, 144), np.uint8)
    cases = [(0, 0, 0), (1, 1, 15), (17, 0, 16), (39, 1, 79), (5, 1, 80), (22, 0, 143), (31, 1, 3)]
    for k, (r, b, off) in enumerate(cases):
        W[r, b, off] = 1 + k
    P = oracle.repack_planar(W, rows, K, oracle.TYPE_Q4_K)
    for k, (r, b, off) in enumerate(cases):
        g, i = divmod(r, 16)
        base = (g * nb + b) * 2304
        if off < 16:                                   # header
            pos = base + 2048 + 16 * i + off
        else:                                          # qs[64u + 16j + e]
            u, rem = divmod(off - 16, 64)
            j, e = divmod(rem, 16)
            pos = base + 512 * j + 16 * (16 * u + i) + e
        assert P[pos] == 1 + k, (r, b, off)
    assert np.count_nonzero(P) == len(cases)


def test_gather_planar_rows_picks_the_named_rows():
    rows, K = 300, 512
    W = synth.q6_k_weights(rows, K, salt=4)
    P = oracle.repack_planar(W, rows, K)
    ids = synth.draft_rows(37, rows)
    G = oracle.gather_planar_rows(P, rows, K, ids)
    assert np.array_equal(oracle.unpack_planar(G, ids.size, K), W[ids])
    xq = oracle.quantize_q8_1(synth.activations(K, 2, salt=4))
    full = oracle.gemv(oracle.TYPE_Q6_K_PLANAR, P, rows, K, xq, 2)
    sub = oracle.gemv(oracle.TYPE_Q6_K_PLANAR, G, ids.size, K, xq, 2)
    assert np.array_equal(sub, full[:, ids])


@pytest.mark.parametrize("T", [1, 4, 8])
def test_route_groups_invariants(T):
    E, k = 256, 8
    topk = synth.routing(T, k, E, salt=T)
    eids, offs, act, slot = oracle.route_groups(topk, E)
    assert np.array_equal(eids, np.arange(E))
    assert offs[0] == 0 and offs[-1] == T * k and np.all(np.diff(offs) >= 0)
    assert np.array_equal(np.sort(slot), np.arange(T * k))          # each slot once
    for e in range(E):
        p0, p1 = offs[e], offs[e + 1]
        toks = act[p0:p1]
        assert np.all(np.diff(toks) > 0)                             # token order
        assert set(toks.tolist()) == {t for t in range(T) if e in topk[t]}
        for p in range(p0, p1):
            assert topk[slot[p] // k, slot[p] % k] == e and slot[p] // k == act[p]
    assert (np.diff(offs) == 0).sum() >= E - T * k                   # empty groups exist


def test_grouped_rows_equal_dense_products_per_expert():
    E, rows, K, T = 6, 20, 512, 5
    W = synth.expert_weights("q4_k", E, rows, K, salt=2)
    topk = synth.routing(T, 2, E, salt=2)
    eids, offs, act, _ = oracle.route_groups(topk, E)
    xq = oracle.quantize_q8_1(synth.activations(K, T, salt=2))
    y = oracle.grouped(oracle.TYPE_Q4_K, W, E, rows, K, eids, offs, act, xq)
    for e in range(E):
        for p in range(offs[e], offs[e + 1]):
            col = np.ascontiguousarray(xq[act[p]:act[p] + 1])
            assert np.array_equal(y[p], oracle.gemv(oracle.TYPE_Q4_K, W[e], rows, K, col, 1)[0])


def test_silu_mul_quantize_against_logistic_and_closed_forms():
    F, n = 768, 9
    gu = synth.gate_up(n, F)
    gu[0, :F] = 0.0                                  # silu(0) = 0 -> h = 0
    xq, h = oracle.silu_mul_quantize(gu, F)
    g = gu[:, :F].astype(np.float64)
    u = gu[:, F:].astype(np.float64)
    ref = g * expit(g) * u
    assert np.all(np.abs(h - ref) <= 4e-7 * np.abs(ref) + 1e-30)
    assert not h[0].any() and not xq[0].any()
    assert np.array_equal(xq, oracle.quantize_q8_1(h))
