"""Planar repack, draft-row gather, expert grouping and the grouped expert
products on the GPU against the oracle.

Repack and gather are byte permutations ("Strata" PR #2340
"STRATA_Q6_PLANAR"), grouping is integer work: all bit for bit.  Grouped
products (PR #2746 "B70 validation": grouped calls with empty groups) are
checked like the dense ones: FP32 within the bound, per position."""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_matvec_gb300 import mmvq, synth
from tests._gpu import assert_within_bound, dev, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,K", [(1, 256), (16, 256), (37, 512), (300, 2560), (45, 10240)])
def test_repack_bit_exact(rows, K):
    W = synth.q6_k_weights(rows, K, salt=rows)
    assert np.array_equal(host(mmvq.repack_planar(dev(W), rows, K)),
                          oracle.repack_planar(W, rows, K))


@pytest.mark.parametrize("rows,K", [(1, 256), (16, 256), (37, 512), (300, 2560), (45, 10240)])
def test_repack_q4_bit_exact(rows, K):
    W = synth.q4_k_weights(rows, K, salt=rows)
    got = host(mmvq.repack_planar(dev(W), rows, K, type_=mmvq.TYPE_Q4_K))
    assert np.array_equal(got, oracle.repack_planar(W, rows, K, oracle.TYPE_Q4_K))


@pytest.mark.parametrize("rows,K", [(1, 256), (16, 256), (37, 512), (300, 2560), (45, 10240)])
def test_repack_q5_bit_exact(rows, K):
    W = synth.q5_k_weights(rows, K, salt=rows + K)
    got = host(mmvq.repack_planar(dev(W), rows, K, type_=mmvq.TYPE_Q5_K))
    assert np.array_equal(got, oracle.repack_planar(W, rows, K, oracle.TYPE_Q5_K))


@pytest.mark.parametrize("rows,K,n", [(300, 512, 37), (1000, 2560, 64), (40, 256, 1)])
def test_gather_bit_exact(rows, K, n):
    W = synth.q6_k_weights(rows, K, salt=n)
    P = oracle.repack_planar(W, rows, K)
    ids = synth.draft_rows(n, rows, salt=n)
    out, status = mmvq.gather_planar_rows(dev(P), rows, K, dev(ids))
    assert np.array_equal(host(out), oracle.gather_planar_rows(P, rows, K, ids))
    assert host(status)[0] == 0


def test_gather_flags_bad_row_ids_and_writes_zero_rows():
    rows, K = 64, 256
    W = synth.q6_k_weights(rows, K, salt=2)
    P = oracle.repack_planar(W, rows, K)
    ids = np.array([3, rows, -1, 7], np.int32)
    out, status = mmvq.gather_planar_rows(dev(P), rows, K, dev(ids))
    assert host(status)[0] == mmvq.ERR_ROUTING
    g = oracle.unpack_planar(host(out), 4, K)
    assert np.array_equal(g[0], W[3]) and np.array_equal(g[3], W[7])
    assert not g[1].any() and not g[2].any()


@pytest.mark.parametrize("T,k,E", [(1, 8, 256), (4, 8, 256), (8, 8, 256), (0, 8, 256),
                                   (300, 6, 64), (20, 2, 4)])
def test_route_groups_bit_exact(T, k, E):
    topk = synth.routing(T, k, E, salt=T) if T else np.zeros((0, k), np.int32)
    eids, offs, act, slot = oracle.route_groups(topk, E) if T else (
        np.arange(E, dtype=np.int32), np.zeros(E + 1, np.int32), None, None)
    td = dev(topk) if T else torch.zeros((0, k), dtype=torch.int32, device="cuda")
    g_eids, g_offs, g_act, g_slot, status = mmvq.route_groups(td, E)
    assert np.array_equal(host(g_eids), eids) and np.array_equal(host(g_offs), offs)
    if T:
        assert np.array_equal(host(g_act), act) and np.array_equal(host(g_slot), slot)
    assert host(status)[0] == 0


def _experts_on_device(kind, W):
    """GGUF experts as they are, planar kinds repacked one expert at a time."""
    if not kind.endswith("_planar"):
        return dev(W)
    E, rows, nb, _ = W.shape
    t = mmvq.TYPE_Q4_K if kind.startswith("q4") else mmvq.TYPE_Q6_K
    return torch.cat([mmvq.repack_planar(dev(W[e]), rows, nb * 256, type_=t) for e in range(E)])


def _grouped_case(kind, T, k, E, rows, K, salt):
    t = {"q4_k": (mmvq.TYPE_Q4_K, oracle.TYPE_Q4_K), "q6_k": (mmvq.TYPE_Q6_K, oracle.TYPE_Q6_K),
         "q4_k_planar": (mmvq.TYPE_Q4_K_PLANAR, oracle.TYPE_Q4_K),
         "q6_k_planar": (mmvq.TYPE_Q6_K_PLANAR, oracle.TYPE_Q6_K)}[kind]
    W = synth.expert_weights(kind.replace("_planar", ""), E, rows, K, salt=salt)
    topk = synth.routing(T, k, E, salt=salt)
    eids, offs, act, _ = oracle.route_groups(topk, E)
    x = synth.activations(K, T, salt=salt)
    xq = oracle.quantize_q8_1(x)
    y_ref, bound = oracle.grouped(t[1], W, E, rows, K, eids, offs, act, xq, with_bound=True)
    Wd = _experts_on_device(kind, W)
    xqd = mmvq.quantize_q8_1(dev(x))
    g_eids, g_offs, g_act, _, _ = mmvq.route_groups(dev(topk), E)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = mmvq.grouped(t[0], Wd, E, rows, K, g_eids, g_offs, g_act, xqd, T, T * k, status=status)
    return host(y), y_ref, bound, host(status)[0]


@pytest.mark.parametrize("kind", ["q4_k", "q4_k_planar", "q6_k_planar"])
@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_grouped_gate_up_shape(kind, T):
    # 256 experts, gate|up 1536 x 2560, top-8 distinct experts per token
    y, y_ref, bound, st = _grouped_case(kind, T, 8, 256, 1536, 2560, salt=T)
    assert st == 0
    assert_within_bound(y, y_ref, bound, f"GU T={T}")


@pytest.mark.parametrize("planar", [False, True])
@pytest.mark.parametrize("T", [1, 8])
def test_grouped_down_shape(T, planar):
    # down 2560 x 768, activations are the requantised SiLU*up columns, one per position
    E, rows, K, k = 256, 2560, 768, 8
    W = synth.expert_weights("q4_k", E, rows, K, salt=10 + T)
    topk = synth.routing(T, k, E, salt=10 + T)
    eids, offs, _, _ = oracle.route_groups(topk, E)
    h = synth.activations(K, T * k, salt=10 + T)
    xq = oracle.quantize_q8_1(h)
    y_ref, bound = oracle.grouped(oracle.TYPE_Q4_K, W, E, rows, K, eids, offs, None, xq,
                                  with_bound=True)
    g_eids, g_offs, _, _, _ = mmvq.route_groups(dev(topk), E)
    Wd, t = dev(W), mmvq.TYPE_Q4_K
    if planar:
        Wd = torch.cat([mmvq.repack_planar(dev(W[e]), rows, K, type_=mmvq.TYPE_Q4_K) for e in range(E)])
        t = mmvq.TYPE_Q4_K_PLANAR
    y = mmvq.grouped(t, Wd, E, rows, K, g_eids, g_offs, None, mmvq.quantize_q8_1(dev(h)), T * k, T * k)
    assert_within_bound(host(y), y_ref, bound, f"down T={T}")


@pytest.mark.parametrize("kind,rows", [("q4_k", 37), ("q6_k", 37), ("q4_k_planar", 48),
                                       ("q6_k_planar", 48)])
def test_grouped_groups_larger_than_eight_and_ragged_rows(kind, rows):
    # 4 experts, 20 tokens, top-2: groups of about 10 positions (processed 8 at a time)
    y, y_ref, bound, st = _grouped_case(kind, 20, 2, 4, rows, 512, salt=3)
    assert st == 0
    assert_within_bound(y, y_ref, bound, kind)


_KIND_TYPE = {"q4_k": mmvq.TYPE_Q4_K, "q4_k_planar": mmvq.TYPE_Q4_K_PLANAR,
              "q6_k_planar": mmvq.TYPE_Q6_K_PLANAR}


@pytest.mark.parametrize("kind", ["q4_k_planar", "q6_k_planar"])
def test_grouped_longest_rows_with_full_position_chunks(kind):
    # K = 16384 with groups of about 10 positions (chunks of 8): the launch
    # shape must still fit its ring beside eight staged activation columns
    y, y_ref, bound, st = _grouped_case(kind, 20, 2, 4, 48, 16384, salt=6)
    assert st == 0
    assert_within_bound(y, y_ref, bound, f"{kind} K=16384")


@pytest.mark.parametrize("kind", ["q4_k", "q4_k_planar", "q6_k_planar"])
def test_grouped_all_groups_empty_writes_nothing(kind):
    E, rows, K = 8, 32, 256
    W = _experts_on_device(kind, synth.expert_weights(kind[:4], E, rows, K))
    xqd = mmvq.quantize_q8_1(dev(synth.activations(K, 1)))
    eids = torch.arange(E, dtype=torch.int32, device="cuda")
    offs = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    out = torch.full((4, rows), 7.0, device="cuda")
    mmvq.grouped(_KIND_TYPE[kind], W, E, rows, K, eids, offs, None, xqd, 1, 4, out=out)
    assert np.all(host(out) == 7.0)


@pytest.mark.parametrize("kind", ["q4_k", "q4_k_planar", "q6_k_planar"])
def test_grouped_flags_bad_routing_without_faulting(kind):
    E, rows, K = 4, 32, 256
    W = _experts_on_device(kind, synth.expert_weights(kind[:4], E, rows, K))
    xqd = mmvq.quantize_q8_1(dev(synth.activations(K, 3)))
    eids = dev(np.array([0, 9, 2], np.int32))           # expert 9 does not exist
    offs = dev(np.array([0, 1, 2, 3], np.int32))
    act = dev(np.array([0, 1, 5], np.int32))            # column 5 does not exist
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((3, rows), 7.0, device="cuda")
    mmvq.grouped(_KIND_TYPE[kind], W, E, rows, K, eids, offs, act, xqd, 3, 3, out=out,
                 status=status)
    o = host(out)
    assert host(status)[0] == mmvq.ERR_ROUTING
    assert np.all(o[1] == 7.0)                           # skipped group
    assert np.all(o[2] == 0.0)                           # zero activation column
    assert np.any(o[0] != 7.0)


@pytest.mark.parametrize("kind", ["q4_k_planar", "q6_k_planar"])
def test_grouped_planar_is_bitwise_repeatable(kind):
    # fixed reduction order: the same call gives the same bits every time
    E, rows, K, T, k = 32, 512, 2560, 8, 8
    W = _experts_on_device(kind, synth.expert_weights(kind[:4], E, rows, K, salt=5))
    topk = synth.routing(T, k, E, salt=5)
    xqd = mmvq.quantize_q8_1(dev(synth.activations(K, T, salt=5)))
    g_eids, g_offs, g_act, _, _ = mmvq.route_groups(dev(topk), E)
    outs = [host(mmvq.grouped(_KIND_TYPE[kind], W, E, rows, K, g_eids, g_offs, g_act, xqd, T,
                              T * k)) for _ in range(3)]
    assert all(np.array_equal(outs[0].view(np.uint32), o.view(np.uint32)) for o in outs[1:])


@pytest.mark.parametrize("T,k,E,K", [(1, 8, 256, 2560), (8, 8, 256, 2560), (3, 2, 1024, 768),
                                     (4, 8, 2048, 256), (5, 3, 7, 512)])
def test_quantize_route_in_one_launch_matches_the_two_calls(T, k, E, K):
    topk = dev(synth.routing(T, k, E, salt=E + T))
    x = dev(synth.activations(K, T, salt=E + T))
    xq, eids, offs, act, slot, status = mmvq.quantize_route_groups(x, topk, E)
    r_eids, r_offs, r_act, r_slot, r_status = mmvq.route_groups(topk, E)
    assert np.array_equal(host(xq), host(mmvq.quantize_q8_1(x)))
    assert np.array_equal(host(xq), oracle.quantize_q8_1(host(x)))
    for a, b in ((eids, r_eids), (offs, r_offs), (act, r_act), (slot, r_slot), (status, r_status)):
        assert np.array_equal(host(a), host(b))
