"""Parity of the one-launch expert FFN (mmvq_expert_ffn) with the oracle's
chain of steps: token lists, Q8_1 of the hidden states, grouped gate|up,
SiLU(gate)*up -> Q8_1, grouped down (PR #2746 "B70 validation": grouped
calls over per-expert token groups; issue #2801: the gate/up and down
kernels and the activation between them).

The requantised SiLU*up is a Q8_1 code decided by floating point, so the
chain is pinned two ways:
  - an exact chain: integer weights (d = 1, unit scales, no mins) and hidden
    states whose 32-blocks hold one 127 or nothing (Q8_1 d = 1), with every
    gate output >= 127, so that 1 + exp(-gate) rounds to 1 on both sides.
    Every block term is then a small integer: gate|up, h and its Q8_1 bytes
    are exact and must equal the oracle's bit for bit; the down output is
    checked within the bound;
  - synthetic weights and activations shaped like the pages' MoE layer:
    gate|up within the bound; the fused requantisation bit-identical to the
    separate SiLU*up kernel run on the same gate|up rows, and on every block
    equal to the oracle's Q8_1 of that kernel's h; h within a few ulps of the
    oracle's; every down row within the bound of the oracle's product of the
    GPU's requantised input.
"""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_matvec_gb300 import mmvq, synth
from tests._gpu import assert_within_bound, dev, host

pytestmark = pytest.mark.gpu

# planar type, GGUF source type for the repack, oracle type
KINDS = {"q4_k_planar": (mmvq.TYPE_Q4_K_PLANAR, mmvq.TYPE_Q4_K, oracle.TYPE_Q4_K),
         "q6_k_planar": (mmvq.TYPE_Q6_K_PLANAR, mmvq.TYPE_Q6_K, oracle.TYPE_Q6_K)}


def _planar(W, src_type):
    E, rows, nb, _ = W.shape
    return torch.cat([mmvq.repack_planar(dev(W[e]), rows, nb * 256, type_=src_type)
                      for e in range(E)])


def _run(kind, W_gu, W_dn, E, H, F, x, topk, sync=None):
    t_planar, t_src, _ = KINDS[kind]
    T = x.shape[0]
    xq = torch.empty((T, H // 32, 36), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if sync is None:
        sync = mmvq.expert_ffn_workspace("cuda")
    out = mmvq.expert_ffn(t_planar, _planar(W_gu, t_src), _planar(W_dn, t_src), E, H, F, dev(x),
                          dev(topk), xq=xq, status=status, sync=sync)
    res = {k: host(v) for k, v in out.items()}
    res["sync"] = host(sync)
    return res, out


def _oracle_chain(kind, W_gu, W_dn, E, H, F, x, topk):
    o_t = KINDS[kind][2]
    eids, offs, act, slot = oracle.route_groups(topk, E)
    xq = oracle.quantize_q8_1(x)
    gu, gu_b = oracle.grouped(o_t, W_gu, E, 2 * F, H, eids, offs, act, xq, with_bound=True)
    hq, _ = oracle.silu_mul_quantize(gu, F)
    y, y_b = oracle.grouped(o_t, W_dn, E, H, F, eids, offs, None, hq, with_bound=True)
    return dict(expert_ids=eids, offsets=offs, act_index=act, slot_of=slot, xq=xq, gu=gu,
                gu_bound=gu_b, hq=hq, y=y, y_bound=y_b)


def _check_lists(got, ref, n_pos):
    assert np.array_equal(got["expert_ids"], ref["expert_ids"])
    assert np.array_equal(got["offsets"], ref["offsets"])
    assert np.array_equal(got["act_index"][:n_pos], ref["act_index"][:n_pos])
    assert np.array_equal(got["slot_of"][:n_pos], ref["slot_of"][:n_pos])
    assert np.array_equal(got["xq"], ref["xq"])


# ----------------------------------------------------------- exact chain --

def _q4_blocks(q):
    """Q4_K blocks with d = 1, dmin = 0, unit scales, zero mins; q [..., 256] in 0..15."""
    q = q.astype(np.uint8)
    out = np.zeros(q.shape[:-1] + (144,), np.uint8)
    out[..., 0:2] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)
    out[..., 4:8] = 1                      # sc[0..3] = 1 (top bits of sc[4..7] zero)
    out[..., 8:12] = 0                     # m[0..3] = 0
    out[..., 12:16] = 1                    # sc[4..7] low nibble 1, m[4..7] = 0
    for c in range(4):
        out[..., 16 + 32 * c:16 + 32 * c + 32] = (q[..., 64 * c:64 * c + 32] |
                                                  (q[..., 64 * c + 32:64 * c + 64] << 4))
    return out


def _q6_blocks(q):
    """Q6_K blocks with d = 1 and unit scales; q [..., 256] in 0..63 (weight q - 32)."""
    q = q.astype(np.int64)
    out = np.zeros(q.shape[:-1] + (210,), np.uint8)
    for h in range(2):
        for r in range(4):
            lo = q[..., 128 * h + 32 * r:128 * h + 32 * r + 32]
            ql = slice(64 * h + 32 * (r % 2), 64 * h + 32 * (r % 2) + 32)
            out[..., ql] |= ((lo & 15) << (4 * (r // 2))).astype(np.uint8)
            qh = slice(128 + 32 * h, 128 + 32 * h + 32)
            out[..., qh] |= ((lo >> 4) << (2 * r)).astype(np.uint8)
    out[..., 192:208] = 1
    out[..., 208:210] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)
    return out


def _exact_case(kind, E, H, F, T, k, salt):
    rng = np.random.default_rng(9000 + salt)
    nb_h, nb_f = H // 256, F // 256
    if kind == "q4_k_planar":
        gate = rng.integers(1, 16, (E, F, nb_h, 256))            # weights 1..15
        up = rng.integers(0, 16, (E, F, nb_h, 256))              # weights 0..15
        down = rng.integers(0, 16, (E, H, nb_f, 256))
        enc = _q4_blocks
    else:
        gate = rng.integers(33, 48, (E, F, nb_h, 256))           # weights 1..15
        up = rng.integers(16, 48, (E, F, nb_h, 256))             # weights -16..15
        down = rng.integers(0, 64, (E, H, nb_f, 256))
        enc = _q6_blocks
    W_gu = enc(np.concatenate([gate, up], axis=1))
    W_dn = enc(down)
    x = np.zeros((T, H), np.float32)
    for t in range(T):                                           # one 127 per token
        x[t, rng.integers(0, H)] = 127.0
    topk = synth.routing(T, k, E, salt=salt)
    return W_gu, W_dn, x, topk


@pytest.mark.parametrize("kind", list(KINDS))
@pytest.mark.parametrize("T", [1, 2, 3, 5, 8])
def test_exact_chain_matches_the_oracle_bit_for_bit(kind, T):
    E, H, F, k = 16, 2560, 768, 4
    W_gu, W_dn, x, topk = _exact_case(kind, E, H, F, T, k, salt=T)
    ref = _oracle_chain(kind, W_gu, W_dn, E, H, F, x, topk)
    got, _ = _run(kind, W_gu, W_dn, E, H, F, x, topk)
    n = T * k
    _check_lists(got, ref, n)
    assert got["status"][0] == 0
    assert np.all(ref["gu"][:, :F] >= 127.0)                    # 1 + exp(-gate) == 1
    assert np.array_equal(got["gu"].view(np.uint32), ref["gu"].view(np.uint32))
    assert np.array_equal(got["hq"], ref["hq"])
    assert_within_bound(got["y"], ref["y"], ref["y_bound"], f"{kind} down T={T}")
    assert got["sync"][0] & 0x7fffffff == 0                     # barrier word restored


# ------------------------------------------------- synthetic MoE layer --

def _synthetic_case(kind, E, H, F, T, k, salt):
    src = kind.replace("_planar", "")
    W_gu = synth.expert_weights(src, E, 2 * F, H, salt=salt)
    W_dn = synth.expert_weights(src, E, H, F, salt=salt + 1)
    x = synth.moe_hidden(H, T, salt=salt)
    topk = synth.routing(T, k, E, salt=salt)
    return W_gu, W_dn, x, topk


def _check_synthetic(kind, E, H, F, T, k, salt, topk=None):
    W_gu, W_dn, x, rtopk = _synthetic_case(kind, E, H, F, T, k, salt)
    topk = rtopk if topk is None else topk
    ref = _oracle_chain(kind, W_gu, W_dn, E, H, F, x, topk)
    got, out = _run(kind, W_gu, W_dn, E, H, F, x, topk)
    n = int(ref["offsets"][E])
    _check_lists(got, ref, n)
    assert got["status"][0] == 0 and got["sync"][0] & 0x7fffffff == 0
    assert np.isfinite(ref["y"]).all()                  # the chain stays in fp16 range
    assert_within_bound(got["gu"][:n], ref["gu"], ref["gu_bound"], f"{kind} gate|up T={T}")
    # the fused requantisation is the separate kernel's, bit for bit, and
    # that is the oracle's Q8_1 of the separate kernel's h on the GPU's own
    # gate|up rows, on every block; h itself is within a few ulps of the
    # oracle's SiLU*up of those rows
    h_t = torch.empty((n, F), dtype=torch.float32, device="cuda")
    sep = host(mmvq.silu_mul_quantize_q8_1(out["gu"][:n].contiguous(), F, h_out=h_t))
    h_gpu = host(h_t)
    assert np.array_equal(got["hq"][:n], sep)
    assert np.array_equal(got["hq"][:n], oracle.quantize_q8_1(h_gpu))
    _, h_orc = oracle.silu_mul_quantize(got["gu"][:n], F)
    assert np.all(np.abs(h_gpu - h_orc) <= 4e-7 * np.abs(h_orc) + 1e-30)
    # down: every row, against the oracle's grouped product of the GPU's own
    # requantised input
    y_ref, y_bound = oracle.grouped(KINDS[kind][2], W_dn, E, H, F, ref["expert_ids"],
                                    ref["offsets"], None, got["hq"][:n], with_bound=True)
    assert_within_bound(got["y"][:n], y_ref, y_bound, f"{kind} down T={T}")


@pytest.mark.parametrize("kind", list(KINDS))
@pytest.mark.parametrize("T", [1, 4, 8])
def test_moe_layer_shape(kind, T):
    # 256 experts, gate|up 1536 x 2560, down 2560 x 768, top-8 distinct experts
    _check_synthetic(kind, 256, 2560, 768, T, 8, salt=20 + T)


@pytest.mark.parametrize("E,H,F,T,k", [(4, 512, 256, 8, 2), (1, 256, 512, 8, 1),
                                       (7, 768, 1024, 3, 3), (64, 256, 256, 6, 8),
                                       (1024, 256, 256, 8, 8)])
def test_small_and_ragged_layers(E, H, F, T, k):
    # few experts (groups up to 8 positions), F > H, one expert for all
    # tokens, six tokens (the 8-position instance with a partial chunk), and
    # the largest expert count
    _check_synthetic("q4_k_planar", E, H, F, T, k, salt=E + H + F)


def test_groups_longer_than_eight_positions():
    # topk repeats an expert within a token: a group can exceed the 8
    # positions of one pass and is processed in two
    E, H, F, T, k = 3, 256, 256, 8, 3
    topk = np.zeros((T, k), np.int32)
    topk[:, 1] = 2
    assert int(oracle.route_groups(topk, E)[1][1]) == 16           # expert 0: 16 positions
    _check_synthetic("q4_k_planar", E, H, F, T, k, salt=7, topk=topk)


def test_two_tokens_with_a_group_longer_than_a_pass():
    # T = 2 requantises SiLU*up inside the down staging; a token that repeats
    # an expert gives a group of six positions, three passes of two
    E, H, F, T, k = 3, 256, 256, 2, 3
    topk = np.zeros((T, k), np.int32)
    topk[1, 1] = 2
    assert int(oracle.route_groups(topk, E)[1][1]) == 5            # expert 0: 5 positions
    _check_synthetic("q4_k_planar", E, H, F, T, k, salt=13, topk=topk)
    _check_synthetic("q6_k_planar", E, H, F, T, k, salt=14, topk=topk)


def test_bad_expert_ids_are_dropped_and_flagged():
    E, H, F, T, k = 8, 256, 256, 4, 2
    W_gu, W_dn, x, topk = _synthetic_case("q4_k_planar", E, H, F, T, k, salt=11)
    topk = topk.copy()
    topk[1, 0] = E + 3
    topk[2, 1] = -1
    got, _ = _run("q4_k_planar", W_gu, W_dn, E, H, F, x, topk)
    assert got["status"][0] == mmvq.ERR_ROUTING
    valid = (topk >= 0) & (topk < E)
    n = int(got["offsets"][E])
    assert n == int(valid.sum())
    # the lists hold exactly the valid entries, in expert order
    assert sorted(got["slot_of"][:n].tolist()) == sorted(np.flatnonzero(valid.reshape(-1)).tolist())
    assert np.all(np.diff(topk.reshape(-1)[got["slot_of"][:n]]) >= 0)
    assert got["sync"][0] & 0x7fffffff == 0


@pytest.mark.parametrize("kind", list(KINDS))
def test_bitwise_repeatable(kind):
    E, H, F, T, k = 32, 2560, 768, 8, 8
    W_gu, W_dn, x, topk = _synthetic_case(kind, E, H, F, T, k, salt=5)
    sync = mmvq.expert_ffn_workspace("cuda")
    runs = [_run(kind, W_gu, W_dn, E, H, F, x, topk, sync=sync)[0] for _ in range(3)]
    for r in runs[1:]:
        assert np.array_equal(r["gu"].view(np.uint32), runs[0]["gu"].view(np.uint32))
        assert np.array_equal(r["hq"], runs[0]["hq"])
        assert np.array_equal(r["y"].view(np.uint32), runs[0]["y"].view(np.uint32))
    assert runs[-1]["sync"][0] & 0x7fffffff == 0


def test_launch_shape_fills_the_gpu():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for T in (1, 2, 4, 8):
        s = mmvq.expert_ffn_shape(mmvq.TYPE_Q4_K_PLANAR, 256, 2560, 768, T, 8)
        C = s["threads"] // 32 - 1                                # consumer warps
        assert s["threads"] in (13 * 32, 5 * 32)
        assert s["grid"] == sms * (1 if C == 12 else 3)
        assert s["G_gate_up"] * s["P_gate_up"] == C and s["G_down"] * s["P_down"] == C
        assert s["stages"] >= 2


def test_shape_rejects_what_does_not_fit():
    with pytest.raises(mmvq.MMVQError) as e:
        mmvq.expert_ffn_shape(mmvq.TYPE_Q6_K_PLANAR, 256, 16384, 768, 8, 8)
    assert e.value.code == mmvq.ERR_SHAPE


def test_grid_barrier_timeout_is_reported_without_a_fault():
    mmvq.read_device_fault()                                     # clear
    word = mmvq.expert_ffn_workspace("cuda")
    mmvq.selftest_grid_barrier_timeout(word, 2000)
    assert mmvq.read_device_fault() & 2
    # the context stays usable: a full call afterwards is correct
    _check_synthetic("q4_k_planar", 8, 256, 256, 2, 2, salt=3)


@pytest.mark.parametrize("T", [1, 2])
def test_hidden_state_quantisation_at_ties_bit_exact(T):
    # one or two tokens: every CTA quantises the hidden states itself, a block
    # per thread, with a reciprocal-multiply candidate checked against the
    # exact quotient; values whose quotient x/d sits exactly on, or one ulp
    # either side of, a half-integer must give the plain definition's bytes
    E, H, F, k = 8, 512, 256, 2
    rng = np.random.default_rng(31 + T)
    x = np.zeros((T, H), np.float32)
    for t in range(T):
        for b in range(H // 32):
            blk = np.zeros(32, np.float32)
            kind = b % 4
            if kind == 0:                                   # d = 1: exact ties k + 0.5
                blk[:] = np.arange(32) - 15.5
                blk[0] = 127.0
            elif kind == 1:                                 # one ulp either side of the ties
                base = (np.arange(32) - 15.5).astype(np.float32)
                away = np.where(rng.random(32) < 0.5, -200.0, 200.0).astype(np.float32)
                blk[:] = np.nextafter(base, away)
                blk[0] = 127.0
            elif kind == 2:                                 # d not a power of two, ties in x/d
                amax = np.float32(rng.uniform(0.5, 4.0))
                d = np.float32(amax / np.float32(127.0))
                m = rng.integers(-126, 126, 32)
                blk[:] = ((m + 0.5) * d).astype(np.float32)
                blk[0] = amax
            else:                                           # plain random values
                blk[:] = rng.standard_normal(32).astype(np.float32) * np.float32(0.02)
            x[t, 32 * b:32 * b + 32] = blk
    W_gu = synth.expert_weights("q4_k", E, 2 * F, H, salt=T)
    W_dn = synth.expert_weights("q4_k", E, H, F, salt=T + 1)
    topk = synth.routing(T, k, E, salt=T)
    got, _ = _run("q4_k_planar", W_gu, W_dn, E, H, F, x, topk)
    assert np.array_equal(got["xq"], oracle.quantize_q8_1(x))
    ref = _oracle_chain("q4_k_planar", W_gu, W_dn, E, H, F, x, topk)
    n = T * k
    assert_within_bound(got["gu"][:n], ref["gu"], ref["gu_bound"], f"gate|up T={T}")
