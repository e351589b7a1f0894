"""mmvq_expert_ffn_noalloc: the one-launch expert layer for callers that
cannot allocate device memory (a plugin whose host engine owns every device
buffer, a C caller holding only the pointers it was given, a decode loop
that must keep cudaMalloc and its device synchronisation out of a step).
Its intermediates live in a fixed array inside the library, so the caller
passes only inputs and outputs.

The GPU test calls it through the C ABI twice in a row, on two different
layers, and checks each output against mmvq_expert_ffn (caller-owned
intermediates) on the same inputs, within the bound the other parity tests
use.  The second call finds the first call's intermediates in the array.
This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_matvec_gb300 import build, mmvq, synth
from tests._gpu import assert_within_bound, dev, host

KINDS = {"q4_k_planar": (mmvq.TYPE_Q4_K_PLANAR, mmvq.TYPE_Q4_K, oracle.TYPE_Q4_K),
         "q6_k_planar": (mmvq.TYPE_Q6_K_PLANAR, mmvq.TYPE_Q6_K, oracle.TYPE_Q6_K)}

A = 0x10000  # an aligned fake device address: these calls fail before any CUDA call


def _scratch_need(H, F, T, k):
    up = lambda v: (v + 255) // 256 * 256
    return 256 + up(T * (H // 32) * 36) + up(T * k * (F // 32) * 36) + T * k * 2 * F * 4


def test_sizes_beyond_the_fixed_scratch_are_rejected_on_the_host():
    build.build()
    lib = mmvq.lib()
    args = lambda H, F, T, k, y=A: (mmvq.TYPE_Q4_K_PLANAR, A, A, 256, H, F, A, H, T, A, k, y,
                                    None, None, None, None, None, None)
    # the pages' layer fits: 256 experts, H = 2560, F = 768, 8 tokens, top-8
    assert _scratch_need(2560, 768, 8, 8) <= mmvq.NOALLOC_SCRATCH_BYTES
    # 64 slots of F = 4096 need 2 MiB of gate|up rows alone
    assert _scratch_need(2560, 4096, 8, 8) > mmvq.NOALLOC_SCRATCH_BYTES
    assert lib.mmvq_expert_ffn_noalloc(*args(2560, 4096, 8, 8)) == mmvq.ERR_SCRATCH
    assert "scratch" in mmvq.strerror(mmvq.ERR_SCRATCH)
    # the other rules are mmvq_expert_ffn's
    assert lib.mmvq_expert_ffn_noalloc(*args(2560, 768, 8, 8, y=None)) == mmvq.ERR_NULL
    assert lib.mmvq_expert_ffn_noalloc(*args(2560, 768, 9, 8)) == mmvq.ERR_NCOLS
    assert lib.mmvq_expert_ffn_noalloc(*args(2560, 700, 8, 8)) == mmvq.ERR_SHAPE


def _planar(W, src_type):
    E, rows, nb, _ = W.shape
    return torch.cat([mmvq.repack_planar(dev(W[e]), rows, nb * 256, type_=src_type)
                      for e in range(E)])


def _layer(kind, E, H, F, T, k, salt):
    src = kind.replace("_planar", "")
    _, t_src, _ = KINDS[kind]
    W_gu = synth.expert_weights(src, E, 2 * F, H, salt=salt)
    W_dn = synth.expert_weights(src, E, H, F, salt=salt + 1)
    x = synth.moe_hidden(H, T, salt=salt)
    topk = synth.routing(T, k, E, salt=salt)
    return dict(W_dn=W_dn, Pgu=_planar(W_gu, t_src), Pdn=_planar(W_dn, t_src), x=dev(x),
                topk=dev(topk), E=E, H=H, F=F, T=T, k=k)


@pytest.mark.gpu
@pytest.mark.parametrize("kind", list(KINDS))
def test_two_calls_in_a_row_match_the_allocating_entry_point(kind):
    t_planar, _, o_t = KINDS[kind]
    # two layers shaped like the pages' MoE layer (256 experts, gate|up
    # 1536 x 2560, down 2560 x 768, top-8), eight tokens then one
    layers = [_layer(kind, 256, 2560, 768, T, 8, salt=60 + T) for T in (8, 1)]
    got = []
    for L in layers:                                   # back to back on one stream
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = mmvq.expert_ffn_noalloc(t_planar, L["Pgu"], L["Pdn"], L["E"], L["H"], L["F"],
                                      L["x"], L["topk"], status=status)
        got.append(out)
    torch.cuda.synchronize()
    for L, out in zip(layers, got):
        ref = mmvq.expert_ffn(t_planar, L["Pgu"], L["Pdn"], L["E"], L["H"], L["F"], L["x"],
                              L["topk"], status=torch.zeros(1, dtype=torch.int32, device="cuda"))
        g = {key: host(v) for key, v in out.items()}
        r = {key: host(v) for key, v in ref.items()}
        n = int(r["offsets"][L["E"]])
        assert n == L["T"] * L["k"]
        assert g["status"][0] == 0
        for key in ("expert_ids", "offsets"):
            assert np.array_equal(g[key], r[key])
        for key in ("act_index", "slot_of"):
            assert np.array_equal(g[key][:n], r[key][:n])
        # the bound of the down product on the allocating call's own requantised input
        _, y_bound = oracle.grouped(o_t, L["W_dn"], L["E"], L["H"], L["F"], r["expert_ids"],
                                    r["offsets"], None, r["hq"][:n], with_bound=True)
        assert_within_bound(g["y"][:n], r["y"][:n], y_bound,
                            f"{kind} no-alloc T={L['T']} against mmvq_expert_ffn")
    assert mmvq.read_device_fault() == 0
