"""The debug build (libmmvq_checked.so: the library compiled with
MMVQ_CHECKED, whose ring kernels test every shared-memory layout, bulk-copy
source range, ring tile and staged K-block against its bounds, set bit 4 of
the device fault word on a failure and skip the access).

On ragged and full-size shapes of every ring kernel (dense planar, with and
without the cluster K-split and the tensor-core consumer, the LM head's
persistent grid, grouped experts, the one-launch expert layer at one and
eight tokens) no check fails and the outputs have the product library's
bits: the checks change no arithmetic.  The checked library is built on
first use (a minute or two); the product library is untouched.
"""
import contextlib
import ctypes

import numpy as np
import pytest
import torch

from block_quantized_matvec_gb300 import build, mmvq, synth
from tests._gpu import dev, host

pytestmark = pytest.mark.gpu

KINDS = {"q4_k_planar": (mmvq.TYPE_Q4_K_PLANAR, mmvq.TYPE_Q4_K, synth.q4_k_weights),
         "q5_k_planar": (mmvq.TYPE_Q5_K_PLANAR, mmvq.TYPE_Q5_K, synth.q5_k_weights),
         "q6_k_planar": (mmvq.TYPE_Q6_K_PLANAR, mmvq.TYPE_Q6_K, synth.q6_k_weights)}


@pytest.fixture(scope="module")
def checked():
    path = build.build(checked=True)
    lib = ctypes.CDLL(path)
    for name, (res, args) in mmvq.SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


@contextlib.contextmanager
def _using(lib):
    """The binding's calls go to `lib` inside the block."""
    mmvq.lib()  # the product library is loaded first
    saved = mmvq._lib
    mmvq._lib = lib
    try:
        yield
    finally:
        mmvq._lib = saved


def _fault(lib):
    with _using(lib):
        return mmvq.read_device_fault()


def _same_bits(a, b):
    return np.array_equal(host(a).view(np.uint32), host(b).view(np.uint32))


@pytest.mark.parametrize("kind", list(KINDS))
def test_dense_shapes_pass_every_check_with_the_products_bits(checked, kind):
    t, src, gen = KINDS[kind]
    assert _fault(checked) == 0
    for rows, K in [(1, 256), (37, 2560), (300, 512), (2560, 10240), (17, 16384)]:
        W = gen(rows, K, salt=rows + K)
        P = mmvq.repack_planar(dev(W), rows, K, type_=src)
        for ncols in (1, 3, 8):
            xq = mmvq.quantize_q8_1(dev(synth.activations(K, ncols, salt=ncols)))
            for flags in ((0, mmvq.FLAG_TENSOR_CORE) if ncols == 8 else (0,)):
                y = mmvq.gemv(t, P, rows, K, xq, ncols, flags=flags)
                with _using(checked):
                    yc = mmvq.gemv(t, P, rows, K, xq, ncols, flags=flags)
                assert _same_bits(y, yc), (kind, rows, K, ncols, flags)
    assert _fault(checked) == 0


def test_lm_head_persistent_grid(checked):
    rows, K = 151936, 2560
    t = mmvq.TYPE_Q6_K_PLANAR
    P = mmvq.repack_planar(dev(synth.q6_k_weights(rows, K, salt=2)), rows, K)
    for ncols in (1, 5):
        xq = mmvq.quantize_q8_1(dev(synth.activations(K, ncols, salt=2)))
        y = mmvq.gemv(t, P, rows, K, xq, ncols)
        with _using(checked):
            yc = mmvq.gemv(t, P, rows, K, xq, ncols)
        assert _same_bits(y, yc)
    assert _fault(checked) == 0


def _planar_experts(kind, E, rows, K, salt):
    _, src, _ = KINDS[kind]
    W = synth.expert_weights(kind.replace("_planar", ""), E, rows, K, salt=salt)
    return torch.cat([mmvq.repack_planar(dev(W[e]), rows, K, type_=src) for e in range(E)])


@pytest.mark.parametrize("kind", ["q4_k_planar", "q6_k_planar"])
def test_grouped_and_expert_layer(checked, kind):
    t = KINDS[kind][0]
    E, H, F, k = 64, 2560, 768, 8
    Pgu = _planar_experts(kind, E, 2 * F, H, 40)
    Pdn = _planar_experts(kind, E, H, F, 41)
    for T in (1, 8):
        x = dev(synth.moe_hidden(H, T, salt=T))
        topk = dev(synth.routing(T, k, E, salt=T))
        out = mmvq.expert_ffn(t, Pgu, Pdn, E, H, F, x, topk,
                              status=torch.zeros(1, dtype=torch.int32, device="cuda"))
        with _using(checked):
            outc = mmvq.expert_ffn(t, Pgu, Pdn, E, H, F, x, topk,
                                   status=torch.zeros(1, dtype=torch.int32, device="cuda"))
        n = T * k
        assert _same_bits(out["y"][:n], outc["y"][:n])
        assert np.array_equal(host(out["hq"][:n]), host(outc["hq"][:n]))
        # the grouped gate|up call over the same lists, product and checked
        xq = out["xq"]
        ids, offs, act = out["expert_ids"], out["offsets"], out["act_index"]
        g = mmvq.grouped(t, Pgu, E, 2 * F, H, ids, offs, act, xq, T, n)
        with _using(checked):
            gc = mmvq.grouped(t, Pgu, E, 2 * F, H, ids, offs, act, xq, T, n)
        assert _same_bits(g[:n], gc[:n])
    assert _fault(checked) == 0
