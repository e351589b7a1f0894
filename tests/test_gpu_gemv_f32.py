"""mmvq_gemv_f32: fp32 activation columns quantised inside the product.

The result must be exactly that of the two calls it replaces: xq the Q8_1
bytes of the plain definition (checked against the oracle), y the same bits
as mmvq_gemv on those bytes, and y within the bound of the oracle's product
("Strata" PR #2340 "int4 activation loads": the wide kernels read Q8_1
columns; PR #2207: weights read once for 1-8 columns).  The cases cover both
the one-launch path and the two-launch one, ragged rows, ldx > K, x that is
only 4-byte aligned, and values whose quotient x/d sits on a half-integer.
"""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_matvec_gb300 import mmvq, synth
from tests._gpu import assert_within_bound, dev, host

pytestmark = pytest.mark.gpu

KINDS = {"q6_k_planar": (mmvq.TYPE_Q6_K_PLANAR, mmvq.TYPE_Q6_K, oracle.TYPE_Q6_K, synth.q6_k_weights),
         "q4_k_planar": (mmvq.TYPE_Q4_K_PLANAR, mmvq.TYPE_Q4_K, oracle.TYPE_Q4_K, synth.q4_k_weights),
         "q5_k_planar": (mmvq.TYPE_Q5_K_PLANAR, mmvq.TYPE_Q5_K, oracle.TYPE_Q5_K, synth.q5_k_weights)}


def _weights(kind, rows, K, salt):
    t_gpu, t_src, t_orc, gen = KINDS[kind]
    W = gen(rows, K, salt=salt)
    return W, mmvq.repack_planar(dev(W), rows, K, type_=t_src), t_gpu, t_orc


def _tie_columns(K, ncols, salt):
    """Columns whose 32-blocks mix exact half-integer quotients, values one ulp
    off them, and plain normal values."""
    rng = np.random.default_rng(salt)
    x = synth.activations(K, ncols, salt=salt).copy()
    for c in range(ncols):
        for b in range(0, K // 32, 3):
            blk = (np.arange(32) - 15.5).astype(np.float32)
            if b % 2:
                away = np.where(rng.random(32) < 0.5, -200.0, 200.0).astype(np.float32)
                blk = np.nextafter(blk, away)
            blk[0] = 127.0
            x[c, 32 * b:32 * b + 32] = blk * np.float32(2.0) ** int(rng.integers(-4, 4))
    return x


def _check(kind, rows, K, ncols, x, flags=0, salt=1):
    W, Wd, t_gpu, t_orc = _weights(kind, rows, K, salt)
    xd = dev(x)
    y, xq = mmvq.gemv_f32(t_gpu, Wd, rows, K, xd[:, :K] if x.shape[1] > K else xd, ncols,
                          flags=flags)
    xq_ref = oracle.quantize_q8_1(x, K=K)
    assert np.array_equal(host(xq), xq_ref)
    y_two = mmvq.gemv(t_gpu, Wd, rows, K, mmvq.quantize_q8_1(xd, K=K), ncols)
    assert np.array_equal(host(y).view(np.uint32), host(y_two).view(np.uint32))
    y_ref, bound = oracle.gemv(t_orc, W, rows, K, xq_ref, ncols, with_bound=True)
    assert_within_bound(host(y), y_ref, bound, f"{kind} {rows}x{K} ncols={ncols}")


@pytest.mark.parametrize("kind", list(KINDS))
@pytest.mark.parametrize("rows,K,ncols", [(2560, 2560, 1), (37, 2560, 2), (300, 512, 8),
                                          (10240, 2560, 1), (2560, 10240, 1), (2560, 10240, 4),
                                          (2560, 10240, 8), (17, 256, 3)])
def test_matches_the_two_calls_it_replaces(kind, rows, K, ncols):
    x = _tie_columns(K, ncols, salt=rows + K + ncols)
    _check(kind, rows, K, ncols, x, salt=rows + ncols)


def test_both_paths_are_exercised():
    t = mmvq.TYPE_Q6_K_PLANAR
    assert mmvq.gemv_f32_fused(t, 2560, 2560, 1)                   # one launch
    assert mmvq.gemv_f32_fused(t, 10240, 2560, 1)
    assert not mmvq.gemv_f32_fused(t, 151936, 2560, 1)             # quantiser + product
    assert not mmvq.gemv_f32_fused(t, 2560, 10240, 8)


def test_ldx_and_unaligned_columns():
    rows, K, ncols = 200, 2560, 3
    big = _tie_columns(K + 64, ncols, salt=5)
    # ldx = K + 64 through a strided view
    W, Wd, t_gpu, t_orc = _weights("q6_k_planar", rows, K, 5)
    xd = dev(big)
    y, xq = mmvq.gemv_f32(t_gpu, Wd, rows, K, xd, ncols)
    assert np.array_equal(host(xq), oracle.quantize_q8_1(big, K=K))
    # x starting one float into an allocation: 4-byte aligned only (scalar loads)
    flat = torch.zeros(ncols * (K + 1) + 1, dtype=torch.float32, device="cuda")
    xu = flat[1:1 + ncols * (K + 1)].view(ncols, K + 1)
    xu.copy_(xd[:, :K + 1])
    assert xu.data_ptr() % 16 != 0
    y2, xq2 = mmvq.gemv_f32(t_gpu, Wd, rows, K, xu, ncols)
    assert np.array_equal(host(xq2), oracle.quantize_q8_1(big[:, :K + 1], K=K))
    assert np.array_equal(host(y).view(np.uint32), host(y2).view(np.uint32))


def test_stable_flag_gives_the_same_bits():
    rows, K, ncols = 2560, 2560, 2
    x = _tie_columns(K, ncols, salt=9)
    W, Wd, t_gpu, _ = _weights("q4_k_planar", rows, K, 9)
    xd = dev(x)
    y0, q0 = mmvq.gemv_f32(t_gpu, Wd, rows, K, xd, ncols)
    y1, q1 = mmvq.gemv_f32(t_gpu, Wd, rows, K, xd, ncols, flags=mmvq.FLAG_XQ_STABLE)
    assert np.array_equal(host(q0), host(q1))
    assert np.array_equal(host(y0).view(np.uint32), host(y1).view(np.uint32))


def test_zero_blocks():
    rows, K, ncols = 64, 512, 2
    x = synth.activations(K, ncols, salt=3).copy()
    x[0, :32] = 0.0                                 # amax = 0: d = 0, q = 0
    x[1, 64:96] = 0.0
    x[1, 96:128] *= np.float32(1e-30)               # d = amax/127 rounds to 0 in fp16
    W, Wd, t_gpu, _ = _weights("q6_k_planar", rows, K, 3)
    y, xq = mmvq.gemv_f32(t_gpu, Wd, rows, K, dev(x), ncols)
    assert np.array_equal(host(xq), oracle.quantize_q8_1(x))
