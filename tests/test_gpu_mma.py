"""The tensor-core consumer of the planar kernel (MMVQ_FLAG_TENSOR_CORE,
4-8 columns: warp-level f16 MMAs, one per 16-weight sub-block) against the
oracle and the default dp4a consumer.

Its per-32-block integer sums equal the oracle's, and y has the same bits
as the dp4a consumer's in the same launch shape: the weights enter the MMA
as exact f16 integers 1024 + code, the activations as exact f16 integers,
and every partial sum is an integer below 2^24.  The extreme cases put
codes, scales and activations at the ends of their ranges, where the sums
come closest to that limit ("Strata" PR #1774 "d * ds * sumi": the integer
sums per sub-block and the fp32 scale chain; PR #2207: 1-8 columns).
"""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_matvec_gb300 import mmvq, synth
from tests._gpu import assert_within_bound, dev, host

pytestmark = pytest.mark.gpu

TC = mmvq.FLAG_TENSOR_CORE
KINDS = {
    "q6_k_planar": (mmvq.TYPE_Q6_K_PLANAR, mmvq.TYPE_Q6_K, oracle.TYPE_Q6_K, synth.q6_k_weights),
    "q4_k_planar": (mmvq.TYPE_Q4_K_PLANAR, mmvq.TYPE_Q4_K, oracle.TYPE_Q4_K, synth.q4_k_weights),
    "q5_k_planar": (mmvq.TYPE_Q5_K_PLANAR, mmvq.TYPE_Q5_K, oracle.TYPE_Q5_K, synth.q5_k_weights),
}


def _planar(kind, W, rows, K):
    return mmvq.repack_planar(dev(W), rows, K, type_=KINDS[kind][1])


def _same_bits(a, b):
    return np.array_equal(host(a).view(np.uint32), host(b).view(np.uint32))


@pytest.mark.parametrize("kind", list(KINDS))
@pytest.mark.parametrize("rows,K", [(1, 256), (37, 2560), (300, 512), (2560, 2560),
                                    (2560, 10240), (10240, 2560), (17, 16384)])
@pytest.mark.parametrize("ncols", [4, 5, 6, 7, 8])
def test_exact_sums_and_the_dp4a_consumers_bits(kind, rows, K, ncols):
    t_gpu, _, t_orc, gen = KINDS[kind]
    salt = 7 * rows + K + ncols
    W = gen(rows, K, salt=salt)
    Wd = _planar(kind, W, rows, K)
    x = synth.activations(K, ncols, salt=salt)
    xq = oracle.quantize_q8_1(x)
    xqd = dev(xq)
    sumi, y_dbg = mmvq.debug_block_sums(t_gpu, Wd, rows, K, xqd, ncols, flags=TC)
    sel = np.unique(np.linspace(0, rows - 1, min(rows, 48)).astype(np.int64))
    s_ref = oracle.block_sums(t_orc, np.ascontiguousarray(W[sel]), sel.size, K, xq, ncols)
    assert np.array_equal(host(sumi)[:, sel], s_ref)
    y = mmvq.gemv(t_gpu, Wd, rows, K, xqd, ncols, flags=TC)
    assert _same_bits(y, y_dbg)
    assert _same_bits(y, mmvq.gemv(t_gpu, Wd, rows, K, xqd, ncols))
    assert _same_bits(y, mmvq.gemv(t_gpu, Wd, rows, K, xqd, ncols, flags=TC | mmvq.FLAG_XQ_STABLE))


@pytest.mark.parametrize("ncols", [4, 5])
def test_lm_head_same_bits_as_the_dp4a_consumer(ncols):
    rows, K = 151936, 2560
    t = mmvq.TYPE_Q6_K_PLANAR
    Wd = mmvq.repack_planar(dev(synth.q6_k_weights(rows, K, salt=3)), rows, K)
    xqd = mmvq.quantize_q8_1(dev(synth.activations(K, ncols, salt=3)))
    y = mmvq.gemv(t, Wd, rows, K, xqd, ncols, flags=TC)
    assert _same_bits(y, mmvq.gemv(t, Wd, rows, K, xqd, ncols))


def _extreme_blocks(kind, rows, nb, rng):
    """GGUF blocks whose codes and scales sit at the ends of their ranges:
    per block one code (lowest or highest), the largest scale magnitudes,
    and d = dmin = 1.0, mixed at random over rows and blocks."""
    one = np.frombuffer(np.float16(1.0).tobytes(), dtype=np.uint8)
    if kind == "q6_k_planar":
        W = np.zeros((rows, nb, 210), dtype=np.uint8)
        hi = rng.random((rows, nb)) < 0.5                     # code 63 (q = +31) or 0 (q = -32)
        W[..., 0:128] = np.where(hi[..., None], 0xFF, 0x00)
        W[..., 128:192] = np.where(hi[..., None], 0xFF, 0x00)
        sc = np.where(rng.random((rows, nb, 16)) < 0.5, -128, 127).astype(np.int8)
        W[..., 192:208] = sc.view(np.uint8)
        W[..., 208:210] = one
        return W
    size = 144 if kind == "q4_k_planar" else 176
    W = np.zeros((rows, nb, size), dtype=np.uint8)
    W[..., 0:2] = one
    W[..., 2:4] = one
    W[..., 4:16] = 0xFF                                       # every scale and min 63
    hi = rng.random((rows, nb)) < 0.75
    W[..., size - 128:] = np.where(hi[..., None], 0xFF, 0x00)  # nibbles 15 or 0
    if size == 176:
        W[..., 16:48] = np.where(hi[..., None], 0xFF, 0x00)   # fifth bits: codes 31 or 0
    return W


@pytest.mark.parametrize("kind", list(KINDS))
@pytest.mark.parametrize("ncols", [4, 8])
def test_extreme_codes_scales_and_activations(kind, ncols):
    rows, K = 64, 2560
    rng = np.random.default_rng(11)
    W = _extreme_blocks(kind, rows, K // 256, rng)
    Wd = _planar(kind, W, rows, K)
    # columns of +1, -1 and mixed signs: every Q8_1 quant is +-127
    x = np.ones((ncols, K), dtype=np.float32)
    x[1] = -1.0
    x[2:] = np.where(rng.random((ncols - 2, K)) < 0.5, -1.0, 1.0)
    t_gpu, _, t_orc, _ = KINDS[kind]
    xq = oracle.quantize_q8_1(x)
    assert np.all(np.abs(xq[..., 4:].view(np.int8)) == 127)
    xqd = dev(xq)
    sumi, y_dbg = mmvq.debug_block_sums(t_gpu, Wd, rows, K, xqd, ncols, flags=TC)
    s_ref = oracle.block_sums(t_orc, W, rows, K, xq, ncols)
    assert np.array_equal(host(sumi), s_ref)
    if kind == "q6_k_planar":  # the largest sums reach 2 * 128 * 16 * 32 * 127 = 16,646,144
        assert np.abs(s_ref).max() == 2 * 128 * 16 * 32 * 127
    y = mmvq.gemv(t_gpu, Wd, rows, K, xqd, ncols, flags=TC)
    assert _same_bits(y, y_dbg)
    assert _same_bits(y, mmvq.gemv(t_gpu, Wd, rows, K, xqd, ncols))
    y_ref, bound = oracle.gemv(t_orc, W, rows, K, xq, ncols, with_bound=True)
    assert_within_bound(host(y), y_ref, bound, f"{kind} extremes ncols={ncols}")


def test_padding_columns_stay_out_of_the_output():
    # five columns: the MMA lanes of columns 5-7 compute on zero fragments
    # and must not write; memory past the output stays untouched
    rows, K, ncols = 37, 2560, 5
    W = synth.q4_k_weights(rows, K, salt=4)
    Wd = _planar("q4_k_planar", W, rows, K)
    xqd = mmvq.quantize_q8_1(dev(synth.activations(K, ncols, salt=4)))
    canary = torch.full((ncols * rows + 256,), 777.0, device="cuda")
    out = canary[:ncols * rows].view(ncols, rows)
    mmvq.gemv(mmvq.TYPE_Q4_K_PLANAR, Wd, rows, K, xqd, ncols, out=out, flags=TC)
    assert np.all(host(canary[ncols * rows:]) == 777.0)
    assert mmvq.read_device_fault() == 0


def test_flag_is_ignored_below_four_columns_and_by_gguf_types():
    rows, K = 100, 2560
    W = synth.q6_k_weights(rows, K, salt=6)
    P = mmvq.repack_planar(dev(W), rows, K)
    for ncols in (1, 2, 3):
        xqd = mmvq.quantize_q8_1(dev(synth.activations(K, ncols, salt=ncols)))
        assert _same_bits(mmvq.gemv(mmvq.TYPE_Q6_K_PLANAR, P, rows, K, xqd, ncols, flags=TC),
                          mmvq.gemv(mmvq.TYPE_Q6_K_PLANAR, P, rows, K, xqd, ncols))
    xqd = mmvq.quantize_q8_1(dev(synth.activations(K, 6, salt=9)))
    Wg = dev(W)
    assert _same_bits(mmvq.gemv(mmvq.TYPE_Q6_K, Wg, rows, K, xqd, 6, flags=TC),
                      mmvq.gemv(mmvq.TYPE_Q6_K, Wg, rows, K, xqd, 6))


def test_fp32_columns_with_the_flag():
    # mmvq_gemv_f32 takes the quantiser and the product for the flag (its
    # one-launch instance is a dp4a one): the same xq bytes and y bits
    rows, K, ncols = 2560, 2560, 6
    W = synth.q6_k_weights(rows, K, salt=12)
    P = mmvq.repack_planar(dev(W), rows, K)
    x = dev(synth.activations(K, ncols, salt=12))
    y0, q0 = mmvq.gemv_f32(mmvq.TYPE_Q6_K_PLANAR, P, rows, K, x, ncols)
    y1, q1 = mmvq.gemv_f32(mmvq.TYPE_Q6_K_PLANAR, P, rows, K, x, ncols, flags=TC)
    assert np.array_equal(host(q0), host(q1))
    assert _same_bits(y0, y1)
    assert np.array_equal(host(q1), oracle.quantize_q8_1(host(x)))
