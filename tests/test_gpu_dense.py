"""Dense MMVQ on the GPU against the oracle, through the C ABI.

Per-32-block integer sums bit for bit; FP32 outputs within
|dy| <= 1e-5 * sum|t_b| + 1e-6 ("Strata" PR #1774: only the sub-block
summation order differs, so only the last bits may move).  Sizes span
several 16-row tiles and a ragged tail, K from one block to the maximum,
and every column count 1-8 (PR #2207)."""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_matvec_gb300 import mmvq, synth
from tests._gpu import assert_within_bound, dev, fnv1a, host

pytestmark = pytest.mark.gpu

KINDS = {
    "q6_k": (mmvq.TYPE_Q6_K, oracle.TYPE_Q6_K, synth.q6_k_weights),
    "q6_k_planar": (mmvq.TYPE_Q6_K_PLANAR, oracle.TYPE_Q6_K, synth.q6_k_weights),
    "q4_k": (mmvq.TYPE_Q4_K, oracle.TYPE_Q4_K, synth.q4_k_weights),
    "q4_k_planar": (mmvq.TYPE_Q4_K_PLANAR, oracle.TYPE_Q4_K, synth.q4_k_weights),
    "q5_k_planar": (mmvq.TYPE_Q5_K_PLANAR, oracle.TYPE_Q5_K, synth.q5_k_weights),
}


def _weights(kind, rows, K, salt):
    t_gpu, t_orc, gen = KINDS[kind]
    W = gen(rows, K, salt=salt)
    Wd = dev(W)
    if kind == "q6_k_planar":
        Wd = mmvq.repack_planar(Wd, rows, K)
    if kind == "q4_k_planar":
        Wd = mmvq.repack_planar(Wd, rows, K, type_=mmvq.TYPE_Q4_K)
    if kind == "q5_k_planar":
        Wd = mmvq.repack_planar(Wd, rows, K, type_=mmvq.TYPE_Q5_K)
    return W, Wd, t_gpu, t_orc


SHAPES = [(1, 256), (17, 512), (37, 2560), (100, 768), (160, 2560), (33, 10240), (5, 16384)]


@pytest.mark.parametrize("kind", list(KINDS))
@pytest.mark.parametrize("rows,K", SHAPES)
@pytest.mark.parametrize("ncols", [1, 2, 3, 4, 5, 6, 7, 8])
def test_block_sums_exact_and_outputs_within_bound(kind, rows, K, ncols):
    salt = rows * 131 + K + ncols
    W, Wd, t_gpu, t_orc = _weights(kind, rows, K, salt)
    x = synth.activations(K, ncols, salt=salt)
    xq = oracle.quantize_q8_1(x)
    xqd = mmvq.quantize_q8_1(dev(x))
    assert np.array_equal(host(xqd), xq)
    sumi, y_dbg = mmvq.debug_block_sums(t_gpu, Wd, rows, K, xqd, ncols)
    y = mmvq.gemv(t_gpu, Wd, rows, K, xqd, ncols)
    s_ref = oracle.block_sums(t_orc, W, rows, K, xq, ncols)
    y_ref, bound = oracle.gemv(t_orc, W, rows, K, xq, ncols, with_bound=True)
    assert np.array_equal(host(sumi), s_ref)
    yh = host(y)
    assert np.array_equal(yh.view(np.uint32), host(y_dbg).view(np.uint32))
    assert_within_bound(yh, y_ref, bound, f"{kind} {rows}x{K} ncols={ncols}")


@pytest.mark.parametrize("kind", list(KINDS))
def test_columns_bit_identical_to_single_column_calls(kind):
    rows, K, ncols = 200, 2560, 8
    W, Wd, t_gpu, _ = _weights(kind, rows, K, 77)
    xqd = mmvq.quantize_q8_1(dev(synth.activations(K, ncols, salt=77)))
    y = host(mmvq.gemv(t_gpu, Wd, rows, K, xqd, ncols))
    for c in range(ncols):
        one = host(mmvq.gemv(t_gpu, Wd, rows, K, xqd[c:c + 1].contiguous(), 1))
        assert np.array_equal(y[c].view(np.uint32), one[0].view(np.uint32))


@pytest.mark.parametrize("kind", list(KINDS))
def test_zero_activations_give_exact_zero_and_runs_are_deterministic(kind):
    rows, K = 300, 2560
    W, Wd, t_gpu, _ = _weights(kind, rows, K, 5)
    xq0 = mmvq.quantize_q8_1(torch.zeros((3, K), dtype=torch.float32, device="cuda"))
    y0 = host(mmvq.gemv(t_gpu, Wd, rows, K, xq0, 3))
    assert np.all(y0 == 0.0)
    xqd = mmvq.quantize_q8_1(dev(synth.activations(K, 4, salt=5)))
    h = {fnv1a(host(mmvq.gemv(t_gpu, Wd, rows, K, xqd, 4))) for _ in range(3)}
    assert len(h) == 1


def test_planar_and_gguf_kernels_agree_within_bound():
    rows, K, ncols = 1000, 2560, 4
    W = synth.q6_k_weights(rows, K, salt=8)
    Wd = dev(W)
    P = mmvq.repack_planar(Wd, rows, K)
    x = synth.activations(K, ncols, salt=8)
    xq = oracle.quantize_q8_1(x)
    xqd = mmvq.quantize_q8_1(dev(x))
    a = host(mmvq.gemv(mmvq.TYPE_Q6_K, Wd, rows, K, xqd, ncols))
    b = host(mmvq.gemv(mmvq.TYPE_Q6_K_PLANAR, P, rows, K, xqd, ncols))
    _, bound = oracle.gemv(oracle.TYPE_Q6_K, W, rows, K, xq, ncols, with_bound=True)
    assert_within_bound(a, b, 2 * bound)


def test_output_rows_outside_the_matrix_are_untouched():
    rows, K = 37, 512
    W, Wd, t_gpu, _ = _weights("q6_k_planar", rows, K, 9)
    xqd = mmvq.quantize_q8_1(dev(synth.activations(K, 2, salt=9)))
    canary = torch.full((2 * rows + 64,), 12345.0, device="cuda")
    out = canary[:2 * rows].view(2, rows)
    mmvq.gemv(t_gpu, Wd, rows, K, xqd, 2, out=out)
    assert np.all(host(canary[2 * rows:]) == 12345.0)


@pytest.mark.parametrize("kind", list(KINDS))
@pytest.mark.parametrize("rows,K,ncols", [(2560, 10240, 8), (2560, 10240, 6), (33, 10240, 7),
                                          (5, 16384, 8)])
def test_cluster_k_split_exact_sums_and_repeatable(kind, rows, K, ncols):
    # six to eight columns of a long row run with each row group's K split
    # over a pair of CTAs (partials added through distributed shared memory)
    if kind.endswith("_planar"):
        t = KINDS[kind][0]
        assert mmvq.launch_shape(t, rows, K, ncols)["cluster"] == 2
    salt = rows + K + ncols
    W, Wd, t_gpu, t_orc = _weights(kind, rows, K, salt)
    x = synth.activations(K, ncols, salt=salt)
    xq = oracle.quantize_q8_1(x)
    xqd = mmvq.quantize_q8_1(dev(x))
    sel = np.unique(np.linspace(0, rows - 1, min(rows, 64)).astype(np.int64))
    sumi, y_dbg = mmvq.debug_block_sums(t_gpu, Wd, rows, K, xqd, ncols)
    s_ref = oracle.block_sums(t_orc, np.ascontiguousarray(W[sel]), sel.size, K, xq, ncols)
    assert np.array_equal(host(sumi)[:, sel], s_ref)
    runs = [host(mmvq.gemv(t_gpu, Wd, rows, K, xqd, ncols)) for _ in range(3)]
    for r in runs[1:]:
        assert np.array_equal(r.view(np.uint32), runs[0].view(np.uint32))
    assert np.array_equal(runs[0].view(np.uint32), host(y_dbg).view(np.uint32))
    y_ref, bound = oracle.gemv(t_orc, np.ascontiguousarray(W[sel]), sel.size, K, xq, ncols,
                               with_bound=True)
    assert_within_bound(runs[0][:, sel], y_ref, bound, f"{kind} {rows}x{K} ncols={ncols}")
