"""Parity at the full workload sizes, in the same launch configuration the
benchmark times: the GPU computes the whole matrix, the oracle recomputes a
seeded sample of rows one by one (block sums bit for bit, outputs within
the bound).  Shapes are the pages' matrices ("Strata" PR #2207 mmvq_bench
Q6_K table; PR #1774 dense matrices; the Q6_K LM head and its draft
subset, PR #2340)."""
import numpy as np
import pytest

import oracle
from block_quantized_matvec_gb300 import mmvq, synth
from tests._gpu import assert_within_bound, dev, host

pytestmark = pytest.mark.gpu

N_SAMPLE = 48


def _check_sampled(t_gpu, t_orc, W, Wd, rows, K, x, ncols, salt):
    xq = oracle.quantize_q8_1(x)
    xqd = mmvq.quantize_q8_1(dev(x))
    sumi, y = mmvq.debug_block_sums(t_gpu, Wd, rows, K, xqd, ncols)
    y_plain = mmvq.gemv(t_gpu, Wd, rows, K, xqd, ncols)
    rng = np.random.default_rng(salt)
    idx = np.unique(np.concatenate([[0, rows - 1], rng.choice(rows, N_SAMPLE, replace=False)]))
    import torch
    it = torch.from_numpy(idx).cuda()
    s_gpu = host(sumi[:, it, :])
    y_gpu = host(y_plain[:, it])
    assert np.array_equal(y_gpu.view(np.uint32), host(y[:, it]).view(np.uint32))
    Ws = np.ascontiguousarray(W[idx])
    assert np.array_equal(s_gpu, oracle.block_sums(t_orc, Ws, idx.size, K, xq, ncols))
    y_ref, bound = oracle.gemv(t_orc, Ws, idx.size, K, xq, ncols, with_bound=True)
    assert_within_bound(y_gpu, y_ref, bound, f"{rows}x{K} ncols={ncols}")


@pytest.mark.parametrize("rows,K", [(2560, 2560), (2560, 10240), (10240, 2560)])
@pytest.mark.parametrize("planar", [True, False])
def test_q6_k_sweep_shapes(rows, K, planar):
    W = synth.q6_k_weights(rows, K, salt=rows + K)
    Wd = dev(W)
    t = mmvq.TYPE_Q6_K
    if planar:
        Wd = mmvq.repack_planar(Wd, rows, K)
        t = mmvq.TYPE_Q6_K_PLANAR
    for ncols in (1, 2, 4, 6, 8):
        x = synth.activations(K, ncols, salt=ncols)
        _check_sampled(t, oracle.TYPE_Q6_K, W, Wd, rows, K, x, ncols, salt=ncols)


@pytest.mark.parametrize("rows,K", [(12288, 2560), (6144, 2560), (2560, 6144), (640, 2560),
                                    (512, 2560)])
@pytest.mark.parametrize("planar", [True, False])
def test_q4_k_dense_shapes(rows, K, planar):
    W = synth.q4_k_weights(rows, K, salt=rows + K)
    Wd = dev(W)
    t = mmvq.TYPE_Q4_K
    if planar:
        Wd = mmvq.repack_planar(Wd, rows, K, type_=mmvq.TYPE_Q4_K)
        t = mmvq.TYPE_Q4_K_PLANAR
    for ncols in (1, 4):
        x = synth.activations(K, ncols, salt=ncols)
        _check_sampled(t, oracle.TYPE_Q4_K, W, Wd, rows, K, x, ncols, salt=ncols)


@pytest.mark.parametrize("rows,K", [(12288, 2560), (6144, 2560), (2560, 6144), (640, 2560),
                                    (512, 2560)])
def test_q5_k_dense_shapes(rows, K):
    W = synth.q5_k_weights(rows, K, salt=rows + K)
    Wd = mmvq.repack_planar(dev(W), rows, K, type_=mmvq.TYPE_Q5_K)
    for ncols in (1, 4):
        x = synth.activations(K, ncols, salt=ncols)
        _check_sampled(mmvq.TYPE_Q5_K_PLANAR, oracle.TYPE_Q5_K, W, Wd, rows, K, x, ncols,
                       salt=ncols)


def test_lm_head_and_draft_head():
    rows, K = 151936, 2560
    W = synth.q6_k_weights(rows, K, salt=7)
    P = mmvq.repack_planar(dev(W), rows, K)
    ids = synth.draft_rows(4096, rows)
    D, status = mmvq.gather_planar_rows(P, rows, K, dev(ids))
    assert host(status)[0] == 0
    Wdraft = np.ascontiguousarray(W[ids])
    for ncols in (1, 2, 3, 4, 5):
        x = synth.activations(K, ncols, salt=20 + ncols)
        _check_sampled(mmvq.TYPE_Q6_K_PLANAR, oracle.TYPE_Q6_K, W, P, rows, K, x, ncols, ncols)
        _check_sampled(mmvq.TYPE_Q6_K_PLANAR, oracle.TYPE_Q6_K, Wdraft, D, 4096, K, x, ncols,
                       ncols)


@pytest.mark.parametrize("kind,rows,K", [("q6_k", 10247, 2560), ("q4_k", 12300, 2560),
                                         ("q5_k", 6151, 2560)])
def test_tall_ragged_matrices_with_several_row_groups_per_cta(kind, rows, K):
    # row counts just past a 16-row multiple, at sizes where the launch shape
    # gives each CTA more than one row group (G > 1); the sample holds the
    # last, partial row group
    gen = {"q6_k": synth.q6_k_weights, "q4_k": synth.q4_k_weights, "q5_k": synth.q5_k_weights}[kind]
    src = {"q6_k": mmvq.TYPE_Q6_K, "q4_k": mmvq.TYPE_Q4_K, "q5_k": mmvq.TYPE_Q5_K}[kind]
    t = {"q6_k": mmvq.TYPE_Q6_K_PLANAR, "q4_k": mmvq.TYPE_Q4_K_PLANAR,
         "q5_k": mmvq.TYPE_Q5_K_PLANAR}[kind]
    t_orc = {"q6_k": oracle.TYPE_Q6_K, "q4_k": oracle.TYPE_Q4_K, "q5_k": oracle.TYPE_Q5_K}[kind]
    W = gen(rows, K, salt=rows)
    Wd = mmvq.repack_planar(dev(W), rows, K, type_=src)
    groups = []
    for ncols in (1, 2, 4):
        groups.append(mmvq.launch_shape(t, rows, K, ncols)["G"])
        x = synth.activations(K, ncols, salt=30 + ncols)
        _check_sampled(t, t_orc, W, Wd, rows, K, x, ncols, salt=ncols)
    assert max(groups) > 1, groups
