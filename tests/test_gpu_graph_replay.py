"""The hot path captured in CUDA graphs and replayed, as decode engines run it
("Strata" PR #2746 "B70 validation": the expert calls were also checked
under graph replay; the pages' timings are graph replays), and the dense
products over several activation patterns (the same validation runs five
activation patterns through the expert kernels).

* Replays of a captured step, with new inputs copied into the captured
  buffers between replays, give the same bits as the same calls made
  eagerly: launches chained by programmatic dependent launch inside a graph
  read what their predecessors wrote.
* Dense products of pattern columns (zeros, a constant, one-hot, tiny
  values whose Q8_1 scale flushes to zero in fp16, large values, mixed
  signs) match the oracle: block sums bit for bit, outputs within the bound.
"""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_matvec_gb300 import mmvq, synth
from tests._gpu import assert_within_bound, dev, host

pytestmark = pytest.mark.gpu


def _graph(fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
        fn()
    torch.cuda.synchronize()
    return g


def _bits(t):
    return host(t).view(np.uint32) if t.dtype == torch.float32 else host(t)


def test_dense_step_replayed_equals_eager_calls():
    # one activation shared by three matrices (the later calls flagged
    # stable), then a call on the first product's output as its activation
    K, ncols = 2560, 4
    mats = []
    for i, (rows, src) in enumerate([(2560, mmvq.TYPE_Q6_K), (10247, mmvq.TYPE_Q4_K),
                                     (640, mmvq.TYPE_Q5_K)]):
        gen = {mmvq.TYPE_Q6_K: synth.q6_k_weights, mmvq.TYPE_Q4_K: synth.q4_k_weights,
               mmvq.TYPE_Q5_K: synth.q5_k_weights}[src]
        t = {mmvq.TYPE_Q6_K: mmvq.TYPE_Q6_K_PLANAR, mmvq.TYPE_Q4_K: mmvq.TYPE_Q4_K_PLANAR,
             mmvq.TYPE_Q5_K: mmvq.TYPE_Q5_K_PLANAR}[src]
        mats.append((t, rows, mmvq.repack_planar(dev(gen(rows, K, salt=40 + i)), rows, K,
                                                 type_=src)))
    x = torch.empty((ncols, K), device="cuda")
    xq = torch.empty((ncols, K // 32, mmvq.Q8_1_BYTES), dtype=torch.uint8, device="cuda")
    ys = [torch.empty((ncols, rows), device="cuda") for _, rows, _ in mats]
    xq2 = torch.empty_like(xq)
    y2 = torch.empty((ncols, 2560), device="cuda")

    def step():
        mmvq.quantize_q8_1(x, out=xq)
        for n, ((t, rows, W), y) in enumerate(zip(mats, ys)):
            mmvq.gemv(t, W, rows, K, xq, ncols, out=y, flags=mmvq.FLAG_XQ_STABLE if n else 0)
        mmvq.quantize_q8_1(ys[0], out=xq2)                # the next product depends on y0
        mmvq.gemv(mats[0][0], mats[0][2], 2560, K, xq2, ncols, out=y2)

    x.copy_(dev(synth.activations(K, ncols, salt=1)))
    g = _graph(step)
    for r in range(3):
        xr = dev(synth.activations(K, ncols, salt=100 + r))
        x.copy_(xr)
        g.replay()
        torch.cuda.synchronize()
        got = [_bits(y) for y in ys] + [_bits(y2)]
        x.copy_(xr)
        step()                                            # the same calls, eagerly
        torch.cuda.synchronize()
        want = [_bits(y) for y in ys] + [_bits(y2)]
        for a, b in zip(got, want):
            assert np.array_equal(a, b)
    assert mmvq.read_device_fault() == 0


@pytest.mark.parametrize("T", [1, 2, 8])
def test_expert_layer_replayed_with_new_routings_equals_eager_launches(T):
    E, H, F, k = 64, 2560, 768, 8
    W = synth.expert_weights("q4_k", E, 2 * F, H, salt=1)
    W_gu = torch.cat([mmvq.repack_planar(dev(W[e]), 2 * F, H, type_=mmvq.TYPE_Q4_K)
                      for e in range(E)])
    W = synth.expert_weights("q4_k", E, H, F, salt=2)
    W_dn = torch.cat([mmvq.repack_planar(dev(W[e]), H, F, type_=mmvq.TYPE_Q4_K)
                      for e in range(E)])
    x = dev(synth.moe_hidden(H, T, salt=3))
    topk = torch.empty((T, k), dtype=torch.int32, device="cuda")
    n = T * k
    bufs = dict(gu=torch.empty((n, 2 * F), device="cuda"),
                hq=torch.empty((n, F // 32, mmvq.Q8_1_BYTES), dtype=torch.uint8, device="cuda"),
                y=torch.empty((n, H), device="cuda"),
                xq=torch.empty((T, H // 32, mmvq.Q8_1_BYTES), dtype=torch.uint8, device="cuda"))
    sync = mmvq.expert_ffn_workspace("cuda")

    def layer():
        return mmvq.expert_ffn(mmvq.TYPE_Q4_K_PLANAR, W_gu, W_dn, E, H, F, x, topk, sync=sync,
                               **bufs)

    topk.copy_(dev(synth.routing(T, k, E, salt=0)))
    holder = {}
    g = _graph(lambda: holder.update(out=layer()))
    gout = holder["out"]                                  # the graph's own output tensors
    keys = ("gu", "hq", "y", "xq", "offsets", "slot_of")
    for r in range(4):
        tk = dev(synth.routing(T, k, E, salt=10 + r))
        topk.copy_(tk)
        g.replay()
        torch.cuda.synchronize()
        got = {key: _bits(gout[key]) for key in keys}
        topk.copy_(tk)
        eager = layer()
        torch.cuda.synchronize()
        for key in keys:
            assert np.array_equal(got[key], _bits(eager[key])), key
    assert host(sync)[0] & 0x7fffffff == 0
    assert mmvq.read_device_fault() == 0


def _patterns(K):
    rng = np.random.default_rng(17)
    cols = [np.zeros(K), np.full(K, 0.75), np.zeros(K), rng.standard_normal(K) * 1e-7,
            rng.standard_normal(K) * 300.0, np.where(np.arange(K) % 2, 1.0, -1.0) *
            rng.uniform(0.5, 2.0, K)]
    cols[2][K // 3] = -5.0                                # one-hot
    return np.stack(cols).astype(np.float32)


@pytest.mark.parametrize("src,t_gpu,t_orc,gen", [
    (mmvq.TYPE_Q6_K, mmvq.TYPE_Q6_K_PLANAR, oracle.TYPE_Q6_K, synth.q6_k_weights),
    (mmvq.TYPE_Q4_K, mmvq.TYPE_Q4_K_PLANAR, oracle.TYPE_Q4_K, synth.q4_k_weights),
    (mmvq.TYPE_Q5_K, mmvq.TYPE_Q5_K_PLANAR, oracle.TYPE_Q5_K, synth.q5_k_weights)])
def test_dense_products_of_activation_patterns(src, t_gpu, t_orc, gen):
    rows, K = 37, 2560
    W = gen(rows, K, salt=6)
    Wd = mmvq.repack_planar(dev(W), rows, K, type_=src)
    x = _patterns(K)
    ncols = x.shape[0]
    xq = oracle.quantize_q8_1(x)
    xqd = mmvq.quantize_q8_1(dev(x))
    assert np.array_equal(host(xqd), xq)
    sumi, _ = mmvq.debug_block_sums(t_gpu, Wd, rows, K, xqd, ncols)
    y = host(mmvq.gemv(t_gpu, Wd, rows, K, xqd, ncols))
    assert np.array_equal(host(sumi), oracle.block_sums(t_orc, W, rows, K, xq, ncols))
    y_ref, bound = oracle.gemv(t_orc, W, rows, K, xq, ncols, with_bound=True)
    assert np.isfinite(y_ref).all()
    assert_within_bound(y, y_ref, bound, "activation patterns")
    assert np.all(y[0] == 0.0)                            # the zero column
