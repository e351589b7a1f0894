"""mmvq_gemv_ex with MMVQ_FLAG_XQ_STABLE: the same bits as mmvq_gemv, and no
ordering race when the activation buffer is re-quantised between calls
(every flagged call must see the columns quantised just before it)."""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_matvec_gb300 import mmvq, synth
from tests._gpu import assert_within_bound, dev, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,K,ncols", [(2560, 2560, 1), (1000, 10240, 4), (37, 512, 8)])
def test_stable_flag_gives_identical_bits(rows, K, ncols):
    W = synth.q6_k_weights(rows, K, salt=3)
    P = mmvq.repack_planar(dev(W), rows, K)
    xq = mmvq.quantize_q8_1(dev(synth.activations(K, ncols, salt=3)))
    a = host(mmvq.gemv(mmvq.TYPE_Q6_K_PLANAR, P, rows, K, xq, ncols))
    b = host(mmvq.gemv(mmvq.TYPE_Q6_K_PLANAR, P, rows, K, xq, ncols, flags=mmvq.FLAG_XQ_STABLE))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_flagged_chain_sees_each_new_activation():
    rows, K, ncols, iters = 2560, 2560, 2, 24
    mats = [synth.q6_k_weights(rows, K, salt=s) for s in range(3)]
    Ps = [mmvq.repack_planar(dev(W), rows, K) for W in mats]
    xs = [synth.activations(K, ncols, salt=100 + i) for i in range(iters)]
    x_dev = torch.empty((ncols, K), device="cuda")
    xq = torch.empty((ncols, K // 32, 36), dtype=torch.uint8, device="cuda")
    outs = torch.empty((iters, 3, ncols, rows), device="cuda")
    xs_dev = [dev(x) for x in xs]
    torch.cuda.synchronize()
    for i in range(iters):
        x_dev.copy_(xs_dev[i])
        mmvq.quantize_q8_1(x_dev, out=xq)
        for m in range(3):
            mmvq.gemv(mmvq.TYPE_Q6_K_PLANAR, Ps[m], rows, K, xq, ncols, out=outs[i, m],
                      flags=mmvq.FLAG_XQ_STABLE if m else 0)
    got = host(outs)
    for i in range(iters):
        xq_ref = oracle.quantize_q8_1(xs[i])
        for m in range(3):
            y, bound = oracle.gemv(oracle.TYPE_Q6_K, mats[m], rows, K, xq_ref, ncols, with_bound=True)
            assert_within_bound(got[i, m], y, bound, f"iter {i} matrix {m}")


def test_unknown_flag_bits_are_rejected():
    t = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(mmvq.MMVQError):
        mmvq.gemv(mmvq.TYPE_Q6_K_PLANAR, t, 16, 256, t, 1, out=torch.empty(16, device="cuda"), flags=4)
