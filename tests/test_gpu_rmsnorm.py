"""RMSNorm then Q8_1 on the GPU against the oracle, through the C ABI: the
normalised values and the Q8_1 bytes bit for bit (the mean square is reduced
in fp64 on both sides, so the fp32 scale agrees; the rest is the same fp32
operations in the same order)."""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_matvec_gb300 import mmvq, synth
from tests._gpu import dev, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("K", [32, 256, 2560, 10240, 16384])
@pytest.mark.parametrize("ncols", [1, 3, 8])
@pytest.mark.parametrize("eps", [0.0, 1e-6])
def test_rmsnorm_quantize_bit_exact(K, ncols, eps):
    x = synth.activations(K, ncols, salt=K + ncols) * 3.0
    w = synth.activations(K, 1, salt=K + 7)[0]
    xq_ref, y_ref = oracle.rmsnorm_quantize_q8_1(x, w, eps)
    y = torch.empty((ncols, K), dtype=torch.float32, device="cuda")
    xq = mmvq.rmsnorm_quantize_q8_1(dev(x), dev(w), eps, y_out=y)
    assert np.array_equal(host(y).view(np.uint32), y_ref.view(np.uint32))
    assert np.array_equal(host(xq), xq_ref)


def test_rmsnorm_strided_columns_and_zero_weights():
    K, ncols, ldx = 512, 4, 640
    xs = synth.activations(ldx, ncols, salt=90)
    w = synth.activations(K, 1, salt=91)[0]
    xq_ref, _ = oracle.rmsnorm_quantize_q8_1(np.ascontiguousarray(xs[:, :K]), w, 1e-5)
    xq = mmvq.rmsnorm_quantize_q8_1(dev(xs)[:, :K], dev(w), 1e-5)
    assert np.array_equal(host(xq), xq_ref)
    z = mmvq.rmsnorm_quantize_q8_1(dev(xs)[:, :K], torch.zeros(K, device="cuda"), 1e-5)
    assert not host(z).any()
