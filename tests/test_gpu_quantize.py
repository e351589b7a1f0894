"""Q8_1 quantiser and SiLU*up requantiser on the GPU against the oracle.
Q8_1 bytes are compared bit for bit ("Strata" PR #2340 / PR #1774 block
format; exact d = amax/127, round-half-away, s = d*sum q)."""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_matvec_gb300 import mmvq, synth
from tests._gpu import dev, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("K,ncols", [(32, 1), (2560, 1), (2560, 8), (10240, 5), (6144, 3),
                                     (768, 64), (96, 7)])
def test_quantize_bit_exact(K, ncols):
    x = synth.activations(K, ncols, salt=K + ncols)
    got = host(mmvq.quantize_q8_1(dev(x)))
    assert np.array_equal(got, oracle.quantize_q8_1(x))


def test_quantize_edge_values_bit_exact():
    rng = np.random.default_rng(5)
    x = np.zeros((6, 256), np.float32)
    x[1, :32] = 127.0 * np.sign(rng.standard_normal(32))        # exact d = 1
    x[1, 32:64] = np.arange(32) - 15.5                            # ties (x.5)
    x[2] = rng.standard_normal(256) * 1e-30                       # tiny values
    x[3] = rng.standard_normal(256) * 1e30                        # huge values
    x[4, ::32] = 3.0                                              # single nonzero per block
    x[5] = np.float32(2.0) ** rng.integers(-20, 20, 256) * np.sign(rng.standard_normal(256))
    got = host(mmvq.quantize_q8_1(dev(x)))
    assert np.array_equal(got, oracle.quantize_q8_1(x))


def test_quantize_respects_ldx():
    x = synth.activations(3000, 3, salt=1)
    got = host(mmvq.quantize_q8_1(dev(x), K=2560))
    assert np.array_equal(got, oracle.quantize_q8_1(x, K=2560))


def test_silu_mul_quantize_matches_oracle():
    F, n = 768, 64
    gu = synth.gate_up(n, F, salt=3)
    gu[0, :F] = 0.0
    gu[1, :F] = -200.0                                            # exp overflow side
    h_gpu_t = torch.empty((n, F), dtype=torch.float32, device="cuda")
    xq_gpu = host(mmvq.silu_mul_quantize_q8_1(dev(gu), F, h_out=h_gpu_t))
    h_gpu = host(h_gpu_t)
    _, h_orc = oracle.silu_mul_quantize(gu, F)
    # h within a few ulps (expf on the GPU and the host may differ by an ulp)
    assert np.all(np.abs(h_gpu - h_orc) <= 4e-7 * np.abs(h_orc) + 1e-30)
    # the Q8_1 bytes are the oracle's quantisation of the GPU's own h, on
    # every block: the requantisation adds no rounding of its own
    assert np.array_equal(xq_gpu, oracle.quantize_q8_1(h_gpu))
