"""Pins for the oracle's RMSNorm-then-Q8_1 prologue (PR #1774 "How it was
checked" names the opt-in fused norm without a formula; the reading is the
plain RMS norm with a weight vector, mean square accumulated in fp64).

Each pin rests on something other than the oracle's own formula:
* exact power-of-two scale invariance (eps = 0): RMSNorm(2^k x) has the same
  bits as RMSNorm(x), since every rounding sees the same mantissas;
* a constant vector (closed form: x = c gives y = w * sign(c) * 1/sqrt(1 + eps/c^2));
* the fp64 sum of squares against math.fsum (the correctly rounded sum);
* zero weights or zero input give all-zero Q8_1 blocks;
* the bytes are the plain quantiser's bytes of the returned y.
"""
import math

import numpy as np
import pytest

import oracle
from block_quantized_matvec_gb300 import synth


@pytest.mark.parametrize("k", [-3, -1, 1, 5])
def test_power_of_two_scaling_leaves_the_bytes_unchanged(k):
    K = 2560
    x = synth.activations(K, 3, salt=70)
    w = synth.activations(K, 1, salt=71)[0]
    a, ya = oracle.rmsnorm_quantize_q8_1(x, w, 0.0)
    b, yb = oracle.rmsnorm_quantize_q8_1(np.ldexp(x, k).astype(np.float32), w, 0.0)
    assert np.array_equal(a, b) and np.array_equal(ya.view(np.uint32), yb.view(np.uint32))


@pytest.mark.parametrize("c,eps", [(3.0, 0.0), (-0.5, 1e-6), (1e-3, 1e-6)])
def test_constant_vector_closed_form(c, eps):
    K = 256
    x = np.full((1, K), c, np.float32)
    w = np.linspace(-2, 2, K).astype(np.float32)
    _, y = oracle.rmsnorm_quantize_q8_1(x, w, eps)
    expect = w.astype(np.float64) * math.copysign(1.0, c) / math.sqrt(1.0 + eps / (c * c))
    assert np.all(np.abs(y[0] - expect) <= 3e-7 * np.abs(expect) + 1e-30)


def test_mean_square_is_accumulated_in_fp64():
    # 1e4 large and 1e4 tiny squares: an fp32 accumulation loses the tiny ones
    K = 20480
    x = np.concatenate([np.full(K // 2, 1000.0, np.float32), np.full(K // 2, 1e-3, np.float32)])
    w = np.ones(K, np.float32)
    _, y = oracle.rmsnorm_quantize_q8_1(x[None, :], w, 0.0)
    ms = math.fsum(float(v) * float(v) for v in x) / K
    scale = np.float32(1.0 / math.sqrt(ms))
    assert y[0, 0] == np.float32(np.float32(1000.0) * scale)
    assert y[0, -1] == np.float32(np.float32(1e-3) * scale)


def test_zeros_give_zero_blocks_and_bytes_match_the_plain_quantiser():
    K = 512
    x = synth.activations(K, 2, salt=72)
    q0, _ = oracle.rmsnorm_quantize_q8_1(x, np.zeros(K, np.float32), 1e-6)
    assert not q0.any()
    qz, _ = oracle.rmsnorm_quantize_q8_1(np.zeros((2, K), np.float32), np.ones(K, np.float32), 1e-6)
    assert not qz.any()
    q, y = oracle.rmsnorm_quantize_q8_1(x, synth.activations(K, 1, salt=73)[0], 1e-6)
    assert np.array_equal(q, oracle.quantize_q8_1(y))


def test_unit_weights_give_unit_rms():
    K = 4096
    x = synth.activations(K, 4, salt=74) * 7.0
    _, y = oracle.rmsnorm_quantize_q8_1(x, np.ones(K, np.float32), 0.0)
    rms = np.sqrt(np.mean(y.astype(np.float64) ** 2, axis=1))
    assert np.all(np.abs(rms - 1.0) < 1e-6)
