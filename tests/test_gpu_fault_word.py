"""Failure detection without a GPU fault: the library's bounded barrier wait,
run to expiry on a barrier nothing completes, reports through the device
fault word on the host, and the context stays usable afterwards."""
import numpy as np
import pytest

import oracle
from block_quantized_matvec_gb300 import mmvq, synth
from tests._gpu import assert_within_bound, dev, host

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_cleared():
    mmvq.read_device_fault()                      # start from a clear word
    mmvq.selftest_wait_timeout(2000)
    assert mmvq.read_device_fault() == 1          # bit 1: a barrier wait ran out
    assert mmvq.read_device_fault() == 0          # reading clears it


def test_context_usable_after_a_timeout():
    mmvq.selftest_wait_timeout(1000)
    assert mmvq.read_device_fault() == 1
    rows, K = 300, 2560
    W = synth.q6_k_weights(rows, K, salt=61)
    Wd = mmvq.repack_planar(dev(W), rows, K)
    x = synth.activations(K, 2, salt=61)
    y = host(mmvq.gemv(mmvq.TYPE_Q6_K_PLANAR, Wd, rows, K, mmvq.quantize_q8_1(dev(x)), 2))
    y_ref, bound = oracle.gemv(oracle.TYPE_Q6_K, W, rows, K, oracle.quantize_q8_1(x), 2,
                               with_bound=True)
    assert_within_bound(y, y_ref, bound, "after timeout")
    assert mmvq.read_device_fault() == 0          # a normal call leaves it clear
