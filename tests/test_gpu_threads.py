"""Several host threads calling the library at once, each on its own stream.

The launch choosers keep per-shape caches and set kernel attributes on first
use (both behind locks); these calls use shapes no other test has chosen a
launch for yet, from four threads at once, and must give the same bits as
the same calls made from one thread."""
import threading

import numpy as np
import pytest
import torch

from block_quantized_matvec_gb300 import mmvq, synth
from tests._gpu import dev, host

pytestmark = pytest.mark.gpu

# (planar type, GGUF source type, generator, rows, K, ncols): shapes used nowhere else
CASES = [(mmvq.TYPE_Q6_K_PLANAR, mmvq.TYPE_Q6_K, synth.q6_k_weights, 3001, 1792, 3),
         (mmvq.TYPE_Q4_K_PLANAR, mmvq.TYPE_Q4_K, synth.q4_k_weights, 4099, 1536, 5),
         (mmvq.TYPE_Q5_K_PLANAR, mmvq.TYPE_Q5_K, synth.q5_k_weights, 2049, 3328, 7),
         (mmvq.TYPE_Q6_K_PLANAR, mmvq.TYPE_Q6_K, synth.q6_k_weights, 777, 4864, 2)]


def test_concurrent_calls_from_four_threads_give_the_single_thread_bits():
    prepared = []
    for t, src, gen, rows, K, ncols in CASES:
        W = mmvq.repack_planar(dev(gen(rows, K, salt=rows)), rows, K, type_=src)
        x = dev(synth.activations(K, ncols, salt=K))
        prepared.append((t, W, rows, K, ncols, x))
    torch.cuda.synchronize()
    results = [None] * len(prepared)
    errors = []
    start = threading.Barrier(len(prepared))

    def worker(i):
        try:
            t, W, rows, K, ncols, x = prepared[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                start.wait()
                outs = []
                for _ in range(20):
                    xq = mmvq.quantize_q8_1(x, stream=s)
                    outs.append(mmvq.gemv(t, W, rows, K, xq, ncols, stream=s))
                s.synchronize()
                results[i] = [host(o).view(np.uint32) for o in outs]
        except Exception as e:                  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(prepared))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for (t, W, rows, K, ncols, x), res in zip(prepared, results):
        want = host(mmvq.gemv(t, W, rows, K, mmvq.quantize_q8_1(x), ncols)).view(np.uint32)
        for r in res:
            assert np.array_equal(r, want)
    assert mmvq.read_device_fault() == 0
