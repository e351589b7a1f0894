"""The pages' printed bandwidth figures pin the metric's byte accounting:
weight bytes of the matrix (rows x K/256 blocks x bytes per block) over the
call time, weights counted once whatever the column count.  Fixture:
tests/golden/pages_bandwidth.txt (each line cites its page and table)."""
import os

import pytest

from block_quantized_matvec_gb300.metrics import gbps, weight_bytes

HERE = os.path.dirname(os.path.abspath(__file__))


def _rows():
    out = []
    with open(os.path.join(HERE, "golden", "pages_bandwidth.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            src, fmt, n_in, n_out, bpb, cols, us, printed = [s.strip() for s in line.split("|")]
            out.append((src, fmt, int(n_in), int(n_out), int(bpb), int(cols), float(us), float(printed)))
    return out


@pytest.mark.parametrize("row", _rows(), ids=lambda r: r[0])
def test_weight_bandwidth_reproduces_printed_figure(row):
    src, fmt, n_in, n_out, bpb, cols, us, printed = row
    nbytes = weight_bytes(fmt, n_out, n_in)
    assert nbytes == n_out * n_in // 256 * bpb
    got = gbps(nbytes, us * 1e-6)
    # the pages print whole GB/s from unrounded times; allow the us rounding
    assert abs(got - printed) <= max(1.0, 0.02 * printed), (got, printed)
