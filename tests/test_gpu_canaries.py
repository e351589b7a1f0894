"""Canary bytes around every output buffer of the library (in place of a
memory checker, which this setup does not offer): each output is the front
of a larger device buffer filled with a byte pattern, and after the call the
bytes past the output, and the rows the contract says are not written, must
still hold the pattern.  Shapes are ragged (row counts off the 16-row tile,
odd column and position counts) so that a tile-rounded store would show."""
import numpy as np
import pytest
import torch

from block_quantized_matvec_gb300 import mmvq, synth
from tests._gpu import dev, host

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


def _guarded(nbytes):
    return torch.full((nbytes + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")


def _front(buf, nbytes, shape, dtype=torch.uint8):
    return buf[:nbytes].view(dtype).view(shape)


def _guard_intact(buf, nbytes):
    tail = host(buf[nbytes:])
    assert np.all(tail == PATTERN), f"{int(np.sum(tail != PATTERN))} guard bytes overwritten"


def _q8_bytes(ncols, K):
    return ncols * (K // 32) * mmvq.Q8_1_BYTES


@pytest.mark.parametrize("K,ncols", [(32, 1), (2560, 3), (10240, 8)])
def test_quantize_writes_only_its_blocks(K, ncols):
    x = dev(synth.activations(K, ncols, salt=K + ncols))
    nb = _q8_bytes(ncols, K)
    buf = _guarded(nb)
    mmvq.quantize_q8_1(x, out=_front(buf, nb, (ncols, K // 32, mmvq.Q8_1_BYTES)))
    _guard_intact(buf, nb)


def test_rmsnorm_quantize_writes_only_its_blocks():
    K, ncols = 2560, 5
    x = dev(synth.activations(K, ncols, salt=3))
    w = torch.linspace(0.5, 1.5, K, device="cuda")
    nb = _q8_bytes(ncols, K)
    buf = _guarded(nb)
    ybytes = ncols * K * 4
    ybuf = _guarded(ybytes)
    mmvq.rmsnorm_quantize_q8_1(x, w, 1e-6, out=_front(buf, nb, (ncols, K // 32, mmvq.Q8_1_BYTES)),
                               y_out=_front(ybuf, ybytes, (ncols, K), torch.float32))
    _guard_intact(buf, nb)
    _guard_intact(ybuf, ybytes)


def test_silu_mul_quantize_writes_only_its_rows():
    n, F = 37, 768
    gu = torch.randn(n, 2 * F, device="cuda")
    nb = _q8_bytes(n, F)
    buf = _guarded(nb)
    hbytes = n * F * 4
    hbuf = _guarded(hbytes)
    mmvq.silu_mul_quantize_q8_1(gu, F, out=_front(buf, nb, (n, F // 32, mmvq.Q8_1_BYTES)),
                                h_out=_front(hbuf, hbytes, (n, F), torch.float32))
    _guard_intact(buf, nb)
    _guard_intact(hbuf, hbytes)


@pytest.mark.parametrize("src", [mmvq.TYPE_Q6_K, mmvq.TYPE_Q4_K, mmvq.TYPE_Q5_K])
def test_repack_and_gather_write_only_their_tiles(src):
    rows, K = 37, 512
    gen = {mmvq.TYPE_Q6_K: synth.q6_k_weights, mmvq.TYPE_Q4_K: synth.q4_k_weights,
           mmvq.TYPE_Q5_K: synth.q5_k_weights}[src]
    W = dev(gen(rows, K, salt=5))
    nb = mmvq.planar_bytes(rows, K, src)
    buf = _guarded(nb)
    P = mmvq.repack_planar(W, rows, K, out=buf[:nb], type_=src)
    _guard_intact(buf, nb)
    if src == mmvq.TYPE_Q6_K:
        ids = torch.tensor([36, 0, 17, 17, 5], dtype=torch.int32, device="cuda")
        gb = mmvq.planar_bytes(ids.numel(), K, src)
        gbuf = _guarded(gb)
        _, status = mmvq.gather_planar_rows(P, rows, K, ids, out=gbuf[:gb])
        assert host(status)[0] == 0
        _guard_intact(gbuf, gb)


@pytest.mark.parametrize("type_,src,gen", [
    (mmvq.TYPE_Q6_K_PLANAR, mmvq.TYPE_Q6_K, synth.q6_k_weights),
    (mmvq.TYPE_Q4_K_PLANAR, mmvq.TYPE_Q4_K, synth.q4_k_weights),
    (mmvq.TYPE_Q5_K_PLANAR, mmvq.TYPE_Q5_K, synth.q5_k_weights),
    (mmvq.TYPE_Q6_K, None, synth.q6_k_weights),
    (mmvq.TYPE_Q4_K, None, synth.q4_k_weights)])
@pytest.mark.parametrize("rows,ncols", [(37, 3), (10247, 8)])
def test_gemv_writes_only_its_outputs(type_, src, gen, rows, ncols):
    K = 2560
    W = dev(gen(rows, K, salt=rows))
    if src is not None:
        W = mmvq.repack_planar(W, rows, K, type_=src)
    xq = mmvq.quantize_q8_1(dev(synth.activations(K, ncols, salt=1)))
    nb = ncols * rows * 4
    buf = _guarded(nb)
    mmvq.gemv(type_, W, rows, K, xq, ncols, out=_front(buf, nb, (ncols, rows), torch.float32))
    _guard_intact(buf, nb)


def _planar_experts(E, rows, K, salt):
    W = synth.expert_weights("q4_k", E, rows, K, salt=salt)
    return torch.cat([mmvq.repack_planar(dev(W[e]), rows, K, type_=mmvq.TYPE_Q4_K)
                      for e in range(E)])


def test_grouped_leaves_dropped_positions_and_the_guard_alone():
    E, H, F, T, k = 8, 512, 256, 4, 2
    topk = synth.routing(T, k, E, salt=3).copy()
    topk[2, 1] = E + 5                                    # dropped: one position fewer
    xq, eids, offs, act, _, status = mmvq.quantize_route_groups(
        dev(synth.activations(H, T, salt=2)), dev(topk), E)
    n_valid = int(host(offs)[E])
    assert n_valid == T * k - 1 and host(status)[0] == mmvq.ERR_ROUTING
    W = _planar_experts(E, 2 * F, H, salt=1)
    nb = T * k * 2 * F * 4
    buf = _guarded(nb)
    mmvq.grouped(mmvq.TYPE_Q4_K_PLANAR, W, E, 2 * F, H, eids, offs, act, xq, T, T * k,
                 out=_front(buf, nb, (T * k, 2 * F), torch.float32))
    _guard_intact(buf, n_valid * 2 * F * 4)               # the unused last row and the guard


def test_expert_ffn_leaves_dropped_positions_and_the_guard_alone():
    E, H, F, T, k = 16, 512, 256, 3, 4
    topk = synth.routing(T, k, E, salt=4).copy()
    topk[0, 2] = -1
    topk[2, 3] = E                                        # two dropped entries
    x = dev(synth.moe_hidden(H, T, salt=4))
    W_gu = _planar_experts(E, 2 * F, H, salt=1)
    W_dn = _planar_experts(E, H, F, salt=2)
    n = T * k
    sizes = {"gu": n * 2 * F * 4, "hq": _q8_bytes(n, F), "y": n * H * 4, "xq": _q8_bytes(T, H)}
    bufs = {key: _guarded(nb) for key, nb in sizes.items()}
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mmvq.expert_ffn(mmvq.TYPE_Q4_K_PLANAR, W_gu, W_dn, E, H, F, x, dev(topk),
                          gu=_front(bufs["gu"], sizes["gu"], (n, 2 * F), torch.float32),
                          hq=_front(bufs["hq"], sizes["hq"], (n, F // 32, mmvq.Q8_1_BYTES)),
                          y=_front(bufs["y"], sizes["y"], (n, H), torch.float32),
                          xq=_front(bufs["xq"], sizes["xq"], (T, H // 32, mmvq.Q8_1_BYTES)),
                          status=status)
    n_valid = int(host(out["offsets"])[E])
    assert n_valid == n - 2 and host(status)[0] == mmvq.ERR_ROUTING
    per_row = {"gu": 2 * F * 4, "hq": (F // 32) * mmvq.Q8_1_BYTES, "y": H * 4}
    for key in ("gu", "hq", "y"):
        _guard_intact(bufs[key], n_valid * per_row[key])  # rows >= n_valid and the guard
    _guard_intact(bufs["xq"], sizes["xq"])
    assert mmvq.read_device_fault() == 0
