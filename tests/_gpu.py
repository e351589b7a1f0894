"""Helpers for the GPU parity tests: device transfer, the output bound and
an FNV-1a hash of float bits (the pages' mmvq_bench checksum, PR #2207)."""
import numpy as np
import torch


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    torch.cuda.synchronize()
    return t.cpu().numpy()


def assert_within_bound(y_gpu: np.ndarray, y_ref: np.ndarray, bound: np.ndarray, what=""):
    """|y_gpu - y_ref| <= 1e-5 * sum|block terms| + 1e-6, element by element.
    Non-finite values (an fp16 Q8_1 field that overflowed) must sit at the
    same places with the same value class on both sides."""
    y_gpu = np.asarray(y_gpu)
    y_ref = np.asarray(y_ref)
    fin_g, fin_r = np.isfinite(y_gpu), np.isfinite(y_ref)
    assert np.array_equal(fin_g, fin_r), f"{what}: non-finite outputs differ in place"
    if not fin_g.all():
        assert np.array_equal(np.isnan(y_gpu), np.isnan(y_ref)), f"{what}: NaN places differ"
        inf = np.isinf(y_ref)
        assert np.array_equal(y_gpu[inf], y_ref[inf]), f"{what}: infinities differ"
        y_gpu, y_ref, bound = y_gpu[fin_r], y_ref[fin_r], np.asarray(bound)[fin_r]
    err = np.abs(y_gpu.astype(np.float64) - y_ref.astype(np.float64))
    lim = 1e-5 * bound.astype(np.float64) + 1e-6
    bad = err > lim
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside the bound; worst "
                           f"{(err - lim).max():.3g} at {np.argwhere(bad)[0]}")


def fnv1a(a: np.ndarray) -> int:
    h = np.uint64(0xcbf29ce484222325)
    prime = np.uint64(0x100000001b3)
    with np.errstate(over="ignore"):
        for b in np.ascontiguousarray(a).reshape(-1).view(np.uint8):
            h = (h ^ np.uint64(b)) * prime
    return int(h)
