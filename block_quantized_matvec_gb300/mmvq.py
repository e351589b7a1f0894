"""Thin Python binding of libmmvq.so (include/mmvq.h).

Argument marshalling only: every step of the path runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors; each call runs on the current
torch stream (or the one passed in).  If the library is missing the first
call raises; there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmmvq.so")

TYPE_Q4_K = 12
TYPE_Q6_K = 14
TYPE_Q6_K_PLANAR = 1014
TYPE_Q4_K_PLANAR = 1012
TYPE_Q5_K = 13
TYPE_Q5_K_PLANAR = 1013
BLOCK_BYTES = {TYPE_Q4_K: 144, TYPE_Q6_K: 210, TYPE_Q6_K_PLANAR: 210, TYPE_Q4_K_PLANAR: 144,
               TYPE_Q5_K: 176, TYPE_Q5_K_PLANAR: 176}
Q8_1_BYTES = 36
MAX_COLS = 8

OK = 0
FLAG_XQ_STABLE = 1
FLAG_TENSOR_CORE = 2
ERR_TYPE, ERR_SHAPE, ERR_NCOLS, ERR_NULL, ERR_ALIGN, ERR_ROUTING, ERR_CUDA = -1, -2, -3, -4, -5, -6, -7
ERR_SCRATCH = -8
NOALLOC_SCRATCH_BYTES = 2 << 20  # MMVQ_NOALLOC_SCRATCH_BYTES

# name -> (restype, argtypes); mirrors include/mmvq.h
_P, _I, _I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
SIGNATURES = {
    "mmvq_version": (_I, []),
    "mmvq_strerror": (ctypes.c_char_p, [_I]),
    "mmvq_quantize_q8_1": (_I, [_P, _I, _I, _I64, _P, _P]),
    "mmvq_gemv": (_I, [_I, _P, _I64, _I, _P, _I, _P, _P]),
    "mmvq_gemv_ex": (_I, [_I, _P, _I64, _I, _P, _I, _P, ctypes.c_uint, _P]),
    "mmvq_debug_block_sums": (_I, [_I, _P, _I64, _I, _P, _I, _P, _P, _P]),
    "mmvq_debug_block_sums_ex": (_I, [_I, _P, _I64, _I, _P, _I, _P, _P, ctypes.c_uint, _P]),
    "mmvq_gemv_f32": (_I, [_I, _P, _I64, _I, _P, _I64, _I, _P, _P, ctypes.c_uint, _P]),
    "mmvq_gemv_f32_fused": (_I, [_I, _I64, _I, _I, _P]),
    "mmvq_grouped": (_I, [_I, _P, _I, _I64, _I, _P, _P, _I, _P, _P, _I, _P, _P, _P]),
    "mmvq_route_groups": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "mmvq_quantize_route_groups": (_I, [_P, _I, _I, _I64, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "mmvq_silu_mul_quantize_q8_1": (_I, [_P, _I, _I, _P, _P, _P]),
    "mmvq_planar_bytes": (_I64, [_I, _I64, _I]),
    "mmvq_repack_planar": (_I, [_I, _P, _I64, _I, _P, _P]),
    "mmvq_gather_planar_rows": (_I, [_P, _I64, _I, _P, _I, _P, _P, _P]),
    "mmvq_read_device_fault": (_I, [_P, _P]),
    "mmvq_selftest_wait_timeout": (_I, [ctypes.c_uint, _P]),
    "mmvq_rmsnorm_quantize_q8_1": (_I, [_P, _P, ctypes.c_float, _I, _I, _I64, _P, _P, _P]),
    "mmvq_launch_shape": (_I, [_I, _I64, _I, _I, _P]),
    "mmvq_launch_shape_ex": (_I, [_I, _I64, _I, _I, _P, _I]),
    "mmvq_expert_ffn": (_I, [_I, _P, _P, _I, _I, _I, _P, _I64, _I, _P, _I, _P, _P, _P, _P, _P,
                             _P, _P, _P, _P, _P, _P]),
    "mmvq_expert_ffn_noalloc": (_I, [_I, _P, _P, _I, _I, _I, _P, _I64, _I, _P, _I, _P, _P, _P,
                                     _P, _P, _P, _P]),
    "mmvq_expert_ffn_shape": (_I, [_I, _I, _I, _I, _I, _I, _P]),
    "mmvq_selftest_grid_barrier_timeout": (_I, [_P, ctypes.c_uint, _P]),
}


class MMVQError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} (code {code})")


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C-ABI library.  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m block_quantized_matvec_gb300.build` (nvcc, sm_103a)")
            l = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(l, name)
                f.restype = res
                f.argtypes = args
            _lib = l
    return _lib


def strerror(code: int) -> str:
    return lib().mmvq_strerror(code).decode()


def _check(rc: int, what: str):
    if rc != OK:
        raise MMVQError(rc, what)


def _ptr(t):
    return None if t is None else t.data_ptr()


# The current stream's handle without building a torch Stream object (about
# 3 us a call otherwise); torch's own raw accessor where it exists.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _dev(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ------------------------------------------------------------- entry points --

def quantize_q8_1(x: torch.Tensor, K: int | None = None, out: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """fp32 x [ncols, ldx] -> Q8_1 bytes [ncols, K/32, 36] (uint8)."""
    _dev(x, "x")
    if x.dtype != torch.float32:
        raise ValueError("x must be float32")
    x2 = x if x.dim() == 2 else x.view(1, -1)
    ncols, ldx = x2.shape
    K = ldx if K is None else K
    if out is None:
        out = torch.empty((ncols, K // 32, Q8_1_BYTES), dtype=torch.uint8, device=x.device)
    _check(lib().mmvq_quantize_q8_1(_ptr(x2), K, ncols, ldx, _ptr(out), _stream(stream)),
           "mmvq_quantize_q8_1")
    return out


def gemv(type_: int, W: torch.Tensor, rows: int, K: int, xq: torch.Tensor, ncols: int,
         out: torch.Tensor | None = None, stream=None, flags: int = 0) -> torch.Tensor:
    """y [ncols, rows] fp32 = W (rows x K, block type ``type_``) times ncols Q8_1 columns.
    flags: FLAG_XQ_STABLE when no still-running kernel writes xq, FLAG_TENSOR_CORE for
    the tensor-core consumer (mmvq_gemv_ex)."""
    _dev(W, "W")
    _dev(xq, "xq")
    if out is None:
        out = torch.empty((ncols, rows), dtype=torch.float32, device=W.device)
    if flags:
        _check(lib().mmvq_gemv_ex(type_, _ptr(W), rows, K, _ptr(xq), ncols, _ptr(out), flags,
                                  _stream(stream)), "mmvq_gemv_ex")
    else:
        _check(lib().mmvq_gemv(type_, _ptr(W), rows, K, _ptr(xq), ncols, _ptr(out),
                               _stream(stream)), "mmvq_gemv")
    return out


def gemv_f32(type_: int, W: torch.Tensor, rows: int, K: int, x: torch.Tensor, ncols: int | None = None,
             xq: torch.Tensor | None = None, out: torch.Tensor | None = None, flags: int = 0,
             stream=None):
    """fp32 x [ncols, ldx] -> (y [ncols, rows], xq [ncols, K/32, 36]): Q8_1 of x and the
    product, in one launch where the columns are small enough."""
    _dev(W, "W")
    if x.dim() == 1:
        x = x.view(1, -1)
    if not x.is_cuda or x.dtype != torch.float32 or x.stride(1) != 1:
        raise ValueError("x must be a CUDA float32 tensor with unit column stride")
    ncols = x.shape[0] if ncols is None else ncols
    if xq is None:
        xq = torch.empty((ncols, K // 32, Q8_1_BYTES), dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty((ncols, rows), dtype=torch.float32, device=x.device)
    _check(lib().mmvq_gemv_f32(type_, _ptr(W), rows, K, _ptr(x), x.stride(0), ncols, _ptr(xq),
                               _ptr(out), flags, _stream(stream)), "mmvq_gemv_f32")
    return out, xq


def gemv_f32_fused(type_: int, rows: int, K: int, ncols: int) -> bool:
    """Whether gemv_f32 runs this call as one launch (host-only)."""
    f = ctypes.c_int32(0)
    _check(lib().mmvq_gemv_f32_fused(type_, rows, K, ncols, ctypes.byref(f)), "mmvq_gemv_f32_fused")
    return bool(f.value)


def debug_block_sums(type_: int, W: torch.Tensor, rows: int, K: int, xq: torch.Tensor, ncols: int,
                     stream=None, flags: int = 0):
    """(sumi [ncols, rows, K/32] int32, y [ncols, rows]) from the gemv kernel itself."""
    _dev(W, "W")
    _dev(xq, "xq")
    sumi = torch.empty((ncols, rows, K // 32), dtype=torch.int32, device=W.device)
    y = torch.empty((ncols, rows), dtype=torch.float32, device=W.device)
    if flags:
        _check(lib().mmvq_debug_block_sums_ex(type_, _ptr(W), rows, K, _ptr(xq), ncols,
                                              _ptr(sumi), _ptr(y), flags, _stream(stream)),
               "mmvq_debug_block_sums_ex")
    else:
        _check(lib().mmvq_debug_block_sums(type_, _ptr(W), rows, K, _ptr(xq), ncols, _ptr(sumi),
                                           _ptr(y), _stream(stream)), "mmvq_debug_block_sums")
    return sumi, y


def grouped(type_: int, W_experts: torch.Tensor, n_experts: int, rows: int, K: int,
            expert_ids: torch.Tensor, offsets: torch.Tensor, act_index: torch.Tensor | None,
            xq: torch.Tensor, n_xq_cols: int, n_positions: int, out: torch.Tensor | None = None,
            status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y [n_positions, rows]: row p = expert of p's group times xq column act_index[p]."""
    for t, n in ((W_experts, "W_experts"), (expert_ids, "expert_ids"), (offsets, "offsets"),
                 (xq, "xq")):
        _dev(t, n)
    if out is None:
        out = torch.empty((max(n_positions, 1), rows), dtype=torch.float32, device=xq.device)
    _check(lib().mmvq_grouped(type_, _ptr(W_experts), n_experts, rows, K, _ptr(expert_ids),
                              _ptr(offsets), expert_ids.numel(), _ptr(act_index), _ptr(xq),
                              n_xq_cols, _ptr(out), _ptr(status), _stream(stream)), "mmvq_grouped")
    return out


def quantize_route_groups(x: torch.Tensor, topk: torch.Tensor, n_experts: int,
                          xq: torch.Tensor | None = None, stream=None):
    """One launch: Q8_1 of x [ncols, K] and the per-expert lists of topk [T, k]
    -> (xq, expert_ids, offsets, act_index, slot_of, status)."""
    _dev(x, "x")
    _dev(topk, "topk")
    if x.dim() == 1:
        x = x.view(1, -1)
    ncols, K = x.shape
    T, k = topk.shape
    dev = x.device
    if xq is None:
        xq = torch.empty((ncols, K // 32, Q8_1_BYTES), dtype=torch.uint8, device=dev)
    eids = torch.empty(n_experts, dtype=torch.int32, device=dev)
    offs = torch.empty(n_experts + 1, dtype=torch.int32, device=dev)
    act = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    slot = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    _check(lib().mmvq_quantize_route_groups(_ptr(x), K, ncols, K, _ptr(xq),
                                            _ptr(topk) if T else None, T, k, n_experts,
                                            _ptr(eids), _ptr(offs), _ptr(act), _ptr(slot),
                                            _ptr(status), _stream(stream)),
           "mmvq_quantize_route_groups")
    return xq, eids, offs, act, slot, status


def expert_ffn_workspace(device) -> torch.Tensor:
    """A zeroed grid-barrier word for expert_ffn (one per concurrently running launch)."""
    return torch.zeros(4, dtype=torch.int32, device=device)


def expert_ffn(type_: int, W_gate_up: torch.Tensor, W_down: torch.Tensor, n_experts: int,
               H: int, F: int, x: torch.Tensor, topk: torch.Tensor, *,
               gu: torch.Tensor | None = None, hq: torch.Tensor | None = None,
               y: torch.Tensor | None = None, lists: bool = True, xq: torch.Tensor | None = None,
               status: torch.Tensor | None = None, sync: torch.Tensor | None = None,
               stream=None) -> dict:
    """The routed-expert FFN of one MoE layer in one launch: x [T, H] fp32 (T <= 8),
    topk [T, k] int32, planar experts W_gate_up (2F x H each) and W_down (H x F
    each).  Returns a dict with xq [T, H/32, 36], gu [T*k, 2F], hq [T*k, F/32, 36],
    y [T*k, H] and, with lists=True, expert_ids, offsets, act_index, slot_of."""
    for t, n in ((W_gate_up, "W_gate_up"), (W_down, "W_down"), (x, "x"), (topk, "topk")):
        _dev(t, n)
    if x.dim() == 1:
        x = x.view(1, -1)
    T, k = topk.shape
    n = T * k
    dev = x.device
    if gu is None:
        gu = torch.empty((n, 2 * F), dtype=torch.float32, device=dev)
    if hq is None:
        hq = torch.empty((n, F // 32, Q8_1_BYTES), dtype=torch.uint8, device=dev)
    if y is None:
        y = torch.empty((n, H), dtype=torch.float32, device=dev)
    out = {"gu": gu, "hq": hq, "y": y}
    if lists:
        out.update(expert_ids=torch.empty(n_experts, dtype=torch.int32, device=dev),
                   offsets=torch.empty(n_experts + 1, dtype=torch.int32, device=dev),
                   act_index=torch.empty(max(n, 1), dtype=torch.int32, device=dev),
                   slot_of=torch.empty(max(n, 1), dtype=torch.int32, device=dev))
    if xq is None:
        xq = torch.empty((T, H // 32, Q8_1_BYTES), dtype=torch.uint8, device=dev)
    out["xq"] = xq
    if status is not None:
        out["status"] = status
    if sync is None:
        sync = expert_ffn_workspace(dev)
    _check(lib().mmvq_expert_ffn(type_, _ptr(W_gate_up), _ptr(W_down), n_experts, H, F, _ptr(x),
                                 x.stride(0), T, _ptr(topk), k, _ptr(gu), _ptr(hq), _ptr(y),
                                 _ptr(out.get("expert_ids")), _ptr(out.get("offsets")),
                                 _ptr(out.get("act_index")), _ptr(out.get("slot_of")),
                                 _ptr(xq), _ptr(status), _ptr(sync), _stream(stream)),
           "mmvq_expert_ffn")
    return out


def expert_ffn_noalloc(type_: int, W_gate_up: torch.Tensor, W_down: torch.Tensor,
                       n_experts: int, H: int, F: int, x: torch.Tensor, topk: torch.Tensor, *,
                       y: torch.Tensor | None = None, lists: bool = True,
                       status: torch.Tensor | None = None, stream=None) -> dict:
    """expert_ffn with its intermediates (xq, gu, hq, barrier word) in the library's
    fixed device array: for callers that cannot allocate.  Pass y (and the list
    outputs) preallocated to allocate nothing here either.  Returns y and, with
    lists=True, expert_ids, offsets, act_index, slot_of."""
    for t, n in ((W_gate_up, "W_gate_up"), (W_down, "W_down"), (x, "x"), (topk, "topk")):
        _dev(t, n)
    if x.dim() == 1:
        x = x.view(1, -1)
    T, k = topk.shape
    n = T * k
    dev = x.device
    if y is None:
        y = torch.empty((n, H), dtype=torch.float32, device=dev)
    out = {"y": y}
    if lists:
        out.update(expert_ids=torch.empty(n_experts, dtype=torch.int32, device=dev),
                   offsets=torch.empty(n_experts + 1, dtype=torch.int32, device=dev),
                   act_index=torch.empty(max(n, 1), dtype=torch.int32, device=dev),
                   slot_of=torch.empty(max(n, 1), dtype=torch.int32, device=dev))
    if status is not None:
        out["status"] = status
    _check(lib().mmvq_expert_ffn_noalloc(type_, _ptr(W_gate_up), _ptr(W_down), n_experts, H, F,
                                         _ptr(x), x.stride(0), T, _ptr(topk), k, _ptr(y),
                                         _ptr(out.get("expert_ids")), _ptr(out.get("offsets")),
                                         _ptr(out.get("act_index")), _ptr(out.get("slot_of")),
                                         _ptr(status), _stream(stream)),
           "mmvq_expert_ffn_noalloc")
    return out


def expert_ffn_shape(type_: int, n_experts: int, H: int, F: int, T: int, k: int) -> dict:
    """The launch shape mmvq_expert_ffn picks (host-only)."""
    info = (ctypes.c_int32 * 8)()
    _check(lib().mmvq_expert_ffn_shape(type_, n_experts, H, F, T, k, info),
           "mmvq_expert_ffn_shape")
    keys = ("grid", "threads", "smem", "stages", "G_gate_up", "P_gate_up", "G_down", "P_down")
    return dict(zip(keys, list(info)))


def selftest_grid_barrier_timeout(sync: torch.Tensor, limit_us: int = 2000, stream=None) -> None:
    """Run the expert FFN's grid barrier to expiry on its own word (sets bit 2 of the fault word)."""
    _dev(sync, "sync")
    _check(lib().mmvq_selftest_grid_barrier_timeout(_ptr(sync), limit_us, _stream(stream)),
           "mmvq_selftest_grid_barrier_timeout")


def route_groups(topk: torch.Tensor, n_experts: int, stream=None):
    """topk [T, k] int32 -> (expert_ids [E], offsets [E+1], act_index [T*k], slot_of [T*k], status)."""
    _dev(topk, "topk")
    T, k = topk.shape
    dev = topk.device
    eids = torch.empty(n_experts, dtype=torch.int32, device=dev)
    offs = torch.empty(n_experts + 1, dtype=torch.int32, device=dev)
    act = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    slot = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    _check(lib().mmvq_route_groups(_ptr(topk) if T else None, T, k, n_experts, _ptr(eids),
                                   _ptr(offs), _ptr(act), _ptr(slot), _ptr(status),
                                   _stream(stream)), "mmvq_route_groups")
    return eids, offs, act, slot, status


def silu_mul_quantize_q8_1(gu: torch.Tensor, F: int, out: torch.Tensor | None = None,
                           h_out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """gu [n, 2F] = [gate | up] -> Q8_1 of silu(gate)*up, [n, F/32, 36]."""
    _dev(gu, "gu")
    n = gu.shape[0]
    if out is None:
        out = torch.empty((n, F // 32, Q8_1_BYTES), dtype=torch.uint8, device=gu.device)
    _check(lib().mmvq_silu_mul_quantize_q8_1(_ptr(gu), F, n, _ptr(out), _ptr(h_out),
                                             _stream(stream)), "mmvq_silu_mul_quantize_q8_1")
    return out


def launch_shape(type_: int, rows: int, K: int, ncols: int) -> dict:
    """The launch shape mmvq_gemv picks (host-only query)."""
    info = (ctypes.c_int32 * 7)()
    _check(lib().mmvq_launch_shape_ex(type_, rows, K, ncols, info, 7), "mmvq_launch_shape_ex")
    keys = (["grid", "threads", "smem", "G", "P", "stages", "cluster"]
            if type_ in (TYPE_Q6_K_PLANAR, TYPE_Q4_K_PLANAR, TYPE_Q5_K_PLANAR)
            else ["grid", "threads", "smem", "WR", "WK", "unused", "cluster"])
    return dict(zip(keys, list(info)))


def read_device_fault(stream=None) -> int:
    """Synchronise the stream, return and clear the device fault word (0 = none)."""
    v = ctypes.c_int(0)
    _check(lib().mmvq_read_device_fault(ctypes.byref(v), _stream(stream)), "mmvq_read_device_fault")
    return v.value


def rmsnorm_quantize_q8_1(x: torch.Tensor, w: torch.Tensor, eps: float,
                          out: torch.Tensor | None = None, y_out: torch.Tensor | None = None,
                          stream=None) -> torch.Tensor:
    """x [ncols, K] fp32 (rows may be strided), w [K] fp32 -> Q8_1 of RMSNorm(x) * w,
    [ncols, K/32, 36]."""
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    _dev(w, "w")
    if x.dim() == 1:
        x = x.view(1, -1)
    ncols, K = x.shape
    if x.dtype != torch.float32 or w.dtype != torch.float32 or x.stride(1) != 1 or \
            not w.is_contiguous() or w.numel() != K:
        raise ValueError("x [ncols, K] with unit inner stride and w [K], both float32")
    if out is None:
        out = torch.empty((ncols, K // 32, Q8_1_BYTES), dtype=torch.uint8, device=x.device)
    _check(lib().mmvq_rmsnorm_quantize_q8_1(_ptr(x), _ptr(w), eps, K, ncols, x.stride(0),
                                            _ptr(out), _ptr(y_out), _stream(stream)),
           "mmvq_rmsnorm_quantize_q8_1")
    return out


def selftest_wait_timeout(limit_us: int = 2000, stream=None) -> None:
    """Run one bounded barrier wait to expiry (sets bit 1 of the fault word)."""
    _check(lib().mmvq_selftest_wait_timeout(limit_us, _stream(stream)),
           "mmvq_selftest_wait_timeout")


def planar_bytes(rows: int, K: int, type_: int = TYPE_Q6_K) -> int:
    n = lib().mmvq_planar_bytes(type_, rows, K)
    if n < 0:
        raise MMVQError(ERR_SHAPE, "mmvq_planar_bytes")
    return int(n)


def repack_planar(W_gguf: torch.Tensor, rows: int, K: int, out: torch.Tensor | None = None,
                  stream=None, type_: int = TYPE_Q6_K) -> torch.Tensor:
    """GGUF Q6_K (or Q4_K) bytes -> planar tiles (uint8, planar_bytes(rows, K, type_))."""
    _dev(W_gguf, "W_gguf")
    if out is None:
        out = torch.empty(planar_bytes(rows, K, type_), dtype=torch.uint8, device=W_gguf.device)
    _check(lib().mmvq_repack_planar(type_, _ptr(W_gguf), rows, K, _ptr(out), _stream(stream)),
           "mmvq_repack_planar")
    return out


def gather_planar_rows(W_planar: torch.Tensor, rows: int, K: int, row_ids: torch.Tensor,
                       out: torch.Tensor | None = None, stream=None):
    """Planar matrix of len(row_ids) rows, row k = row row_ids[k] of W_planar; returns (out, status)."""
    _dev(W_planar, "W_planar")
    _dev(row_ids, "row_ids")
    n = row_ids.numel()
    if out is None:
        out = torch.empty(planar_bytes(n, K), dtype=torch.uint8, device=W_planar.device)
    status = torch.zeros(1, dtype=torch.int32, device=W_planar.device)
    _check(lib().mmvq_gather_planar_rows(_ptr(W_planar), rows, K, _ptr(row_ids), n, _ptr(out),
                                         _ptr(status), _stream(stream)), "mmvq_gather_planar_rows")
    return out, status
