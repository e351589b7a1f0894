"""CPU oracle for the MMVQ path: a thin ctypes wrapper over ``mmvq_oracle.cpp``.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
path (``block_quantized_matvec_gb300``) never imports it, and the oracle
never imports the product path.  Inputs come from
``block_quantized_matvec_gb300.synth`` (random draws only).

Every function is pinned in ``tests/test_oracle_*.py`` against something
other than itself; see the header of ``mmvq_oracle.cpp``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mmvq_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

TYPE_Q4_K = 12
TYPE_Q5_K = 13
TYPE_Q6_K = 14
TYPE_Q6_K_PLANAR = 1014
TYPE_Q4_K_PLANAR = 1012
TYPE_Q5_K_PLANAR = 1013

Q81_BYTES = 36
BLOCK_BYTES = {TYPE_Q4_K: 144, TYPE_Q5_K: 176, TYPE_Q6_K: 210}


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (-O2, no FMA contraction), single-threaded."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            lib.orc_f32_to_f16_array.argtypes = [P, P, I64]
            lib.orc_f16_to_f32_array.argtypes = [P, P, I64]
            lib.orc_quantize_q8_1.argtypes = [P, I, I, I64, P]
            lib.orc_decode_q6_k.argtypes = [P, P, P, P]
            lib.orc_decode_q4_k.argtypes = [P, P, P, P, P, P]
            lib.orc_planar_bytes.argtypes = [I64, I]
            lib.orc_planar_bytes.restype = I64
            lib.orc_planar_bytes_q4.argtypes = [I64, I]
            lib.orc_planar_bytes_q4.restype = I64
            lib.orc_planar_bytes_q5.argtypes = [I64, I]
            lib.orc_planar_bytes_q5.restype = I64
            lib.orc_repack_planar_q5.argtypes = [P, I64, I, P]
            lib.orc_unpack_planar_q5.argtypes = [P, I64, I, P]
            lib.orc_decode_q5_k.argtypes = [P, P, P, P, P, P]
            lib.orc_repack_planar_q4.argtypes = [P, I64, I, P]
            lib.orc_unpack_planar_q4.argtypes = [P, I64, I, P]
            lib.orc_repack_planar.argtypes = [P, I64, I, P]
            lib.orc_unpack_planar.argtypes = [P, I64, I, P]
            lib.orc_gather_planar_rows.argtypes = [P, I64, I, P, I, P]
            lib.orc_gemv.argtypes = [I, P, I64, I, P, I, P, P]
            lib.orc_block_sums.argtypes = [I, P, I64, I, P, I, P]
            lib.orc_route_groups.argtypes = [P, I, I, I, P, P, P, P]
            lib.orc_grouped.argtypes = [I, P, I, I64, I, P, P, I, P, P, P, P]
            lib.orc_silu_mul_quantize.argtypes = [P, I, I, P, P]
            lib.orc_rmsnorm_quantize_q8_1.argtypes = [P, P, ctypes.c_float, I, I, I64, P, P]
            _lib = lib
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().orc_f32_to_f16_array(_p(x), _p(out), x.size)
    return out


def f16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    _load().orc_f16_to_f32_array(_p(h), _p(out), h.size)
    return out


def quantize_q8_1(x: np.ndarray, K: int | None = None) -> np.ndarray:
    """x [ncols, ldx] fp32 -> Q8_1 bytes [ncols, K/32, 36]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    ncols, ldx = x.shape
    K = ldx if K is None else K
    out = np.empty((ncols, K // 32, Q81_BYTES), dtype=np.uint8)
    _check(_load().orc_quantize_q8_1(_p(x), K, ncols, ldx, _p(out)), "quantize_q8_1")
    return out


def decode_q6_k(block: np.ndarray):
    b = np.ascontiguousarray(block, dtype=np.uint8)
    assert b.size == 210
    q = np.empty(256, np.uint8)
    sc = np.empty(16, np.int8)
    d = np.empty(1, np.float32)
    _load().orc_decode_q6_k(_p(b), _p(q), _p(sc), _p(d))
    return q, sc, float(d[0])


def decode_q5_k(block: np.ndarray):
    b = np.ascontiguousarray(block, dtype=np.uint8)
    assert b.size == 176
    q = np.empty(256, np.uint8)
    sc = np.empty(8, np.uint8)
    m = np.empty(8, np.uint8)
    d = np.empty(1, np.float32)
    dmin = np.empty(1, np.float32)
    _load().orc_decode_q5_k(_p(b), _p(q), _p(sc), _p(m), _p(d), _p(dmin))
    return q, sc, m, float(d[0]), float(dmin[0])


def decode_q4_k(block: np.ndarray):
    b = np.ascontiguousarray(block, dtype=np.uint8)
    assert b.size == 144
    q = np.empty(256, np.uint8)
    sc = np.empty(8, np.uint8)
    m = np.empty(8, np.uint8)
    d = np.empty(1, np.float32)
    dmin = np.empty(1, np.float32)
    _load().orc_decode_q4_k(_p(b), _p(q), _p(sc), _p(m), _p(d), _p(dmin))
    return q, sc, m, float(d[0]), float(dmin[0])


def _planar_fns(type_: int):
    lib = _load()
    if type_ == TYPE_Q4_K:
        return lib.orc_planar_bytes_q4, lib.orc_repack_planar_q4, lib.orc_unpack_planar_q4
    if type_ == TYPE_Q5_K:
        return lib.orc_planar_bytes_q5, lib.orc_repack_planar_q5, lib.orc_unpack_planar_q5
    return lib.orc_planar_bytes, lib.orc_repack_planar, lib.orc_unpack_planar


def planar_bytes(rows: int, K: int, type_: int = TYPE_Q6_K) -> int:
    return int(_planar_fns(type_)[0](rows, K))


def repack_planar(W: np.ndarray, rows: int, K: int, type_: int = TYPE_Q6_K) -> np.ndarray:
    """GGUF blocks of type_ (Q6_K, Q5_K or Q4_K) -> planar tiles."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    out = np.empty(planar_bytes(rows, K, type_), dtype=np.uint8)
    _check(_planar_fns(type_)[1](_p(W), rows, K, _p(out)), "repack_planar")
    return out


def unpack_planar(P: np.ndarray, rows: int, K: int, type_: int = TYPE_Q6_K) -> np.ndarray:
    P = np.ascontiguousarray(P, dtype=np.uint8)
    out = np.empty((rows, K // 256, BLOCK_BYTES[type_]), dtype=np.uint8)
    _check(_planar_fns(type_)[2](_p(P), rows, K, _p(out)), "unpack_planar")
    return out


def gather_planar_rows(P: np.ndarray, rows: int, K: int, row_ids: np.ndarray) -> np.ndarray:
    P = np.ascontiguousarray(P, dtype=np.uint8)
    ids = np.ascontiguousarray(row_ids, dtype=np.int32)
    out = np.empty(planar_bytes(ids.size, K), dtype=np.uint8)
    _check(_load().orc_gather_planar_rows(_p(P), rows, K, _p(ids), ids.size, _p(out)),
           "gather_planar_rows")
    return out


def gemv(type_: int, W: np.ndarray, rows: int, K: int, xq: np.ndarray, ncols: int,
         with_bound: bool = False):
    """y [ncols, rows] fp32 (and the bound sum|t_b| when asked)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    y = np.empty((ncols, rows), dtype=np.float32)
    bnd = np.empty((ncols, rows), dtype=np.float32) if with_bound else None
    _check(_load().orc_gemv(type_, _p(W), rows, K, _p(xq), ncols, _p(y), _p(bnd)), "gemv")
    return (y, bnd) if with_bound else y


def block_sums(type_: int, W: np.ndarray, rows: int, K: int, xq: np.ndarray, ncols: int):
    """Per-32-block integer sums, [ncols, rows, K/32] int32."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    s = np.empty((ncols, rows, K // 32), dtype=np.int32)
    _check(_load().orc_block_sums(type_, _p(W), rows, K, _p(xq), ncols, _p(s)), "block_sums")
    return s


def route_groups(topk: np.ndarray, n_experts: int):
    """-> (expert_ids [E], offsets [E+1], act_index [T*k], slot_of [T*k])."""
    topk = np.ascontiguousarray(topk, dtype=np.int32)
    T, k = topk.shape
    eids = np.empty(n_experts, np.int32)
    offs = np.empty(n_experts + 1, np.int32)
    act = np.empty(T * k, np.int32)
    slot = np.empty(T * k, np.int32)
    _check(_load().orc_route_groups(_p(topk), T, k, n_experts, _p(eids), _p(offs), _p(act),
                                    _p(slot)), "route_groups")
    return eids, offs, act, slot


def grouped(type_: int, W: np.ndarray, n_experts: int, rows: int, K: int,
            expert_ids: np.ndarray, offsets: np.ndarray, act_index: np.ndarray | None,
            xq: np.ndarray, with_bound: bool = False):
    """y [n_pos, rows] for the positions covered by the groups."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    eids = np.ascontiguousarray(expert_ids, dtype=np.int32)
    offs = np.ascontiguousarray(offsets, dtype=np.int32)
    act = None if act_index is None else np.ascontiguousarray(act_index, dtype=np.int32)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    n_groups = eids.size
    n_pos = int(offs[n_groups])
    y = np.zeros((n_pos, rows), dtype=np.float32)
    bnd = np.zeros((n_pos, rows), dtype=np.float32) if with_bound else None
    _check(_load().orc_grouped(type_, _p(W), n_experts, rows, K, _p(eids), _p(offs), n_groups,
                               _p(act), _p(xq), _p(y), _p(bnd)), "grouped")
    return (y, bnd) if with_bound else y


def silu_mul_quantize(gu: np.ndarray, F: int):
    """gu [n, 2F] -> (xq [n, F/32, 36], h [n, F])."""
    gu = np.ascontiguousarray(gu, dtype=np.float32)
    n = gu.shape[0]
    xq = np.empty((n, F // 32, Q81_BYTES), dtype=np.uint8)
    h = np.empty((n, F), dtype=np.float32)
    _check(_load().orc_silu_mul_quantize(_p(gu), F, n, _p(xq), _p(h)), "silu_mul_quantize")
    return xq, h


def rmsnorm_quantize_q8_1(x: np.ndarray, w: np.ndarray, eps: float):
    """x [ncols, K], w [K] -> (xq [ncols, K/32, 36], y [ncols, K]) of RMSNorm(x) * w."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    w = np.ascontiguousarray(w, dtype=np.float32)
    ncols, K = x.shape
    xq = np.empty((ncols, K // 32, Q81_BYTES), dtype=np.uint8)
    y = np.empty((ncols, K), dtype=np.float32)
    _check(_load().orc_rmsnorm_quantize_q8_1(_p(x), _p(w), eps, K, ncols, K, _p(xq), _p(y)),
           "rmsnorm_quantize_q8_1")
    return xq, y
