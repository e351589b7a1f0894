"""The C-ABI library builds, loads without a GPU, exports exactly the entry
points include/mmvq.h declares, and rejects bad arguments on the host
before any CUDA call (so these run on a machine with no GPU)."""
import ctypes
import os
import re

import pytest

from block_quantized_matvec_gb300 import build, mmvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return mmvq.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "mmvq.h")).read()
    return set(re.findall(r"MMVQ_API\s+[\w\s\*]+?\b(mmvq_\w+)\s*\(", text))


def test_header_declares_the_binding_signatures():
    assert _declared() == set(mmvq.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {mmvq.LIB_PATH}").read().split("\n")
    exported = {l.split()[-1] for l in out if l.strip() and l.split()[-1].startswith("mmvq_")}
    assert exported == _declared()


def test_version_and_strerror(lib):
    assert lib.mmvq_version() == 10000
    for code in range(0, -9, -1):
        assert mmvq.strerror(code) and "unknown" not in mmvq.strerror(code)
    assert "unknown" in mmvq.strerror(-99)


def test_planar_bytes_host_only(lib):
    assert mmvq.planar_bytes(151936, 2560) == 151936 // 16 * 10 * 3360 == 151936 * 10 * 210
    assert mmvq.planar_bytes(17, 256) == 2 * 1 * 3360
    assert mmvq.planar_bytes(17, 512, mmvq.TYPE_Q4_K) == 2 * 2 * 2304
    assert mmvq.planar_bytes(17, 512, mmvq.TYPE_Q5_K) == 2 * 2 * 2816 == 32 * 2 * 176
    assert lib.mmvq_planar_bytes(14, 16, 100) == -1
    assert lib.mmvq_planar_bytes(14, 0, 256) == -1
    assert lib.mmvq_planar_bytes(1014, 16, 256) == -1


A = 0x10000  # an aligned fake device address: never dereferenced, calls fail before CUDA


@pytest.mark.parametrize("args,code", [
    ((99, A, 16, 256, A, 1, A, None), mmvq.ERR_TYPE),
    ((14, A, 16, 255, A, 1, A, None), mmvq.ERR_SHAPE),
    ((14, A, 16, 128, A, 1, A, None), mmvq.ERR_SHAPE),
    ((14, A, 16, 16384 + 256, A, 1, A, None), mmvq.ERR_SHAPE),
    ((14, A, 0, 256, A, 1, A, None), mmvq.ERR_SHAPE),
    ((14, A, 16, 256, A, 0, A, None), mmvq.ERR_NCOLS),
    ((14, A, 16, 256, A, 9, A, None), mmvq.ERR_NCOLS),
    ((14, None, 16, 256, A, 1, A, None), mmvq.ERR_NULL),
    ((14, A, 16, 256, None, 1, A, None), mmvq.ERR_NULL),
    ((14, A, 16, 256, A, 1, None, None), mmvq.ERR_NULL),
    ((14, A + 8, 16, 256, A, 1, A, None), mmvq.ERR_ALIGN),
    ((1014, A, 16, 256, A + 4, 1, A, None), mmvq.ERR_ALIGN),
    ((12, A, 16, 256, A, 1, A + 2, None), mmvq.ERR_ALIGN),
    ((1012, A + 4, 16, 256, A, 1, A, None), mmvq.ERR_ALIGN),
    ((1012, A, 16, 200, A, 1, A, None), mmvq.ERR_SHAPE),
    ((13, A, 16, 256, A, 1, A, None), mmvq.ERR_TYPE),          # Q5_K runs from planar tiles
    ((1013, A + 8, 16, 256, A, 1, A, None), mmvq.ERR_ALIGN),
    ((1013, A, 16, 256, A, 9, A, None), mmvq.ERR_NCOLS),
])
def test_gemv_rejects_bad_arguments_on_host(lib, args, code):
    assert lib.mmvq_gemv(*args) == code


def test_other_entry_points_reject_bad_arguments_on_host(lib):
    L = lib
    assert L.mmvq_quantize_q8_1(A, 48, 1, 48, A, None) == mmvq.ERR_SHAPE
    assert L.mmvq_quantize_q8_1(A, 64, 1, 32, A, None) == mmvq.ERR_SHAPE
    assert L.mmvq_quantize_q8_1(None, 64, 1, 64, A, None) == mmvq.ERR_NULL
    assert L.mmvq_quantize_q8_1(A, 64, 1, 64, A + 4, None) == mmvq.ERR_ALIGN
    assert L.mmvq_quantize_q8_1(A, 64, 0, 64, A, None) == mmvq.ERR_SHAPE
    g = (12, A, 256, 1536, 2560, A, A, 256, A, A, 1, A, None, None)
    assert L.mmvq_grouped(1012, A, 256, 1530, 2560, A, A, 256, A, A, 1, A, None, None) == mmvq.ERR_SHAPE
    assert L.mmvq_grouped(1014, A, 256, 1530, 2560, A, A, 256, A, A, 1, A, None, None) == mmvq.ERR_SHAPE
    assert L.mmvq_grouped(*g[:0], 99, *g[1:]) == mmvq.ERR_TYPE
    assert L.mmvq_grouped(*g[:0], 1013, *g[1:]) == mmvq.ERR_TYPE
    assert L.mmvq_grouped(*g[:7], 0, *g[8:]) == mmvq.ERR_ROUTING
    assert L.mmvq_grouped(*g[:7], 4097, *g[8:]) == mmvq.ERR_ROUTING
    assert L.mmvq_grouped(*g[:4], 2560 + 32, *g[5:]) == mmvq.ERR_SHAPE
    assert L.mmvq_grouped(*g[:5], None, *g[6:]) == mmvq.ERR_NULL
    assert L.mmvq_grouped(*g[:9], A + 4, *g[10:]) == mmvq.ERR_ALIGN
    r = (A, A, 1e-6, 2560, 2, 2560, A, None, None)
    assert L.mmvq_rmsnorm_quantize_q8_1(None, *r[1:]) == mmvq.ERR_NULL
    assert L.mmvq_rmsnorm_quantize_q8_1(*r[:3], 2560 + 16, *r[4:]) == mmvq.ERR_SHAPE
    assert L.mmvq_rmsnorm_quantize_q8_1(*r[:4], 0, *r[5:]) == mmvq.ERR_SHAPE
    assert L.mmvq_rmsnorm_quantize_q8_1(*r[:5], 2048, *r[6:]) == mmvq.ERR_SHAPE   # ldx < K
    assert L.mmvq_rmsnorm_quantize_q8_1(*r[:2], -1.0, *r[3:]) == mmvq.ERR_SHAPE
    assert L.mmvq_rmsnorm_quantize_q8_1(*r[:2], float("nan"), *r[3:]) == mmvq.ERR_SHAPE
    assert L.mmvq_rmsnorm_quantize_q8_1(*r[:6], A + 4, *r[7:]) == mmvq.ERR_ALIGN
    qr = (A, 2560, 1, 2560, A, A, 1, 8, 256, A, A, A, A, None, None)
    assert L.mmvq_quantize_route_groups(*qr[:5], None, *qr[6:]) == mmvq.ERR_NULL      # topk, T > 0
    assert L.mmvq_quantize_route_groups(*qr[:1], 2560 + 16, *qr[2:]) == mmvq.ERR_SHAPE
    assert L.mmvq_quantize_route_groups(*qr[:8], 4097, *qr[9:]) == mmvq.ERR_SHAPE
    assert L.mmvq_quantize_route_groups(*qr[:4], A + 4, *qr[5:]) == mmvq.ERR_ALIGN
    assert L.mmvq_selftest_wait_timeout(0, None) == mmvq.ERR_SHAPE
    assert L.mmvq_selftest_wait_timeout(100001, None) == mmvq.ERR_SHAPE
    assert L.mmvq_route_groups(A, 4, 8, 0, A, A, A, A, None, None) == mmvq.ERR_SHAPE
    assert L.mmvq_route_groups(A, 10000, 8, 256, A, A, A, A, None, None) == mmvq.ERR_SHAPE
    assert L.mmvq_route_groups(None, 4, 8, 256, A, A, A, A, None, None) == mmvq.ERR_NULL
    assert L.mmvq_silu_mul_quantize_q8_1(A, 768 + 16, 1, A, None, None) == mmvq.ERR_SHAPE
    assert L.mmvq_silu_mul_quantize_q8_1(A, 768, 0, A, None, None) == mmvq.ERR_SHAPE
    assert L.mmvq_repack_planar(99, A, 16, 256, A, None) == mmvq.ERR_TYPE
    assert L.mmvq_repack_planar(12, A + 8, 16, 256, A, None) == mmvq.ERR_ALIGN
    assert L.mmvq_repack_planar(13, A + 8, 16, 256, A, None) == mmvq.ERR_ALIGN
    assert L.mmvq_repack_planar(1013, A, 16, 256, A, None) == mmvq.ERR_TYPE
    assert L.mmvq_repack_planar(14, A, 16, 256, A + 8, None) == mmvq.ERR_ALIGN
    assert L.mmvq_gather_planar_rows(A, 16, 256, A, 0, A, None, None) == mmvq.ERR_SHAPE
    assert L.mmvq_gather_planar_rows(A, 16, 256, A, 4, A + 8, None, None) == mmvq.ERR_ALIGN
    # expert FFN: type, pointer, shape, token and expert-count rules, checked on the host
    f = [1012, A, A, 256, 2560, 768, A, 2560, 4, A, 8, A, A, A, None, None, None, None, A,
         None, A, None]

    def ffn(**kw):
        a = list(f)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return L.mmvq_expert_ffn(*a)
    assert ffn(a0=12) == mmvq.ERR_TYPE                       # GGUF experts: use mmvq_grouped
    assert ffn(a0=1013) == mmvq.ERR_TYPE
    assert ffn(a1=None) == mmvq.ERR_NULL
    assert ffn(a20=None) == mmvq.ERR_NULL                    # sync word
    assert ffn(a12=None) == mmvq.ERR_NULL                    # hq
    assert ffn(a4=2560 + 128) == mmvq.ERR_SHAPE              # H % 256
    assert ffn(a5=0) == mmvq.ERR_SHAPE
    assert ffn(a7=2048) == mmvq.ERR_SHAPE                    # ldx < H
    assert ffn(a8=0) == mmvq.ERR_NCOLS and ffn(a8=9) == mmvq.ERR_NCOLS
    assert ffn(a10=0) == mmvq.ERR_SHAPE and ffn(a10=65) == mmvq.ERR_SHAPE   # T*k > 256
    assert ffn(a3=0) == mmvq.ERR_ROUTING and ffn(a3=1025) == mmvq.ERR_ROUTING
    assert ffn(a12=A + 4) == mmvq.ERR_ALIGN                  # hq 16-byte
    assert ffn(a18=A + 4) == mmvq.ERR_ALIGN                  # xq 16-byte
    assert ffn(a18=None) == mmvq.ERR_NULL                    # xq is required
    assert ffn(a2=A + 8) == mmvq.ERR_ALIGN
    info = (ctypes.c_int32 * 8)()
    assert L.mmvq_expert_ffn_shape(12, 256, 2560, 768, 4, 8, info) == mmvq.ERR_TYPE
    assert L.mmvq_expert_ffn_shape(1012, 256, 2560, 768, 9, 8, info) == mmvq.ERR_NCOLS
    assert L.mmvq_expert_ffn_shape(1012, 256, 2560, 768, 4, 8, None) == mmvq.ERR_NULL
    assert L.mmvq_selftest_grid_barrier_timeout(None, 1000, None) == mmvq.ERR_NULL
    assert L.mmvq_selftest_grid_barrier_timeout(A + 2, 1000, None) == mmvq.ERR_ALIGN
    assert L.mmvq_selftest_grid_barrier_timeout(A, 0, None) == mmvq.ERR_SHAPE


def test_flag_words_are_checked_on_host(lib):
    L = lib
    A = 0x10000
    # mmvq_gemv_ex / mmvq_gemv_f32 / mmvq_debug_block_sums_ex: bits other than
    # MMVQ_FLAG_XQ_STABLE (1) and MMVQ_FLAG_TENSOR_CORE (2) are rejected
    assert mmvq.FLAG_XQ_STABLE == 1 and mmvq.FLAG_TENSOR_CORE == 2
    for bad in (4, 8, 1 << 31, 3 | 4):
        assert L.mmvq_gemv_ex(1014, A, 16, 256, A, 1, A, bad, None) == mmvq.ERR_SHAPE
        assert L.mmvq_gemv_f32(1014, A, 16, 256, A, 256, 1, A, A, bad, None) == mmvq.ERR_SHAPE
        assert L.mmvq_debug_block_sums_ex(1014, A, 16, 256, A, 1, A, A, bad, None) == mmvq.ERR_SHAPE
    # the other rules come first, as for mmvq_debug_block_sums
    assert L.mmvq_debug_block_sums_ex(1014, A, 16, 255, A, 1, A, A, 2, None) == mmvq.ERR_SHAPE
    assert L.mmvq_debug_block_sums_ex(1014, A, 16, 256, A, 9, A, A, 2, None) == mmvq.ERR_NCOLS
    assert L.mmvq_debug_block_sums_ex(1014, A, 16, 256, A, 1, A, None, 2, None) == mmvq.ERR_NULL
    assert L.mmvq_debug_block_sums_ex(7, A, 16, 256, A, 1, A, A, 2, None) == mmvq.ERR_TYPE


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "block_quantized_matvec_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "mmvq_oracle" not in text, f
