// Device helpers shared by the MMVQ kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mmvq.h"

namespace mmvq {

constexpr int kQK = 256;          // weights per K-quant block
constexpr int kQK8 = 32;          // values per Q8_1 block
constexpr int kQ81Bytes = 36;     // fp16 d, fp16 s, int8 q[32]
constexpr int kQ6KBytes = 210;
constexpr int kQ4KBytes = 144;
constexpr int kQ5KBytes = 176;
constexpr int kTileRows = 16;     // rows per planar tile / per warp
constexpr int kTileBytes = 3360;  // 16 rows x one Q6_K block
constexpr int kTileBytesQ4 = 2304;  // 16 rows x one Q4_K block
constexpr int kTileBytesQ5 = 2816;  // 16 rows x one Q5_K block
constexpr int kMaxCols = 8;

// Weight layouts the kernels read.
enum Layout { kQ6Planar = 0, kQ6Gguf = 1, kQ4Gguf = 2, kQ4Planar = 3, kQ5Planar = 4 };
constexpr int kMaxK = 16384;

// Activation quants in shared memory: per column, K bytes with 16 bytes of
// padding after every 128 (four Q8_1 blocks), so that the two halves of a
// 256-block (lanes 0-15 and 16-31 of a warp) hit different banks, and the
// column stride rounded up to 16 more than a multiple of 128 bytes, so that
// eight lanes reading the same word of eight columns hit eight different
// groups of four banks (the tensor-core consumer's activation fragments).
__host__ __device__ constexpr int act_row_bytes(int K) {
  return K + K / 8 + (((16 - (K + K / 8)) % 128) + 128) % 128;
}
__device__ __forceinline__ int act_off(int kb) { return kb * 32 + (kb >> 2) * 16; }

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ int dp4a(int a, int b, int c) { return __dp4a(a, b, c); }

// Q6_K 6-bit offset as SWAR: every byte of v is a code in 0..63; returns
// the four bytes (code - 32) as int8.  Setting bit 7 first keeps the byte
// subtraction from borrowing across bytes; the final xor clears it again.
__device__ __forceinline__ int q6_minus_32(uint32_t v) {
  return (int)(((v | 0x80808080u) - 0x20202020u) ^ 0x80808080u);
}

// Programmatic dependent launch: wait for the preceding kernel in the stream
// (no-op when launched without the attribute).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;");
}

// Prefetch [p, p + bytes) into L2 (bulk, asynchronous, no completion to
// wait for).  p is rounded down and the size up to 16 bytes; the caller
// keeps the range inside its allocation.  Safe before griddepcontrol.wait:
// L2 is the point of coherence, so data written afterwards by the preceding
// kernel still wins, and nothing is held in L1 or registers.
__device__ __forceinline__ void prefetch_l2(const void* p, int64_t bytes) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p) & ~uintptr_t(15);
  int64_t n = (int64_t)(reinterpret_cast<uintptr_t>(p) + bytes - a);
  n &= ~int64_t(15);
  while (n > 0) {
    const uint32_t chunk = (uint32_t)(n > (1 << 20) ? (1 << 20) : n);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"(chunk) : "memory");
    n -= chunk;
    a += chunk;
  }
}

// Stage Q8_1 columns into shared memory: quants into the padded byte rows,
// d (and s when wanted) as floats.  act: [ncols][act_row_bytes(K)] bytes,
// da/sa: [ncols][K/32].  col_of(c) gives the xq column for local column c,
// or -1 for a column to stage as zeros.  A column's blocks are one
// contiguous, 16-byte aligned run of 36*K/32 bytes (K % 256 == 0), read
// here 16 bytes per thread and scattered word by word.  kCoherent reads
// through L2 only (ld.global.cg), for columns written earlier in the same
// launch by other CTAs; otherwise the read-only path.
template <bool kCoherent = false, typename ColOf>
__device__ __forceinline__ void stage_q8_1(const uint8_t* __restrict__ xq, int K, int ncols,
                                           ColOf col_of, uint8_t* act, float* da, float* sa,
                                           int tid, int nthreads) {
  const int nbq = K / kQK8;
  const int vec_per_col = nbq * 9 / 4;  // 16-byte vectors per column
  const int rb = act_row_bytes(K);
  for (int c = 0; c < ncols; ++c)
  for (int vi = tid; vi < vec_per_col; vi += nthreads) {
    const int col = col_of(c);
    uint4 q = make_uint4(0u, 0u, 0u, 0u);
    if (col >= 0)
    {
      const uint4* src = reinterpret_cast<const uint4*>(xq + (size_t)col * nbq * kQ81Bytes) + vi;
      q = kCoherent ? __ldcg(src) : __ldg(src);
    }
    const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int w = 4 * vi + e;  // word index in the column
      const int kb = w / 9;
      const int k = w - kb * 9;
      if (k == 0) {
        da[c * nbq + kb] = half_bits_to_float((uint16_t)(w4[e] & 0xffff));
        if (sa) sa[c * nbq + kb] = half_bits_to_float((uint16_t)(w4[e] >> 16));
      } else {
        *reinterpret_cast<uint32_t*>(act + c * rb + act_off(kb) + 4 * (k - 1)) = w4[e];
      }
    }
  }
}

// stage_q8_1 for a K-slice of the columns: the 32-blocks [kb0, kb0 + Kc/32)
// of each column (column stride nbq_total blocks) into a staging area laid
// out as for a K = Kc matrix.  kb0 and Kc are multiples of 8 blocks / 256
// values, so every source vector is 16-byte aligned.
__device__ __forceinline__ void stage_q8_1_slice(const uint8_t* __restrict__ xq, int nbq_total,
                                                 int kb0, int Kc, int ncols, uint8_t* act,
                                                 float* da, float* sa, int tid, int nthreads) {
  const int nbq = Kc / kQK8;
  const int vec_per_col = nbq * 9 / 4;
  const int rb = act_row_bytes(Kc);
  for (int c = 0; c < ncols; ++c)
  for (int vi = tid; vi < vec_per_col; vi += nthreads) {
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(
                              xq + ((size_t)c * nbq_total + kb0) * kQ81Bytes) + vi);
    const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int w = 4 * vi + e;
      const int kb = w / 9;
      const int k = w - kb * 9;
      if (k == 0) {
        da[c * nbq + kb] = half_bits_to_float((uint16_t)(w4[e] & 0xffff));
        if (sa) sa[c * nbq + kb] = half_bits_to_float((uint16_t)(w4[e] >> 16));
      } else {
        *reinterpret_cast<uint32_t*>(act + c * rb + act_off(kb) + 4 * (k - 1)) = w4[e];
      }
    }
  }
}

// Launches `kern` with programmatic stream serialization allowed, so that
// it may start while the preceding kernel in the stream drains; every kernel
// of this library waits (griddepcontrol.wait) before it reads anything the
// preceding kernel may write, and lets its own dependents launch early.
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...) == cudaSuccess ? MMVQ_OK : MMVQ_ERR_CUDA;
}

}  // namespace mmvq
