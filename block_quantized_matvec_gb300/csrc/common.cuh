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
constexpr int kTileRows = 16;     // rows per planar tile / per warp
constexpr int kTileBytes = 3360;  // 16 rows x one Q6_K block
constexpr int kMaxCols = 8;
constexpr int kMaxK = 16384;

// Activation quants in shared memory: per column, K bytes with 16 bytes of
// padding after every 128 (four Q8_1 blocks), so that the two halves of a
// 256-block (lanes 0-15 and 16-31 of a warp) hit different banks.
__host__ __device__ constexpr int act_row_bytes(int K) { return K + K / 8; }
__device__ __forceinline__ int act_off(int kb) { return kb * 32 + (kb >> 2) * 16; }

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint2 ldg_nc_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(r.x), "=r"(r.y)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint16_t ldg_nc_u16(const void* p) {
  uint16_t r;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
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

// Stage Q8_1 columns into shared memory: quants into the padded byte rows,
// d (and s when wanted) as floats.  act: [ncols][act_row_bytes(K)] bytes,
// da/sa: [ncols][K/32].  col_of(c) gives the xq column for local column c.
template <typename ColOf>
__device__ __forceinline__ void stage_q8_1(const uint8_t* __restrict__ xq, int K, int ncols,
                                           ColOf col_of, uint8_t* act, float* da, float* sa,
                                           int tid, int nthreads) {
  const int nbq = K / kQK8;
  const int total = ncols * nbq * 9;  // 9 words per block: header + 8 quant words
  const int rb = act_row_bytes(K);
  for (int w = tid; w < total; w += nthreads) {
    const int c = w / (nbq * 9);
    const int rem = w - c * nbq * 9;
    const int kb = rem / 9;
    const int k = rem - kb * 9;
    const uint8_t* blk = xq + ((size_t)col_of(c) * nbq + kb) * kQ81Bytes;
    const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(blk) + k);
    if (k == 0) {
      da[c * nbq + kb] = half_bits_to_float((uint16_t)(v & 0xffff));
      if (sa) sa[c * nbq + kb] = half_bits_to_float((uint16_t)(v >> 16));
    } else {
      *reinterpret_cast<uint32_t*>(act + c * rb + act_off(kb) + 4 * (k - 1)) = v;
    }
  }
}

}  // namespace mmvq
