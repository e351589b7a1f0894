// Q8_1 quantisation of one 32-value block by one warp, and the SiLU(gate)*up
// value that feeds it between the gate|up and down products.
//
// Q8_1 ("Strata" PR #2340 "int4 activation loads"; PR #1774 "d * ds *
// sumi"): per 32 values, amax, d = amax/127, q = round-half-away(x/d),
// s = d*sum(q); d and s stored as fp16 (round to nearest even).  One value
// per lane; IEEE division and roundf (no fast-math), so the bytes are
// exactly those of the plain definition, whichever kernel runs them.
#pragma once
#include "common.cuh"

namespace mmvq {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// The block of the warp's 32 values: `word` is quants 4*(lane/4) .. +3 as
// one little-endian word (valid on lanes with lane % 4 == 0) and `header`
// the fp16 bits of d (low half) and s (high half), the same on every lane.
__device__ __forceinline__ void quantize_block_warp(float v, uint32_t& word, uint32_t& header) {
  const float amax = warp_max(fabsf(v));
  const float d = __fdiv_rn(amax, 127.0f);
  const int q = (d != 0.0f) ? (int)roundf(__fdiv_rn(v, d)) : 0;
  const int sum = warp_sum(q);
  const uint32_t b = (uint32_t)(q & 0xff);
  const uint32_t b1 = __shfl_down_sync(0xffffffffu, b, 1);
  const uint32_t b2 = __shfl_down_sync(0xffffffffu, b, 2);
  const uint32_t b3 = __shfl_down_sync(0xffffffffu, b, 3);
  word = b | (b1 << 8) | (b2 << 16) | (b3 << 24);
  const float s = __fmul_rn(d, (float)sum);
  header = (uint32_t)__half_as_ushort(__float2half_rn(d)) |
           ((uint32_t)__half_as_ushort(__float2half_rn(s)) << 16);
}

// One lane's value v of a 32-value block -> writes the 36-byte block at out
// (global or shared memory, 4-byte aligned).
__device__ __forceinline__ void quantize_lane(float v, uint8_t* out, int lane) {
  uint32_t word, header;
  quantize_block_warp(v, word, header);
  uint32_t* o32 = reinterpret_cast<uint32_t*>(out);
  if ((lane & 3) == 0) o32[1 + (lane >> 2)] = word;
  if (lane == 0) o32[0] = header;
}

// The same block written into the shared-memory staging layout of the MMVQ
// kernels (quants at act_col + act_off(kb), d and s as floats into da[kb],
// sa[kb]; sa may be NULL) and, when out != NULL, also as the 36-byte block
// at out: the values a kernel stages from that block.
__device__ __forceinline__ void quantize_lane_staged(float v, uint8_t* act_col, float* da,
                                                     float* sa, int kb, uint8_t* out, int lane) {
  uint32_t word, header;
  quantize_block_warp(v, word, header);
  if ((lane & 3) == 0) {
    *reinterpret_cast<uint32_t*>(act_col + act_off(kb) + 4 * (lane >> 2)) = word;
    if (out) reinterpret_cast<uint32_t*>(out)[1 + (lane >> 2)] = word;
  }
  if (lane == 0) {
    da[kb] = half_bits_to_float((uint16_t)(header & 0xffffu));
    if (sa) sa[kb] = half_bits_to_float((uint16_t)(header >> 16));
    if (out) reinterpret_cast<uint32_t*>(out)[0] = header;
  }
}

// h = gate/(1+exp(-gate)) * up in fp32 (expf, IEEE division).
__device__ __forceinline__ float silu_mul(float g, float u) {
  const float sg = __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
  return __fmul_rn(sg, u);
}

}  // namespace mmvq
