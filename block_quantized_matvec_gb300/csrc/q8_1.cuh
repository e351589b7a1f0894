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

// roundf(v / d) for a value of a block whose d = amax/127 (so |v/d| <= 127
// up to rounding), with the same result as roundf of the IEEE quotient.
// A candidate q = roundf(v * r), r the hardware's approximate reciprocal of
// d (PTX rcp.approx), is accepted when the exact quotient z = v/d provably
// lies in (q - 1/2 + 2^-17, q + 1/2 - 2^-17): the IEEE quotient is within
// half an ulp (at most 2^-18 below 128) of z, so it rounds to q as well.
// The two bounds q -+ (1/2 - 2^-17) are exact in fp32 for |q| <= 127 (24
// significant bits), and the sign of v - c*d is that of one fmaf, which
// rounds once and so keeps the sign of the exact value.  This needs no bound
// on the reciprocal's error; a candidate that fails (near a half-integer,
// or non-finite) takes the IEEE division.
__device__ __forceinline__ int round_div_q8(float v, float d, float r) {
  const float q = roundf(__fmul_rn(v, r));
  const float half_in = 0.5f - 0x1p-17f;
  const float lo = __fsub_rn(q, half_in);
  const float hi = __fadd_rn(q, half_in);
  if (fabsf(q) <= 127.0f && fmaf(-lo, d, v) > 0.0f && fmaf(-hi, d, v) < 0.0f) return (int)q;
  return (int)roundf(__fdiv_rn(v, d));
}

__device__ __forceinline__ float rcp_approx(float d) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
  return r;
}

// A 32-value block by four consecutive lanes (a quad), eight values each:
// v[8] = values 8*j .. 8*j+7 for quad lane j.  The same bytes as
// quantize_block_warp: the quad's max and sum by two xor shuffles each, the
// division by round_div_q8.  Returns the lane's eight quants as two
// little-endian words; header: fp16 d (low) and s (high), on every lane.
// All 32 lanes of the warp must call it (inactive quads with zeros).
__device__ __forceinline__ void quantize_block_quad(const float (&v)[8], uint32_t& w0,
                                                    uint32_t& w1, uint32_t& header) {
  float m = fabsf(v[0]);
#pragma unroll
  for (int i = 1; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  const float d = __fdiv_rn(m, 127.0f);
  const float r = rcp_approx(d);
  int sum = 0;
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int q = (d != 0.0f) ? round_div_q8(v[i], d, r) : 0;
    sum += q;
    w[i >> 2] |= (uint32_t)(q & 0xff) << (8 * (i & 3));
  }
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  w0 = w[0];
  w1 = w[1];
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
