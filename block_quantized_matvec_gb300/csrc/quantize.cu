// Q8_1 activation quantisation and the SiLU(gate)*up requantisation.
//
// Q8_1 ("Strata" PR #2340 "int4 activation loads"; PR #1774 "d * ds *
// sumi"): per 32 values, amax, d = amax/127, q = round-half-away(x/d),
// s = d*sum(q); d and s stored as fp16 (round to nearest even).  One warp
// per block, one value per lane; IEEE division and roundf (no fast-math),
// so the bytes are exactly those of the plain definition.
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

// One lane's value v of a 32-value block -> writes the 36-byte block at out.
__device__ __forceinline__ void quantize_lane(float v, uint8_t* out, int lane) {
  const float amax = warp_max(fabsf(v));
  const float d = __fdiv_rn(amax, 127.0f);
  const int q = (d != 0.0f) ? (int)roundf(__fdiv_rn(v, d)) : 0;
  const int sum = warp_sum(q);
  // Pack four quants per lane 0..7 so the block is written with word stores.
  const uint32_t b = (uint32_t)(q & 0xff);
  const uint32_t b1 = __shfl_down_sync(0xffffffffu, b, 1);
  const uint32_t b2 = __shfl_down_sync(0xffffffffu, b, 2);
  const uint32_t b3 = __shfl_down_sync(0xffffffffu, b, 3);
  const uint32_t word = b | (b1 << 8) | (b2 << 16) | (b3 << 24);
  uint32_t* o32 = reinterpret_cast<uint32_t*>(out);
  if ((lane & 3) == 0) o32[1 + (lane >> 2)] = word;
  if (lane == 0) {
    const float s = __fmul_rn(d, (float)sum);
    const uint32_t hd = __half_as_ushort(__float2half_rn(d));
    const uint32_t hs = __half_as_ushort(__float2half_rn(s));
    o32[0] = hd | (hs << 16);
  }
}

__global__ void __launch_bounds__(256) quantize_q8_1_kernel(const float* __restrict__ x, int K,
                                                            int ncols, int64_t ldx,
                                                            uint8_t* __restrict__ xq) {
  // Writes activations: the next kernel may not start before this one ends
  // (no early trigger), which is what MMVQ_FLAG_XQ_STABLE relies on.
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const int nbq = K / kQK8;
  const int64_t blk = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (blk >= (int64_t)ncols * nbq) return;
  const int c = (int)(blk / nbq);
  const int kb = (int)(blk - (int64_t)c * nbq);
  const float v = x[(int64_t)c * ldx + kb * kQK8 + lane];
  quantize_lane(v, xq + blk * kQ81Bytes, lane);
}

// gu: [n][2F] = [gate | up]; h = gate/(1+exp(-gate)) * up (fp32, expf).
__global__ void __launch_bounds__(256) silu_mul_quantize_kernel(const float* __restrict__ gu, int F,
                                                                int n, uint8_t* __restrict__ xq,
                                                                float* __restrict__ h_out) {
  // Writes activations: no early start of the next kernel (see above).
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const int nbq = F / kQK8;
  const int64_t blk = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (blk >= (int64_t)n * nbq) return;
  const int r = (int)(blk / nbq);
  const int kb = (int)(blk - (int64_t)r * nbq);
  const float* row = gu + (int64_t)r * 2 * F;
  const float g = row[kb * kQK8 + lane];
  const float u = row[F + kb * kQK8 + lane];
  const float sg = __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
  const float h = __fmul_rn(sg, u);
  if (h_out) h_out[(int64_t)r * F + kb * kQK8 + lane] = h;
  quantize_lane(h, xq + blk * kQ81Bytes, lane);
}

int launch_quantize_q8_1(const float* x, int K, int ncols, int64_t ldx, void* xq,
                         cudaStream_t stream) {
  const int64_t blocks = (int64_t)ncols * (K / kQK8);
  const int grid = (int)((blocks + 7) / 8);
  return launch_pdl(quantize_q8_1_kernel, dim3(grid), dim3(256), 0, stream, x, K, ncols, ldx,
                    static_cast<uint8_t*>(xq));
}

int launch_silu_mul_quantize(const float* gu, int F, int n, void* xq, float* h_out,
                             cudaStream_t stream) {
  const int64_t blocks = (int64_t)n * (F / kQK8);
  const int grid = (int)((blocks + 7) / 8);
  return launch_pdl(silu_mul_quantize_kernel, dim3(grid), dim3(256), 0, stream, gu, F, n,
                    static_cast<uint8_t*>(xq), h_out);
}

}  // namespace mmvq
