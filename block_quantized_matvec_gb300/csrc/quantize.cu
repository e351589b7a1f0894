// Q8_1 activation quantisation and the SiLU(gate)*up requantisation: one
// warp per 32-value block, the arithmetic of q8_1.cuh.
#include "common.cuh"
#include "q8_1.cuh"
#include "route.cuh"

namespace mmvq {

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
  const float h = silu_mul(row[kb * kQK8 + lane], row[F + kb * kQK8 + lane]);
  if (h_out) h_out[(int64_t)r * F + kb * kQK8 + lane] = h;
  quantize_lane(h, xq + blk * kQ81Bytes, lane);
}

// RMSNorm then Q8_1 (the opt-in fused norm named in PR #1774 "How it was
// checked"; no formula is given there, so the plain RMS norm with a weight
// vector).  CTA (slice, column) quantises the column's 32-blocks 8*slice ..
// 8*slice + 7, one per warp as in quantize_q8_1_kernel; every CTA of a column
// first reduces the whole column's mean square in the same order (each
// thread's share compensated in fp32, then fp64 across threads; close to the
// exact sum), so all of them get the same scale = fp32(1/sqrt(ms + eps))
// (computed in fp64); y = (x*scale)*w in fp32.
__global__ void __launch_bounds__(256) rmsnorm_quantize_kernel(const float* __restrict__ x,
                                                               const float* __restrict__ w,
                                                               float eps, int K, int64_t ldx,
                                                               uint8_t* __restrict__ xq,
                                                               float* __restrict__ y_out) {
  __shared__ double part[8];
  __shared__ float scale_s;
  // writes activations: no early start of the next kernel (see above)
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int c = blockIdx.y;
  const float* xc = x + (int64_t)c * ldx;
  // This thread's element of its warp's block is i0 = 256 * slice + tid, one
  // of those it sums: kept, and its weight loaded before the reduction.
  const int nbq = K / kQK8;
  const int kb = blockIdx.x * (blockDim.x >> 5) + warp;
  const int i0 = kb * kQK8 + lane;
  const float w0 = kb < nbq ? w[i0] : 0.0f;
  // Per thread: the exact square x*x = p + e (e from an fma) added into a
  // compensated fp32 pair (TwoSum), about 48 bits, with eight loads in
  // flight before the serial adds; the pairs are then combined in fp64 (FP64
  // units are scarce on this part).
  float x0 = 0.0f;
  float sh = 0.0f, sl = 0.0f;
  constexpr int kU = 8;
  for (int i = threadIdx.x; i < K; i += kU * blockDim.x) {
    float vs[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int iu = i + u * blockDim.x;
      vs[u] = iu < K ? xc[iu] : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int iu = i + u * blockDim.x;
      const float v = vs[u];
      if (iu == i0) x0 = v;
      const float p = __fmul_rn(v, v);
      const float e = __fmaf_rn(v, v, -p);
      const float t = __fadd_rn(sh, p);
      const float z = __fsub_rn(t, sh);
      const float err = __fadd_rn(__fsub_rn(sh, __fsub_rn(t, z)), __fsub_rn(p, z));
      sh = t;
      sl = __fadd_rn(sl, __fadd_rn(err, e));
    }
  }
  double ss = (double)sh + (double)sl;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) part[warp] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += part[i];
    scale_s = (float)(1.0 / sqrt(t / (double)K + (double)eps));
  }
  __syncthreads();
  const float scale = scale_s;
  if (kb >= nbq) return;
  const float v = __fmul_rn(__fmul_rn(x0, scale), w0);
  if (y_out) y_out[(int64_t)c * K + i0] = v;
  quantize_lane(v, xq + ((int64_t)c * nbq + kb) * kQ81Bytes, lane);
}

int launch_rmsnorm_quantize(const float* x, const float* w, float eps, int K, int ncols,
                            int64_t ldx, void* xq, float* y_out, cudaStream_t stream) {
  const int slices = (K / kQK8 + 7) / 8;
  return launch_pdl(rmsnorm_quantize_kernel, dim3(slices, ncols), dim3(256), 0, stream, x, w, eps,
                    K, ldx, static_cast<uint8_t*>(xq), y_out);
}

// The first step of an expert layer in one launch: blocks 0 .. n-2 quantise
// the hidden states as quantize_q8_1_kernel, the last block builds the
// per-expert token lists as route_groups_kernel (the two are independent).
// Writes activations, so no early start of the next kernel.
__global__ void __launch_bounds__(256) quantize_route_kernel(
    const float* __restrict__ x, int K, int ncols, int64_t ldx, uint8_t* __restrict__ xq,
    const int32_t* __restrict__ topk, int n_slots, int k, int n_experts,
    int32_t* __restrict__ expert_ids, int32_t* __restrict__ offsets,
    int32_t* __restrict__ act_index, int32_t* __restrict__ slot_of, int32_t* __restrict__ status) {
  grid_dependency_wait();
  if (blockIdx.x == gridDim.x - 1) {
    route_groups_cta(topk, n_slots, k, n_experts, expert_ids, offsets, act_index, slot_of, status);
    return;
  }
  const int lane = threadIdx.x & 31;
  const int nbq = K / kQK8;
  const int64_t blk = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (blk >= (int64_t)ncols * nbq) return;
  const int c = (int)(blk / nbq);
  const int kb = (int)(blk - (int64_t)c * nbq);
  quantize_lane(x[(int64_t)c * ldx + kb * kQK8 + lane], xq + blk * kQ81Bytes, lane);
}

int launch_route_groups(const int32_t* topk, int T, int k, int n_experts, int32_t* expert_ids,
                        int32_t* token_offsets, int32_t* act_index, int32_t* slot_of,
                        int32_t* status, cudaStream_t s);

int launch_quantize_route(const float* x, int K, int ncols, int64_t ldx, void* xq,
                          const int32_t* topk, int T, int k, int n_experts, int32_t* expert_ids,
                          int32_t* token_offsets, int32_t* act_index, int32_t* slot_of,
                          int32_t* status, cudaStream_t stream);

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

// One launch when the routing fits one 256-thread block (four experts per
// thread), else the two kernels back to back.
int launch_quantize_route(const float* x, int K, int ncols, int64_t ldx, void* xq,
                          const int32_t* topk, int T, int k, int n_experts, int32_t* expert_ids,
                          int32_t* token_offsets, int32_t* act_index, int32_t* slot_of,
                          int32_t* status, cudaStream_t stream) {
  if (n_experts > 4 * 256) {
    const int rc = launch_quantize_q8_1(x, K, ncols, ldx, xq, stream);
    if (rc != MMVQ_OK) return rc;
    return launch_route_groups(topk, T, k, n_experts, expert_ids, token_offsets, act_index,
                               slot_of, status, stream);
  }
  const int64_t blocks = (int64_t)ncols * (K / kQK8);
  const int grid = (int)((blocks + 7) / 8) + 1;
  return launch_pdl(quantize_route_kernel, dim3(grid), dim3(256), 0, stream, x, K, ncols, ldx,
                    static_cast<uint8_t*>(xq), topk, T * k, k, n_experts, expert_ids,
                    token_offsets, act_index, slot_of, status);
}

}  // namespace mmvq
