// Per-expert token lists: the routing step of the grouped expert calls
// ("Strata" PR #2746 "B70 validation": per-expert token groups, empty groups
// allowed), as the work of one CTA: counting sort of the routing slots by
// expert, stable in slot order.  Slot s = t*k + j.  Thread t owns the
// ceil(n_experts / blockDim.x) consecutive experts from t times that count
// (n_experts <= kMaxE, blockDim.x a multiple of 32, at most 1024).  The
// outputs may live in global or shared memory; expert_ids and status may be
// NULL.
#pragma once
#include "common.cuh"

namespace mmvq {

template <int kMaxE = 4096>
__device__ __forceinline__ void route_groups_cta(const int32_t* __restrict__ topk, int n_slots,
                                                 int k, int n_experts,
                                                 int32_t* __restrict__ expert_ids,
                                                 int32_t* __restrict__ offsets,
                                                 int32_t* __restrict__ act_index,
                                                 int32_t* __restrict__ slot_of,
                                                 int32_t* __restrict__ status) {
  __shared__ int cnt[kMaxE];
  __shared__ int wsum[33];
  const int tid = threadIdx.x;
  for (int e = tid; e < n_experts; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  for (int s = tid; s < n_slots; s += blockDim.x) {
    const int e = topk[s];
    if (e >= 0 && e < n_experts) {
      atomicAdd(&cnt[e], 1);
    } else if (status) {
      *status = MMVQ_ERR_ROUTING;
    }
  }
  __syncthreads();
  // exclusive scan over the experts, each thread's run of them in order
  const int per = (n_experts + (int)blockDim.x - 1) / (int)blockDim.x;
  const int e_lo = min(n_experts, tid * per), e_hi = min(n_experts, e_lo + per);
  int sum = 0;
  for (int e = e_lo; e < e_hi; ++e) sum += cnt[e];
  const int lane = tid & 31, warp = tid >> 5;
  int x = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += v;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the warp totals, by shuffles
    const int nw = (int)(blockDim.x >> 5);
    const int v = lane < nw ? wsum[lane] : 0;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane < nw) wsum[lane] = inc - v;
    if (lane == 31) wsum[32] = inc;
  }
  __syncthreads();
  int run = wsum[warp] + x - sum;
  for (int e = e_lo; e < e_hi; ++e) {
    const int c = cnt[e];
    offsets[e] = run;
    if (expert_ids) expert_ids[e] = e;
    cnt[e] = run;  // becomes the placement cursor
    run += c;
  }
  if (tid == 0) offsets[n_experts] = wsum[32];
  __syncthreads();
  // stable placement by one warp, 32 slots at a time in slot order
  if (warp == 0) {
    for (int base = 0; base < n_slots; base += 32) {
      const int s = base + lane;
      int e = -1;
      if (s < n_slots) {
        const int v = topk[s];
        if (v >= 0 && v < n_experts) e = v;
      }
      const unsigned same = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(same & ((1u << lane) - 1u));
      if (e >= 0) {
        const int p = cnt[e] + rank;
        act_index[p] = s / k;
        slot_of[p] = s;
      }
      __syncwarp();
      if (e >= 0 && rank == 0) cnt[e] += __popc(same);
      __syncwarp();
    }
  }
}

}  // namespace mmvq
