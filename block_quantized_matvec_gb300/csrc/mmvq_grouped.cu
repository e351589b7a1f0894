// Grouped expert MMVQ over per-expert token lists ("Strata" PR #2746, "B70
// validation": grouped expert calls with empty groups; issue #2801: the
// native_gu_kernel / native_down_kernel grouped gate/up and down kernels).
//
// GB300 design: one persistent launch for all groups.  Every CTA compacts
// the non-empty groups from the offsets into shared memory, so empty groups
// cost neither a launch nor a CTA pass; the work items (non-empty group x
// 16-row group) are then split into equal contiguous ranges, one per CTA, in
// group-major order, so a CTA restages its Q8_1 columns only when its range
// crosses into the next group.  Each item runs the dense row-group routine
// with as many columns as the group has positions (up to 8 at a time).
#include <algorithm>

#include "rowgroup.cuh"

namespace mmvq {

int device_sms();
size_t max_smem_optin();
int divisor_at_least(int nb, int want);
int ensure_smem(const void* kern, size_t smem);

constexpr int kMaxGroups = 4096;

// Exclusive prefix sum over the CTA; returns the total in *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31;
  const int tid = threadIdx.x + blockDim.x * (threadIdx.y + blockDim.y * threadIdx.z);
  const int warp = tid >> 5;
  const int nwarps = (blockDim.x * blockDim.y * blockDim.z) >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int w = 0; w < nwarps; ++w) {
      const int s = warp_sums[w];
      warp_sums[w] = run;
      run += s;
    }
    warp_sums[nwarps] = run;
  }
  __syncthreads();
  const int out = warp_sums[warp] + x - v;
  *total = warp_sums[nwarps];
  __syncthreads();
  return out;
}

template <int LAYOUT, int NC>
__device__ __forceinline__ void grouped_item(const uint8_t* Wexp, int64_t rows, int nb, int64_t rg,
                                             int wk, int WK, int lane, const uint8_t* act, int rb,
                                             const float* da, const float* sa, int nbq, float* red,
                                             float* ybase, uint8_t* stage) {
  float acc[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) acc[c] = 0.0f;
  rowgroup_dot<LAYOUT, NC>(Wexp, rows, nb, rg, wk, WK, lane, act, rb, da, sa, nbq, acc, nullptr, 0,
                           stage);
  reduce_store<NC>(acc, lane, wk, WK, 0, true, rg * kTileRows + (lane & 15), rows, red, ybase, rows);
}

template <int LAYOUT>
__global__ void __launch_bounds__(512) mmvq_grouped_kernel(
    const uint8_t* __restrict__ W, int n_experts, int64_t rows, int K,
    const int32_t* __restrict__ expert_ids, const int32_t* __restrict__ offsets, int n_groups,
    const int32_t* __restrict__ act_index, const uint8_t* __restrict__ xq, int n_xq_cols,
    float* __restrict__ y, int32_t* __restrict__ status) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int active[kMaxGroups];
  __shared__ int warp_sums[17];
  __shared__ int cols_s[kMaxCols];

  const int lane = threadIdx.x;
  const int wk = threadIdx.y, WK = blockDim.y;
  const int tid = lane + 32 * wk;
  const int nthreads = 32 * WK;
  const int nb = K / kQK;
  const int nbq = K / kQK8;
  const int rb = act_row_bytes(K);
  const int64_t n_rg = (rows + kTileRows - 1) / kTileRows;
  const int64_t expert_bytes = rows * nb * (LAYOUT == kQ4Gguf ? kQ4KBytes : kQ6KBytes);

  uint8_t* act = smem;
  float* da = reinterpret_cast<float*>(smem + kMaxCols * rb);
  float* sa = da + kMaxCols * nbq;
  float* red = sa + (LAYOUT == kQ4Gguf ? kMaxCols * nbq : 0);
  uint8_t* stage =
      reinterpret_cast<uint8_t*>(red + WK * kMaxCols * kTileRows) + (size_t)wk * 2 * kGgufStage;

  grid_launch_dependents();
  grid_dependency_wait();

  // 1. compact the valid non-empty groups, in group order
  const int per = (n_groups + nthreads - 1) / nthreads;
  const int g0 = tid * per;
  const int g1 = min(n_groups, g0 + per);
  int cnt = 0;
  bool bad = false;
  for (int g = g0; g < g1; ++g) {
    const int e = expert_ids[g];
    const int o0 = offsets[g], o1 = offsets[g + 1];
    const bool ok = e >= 0 && e < n_experts && o0 >= 0 && o1 >= o0;
    bad |= !ok;
    cnt += (ok && o1 > o0) ? 1 : 0;
  }
  if (bad && status && blockIdx.x == 0) *status = MMVQ_ERR_ROUTING;
  int n_active = 0;
  int pos = block_exclusive_scan(cnt, warp_sums, &n_active);
  for (int g = g0; g < g1; ++g) {
    const int e = expert_ids[g];
    const int o0 = offsets[g], o1 = offsets[g + 1];
    if (e >= 0 && e < n_experts && o0 >= 0 && o1 > o0) active[pos++] = g;
  }
  __syncthreads();

  // 2. this CTA's contiguous share of the (group, row group) items
  const int64_t n_items = (int64_t)n_active * n_rg;
  const int64_t it0 = n_items * blockIdx.x / gridDim.x;
  const int64_t it1 = n_items * (blockIdx.x + 1) / gridDim.x;
  int staged_g = -1, staged_p0 = -1;
  for (int64_t it = it0; it < it1; ++it) {
    const int a = (int)(it / n_rg);
    const int64_t rg = it - (int64_t)a * n_rg;
    const int g = active[a];
    const int e = expert_ids[g];
    const int pe = offsets[g + 1];
    for (int p0 = offsets[g]; p0 < pe; p0 += kMaxCols) {
      const int n = min(kMaxCols, pe - p0);
      if (g != staged_g || p0 != staged_p0) {
        __syncthreads();  // the previous columns are no longer read
        if (tid < n) {
          const int col = act_index ? act_index[p0 + tid] : p0 + tid;
          const bool ok = col >= 0 && col < n_xq_cols;
          if (!ok && status) *status = MMVQ_ERR_ROUTING;
          cols_s[tid] = ok ? col : -1;
        }
        __syncthreads();
        // an invalid column is staged as zeros (d = 0, q = 0): its rows come out 0
        stage_q8_1(xq, K, n, [&](int c) { return cols_s[c]; }, act, da,
                   LAYOUT == kQ4Gguf ? sa : nullptr, tid, nthreads);
        __syncthreads();
        staged_g = g;
        staged_p0 = p0;
      }
      const uint8_t* Wexp = W + (size_t)e * expert_bytes;
      float* ybase = y + (size_t)p0 * rows;
      switch (n) {
        case 1: grouped_item<LAYOUT, 1>(Wexp, rows, nb, rg, wk, WK, lane, act, rb, da, sa, nbq, red, ybase, stage); break;
        case 2: grouped_item<LAYOUT, 2>(Wexp, rows, nb, rg, wk, WK, lane, act, rb, da, sa, nbq, red, ybase, stage); break;
        case 3: grouped_item<LAYOUT, 3>(Wexp, rows, nb, rg, wk, WK, lane, act, rb, da, sa, nbq, red, ybase, stage); break;
        case 4: grouped_item<LAYOUT, 4>(Wexp, rows, nb, rg, wk, WK, lane, act, rb, da, sa, nbq, red, ybase, stage); break;
        case 5: grouped_item<LAYOUT, 5>(Wexp, rows, nb, rg, wk, WK, lane, act, rb, da, sa, nbq, red, ybase, stage); break;
        case 6: grouped_item<LAYOUT, 6>(Wexp, rows, nb, rg, wk, WK, lane, act, rb, da, sa, nbq, red, ybase, stage); break;
        case 7: grouped_item<LAYOUT, 7>(Wexp, rows, nb, rg, wk, WK, lane, act, rb, da, sa, nbq, red, ybase, stage); break;
        default: grouped_item<LAYOUT, 8>(Wexp, rows, nb, rg, wk, WK, lane, act, rb, da, sa, nbq, red, ybase, stage); break;
      }
    }
  }
}

template <int LAYOUT>
static int launch_grouped_t(const uint8_t* W, int n_experts, int64_t rows, int K,
                            const int32_t* expert_ids, const int32_t* offsets, int n_groups,
                            const int32_t* act_index, const uint8_t* xq, int n_xq_cols, float* y,
                            int32_t* status, cudaStream_t stream) {
  auto kern = mmvq_grouped_kernel<LAYOUT>;
  const int sms = device_sms();
  if (sms <= 0) return MMVQ_ERR_CUDA;
  const int nb = K / kQK;
  // Small K: one warp per 256-block of the row group; large K: about 4 slices.
  int wk = std::min(16, divisor_at_least(nb, std::min(nb, 3)));
  size_t smem = mmvq_smem_bytes(LAYOUT, K, kMaxCols, wk);
  // the kernel also holds ~16.5 KB of static shared memory (the group list)
  const size_t limit = max_smem_optin() - (kMaxGroups + 32) * sizeof(int);
  while (smem > limit && wk > 1) {
    wk = std::max(1, wk / 2);
    smem = mmvq_smem_bytes(LAYOUT, K, kMaxCols, wk);
  }
  if (smem > limit) return MMVQ_ERR_SHAPE;
  if (ensure_smem((const void*)kern, smem) != MMVQ_OK) return MMVQ_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * wk, smem) != cudaSuccess ||
      per_sm <= 0)
    return MMVQ_ERR_CUDA;
  const int64_t n_rg = (rows + kTileRows - 1) / kTileRows;
  const int64_t max_items = (int64_t)n_groups * n_rg;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(max_items, (int64_t)sms * per_sm));
  return launch_pdl(kern, dim3(grid), dim3(32, wk, 1), smem, stream, W, n_experts, rows, K,
                    expert_ids, offsets, n_groups, act_index, xq, n_xq_cols, y, status);
}

int launch_grouped_tma(int type, const void* W, int n_experts, int64_t rows, int K,
                       const int32_t* expert_ids, const int32_t* offsets, int n_groups,
                       const int32_t* act_index, const void* xq, int n_xq_cols, float* y,
                       int32_t* status, cudaStream_t s);

int launch_grouped(int type, const void* W, int n_experts, int64_t rows, int K,
                   const int32_t* expert_ids, const int32_t* offsets, int n_groups,
                   const int32_t* act_index, const void* xq, int n_xq_cols, float* y,
                   int32_t* status, cudaStream_t s) {
  const uint8_t* w = static_cast<const uint8_t*>(W);
  const uint8_t* x = static_cast<const uint8_t*>(xq);
  switch (type) {
    case MMVQ_Q4_K:
      return launch_grouped_t<kQ4Gguf>(w, n_experts, rows, K, expert_ids, offsets, n_groups,
                                       act_index, x, n_xq_cols, y, status, s);
    case MMVQ_Q6_K:
      return launch_grouped_t<kQ6Gguf>(w, n_experts, rows, K, expert_ids, offsets, n_groups,
                                       act_index, x, n_xq_cols, y, status, s);
    case MMVQ_Q4_K_PLANAR:
    case MMVQ_Q6_K_PLANAR:
      return launch_grouped_tma(type, W, n_experts, rows, K, expert_ids, offsets, n_groups,
                                act_index, xq, n_xq_cols, y, status, s);
  }
  return MMVQ_ERR_TYPE;
}

}  // namespace mmvq
