// Dense MMVQ: y[c][row] = sum over 32-blocks of d_w*d_a*sumi (Q4_K: minus
// dmin*m*s_a), for 1-8 Q8_1 activation columns ("Strata" PR #2207: the wide
// kernels at 1-8 columns; PR #1774 "What changed": the same integer sum and
// d*ds*sumi per sub-block, only the summation order differs).
//
// GB300 design: a CTA stages its Q8_1 columns into shared memory once (the
// quants re-laid 16-byte aligned and padded, d and s as floats: PR #2340's
// "ld_i4_a4" idea as one aligned shared load), then walks row groups of 16
// rows.  Its warps are arranged WR row groups x WK K-slices; each warp
// streams its blocks with 16-byte loads, decodes in registers and
// accumulates with dp4a; the K-slices are summed through shared memory in
// a fixed order, so results are run-to-run deterministic.
#include <algorithm>
#include <mutex>

#include "rowgroup.cuh"

namespace mmvq {

template <int LAYOUT, int NCOLS>
__global__ void __launch_bounds__(512) mmvq_dense_kernel(const uint8_t* __restrict__ W,
                                                         int64_t rows, int K,
                                                         const uint8_t* __restrict__ xq,
                                                         float* __restrict__ y,
                                                         int32_t* __restrict__ sumi) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int lane = threadIdx.x;
  const int wk = threadIdx.y, WK = blockDim.y;
  const int wr = threadIdx.z, WR = blockDim.z;
  const int warp = wr * WK + wk;
  const int nwarps = WK * WR;
  const int tid = lane + 32 * warp;
  const int nb = K / kQK;
  const int nbq = K / kQK8;
  const int rb = act_row_bytes(K);
  const int64_t n_rg = (rows + kTileRows - 1) / kTileRows;

  uint8_t* act = smem;
  float* da = reinterpret_cast<float*>(smem + NCOLS * rb);
  float* sa = da + NCOLS * nbq;
  float* red = sa + (LAYOUT == kQ4Gguf ? NCOLS * nbq : 0);
  uint8_t* stage =
      reinterpret_cast<uint8_t*>(red + nwarps * kMaxCols * kTileRows) + (size_t)warp * 2 * kGgufStage;

  grid_dependency_wait();
  stage_q8_1(xq, K, NCOLS, [](int c) { return c; }, act, da, LAYOUT == kQ4Gguf ? sa : nullptr,
             tid, 32 * nwarps);
  __syncthreads();

  for (int64_t rg0 = (int64_t)blockIdx.x * WR; rg0 < n_rg; rg0 += (int64_t)gridDim.x * WR) {
    const int64_t rg = rg0 + wr;
    const int64_t row = rg * kTileRows + (lane & 15);
    float acc[NCOLS];
#pragma unroll
    for (int c = 0; c < NCOLS; ++c) acc[c] = 0.0f;
    if (rg < n_rg) {
      int32_t* srow = (sumi && row < rows) ? sumi + row * nbq : nullptr;
      rowgroup_dot<LAYOUT, NCOLS>(W, rows, nb, rg, wk, WK, lane, act, rb, da, sa, nbq, acc, srow,
                                  rows * nbq, stage);
    }
    reduce_store<NCOLS>(acc, lane, wk, WK, wr, rg < n_rg, row, rows, red, y, rows);
  }
}

// ------------------------------------------------------------ host side ----

// Largest dynamic shared memory a CTA may opt into on this device.
size_t max_smem_optin() {
  static int v = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      v = 0;
  });
  return (size_t)v;
}

int device_sms() {
  static int sms = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      sms = 0;
    }
  });
  return sms;
}

// Smallest divisor of nb that is >= want (nb itself when there is none below).
int divisor_at_least(int nb, int want) {
  for (int d = std::max(want, 1); d < nb; ++d)
    if (nb % d == 0) return d;
  return nb;
}

// Raises a kernel's dynamic shared memory limit once it is first needed.
int ensure_smem(const void* kern, size_t smem, size_t* smem_set, std::mutex* mu) {
  std::lock_guard<std::mutex> lock(*mu);
  if (smem > *smem_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return MMVQ_ERR_CUDA;
    *smem_set = smem;
  }
  return MMVQ_OK;
}

template <int LAYOUT, int NCOLS>
static int launch_dense_t(const uint8_t* W, int64_t rows, int K, const uint8_t* xq, float* y,
                          int32_t* sumi, cudaStream_t stream) {
  auto kern = mmvq_dense_kernel<LAYOUT, NCOLS>;
  const int sms = device_sms();
  if (sms <= 0) return MMVQ_ERR_CUDA;
  const int nb = K / kQK;
  const int64_t n_rg = (rows + kTileRows - 1) / kTileRows;
  // Enough warps in flight to cover HBM latency: about 16 per SM.  Small
  // matrices split K across the warps of a CTA.
  const int64_t want_warps = (int64_t)sms * 16;
  int wk = 1;
  if (n_rg < want_warps) {
    const int64_t w = (want_warps + n_rg - 1) / n_rg;
    wk = divisor_at_least(nb, (int)std::min<int64_t>(w, nb));
    if (wk > 16) wk = 16;
  }
  int wr = std::max(1, 8 / wk);
  if ((int64_t)wr > n_rg) wr = (int)n_rg;
  int nwarps = wk * wr;
  size_t smem = mmvq_smem_bytes(LAYOUT, K, NCOLS, nwarps);
  const size_t limit = max_smem_optin();
  while (smem > limit && nwarps > 1) {  // long rows x many columns: fewer warps
    if (wr > 1) --wr; else wk = std::max(1, wk / 2);
    nwarps = wk * wr;
    smem = mmvq_smem_bytes(LAYOUT, K, NCOLS, nwarps);
  }
  if (smem > limit) return MMVQ_ERR_SHAPE;

  static std::mutex mu;
  static size_t smem_set = 48 * 1024;
  if (ensure_smem((const void*)kern, smem, &smem_set, &mu) != MMVQ_OK) return MMVQ_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * nwarps, smem) !=
          cudaSuccess ||
      per_sm <= 0)
    return MMVQ_ERR_CUDA;
  const int64_t ctas_needed = (n_rg + wr - 1) / wr;
  const int grid = (int)std::min<int64_t>(ctas_needed, (int64_t)sms * per_sm);
  dim3 block(32, wk, wr);
  kern<<<grid, block, smem, stream>>>(W, rows, K, xq, y, sumi);
  return cudaGetLastError() == cudaSuccess ? MMVQ_OK : MMVQ_ERR_CUDA;
}

template <int LAYOUT>
static int launch_dense_layout(const uint8_t* W, int64_t rows, int K, const uint8_t* xq, int ncols,
                               float* y, int32_t* sumi, cudaStream_t s) {
  switch (ncols) {
    case 1: return launch_dense_t<LAYOUT, 1>(W, rows, K, xq, y, sumi, s);
    case 2: return launch_dense_t<LAYOUT, 2>(W, rows, K, xq, y, sumi, s);
    case 3: return launch_dense_t<LAYOUT, 3>(W, rows, K, xq, y, sumi, s);
    case 4: return launch_dense_t<LAYOUT, 4>(W, rows, K, xq, y, sumi, s);
    case 5: return launch_dense_t<LAYOUT, 5>(W, rows, K, xq, y, sumi, s);
    case 6: return launch_dense_t<LAYOUT, 6>(W, rows, K, xq, y, sumi, s);
    case 7: return launch_dense_t<LAYOUT, 7>(W, rows, K, xq, y, sumi, s);
    case 8: return launch_dense_t<LAYOUT, 8>(W, rows, K, xq, y, sumi, s);
  }
  return MMVQ_ERR_NCOLS;
}

int launch_dense(int type, const void* W, int64_t rows, int K, const void* xq, int ncols, float* y,
                 int32_t* sumi, cudaStream_t s) {
  const uint8_t* w = static_cast<const uint8_t*>(W);
  const uint8_t* x = static_cast<const uint8_t*>(xq);
  switch (type) {
    case MMVQ_Q6_K_PLANAR: return launch_dense_layout<kQ6Planar>(w, rows, K, x, ncols, y, sumi, s);
    case MMVQ_Q6_K: return launch_dense_layout<kQ6Gguf>(w, rows, K, x, ncols, y, sumi, s);
    case MMVQ_Q4_K: return launch_dense_layout<kQ4Gguf>(w, rows, K, x, ncols, y, sumi, s);
  }
  return MMVQ_ERR_TYPE;
}

}  // namespace mmvq
