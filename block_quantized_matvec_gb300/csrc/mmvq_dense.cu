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
//
// Latency: the launch lets the next kernel in the stream start early
// (programmatic dependent launch), and before waiting for the preceding
// kernel each CTA asks L2 for the weight bytes of its first row groups, so
// the weight stream overlaps the previous kernel's tail and the activation
// staging.  The host picks the K-split so that all row groups of small and
// mid-size matrices are resident in one wave; large ones run persistently
// and prefetch the next row group into L2 while computing the current one.
#include <algorithm>
#include <cstdint>
#include <map>
#include <mutex>
#include <unordered_map>

#include "rowgroup.cuh"

namespace mmvq {

// Byte range of the weights of row group rg (16 rows, all K).
template <int LAYOUT>
__device__ __forceinline__ void rowgroup_range(const uint8_t* W, int64_t rows, int nb, int64_t rg,
                                               const uint8_t** p, int64_t* bytes) {
  const int bb = (LAYOUT == kQ4Gguf) ? kQ4KBytes : kQ6KBytes;
  const int64_t r0 = rg * kTileRows;
  const int64_t r1 = min(r0 + kTileRows, rows);
  *p = W + r0 * nb * bb;
  *bytes = (r1 - r0) * nb * bb;
}

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
  const int64_t rg_stride = (int64_t)gridDim.x * WR;

  uint8_t* act = smem;
  float* da = reinterpret_cast<float*>(smem + NCOLS * rb);
  float* sa = da + NCOLS * nbq;
  float* red = sa + (LAYOUT == kQ4Gguf ? NCOLS * nbq : 0);
  uint8_t* stage =
      reinterpret_cast<uint8_t*>(red + nwarps * kMaxCols * kTileRows) + (size_t)warp * 2 * kGgufStage;

  grid_launch_dependents();
  if (wk == 0 && lane == 0) {
    const int64_t rg = (int64_t)blockIdx.x * WR + wr;
    if (rg < n_rg) {
      const uint8_t* p;
      int64_t bytes;
      rowgroup_range<LAYOUT>(W, rows, nb, rg, &p, &bytes);
      prefetch_l2(p, bytes);
    }
  }
  grid_dependency_wait();
  stage_q8_1(xq, K, NCOLS, [](int c) { return c; }, act, da, LAYOUT == kQ4Gguf ? sa : nullptr,
             tid, 32 * nwarps);
  __syncthreads();

  for (int64_t rg0 = (int64_t)blockIdx.x * WR; rg0 < n_rg; rg0 += rg_stride) {
    const int64_t rg = rg0 + wr;
    const int64_t row = rg * kTileRows + (lane & 15);
    if (wk == 0 && lane == 0 && rg + rg_stride < n_rg) {  // next row group into L2
      const uint8_t* p;
      int64_t bytes;
      rowgroup_range<LAYOUT>(W, rows, nb, rg + rg_stride, &p, &bytes);
      prefetch_l2(p, bytes);
    }
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
// Raises the kernel's dynamic shared-memory limit on the current device to
// at least `smem` (the attribute is per kernel and per device).
int ensure_smem(const void* kern, size_t smem) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> set;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MMVQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  size_t& have = set[{kern, dev}];
  if (smem > have) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return MMVQ_ERR_CUDA;
    have = smem;
  }
  return MMVQ_OK;
}

struct DenseCfg {
  int wk, wr, grid;
  size_t smem;
};

// Launch shape for a (rows, K) matrix, cached per shape:
//  - many row groups (>= 8 per SM): one warp per row group, 8 per CTA,
//    persistent grid of (CTAs resident per SM) x SMs;
//  - otherwise the largest K-split WK (a divisor of K/256, at most 16 warps)
//    that still keeps every row group's CTA resident in a single wave;
//  - unless no WK fits in one wave, or the one that does leaves each warp
//    more than 8 blocks of K (wide activations crowd the shared memory out):
//    then the WK with the fewest waves x K/256/WK, ties to fewer waves.
//    Measured on GB300: 2560 x 10240 at 8 columns took 110.6 us at WK = 1
//    (one wave) and 41.7 us at WK = 10 (two waves); 2560 x 16384 at 8
//    columns 192.8 us on the persistent shape (20 CTAs) and 66.2 us at
//    WK = 8 (two waves).
template <int LAYOUT, int NCOLS>
static int dense_config(int64_t rows, int K, DenseCfg* out) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, DenseCfg> cache;
  const uint64_t key = ((uint64_t)rows << 8) | (uint64_t)(K / kQK);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *out = it->second;
      return MMVQ_OK;
    }
  }
  auto kern = mmvq_dense_kernel<LAYOUT, NCOLS>;
  const int sms = device_sms();
  const size_t limit = max_smem_optin();
  if (sms <= 0 || limit == 0) return MMVQ_ERR_CUDA;
  const int nb = K / kQK;
  const int64_t n_rg = (rows + kTileRows - 1) / kTileRows;

  auto occupancy = [&](int nwarps, size_t smem, int* per_sm) -> int {
    if (smem > limit) return MMVQ_ERR_SHAPE;
    if (ensure_smem((const void*)kern, smem) != MMVQ_OK) return MMVQ_ERR_CUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, kern, 32 * nwarps, smem) !=
        cudaSuccess)
      return MMVQ_ERR_CUDA;
    return MMVQ_OK;
  };

  DenseCfg cfg = {0, 0, 0, 0};
  if (n_rg < (int64_t)sms * 8) {
    for (int wk = std::min(nb, 16); wk >= 1; --wk) {
      if (nb % wk) continue;
      const size_t smem = mmvq_smem_bytes(LAYOUT, K, NCOLS, wk);
      int per_sm = 0;
      const int rc = occupancy(wk, smem, &per_sm);
      if (rc == MMVQ_ERR_CUDA) return rc;
      if (rc != MMVQ_OK || per_sm < 1) continue;
      if (n_rg <= (int64_t)sms * per_sm) {
        cfg = {wk, 1, (int)n_rg, smem};
        break;
      }
    }
  }
  if (n_rg < (int64_t)sms * 8 && (cfg.wk == 0 || nb / cfg.wk > 8)) {
    // the one-wave choice, if any, against every larger K-split
    int64_t best = cfg.wk != 0 ? nb / cfg.wk : INT64_MAX;
    int64_t best_waves = cfg.wk != 0 ? 1 : INT64_MAX;
    for (int wk = std::min(nb, 16); wk > cfg.wk; --wk) {
      if (nb % wk) continue;
      const size_t smem = mmvq_smem_bytes(LAYOUT, K, NCOLS, wk);
      int per_sm = 0;
      const int rc = occupancy(wk, smem, &per_sm);
      if (rc == MMVQ_ERR_CUDA) return rc;
      if (rc != MMVQ_OK || per_sm < 1) continue;
      const int64_t waves = (n_rg + (int64_t)sms * per_sm - 1) / ((int64_t)sms * per_sm);
      const int64_t cost = waves * (nb / wk);
      if (cost < best || (cost == best && waves < best_waves)) {
        best = cost;
        best_waves = waves;
        cfg = {wk, 1, (int)n_rg, smem};
      }
    }
  }
  if (cfg.wk == 0) {
    // persistent: 8 row groups per CTA iteration (fewer if shared memory is short)
    for (int wr = 8; wr >= 1; --wr) {
      const size_t smem = mmvq_smem_bytes(LAYOUT, K, NCOLS, wr);
      int per_sm = 0;
      const int rc = occupancy(wr, smem, &per_sm);
      if (rc == MMVQ_ERR_CUDA) return rc;
      if (rc != MMVQ_OK || per_sm < 1) continue;
      const int64_t ctas = (n_rg + wr - 1) / wr;
      cfg = {1, wr, (int)std::min<int64_t>(ctas, (int64_t)sms * per_sm), smem};
      break;
    }
  }
  if (cfg.wk == 0) return MMVQ_ERR_SHAPE;
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = cfg;
  *out = cfg;
  return MMVQ_OK;
}

template <int LAYOUT, int NCOLS>
static int launch_dense_t(const uint8_t* W, int64_t rows, int K, const uint8_t* xq, float* y,
                          int32_t* sumi, cudaStream_t stream) {
  DenseCfg cfg;
  const int rc = dense_config<LAYOUT, NCOLS>(rows, K, &cfg);
  if (rc != MMVQ_OK) return rc;
  return launch_pdl(mmvq_dense_kernel<LAYOUT, NCOLS>, dim3(cfg.grid), dim3(32, cfg.wk, cfg.wr),
                    cfg.smem, stream, W, rows, K, xq, y, sumi);
}

template <int LAYOUT, int NCOLS>
static int dense_shape_t(int64_t rows, int K, int32_t* info) {
  DenseCfg cfg;
  const int rc = dense_config<LAYOUT, NCOLS>(rows, K, &cfg);
  if (rc != MMVQ_OK) return rc;
  info[0] = cfg.grid;
  info[1] = 32 * cfg.wk * cfg.wr;
  info[2] = (int32_t)cfg.smem;
  info[3] = cfg.wr;
  info[4] = cfg.wk;
  info[5] = 0;
  info[6] = 1;
  return MMVQ_OK;
}

template <int LAYOUT>
static int dense_shape_layout(int64_t rows, int K, int ncols, int32_t* info) {
  switch (ncols) {
    case 1: return dense_shape_t<LAYOUT, 1>(rows, K, info);
    case 2: return dense_shape_t<LAYOUT, 2>(rows, K, info);
    case 3: return dense_shape_t<LAYOUT, 3>(rows, K, info);
    case 4: return dense_shape_t<LAYOUT, 4>(rows, K, info);
    case 5: return dense_shape_t<LAYOUT, 5>(rows, K, info);
    case 6: return dense_shape_t<LAYOUT, 6>(rows, K, info);
    case 7: return dense_shape_t<LAYOUT, 7>(rows, K, info);
    case 8: return dense_shape_t<LAYOUT, 8>(rows, K, info);
  }
  return MMVQ_ERR_NCOLS;
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

int planar_tma_shape(int type, int64_t rows, int K, int ncols, int32_t* info);

int dense_shape(int type, int64_t rows, int K, int ncols, int32_t* info) {
  switch (type) {
    case MMVQ_Q6_K_PLANAR:
    case MMVQ_Q4_K_PLANAR:
    case MMVQ_Q5_K_PLANAR: return planar_tma_shape(type, rows, K, ncols, info);
    case MMVQ_Q6_K: return dense_shape_layout<kQ6Gguf>(rows, K, ncols, info);
    case MMVQ_Q4_K: return dense_shape_layout<kQ4Gguf>(rows, K, ncols, info);
  }
  return MMVQ_ERR_TYPE;
}

int launch_planar_tma(int type, const void* W, int64_t rows, int K, const void* xq, int ncols,
                      float* y, int32_t* sumi, uint32_t flags, cudaStream_t s);

int launch_dense(int type, const void* W, int64_t rows, int K, const void* xq, int ncols, float* y,
                 int32_t* sumi, uint32_t flags, cudaStream_t s) {
  const uint8_t* w = static_cast<const uint8_t*>(W);
  const uint8_t* x = static_cast<const uint8_t*>(xq);
  switch (type) {
    case MMVQ_Q6_K_PLANAR:
    case MMVQ_Q4_K_PLANAR:
    case MMVQ_Q5_K_PLANAR: return launch_planar_tma(type, W, rows, K, xq, ncols, y, sumi, flags, s);
    case MMVQ_Q6_K: return launch_dense_layout<kQ6Gguf>(w, rows, K, x, ncols, y, sumi, s);
    case MMVQ_Q4_K: return launch_dense_layout<kQ4Gguf>(w, rows, K, x, ncols, y, sumi, s);
  }
  return MMVQ_ERR_TYPE;
}

}  // namespace mmvq
