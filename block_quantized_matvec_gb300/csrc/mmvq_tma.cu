// Planar Q6_K MMVQ fed by bulk copies (cp.async.bulk, the 1-D TMA path) into
// a shared-memory ring ("Strata" PR #2340 "STRATA_Q6_PLANAR": the head's
// planes are laid out so every lane load is one aligned 16-byte load; PR
// #2207: the weights are read once for all 1-8 columns).
//
// GB300 design.  One producer warp per CTA streams the CTA's weights from
// HBM into a ring of S stages with one bulk copy per stage; a stage is C
// consecutive 3360-byte tiles (16 rows x one 256-block each) of one row
// group, one tile per consumer warp.  Each stage has a pair of mbarriers
// (full: bytes landed; empty: all C consumer warps have read it).  The bytes
// in flight per SM are set by the ring depth, not by how many warps hold
// loads in registers.  Every consumer warp walks every stage in order, so a
// warp waiting for round r of a slot has itself consumed round r-1 there and
// the parity wait cannot alias an older phase.  A warp copies its tile's
// lane bytes out of the ring with 16-byte shared loads (the tile order makes
// them conflict-free), releases the stage, decodes and accumulates with
// dp4a; the K-slices are summed in a fixed warp order.
//
// Weights are never written by a kernel of this library that lets its
// successor launch early (repack and gather wait for completion), so the
// producer starts streaming before griddepcontrol.wait: a call's weights
// arrive while the preceding kernel in the stream is still finishing.  The
// consumers wait for the preceding kernel before they read activations.
//
// Every mbarrier wait is bounded (about one second of %globaltimer); on
// expiry the CTA records a fault in a device word (read with
// mmvq_read_device_fault), stops waiting, waits a bounded time for its
// copies still in flight and returns.  No trap, no unbounded spin.
#include <algorithm>
#include <mutex>
#include <unordered_map>

#include "kquant.cuh"

namespace mmvq {

int device_sms();
size_t max_smem_optin();
int ensure_smem(const void* kern, size_t smem, size_t* smem_set, std::mutex* mu);

__device__ unsigned int g_fault_word = 0;

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per wait
constexpr int kFaultMbarTimeout = 1;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(20000)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Waits for the phase with the given parity to complete; false after ~1 s.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// Tile bytes of lane L out of a ring slot: the same offsets as in global
// memory, so each warp-wide 16-byte load covers 512 consecutive bytes.
__device__ __forceinline__ void load_q6_tile_smem(const uint8_t* tile, int lane, Q6Half& w) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 v = *reinterpret_cast<const uint4*>(tile + 512 * j + 16 * lane);
    w.ql[4 * j + 0] = v.x;
    w.ql[4 * j + 1] = v.y;
    w.ql[4 * j + 2] = v.z;
    w.ql[4 * j + 3] = v.w;
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint4 v = *reinterpret_cast<const uint4*>(tile + 2048 + 512 * j + 16 * lane);
    w.qh[4 * j + 0] = v.x;
    w.qh[4 * j + 1] = v.y;
    w.qh[4 * j + 2] = v.z;
    w.qh[4 * j + 3] = v.w;
  }
  const uint2 s = *reinterpret_cast<const uint2*>(tile + 3072 + 8 * lane);
  w.sc[0] = s.x;
  w.sc[1] = s.y;
  w.d = *reinterpret_cast<const uint16_t*>(tile + 3328 + 2 * (lane & 15));
}

// Shared memory: [full S][empty S] mbarriers, a fail flag, the ring
// (S stages of C tiles, 128-byte aligned), the activation quants and d, the
// K-slice partials [C][8][16].
__host__ __device__ inline size_t tma_ring_offset(int S) { return ((size_t)16 * S + 16 + 127) & ~size_t(127); }
__host__ __device__ inline size_t tma_smem_bytes(int S, int K, int ncols, int C) {
  return tma_ring_offset(S) + (size_t)S * C * kTileBytes + (size_t)ncols * act_row_bytes(K) +
         (size_t)ncols * (K / kQK8) * 4 + (size_t)C * kMaxCols * kTileRows * 4;
}

template <int NCOLS>
__global__ void __launch_bounds__(13 * 32) mmvq_q6p_tma_kernel(const uint8_t* __restrict__ W,
                                                               int64_t rows, int K,
                                                               const uint8_t* __restrict__ xq,
                                                               float* __restrict__ y,
                                                               int32_t* __restrict__ sumi, int S) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int C = (int)(blockDim.x >> 5) - 1;  // consumer warps; warp C produces
  const int nb = K / kQK;
  const int nbq = K / kQK8;
  const int rb = act_row_bytes(K);
  const int64_t n_rg = (rows + kTileRows - 1) / kTileRows;

  const int spr = nb / C;  // stages per row group
  const size_t stage_bytes = (size_t)C * kTileBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + S;
  volatile int* fail = reinterpret_cast<volatile int*>(empty + S);
  uint8_t* ring = smem + tma_ring_offset(S);
  uint8_t* act = ring + (size_t)S * stage_bytes;
  float* da = reinterpret_cast<float*>(act + NCOLS * rb);
  float* red = da + NCOLS * nbq;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C);
    }
    *fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  grid_launch_dependents();

  // this CTA's row groups: blockIdx.x, + gridDim.x, ...
  const int64_t my_rgs = (blockIdx.x < n_rg) ? (n_rg - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int64_t total = my_rgs * spr;

  if (warp == C) {  // ------------------------------------------ producer
    if (lane == 0) {
      int64_t it = 0;
      for (; it < total; ++it) {
        const int s = (int)(it % S);
        const int64_t round = it / S;
        if (round > 0 && !*fail && !mbar_wait(&empty[s], (uint32_t)((round - 1) & 1))) {
          *fail = 1;
          atomicOr(&g_fault_word, kFaultMbarTimeout);
        }
        if (*fail) break;
        const int64_t rg = blockIdx.x + (it / spr) * gridDim.x;
        const int b0 = (int)(it % spr) * C;
        mbar_expect_tx(&full[s], (uint32_t)stage_bytes);
        bulk_g2s(ring + (size_t)s * stage_bytes, W + (rg * nb + b0) * kTileBytes,
                 (uint32_t)stage_bytes, &full[s]);
      }
      // no copy of this CTA may land after it exits: wait (bounded) for the
      // last phase of every slot that was filled
      const int64_t issued = it;
      for (int s = 0; s < S && s < issued; ++s) {
        const int64_t last = issued - 1 - ((issued - 1 - s) % S);
        mbar_wait(&full[s], (uint32_t)((last / S) & 1));
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int nthreads = 32 * C;
  const int tid = threadIdx.x;
  grid_dependency_wait();
  stage_q8_1(xq, K, NCOLS, [](int c) { return c; }, act, da, nullptr, tid, nthreads);
  consumer_sync(nthreads);

  const int i = lane & 15;
  const int h = lane >> 4;
  for (int64_t k = 0; k < my_rgs; ++k) {
    const int64_t rg = blockIdx.x + k * gridDim.x;
    const int64_t row = rg * kTileRows + i;
    int32_t* srow = (sumi && row < rows) ? sumi + row * nbq : nullptr;
    float acc[NCOLS];
#pragma unroll
    for (int c = 0; c < NCOLS; ++c) acc[c] = 0.0f;
    for (int j = 0; j < spr; ++j) {
      const int64_t it = k * spr + j;
      const int s = (int)(it % S);
      if (!*fail && !mbar_wait(&full[s], (uint32_t)((it / S) & 1))) {
        *fail = 1;
        atomicOr(&g_fault_word, kFaultMbarTimeout);
      }
      Q6Half w;
      load_q6_tile_smem(ring + (size_t)s * stage_bytes + (size_t)warp * kTileBytes, lane, w);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      q6_dot<NCOLS>(w, h, j * C + warp, act, rb, da, nbq, acc, srow, rows * nbq);
    }
    // halves of each row, then the K-slices in warp order
#pragma unroll
    for (int c = 0; c < NCOLS; ++c) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], 16);
    if (C == 1) {
      if (h == 0 && row < rows) {
#pragma unroll
        for (int c = 0; c < NCOLS; ++c) y[c * rows + row] = acc[c];
      }
      continue;
    }
    if (h == 0) {
#pragma unroll
      for (int c = 0; c < NCOLS; ++c) red[(warp * kMaxCols + c) * kTileRows + i] = acc[c];
    }
    consumer_sync(nthreads);
    if (warp == 0 && h == 0 && row < rows) {
#pragma unroll
      for (int c = 0; c < NCOLS; ++c) {
        float sum = 0.0f;
        for (int wq = 0; wq < C; ++wq) sum += red[(wq * kMaxCols + c) * kTileRows + i];
        y[c * rows + row] = sum;
      }
    }
    consumer_sync(nthreads);
  }
}

// ------------------------------------------------------------ host side ----

struct TmaCfg {
  int consumers, slots, grid;
  size_t smem;
};

// Consumers C: a divisor of K/256 (each row group's blocks split evenly),
// as many as possible up to 12 while the ring still holds two stages.  Ring
// depth: as many stages as fit in about 110 KB of shared memory (so this
// call's CTA and the next call's can share an SM), and at least two.
template <int NCOLS>
static int tma_config(int64_t rows, int K, TmaCfg* out) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, TmaCfg> cache;
  static size_t smem_set = 48 * 1024;
  const uint64_t key = ((uint64_t)rows << 8) | (uint64_t)(K / kQK);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *out = it->second;
      return MMVQ_OK;
    }
  }
  auto kern = mmvq_q6p_tma_kernel<NCOLS>;
  const int sms = device_sms();
  const size_t limit = max_smem_optin();
  if (sms <= 0 || limit == 0) return MMVQ_ERR_CUDA;
  const int nb = K / kQK;
  const size_t budget = std::min<size_t>(limit, 110 * 1024);
  int C = 0, S = 0;
  size_t smem = 0;
  for (int d = std::min(nb, 12); d >= 1 && C == 0; --d) {
    if (nb % d) continue;
    for (int s = 64; s >= 2; --s) {
      const size_t b = tma_smem_bytes(s, K, NCOLS, d);
      if (b <= budget || (s == 2 && b <= limit)) {
        C = d;
        S = s;
        smem = b;
        break;
      }
    }
  }
  if (C == 0) return MMVQ_ERR_SHAPE;
  if (ensure_smem((const void*)kern, smem, &smem_set, &mu) != MMVQ_OK) return MMVQ_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * (C + 1), smem) !=
          cudaSuccess ||
      per_sm < 1)
    return MMVQ_ERR_CUDA;
  const int64_t n_rg = (rows + kTileRows - 1) / kTileRows;
  TmaCfg cfg = {C, S, (int)std::min<int64_t>(n_rg, (int64_t)sms * per_sm), smem};
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = cfg;
  *out = cfg;
  return MMVQ_OK;
}

template <int NCOLS>
static int launch_tma_t(const uint8_t* W, int64_t rows, int K, const uint8_t* xq, float* y,
                        int32_t* sumi, cudaStream_t stream) {
  TmaCfg cfg;
  const int rc = tma_config<NCOLS>(rows, K, &cfg);
  if (rc != MMVQ_OK) return rc;
  return launch_pdl(mmvq_q6p_tma_kernel<NCOLS>, dim3(cfg.grid), dim3(32 * (cfg.consumers + 1)),
                    cfg.smem, stream, W, rows, K, xq, y, sumi, cfg.slots);
}

int launch_q6_planar_tma(const void* W, int64_t rows, int K, const void* xq, int ncols, float* y,
                         int32_t* sumi, cudaStream_t s) {
  const uint8_t* w = static_cast<const uint8_t*>(W);
  const uint8_t* x = static_cast<const uint8_t*>(xq);
  switch (ncols) {
    case 1: return launch_tma_t<1>(w, rows, K, x, y, sumi, s);
    case 2: return launch_tma_t<2>(w, rows, K, x, y, sumi, s);
    case 3: return launch_tma_t<3>(w, rows, K, x, y, sumi, s);
    case 4: return launch_tma_t<4>(w, rows, K, x, y, sumi, s);
    case 5: return launch_tma_t<5>(w, rows, K, x, y, sumi, s);
    case 6: return launch_tma_t<6>(w, rows, K, x, y, sumi, s);
    case 7: return launch_tma_t<7>(w, rows, K, x, y, sumi, s);
    case 8: return launch_tma_t<8>(w, rows, K, x, y, sumi, s);
  }
  return MMVQ_ERR_NCOLS;
}

// Reads and clears the device fault word (after synchronising `stream`).
int read_device_fault(int* fault, cudaStream_t stream) {
  unsigned int v = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MMVQ_ERR_CUDA;
  if (cudaMemcpyFromSymbol(&v, g_fault_word, sizeof(v)) != cudaSuccess) return MMVQ_ERR_CUDA;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(zero)) != cudaSuccess) return MMVQ_ERR_CUDA;
  *fault = (int)v;
  return MMVQ_OK;
}

}  // namespace mmvq
