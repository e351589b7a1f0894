// The bulk-copy ring shared by the MMVQ kernels: mbarrier helpers with
// bounded waits, 1-D bulk copies (cp.async.bulk) into shared memory, the
// planar tile loads out of a ring slot, the ring's shared-memory layout, and
// the grouped-expert consume routine (one item and chunk for one consumer
// warp).  Included by each translation unit that runs a ring kernel.
#pragma once
#include "kquant.cuh"

namespace mmvq {

int device_sms();
size_t max_smem_optin();
int ensure_smem(const void* kern, size_t smem);

// The device fault word of the translation unit that includes this header
// (each unit has its own; mmvq_read_device_fault reads and clears them all).
static __device__ unsigned int g_fault_word = 0;

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per wait
constexpr int kFaultMbarTimeout = 1;

// Debug build (compiled with MMVQ_CHECKED, libmmvq_checked.so): device-side
// index checks in the ring kernels.  Each check tests an index or an extent
// against the bounds of its buffer: the kernel's shared-memory layout
// against the dynamic shared memory it was launched with, every bulk copy's
// source range against the weights' extent, every tile a consumer reads
// against the ring, every K-block it uses against the staged columns.  A
// failed check sets bit 4 of this translation unit's fault word (read with
// mmvq_read_device_fault), and the kernel skips the access and stops its
// ring (whose bounded waits then end it): no trap, the context stays usable.
// In the product build every check is the constant true and compiles away.
constexpr int kFaultIndexCheck = 4;
#ifdef MMVQ_CHECKED
__device__ __forceinline__ bool index_ok(bool ok) {
  if (!ok) atomicOr(&g_fault_word, kFaultIndexCheck);
  return ok;
}
__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
  uint32_t r;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(r));
  return r;
}
// MMVQ_SMEM_OK(base, end): [base, end) lies inside the launch's dynamic
// shared memory (base: its start).
#define MMVQ_INDEX_OK(cond) ::mmvq::index_ok(cond)
#define MMVQ_SMEM_OK(base, end) \
  ::mmvq::index_ok((size_t)((const uint8_t*)(end) - (const uint8_t*)(base)) <= \
                   (size_t)::mmvq::dynamic_smem_bytes())
#else
#define MMVQ_INDEX_OK(cond) true
#define MMVQ_SMEM_OK(base, end) true
#endif

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
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Waits for the phase with the given parity to complete; false once
// `limit_ns` (about 1 s by default) has passed.  The timer is read once every
// 64 tries; `backoff_ns` > 0 sleeps between tries (the producer, whose waits
// are not on the critical path).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int backoff_ns = 0,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = 0;
  for (uint32_t i = 1;; ++i) {
    if (backoff_ns) __nanosleep(backoff_ns);
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      const uint64_t t = global_ns();
      if (t0 == 0) {
        t0 = t;
      } else if (t - t0 > limit_ns) {
        return false;
      }
    }
  }
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---- thread-block clusters (the dense kernel's K-split over CTAs) ----
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The shared::cluster address of `p` (a shared variable of this CTA) in
// the CTA of the cluster with the given rank.
__device__ __forceinline__ uint32_t cluster_map(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  return a;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// Arrival on an mbarrier of another CTA of the cluster; release at cluster
// scope, so this thread's earlier stores into that CTA are visible to a
// thread whose wait observes the phase.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// mbar_wait with acquire at cluster scope (arrivals from other CTAs).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  uint64_t t0 = 0;
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 63u) == 0) {
      const uint64_t t = global_ns();
      if (t0 == 0) {
        t0 = t;
      } else if (t - t0 > limit_ns) {
        return false;
      }
    }
  }
}
// All threads of every CTA of the cluster (used once, after the mbarriers
// are initialised and before any CTA touches another's shared memory).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
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
// (S stages of G*P tiles, 128-byte aligned), the activation quants, d_a as
// floats, the K-slice partials [C][8][16].
__host__ __device__ inline size_t tma_ring_offset(int S) { return ((size_t)16 * S + 16 + 127) & ~size_t(127); }
// Layouts whose blocks carry a min term (d*sc*q - dmin*m): the Q8_1 sums s
// are staged beside d.
__host__ __device__ constexpr bool has_min(int layout) {
  return layout == kQ4Planar || layout == kQ5Planar;
}
__host__ __device__ constexpr int tile_bytes(int layout) {
  return layout == kQ4Planar ? kTileBytesQ4 : layout == kQ5Planar ? kTileBytesQ5 : kTileBytes;
}
// With a K-split over a cluster of CS CTAs each stages K/CS of the
// activations and holds the exchange buffers [2][CS][G][ncols][16] floats
// and two pairs of mbarriers.  mma: the tensor-core consumer's table of
// 32 floats per 32-block (tma_mma.cuh).  The K-slice partials [C][8][16]
// floats are double-buffered when P > 1.
__host__ __device__ inline size_t tma_smem_bytes(int layout, int S, int K, int ncols, int G, int P,
                                                 int CS = 1, bool mma = false) {
  const int C = G * P;
  const int Kc = K / CS;
  const size_t cols = (size_t)ncols * act_row_bytes(Kc) +
                      (size_t)ncols * (Kc / kQK8) * 4 * (has_min(layout) ? 2 : 1) +
                      (mma ? (size_t)(Kc / kQK8) * 32 * 4 : 0);
  return tma_ring_offset(S) + (size_t)S * C * tile_bytes(layout) + cols +
         (size_t)C * kMaxCols * kTileRows * 4 * (P > 1 ? 2 : 1) +
         (CS > 1 ? (size_t)2 * CS * G * ncols * kTileRows * 4 + 32 : 0);
}

__device__ __forceinline__ void group_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ int block_scan_excl(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int w = 0; w < nwarps; ++w) {
      const int t = warp_sums[w];
      warp_sums[w] = run;
      run += t;
    }
    warp_sums[nwarps] = run;
  }
  __syncthreads();
  const int out = warp_sums[warp] + x - v;
  *total = warp_sums[nwarps];
  __syncthreads();
  return out;
}

struct GroupedRing {
  const uint8_t* ring;
  size_t stage_bytes;
  uint64_t* full;
  uint64_t* empty;
  volatile int* fail;
  int S;
};

// One (item, chunk) for consumer warp (g, p): row group rg, K-slice p.
template <int LAYOUT, int NC>
__device__ __forceinline__ void grouped_consume(const GroupedRing& r, int& slot, uint32_t& par,
                                                int g, int p, int P, int lane, int spb,
                                                const uint8_t* act, int rb, const float* da,
                                                const float* sa, int nbq, float* red,
                                                float* ybase, int64_t rg, bool valid,
                                                int64_t rows) {
  constexpr int TB = tile_bytes(LAYOUT);
  const int i = lane & 15;
  const int h = lane >> 4;
  float acc[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) acc[c] = 0.0f;
  const size_t tile_off = (size_t)(g * P + p) * TB;
  for (int bb = 0; bb < spb; ++bb) {
    const int s = slot;
    if (!*r.fail && !mbar_wait(&r.full[s], par)) {
      *r.fail = 1;
      atomicOr(&g_fault_word, kFaultMbarTimeout);
    }
    if (++slot == r.S) {
      slot = 0;
      par ^= 1u;
    }
    // a row group past the end reads a stale (in-bounds) tile and stores nothing
    const uint8_t* tile = r.ring + (size_t)s * r.stage_bytes + tile_off;
    // debug build: the tile lies in the ring, its K-block in the staging
    const bool in = MMVQ_INDEX_OK(s < r.S && tile_off + TB <= r.stage_bytes && bb * P + p < nbq / 8);
    if (LAYOUT == kQ4Planar) {
      Q4Half w;
      if (in) load_q4_tile_smem(tile, lane, w);
      __syncwarp();
      if (lane == 0) mbar_arrive(&r.empty[s]);
      if (valid && in) q4_dot<NC>(w, h, bb * P + p, act, rb, da, sa, nbq, acc, nullptr, 0);
    } else {
      Q6Half w;
      if (in) load_q6_tile_smem(tile, lane, w);
      __syncwarp();
      if (lane == 0) mbar_arrive(&r.empty[s]);
      if (valid && in) q6_dot<NC>(w, h, bb * P + p, act, rb, da, nbq, acc, nullptr, 0);
    }
  }
#pragma unroll
  for (int c = 0; c < NC; ++c) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], 16);
  const int64_t row = rg * kTileRows + i;
  if (P == 1) {
    if (valid && h == 0 && row < rows) {
#pragma unroll
      for (int c = 0; c < NC; ++c) ybase[c * rows + row] = acc[c];
    }
    return;
  }
  float* rg_red = red + (size_t)g * P * kMaxCols * kTileRows;
  if (h == 0) {
#pragma unroll
    for (int c = 0; c < NC; ++c) rg_red[(p * kMaxCols + c) * kTileRows + i] = acc[c];
  }
  group_sync(2 + g, 32 * P);
  if (p == 0 && valid && h == 0 && row < rows) {
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      float sum = 0.0f;
      for (int q = 0; q < P; ++q) sum += rg_red[(q * kMaxCols + c) * kTileRows + i];
      ybase[c * rows + row] = sum;
    }
  }
  group_sync(2 + g, 32 * P);
}

// Reads and clears this translation unit's fault word (the caller has
// synchronised the stream).
static inline int read_clear_fault_word(unsigned int* v) {
  if (cudaMemcpyFromSymbol(v, g_fault_word, sizeof(*v)) != cudaSuccess) return MMVQ_ERR_CUDA;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(zero)) != cudaSuccess) return MMVQ_ERR_CUDA;
  return MMVQ_OK;
}

}  // namespace mmvq
