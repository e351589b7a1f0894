// Planar (Q6_K, Q4_K and Q5_K tile) MMVQ fed by bulk copies (cp.async.bulk, the 1-D TMA path)
// into a shared-memory ring ("Strata" PR #2340 "STRATA_Q6_PLANAR": the head's
// planes are laid out so every lane load is one aligned 16-byte load; PR
// #2207: the weights are read once for all 1-8 columns).
//
// GB300 design.  One producer warp per CTA streams the CTA's weights from
// HBM into a ring of S stages; a stage holds, for each of the batch's G row
// groups, P consecutive tiles (16 rows x one 256-block each: 3360 bytes for
// Q6_K, 2304 for Q4_K, 2816 for Q5_K), one bulk copy per row group, one tile
// per consumer warp.  Each stage has a pair of mbarriers
// (full: bytes landed; empty: all C consumer warps have read it).  The bytes
// in flight per SM are set by the ring depth, not by how many warps hold
// loads in registers.  Every consumer warp walks every stage in order, so a
// warp waiting for round r of a slot has itself consumed round r-1 there and
// the parity wait cannot alias an older phase.  A warp copies its tile's
// lane bytes out of the ring with 16-byte shared loads (the tile order makes
// them conflict-free), releases the stage, decodes and accumulates with
// dp4a; the K-slices are summed in a fixed warp order.  For 4-8 columns,
// MMVQ_FLAG_TENSOR_CORE swaps in the tensor-core consumer of tma_mma.cuh
// (same tiles, same staging, same launch shape, same bits).
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

#include "tma_dense.cuh"

namespace mmvq {

// ------------------------------------------------- grouped (experts) ----
// Grouped expert MMVQ on the same ring ("Strata" PR #2746 "B70 validation":
// grouped calls over per-expert token groups, empty groups allowed; issue
// #2801: the grouped gate/up and down kernels).  Each CTA compacts the
// non-empty groups from the offsets (after the grid dependency: the lists
// come from the preceding kernel) and takes an equal contiguous range of
// items; an item is G consecutive row groups of one group's expert.  Per
// item and per chunk of up to CM positions a stage holds, for each of the G
// row groups, P consecutive tiles (one bulk copy each); consumer warp (g, p)
// takes row group g and the K-slice p.  Producer and consumers walk the same
// (item, chunk, stage) sequence, so their slot and phase counters agree.

constexpr int kMaxGroupsTma = 4096;

__host__ __device__ inline size_t grouped_smem_bytes(int layout, int S, int K, int CM, int G,
                                                     int P) {
  return tma_ring_offset(S) + (size_t)S * G * P * tile_bytes(layout) +
         (size_t)CM * act_row_bytes(K) + (size_t)CM * (K / kQK8) * 8 +
         (size_t)G * P * kMaxCols * kTileRows * 4;
}

template <int LAYOUT, int CM>
__global__ void __launch_bounds__(13 * 32) mmvq_grouped_tma_kernel(
    const uint8_t* __restrict__ W, int n_experts, int64_t rows, int K,
    const int32_t* __restrict__ expert_ids, const int32_t* __restrict__ offsets, int n_groups,
    const int32_t* __restrict__ act_index, const uint8_t* __restrict__ xq, int n_xq_cols,
    float* __restrict__ y, int32_t* __restrict__ status, int S, int G, int P) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int active[kMaxGroupsTma];
  __shared__ int warp_sums[17];
  __shared__ int cols_s[kMaxCols];
  constexpr int TB = tile_bytes(LAYOUT);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int C = G * P;
  const int nb = K / kQK;
  const int nbq = K / kQK8;
  const int rb = act_row_bytes(K);
  const int64_t n_rg = (rows + kTileRows - 1) / kTileRows;
  const int64_t n_rgb = (n_rg + G - 1) / G;
  const int spb = nb / P;
  const size_t slice_bytes = (size_t)P * TB;
  const int64_t expert_bytes = n_rg * nb * TB;

  GroupedRing r;
  r.full = reinterpret_cast<uint64_t*>(smem);
  r.empty = r.full + S;
  r.fail = reinterpret_cast<volatile int*>(r.empty + S);
  r.ring = smem + tma_ring_offset(S);
  r.stage_bytes = (size_t)G * slice_bytes;
  r.S = S;
  uint8_t* ring = smem + tma_ring_offset(S);
  uint8_t* act = ring + (size_t)S * r.stage_bytes;
  float* da = reinterpret_cast<float*>(act + (size_t)CM * rb);
  float* sa = da + CM * nbq;
  float* red = sa + CM * nbq;
  // debug build: the layout must fit the launch
  if (!MMVQ_SMEM_OK(smem, red + (size_t)C * kMaxCols * kTileRows)) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&r.full[s], 1);
      mbar_init(&r.empty[s], C);
    }
    *r.fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  grid_launch_dependents();
  grid_dependency_wait();

  // 1. compact the valid non-empty groups, in group order (all threads)
  const int per = (n_groups + (int)blockDim.x - 1) / (int)blockDim.x;
  const int g0 = threadIdx.x * per;
  const int g1 = min(n_groups, g0 + per);
  int cnt = 0;
  bool bad = false;
  for (int q = g0; q < g1; ++q) {
    const int e = expert_ids[q];
    const int o0 = offsets[q], o1 = offsets[q + 1];
    const bool ok = e >= 0 && e < n_experts && o0 >= 0 && o1 >= o0;
    bad |= !ok;
    cnt += (ok && o1 > o0) ? 1 : 0;
  }
  if (bad && status && blockIdx.x == 0) *status = MMVQ_ERR_ROUTING;
  int n_active = 0;
  int pos = block_scan_excl(cnt, warp_sums, &n_active);
  for (int q = g0; q < g1; ++q) {
    const int e = expert_ids[q];
    const int o0 = offsets[q], o1 = offsets[q + 1];
    if (e >= 0 && e < n_experts && o0 >= 0 && o1 > o0) active[pos++] = q;
  }
  __syncthreads();

  // 2. this CTA's contiguous share of the (group, row-group block) items
  const int64_t n_items = (int64_t)n_active * n_rgb;
  const int64_t it0 = n_items * blockIdx.x / gridDim.x;
  const int64_t it1 = n_items * (blockIdx.x + 1) / gridDim.x;
  if (it0 >= it1) return;
  int a = (int)(it0 / n_rgb);
  int64_t rgb = it0 - (int64_t)a * n_rgb;

  if (warp == C) {  // ------------------------------------------ producer
    if (lane == 0) {
      int slot = 0;
      uint32_t par = 0;
      int64_t issued = 0;
      for (int64_t it = it0; it < it1 && !*r.fail; ++it) {
        const int grp = active[a];
        const uint8_t* Wexp = W + (size_t)expert_ids[grp] * expert_bytes;
        const int64_t rg0 = rgb * G;
        const int nvalid = (int)min((int64_t)G, n_rg - rg0);
        const int pe = offsets[grp + 1];
        // debug build: the item's tiles lie inside its expert's weights
        if (!MMVQ_INDEX_OK(expert_ids[grp] >= 0 && expert_ids[grp] < n_experts && rg0 >= 0 &&
                           rg0 + nvalid <= n_rg && spb * P <= nb)) {
          *r.fail = 1;
          break;
        }
        for (int p0 = offsets[grp]; p0 < pe && !*r.fail; p0 += CM) {
          for (int bb = 0; bb < spb; ++bb) {
            if (issued >= S && !mbar_wait(&r.empty[slot], par ^ 1u, 128)) {
              *r.fail = 1;
              atomicOr(&g_fault_word, kFaultMbarTimeout);
              break;
            }
            mbar_expect_tx(&r.full[slot], (uint32_t)(nvalid * slice_bytes));
            uint8_t* dst = ring + (size_t)slot * r.stage_bytes;
            const uint8_t* src = Wexp + (rg0 * nb + (int64_t)bb * P) * TB;
            for (int g = 0; g < nvalid; ++g)
              bulk_g2s(dst + (size_t)g * slice_bytes, src + (int64_t)g * nb * TB,
                       (uint32_t)slice_bytes, &r.full[slot]);
            ++issued;
            if (++slot == S) {
              slot = 0;
              par ^= 1u;
            }
          }
        }
        if (++rgb == n_rgb) {
          rgb = 0;
          ++a;
        }
      }
      // wait (bounded) for the last phase of every filled slot
      for (int s = 0; s < S && s < issued; ++s) {
        const int64_t last = issued - 1 - ((issued - 1 - s) % S);
        mbar_wait(&r.full[s], (uint32_t)((last / S) & 1));
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int nthreads = 32 * C;
  const int g = warp / P;
  const int p = warp - g * P;
  int slot = 0;
  uint32_t par = 0;
  int staged_grp = -1, staged_p0 = -1;
  for (int64_t it = it0; it < it1; ++it) {
    const int grp = active[a];
    const int pe = offsets[grp + 1];
    const int64_t rg = rgb * G + g;
    const bool valid = rg < n_rg;
    for (int p0 = offsets[grp]; p0 < pe; p0 += CM) {
      const int n = min(CM, pe - p0);
      if (grp != staged_grp || p0 != staged_p0) {
        group_sync(1, nthreads);  // the previous columns are no longer read
        if (threadIdx.x < n) {
          const int col = act_index ? act_index[p0 + threadIdx.x] : p0 + threadIdx.x;
          const bool ok = col >= 0 && col < n_xq_cols;
          if (!ok && status) *status = MMVQ_ERR_ROUTING;
          cols_s[threadIdx.x] = ok ? col : -1;
        }
        group_sync(1, nthreads);
        // an invalid column is staged as zeros: its outputs come out 0
        stage_q8_1(xq, K, n, [&](int c) { return cols_s[c]; }, act, da,
                   LAYOUT == kQ4Planar ? sa : nullptr, threadIdx.x, nthreads);
        group_sync(1, nthreads);
        staged_grp = grp;
        staged_p0 = p0;
      }
      float* ybase = y + (size_t)p0 * rows;
#define MMVQ_GC(NC)                                                                           \
  grouped_consume<LAYOUT, NC>(r, slot, par, g, p, P, lane, spb, act, rb, da, sa, nbq, red, \
                              ybase, rg, valid, rows)
      if constexpr (CM == 1) {
        MMVQ_GC(1);
      } else if constexpr (CM == 2) {
        if (n == 1) MMVQ_GC(1); else MMVQ_GC(2);
      } else if constexpr (CM == 4) {
        switch (n) {
          case 1: MMVQ_GC(1); break;
          case 2: MMVQ_GC(2); break;
          case 3: MMVQ_GC(3); break;
          default: MMVQ_GC(4); break;
        }
      } else {
        switch (n) {
          case 1: MMVQ_GC(1); break;
          case 2: MMVQ_GC(2); break;
          case 3: MMVQ_GC(3); break;
          case 4: MMVQ_GC(4); break;
          case 5: MMVQ_GC(5); break;
          case 6: MMVQ_GC(6); break;
          case 7: MMVQ_GC(7); break;
          default: MMVQ_GC(8); break;
        }
      }
#undef MMVQ_GC
    }
    if (++rgb == n_rgb) {
      rgb = 0;
      ++a;
    }
  }
}

// ------------------------------------------------------------ host side ----

// Launch shape.  Candidates (G, P) with P | K/256 and C = G*P <= 12; the ring
// gets as many stages as fit in ~110 KB (two CTAs per SM when registers
// allow), at least two.  Cost model: a CTA's time is its batches x (stages
// per batch + the batch's K-slice reduction over P warps, (P-1)/18 of a
// stage), each stage one tile per consumer warp; the SM's issue rate is
// shared by all resident consumer warps once they exceed 20.  The cheapest
// shape wins; ties go to more consumer warps.  The two constants were fitted
// on GB300 to every (G, P) of the Q6_K 2560 x 2560, 2560 x 10240 and
// 10240 x 2560 calls at 1-8 columns, timed back to back and as a dependent
// chain: they pick G = 2, P = 5 over G = 1, P = 10 for 10240 x 2560 at 1-4
// columns (one batch per CTA instead of three), faster in both timings.
template <int LAYOUT, int NCOLS>
static int tma_config(int64_t rows, int K, TmaCfg* out) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, TmaCfg> cache;
  const uint64_t key = ((uint64_t)rows << 8) | (uint64_t)(K / kQK);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *out = it->second;
      return MMVQ_OK;
    }
  }
  auto kern = mmvq_planar_tma_kernel<LAYOUT, NCOLS, false, false, false>;
  const int sms = device_sms();
  const size_t limit = max_smem_optin();
  if (sms <= 0 || limit == 0) return MMVQ_ERR_CUDA;
  const int nb = K / kQK;
  const int64_t n_rg = (rows + kTileRows - 1) / kTileRows;
  const size_t budget = std::min<size_t>(limit, 110 * 1024);
  TmaCfg best = {0, 0, 0, 0, 0, 1};
  double best_cost = 1e300;
  int best_c = 0;
  // Very tall matrices (an LM head): one warp per row group (no K-split, no
  // barriers), a two-stage ring, several CTAs per SM.  Measured on GB300:
  // ~15% faster than the split-K shapes for 151936 x 2560.
  // At one column, four CTAs of four row groups per SM: a persistent CTA
  // takes a fixed share of the row groups, and CTAs finish up to ~17 us
  // apart in a 50 us head call (measured per CTA); with more, smaller
  // CTAs per SM the spread shrinks.  Measured for 151936 x 2560 at one
  // column: 44.8 / 47.0 us back to back / dependent, against 44.0 / 51.2 us
  // for seven row groups, three CTAs per SM, which stays best from two
  // columns on (a fourth CTA of seven row groups was ~6% slower there).
  const bool tall = n_rg >= (int64_t)16 * sms;
  if (tall) {
    const int g_top = NCOLS == 1 ? 4 : 7;
    const int per_cap = NCOLS == 1 ? 4 : 3;
    for (int G = g_top; G >= 1 && best.G == 0; --G) {
      const size_t smem = tma_smem_bytes(LAYOUT, 2, K, NCOLS, G, 1);
      if (smem > limit) continue;
      if (ensure_smem((const void*)kern, smem) != MMVQ_OK) return MMVQ_ERR_CUDA;
      int per_sm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * (G + 1), smem) !=
          cudaSuccess)
        return MMVQ_ERR_CUDA;
      if (per_sm < 1) continue;
      per_sm = std::min(per_sm, per_cap);
      const int64_t ctas = std::min<int64_t>((n_rg + G - 1) / G, (int64_t)sms * per_sm);
      best = {G, 1, 2, (int)ctas, smem, 1};
    }
  }
  const bool search = !tall || best.G == 0;
  for (int P = 1; P <= std::min(nb, 12) && search; ++P) {
    if (nb % P) continue;
    for (int G = 1; G * P <= 12; ++G) {
      int S = 0;
      size_t smem = 0;
      for (int s = 32; s >= 2; --s) {
        const size_t b = tma_smem_bytes(LAYOUT, s, K, NCOLS, G, P);
        if (b <= budget || (s == 2 && b <= limit)) {
          S = s;
          smem = b;
          break;
        }
      }
      if (S == 0) continue;
      if (ensure_smem((const void*)kern, smem) != MMVQ_OK) return MMVQ_ERR_CUDA;
      int per_sm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * (G * P + 1), smem) !=
          cudaSuccess)
        return MMVQ_ERR_CUDA;
      if (per_sm < 1) continue;
      const int64_t ctas = std::min<int64_t>((n_rg + G - 1) / G, (int64_t)sms * per_sm);
      const int64_t rgs_per_cta = (n_rg + ctas - 1) / ctas;
      const int64_t batches = (rgs_per_cta + G - 1) / G;
      const double ctas_per_sm = std::min<double>(per_sm, (double)ctas / sms);
      const double warps_per_sm = std::max(1.0, ctas_per_sm) * G * P;
      // stage time: one tile per warp, slowed once the SM holds > 20 warps
      const double stage = std::max(1.0, warps_per_sm / 20.0);
      const double cost = (double)batches * ((double)(nb / P) + (P - 1) / 18.0) * stage;
      if (cost < best_cost * 0.999 || (cost < best_cost * 1.001 && G * P > best_c)) {
        best_cost = cost;
        best_c = G * P;
        best = {G, P, S, (int)ctas, smem, 1};
      }
    }
  }
  if (best.G == 0) return MMVQ_ERR_SHAPE;
  // Six to eight columns of a long row (K >= 8192): the staged columns
  // (>= 72 KB) leave the ring two stages and one CTA per SM, and a matrix of
  // few row groups covers part of the GPU (2560 x 10240: 80 CTAs).  A K-split
  // over CTA pairs halves the staging and spreads each row group over two
  // SMs: three row groups of four K-slices per CTA.  Measured on GB300 for
  // 2560 x 10240 at 6 / 8 columns: 18.4 / 19.5 -> 13.1 / 14.5 us as a
  // dependent chain, 10.1 / 10.9 -> 9.9 / 11.0 us back to back.
  if (NCOLS >= 6 && nb >= 32 && (nb / 2) % 4 == 0 && best.grid < sms) {
    auto ckern = mmvq_planar_tma_kernel<LAYOUT, NCOLS, false, true, false>;
    const int G = 3, P = 4, CS = 2;
    int S = 0;
    size_t smem = 0;
    for (int s = 32; s >= 2; --s) {
      const size_t b = tma_smem_bytes(LAYOUT, s, K, NCOLS, G, P, CS);
      if (b <= budget || (s == 2 && b <= limit)) {
        S = s;
        smem = b;
        break;
      }
    }
    if (S >= 2) {
      if (ensure_smem((const void*)ckern, smem) != MMVQ_OK) return MMVQ_ERR_CUDA;
      cudaLaunchConfig_t lc = {};
      lc.blockDim = dim3(32 * (G * P + 1));
      lc.gridDim = dim3(2 * sms);
      lc.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = CS;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      lc.attrs = attr;
      lc.numAttrs = 1;
      int max_cl = 0;
      if (cudaOccupancyMaxActiveClusters(&max_cl, (void*)ckern, &lc) == cudaSuccess && max_cl >= 1) {
        const int64_t n_batch = (n_rg + G - 1) / G;
        const int64_t ncl = std::min<int64_t>(n_batch, max_cl);
        best = {G, P, S, (int)(ncl * CS), smem, CS};
      }
    }
  }
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = best;
  *out = best;
  return MMVQ_OK;
}

// A launch shape the kernel can run: a ring of at least two stages, at most
// 12 consumer warps, CS | K/256 and P | (K/256)/CS, a grid of whole clusters
// of 1-8 CTAs, and the shared memory the shape needs.
static bool tma_shape_ok(const TmaCfg& c, int K, int layout, int ncols, bool mma) {
  const int nb = K / kQK;
  if (c.slots < 2 || c.G < 1 || c.P < 1 || c.G * c.P > 12) return false;
  if (c.CS < 1 || c.CS > 8) return false;
  if (nb % c.CS != 0 || (nb / c.CS) % c.P != 0 || c.grid < c.CS || c.grid % c.CS != 0) return false;
  return c.smem >= tma_smem_bytes(layout, c.slots, K, ncols, c.G, c.P, c.CS, mma) &&
         c.smem <= max_smem_optin();
}

// The instance that also stores the per-block sums runs in the product
// instance's launch shape, so y comes out with the same bits.
template <int LAYOUT, int NCOLS, bool SUMI, bool MMA>
static int launch_tma_cfg_k(const uint8_t* W, int64_t rows, int K, const uint8_t* xq, float* y,
                            int32_t* sumi, const TmaCfg& cfg, uint32_t flags,
                            cudaStream_t stream) {
  if (!tma_shape_ok(cfg, K, LAYOUT, NCOLS, MMA)) return MMVQ_ERR_SHAPE;
  if (cfg.CS == 1) {
    auto kern = mmvq_planar_tma_kernel<LAYOUT, NCOLS, SUMI, false, false, MMA>;
    if (ensure_smem((const void*)kern, cfg.smem) != MMVQ_OK) return MMVQ_ERR_CUDA;
    return launch_pdl(kern, dim3(cfg.grid), dim3(32 * (cfg.G * cfg.P + 1)), cfg.smem, stream, W,
                      rows, K, xq, y, sumi, cfg.slots, cfg.G, cfg.P, 1, flags,
                      static_cast<const float*>(nullptr), (int64_t)0,
                      static_cast<uint8_t*>(nullptr));
  }
  auto kern = mmvq_planar_tma_kernel<LAYOUT, NCOLS, SUMI, true, false, MMA>;
  if (ensure_smem((const void*)kern, cfg.smem) != MMVQ_OK) return MMVQ_ERR_CUDA;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(cfg.grid);
  lc.blockDim = dim3(32 * (cfg.G * cfg.P + 1));
  lc.dynamicSmemBytes = cfg.smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)cfg.CS;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 2;
  return cudaLaunchKernelEx(&lc, kern, W, rows, K, xq, y, sumi, cfg.slots, cfg.G, cfg.P, cfg.CS,
                            flags, static_cast<const float*>(nullptr), (int64_t)0,
                            static_cast<uint8_t*>(nullptr)) == cudaSuccess
             ? MMVQ_OK
             : MMVQ_ERR_CUDA;
}

// The consumer of the shape (cfg.mma, set by the explicit-shape entry), or
// with MMVQ_FLAG_TENSOR_CORE the tensor-core one in the chosen shape, its
// table added to the shared memory where that still fits (the dp4a
// consumer otherwise: same sums, same bits).
template <int LAYOUT, int NCOLS, bool SUMI>
static int launch_tma_cfg(const uint8_t* W, int64_t rows, int K, const uint8_t* xq, float* y,
                          int32_t* sumi, const TmaCfg& cfg, uint32_t flags, cudaStream_t stream) {
  if constexpr (NCOLS >= kMmaMinCols) {
    if (cfg.mma)
      return launch_tma_cfg_k<LAYOUT, NCOLS, SUMI, true>(W, rows, K, xq, y, sumi, cfg, flags,
                                                         stream);
    if (flags & MMVQ_FLAG_TENSOR_CORE) {
      TmaCfg m = cfg;
      m.smem = tma_smem_bytes(LAYOUT, cfg.slots, K, NCOLS, cfg.G, cfg.P, cfg.CS, true);
      m.mma = 1;
      if (m.smem <= max_smem_optin())
        return launch_tma_cfg_k<LAYOUT, NCOLS, SUMI, true>(W, rows, K, xq, y, sumi, m, flags,
                                                           stream);
    }
  } else {
    if (cfg.mma) return MMVQ_ERR_SHAPE;
  }
  return launch_tma_cfg_k<LAYOUT, NCOLS, SUMI, false>(W, rows, K, xq, y, sumi, cfg, flags, stream);
}

template <int LAYOUT, int NCOLS, bool SUMI>
static int launch_tma_s(const uint8_t* W, int64_t rows, int K, const uint8_t* xq, float* y,
                        int32_t* sumi, uint32_t flags, cudaStream_t stream) {
  TmaCfg cfg;
  const int rc = tma_config<LAYOUT, NCOLS>(rows, K, &cfg);
  if (rc != MMVQ_OK) return rc;
  return launch_tma_cfg<LAYOUT, NCOLS, SUMI>(W, rows, K, xq, y, sumi, cfg, flags, stream);
}

template <int LAYOUT, int NCOLS>
static int launch_tma_t(const uint8_t* W, int64_t rows, int K, const uint8_t* xq, float* y,
                        int32_t* sumi, uint32_t flags, cudaStream_t stream) {
  if (sumi) return launch_tma_s<LAYOUT, NCOLS, true>(W, rows, K, xq, y, sumi, flags, stream);
  return launch_tma_s<LAYOUT, NCOLS, false>(W, rows, K, xq, y, sumi, flags, stream);
}

template <int LAYOUT>
static int launch_tma_layout(const uint8_t* w, int64_t rows, int K, const uint8_t* x, int ncols,
                             float* y, int32_t* sumi, uint32_t flags, cudaStream_t s) {
  switch (ncols) {
    case 1: return launch_tma_t<LAYOUT, 1>(w, rows, K, x, y, sumi, flags, s);
    case 2: return launch_tma_t<LAYOUT, 2>(w, rows, K, x, y, sumi, flags, s);
    case 3: return launch_tma_t<LAYOUT, 3>(w, rows, K, x, y, sumi, flags, s);
    case 4: return launch_tma_t<LAYOUT, 4>(w, rows, K, x, y, sumi, flags, s);
    case 5: return launch_tma_t<LAYOUT, 5>(w, rows, K, x, y, sumi, flags, s);
    case 6: return launch_tma_t<LAYOUT, 6>(w, rows, K, x, y, sumi, flags, s);
    case 7: return launch_tma_t<LAYOUT, 7>(w, rows, K, x, y, sumi, flags, s);
    case 8: return launch_tma_t<LAYOUT, 8>(w, rows, K, x, y, sumi, flags, s);
  }
  return MMVQ_ERR_NCOLS;
}

int launch_planar_tma(int type, const void* W, int64_t rows, int K, const void* xq, int ncols,
                      float* y, int32_t* sumi, uint32_t flags, cudaStream_t s) {
  const uint8_t* w = static_cast<const uint8_t*>(W);
  const uint8_t* x = static_cast<const uint8_t*>(xq);
  if (type == MMVQ_Q4_K_PLANAR)
    return launch_tma_layout<kQ4Planar>(w, rows, K, x, ncols, y, sumi, flags, s);
  if (type == MMVQ_Q5_K_PLANAR)
    return launch_tma_layout<kQ5Planar>(w, rows, K, x, ncols, y, sumi, flags, s);
  return launch_tma_layout<kQ6Planar>(w, rows, K, x, ncols, y, sumi, flags, s);
}

template <int LAYOUT>
static int launch_tma_cfg_l(const uint8_t* w, int64_t rows, int K, const uint8_t* x, int ncols,
                            float* y, int32_t* sumi, const TmaCfg& c, uint32_t flags,
                            cudaStream_t s) {
#define MMVQ_TC(N)                                                                         \
  return sumi ? launch_tma_cfg<LAYOUT, N, true>(w, rows, K, x, y, sumi, c, flags, s)     \
              : launch_tma_cfg<LAYOUT, N, false>(w, rows, K, x, y, sumi, c, flags, s)
  switch (ncols) {
    case 1: MMVQ_TC(1);
    case 2: MMVQ_TC(2);
    case 3: MMVQ_TC(3);
    case 4: MMVQ_TC(4);
    case 5: MMVQ_TC(5);
    case 6: MMVQ_TC(6);
    case 7: MMVQ_TC(7);
    case 8: MMVQ_TC(8);
  }
#undef MMVQ_TC
  return MMVQ_ERR_NCOLS;
}

// The ring kernel in an explicit launch shape (G, P, stages, CS, grid), with
// the shared memory the shape needs; the shape is checked as the chooser's.
int launch_planar_tma_shape(int type, const void* W, int64_t rows, int K, const void* xq,
                            int ncols, float* y, int32_t* sumi, int G, int P, int S, int CS,
                            int grid, int mma, uint32_t flags, cudaStream_t s) {
  const int layout =
      type == MMVQ_Q4_K_PLANAR ? kQ4Planar : type == MMVQ_Q5_K_PLANAR ? kQ5Planar : kQ6Planar;
  if (G < 1 || P < 1 || S < 2 || CS < 1 || CS > 8) return MMVQ_ERR_SHAPE;
  if (mma && ncols < kMmaMinCols) return MMVQ_ERR_SHAPE;
  TmaCfg c = {G, P, S, grid, tma_smem_bytes(layout, S, K, ncols, G, P, CS, mma != 0), CS,
              mma ? 1 : 0};
  const uint8_t* w = static_cast<const uint8_t*>(W);
  const uint8_t* x = static_cast<const uint8_t*>(xq);
  if (layout == kQ4Planar) return launch_tma_cfg_l<kQ4Planar>(w, rows, K, x, ncols, y, sumi, c, flags, s);
  if (layout == kQ5Planar) return launch_tma_cfg_l<kQ5Planar>(w, rows, K, x, ncols, y, sumi, c, flags, s);
  return launch_tma_cfg_l<kQ6Planar>(w, rows, K, x, ncols, y, sumi, c, flags, s);
}

template <int LAYOUT>
static int tma_config_l(int64_t rows, int K, int ncols, TmaCfg* out) {
  switch (ncols) {
    case 1: return tma_config<LAYOUT, 1>(rows, K, out);
    case 2: return tma_config<LAYOUT, 2>(rows, K, out);
    case 3: return tma_config<LAYOUT, 3>(rows, K, out);
    case 4: return tma_config<LAYOUT, 4>(rows, K, out);
    case 5: return tma_config<LAYOUT, 5>(rows, K, out);
    case 6: return tma_config<LAYOUT, 6>(rows, K, out);
    case 7: return tma_config<LAYOUT, 7>(rows, K, out);
    case 8: return tma_config<LAYOUT, 8>(rows, K, out);
  }
  return MMVQ_ERR_NCOLS;
}

int planar_tma_config(int type, int64_t rows, int K, int ncols, TmaCfg* out) {
  if (type == MMVQ_Q4_K_PLANAR) return tma_config_l<kQ4Planar>(rows, K, ncols, out);
  if (type == MMVQ_Q5_K_PLANAR) return tma_config_l<kQ5Planar>(rows, K, ncols, out);
  return tma_config_l<kQ6Planar>(rows, K, ncols, out);
}

template <int LAYOUT, int NCOLS>
static int tma_shape_t(int64_t rows, int K, int32_t* info) {
  TmaCfg cfg;
  const int rc = tma_config<LAYOUT, NCOLS>(rows, K, &cfg);
  if (rc != MMVQ_OK) return rc;
  info[0] = cfg.grid;
  info[1] = 32 * (cfg.G * cfg.P + 1);
  info[2] = (int32_t)cfg.smem;
  info[3] = cfg.G;
  info[4] = cfg.P;
  info[5] = cfg.slots;
  info[6] = cfg.CS;
  return MMVQ_OK;
}

template <int LAYOUT>
static int tma_shape_layout(int64_t rows, int K, int ncols, int32_t* info) {
  switch (ncols) {
    case 1: return tma_shape_t<LAYOUT, 1>(rows, K, info);
    case 2: return tma_shape_t<LAYOUT, 2>(rows, K, info);
    case 3: return tma_shape_t<LAYOUT, 3>(rows, K, info);
    case 4: return tma_shape_t<LAYOUT, 4>(rows, K, info);
    case 5: return tma_shape_t<LAYOUT, 5>(rows, K, info);
    case 6: return tma_shape_t<LAYOUT, 6>(rows, K, info);
    case 7: return tma_shape_t<LAYOUT, 7>(rows, K, info);
    case 8: return tma_shape_t<LAYOUT, 8>(rows, K, info);
  }
  return MMVQ_ERR_NCOLS;
}

int planar_tma_shape(int type, int64_t rows, int K, int ncols, int32_t* info) {
  if (type == MMVQ_Q4_K_PLANAR) return tma_shape_layout<kQ4Planar>(rows, K, ncols, info);
  if (type == MMVQ_Q5_K_PLANAR) return tma_shape_layout<kQ5Planar>(rows, K, ncols, info);
  return tma_shape_layout<kQ6Planar>(rows, K, ncols, info);
}


// ------------------------------------------------------ grouped launch ----

struct GroupedCfg {
  int G, P, S, per_sm;
  size_t smem;
};

// Launch shape for the grouped ring kernel.  The number of non-empty groups
// is only known on the device; `est_active` is an estimate from the call's
// sizes, and R = est_active x row groups the work it implies.  Rules, from
// sweeps of G, P and S on GB300 over the gate|up and down shapes of a
// 256-expert MoE at 1-8 tokens:
//  * P = 1 (whole rows per warp, no reduction) once R >= 8 x SMs, else the
//    smallest divisor of K/256 above 1, so that enough warps are busy;
//  * if some G <= 12 / P puts every item in one CTA per SM, the smallest
//    such G with a ring as deep as fits (at most 6 stages): one wave, the
//    most bytes in flight per SM;
//  * otherwise G = 4 (at most 12 / P) and 3 stages, so that several CTAs
//    share each SM.
template <int LAYOUT, int CM>
static int grouped_config(int64_t rows, int K, int64_t est_active, GroupedCfg* out) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, GroupedCfg> cache;
  const uint64_t key = ((uint64_t)rows << 28) | ((uint64_t)(K / kQK) << 16) | (uint64_t)est_active;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *out = it->second;
      return MMVQ_OK;
    }
  }
  auto kern = mmvq_grouped_tma_kernel<LAYOUT, CM>;
  const int sms = device_sms();
  const size_t static_smem = (size_t)(kMaxGroupsTma + 17 + kMaxCols) * sizeof(int);
  const size_t optin = max_smem_optin();
  if (sms <= 0 || optin <= static_smem) return MMVQ_ERR_CUDA;
  const size_t limit = optin - static_smem;
  const int nb = K / kQK;
  const int64_t n_rg = (rows + kTileRows - 1) / kTileRows;
  const int64_t R = est_active * n_rg;
  int P = 1;
  if (R < (int64_t)8 * sms)
    for (int d = 2; d <= std::min(nb, 12); ++d)
      if (nb % d == 0) {
        P = d;
        break;
      }
  int G = 0, S = 3;
  for (int g = 1; g * P <= 12; ++g)
    if (est_active * ((n_rg + g - 1) / g) <= sms) {
      G = g;
      S = 6;
      break;
    }
  if (G == 0) G = std::max(1, std::min(4, 12 / P));
  // long rows with 8-position chunks: fewer stages, then fewer row groups
  // and K-slices per stage, until the ring fits beside the activations
  while (grouped_smem_bytes(LAYOUT, S, K, CM, G, P) > limit) {
    if (S > 2) {
      --S;
    } else if (G > 1) {
      --G;
    } else if (P > 1) {
      int d = P - 1;
      while (d > 1 && nb % d) --d;
      P = d;
    } else {
      break;
    }
  }
  const size_t smem = grouped_smem_bytes(LAYOUT, S, K, CM, G, P);
  if (smem > limit) return MMVQ_ERR_SHAPE;
  if (ensure_smem((const void*)kern, smem) != MMVQ_OK) return MMVQ_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * (G * P + 1), smem) !=
          cudaSuccess ||
      per_sm < 1)
    return MMVQ_ERR_CUDA;
  const GroupedCfg best = {G, P, S, per_sm, smem};
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = best;
  *out = best;
  return MMVQ_OK;
}

// CM, the positions per pass, is min(8, n_xq_cols) rounded up to 1, 2, 4
// or 8 (one kernel instance each): a group rarely holds more positions than
// there are activation columns, and a larger one is simply processed in
// more passes.  Active groups are estimated as min(n_groups, n_xq_cols)
// when the positions index the columns directly, else
// min(n_groups, 8 n_xq_cols) (a top-8 routing of n_xq_cols tokens); the
// estimate only steers the shape.
template <int LAYOUT, int CM>
static int launch_grouped_tma_cm(const uint8_t* W, int n_experts, int64_t rows, int K,
                                 const int32_t* expert_ids, const int32_t* offsets, int n_groups,
                                 const int32_t* act_index, const uint8_t* xq, int n_xq_cols,
                                 float* y, int32_t* status, cudaStream_t stream) {
  const int64_t est_active = std::max<int64_t>(
      1, std::min<int64_t>(n_groups, act_index ? (int64_t)8 * n_xq_cols : (int64_t)n_xq_cols));
  GroupedCfg cfg;
  const int rc = grouped_config<LAYOUT, CM>(rows, K, est_active, &cfg);
  if (rc != MMVQ_OK) return rc;
  const int64_t n_rg = (rows + kTileRows - 1) / kTileRows;
  const int64_t max_items = (int64_t)n_groups * ((n_rg + cfg.G - 1) / cfg.G);
  const int grid = (int)std::max<int64_t>(
      1, std::min<int64_t>(max_items, (int64_t)device_sms() * cfg.per_sm));
  return launch_pdl(mmvq_grouped_tma_kernel<LAYOUT, CM>, dim3(grid),
                    dim3(32 * (cfg.G * cfg.P + 1)), cfg.smem, stream, W, n_experts, rows, K,
                    expert_ids, offsets, n_groups, act_index, xq, n_xq_cols, y, status, cfg.S,
                    cfg.G, cfg.P);
}

template <int LAYOUT>
static int launch_grouped_tma_t(const uint8_t* W, int n_experts, int64_t rows, int K,
                                const int32_t* expert_ids, const int32_t* offsets, int n_groups,
                                const int32_t* act_index, const uint8_t* xq, int n_xq_cols,
                                float* y, int32_t* status, cudaStream_t s) {
  if (n_xq_cols <= 1)
    return launch_grouped_tma_cm<LAYOUT, 1>(W, n_experts, rows, K, expert_ids, offsets,
                                            n_groups, act_index, xq, n_xq_cols, y, status, s);
  if (n_xq_cols == 2)
    return launch_grouped_tma_cm<LAYOUT, 2>(W, n_experts, rows, K, expert_ids, offsets,
                                            n_groups, act_index, xq, n_xq_cols, y, status, s);
  if (n_xq_cols <= 4)
    return launch_grouped_tma_cm<LAYOUT, 4>(W, n_experts, rows, K, expert_ids, offsets,
                                            n_groups, act_index, xq, n_xq_cols, y, status, s);
  return launch_grouped_tma_cm<LAYOUT, 8>(W, n_experts, rows, K, expert_ids, offsets, n_groups,
                                          act_index, xq, n_xq_cols, y, status, s);
}

int launch_grouped_tma(int type, const void* W, int n_experts, int64_t rows, int K,
                       const int32_t* expert_ids, const int32_t* offsets, int n_groups,
                       const int32_t* act_index, const void* xq, int n_xq_cols, float* y,
                       int32_t* status, cudaStream_t s) {
  const uint8_t* w = static_cast<const uint8_t*>(W);
  const uint8_t* x = static_cast<const uint8_t*>(xq);
  if (type == MMVQ_Q4_K_PLANAR)
    return launch_grouped_tma_t<kQ4Planar>(w, n_experts, rows, K, expert_ids, offsets, n_groups,
                                           act_index, x, n_xq_cols, y, status, s);
  return launch_grouped_tma_t<kQ6Planar>(w, n_experts, rows, K, expert_ids, offsets, n_groups,
                                         act_index, x, n_xq_cols, y, status, s);
}

// Self-test of the bounded waits: one warp waits on a shared-memory barrier
// that nothing completes, with the kernels' own wait routine and a short
// limit, and reports the timeout through the fault word as they do.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0u, 0, limit_ns))
    atomicOr(&g_fault_word, kFaultMbarTimeout);
}

int launch_wait_timeout_selftest(uint32_t limit_us, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>((uint64_t)limit_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? MMVQ_OK : MMVQ_ERR_CUDA;
}

int read_clear_ffn_fault_word(unsigned int* v);
int read_clear_f32_fault_word(unsigned int* v);

// Reads and clears the device fault words of the ring kernels and of the
// expert layer (after synchronising `stream`); returns their OR.
int read_device_fault(int* fault, cudaStream_t stream) {
  unsigned int a = 0, b = 0, c = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MMVQ_ERR_CUDA;
  if (read_clear_fault_word(&a) != MMVQ_OK || read_clear_ffn_fault_word(&b) != MMVQ_OK ||
      read_clear_f32_fault_word(&c) != MMVQ_OK)
    return MMVQ_ERR_CUDA;
  *fault = (int)(a | b | c);
  return MMVQ_OK;
}

}  // namespace mmvq
