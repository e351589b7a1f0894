// The routed-expert FFN of one MoE layer in one cooperative launch: Q8_1 of
// the hidden states, the per-expert token lists, the grouped gate|up MMVQ,
// SiLU(gate)*up requantised to Q8_1, and the grouped down MMVQ ("Strata" PR
// #2746 "B70 validation": grouped calls over per-expert token groups; issue
// #2801: the grouped gate/up and down kernels and the activation between
// them).  Each step computes exactly what its separate entry point computes
// (the same device routines); only the schedule differs.
//
// GB300 design.  A cooperative launch (every CTA resident): one CTA per SM
// with 12 consumer warps, or three per SM with 4 each, plus one producer
// warp per CTA, on the bulk-copy ring of the grouped kernel.
//  - Every CTA builds the token lists itself, in shared memory, from topk
//    (a few hundred slots at most), so its producer starts the gate|up
//    weight stream at once; CTA 0 also publishes the lists.
//  - One or two tokens: every CTA quantises the hidden states itself into
//    its own staging, one 32-block per four lanes (values loaded by volatile
//    loads at entry, so they arrive before the CTA's weight stream starts;
//    the division done as a checked reciprocal multiply with the same bytes
//    as the IEEE quotient), so no grid barrier precedes gate|up; CTA 0 also
//    writes xq.  Three or more tokens: the hidden states are quantised to
//    Q8_1 by all consumer warps of the grid, one 32-block each, into the
//    caller's xq, behind a grid barrier; a CTA stages a group's columns from
//    there (through L2) when the group changes.
//  - The producer streams the CTA's gate|up items and then, through the same
//    ring, its down items: the down weights are in flight while the
//    consumers finish gate|up and wait at the grid barriers.
//  - Grid barriers over the consumer threads: after the Q8_1 of the hidden
//    states (three or more tokens), and after gate|up (every row of every
//    position written).  One or two tokens: a CTA then requantises the
//    SiLU*up of its down columns itself while staging them.  Three or more:
//    all consumer warps of the grid share SiLU*up -> Q8_1 out block by block,
//    behind a third barrier.
//    The producer does not wait at them.
// Items, shares and the consume routine are those of the grouped kernel: an
// item is G row groups of one non-empty group's expert, each CTA takes an
// equal contiguous range of items per phase, warp (g, p) takes row group g
// and K-slice p of each stage.
//
// The barrier counter is a caller-owned word.  Block 0 adds 2^31 - (n-1),
// every other block adds 1, so its top bit flips exactly when the last block
// arrives and its low 31 bits come back unchanged: a word whose low 31 bits
// are zero stays so after every completed launch (the top bit alternates).
// Every wait is bounded: a barrier that does not open within about a second
// sets bit 2 of the device fault word and lets the CTA go on (its outputs
// are then undefined; the word must be zeroed again before the next launch).
#ifndef FFN_WARPS12_MAX_T
#define FFN_WARPS12_MAX_T 2
#endif
#include <algorithm>
#include <mutex>
#include <unordered_map>

#include "ffn_args.cuh"
#include "q8_1.cuh"
#include "ring.cuh"
#include "route.cuh"

namespace mmvq {

constexpr int kFaultGridBarrier = 2;
constexpr int kFfnMaxExperts = 1024;
constexpr int kFfnMaxSlots = 256;

// Shared memory of a CTA with C consumer warps: the ring (S stages of C
// tiles), one group's staged columns (CM x max(H, F) quants, d and s), the
// K-slice partials.
// One or two tokens (CM <= 2) add the CTA's own Q8_1 of the hidden states
// (CM x act_row_bytes(H) quants, d and s).
__host__ __device__ inline size_t ffn_smem_bytes(int layout, int S, int H, int F, int CM, int C) {
  const int Km = H > F ? H : F;
  return tma_ring_offset(S) + (size_t)S * C * tile_bytes(layout) +
         (size_t)CM * act_row_bytes(Km) + (size_t)CM * (Km / kQK8) * 8 +
         (size_t)C * kMaxCols * kTileRows * 4 +
         (CM <= 2 ? (size_t)CM * act_row_bytes(H) + (size_t)CM * (H / kQK8) * 8 : 0);
}

// The counter's top bit as a barrier finds it: read once per CTA before the
// first barrier (no barrier instance can flip it before this CTA arrives),
// then flipped by the CTA itself after each barrier it passes.
__device__ __forceinline__ uint32_t grid_barrier_phase(const uint32_t* ctr) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
  return v & 0x80000000u;
}

// Barrier over the consumer threads of every CTA of the grid (see above).
// The CTA's threads meet first; thread 0's add is a release at GPU scope
// (cumulative over what the CTA's threads wrote before they met), issued
// without waiting for its result, and its polling load an acquire, so the
// writes of every CTA before the barrier are visible to every CTA after it.
// No full fence: one would also wait for the producer's bulk copies in
// flight.  phase: the top bit before this barrier (grid_barrier_phase), updated
// here.  Returns false when it gave up after limit_ns.
__device__ __forceinline__ bool grid_barrier_bounded(uint32_t* ctr, uint32_t nblocks,
                                                     int nthreads, volatile int* ok_s,
                                                     uint64_t limit_ns, uint32_t& phase) {
  group_sync(1, nthreads);
  if (threadIdx.x == 0) {
    const uint32_t inc = blockIdx.x == 0 ? 0x80000000u - (nblocks - 1u) : 1u;
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(ctr), "r"(inc) : "memory");
    int ok = 1;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0;; ++i) {
      uint32_t v;
      asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
      if ((v ^ phase) & 0x80000000u) break;
      if ((i & 15u) == 15u && global_ns() - t0 > limit_ns) {
        ok = 0;
        break;
      }
      __nanosleep(32);
    }
    *ok_s = ok;
  }
  phase ^= 0x80000000u;
  group_sync(1, nthreads);
  return *ok_s != 0;
}

// Producer: the stages of items [it0, it1) of one phase (as the grouped
// kernel's producer), continuing the ring's slot and phase counters.
template <int LAYOUT, int CM>
__device__ __forceinline__ void ffn_stream(const GroupedRing& r, uint8_t* ring, int& slot,
                                           uint32_t& par, int& issued, const uint8_t* W,
                                           int n_rg, int nb, int G, int P, int n_rgb, int it0,
                                           int it1, const int* active, const int* offs) {
  constexpr int TB = tile_bytes(LAYOUT);
  if (it0 >= it1) return;
  const int spb = nb / P;
  const size_t slice_bytes = (size_t)P * TB;
  const size_t expert_bytes = (size_t)n_rg * nb * TB;
  int a = it0 / n_rgb;
  int rgb = it0 - a * n_rgb;
  for (int it = it0; it < it1 && !*r.fail; ++it) {
    const int grp = active[a];
    const uint8_t* Wexp = W + (size_t)grp * expert_bytes;
    const int rg0 = rgb * G;
    const int nvalid = min(G, n_rg - rg0);
    const int pe = offs[grp + 1];
    // debug build: the item's tiles lie inside its expert's weights
    if (!MMVQ_INDEX_OK(grp >= 0 && rg0 >= 0 && rg0 + nvalid <= n_rg && spb * P <= nb)) {
      *r.fail = 1;
      break;
    }
    for (int p0 = offs[grp]; p0 < pe && !*r.fail; p0 += CM) {
      for (int bb = 0; bb < spb; ++bb) {
        if (issued >= r.S && !mbar_wait(&r.empty[slot], par ^ 1u, 128)) {
          *r.fail = 1;
          atomicOr(&g_fault_word, kFaultMbarTimeout);
          break;
        }
        mbar_expect_tx(&r.full[slot], (uint32_t)(nvalid * slice_bytes));
        uint8_t* dst = ring + (size_t)slot * r.stage_bytes;
        const uint8_t* src = Wexp + ((size_t)rg0 * nb + (size_t)bb * P) * TB;
        for (int g = 0; g < nvalid; ++g)
          bulk_g2s(dst + (size_t)g * slice_bytes, src + (size_t)g * nb * TB,
                   (uint32_t)slice_bytes, &r.full[slot]);
        ++issued;
        if (++slot == r.S) {
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
}

// Consumers: items [it0, it1) of one phase.  stage(p0, n, first) fills the
// chunk buffers with the columns of positions p0 .. p0+n-1; first tells that
// the item is its group's first (row groups from 0).
template <int LAYOUT, int CM, typename Stage>
__device__ __forceinline__ void ffn_consume(const GroupedRing& r, int& slot, uint32_t& par,
                                            int warp, int lane, int nthreads, int G, int P,
                                            int K, int n_rg, int n_rgb, int it0, int it1,
                                            const int* active, const int* offs,
                                            const uint8_t* act, const float* da, const float* sa,
                                            float* red, float* y, int64_t rows, Stage stage) {
  if (it0 >= it1) return;
  const int g = warp / P;
  const int p = warp - g * P;
  const int spb = K / kQK / P;
  const int nbq = K / kQK8;
  const int rb = act_row_bytes(K);
  int a = it0 / n_rgb;
  int rgb = it0 - a * n_rgb;
  int staged_grp = -1, staged_p0 = -1;
  for (int it = it0; it < it1; ++it) {
    const int grp = active[a];
    const int pe = offs[grp + 1];
    const int rg = rgb * G + g;
    const bool valid = rg < n_rg;
    for (int p0 = offs[grp]; p0 < pe; p0 += CM) {
      const int n = min(CM, pe - p0);
      if (grp != staged_grp || p0 != staged_p0) {
        group_sync(1, nthreads);  // the previous columns are no longer read
        stage(p0, n, rgb == 0);
        group_sync(1, nthreads);
        staged_grp = grp;
        staged_p0 = p0;
      }
      float* ybase = y + (size_t)p0 * rows;
#define MMVQ_FC(NC)                                                                          \
  grouped_consume<LAYOUT, NC>(r, slot, par, g, p, P, lane, spb, act, rb, da, sa, nbq, red, \
                              ybase, rg, valid, rows)
      if constexpr (CM == 1) {
        MMVQ_FC(1);
      } else if constexpr (CM == 2) {
        if (n == 1) MMVQ_FC(1); else MMVQ_FC(2);
      } else if constexpr (CM == 4) {
        switch (n) {
          case 1: MMVQ_FC(1); break;
          case 2: MMVQ_FC(2); break;
          case 3: MMVQ_FC(3); break;
          default: MMVQ_FC(4); break;
        }
      } else {
        switch (n) {
          case 1: MMVQ_FC(1); break;
          case 2: MMVQ_FC(2); break;
          case 3: MMVQ_FC(3); break;
          case 4: MMVQ_FC(4); break;
          case 5: MMVQ_FC(5); break;
          case 6: MMVQ_FC(6); break;
          case 7: MMVQ_FC(7); break;
          default: MMVQ_FC(8); break;
        }
      }
#undef MMVQ_FC
    }
    if (++rgb == n_rgb) {
      rgb = 0;
      ++a;
    }
  }
}

template <int LAYOUT, int CM, int FC>
__global__ void __launch_bounds__(32 * (FC + 1), FC < 12 ? 3 : 1)
    mmvq_expert_ffn_kernel(const FfnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int offs_s[kFfnMaxExperts + 1];
  __shared__ int active[kFfnMaxExperts];
  __shared__ int tok_s[kFfnMaxSlots];
  __shared__ int slot_s[kFfnMaxSlots];
  __shared__ int warp_sums[17];
  __shared__ volatile int ok_s;
  constexpr int C = FC;  // consumer warps
  constexpr int TB = tile_bytes(LAYOUT);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int E = a.n_experts, H = a.H, F = a.F;
  const int Km = H > F ? H : F;
  const int nbq_h = H / kQK8, nbq_f = F / kQK8;
  const int S = a.S;

  GroupedRing r;
  r.full = reinterpret_cast<uint64_t*>(smem);
  r.empty = r.full + S;
  r.fail = reinterpret_cast<volatile int*>(r.empty + S);
  r.ring = smem + tma_ring_offset(S);
  r.stage_bytes = (size_t)C * TB;
  r.S = S;
  uint8_t* ring = smem + tma_ring_offset(S);
  uint8_t* act = ring + (size_t)S * r.stage_bytes;  // chunk: [CM][act_row_bytes(Km)]
  float* da = reinterpret_cast<float*>(act + (size_t)CM * act_row_bytes(Km));
  float* sa = da + CM * (Km / kQK8);
  float* red = sa + CM * (Km / kQK8);
  // T <= 2: the CTA's own Q8_1 of the hidden states, [T][act_row_bytes(H)]
  // quants, then d and s as floats [T][H/32] each
  uint8_t* xact = reinterpret_cast<uint8_t*>(red + C * kMaxCols * kTileRows);
  float* xda = reinterpret_cast<float*>(xact + (size_t)(CM <= 2 ? CM : 0) * act_row_bytes(H));
  float* xsa = xda + (CM <= 2 ? CM : 0) * nbq_h;
  // debug build: the layout must fit the launch (the same outcome in every
  // CTA, so none is left at a grid barrier)
  if (!MMVQ_SMEM_OK(smem, xsa + (CM <= 2 ? CM : 0) * nbq_h)) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&r.full[s], 1);
      mbar_init(&r.empty[s], C);
    }
    *r.fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  grid_dependency_wait();  // x and topk may come from the preceding kernel
  // the barrier word's top bit, as left by earlier launches (read now, used
  // at the first barrier)
  uint32_t phase = grid_barrier_phase(a.sync);
  const int gwarp = blockIdx.x * C + warp;  // this warp's index in the grid
  const int nwarps = gridDim.x * C;
  const int n_xblk = a.T * nbq_h;
  // The hidden-state values, loaded now (volatile loads, issued here) so
  // that they arrive before the CTA's weight stream starts.  T <= 2: every
  // CTA quantises all of them itself, one 32-block per consumer thread
  // (16-byte loads when x allows them), so no grid barrier comes before
  // gate|up.  Otherwise each consumer warp of the grid takes one 32-block
  // (at most one per warp for T <= 8 on a full GPU).
  float x_first = 0.0f;
  float4 xr[CM <= 2 ? 2 : 1];
  const bool x_vec = ((reinterpret_cast<uintptr_t>(a.x) & 15) == 0) && (a.ldx % 4 == 0);
  if constexpr (CM <= 2) {
    // quad q = threadIdx.x / 4 takes block q, its lane j values 8j .. 8j+7
    const int blk = threadIdx.x >> 2;
    if (threadIdx.x < 32 * C && blk < n_xblk && x_vec) {
      const int t = blk / nbq_h;
      const float* src = a.x + (int64_t)t * a.ldx + (blk - t * nbq_h) * kQK8 + 8 * (lane & 3);
#pragma unroll
      for (int i = 0; i < 2; ++i)
        asm volatile("ld.global.v4.f32 {%0,%1,%2,%3}, [%4];"
                     : "=f"(xr[i].x), "=f"(xr[i].y), "=f"(xr[i].z), "=f"(xr[i].w)
                     : "l"(src + 4 * i));
    }
  } else {
    if (warp < C && gwarp < n_xblk) {
      const int t = gwarp / nbq_h;
      x_first = a.x[(int64_t)t * a.ldx + (gwarp - t * nbq_h) * kQK8 + lane];
    }
  }

  // 1. token lists, in shared memory (every CTA; CTA 0 reports bad ids)
  route_groups_cta<kFfnMaxExperts>(a.topk, a.T * a.k, a.k, E, nullptr, offs_s, tok_s, slot_s,
                                   blockIdx.x == 0 ? a.status : nullptr);
  __syncthreads();
  const int n_pos = offs_s[E];
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
      if (a.offsets) a.offsets[e] = offs_s[e];
      if (a.expert_ids && e < E) a.expert_ids[e] = e;
    }
    for (int q = threadIdx.x; q < n_pos; q += blockDim.x) {
      if (a.act_index) a.act_index[q] = tok_s[q];
      if (a.slot_of) a.slot_of[q] = slot_s[q];
    }
  }
  // 2. the non-empty groups, in group order
  const int per = (E + (int)blockDim.x - 1) / (int)blockDim.x;
  const int q0 = threadIdx.x * per;
  const int q1 = min(E, q0 + per);
  int cnt = 0;
  for (int q = q0; q < q1; ++q) cnt += offs_s[q + 1] > offs_s[q] ? 1 : 0;
  int n_active = 0;
  int pos = block_scan_excl(cnt, warp_sums, &n_active);
  for (int q = q0; q < q1; ++q)
    if (offs_s[q + 1] > offs_s[q]) active[pos++] = q;
  __syncthreads();

  // 3. this CTA's items of each phase: the first (items mod grid) CTAs take
  // one item more than the rest (item counts < 2^22, so int arithmetic)
  const int nrg_gu = 2 * F / kTileRows, nrg_dn = H / kTileRows;
  const int nrgb_gu = (nrg_gu + a.g_gu - 1) / a.g_gu;
  const int nrgb_dn = (nrg_dn + a.g_dn - 1) / a.g_dn;
  const int b = blockIdx.x, nbk = gridDim.x;
  const int ni_gu = n_active * nrgb_gu, ni_dn = n_active * nrgb_dn;
  const int i0 = b * (ni_gu / nbk) + min(b, ni_gu % nbk);
  const int i1 = i0 + ni_gu / nbk + (b < ni_gu % nbk ? 1 : 0);
  const int j0 = b * (ni_dn / nbk) + min(b, ni_dn % nbk);
  const int j1 = j0 + ni_dn / nbk + (b < ni_dn % nbk ? 1 : 0);

  if (warp == C) {  // ------------------------------------------ producer
    if (lane == 0) {
      int slot = 0;
      uint32_t par = 0;
      int issued = 0;
      ffn_stream<LAYOUT, CM>(r, ring, slot, par, issued, a.w_gu, nrg_gu, H / kQK, a.g_gu, a.p_gu,
                             nrgb_gu, i0, i1, active, offs_s);
      ffn_stream<LAYOUT, CM>(r, ring, slot, par, issued, a.w_dn, nrg_dn, F / kQK, a.g_dn, a.p_dn,
                             nrgb_dn, j0, j1, active, offs_s);
      // wait (bounded) for the last phase of every filled slot
      for (int s = 0; s < S && s < issued; ++s) {
        const int last = issued - 1 - ((issued - 1 - s) % S);
        mbar_wait(&r.full[s], (uint32_t)((last / S) & 1));
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int nthreads = 32 * C;
  int slot = 0;
  uint32_t par = 0;
  const uint8_t* xq = a.xq;
  if constexpr (CM <= 2) {
    // 4. one or two tokens: the CTA quantises the T hidden states into its
    // own staging, a 32-block per quad of lanes (CTA 0 also writes xq); the
    // bytes are those of the plain quantiser
    const int nquads = nthreads / 4;
    for (int blk0 = 0; blk0 < n_xblk; blk0 += nquads) {
      const int blk = blk0 + (int)(threadIdx.x >> 2);
      const bool on = blk < n_xblk;
      const int j = lane & 3;
      const int t = on ? blk / nbq_h : 0;
      const int kb = on ? blk - t * nbq_h : 0;
      float v[8];
      if (on && blk0 == 0 && x_vec) {
        v[0] = xr[0].x; v[1] = xr[0].y; v[2] = xr[0].z; v[3] = xr[0].w;
        v[4] = xr[1].x; v[5] = xr[1].y; v[6] = xr[1].z; v[7] = xr[1].w;
      } else {
        const float* src = a.x + (int64_t)t * a.ldx + kb * kQK8 + 8 * j;
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = on ? src[i] : 0.0f;
      }
      uint32_t w0, w1, header;
      quantize_block_quad(v, w0, w1, header);
      if (on) {
        *reinterpret_cast<uint2*>(xact + (size_t)t * act_row_bytes(H) + act_off(kb) + 8 * j) =
            make_uint2(w0, w1);
        if (j == 0) {
          xda[t * nbq_h + kb] = half_bits_to_float((uint16_t)(header & 0xffffu));
          if (has_min(LAYOUT)) xsa[t * nbq_h + kb] = half_bits_to_float((uint16_t)(header >> 16));
        }
        if (blockIdx.x == 0) {
          uint32_t* o = reinterpret_cast<uint32_t*>(a.xq + (size_t)blk * kQ81Bytes);
          if (j == 0) o[0] = header;
          o[1 + 2 * j] = w0;
          o[2 + 2 * j] = w1;
        }
      }
    }
    group_sync(1, nthreads);
  } else {
    // 4. the T hidden states as Q8_1, one 32-block per warp of the grid
    for (int blk = gwarp; blk < n_xblk; blk += nwarps) {
      const int t = blk / nbq_h;
      const int kb = blk - t * nbq_h;
      const float v = blk == gwarp ? x_first : a.x[(int64_t)t * a.ldx + kb * kQK8 + lane];
      quantize_lane(v, a.xq + (size_t)blk * kQ81Bytes, lane);
    }
    if (!grid_barrier_bounded(a.sync, gridDim.x, nthreads, &ok_s, kWaitLimitNs, phase) &&
        threadIdx.x == 0)
      atomicOr(&g_fault_word, kFaultGridBarrier);
  }
  // 5. gate|up: a group's columns are its tokens' hidden states (copied from
  // the CTA's own staging for T <= 2, else staged from xq through L2)
  auto stage_gu = [=](int p0, int n, bool) {
    if constexpr (CM <= 2) {
      // the chunk layout of the gate|up phase (K = H): rows of
      // act_row_bytes(H), d and s at [c][H/32]
      const int rbh = act_row_bytes(H);
      for (int c = 0; c < n; ++c) {
        const int t = tok_s[p0 + c];
        const uint4* src = reinterpret_cast<const uint4*>(xact + (size_t)t * rbh);
        uint4* dst = reinterpret_cast<uint4*>(act + (size_t)c * rbh);
        for (int v = threadIdx.x; v < rbh / 16; v += nthreads) dst[v] = src[v];
        for (int v = threadIdx.x; v < nbq_h; v += nthreads) {
          da[c * nbq_h + v] = xda[t * nbq_h + v];
          if (has_min(LAYOUT)) sa[c * nbq_h + v] = xsa[t * nbq_h + v];
        }
      }
    } else {
      stage_q8_1<true>(xq, H, n, [=](int c) { return tok_s[p0 + c]; }, act, da,
                       has_min(LAYOUT) ? sa : nullptr, threadIdx.x, nthreads);
    }
  };
  ffn_consume<LAYOUT, CM>(r, slot, par, warp, lane, nthreads, a.g_gu, a.p_gu, H, nrg_gu, nrgb_gu,
                          i0, i1, active, offs_s, act, da, sa, red, a.gu, 2 * F, stage_gu);
  if (!grid_barrier_bounded(a.sync, gridDim.x, nthreads, &ok_s, kWaitLimitNs, phase) &&
      threadIdx.x == 0)
    atomicOr(&g_fault_word, kFaultGridBarrier);
  const uint8_t* hq_in = a.hq;
  if constexpr (CM <= 2) {
    // 6-7. one or two tokens: a CTA's down work covers one or two positions,
    // so it requantises their SiLU(gate)*up itself, straight into its staged
    // columns (no third barrier); the CTA holding a group's first down item
    // also writes the group's rows of hq
    auto stage_dn = [=](int p0, int n, bool first) {
      const int nblk = n * nbq_f;
      for (int b0 = warp; b0 < nblk; b0 += 4 * C) {
        float gv[4], uv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int blk = b0 + j * C;
          if (blk < nblk) {
            const int q = blk / nbq_f;
            const float* row = a.gu + (size_t)(p0 + q) * 2 * F + (blk - q * nbq_f) * kQK8 + lane;
            gv[j] = __ldcg(row);
            uv[j] = __ldcg(row + F);
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int blk = b0 + j * C;
          if (blk < nblk) {
            const int q = blk / nbq_f;
            const int kb = blk - q * nbq_f;
            quantize_lane_staged(silu_mul(gv[j], uv[j]), act + (size_t)q * act_row_bytes(F),
                                 da + q * nbq_f, has_min(LAYOUT) ? sa + q * nbq_f : nullptr, kb,
                                 first ? a.hq + ((size_t)p0 * nbq_f + blk) * kQ81Bytes : nullptr,
                                 lane);
          }
        }
      }
    };
    ffn_consume<LAYOUT, CM>(r, slot, par, warp, lane, nthreads, a.g_dn, a.p_dn, F, nrg_dn,
                            nrgb_dn, j0, j1, active, offs_s, act, da, sa, red, a.y, H, stage_dn);
  } else {
    // 6. SiLU(gate)*up -> Q8_1, one block per warp over the whole grid
    const int nblk = n_pos * nbq_f;
    for (int blk = gwarp; blk < nblk; blk += nwarps) {
      const int q = blk / nbq_f;
      const int kb = blk - q * nbq_f;
      const float* row = a.gu + (size_t)q * 2 * F;
      const float h = silu_mul(__ldcg(row + kb * kQK8 + lane), __ldcg(row + F + kb * kQK8 + lane));
      quantize_lane(h, a.hq + (size_t)blk * kQ81Bytes, lane);
    }
    if (!grid_barrier_bounded(a.sync, gridDim.x, nthreads, &ok_s, kWaitLimitNs, phase) &&
        threadIdx.x == 0)
      atomicOr(&g_fault_word, kFaultGridBarrier);
    // 7. down: a group's columns are its positions' requantised activations
    auto stage_dn = [=](int p0, int n, bool) {
      stage_q8_1<true>(hq_in, F, n, [=](int c) { return p0 + c; }, act, da,
                       has_min(LAYOUT) ? sa : nullptr, threadIdx.x, nthreads);
    };
    ffn_consume<LAYOUT, CM>(r, slot, par, warp, lane, nthreads, a.g_dn, a.p_dn, F, nrg_dn,
                            nrgb_dn, j0, j1, active, offs_s, act, da, sa, red, a.y, H, stage_dn);
  }
}

// ------------------------------------------------------------ host side ----

struct FfnCfg {
  int S, g_gu, p_gu, g_dn, p_dn, grid;
  size_t smem;
};

// Consumer warps per CTA for CM positions per pass (T rounded up to a power
// of two).  Measured on GB300 (256 experts, gate|up 1536 x 2560, down
// 2560 x 768): one 12-warp CTA per SM is faster for one token (15.7 against
// 17.6 us per layer), three 4-warp CTAs per SM from four tokens on (33.1 /
// 52.6 us at T = 4 / 8 against 34.1 / 56.8 us): more producers per SM keep
// more of the larger step's bytes in flight.
template <int CM>
constexpr int ffn_warps() { return CM <= FFN_WARPS12_MAX_T ? 12 : 4; }

// (G, P) of one phase: P | K/256, G*P = C, and each warp's K-slice at least
// three stages long (or all of K when K/256 < 3): items of a stage or two
// spend more on the K-slice reduction and the item switch than they save.
// Among those the busiest CTA's stages, ceil(items / grid) * (K/256) / P,
// decide; ties go to the larger P (more, smaller items over more CTAs).
// est_active estimates the non-empty groups (the lists are device data).
static void ffn_split(int64_t n_rg, int nb, int64_t est_active, int grid, int C, int* G, int* P) {
  int64_t best = -1;
  for (int p = 1; p <= C; ++p) {
    if (C % p || nb % p || (p > 1 && nb / p < 3)) continue;
    const int g = C / p;
    const int64_t items = est_active * ((n_rg + g - 1) / g);
    const int64_t cost = (items + grid - 1) / grid * (nb / p);
    if (best < 0 || cost <= best) {
      best = cost;
      *G = g;
      *P = p;
    }
  }
}

// CM: positions per pass, T rounded up to 1, 2, 4 or 8.  The ring takes as
// many stages (2..8) as fit beside the activations; the grid is every CTA
// that can be resident at once (FC = 12: one per SM; FC = 4: three).
template <int LAYOUT, int CM, int FC>
static int ffn_config(int n_experts, int H, int F, int T, int k, FfnCfg* out) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, FfnCfg> cache;
  const uint64_t key = ((uint64_t)(H / kQK) << 40) | ((uint64_t)(F / kQK) << 24) |
                       ((uint64_t)n_experts << 8) | (uint64_t)(T * k > 255 ? 255 : T * k);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *out = it->second;
      return MMVQ_OK;
    }
  }
  auto kern = mmvq_expert_ffn_kernel<LAYOUT, CM, FC>;
  constexpr int threads = 32 * (FC + 1);
  const int sms = device_sms();
  if (sms <= 0) return MMVQ_ERR_CUDA;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, (const void*)kern) != cudaSuccess) return MMVQ_ERR_CUDA;
  const size_t optin = max_smem_optin();
  if (optin <= fa.sharedSizeBytes) return MMVQ_ERR_CUDA;
  // three CTAs per SM share its shared memory (about 1 KB each is reserved)
  const int want = FC < 12 ? 3 : 1;
  const size_t per_cta = (optin + 1024) / want - 1024;
  if (per_cta <= fa.sharedSizeBytes) return MMVQ_ERR_CUDA;
  const size_t limit = per_cta - fa.sharedSizeBytes;
  int S = 0;
  for (int s = 8; s >= 2 && S == 0; --s)
    if (ffn_smem_bytes(LAYOUT, s, H, F, CM, FC) <= limit) S = s;
  if (S == 0) return MMVQ_ERR_SHAPE;
  const size_t smem = ffn_smem_bytes(LAYOUT, S, H, F, CM, FC);
  if (ensure_smem((const void*)kern, smem) != MMVQ_OK) return MMVQ_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) !=
          cudaSuccess ||
      per_sm < 1)
    return MMVQ_ERR_CUDA;
  FfnCfg cfg = {S, 0, 0, 0, 0, sms * per_sm, smem};
  const int64_t est_active = std::max<int64_t>(1, std::min<int64_t>(n_experts, (int64_t)T * k));
  ffn_split((int64_t)2 * F / kTileRows, H / kQK, est_active, cfg.grid, FC, &cfg.g_gu, &cfg.p_gu);
  ffn_split(H / kTileRows, F / kQK, est_active, cfg.grid, FC, &cfg.g_dn, &cfg.p_dn);
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = cfg;
  *out = cfg;
  return MMVQ_OK;
}

template <int LAYOUT, int CM, int FC>
static int launch_ffn_fc(FfnArgs args, cudaStream_t stream, int32_t* info) {
  FfnCfg cfg;
  const int rc = ffn_config<LAYOUT, CM, FC>(args.n_experts, args.H, args.F, args.T, args.k, &cfg);
  if (rc != MMVQ_OK) return rc;
  if (info) {
    info[0] = cfg.grid;
    info[1] = 32 * (FC + 1);
    info[2] = (int32_t)cfg.smem;
    info[3] = cfg.S;
    info[4] = cfg.g_gu;
    info[5] = cfg.p_gu;
    info[6] = cfg.g_dn;
    info[7] = cfg.p_dn;
    return MMVQ_OK;
  }
  args.S = cfg.S;
  args.g_gu = cfg.g_gu;
  args.p_gu = cfg.p_gu;
  args.g_dn = cfg.g_dn;
  args.p_dn = cfg.p_dn;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(cfg.grid);
  lc.blockDim = dim3(32 * (FC + 1));
  lc.dynamicSmemBytes = cfg.smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 2;
  return cudaLaunchKernelEx(&lc, mmvq_expert_ffn_kernel<LAYOUT, CM, FC>, args) == cudaSuccess
             ? MMVQ_OK
             : MMVQ_ERR_CUDA;
}

template <int LAYOUT, int CM>
static int launch_ffn_cm(const FfnArgs& args, cudaStream_t stream, int32_t* info) {
  return launch_ffn_fc<LAYOUT, CM, ffn_warps<CM>()>(args, stream, info);
}

template <int LAYOUT>
static int launch_ffn_layout(const FfnArgs& args, cudaStream_t s, int32_t* info) {
  if (args.T <= 1) return launch_ffn_cm<LAYOUT, 1>(args, s, info);
  if (args.T == 2) return launch_ffn_cm<LAYOUT, 2>(args, s, info);
  if (args.T <= 4) return launch_ffn_cm<LAYOUT, 4>(args, s, info);
  return launch_ffn_cm<LAYOUT, 8>(args, s, info);
}

// info != NULL: report the launch shape (8 ints) instead of launching.
int launch_expert_ffn(int type, const FfnArgs& args, cudaStream_t s, int32_t* info) {
  if (type == MMVQ_Q4_K_PLANAR) return launch_ffn_layout<kQ4Planar>(args, s, info);
  return launch_ffn_layout<kQ6Planar>(args, s, info);
}

// Self-test of the grid barrier's bound: one CTA waits for a second block
// that is never launched, with a short limit, and reports through the fault
// word as the kernel does.  The counter word is left changed.
__global__ void grid_barrier_selftest_kernel(uint32_t* ctr, uint64_t limit_ns) {
  __shared__ volatile int ok_s;
  uint32_t phase = grid_barrier_phase(ctr);
  if (!grid_barrier_bounded(ctr, 2u, (int)blockDim.x, &ok_s, limit_ns, phase) &&
      threadIdx.x == 0)
    atomicOr(&g_fault_word, kFaultGridBarrier);
}

int launch_grid_barrier_selftest(uint32_t* ctr, uint32_t limit_us, cudaStream_t stream) {
  grid_barrier_selftest_kernel<<<1, 32, 0, stream>>>(ctr, (uint64_t)limit_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? MMVQ_OK : MMVQ_ERR_CUDA;
}

// ----------------------------------------------- fixed-scratch variant ----
//
// mmvq_expert_ffn_noalloc keeps the layer's intermediates (the barrier word,
// xq, hq and gu) in this array instead of buffers from the caller.  It is a
// file-scope device variable, so every GPU that loads the library holds it
// until the process exits, and every call on a device shares it.  Host code
// must not hand the name itself to a kernel (on the host it names a
// stand-in, not device memory): its device address is looked up once per
// device with cudaGetSymbolAddress, with that device current, and cached.
static __device__ __align__(256) uint8_t g_ffn_scratch[kFfnScratchBytes];

static int ffn_scratch_address(uint8_t** p) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return MMVQ_ERR_CUDA;
  static std::mutex mu;
  static std::unordered_map<int, uint8_t*> addr;
  std::lock_guard<std::mutex> lock(mu);
  auto it = addr.find(dev);
  if (it != addr.end()) {
    *p = it->second;
    return MMVQ_OK;
  }
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_ffn_scratch) != cudaSuccess || ptr == nullptr)
    return MMVQ_ERR_CUDA;
  addr[dev] = static_cast<uint8_t*>(ptr);
  *p = static_cast<uint8_t*>(ptr);
  return MMVQ_OK;
}

int launch_expert_ffn_noalloc(int type, FfnArgs a, cudaStream_t s) {
  const FfnScratchLayout l = ffn_scratch_layout(a.H, a.F, a.T, a.k);
  if (l.end > kFfnScratchBytes) return MMVQ_ERR_SCRATCH;
  uint8_t* base = nullptr;
  const int rc = ffn_scratch_address(&base);
  if (rc != MMVQ_OK) return rc;
  a.sync = reinterpret_cast<uint32_t*>(base);
  a.xq = base + l.xq;
  a.hq = base + l.hq;
  a.gu = reinterpret_cast<float*>(base + l.gu);
  // the grid barrier needs a word whose low 31 bits are zero; a launch that
  // gave up at a barrier leaves it otherwise, so it is cleared every call
  // (xq, hq and gu are written before they are read)
  if (cudaMemsetAsync(a.sync, 0, sizeof(uint32_t), s) != cudaSuccess) return MMVQ_ERR_CUDA;
  return launch_expert_ffn(type, a, s, nullptr);
}

// This translation unit's fault word, for mmvq_read_device_fault.
int read_clear_ffn_fault_word(unsigned int* v) { return read_clear_fault_word(v); }

}  // namespace mmvq
