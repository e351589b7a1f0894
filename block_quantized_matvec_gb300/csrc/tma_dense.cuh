// The dense ring kernel over planar tiles (Q6_K, Q4_K, Q5_K), shared by the
// translation units that instantiate it: mmvq_tma.cu (Q8_1 columns, with
// and without a cluster K-split, the parity-debug instance, and for 4-8
// columns the tensor-core consumer's instances) and mmvq_tma_f32.cu (fp32
// columns quantised inside the kernel).  The design notes are at the top of
// mmvq_tma.cu.
#pragma once
#include "q8_1.cuh"
#include "tma_mma.cuh"

namespace mmvq {

// Quantise NCOLS fp32 columns (x [ncols][ldx], the first K values of each)
// into the staging of the ring kernels, a 32-block per four lanes
// (quantize_block_quad: the plain quantiser's bytes), all nthreads threads
// (whole warps) taking part; xq_out (may be NULL) also receives the 36-byte
// blocks.  16-byte loads when x and ldx allow them.
__device__ __forceinline__ void quantize_columns_quad(const float* __restrict__ x, int64_t ldx,
                                                      int K, int ncols, uint8_t* act, float* da,
                                                      float* sa, uint8_t* xq_out, int tid,
                                                      int nthreads) {
  const int nbq = K / kQK8;
  const int rb = act_row_bytes(K);
  const int nblk = ncols * nbq;
  const int nquads = nthreads / 4;
  const int j = tid & 3;
  const bool vec = ((reinterpret_cast<uintptr_t>(x) & 15) == 0) && (ldx % 4 == 0);
  for (int blk0 = 0; blk0 < nblk; blk0 += nquads) {
    const int blk = blk0 + tid / 4;
    const bool on = blk < nblk;
    const int c = on ? blk / nbq : 0;
    const int kb = on ? blk - c * nbq : 0;
    const float* src = x + (int64_t)c * ldx + kb * kQK8 + 8 * j;
    float v[8];
    if (on && vec) {
      const float4 a = reinterpret_cast<const float4*>(src)[0];
      const float4 b = reinterpret_cast<const float4*>(src)[1];
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = on ? src[i] : 0.0f;
    }
    uint32_t w0, w1, header;
    quantize_block_quad(v, w0, w1, header);
    if (on) {
      *reinterpret_cast<uint2*>(act + c * rb + act_off(kb) + 8 * j) = make_uint2(w0, w1);
      if (j == 0) {
        da[c * nbq + kb] = half_bits_to_float((uint16_t)(header & 0xffffu));
        if (sa) sa[c * nbq + kb] = half_bits_to_float((uint16_t)(header >> 16));
      }
      if (xq_out) {
        uint32_t* o = reinterpret_cast<uint32_t*>(xq_out + (size_t)blk * kQ81Bytes);
        if (j == 0) o[0] = header;
        o[1 + 2 * j] = w0;
        o[2 + 2 * j] = w1;
      }
    }
  }
}

// Consumers are G groups of P warps (C = G*P); warp C is the producer.  A
// batch is G of the row groups of the CTA's cluster (group g takes the g-th);
// within a batch, stage bb holds, for each group, the P consecutive tiles
// bb*P .. bb*P+P-1 of the CTA's K-range of its row group, and warp (g, p)
// takes tile bb*P+p.  The P partial sums of a row group are added in warp
// order at the batch end.
//
// K-split over a cluster (CS = 2..8 CTAs): CTA rank q of a cluster takes
// the 256-blocks [q*nb/CS, (q+1)*nb/CS) of every row group of the cluster's
// batches and stages only those activations, so a matrix with few row groups
// still covers every SM, and the staged columns take 1/CS of the shared
// memory.  At each batch end the CTAs of ranks 1..CS-1 write their row sums
// into rank 0's shared memory (distributed shared memory) and arrive on its
// `xfull` mbarrier (release at cluster scope); rank 0 adds them in rank order
// after its own (a fixed order, so results repeat bit for bit) and stores y.
// The partials are double-buffered by batch parity; before a rank overwrites
// a buffer two batches on, it waits on its own `xempty` mbarrier, on which
// rank 0 arrives once it has read that buffer.  Rank 0 arrives only where a
// later batch will wait, and waits itself for every batch's partials, so no
// CTA's shared memory is touched by another CTA after it exits.  Every wait
// is bounded, as the ring's; a cluster barrier is passed once, after the
// mbarriers are initialised.
// SUMI: also store every per-32-block integer sum (the parity-debug entry);
// a separate instance, so the product path carries no per-block test.
// CLUSTER: the cluster instance (CS = cs); the plain instance has CS = 1
// folded in.
// XF32: the columns come as fp32 x [NCOLS][ldx] and the CTA quantises them
// itself into its staging (a 32-block per four lanes, the plain quantiser's
// bytes); CTA 0 also writes them to xq (plain instance only).
// MMA: the tensor-core consumer (tma_mma.cuh; same sums, same bits) on the
// same staging, plus a table of d_a, s_a and MMA start values built after
// it; MMA lane (g, t) holds rows g and g + 8, columns 2t and 2t + 1, and
// both halves of each block, and the lane sums pass through shared memory
// into the dp4a lanes' layout before the K-slice reduction, which is
// common to both.
template <int LAYOUT, int NCOLS, bool SUMI, bool CLUSTER, bool XF32, bool MMA = false>
__global__ void __launch_bounds__(13 * 32) mmvq_planar_tma_kernel(const uint8_t* __restrict__ W,
                                                               int64_t rows, int K,
                                                               const uint8_t* __restrict__ xq,
                                                               float* __restrict__ y,
                                                               int32_t* __restrict__ sumi, int S,
                                                               int G, int P, int cs,
                                                               uint32_t flags,
                                                               const float* __restrict__ xf,
                                                               int64_t ldx, uint8_t* xq_out) {
  static_assert(!(XF32 && (CLUSTER || SUMI || MMA)), "fp32 columns: plain dp4a instance only");
  const int CS = CLUSTER ? cs : 1;
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int C = G * P;  // consumer warps; warp C produces
  const int nb = K / kQK;
  const int nbc = nb / CS;   // 256-blocks of this CTA's K-range
  const int Kc = K / CS;
  const int nbq = Kc / kQK8;  // 32-blocks of the K-range (staged)
  const int rb = act_row_bytes(Kc);
  const int rank = CLUSTER ? (int)cluster_ctarank() : 0;
  const int cid = blockIdx.x / CS;  // cluster index (1-D clusters of CS CTAs)
  const int ncl = gridDim.x / CS;
  const int64_t n_rg = (rows + kTileRows - 1) / kTileRows;
  constexpr int TB = tile_bytes(LAYOUT);
  const int spb = nbc / P;  // stages per batch
  const size_t stage_bytes = (size_t)C * TB;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + S;
  volatile int* fail = reinterpret_cast<volatile int*>(empty + S);
  uint8_t* ring = smem + tma_ring_offset(S);
  uint8_t* act = ring + (size_t)S * stage_bytes;
  float* da = reinterpret_cast<float*>(act + NCOLS * rb);
  float* sa = da + NCOLS * nbq;  // Q4_K only
  float* tab = sa + (has_min(LAYOUT) ? NCOLS * nbq : 0);  // MMA: [nbq][4][8]
  // K-slice partials [C][8][16] floats, two buffers by batch parity when
  // P > 1 (so one group barrier per batch orders them)
  float* red = tab + (MMA ? nbq * 32 : 0);
  // cluster exchange: xred [2][CS][G][NCOLS][16] floats (rank 0's is used),
  // then xfull[2], xempty[2]
  float* xred = red + C * kMaxCols * kTileRows * (P > 1 ? 2 : 1);
  uint64_t* xfull = reinterpret_cast<uint64_t*>(xred + (CS > 1 ? 2 * CS * G * NCOLS * kTileRows : 0));
  uint64_t* xempty = xfull + 2;
  // debug build: the layout must fit the launch (the same outcome in every
  // CTA of a cluster, so none is left at the cluster barrier)
  if (!MMVQ_SMEM_OK(smem, CLUSTER ? reinterpret_cast<uint8_t*>(xempty + 2)
                                  : reinterpret_cast<uint8_t*>(xred)))
    return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C);
    }
    if (CLUSTER) {
      for (int q = 0; q < 2; ++q) {
        mbar_init(&xfull[q], (CS - 1) * G);
        mbar_init(&xempty[q], G);
      }
    }
    *fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (CLUSTER) cluster_sync_all();
  grid_launch_dependents();

  // this cluster's row groups: cid, + ncl, ... (row groups < 2^27: 32-bit
  // divisions, which stay inline)
  const int64_t my_rgs = (cid < n_rg) ? (uint32_t)(n_rg - 1 - cid) / ncl + 1 : 0;
  const int64_t batches = (uint32_t)(my_rgs + G - 1) / (uint32_t)G;
  const int64_t total = batches * spb;
  const int64_t blk0 = (int64_t)rank * nbc;  // first 256-block of the K-range

  if (warp == C) {  // ------------------------------------------ producer
    if (lane == 0) {
      // slot and round parity are kept incrementally (no divisions per stage)
      int64_t it = 0;
      int slot = 0;
      uint32_t par = 0;
      int64_t j = 0;
      int bb = 0;
      for (; it < total; ++it) {
        if (it >= S && !*fail && !mbar_wait(&empty[slot], par ^ 1u, 128)) {
          *fail = 1;
          atomicOr(&g_fault_word, kFaultMbarTimeout);
        }
        if (*fail) break;
        const int64_t left = my_rgs - j * G;
        const int valid = (int)(left < G ? left : G);
        // debug build: the stage's tiles lie inside the weights
        if (!MMVQ_INDEX_OK(cid + (j * G + valid - 1) * (int64_t)ncl < n_rg &&
                           blk0 + (int64_t)(bb + 1) * P <= nb)) {
          *fail = 1;
          break;
        }
        mbar_expect_tx(&full[slot], (uint32_t)(valid * P * TB));
        for (int g = 0; g < valid; ++g) {
          const int64_t rg = cid + (j * G + g) * (int64_t)ncl;
          bulk_g2s(ring + (size_t)slot * stage_bytes + (size_t)g * P * TB,
                   W + (rg * nb + blk0 + (int64_t)bb * P) * TB, (uint32_t)(P * TB), &full[slot]);
        }
        if (++bb == spb) {
          bb = 0;
          ++j;
        }
        if (++slot == S) {
          slot = 0;
          par ^= 1u;
        }
      }
      // no copy of this CTA may land after it exits: wait (bounded) for the
      // last phase of every slot that was filled
      const int64_t issued = it;  // a CTA's stages: < 2^31
      for (int s = 0; s < S && s < issued; ++s) {
        const uint32_t last = (uint32_t)(issued - 1) - ((uint32_t)(issued - 1 - s) % (uint32_t)S);
        mbar_wait(&full[s], (last / (uint32_t)S) & 1u);
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int nthreads = 32 * C;
  const int tid = threadIdx.x;
  // With MMVQ_FLAG_XQ_STABLE no kernel that may still run writes xq, so the
  // whole product runs before the grid dependency; only the stores of y
  // wait for the preceding kernel.
  const bool stable = (flags & MMVQ_FLAG_XQ_STABLE) != 0;
  bool waited = !stable;
  if (!stable) grid_dependency_wait();
  if constexpr (XF32) {
    quantize_columns_quad(xf, ldx, K, NCOLS, act, da, has_min(LAYOUT) ? sa : nullptr,
                          blockIdx.x == 0 ? xq_out : nullptr, tid, nthreads);
  } else if constexpr (!CLUSTER) {
    stage_q8_1(xq, K, NCOLS, [](int c) { return c; }, act, da,
               has_min(LAYOUT) ? sa : nullptr, tid, nthreads);
  } else {
    stage_q8_1_slice(xq, K / kQK8, (int)blk0 * 8, Kc, NCOLS, act, da,
                     has_min(LAYOUT) ? sa : nullptr, tid, nthreads);
  }
  group_sync(1, nthreads);
  if constexpr (MMA) {
    mma_build_table<LAYOUT>(act, rb, da, sa, nbq, NCOLS, tab, tid, nthreads);
    group_sync(1, nthreads);
  }

  const int g = warp / P;
  const int p = warp - g * P;
  const int i = lane & 15;
  const int h = lane >> 4;
  const int mg = lane >> 2;  // MMA lane (mg, mt): rows mg, mg + 8; columns 2mt, 2mt + 1
  const int mt = lane & 3;
  int slot = 0;
  uint32_t par = 0;
  for (int64_t j = 0; j < batches; ++j) {
    const int64_t k = j * G + g;
    const bool valid = k < my_rgs;
    const int64_t rg = cid + k * (int64_t)ncl;
    const int64_t row = rg * kTileRows + i;
    // per-block sums of this row at its global 32-block index
    int32_t* srow =
        (SUMI && sumi && valid && row < rows) ? sumi + row * (K / kQK8) + blk0 * 8 : nullptr;
    if (srow && !waited) {
      grid_dependency_wait();
      waited = true;
    }
    float acc[NCOLS];
#pragma unroll
    for (int c = 0; c < NCOLS; ++c) acc[c] = 0.0f;
    float macc[2][2][2] = {{{0.0f, 0.0f}, {0.0f, 0.0f}}, {{0.0f, 0.0f}, {0.0f, 0.0f}}};
    int32_t* msrow[2] = {nullptr, nullptr};
    if (SUMI && MMA && sumi && valid) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int64_t mrow = rg * kTileRows + mg + 8 * rr;
        if (mrow < rows) msrow[rr] = sumi + mrow * (K / kQK8) + blk0 * 8;
      }
      if ((msrow[0] || msrow[1]) && !waited) {
        grid_dependency_wait();
        waited = true;
      }
    }
    for (int bb = 0; bb < spb; ++bb) {
      const int s = slot;
      if (!*fail && !mbar_wait(&full[s], par)) {
        *fail = 1;
        atomicOr(&g_fault_word, kFaultMbarTimeout);
      }
      if (++slot == S) {
        slot = 0;
        par ^= 1u;
      }
      const uint8_t* tile = ring + (size_t)s * stage_bytes + (size_t)warp * TB;
      const int64_t scs = rows * (K / kQK8);
      // debug build: the tile lies in the ring, its K-block in the staging
      const bool use = valid && MMVQ_INDEX_OK(s < S && warp < C && bb * P + p < nbc);
      if constexpr (MMA) {
        if (LAYOUT == kQ6Planar) {
          Q6Mma w;
          if (use) load_q6_mma(tile, mg, mt, w);
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
          if (use) q6_mma<NCOLS, SUMI>(w, bb * P + p, lane, act, rb, tab, macc, msrow, scs);
        } else {
          Q45Mma w;
          if (use) load_q45_mma<LAYOUT == kQ5Planar>(tile, mg, mt, w);
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
          if (use)
            q45_mma<NCOLS, LAYOUT == kQ5Planar, SUMI>(w, bb * P + p, lane, act, rb, tab, macc,
                                                      msrow, scs);
        }
      } else if (LAYOUT == kQ4Planar) {
        Q4Half w;
        if (use) load_q4_tile_smem(tile, lane, w);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (use) q4_dot<NCOLS>(w, h, bb * P + p, act, rb, da, sa, nbq, acc, srow, scs);
      } else if (LAYOUT == kQ5Planar) {
        Q5Half w;
        if (use) load_q5_tile_smem(tile, lane, w);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (use) q5_dot<NCOLS>(w, h, bb * P + p, act, rb, da, sa, nbq, acc, srow, scs);
      } else {
        Q6Half w;
        if (use) load_q6_tile_smem(tile, lane, w);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (use) q6_dot<NCOLS>(w, h, bb * P + p, act, rb, da, nbq, acc, srow, scs);
      }
    }
    // halves of each row, then the group's K-slices in warp order.  With
    // P > 1 the batch's partials go to buffer j % 2: a warp writes the
    // buffer of batch j + 2 only after the group barrier of batch j + 1,
    // which the warp that reads batch j's partials passes after reading
    // them.
    if constexpr (MMA) {
      // the MMA lanes' row sums into the dp4a lanes' layout (row i, all
      // columns on lanes i and 16 + i), through this warp's partials
      float* wred = red + (P > 1 ? (size_t)(j & 1) * C * kMaxCols * kTileRows : 0) +
                    (size_t)warp * kMaxCols * kTileRows;
      __syncwarp();
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int col = 2 * mt + cc;
          if (col < NCOLS) wred[col * kTileRows + mg + 8 * rr] = macc[rr][cc][0] + macc[rr][cc][1];
        }
      __syncwarp();
#pragma unroll
      for (int c = 0; c < NCOLS; ++c) acc[c] = wred[c * kTileRows + i];
      __syncwarp();
    } else {
#pragma unroll
      for (int c = 0; c < NCOLS; ++c) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], 16);
    }
    if (!waited) {
      grid_dependency_wait();
      waited = true;
    }
    if constexpr (!CLUSTER) {
      if (P == 1) {
        if (valid && h == 0 && row < rows) {
#pragma unroll
          for (int c = 0; c < NCOLS; ++c) y[c * rows + row] = acc[c];
        }
        continue;
      }
      float* redj = red + (size_t)(j & 1) * C * kMaxCols * kTileRows;
      if (h == 0) {
#pragma unroll
        for (int c = 0; c < NCOLS; ++c) redj[(warp * kMaxCols + c) * kTileRows + i] = acc[c];
      }
      group_sync(2 + g, 32 * P);
      if (p == 0 && valid && h == 0 && row < rows) {
#pragma unroll
        for (int c = 0; c < NCOLS; ++c) {
          float sum = 0.0f;
          for (int q = 0; q < P; ++q) sum += redj[((g * P + q) * kMaxCols + c) * kTileRows + i];
          y[c * rows + row] = sum;
        }
      }
    } else {
      // this CTA's sum over its P K-slices, then the cluster's K-slices:
      // ranks 1..CS-1 send, rank 0 adds in rank order
      float part[NCOLS];
      if (P == 1) {
#pragma unroll
        for (int c = 0; c < NCOLS; ++c) part[c] = acc[c];
      } else {
        float* redj = red + (size_t)(j & 1) * C * kMaxCols * kTileRows;
        if (h == 0) {
#pragma unroll
          for (int c = 0; c < NCOLS; ++c) redj[(warp * kMaxCols + c) * kTileRows + i] = acc[c];
        }
        group_sync(2 + g, 32 * P);
#pragma unroll
        for (int c = 0; c < NCOLS; ++c) {
          float sum = 0.0f;
          if (p == 0 && h == 0)
            for (int q = 0; q < P; ++q) sum += redj[((g * P + q) * kMaxCols + c) * kTileRows + i];
          part[c] = sum;
        }
      }
      if (p == 0) {
        const int xb = (int)(j & 1);
        const uint32_t use = (uint32_t)(j >> 1);
        float* slot_base = xred + (size_t)xb * CS * G * NCOLS * kTileRows;
        if (rank != 0) {
          if (j >= 2 && !*fail && !mbar_wait_cluster(&xempty[xb], (use - 1) & 1u)) {
            *fail = 1;
            atomicOr(&g_fault_word, kFaultMbarTimeout);
          }
          if (h == 0) {
            float* mine = slot_base + ((size_t)(rank * G + g) * NCOLS) * kTileRows;
#pragma unroll
            for (int c = 0; c < NCOLS; ++c)
              st_cluster_f32(cluster_map(mine + c * kTileRows + i, 0), part[c]);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(cluster_map(&xfull[xb], 0));
        } else {
          if (!*fail && !mbar_wait_cluster(&xfull[xb], use & 1u)) {
            *fail = 1;
            atomicOr(&g_fault_word, kFaultMbarTimeout);
          }
          if (valid && h == 0 && row < rows) {
#pragma unroll
            for (int c = 0; c < NCOLS; ++c) {
              float sum = part[c];
              for (int q = 1; q < CS; ++q)
                sum += slot_base[((size_t)(q * G + g) * NCOLS + c) * kTileRows + i];
              y[c * rows + row] = sum;
            }
          }
          __syncwarp();
          // the buffer is free again; only where a later batch waits for it
          if (j + 2 < batches && lane > 0 && lane < CS)
            mbar_arrive_cluster(cluster_map(&xempty[xb], lane));
        }
      }
    }
  }
}

// ------------------------------------------------------------ host side ----

struct TmaCfg {
  int G, P, slots, grid;
  size_t smem;
  int CS;       // CTAs per cluster (K-split); 1: no cluster
  int mma = 0;  // 1: the tensor-core consumer (tma_mma.cuh)
};

// Column counts with a tensor-core instance (MMVQ_FLAG_TENSOR_CORE).
constexpr int kMmaMinCols = 4;

// The launch shape mmvq_gemv takes for a planar matrix (mmvq_tma.cu).
int planar_tma_config(int type, int64_t rows, int K, int ncols, TmaCfg* out);

}  // namespace mmvq
