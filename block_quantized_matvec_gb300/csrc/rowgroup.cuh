// One warp's share of a 16-row group: its K-slice of blocks, streamed with
// register double buffering (planar Q6_K, GGUF Q4_K) or through a two-stage
// cp.async ring in shared memory (GGUF Q6_K, whose 210-byte blocks are only
// 2-byte aligned), then the fixed-order sum of the K-slices.
#pragma once

#include "kquant.cuh"

namespace mmvq {

constexpr int kGgufSlot = 224;                     // 14 aligned 16-byte chunks per Q6_K block
constexpr int kGgufStage = kTileRows * kGgufSlot;  // one warp, one block step

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* src, int src_bytes) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait1() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// Copies, for one warp, block b of the 16 rows of group rg into a stage:
// row i's 210 bytes sit in a 224-byte window starting at the 16-byte
// boundary (of the absolute address) at or below the block.  W itself need
// not be 16-byte aligned (an expert inside a stack of experts); a window
// may then start up to 15 bytes before W, inside the caller's allocation.
// Chunks past the end of the matrix are zero-filled, never read.
__device__ __forceinline__ void stage_q6_gguf(const uint8_t* __restrict__ W, int64_t total_bytes,
                                              int64_t rows, int nb, int64_t rg, int b, int lane,
                                              uint8_t* stage) {
  const uint8_t* end = W + total_bytes;
#pragma unroll
  for (int t = 0; t < 7; ++t) {
    const int q = lane + 32 * t;  // 0..223
    const int i = q / 14;
    const int ch = q - i * 14;
    const int64_t row = min(rg * kTileRows + i, rows - 1);
    const uint8_t* blk = W + (row * nb + b) * kQ6KBytes;
    const uint8_t* src =
        reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(blk) & ~uintptr_t(15)) + 16 * ch;
    const int64_t left = end - src;
    const int nbytes = left >= 16 ? 16 : (left > 0 ? (int)left : 0);
    cp_async16(stage + i * kGgufSlot + 16 * ch, nbytes ? src : W, nbytes);
  }
  cp_async_commit();
}

// Accumulates into acc[] this warp's blocks b = wk, wk+WK, ... of row group
// rg of matrix W (rows x nb blocks).  Lane L = 16h + i works on row 16rg+i,
// half h.  srow: per-row block-sum output (NULL unless dumping).
template <int LAYOUT, int NC>
__device__ __forceinline__ void rowgroup_dot(const uint8_t* __restrict__ W, int64_t rows, int nb,
                                             int64_t rg, int wk, int WK, int lane,
                                             const uint8_t* act, int rb, const float* da,
                                             const float* sa, int nbq, float (&acc)[NC],
                                             int32_t* srow, int64_t scs, uint8_t* stage) {
  const int i = lane & 15;
  const int h = lane >> 4;
  const int64_t row = rg * kTileRows + i;
  if (LAYOUT == kQ6Gguf) {
    const int64_t total_bytes = rows * nb * kQ6KBytes;
    const int64_t rr = min(row, rows - 1);
    int b = wk;
    int slot = 0;
    if (b < nb) stage_q6_gguf(W, total_bytes, rows, nb, rg, b, lane, stage);
    for (; b < nb; b += WK) {
      if (b + WK < nb)
        stage_q6_gguf(W, total_bytes, rows, nb, rg, b + WK, lane, stage + (slot ^ 1) * kGgufStage);
      else
        cp_async_commit();
      cp_async_wait1();
      __syncwarp();
      const int off = (int)(reinterpret_cast<uintptr_t>(W + (rr * nb + b) * kQ6KBytes) & 15);
      Q6Half cur;
      load_q6_gguf_smem(stage + slot * kGgufStage + i * kGgufSlot + off, h, cur);
      __syncwarp();
      q6_dot<NC>(cur, h, b, act, rb, da, nbq, acc, srow, scs);
      slot ^= 1;
    }
  } else {
    const int64_t rr = min(row, rows - 1);
    const uint8_t* wrow = W + (size_t)rr * nb * kQ4KBytes;
    int b = wk;
    Q4Half cur;
    if (b < nb) load_q4_gguf(wrow + (size_t)b * kQ4KBytes, h, cur);
    for (; b < nb; b += WK) {
      Q4Half nxt;
      if (b + WK < nb) load_q4_gguf(wrow + (size_t)(b + WK) * kQ4KBytes, h, nxt);
      q4_dot<NC>(cur, h, b, act, rb, da, sa, nbq, acc, srow, scs);
      cur = nxt;
    }
  }
}

// Sums the two halves of each row, then (WK > 1) the K-slices of the WR*WK
// warps in warp order through red[], and stores y[c*ldc + row].  Every
// thread of the CTA must call it (it holds __syncthreads when WK > 1).
template <int NC>
__device__ __forceinline__ void reduce_store(float (&acc)[NC], int lane, int wk, int WK, int wr,
                                             bool valid, int64_t row, int64_t rows, float* red,
                                             float* y, int64_t ldc) {
  const int i = lane & 15;
  const int h = lane >> 4;
#pragma unroll
  for (int c = 0; c < NC; ++c) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], 16);
  if (WK == 1) {
    if (h == 0 && valid && row < rows) {
#pragma unroll
      for (int c = 0; c < NC; ++c) y[c * ldc + row] = acc[c];
    }
    return;
  }
  const int warp = wr * WK + wk;
  if (h == 0) {
#pragma unroll
    for (int c = 0; c < NC; ++c) red[(warp * kMaxCols + c) * kTileRows + i] = acc[c];
  }
  __syncthreads();
  if (wk == 0 && h == 0 && valid && row < rows) {
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      float s = 0.0f;
      for (int k = 0; k < WK; ++k) s += red[((wr * WK + k) * kMaxCols + c) * kTileRows + i];
      y[c * ldc + row] = s;
    }
  }
  __syncthreads();
}

// Dynamic shared memory of a CTA with `nwarps` warps and `ncols` staged columns.
__host__ __device__ inline size_t mmvq_smem_bytes(int layout, int K, int ncols, int nwarps) {
  size_t s = (size_t)ncols * act_row_bytes(K);                            // quants
  s += (size_t)ncols * (K / kQK8) * 4 * (layout == kQ4Gguf ? 2 : 1);
  s += (size_t)nwarps * kMaxCols * kTileRows * 4;                          // K-slice partials
  if (layout == kQ6Gguf) s += (size_t)nwarps * 2 * kGgufStage;             // cp.async ring
  return s;
}

}  // namespace mmvq
