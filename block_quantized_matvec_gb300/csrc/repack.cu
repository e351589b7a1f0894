// Load-time planar repack of Q6_K, draft-head row gather, and per-expert
// token lists from top-k routing.
//
// Planar ("Strata" PR #2340 "STRATA_Q6_PLANAR": the head is converted at
// load into ql / qh / scales / d planes, the same bytes, so each lane's
// loads are aligned 16-byte loads; the draft head's subset is gathered from
// the planar head).  Here the planes are kept per 16-row x 256-column tile
// in the order the MMVQ warps read them (see include/mmvq.h).
#include <algorithm>

#include "common.cuh"
#include "route.cuh"

namespace mmvq {

// What the 16-byte tile chunk q (0..209) holds: `pieces` pieces of `len`
// bytes, for consecutive tile lanes (or rows, for d) starting at lane0.
struct ChunkMap {
  int pieces;     // 1 (16-byte piece), 2 (two 8-byte scale pieces) or 8 (eight d's)
  int len;        // bytes per piece
  int lane0;      // first tile lane (ql/qh/scale pieces) or first row (d pieces)
  int blk_off;    // offset of the piece in the GGUF block for lane0 (h from lane)
};

__device__ __forceinline__ ChunkMap chunk_map(int q) {
  ChunkMap m;
  if (q < 128) {  // ql: j = q/32, lane = q%32 -> ql[64h + 16j]
    const int j = q >> 5, L = q & 31;
    m.pieces = 1; m.len = 16; m.lane0 = L; m.blk_off = 64 * (L >> 4) + 16 * j;
  } else if (q < 192) {  // qh: j = (q-128)/32 -> qh[32h + 16j]
    const int j = (q - 128) >> 5, L = (q - 128) & 31;
    m.pieces = 1; m.len = 16; m.lane0 = L; m.blk_off = 128 + 32 * (L >> 4) + 16 * j;
  } else if (q < 208) {  // scales: lanes 2(q-192), +1 -> scales[8h]
    const int L = 2 * (q - 192);
    m.pieces = 2; m.len = 8; m.lane0 = L; m.blk_off = 192 + 8 * (L >> 4);
  } else {  // d: rows 8(q-208) .. +7
    m.pieces = 8; m.len = 2; m.lane0 = 8 * (q - 208); m.blk_off = 208;
  }
  return m;
}

// One CTA per tile T(g, b); thread q < 210 writes tile chunk q.
__global__ void __launch_bounds__(256) repack_planar_kernel(const uint8_t* __restrict__ W,
                                                            int64_t rows, int nb,
                                                            uint8_t* __restrict__ P) {
  // Writes weights: no early launch of the next kernel, whose weight
  // stream may start before its own griddepcontrol.wait.
  grid_dependency_wait();
  const int64_t t = blockIdx.x;
  const int64_t g = t / nb;
  const int b = (int)(t - g * nb);
  const int q = threadIdx.x;
  if (q >= kTileBytes / 16) return;
  const ChunkMap m = chunk_map(q);
  alignas(16) uint8_t buf[16];
  for (int p = 0; p < m.pieces; ++p) {
    const int lane_or_row = m.lane0 + p;
    int i, off;
    if (m.pieces == 8) {
      i = lane_or_row;
      off = m.blk_off;
    } else {
      i = lane_or_row & 15;
      off = (m.pieces == 2) ? 192 + 8 * (lane_or_row >> 4) : m.blk_off;
    }
    const int64_t row = g * kTileRows + i;
    const uint8_t* src = W + (row * nb + b) * kQ6KBytes + off;
    for (int k = 0; k < m.len; k += 2) {
      uint16_t v = 0;
      if (row < rows) v = *reinterpret_cast<const uint16_t*>(src + k);
      buf[p * m.len + k] = (uint8_t)(v & 0xff);
      buf[p * m.len + k + 1] = (uint8_t)(v >> 8);
    }
  }
  *reinterpret_cast<uint4*>(P + t * kTileBytes + 16 * q) = *reinterpret_cast<const uint4*>(buf);
}

// Planar Q4_K: one CTA per tile; thread q < 144 writes 16-byte chunk q
// (q < 128: qs[64u + 16j] of lane L = q % 32, j = q / 32; else the header
// of row q - 128).  Q4_K blocks are 16-byte aligned, so reads are uint4.
__global__ void __launch_bounds__(256) repack_planar_q4_kernel(const uint8_t* __restrict__ W,
                                                               int64_t rows, int nb,
                                                               uint8_t* __restrict__ P) {
  // Writes weights: no early launch of the next kernel.
  grid_dependency_wait();
  const int64_t t = blockIdx.x;
  const int64_t g = t / nb;
  const int b = (int)(t - g * nb);
  const int q = threadIdx.x;
  if (q >= kTileBytesQ4 / 16) return;
  int i, off;
  if (q < 128) {
    const int j = q >> 5, L = q & 31;
    i = L & 15;
    off = 16 + 64 * (L >> 4) + 16 * j;
  } else {
    i = q - 128;
    off = 0;
  }
  const int64_t row = g * kTileRows + i;
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (row < rows) v = *reinterpret_cast<const uint4*>(W + (row * nb + b) * kQ4KBytes + off);
  *reinterpret_cast<uint4*>(P + t * kTileBytesQ4 + 16 * q) = v;
}

// Q5_K blocks -> planar Q5_K tiles (include/mmvq.h): one thread per 16-byte
// vector of the 2816-byte tile: 128 qs vectors, 16 headers, 32 qh halves.
__global__ void __launch_bounds__(256) repack_planar_q5_kernel(const uint8_t* __restrict__ W,
                                                               int64_t rows, int nb,
                                                               uint8_t* __restrict__ P) {
  // Writes weights: no early launch of the next kernel.
  grid_dependency_wait();
  const int64_t t = blockIdx.x;
  const int64_t g = t / nb;
  const int b = (int)(t - g * nb);
  const int q = threadIdx.x;
  if (q >= kTileBytesQ5 / 16) return;
  int i, off;
  if (q < 128) {  // qs[64u + 16j ..] of lane L = 16u + i at 512j + 16L
    const int j = q >> 5, L = q & 31;
    i = L & 15;
    off = 48 + 64 * (L >> 4) + 16 * j;
  } else if (q < 144) {  // header of row i at 2048 + 16i
    i = q - 128;
    off = 0;
  } else {  // qh half of row i at 2304 + 32i + 16 * half
    i = (q - 144) >> 1;
    off = 16 + 16 * ((q - 144) & 1);
  }
  const int64_t row = g * kTileRows + i;
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (row < rows) v = *reinterpret_cast<const uint4*>(W + (row * nb + b) * kQ5KBytes + off);
  *reinterpret_cast<uint4*>(P + t * kTileBytesQ5 + 16 * q) = v;
}

// One CTA per output tile; out row k = source row row_ids[k] (zero bytes
// for k >= n or an invalid id).
__global__ void __launch_bounds__(256) gather_planar_kernel(const uint8_t* __restrict__ P,
                                                            int64_t rows, int nb,
                                                            const int32_t* __restrict__ row_ids,
                                                            int n, uint8_t* __restrict__ out,
                                                            int32_t* __restrict__ status) {
  // Writes weights: no early launch of the next kernel, whose weight
  // stream may start before its own griddepcontrol.wait.
  grid_dependency_wait();
  const int64_t t = blockIdx.x;
  const int64_t g = t / nb;
  const int b = (int)(t - g * nb);
  const int q = threadIdx.x;
  if (q >= kTileBytes / 16) return;
  const ChunkMap m = chunk_map(q);
  alignas(16) uint8_t buf[16];
  for (int p = 0; p < m.pieces; ++p) {
    const int lane_or_row = m.lane0 + p;
    const int i = (m.pieces == 8) ? lane_or_row : (lane_or_row & 15);
    const int64_t k = g * kTileRows + i;
    int64_t src_row = -1;
    if (k < n) {
      const int32_t r = row_ids[k];
      if (r >= 0 && r < rows) {
        src_row = r;
      } else if (status) {
        *status = MMVQ_ERR_ROUTING;
      }
    }
    // same section and half in the source tile, the source row's lane
    int src_off;
    if (src_row < 0) {
      for (int k2 = 0; k2 < m.len; ++k2) buf[p * m.len + k2] = 0;
      continue;
    }
    const int si = (int)(src_row % kTileRows);
    if (m.pieces == 8) {
      src_off = 3328 + 2 * si;
    } else {
      const int h = lane_or_row >> 4;
      const int src_lane = 16 * h + si;
      if (m.pieces == 2) {
        src_off = 3072 + 8 * src_lane;
      } else if (q < 128) {
        src_off = 512 * (q >> 5) + 16 * src_lane;
      } else {
        src_off = 2048 + 512 * ((q - 128) >> 5) + 16 * src_lane;
      }
    }
    const uint8_t* src = P + ((src_row / kTileRows) * nb + b) * kTileBytes + src_off;
    for (int k2 = 0; k2 < m.len; k2 += 2) {
      const uint16_t v = *reinterpret_cast<const uint16_t*>(src + k2);
      buf[p * m.len + k2] = (uint8_t)(v & 0xff);
      buf[p * m.len + k2 + 1] = (uint8_t)(v >> 8);
    }
  }
  *reinterpret_cast<uint4*>(out + t * kTileBytes + 16 * q) = *reinterpret_cast<const uint4*>(buf);
}

// Per-expert token lists, one CTA (route_groups_cta); the next kernel may
// start at once (it waits for this one before it reads the lists).
__global__ void __launch_bounds__(1024) route_groups_kernel(const int32_t* __restrict__ topk,
                                                            int n_slots, int k, int n_experts,
                                                            int32_t* __restrict__ expert_ids,
                                                            int32_t* __restrict__ offsets,
                                                            int32_t* __restrict__ act_index,
                                                            int32_t* __restrict__ slot_of,
                                                            int32_t* __restrict__ status) {
  grid_launch_dependents();
  grid_dependency_wait();
  route_groups_cta(topk, n_slots, k, n_experts, expert_ids, offsets, act_index, slot_of, status);
}

int launch_repack_planar(int type, const void* W, int64_t rows, int K, void* P, cudaStream_t s) {
  const int nb = K / kQK;
  const int64_t tiles = ((rows + kTileRows - 1) / kTileRows) * nb;
  if (tiles > 0x7fffffff) return MMVQ_ERR_SHAPE;
  if (type == MMVQ_Q4_K)
    return launch_pdl(repack_planar_q4_kernel, dim3((unsigned)tiles), dim3(256), 0, s,
                      static_cast<const uint8_t*>(W), rows, nb, static_cast<uint8_t*>(P));
  if (type == MMVQ_Q5_K)
    return launch_pdl(repack_planar_q5_kernel, dim3((unsigned)tiles), dim3(256), 0, s,
                      static_cast<const uint8_t*>(W), rows, nb, static_cast<uint8_t*>(P));
  return launch_pdl(repack_planar_kernel, dim3((unsigned)tiles), dim3(256), 0, s,
                    static_cast<const uint8_t*>(W), rows, nb, static_cast<uint8_t*>(P));
}

int launch_gather_planar(const void* P, int64_t rows, int K, const int32_t* row_ids, int n,
                         void* out, int32_t* status, cudaStream_t s) {
  const int nb = K / kQK;
  const int64_t tiles = ((int64_t)(n + kTileRows - 1) / kTileRows) * nb;
  if (tiles > 0x7fffffff) return MMVQ_ERR_SHAPE;
  return launch_pdl(gather_planar_kernel, dim3((unsigned)tiles), dim3(256), 0, s,
                    static_cast<const uint8_t*>(P), rows, nb, row_ids, n,
                    static_cast<uint8_t*>(out), status);
}

int launch_route_groups(const int32_t* topk, int T, int k, int n_experts, int32_t* expert_ids,
                        int32_t* offsets, int32_t* act_index, int32_t* slot_of, int32_t* status,
                        cudaStream_t s) {
  // each thread owns four experts; at least two warps
  const int threads = std::max(64, std::min(1024, ((n_experts + 3) / 4 + 31) / 32 * 32));
  return launch_pdl(route_groups_kernel, dim3(1), dim3(threads), 0, s, topk, T * k, k, n_experts,
                    expert_ids, offsets, act_index, slot_of, status);
}

}  // namespace mmvq
