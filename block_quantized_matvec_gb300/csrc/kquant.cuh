// Per-lane decode and integer dot products for one 256-weight block.
//
// Warp mapping (all kernels): a warp owns 16 rows; lane L = 16*h + i takes
// row i of the group and half h of each 256-block, i.e. the four Q8_1
// blocks 4h..4h+3 (128 weights).  The 16 lanes with the same h read the same
// activation bytes, so the activation loads from shared memory are
// broadcasts and the weight bytes are read from HBM exactly once for all
// columns ("Strata" PR #2207 / PR #1774: the wide kernels read the weights
// once for 1-8 columns).
#pragma once

#include "common.cuh"

namespace mmvq {

// ----------------------------------------------------------------- Q6_K ----
// Registers of one lane for one Q6_K block half: ql[64h..64h+63] as 16
// words, qh[32h..32h+31] as 8 words, scales[8h..8h+7] as 2 words, fp16 d.
struct Q6Half {
  uint32_t ql[16];
  uint32_t qh[8];
  uint32_t sc[2];
  uint32_t d;  // fp16 bits in the low half
};

// GGUF block staged in shared memory at a 2-byte aligned address `blk`:
// aligned word loads, realigned with a funnel shift when the block starts
// on an odd half-word.
__device__ __forceinline__ void load_q6_gguf_smem(const uint8_t* blk, int h, Q6Half& w) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(blk);
  const uint32_t* base = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
  const int sh = (int)(a & 2) * 8;  // 0 or 16
  {
    const uint32_t* p = base + 16 * h;  // ql[64h]
    uint32_t prev = p[0];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint32_t nxt = p[k + 1];
      w.ql[k] = __funnelshift_r(prev, nxt, sh);
      prev = nxt;
    }
  }
  {
    const uint32_t* p = base + 32 + 8 * h;  // qh[32h]
    uint32_t prev = p[0];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t nxt = p[k + 1];
      w.qh[k] = __funnelshift_r(prev, nxt, sh);
      prev = nxt;
    }
  }
  {
    const uint32_t* p = base + 48 + 2 * h;  // scales[8h]
    const uint32_t s0 = p[0], s1 = p[1], s2 = p[2];
    w.sc[0] = __funnelshift_r(s0, s1, sh);
    w.sc[1] = __funnelshift_r(s1, s2, sh);
  }
  w.d = *reinterpret_cast<const uint16_t*>(blk + 208);
}

__device__ __forceinline__ int sext8(uint32_t v) { return (int)(int8_t)(v & 0xff); }

// One lane's 128 weights of block `b` against NCOLS activation columns.
// act: padded quant rows (act_row_bytes(K) per column), da: d_a as floats
// [NCOLS][nbq].  acc[c] += d_w * sum_r d_a * sumi_r.  When sumi_out is set
// the per-32-block integer sums are stored at sumi_out[c*sumi_cs + kb].
template <int NCOLS>
__device__ __forceinline__ void q6_dot(const Q6Half& w, int h, int b, const uint8_t* act, int rb,
                                       const float* da, int nbq, float (&acc)[NCOLS],
                                       int32_t* sumi_out, int64_t sumi_cs) {
  float inner[NCOLS];
#pragma unroll
  for (int c = 0; c < NCOLS; ++c) inner[c] = 0.0f;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    int wv[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      uint32_t lo = (r & 1) ? w.ql[8 + m] : w.ql[m];
      if (r & 2) lo >>= 4;
      const uint32_t hi = ((w.qh[m] >> (2 * r)) & 0x03030303u) << 4;
      wv[m] = q6_minus_32((lo & 0x0f0f0f0fu) | hi);
    }
    const uint32_t scw = w.sc[r >> 1] >> (16 * (r & 1));
    const int sc0 = sext8(scw), sc1 = sext8(scw >> 8);
    const int kb = 8 * b + 4 * h + r;
#pragma unroll
    for (int c = 0; c < NCOLS; ++c) {
      const int4* a = reinterpret_cast<const int4*>(act + c * rb + act_off(kb));
      const int4 a0 = a[0];
      const int4 a1 = a[1];
      int s0 = dp4a(wv[0], a0.x, 0);
      s0 = dp4a(wv[1], a0.y, s0);
      s0 = dp4a(wv[2], a0.z, s0);
      s0 = dp4a(wv[3], a0.w, s0);
      int s1 = dp4a(wv[4], a1.x, 0);
      s1 = dp4a(wv[5], a1.y, s1);
      s1 = dp4a(wv[6], a1.z, s1);
      s1 = dp4a(wv[7], a1.w, s1);
      const int sumi = sc0 * s0 + sc1 * s1;
      if (sumi_out) sumi_out[c * sumi_cs + kb] = sumi;
      inner[c] = fmaf(da[c * nbq + kb], (float)sumi, inner[c]);
    }
  }
  const float dw = half_bits_to_float((uint16_t)w.d);
#pragma unroll
  for (int c = 0; c < NCOLS; ++c) acc[c] = fmaf(dw, inner[c], acc[c]);
}

// ----------------------------------------------------------------- Q4_K ----
// Registers of one lane for one Q4_K block half u: the 16-byte header (d,
// dmin, 12 scale bytes) and qs[64u..64u+63] as 16 words, i.e. qs chunks
// 2u and 2u+1 = sub-blocks 4u..4u+3.
struct Q4Half {
  uint32_t hdr[4];
  uint32_t qs[16];
};

__device__ __forceinline__ void load_q4_gguf(const uint8_t* __restrict__ blk, int u, Q4Half& w) {
  const uint4 hv = __ldg(reinterpret_cast<const uint4*>(blk));
  w.hdr[0] = hv.x;
  w.hdr[1] = hv.y;
  w.hdr[2] = hv.z;
  w.hdr[3] = hv.w;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(blk + 16 + 64 * u + 16 * j));
    w.qs[4 * j + 0] = v.x;
    w.qs[4 * j + 1] = v.y;
    w.qs[4 * j + 2] = v.z;
    w.qs[4 * j + 3] = v.w;
  }
}

// The same tile staged in shared memory.
__device__ __forceinline__ void load_q4_tile_smem(const uint8_t* tile, int lane, Q4Half& w) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 v = *reinterpret_cast<const uint4*>(tile + 512 * j + 16 * lane);
    w.qs[4 * j + 0] = v.x;
    w.qs[4 * j + 1] = v.y;
    w.qs[4 * j + 2] = v.z;
    w.qs[4 * j + 3] = v.w;
  }
  const uint4 hv = *reinterpret_cast<const uint4*>(tile + 2048 + 16 * (lane & 15));
  w.hdr[0] = hv.x;
  w.hdr[1] = hv.y;
  w.hdr[2] = hv.z;
  w.hdr[3] = hv.w;
}

__device__ __forceinline__ uint32_t byte_of(const uint32_t (&hdr)[4], int k) {
  // byte k (0..15) of the header; k is a compile-time constant after unrolling
  return (hdr[k >> 2] >> (8 * (k & 3))) & 0xffu;
}

// Scale and min of sub-block j of a Q4_K block from the header (scale bytes
// start at header byte 4).
__device__ __forceinline__ void q4_scale_min(const uint32_t (&hdr)[4], int j, int& sc, int& m) {
  if (j < 4) {
    sc = (int)(byte_of(hdr, 4 + j) & 63);
    m = (int)(byte_of(hdr, 8 + j) & 63);
  } else {
    sc = (int)((byte_of(hdr, 12 + (j - 4)) & 15) | ((byte_of(hdr, 4 + (j - 4)) >> 6) << 4));
    m = (int)((byte_of(hdr, 12 + (j - 4)) >> 4) | ((byte_of(hdr, 8 + (j - 4)) >> 6) << 4));
  }
}

// One lane's 128 weights (sub-blocks 4u..4u+3) of block b against NCOLS
// columns: acc[c] += d * sum d_a*sumi - dmin * sum s_a*m.
// FIFTH (Q5_K): the code's fifth bit, bit 4u+s of qh byte l, is added to
// the nibble of sub-block 4u+s (qh: the block's 32 qh bytes as 8 words).
template <int NCOLS, bool FIFTH>
__device__ __forceinline__ void q45_dot(const Q4Half& w, const uint32_t* qh, int u, int b,
                                        const uint8_t* act, int rb, const float* da,
                                        const float* sa, int nbq, float (&acc)[NCOLS],
                                        int32_t* sumi_out, int64_t sumi_cs) {
  float inner_d[NCOLS], inner_m[NCOLS];
#pragma unroll
  for (int c = 0; c < NCOLS; ++c) {
    inner_d[c] = 0.0f;
    inner_m[c] = 0.0f;
  }
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    // sub-block j = 4u + s: chunk 2u + (s >> 1), nibble s & 1
    int sc, m;
    int sc_lo, m_lo, sc_hi, m_hi;
    q4_scale_min(w.hdr, s, sc_lo, m_lo);
    q4_scale_min(w.hdr, 4 + s, sc_hi, m_hi);
    sc = u ? sc_hi : sc_lo;
    m = u ? m_hi : m_lo;
    int wv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint32_t v = w.qs[8 * (s >> 1) + k];
      if (s & 1) v >>= 4;
      wv[k] = (int)(v & 0x0f0f0f0fu);
      if (FIFTH) wv[k] |= (int)(((qh[k] >> (4 * u + s)) & 0x01010101u) << 4);
    }
    const int kb = 8 * b + 4 * u + s;
    const float mf = (float)m;
#pragma unroll
    for (int c = 0; c < NCOLS; ++c) {
      const int4* a = reinterpret_cast<const int4*>(act + c * rb + act_off(kb));
      const int4 a0 = a[0];
      const int4 a1 = a[1];
      int t = dp4a(wv[0], a0.x, 0);
      t = dp4a(wv[1], a0.y, t);
      t = dp4a(wv[2], a0.z, t);
      t = dp4a(wv[3], a0.w, t);
      t = dp4a(wv[4], a1.x, t);
      t = dp4a(wv[5], a1.y, t);
      t = dp4a(wv[6], a1.z, t);
      t = dp4a(wv[7], a1.w, t);
      const int sumi = sc * t;
      if (sumi_out) sumi_out[c * sumi_cs + kb] = sumi;
      inner_d[c] = fmaf(da[c * nbq + kb], (float)sumi, inner_d[c]);
      inner_m[c] = fmaf(sa[c * nbq + kb], mf, inner_m[c]);
    }
  }
  const float d = half_bits_to_float((uint16_t)(w.hdr[0] & 0xffff));
  const float dmin = half_bits_to_float((uint16_t)(w.hdr[0] >> 16));
#pragma unroll
  for (int c = 0; c < NCOLS; ++c) acc[c] = fmaf(d, inner_d[c], fmaf(-dmin, inner_m[c], acc[c]));
}

template <int NCOLS>
__device__ __forceinline__ void q4_dot(const Q4Half& w, int u, int b, const uint8_t* act, int rb,
                                       const float* da, const float* sa, int nbq,
                                       float (&acc)[NCOLS], int32_t* sumi_out, int64_t sumi_cs) {
  q45_dot<NCOLS, false>(w, nullptr, u, b, act, rb, da, sa, nbq, acc, sumi_out, sumi_cs);
}

// ----------------------------------------------------------------- Q5_K ----
// A Q5_K block half is a Q4_K half plus the block's qh bytes (every lane of
// a row needs all 32: bit 4u+s of qh[l] belongs to sub-block 4u+s).
struct Q5Half {
  Q4Half q4;
  uint32_t qh[8];
};

// Planar Q5_K tile in shared memory: qs and header as the Q4_K tile, the
// row's qh at [2304 + 32i, +32).
__device__ __forceinline__ void load_q5_tile_smem(const uint8_t* tile, int lane, Q5Half& w) {
  load_q4_tile_smem(tile, lane, w.q4);
  const uint4* hp = reinterpret_cast<const uint4*>(tile + 2304 + 32 * (lane & 15));
  const uint4 h0 = hp[0], h1 = hp[1];
  w.qh[0] = h0.x;
  w.qh[1] = h0.y;
  w.qh[2] = h0.z;
  w.qh[3] = h0.w;
  w.qh[4] = h1.x;
  w.qh[5] = h1.y;
  w.qh[6] = h1.z;
  w.qh[7] = h1.w;
}

template <int NCOLS>
__device__ __forceinline__ void q5_dot(const Q5Half& w, int u, int b, const uint8_t* act, int rb,
                                       const float* da, const float* sa, int nbq,
                                       float (&acc)[NCOLS], int32_t* sumi_out, int64_t sumi_cs) {
  q45_dot<NCOLS, true>(w.q4, w.qh, u, b, act, rb, da, sa, nbq, acc, sumi_out, sumi_cs);
}

}  // namespace mmvq
