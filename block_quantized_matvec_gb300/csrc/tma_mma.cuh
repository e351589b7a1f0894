// Tensor-core consumer of the dense ring kernel for several columns: the
// integer dot products of a 16-row planar tile against up to eight Q8_1
// columns as warp-level f16 MMAs (mma.sync m16n8k16, fp32 accumulate), one
// per 16-weight sub-block, with the same sums as the dp4a consumer
// ("Strata" PR #2207: 1-8 columns read the weights once; the products per
// sub-block and the fp32 scale chain are those of PR #1774 "d * ds * sumi").
// It reads the same staged columns and the same tiles, so the two consumers
// run in the same launch shapes.
//
// Why the products stay exact.  A weight enters as the f16 value 1024 + u,
// u its unsigned code (Q6_K 0..63, Q4_K 0..15, Q5_K 0..31), built by a byte
// permute that puts 0x64 above the code byte: integers below 2048 are exact
// in f16.  An activation q (-127..127) enters as the f16 integer q (the
// same permute on q + 128, less 1152).  Each product is then an integer
// below 2^17, and each MMA adds sixteen of them (or 32, two MMAs chained,
// for the 32-weight sub-blocks of Q4_K and Q5_K) to an fp32 start value
// C = -(1024 + o) * sum(q) over the same weights, o the code offset (32 for
// Q6_K, 0 otherwise), so that D = sum((u - o) * q): every term and partial
// sum is an integer below 2^23, exact in fp32 whatever order the tensor
// core adds them in.  The scale chain after the MMA is the dp4a consumer's:
// sc * D is that consumer's integer sum (exact in fp32 below 2^24), and the
// fp32 accumulation per 32-block, per block half and per 256-block follows
// the same order, so the two consumers give the same bits.
//
// Layout.  MMA lane (g, t) = (lane / 4, lane % 4) holds rows g and g + 8 of
// the tile, and of each 16-weight sub-block the four weights 4t .. 4t+3
// (one 32-bit word of codes); the MMA's k positions 2t, 2t+1 carry weights
// 4t, 4t+2 and its positions 2t+8, 2t+9 weights 4t+1, 4t+3 (any pairing of
// k with the weights works as long as A and B agree).  Its B fragment is
// word t of that sub-block in the staged column g (the column stride of
// the staging keeps the eight columns' words in different banks).  The
// start values, with d_a (and s_a) of columns 2t and 2t + 1, are built once
// per CTA after the staging into a table of eight floats per 32-block and
// t; the tile is read from the ring with 4-byte loads, conflict-free: a
// warp-wide load covers 32 consecutive words.
#pragma once
#include "ring.cuh"

namespace mmvq {

// Per 32-block kb and t: {d_a(c0), d_a(c1), then Q6_K: C(2kb, c0), C(2kb, c1),
// C(2kb+1, c0), C(2kb+1, c1); Q4_K/Q5_K: s_a(c0), s_a(c1), C(kb, c0),
// C(kb, c1)}, c0 = 2t, c1 = 2t + 1, zeros past ncols.  act, da, sa: the
// staging (act_row_bytes(Kc) bytes per column, d and s as [c][Kc/32]).
template <int LAYOUT>
__device__ __forceinline__ void mma_build_table(const uint8_t* act, int rb, const float* da,
                                                const float* sa, int nbq, int ncols, float* tab,
                                                int tid, int nthreads) {
  for (int e = tid; e < nbq * 4; e += nthreads) {
    const int kb = e >> 2, t = e & 3;
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int c = 2 * t + cc;
      if (c >= ncols) continue;
      const int4* q = reinterpret_cast<const int4*>(act + c * rb + act_off(kb));
      const int4 a = q[0], b = q[1];
      const int s0 = dp4a(a.w, 0x01010101, dp4a(a.z, 0x01010101, dp4a(a.y, 0x01010101,
                     dp4a(a.x, 0x01010101, 0))));
      const int s1 = dp4a(b.w, 0x01010101, dp4a(b.z, 0x01010101, dp4a(b.y, 0x01010101,
                     dp4a(b.x, 0x01010101, 0))));
      v[cc] = da[c * nbq + kb];
      if (LAYOUT == kQ6Planar) {
        v[2 + cc] = -1056.0f * (float)s0;
        v[4 + cc] = -1056.0f * (float)s1;
      } else {
        v[2 + cc] = sa[c * nbq + kb];
        v[4 + cc] = -1024.0f * (float)(s0 + s1);
      }
    }
    float4* o = reinterpret_cast<float4*>(tab + (size_t)e * 8);
    o[0] = make_float4(v[0], v[1], v[2], v[3]);
    o[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1, float c0,
                                          float c1, float c2, float c3) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2),
        "f"(c3));
}

// Codes (bytes u0..u3) of one row's word -> the A registers 1024 + u for
// weights (4t, 4t+2) and (4t+1, 4t+3).
__device__ __forceinline__ uint32_t codes_f16_even(uint32_t u) {
  return __byte_perm(u, 0x64646464u, 0x4240);
}
__device__ __forceinline__ uint32_t codes_f16_odd(uint32_t u) {
  return __byte_perm(u, 0x64646464u, 0x4341);
}

// The lane's base in the staging for 256-block blk: word t of column g
// (column 0 for a lane past ncols, whose B stays zero), so that the word of
// 16-block 2kb + half, kb = 8 blk + j, sits at base + act_off(j) + 16 half
// (act_off(8 blk + j) = 288 blk + act_off(j) for j < 8).
template <int NCOLS>
__device__ __forceinline__ const uint8_t* act_lane_base(const uint8_t* act, int rb, int blk, int g,
                                                        int t) {
  return act + ((NCOLS >= 8 || g < NCOLS) ? g : 0) * rb + 288 * blk + 4 * t;
}

// Word w (int8 q0..q3) of a 16-block of staged column g -> the B registers
// f16 (q0, q2) and (q1, q3), exact; zeros past ncols (no branch).
template <int NCOLS>
__device__ __forceinline__ void act_f16_pairs(const uint8_t* p, int g, uint32_t& b0,
                                              uint32_t& b1) {
  const bool on = NCOLS >= 8 || g < NCOLS;
  const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
  const uint32_t u = w ^ 0x80808080u;  // q + 128 per byte
  const __half2 off = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  const uint32_t lo = __byte_perm(u, 0x64646464u, 0x4240);  // 1152 + q0, 1152 + q2
  const uint32_t hi = __byte_perm(u, 0x64646464u, 0x4341);  // 1152 + q1, 1152 + q3
  const __half2 x = __hsub2(*reinterpret_cast<const __half2*>(&lo), off);
  const __half2 y = __hsub2(*reinterpret_cast<const __half2*>(&hi), off);
  b0 = on ? *reinterpret_cast<const uint32_t*>(&x) : 0u;
  b1 = on ? *reinterpret_cast<const uint32_t*>(&y) : 0u;
}

// ------------------------------------------------------------------ Q6_K --
// One lane's words of a planar Q6_K tile (rows g, g + 8): ql words
// 16h + 8a + 4b + t of each row (a: 32-chunk parity, b: 16-block in the
// chunk), qh words 8h + 4b + t, the row's 16 scale bytes and d.
struct Q6Mma {
  uint32_t ql[2][2][2][2];  // [row][h][a][b]
  uint32_t qh[2][2][2];     // [row][h][b]
  uint32_t sc[2][4];        // [row][word]
  uint32_t d[2];
};

__device__ __forceinline__ void load_q6_mma(const uint8_t* tile, int g, int t, Q6Mma& w) {
  const uint32_t* t32 = reinterpret_cast<const uint32_t*>(tile);
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int i = g + 8 * rr;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b) w.ql[rr][h][a][b] = t32[4 * (32 * (2 * a + b) + 16 * h + i) + t];
#pragma unroll
      for (int b = 0; b < 2; ++b) w.qh[rr][h][b] = t32[4 * (128 + 32 * b + 16 * h + i) + t];
      const uint2 s = *reinterpret_cast<const uint2*>(tile + 3072 + 8 * (16 * h + i));
      w.sc[rr][2 * h] = s.x;
      w.sc[rr][2 * h + 1] = s.y;
    }
    w.d[rr] = *reinterpret_cast<const uint16_t*>(tile + 3328 + 2 * i);
  }
}

// acc[row][col][h] += the tile's contribution (256-block blk of the staged
// K-range), per block half h as the dp4a consumer's lane of that half.
// SUMI: also store each per-32-block integer sum at srow[rr][col*scs + kb].
template <int NCOLS, bool SUMI>
__device__ __forceinline__ void q6_mma(const Q6Mma& w, int blk, int lane, const uint8_t* act,
                                       int rb, const float* tab, float (&acc)[2][2][2],
                                       int32_t* const (&srow)[2], int64_t scs) {
  const int g = lane >> 2, t = lane & 3;
  const uint8_t* ab = act_lane_base<NCOLS>(act, rb, blk, g, t);
  const float* tb = tab + 256 * blk + 8 * t;  // entry (kb, t) at 32 kb + 8 t
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float inner[2][2] = {{0.0f, 0.0f}, {0.0f, 0.0f}};
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int kb = 8 * blk + 4 * h + r;
      const float4* tp = reinterpret_cast<const float4*>(tb + 32 * (4 * h + r));
      const float4 t0 = tp[0], t1 = tp[1];
      float D[2][4];
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        uint32_t A[4];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const uint32_t lo = (w.ql[rr][h][r & 1][b] >> (4 * (r >> 1))) & 0x0f0f0f0fu;
          const uint32_t hi = ((w.qh[rr][h][b] >> (2 * r)) & 0x03030303u) << 4;
          const uint32_t u = lo | hi;
          A[rr] = codes_f16_even(u);
          A[2 + rr] = codes_f16_odd(u);
        }
        uint32_t b0, b1;
        act_f16_pairs<NCOLS>(ab + 144 * h + 32 * r + 16 * b, g, b0, b1);
        const float c0 = b ? t1.x : t0.z, c1 = b ? t1.y : t0.w;
        mma_16816(D[b], A[0], A[1], A[2], A[3], b0, b1, c0, c1, c0, c1);
      }
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const uint32_t scw = w.sc[rr][2 * h + (r >> 1)] >> (16 * (r & 1));
        const float sc0 = (float)sext8(scw), sc1 = (float)sext8(scw >> 8);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int v = 2 * rr + cc;
          const float s = fmaf(sc1, D[1][v], sc0 * D[0][v]);
          if (SUMI) {
            const int col = 2 * t + cc;
            if (srow[rr] && col < NCOLS) srow[rr][col * scs + kb] = (int)s;
          }
          inner[rr][cc] = fmaf(cc ? t0.y : t0.x, s, inner[rr][cc]);
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const float dw = half_bits_to_float((uint16_t)w.d[rr]);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) acc[rr][cc][h] = fmaf(dw, inner[rr][cc], acc[rr][cc][h]);
    }
  }
}

// ------------------------------------------------------------ Q4_K, Q5_K --
// One lane's words of a planar Q4_K / Q5_K tile (rows g, g + 8): qs words
// 8c + 4m + t of each row (c: 32-byte chunk = sub-block pair, m: 16-block in
// the sub-block), the 16-byte header, and for Q5_K the qh words 4m + t.
struct Q45Mma {
  uint32_t qs[2][4][2];  // [row][chunk][m]
  uint32_t hdr[2][4];
  uint32_t qh[2][2];     // [row][m] (Q5_K)
};

template <bool FIFTH>
__device__ __forceinline__ void load_q45_mma(const uint8_t* tile, int g, int t, Q45Mma& w) {
  const uint32_t* t32 = reinterpret_cast<const uint32_t*>(tile);
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int i = g + 8 * rr;
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int mm = 0; mm < 2; ++mm)
        w.qs[rr][c][mm] = t32[4 * (32 * (2 * (c & 1) + mm) + 16 * (c >> 1) + i) + t];
    const uint4 hv = *reinterpret_cast<const uint4*>(tile + 2048 + 16 * i);
    w.hdr[rr][0] = hv.x;
    w.hdr[rr][1] = hv.y;
    w.hdr[rr][2] = hv.z;
    w.hdr[rr][3] = hv.w;
    if (FIFTH) {
#pragma unroll
      for (int mm = 0; mm < 2; ++mm) w.qh[rr][mm] = t32[(2304 + 32 * i) / 4 + 4 * mm + t];
    }
  }
}

template <int NCOLS, bool FIFTH, bool SUMI>
__device__ __forceinline__ void q45_mma(const Q45Mma& w, int blk, int lane, const uint8_t* act,
                                        int rb, const float* tab, float (&acc)[2][2][2],
                                        int32_t* const (&srow)[2], int64_t scs) {
  const int g = lane >> 2, t = lane & 3;
  const uint8_t* ab = act_lane_base<NCOLS>(act, rb, blk, g, t);
  const float* tb = tab + 256 * blk + 8 * t;  // entry (kb, t) at 32 kb + 8 t
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float inner_d[2][2] = {{0.0f, 0.0f}, {0.0f, 0.0f}};
    float inner_m[2][2] = {{0.0f, 0.0f}, {0.0f, 0.0f}};
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int S = 4 * h + s;  // sub-block of 32
      const int kb = 8 * blk + S;
      const float4* tp = reinterpret_cast<const float4*>(tb + 32 * S);
      const float4 t0 = tp[0], t1 = tp[1];
      float D[4] = {t1.x, t1.y, t1.x, t1.y};
#pragma unroll
      for (int mm = 0; mm < 2; ++mm) {
        uint32_t A[4];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          uint32_t u = (w.qs[rr][S >> 1][mm] >> (4 * (S & 1))) & 0x0f0f0f0fu;
          if (FIFTH) u |= ((w.qh[rr][mm] >> S) & 0x01010101u) << 4;
          A[rr] = codes_f16_even(u);
          A[2 + rr] = codes_f16_odd(u);
        }
        uint32_t b0, b1;
        act_f16_pairs<NCOLS>(ab + 144 * h + 32 * s + 16 * mm, g, b0, b1);
        mma_16816(D, A[0], A[1], A[2], A[3], b0, b1, D[0], D[1], D[2], D[3]);
      }
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        int sc, mn;
        q4_scale_min(w.hdr[rr], S, sc, mn);
        const float scf = (float)sc, mf = (float)mn;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const float sumi = scf * D[2 * rr + cc];
          if (SUMI) {
            const int col = 2 * t + cc;
            if (srow[rr] && col < NCOLS) srow[rr][col * scs + kb] = (int)sumi;
          }
          inner_d[rr][cc] = fmaf(cc ? t0.y : t0.x, sumi, inner_d[rr][cc]);
          inner_m[rr][cc] = fmaf(cc ? t0.w : t0.z, mf, inner_m[rr][cc]);
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const float d = half_bits_to_float((uint16_t)(w.hdr[rr][0] & 0xffff));
      const float dmin = half_bits_to_float((uint16_t)(w.hdr[rr][0] >> 16));
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
        acc[rr][cc][h] = fmaf(d, inner_d[rr][cc], fmaf(-dmin, inner_m[rr][cc], acc[rr][cc][h]));
    }
  }
}

}  // namespace mmvq
