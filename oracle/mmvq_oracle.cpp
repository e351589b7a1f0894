// Plain single-threaded CPU oracle for block-quantized matrix-vector products
// (MMVQ) with Q8_1 activations.  TEST INFRASTRUCTURE ONLY: nothing on the
// product path may call it.  Only tests/, the smoke check and the bench's
// CPU-baseline leg use it.  It shares no code, header, table or constant
// generator with the CUDA path.
//
// What it computes, and where each step comes from:
//
//  * Q8_1 activation blocks (32 int8 quants, fp16 d and fp16 s = d*sum(q)).
//    "Strata" PR #2340 ("int4 activation loads"): the Q8_1 quants are 4-byte
//    aligned behind a small header; PR #1774 ("What changed"): each
//    sub-block value is "d * ds * sumi".  Per 32 values: amax, d = amax/127,
//    q = round-half-away(x/d), s = d*sum(q), d and s stored as fp16 (RNE).
//  * Q6_K weights (210 B per 256): ql[128] low nibbles, qh[64] 2-bit high
//    fields, int8 scales[16] (one per 16 weights), fp16 d; value
//    d*scale*(q-32).  PR #2340 ("Q6_K six-bit offset as SWAR"): the decode
//    subtracts 32 from the 6-bit code.  Field placement is the GGUF Q6_K
//    arrangement.
//  * Q4_K weights (144 B per 256): fp16 d, fp16 dmin, 12 bytes of packed
//    6-bit scales/mins for 8 sub-blocks of 32, qs[128] nibbles; value
//    d*sc*q - dmin*m (GGUF Q4_K arrangement).  The min term reaches the dot
//    product through the Q8_1 sum s.
//  * Q5_K weights (176 B per 256): the pages run Q5_K matrices through the
//    same wide kernels (PR #2340 "ld_i4_a4"; the A770 dense_bench table)
//    without giving the block; read as the GGUF Q5_K arrangement: fp16 d,
//    fp16 dmin, the Q4_K scale/min bytes, qh[32] (bit j of qh[l] is the
//    fifth bit of weight l of sub-block j) and qs[128] as in Q4_K; code
//    q in 0..31, value d*sc*q - dmin*m.
//  * Per-32-block integer sums (int8 dot products, PR #2746 "INT8 DP4A
//    operations, scales, FP32 accumulation"), the FP32 block term
//    d_w*d_a*sumi (minus dmin*m*s_a for Q4_K), and the FP32 sum over blocks
//    in index order (PR #1774: the sub-block order only changes last bits).
//  * Planar Q6_K repack and draft-row gather (PR #2340 "STRATA_Q6_PLANAR":
//    the head is converted at load into ql/qh/scales/d planes, same bytes;
//    the draft head's subset is gathered from the planar head).  The tile
//    order of the planes is this library's own layout, restated below from
//    its specification.
//  * Grouped expert products over per-expert token lists with empty groups
//    (PR #2746 "B70 validation": "empty groups"; issue #2801: the grouped
//    gate/up and down kernels), and SiLU(gate)*up requantised to Q8_1
//    between the gate/up and down calls.
//  * RMSNorm folded into the Q8_1 quantiser (PR #1774 "How it was checked" names the
//    opt-in fused norm, #1775, without a formula): the plain RMS norm with a
//    weight vector, mean square accumulated in fp64.
//
// Floating point: compiled with -O2 -ffp-contract=off, so every a*b+c below
// is two roundings, exactly as written.
//
// Parity pins: every function here is checked by tests/test_oracle_*.py
// against something other than itself (numpy's fp16 conversion, brute force
// over byte and field values with independently written encoders, closed
// forms, fp64 dot products of the original fields, invariants).  None is
// left unpinned.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

const int kQK = 256;        // weights per K-quant super-block
const int kQK8 = 32;        // values per Q8_1 block
const int kQ81Bytes = 36;   // fp16 d, fp16 s, int8 q[32]
const int kQ6KBytes = 210;  // ql[128] qh[64] scales[16] d
const int kQ4KBytes = 144;  // d dmin scales[12] qs[128]

const int kTypeQ4K = 12;
const int kTypeQ5K = 13;
const int kQ5KBytes = 176;  // d dmin scales[12] qh[32] qs[128]
const int kTypeQ5KPlanar = 1013;
const int kTileBytesQ5 = 2816;  // 16 x 176
const int kTypeQ6K = 14;
const int kTypeQ6KPlanar = 1014;
const int kTypeQ4KPlanar = 1012;

// Planar tile: 16 rows x one 256-block.
const int kTileRows = 16;
const int kTileBytes = 3360;     // Q6_K
const int kTileBytesQ4 = 2304;   // Q4_K

// ---------------------------------------------------------------- fp16 ----
// IEEE 754 binary16 <-> binary32, written from the format definition:
// 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; subnormals have
// exponent field 0 and value fraction * 2^-24.  Conversion to fp16 rounds to
// nearest, ties to even.

float f16_to_f32(uint16_t h) {
  const uint32_t sign = (uint32_t)(h >> 15) << 31;
  const uint32_t e = (h >> 10) & 0x1f;
  const uint32_t f = h & 0x3ff;
  uint32_t bits;
  if (e == 0) {
    if (f == 0) {
      bits = sign;
    } else {
      // Subnormal: value = f * 2^-24.  Normalise so the leading 1 is implicit.
      int exp = -14;  // exponent of the leading bit position 10
      uint32_t m = f;
      while ((m & 0x400) == 0) {
        m <<= 1;
        exp -= 1;
      }
      m &= 0x3ff;
      bits = sign | ((uint32_t)(exp + 127) << 23) | (m << 13);
    }
  } else if (e == 31) {
    bits = sign | 0x7f800000u | (f << 13);  // inf / nan (payload kept)
  } else {
    bits = sign | ((e - 15 + 127) << 23) | (f << 13);
  }
  float out;
  std::memcpy(&out, &bits, 4);
  return out;
}

uint16_t f32_to_f16(float v) {
  uint32_t x;
  std::memcpy(&x, &v, 4);
  const uint16_t sign = (uint16_t)((x >> 16) & 0x8000);
  const uint32_t e32 = (x >> 23) & 0xff;
  const uint32_t m32 = x & 0x7fffff;
  if (e32 == 0xff) {
    if (m32 == 0) return sign | 0x7c00;                        // inf
    return sign | 0x7c00 | 0x200 | (uint16_t)(m32 >> 13);      // quiet nan
  }
  const int e = (int)e32 - 127 + 15;  // re-biased exponent
  if (e >= 31) return sign | 0x7c00;  // too large even before rounding
  if (e <= 0) {
    // Result is subnormal (or zero) in fp16.  Value = M * 2^(e32-150) with
    // M the 24-bit significand; in units of 2^-24 that is M >> (14 - e).
    if (e < -10) return sign;  // |v| < 2^-25: rounds to zero
    const uint32_t M = m32 | 0x800000;
    const int shift = 14 - e;  // 14..24
    uint32_t r = M >> shift;
    const uint32_t rem = M & ((1u << shift) - 1);
    const uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (r & 1))) r += 1;
    return sign | (uint16_t)r;  // r may carry into the smallest normal
  }
  uint32_t r = ((uint32_t)e << 10) | (m32 >> 13);
  const uint32_t rem = m32 & 0x1fff;
  if (rem > 0x1000 || (rem == 0x1000 && (r & 1))) r += 1;  // may carry to inf
  return sign | (uint16_t)r;
}

uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
void wr16(uint8_t* p, uint16_t v) {
  p[0] = (uint8_t)(v & 0xff);
  p[1] = (uint8_t)(v >> 8);
}

// ---------------------------------------------------------------- Q8_1 ----

void quantize_block_q8_1(const float* x, uint8_t* out) {
  float amax = 0.0f;
  for (int i = 0; i < kQK8; ++i) {
    const float a = std::fabs(x[i]);
    if (a > amax) amax = a;
  }
  const float d = amax / 127.0f;
  int8_t q[kQK8];
  int sum = 0;
  for (int i = 0; i < kQK8; ++i) {
    int v = 0;
    if (d != 0.0f) v = (int)std::roundf(x[i] / d);  // half away from zero
    q[i] = (int8_t)v;
    sum += v;
  }
  const float s = d * (float)sum;
  wr16(out + 0, f32_to_f16(d));
  wr16(out + 2, f32_to_f16(s));
  std::memcpy(out + 4, q, kQK8);
}

// ---------------------------------------------------------------- Q6_K ----
// GGUF Q6_K: for half h (128 weights) and l = 0..31, with ql offset 64h and
// qh offset 32h:
//   w[128h + l]      = ql[64h+l]    low nibble | qh[32h+l] bits 0-1 << 4
//   w[128h + l + 32] = ql[64h+l+32] low nibble | qh[32h+l] bits 2-3 << 4
//   w[128h + l + 64] = ql[64h+l]   high nibble | qh[32h+l] bits 4-5 << 4
//   w[128h + l + 96] = ql[64h+l+32] high nibble| qh[32h+l] bits 6-7 << 4
// Signed weight q - 32, scale index = weight index / 16.

void decode_q6_k(const uint8_t* blk, uint8_t q[kQK], int8_t sc[16], float* d) {
  const uint8_t* ql = blk;
  const uint8_t* qh = blk + 128;
  for (int h = 0; h < 2; ++h) {
    for (int l = 0; l < 32; ++l) {
      const uint8_t lo0 = ql[64 * h + l];
      const uint8_t lo1 = ql[64 * h + l + 32];
      const uint8_t hi = qh[32 * h + l];
      q[128 * h + l + 0] = (uint8_t)((lo0 & 0xf) | (((hi >> 0) & 3) << 4));
      q[128 * h + l + 32] = (uint8_t)((lo1 & 0xf) | (((hi >> 2) & 3) << 4));
      q[128 * h + l + 64] = (uint8_t)((lo0 >> 4) | (((hi >> 4) & 3) << 4));
      q[128 * h + l + 96] = (uint8_t)((lo1 >> 4) | (((hi >> 6) & 3) << 4));
    }
  }
  std::memcpy(sc, blk + 192, 16);
  *d = f16_to_f32(rd16(blk + 208));
}

// ---------------------------------------------------------------- Q4_K ----
// GGUF Q4_K scales: 8 sub-blocks j of 32 weights.
//   j < 4:  sc = s[j] & 63,                    m = s[j+4] & 63
//   j >= 4: sc = (s[j+4] & 15) | (s[j-4] >> 6) << 4,
//           m  = (s[j+4] >> 4) | (s[j]   >> 6) << 4
// qs chunk c (32 bytes qs[32c..32c+31]): low nibbles are sub-block 2c, high
// nibbles sub-block 2c+1.  Value = d*sc*q - dmin*m.

void unpack_scales_mins(const uint8_t* s, uint8_t sc[8], uint8_t m[8]) {
  for (int j = 0; j < 8; ++j) {
    if (j < 4) {
      sc[j] = s[j] & 63;
      m[j] = s[j + 4] & 63;
    } else {
      sc[j] = (uint8_t)((s[j + 4] & 0xf) | ((s[j - 4] >> 6) << 4));
      m[j] = (uint8_t)((s[j + 4] >> 4) | ((s[j] >> 6) << 4));
    }
  }
}

void decode_q4_k(const uint8_t* blk, uint8_t q[kQK], uint8_t sc[8], uint8_t m[8], float* d,
                 float* dmin) {
  *d = f16_to_f32(rd16(blk + 0));
  *dmin = f16_to_f32(rd16(blk + 2));
  unpack_scales_mins(blk + 4, sc, m);
  const uint8_t* qs = blk + 16;
  for (int c = 0; c < 4; ++c) {
    for (int l = 0; l < 32; ++l) {
      q[64 * c + l] = qs[32 * c + l] & 0xf;
      q[64 * c + 32 + l] = qs[32 * c + l] >> 4;
    }
  }
}

// ---------------------------------------------------------------- Q5_K ----
// GGUF Q5_K: d | dmin | scales[12] (as Q4_K) | qh[32] | qs[128].  Sub-block j
// (weights 32j .. 32j+31) takes its low 4 bits from qs chunk j/2 (low nibble
// for even j, high for odd j) and, for weight l of the sub-block, its fifth
// bit from bit j of qh[l].  Value = d*sc*q - dmin*m, q in 0..31.
void decode_q5_k(const uint8_t* blk, uint8_t q[kQK], uint8_t sc[8], uint8_t m[8], float* d,
                 float* dmin) {
  *d = f16_to_f32(rd16(blk + 0));
  *dmin = f16_to_f32(rd16(blk + 2));
  unpack_scales_mins(blk + 4, sc, m);
  const uint8_t* qh = blk + 16;
  const uint8_t* qs = blk + 48;
  for (int j = 0; j < 8; ++j) {
    for (int l = 0; l < 32; ++l) {
      const int lo = (qs[32 * (j / 2) + l] >> (4 * (j % 2))) & 0xf;
      const int hi = (qh[l] >> j) & 1;
      q[32 * j + l] = (uint8_t)(lo | (hi << 4));
    }
  }
}

// ---------------------------------------------------- planar Q6_K tiles ----
// Tile T(g, b): rows 16g..16g+15, 256-block b; tiles ordered g-major.
// Lane L = 16h + i (i = row in group, h = half of the block):
//   [512j + 16L, +16),  j=0..3 : ql[64h + 16j .. +15]
//   [2048 + 512j + 16L, +16), j=0..1 : qh[32h + 16j .. +15]
//   [3072 + 8L, +8)            : scales[8h .. 8h+7]
//   [3328 + 2i, +2)            : d
// Rows beyond the matrix (padding of the last group) are zero bytes.

int64_t planar_bytes(int64_t rows, int K) {
  const int64_t groups = (rows + kTileRows - 1) / kTileRows;
  return groups * (int64_t)(K / kQK) * kTileBytes;
}

// Planar Q4_K tile T(g, b), 2304 bytes, lane L = 16u + i (u = half of the
// block: sub-blocks 4u..4u+3):
//   [512j + 16L, +16),  j=0..3 : qs[64u + 16j .. +15]
//   [2048 + 16i, +16)           : the 16-byte header (d, dmin, scales[12])
int64_t planar_bytes_q4(int64_t rows, int K) {
  const int64_t groups = (rows + kTileRows - 1) / kTileRows;
  return groups * (int64_t)(K / kQK) * kTileBytesQ4;
}

void block_to_tile_q4(const uint8_t* blk, int i, uint8_t* tile) {
  for (int u = 0; u < 2; ++u)
    for (int j = 0; j < 4; ++j)
      std::memcpy(tile + 512 * j + 16 * (16 * u + i), blk + 16 + 64 * u + 16 * j, 16);
  std::memcpy(tile + 2048 + 16 * i, blk, 16);
}

void tile_to_block_q4(const uint8_t* tile, int i, uint8_t* blk) {
  for (int u = 0; u < 2; ++u)
    for (int j = 0; j < 4; ++j)
      std::memcpy(blk + 16 + 64 * u + 16 * j, tile + 512 * j + 16 * (16 * u + i), 16);
  std::memcpy(blk, tile + 2048 + 16 * i, 16);
}

void unpack_planar_q4(const uint8_t* P, int64_t rows, int K, uint8_t* W) {
  const int nb = K / kQK;
  for (int64_t r = 0; r < rows; ++r)
    for (int b = 0; b < nb; ++b)
      tile_to_block_q4(P + ((r / kTileRows) * nb + b) * kTileBytesQ4, (int)(r % kTileRows),
                       W + (r * nb + b) * kQ4KBytes);
}

// Planar Q5_K tile T(g, b), 2816 bytes, lane L = 16u + i (u = half of the
// block: sub-blocks 4u..4u+3):
//   [512j + 16L, +16),  j=0..3 : qs[64u + 16j .. +15]
//   [2048 + 16i, +16)           : the 16-byte header (d, dmin, scales[12])
//   [2304 + 32i, +32)           : qh[0..31] (both halves read all of it)
int64_t planar_bytes_q5(int64_t rows, int K) {
  const int64_t groups = (rows + kTileRows - 1) / kTileRows;
  return groups * (int64_t)(K / kQK) * kTileBytesQ5;
}

void block_to_tile_q5(const uint8_t* blk, int i, uint8_t* tile) {
  for (int u = 0; u < 2; ++u)
    for (int j = 0; j < 4; ++j)
      std::memcpy(tile + 512 * j + 16 * (16 * u + i), blk + 48 + 64 * u + 16 * j, 16);
  std::memcpy(tile + 2048 + 16 * i, blk, 16);
  std::memcpy(tile + 2304 + 32 * i, blk + 16, 32);
}

void tile_to_block_q5(const uint8_t* tile, int i, uint8_t* blk) {
  for (int u = 0; u < 2; ++u)
    for (int j = 0; j < 4; ++j)
      std::memcpy(blk + 48 + 64 * u + 16 * j, tile + 512 * j + 16 * (16 * u + i), 16);
  std::memcpy(blk, tile + 2048 + 16 * i, 16);
  std::memcpy(blk + 16, tile + 2304 + 32 * i, 32);
}

void unpack_planar_q5(const uint8_t* P, int64_t rows, int K, uint8_t* W) {
  const int nb = K / kQK;
  for (int64_t r = 0; r < rows; ++r)
    for (int b = 0; b < nb; ++b)
      tile_to_block_q5(P + ((r / kTileRows) * nb + b) * kTileBytesQ5, (int)(r % kTileRows),
                       W + (r * nb + b) * kQ5KBytes);
}

// Copies one GGUF block (row i of tile) into / out of its tile slots.
void block_to_tile(const uint8_t* blk, int i, uint8_t* tile) {
  for (int h = 0; h < 2; ++h) {
    const int L = 16 * h + i;
    for (int j = 0; j < 4; ++j) std::memcpy(tile + 512 * j + 16 * L, blk + 64 * h + 16 * j, 16);
    for (int j = 0; j < 2; ++j)
      std::memcpy(tile + 2048 + 512 * j + 16 * L, blk + 128 + 32 * h + 16 * j, 16);
    std::memcpy(tile + 3072 + 8 * L, blk + 192 + 8 * h, 8);
  }
  std::memcpy(tile + 3328 + 2 * i, blk + 208, 2);
}

void tile_to_block(const uint8_t* tile, int i, uint8_t* blk) {
  for (int h = 0; h < 2; ++h) {
    const int L = 16 * h + i;
    for (int j = 0; j < 4; ++j) std::memcpy(blk + 64 * h + 16 * j, tile + 512 * j + 16 * L, 16);
    for (int j = 0; j < 2; ++j)
      std::memcpy(blk + 128 + 32 * h + 16 * j, tile + 2048 + 512 * j + 16 * L, 16);
    std::memcpy(blk + 192 + 8 * h, tile + 3072 + 8 * L, 8);
  }
  std::memcpy(blk + 208, tile + 3328 + 2 * i, 2);
}

// ------------------------------------------------------- block products ----

int block_bytes(int type) {
  if (type == kTypeQ6K) return kQ6KBytes;
  if (type == kTypeQ4K) return kQ4KBytes;
  if (type == kTypeQ5K) return kQ5KBytes;
  return 0;
}

struct Q81 {
  float d;
  float s;
  const int8_t* q;
};

Q81 q81_at(const uint8_t* xq, int nblk_per_col, int col, int kb) {
  const uint8_t* p = xq + ((int64_t)col * nblk_per_col + kb) * kQ81Bytes;
  Q81 r;
  r.d = f16_to_f32(rd16(p));
  r.s = f16_to_f32(rd16(p + 2));
  r.q = (const int8_t*)(p + 4);
  return r;
}

// For one 256-block of weights and one activation column: the 8 integer
// sums and the 8 FP32 block terms (and their magnitudes for the error bound).
void block_terms(int type, const uint8_t* blk, const uint8_t* xq, int nbq, int col, int b,
                 int32_t sumi_out[8], float t_out[8], float abs_out[8]) {
  if (type == kTypeQ6K) {
    uint8_t q[kQK];
    int8_t sc[16];
    float d;
    decode_q6_k(blk, q, sc, &d);
    for (int j = 0; j < 8; ++j) {
      const Q81 a = q81_at(xq, nbq, col, 8 * b + j);
      int32_t sumi = 0;
      for (int half = 0; half < 2; ++half) {
        int32_t acc = 0;
        for (int i = 0; i < 16; ++i) {
          const int n = 32 * j + 16 * half + i;
          acc += ((int32_t)q[n] - 32) * (int32_t)a.q[16 * half + i];
        }
        sumi += (int32_t)sc[2 * j + half] * acc;
      }
      const float t = (d * a.d) * (float)sumi;
      sumi_out[j] = sumi;
      t_out[j] = t;
      abs_out[j] = std::fabs(t);
    }
  } else {  // Q4_K and Q5_K: codes without offset, scale and min per 32
    uint8_t q[kQK], sc[8], m[8];
    float d, dmin;
    if (type == kTypeQ5K)
      decode_q5_k(blk, q, sc, m, &d, &dmin);
    else
      decode_q4_k(blk, q, sc, m, &d, &dmin);
    for (int j = 0; j < 8; ++j) {
      const Q81 a = q81_at(xq, nbq, col, 8 * b + j);
      int32_t acc = 0;
      for (int i = 0; i < 32; ++i) acc += (int32_t)q[32 * j + i] * (int32_t)a.q[i];
      const int32_t sumi = (int32_t)sc[j] * acc;
      const float tq = (d * a.d) * (float)sumi;
      const float tm = (dmin * (float)m[j]) * a.s;
      sumi_out[j] = sumi;
      t_out[j] = tq - tm;
      abs_out[j] = std::fabs(tq) + std::fabs(tm);
    }
  }
}

// Dense product over GGUF blocks: y[col][row] (ldy = row stride of y per
// column), optional bound[col][row] = sum |block terms|, optional
// sumi[col][row][K/32].
void gemv_gguf(int type, const uint8_t* W, int64_t rows, int K, const uint8_t* xq, int ncols,
               const int* col_of, float* y, int64_t ldy, float* bound, int32_t* sumi) {
  const int nb = K / kQK;
  const int nbq = K / kQK8;
  const int bb = block_bytes(type);
  for (int c = 0; c < ncols; ++c) {
    const int col = col_of ? col_of[c] : c;
    for (int64_t r = 0; r < rows; ++r) {
      float acc = 0.0f;
      float mag = 0.0f;
      for (int b = 0; b < nb; ++b) {
        int32_t s8[8];
        float t8[8], a8[8];
        block_terms(type, W + (r * nb + b) * bb, xq, nbq, col, b, s8, t8, a8);
        for (int j = 0; j < 8; ++j) {
          acc = acc + t8[j];
          mag = mag + a8[j];
          if (sumi) sumi[((int64_t)c * rows + r) * nbq + 8 * b + j] = s8[j];
        }
      }
      y[(int64_t)c * ldy + r] = acc;
      if (bound) bound[(int64_t)c * ldy + r] = mag;
    }
  }
}

void unpack_planar(const uint8_t* P, int64_t rows, int K, uint8_t* W) {
  const int nb = K / kQK;
  for (int64_t r = 0; r < rows; ++r) {
    const int64_t g = r / kTileRows;
    const int i = (int)(r % kTileRows);
    for (int b = 0; b < nb; ++b)
      tile_to_block(P + (g * nb + b) * kTileBytes, i, W + (r * nb + b) * kQ6KBytes);
  }
}

}  // namespace

// ================================================================ C ABI ====
// Return codes: 0 ok, -1 bad type, -2 bad shape.

extern "C" {

uint16_t orc_f32_to_f16(float v) { return f32_to_f16(v); }
float orc_f16_to_f32(uint16_t h) { return f16_to_f32(h); }

void orc_f32_to_f16_array(const float* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_f16(x[i]);
}
void orc_f16_to_f32_array(const uint16_t* x, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = f16_to_f32(x[i]);
}

// x: [ncols][ldx] fp32; quantises the first K of each column.
// xq: [ncols][K/32] Q8_1 blocks of 36 bytes.
int orc_quantize_q8_1(const float* x, int K, int ncols, int64_t ldx, uint8_t* xq) {
  if (K <= 0 || K % kQK8 != 0 || ncols < 0 || ldx < K) return -2;
  const int nbq = K / kQK8;
  for (int c = 0; c < ncols; ++c)
    for (int kb = 0; kb < nbq; ++kb)
      quantize_block_q8_1(x + (int64_t)c * ldx + kb * kQK8,
                          xq + ((int64_t)c * nbq + kb) * kQ81Bytes);
  return 0;
}

// Decoded fields of one block, for the pin tests.
void orc_decode_q6_k(const uint8_t* blk, uint8_t* q256, int8_t* sc16, float* d) {
  decode_q6_k(blk, q256, sc16, d);
}
void orc_decode_q4_k(const uint8_t* blk, uint8_t* q256, uint8_t* sc8, uint8_t* m8, float* d,
                     float* dmin) {
  decode_q4_k(blk, q256, sc8, m8, d, dmin);
}

int64_t orc_planar_bytes(int64_t rows, int K) { return planar_bytes(rows, K); }
int64_t orc_planar_bytes_q4(int64_t rows, int K) { return planar_bytes_q4(rows, K); }
int64_t orc_planar_bytes_q5(int64_t rows, int K) { return planar_bytes_q5(rows, K); }

void orc_decode_q5_k(const uint8_t* blk, uint8_t* q256, uint8_t* sc8, uint8_t* m8, float* d,
                     float* dmin) {
  decode_q5_k(blk, q256, sc8, m8, d, dmin);
}

int orc_repack_planar_q5(const uint8_t* W, int64_t rows, int K, uint8_t* P) {
  if (rows <= 0 || K <= 0 || K % kQK != 0) return -2;
  const int nb = K / kQK;
  std::memset(P, 0, (size_t)planar_bytes_q5(rows, K));
  for (int64_t r = 0; r < rows; ++r)
    for (int b = 0; b < nb; ++b)
      block_to_tile_q5(W + (r * nb + b) * kQ5KBytes, (int)(r % kTileRows),
                       P + ((r / kTileRows) * nb + b) * kTileBytesQ5);
  return 0;
}

int orc_unpack_planar_q5(const uint8_t* P, int64_t rows, int K, uint8_t* W) {
  if (rows <= 0 || K <= 0 || K % kQK != 0) return -2;
  unpack_planar_q5(P, rows, K, W);
  return 0;
}

int orc_repack_planar_q4(const uint8_t* W, int64_t rows, int K, uint8_t* P) {
  if (rows <= 0 || K <= 0 || K % kQK != 0) return -2;
  const int nb = K / kQK;
  std::memset(P, 0, (size_t)planar_bytes_q4(rows, K));
  for (int64_t r = 0; r < rows; ++r)
    for (int b = 0; b < nb; ++b)
      block_to_tile_q4(W + (r * nb + b) * kQ4KBytes, (int)(r % kTileRows),
                       P + ((r / kTileRows) * nb + b) * kTileBytesQ4);
  return 0;
}

int orc_unpack_planar_q4(const uint8_t* P, int64_t rows, int K, uint8_t* W) {
  if (rows <= 0 || K <= 0 || K % kQK != 0) return -2;
  unpack_planar_q4(P, rows, K, W);
  return 0;
}

int orc_repack_planar(const uint8_t* W, int64_t rows, int K, uint8_t* P) {
  if (rows <= 0 || K <= 0 || K % kQK != 0) return -2;
  const int nb = K / kQK;
  std::memset(P, 0, (size_t)planar_bytes(rows, K));
  for (int64_t r = 0; r < rows; ++r) {
    const int64_t g = r / kTileRows;
    const int i = (int)(r % kTileRows);
    for (int b = 0; b < nb; ++b)
      block_to_tile(W + (r * nb + b) * kQ6KBytes, i, P + (g * nb + b) * kTileBytes);
  }
  return 0;
}

int orc_unpack_planar(const uint8_t* P, int64_t rows, int K, uint8_t* W) {
  if (rows <= 0 || K <= 0 || K % kQK != 0) return -2;
  unpack_planar(P, rows, K, W);
  return 0;
}

// out = planar matrix of n rows: row k of out is row row_ids[k] of P.
int orc_gather_planar_rows(const uint8_t* P, int64_t rows, int K, const int32_t* row_ids, int n,
                           uint8_t* out) {
  if (rows <= 0 || K <= 0 || K % kQK != 0 || n <= 0) return -2;
  const int nb = K / kQK;
  std::vector<uint8_t> blk(kQ6KBytes);
  std::memset(out, 0, (size_t)planar_bytes(n, K));
  for (int k = 0; k < n; ++k) {
    const int64_t r = row_ids[k];
    if (r < 0 || r >= rows) return -2;
    for (int b = 0; b < nb; ++b) {
      tile_to_block(P + ((r / kTileRows) * nb + b) * kTileBytes, (int)(r % kTileRows), blk.data());
      block_to_tile(blk.data(), k % kTileRows, out + ((int64_t)(k / kTileRows) * nb + b) * kTileBytes);
    }
  }
  return 0;
}

// y: [ncols][rows]; bound (may be NULL): [ncols][rows] sum of |block terms|.
int orc_gemv(int type, const uint8_t* W, int64_t rows, int K, const uint8_t* xq, int ncols,
             float* y, float* bound) {
  if (rows <= 0 || K <= 0 || K % kQK != 0 || ncols < 1) return -2;
  if (type == kTypeQ6K || type == kTypeQ4K || type == kTypeQ5K) {
    gemv_gguf(type, W, rows, K, xq, ncols, nullptr, y, rows, bound, nullptr);
    return 0;
  }
  if (type == kTypeQ5KPlanar) {
    std::vector<uint8_t> g((size_t)(rows * (K / kQK) * kQ5KBytes));
    unpack_planar_q5(W, rows, K, g.data());
    gemv_gguf(kTypeQ5K, g.data(), rows, K, xq, ncols, nullptr, y, rows, bound, nullptr);
    return 0;
  }
  if (type == kTypeQ6KPlanar) {
    std::vector<uint8_t> g((size_t)(rows * (K / kQK) * kQ6KBytes));
    unpack_planar(W, rows, K, g.data());
    gemv_gguf(kTypeQ6K, g.data(), rows, K, xq, ncols, nullptr, y, rows, bound, nullptr);
    return 0;
  }
  if (type == kTypeQ4KPlanar) {
    std::vector<uint8_t> g((size_t)(rows * (K / kQK) * kQ4KBytes));
    unpack_planar_q4(W, rows, K, g.data());
    gemv_gguf(kTypeQ4K, g.data(), rows, K, xq, ncols, nullptr, y, rows, bound, nullptr);
    return 0;
  }
  return -1;
}

// sumi: [ncols][rows][K/32] per-32-block integer sums.
int orc_block_sums(int type, const uint8_t* W, int64_t rows, int K, const uint8_t* xq, int ncols,
                   int32_t* sumi) {
  if (rows <= 0 || K <= 0 || K % kQK != 0 || ncols < 1) return -2;
  std::vector<float> y((size_t)(ncols * rows));
  if (type == kTypeQ6K || type == kTypeQ4K || type == kTypeQ5K) {
    gemv_gguf(type, W, rows, K, xq, ncols, nullptr, y.data(), rows, nullptr, sumi);
    return 0;
  }
  if (type == kTypeQ5KPlanar) {
    std::vector<uint8_t> g((size_t)(rows * (K / kQK) * kQ5KBytes));
    unpack_planar_q5(W, rows, K, g.data());
    gemv_gguf(kTypeQ5K, g.data(), rows, K, xq, ncols, nullptr, y.data(), rows, nullptr, sumi);
    return 0;
  }
  if (type == kTypeQ6KPlanar) {
    std::vector<uint8_t> g((size_t)(rows * (K / kQK) * kQ6KBytes));
    unpack_planar(W, rows, K, g.data());
    gemv_gguf(kTypeQ6K, g.data(), rows, K, xq, ncols, nullptr, y.data(), rows, nullptr, sumi);
    return 0;
  }
  if (type == kTypeQ4KPlanar) {
    std::vector<uint8_t> g((size_t)(rows * (K / kQK) * kQ4KBytes));
    unpack_planar_q4(W, rows, K, g.data());
    gemv_gguf(kTypeQ4K, g.data(), rows, K, xq, ncols, nullptr, y.data(), rows, nullptr, sumi);
    return 0;
  }
  return -1;
}

// Per-expert token lists from top-k routing.  Groups are all experts in id
// order (expert_ids[e] = e, offsets has n_experts+1 entries); within a group
// the positions follow token order.  act_index[p] = token of position p,
// slot_of[p] = t*k + kk (the routing slot), both [T*k].
int orc_route_groups(const int32_t* topk, int T, int k, int n_experts, int32_t* expert_ids,
                     int32_t* offsets, int32_t* act_index, int32_t* slot_of) {
  if (T < 0 || k <= 0 || n_experts <= 0) return -2;
  int p = 0;
  for (int e = 0; e < n_experts; ++e) {
    expert_ids[e] = e;
    offsets[e] = p;
    for (int t = 0; t < T; ++t) {
      for (int kk = 0; kk < k; ++kk) {
        const int32_t x = topk[t * k + kk];
        if (x < 0 || x >= n_experts) return -2;
        if (x == e) {
          act_index[p] = t;
          slot_of[p] = t * k + kk;
          ++p;
        }
      }
    }
  }
  offsets[n_experts] = p;
  return 0;
}

// Grouped product: for group g, expert expert_ids[g], positions p in
// [offsets[g], offsets[g+1]): y[p][:rows] = W_expert x xq column act_index[p]
// (column p when act_index is NULL).  W: [n_experts][rows][K/256] blocks.
int orc_grouped(int type, const uint8_t* W, int n_experts, int64_t rows, int K,
                const int32_t* expert_ids, const int32_t* offsets, int n_groups,
                const int32_t* act_index, const uint8_t* xq, float* y, float* bound) {
  if (type != kTypeQ6K && type != kTypeQ4K) return -1;
  if (rows <= 0 || K <= 0 || K % kQK != 0 || n_groups < 0) return -2;
  const int64_t expert_bytes = rows * (K / kQK) * block_bytes(type);
  for (int g = 0; g < n_groups; ++g) {
    const int e = expert_ids[g];
    if (e < 0 || e >= n_experts) return -2;
    if (offsets[g + 1] < offsets[g]) return -2;
    for (int p = offsets[g]; p < offsets[g + 1]; ++p) {
      const int col = act_index ? act_index[p] : p;
      gemv_gguf(type, W + e * expert_bytes, rows, K, xq, 1, &col, y + (int64_t)p * rows, rows,
                bound ? bound + (int64_t)p * rows : nullptr, nullptr);
    }
  }
  return 0;
}

// RMSNorm then Q8_1, per column: the step before the activation quantiser
// when the norm is folded into it ("Strata" PR #1774 "How it was checked": the opt-in
// STRATA_GR_FUSE_NORM, #1775; the pages give no formula, so this is the
// plain RMS norm with a weight vector).  ms = (sum x_i^2 in fp64, index
// order) / K; scale = fp32(1 / sqrt(ms + eps)) in fp64; y_i = (x_i * scale)
// * w_i in fp32 (two roundings); then Q8_1 of y as orc_quantize_q8_1.
int orc_rmsnorm_quantize_q8_1(const float* x, const float* w, float eps, int K, int ncols,
                              int64_t ldx, uint8_t* xq, float* y_out) {
  if (K <= 0 || K % kQK8 != 0 || ncols < 0 || ldx < K || !(eps >= 0.0f)) return -2;
  const int nbq = K / kQK8;
  std::vector<float> y((size_t)K);
  for (int c = 0; c < ncols; ++c) {
    const float* xc = x + (int64_t)c * ldx;
    double ss = 0.0;
    for (int i = 0; i < K; ++i) ss += (double)xc[i] * (double)xc[i];
    const float scale = (float)(1.0 / std::sqrt(ss / (double)K + (double)eps));
    for (int i = 0; i < K; ++i) {
      const float t = xc[i] * scale;
      y[i] = t * w[i];
    }
    if (y_out) std::memcpy(y_out + (int64_t)c * K, y.data(), sizeof(float) * K);
    for (int kb = 0; kb < nbq; ++kb)
      quantize_block_q8_1(y.data() + kb * kQK8, xq + ((int64_t)c * nbq + kb) * kQ81Bytes);
  }
  return 0;
}

// gu: [n][2F] rows laid out [gate F | up F].  h = g/(1+exp(-g)) * u in fp32,
// then Q8_1 per 32 into xq [n][F/32].  h_out (may be NULL): [n][F].
int orc_silu_mul_quantize(const float* gu, int F, int n, uint8_t* xq, float* h_out) {
  if (F <= 0 || F % kQK8 != 0 || n < 0) return -2;
  std::vector<float> h((size_t)F);
  for (int r = 0; r < n; ++r) {
    const float* g = gu + (int64_t)r * 2 * F;
    const float* u = g + F;
    for (int i = 0; i < F; ++i) {
      const float sg = g[i] / (1.0f + std::exp(-g[i]));
      h[i] = sg * u[i];
    }
    if (h_out) std::memcpy(h_out + (int64_t)r * F, h.data(), sizeof(float) * F);
    for (int kb = 0; kb < F / kQK8; ++kb)
      quantize_block_q8_1(h.data() + kb * kQK8, xq + ((int64_t)r * (F / kQK8) + kb) * kQ81Bytes);
  }
  return 0;
}

}  // extern "C"
