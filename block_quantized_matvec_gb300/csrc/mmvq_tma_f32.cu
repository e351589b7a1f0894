// MMVQ with fp32 activation columns: the dense ring kernel of tma_dense.cuh
// in its fp32 instance, whose CTAs quantise the columns to Q8_1 themselves
// while the first weight stages stream in, so a decode step has no separate
// quantisation launch ("Strata" PR #2340 "int4 activation loads": the Q8_1
// columns are what the wide kernels read; PR #2207: the weights are read
// once for all 1-8 columns).  Every CTA needs every 32-block of every column,
// so this pays only while the quantisation is a round or two of the CTA's
// quads; larger calls (and the shapes the chooser runs on CTA pairs) take the
// quantiser kernel and the Q8_1 product instead, with the same results.
#include "tma_dense.cuh"

namespace mmvq {

int launch_quantize_q8_1(const float* x, int K, int ncols, int64_t ldx, void* xq, cudaStream_t s);
int launch_planar_tma(int type, const void* W, int64_t rows, int K, const void* xq, int ncols,
                      float* y, int32_t* sumi, uint32_t flags, cudaStream_t s);
int ensure_smem(const void* kern, size_t smem);
int device_sms();

// Rounds of quads (a 32-block per four lanes of the CTA's consumer warps)
// up to which the CTAs quantise the columns themselves.  Measured on GB300,
// one column as a dependent chain of decode steps: 2560 x 2560 5.6 -> 3.8 us,
// 10240 x 2560 9.0 -> 6.8 us, Q4_K 12288 x 2560 8.9 -> 6.5 us (one or two
// rounds); 2560 x 10240 (four rounds) 10.0 -> 11.1 us, so it stays two
// launches.
constexpr int kF32MaxRounds = 2;

template <int LAYOUT, int NCOLS>
static int launch_f32_t(const uint8_t* W, int64_t rows, int K, const float* x, int64_t ldx,
                        uint8_t* xq, float* y, uint32_t flags, const TmaCfg& cfg,
                        cudaStream_t stream) {
  auto kern = mmvq_planar_tma_kernel<LAYOUT, NCOLS, false, false, true>;
  if (ensure_smem((const void*)kern, cfg.smem) != MMVQ_OK) return MMVQ_ERR_CUDA;
  return launch_pdl(kern, dim3(cfg.grid), dim3(32 * (cfg.G * cfg.P + 1)), cfg.smem, stream, W,
                    rows, K, static_cast<const uint8_t*>(nullptr), y,
                    static_cast<int32_t*>(nullptr), cfg.slots, cfg.G, cfg.P, 1, flags, x, ldx, xq);
}

template <int LAYOUT>
static int launch_f32_l(const uint8_t* W, int64_t rows, int K, const float* x, int64_t ldx,
                        int ncols, uint8_t* xq, float* y, uint32_t flags, const TmaCfg& cfg,
                        cudaStream_t s) {
  switch (ncols) {
    case 1: return launch_f32_t<LAYOUT, 1>(W, rows, K, x, ldx, xq, y, flags, cfg, s);
    case 2: return launch_f32_t<LAYOUT, 2>(W, rows, K, x, ldx, xq, y, flags, cfg, s);
    case 3: return launch_f32_t<LAYOUT, 3>(W, rows, K, x, ldx, xq, y, flags, cfg, s);
    case 4: return launch_f32_t<LAYOUT, 4>(W, rows, K, x, ldx, xq, y, flags, cfg, s);
    case 5: return launch_f32_t<LAYOUT, 5>(W, rows, K, x, ldx, xq, y, flags, cfg, s);
    case 6: return launch_f32_t<LAYOUT, 6>(W, rows, K, x, ldx, xq, y, flags, cfg, s);
    case 7: return launch_f32_t<LAYOUT, 7>(W, rows, K, x, ldx, xq, y, flags, cfg, s);
    case 8: return launch_f32_t<LAYOUT, 8>(W, rows, K, x, ldx, xq, y, flags, cfg, s);
  }
  return MMVQ_ERR_NCOLS;
}

// One launch when the columns are a few rounds of the CTA's quads and the
// grid is at most two CTAs per SM: a persistent grid over a tall matrix (an
// LM head, three CTAs per SM) would quantise the columns in hundreds of CTAs
// for a product of tens of microseconds (measured 53.5 against 50.1 us per
// head step as two launches).
// MMVQ_FLAG_TENSOR_CORE: the fp32 instance is a dp4a one, so the flag
// takes the two launches.
static bool f32_fuses(const TmaCfg& cfg, int ncols, int K, uint32_t flags) {
  const int nquads = 8 * cfg.G * cfg.P;  // consumer threads / 4
  return cfg.CS == 1 && !(flags & MMVQ_FLAG_TENSOR_CORE) &&
         ncols * (K / kQK8) <= kF32MaxRounds * nquads &&
         cfg.grid <= 2 * device_sms();
}

// 1: the call runs as one launch (the CTAs quantise); 0: as the quantiser
// and the Q8_1 product.  Host-only.
int gemv_f32_fused(int type, int64_t rows, int K, int ncols, int* fused) {
  TmaCfg cfg;
  const int rc = planar_tma_config(type, rows, K, ncols, &cfg);
  if (rc != MMVQ_OK) return rc;
  *fused = f32_fuses(cfg, ncols, K, 0u) ? 1 : 0;
  return MMVQ_OK;
}

int launch_gemv_f32(int type, const void* W, int64_t rows, int K, const float* x, int64_t ldx,
                    int ncols, void* xq, float* y, uint32_t flags, cudaStream_t s) {
  TmaCfg cfg;
  int rc = planar_tma_config(type, rows, K, ncols, &cfg);
  if (rc != MMVQ_OK) return rc;
  uint8_t* q = static_cast<uint8_t*>(xq);
  if (!f32_fuses(cfg, ncols, K, flags)) {
    rc = launch_quantize_q8_1(x, K, ncols, ldx, xq, s);
    if (rc != MMVQ_OK) return rc;
    return launch_planar_tma(type, W, rows, K, xq, ncols, y, nullptr, flags, s);
  }
  const uint8_t* w = static_cast<const uint8_t*>(W);
  if (type == MMVQ_Q4_K_PLANAR) return launch_f32_l<kQ4Planar>(w, rows, K, x, ldx, ncols, q, y, flags, cfg, s);
  if (type == MMVQ_Q5_K_PLANAR) return launch_f32_l<kQ5Planar>(w, rows, K, x, ldx, ncols, q, y, flags, cfg, s);
  return launch_f32_l<kQ6Planar>(w, rows, K, x, ldx, ncols, q, y, flags, cfg, s);
}

// This translation unit's fault word, for mmvq_read_device_fault.
int read_clear_f32_fault_word(unsigned int* v) { return read_clear_fault_word(v); }

}  // namespace mmvq
