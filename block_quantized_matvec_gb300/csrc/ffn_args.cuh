// Arguments of the one-launch expert FFN (expert_ffn.cu), shared with the
// C ABI layer.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace mmvq {

struct FfnArgs {
  const uint8_t* w_gu;  // [E] planar experts of 2F x H (gate rows, then up rows)
  const uint8_t* w_dn;  // [E] planar experts of H x F
  int n_experts, H, F;
  const float* x;  // [T][ldx] hidden states
  int64_t ldx;
  int T;
  const int32_t* topk;  // [T][k]
  int k;
  float* gu;    // [T*k][2F]
  uint8_t* hq;  // [T*k][F/32] Q8_1
  float* y;     // [T*k][H]
  int32_t* expert_ids;  // optional outputs: the token lists
  int32_t* offsets;
  int32_t* act_index;
  int32_t* slot_of;
  uint8_t* xq;  // optional: [T][H/32] Q8_1 of x
  int32_t* status;
  uint32_t* sync;
  int S, g_gu, p_gu, g_dn, p_dn;
};

// Launches the expert FFN (type: MMVQ_Q4_K_PLANAR or MMVQ_Q6_K_PLANAR); with
// info != NULL it only reports the launch shape (8 ints).
int launch_expert_ffn(int type, const FfnArgs& args, cudaStream_t s, int32_t* info);
int launch_grid_barrier_selftest(uint32_t* ctr, uint32_t limit_us, cudaStream_t stream);

// mmvq_expert_ffn_noalloc: the layer's intermediates live in one fixed
// device array of kFfnScratchBytes (expert_ffn.cu), carved as
// [barrier word | xq | hq | gu], each part starting on a 256-byte boundary.
constexpr size_t kFfnScratchBytes = (size_t)2 << 20;

struct FfnScratchLayout {
  size_t xq, hq, gu, end;  // byte offsets; the barrier word sits at 0
};

inline FfnScratchLayout ffn_scratch_layout(int H, int F, int T, int k) {
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  const size_t n = (size_t)T * (size_t)k;
  FfnScratchLayout l;
  l.xq = 256;
  l.hq = l.xq + up((size_t)T * (size_t)(H / 32) * 36);
  l.gu = l.hq + up(n * (size_t)(F / 32) * 36);
  l.end = l.gu + n * 2 * (size_t)F * sizeof(float);
  return l;
}

// Fills args.sync, xq, hq and gu from the fixed array of the current device
// and launches as launch_expert_ffn does.
int launch_expert_ffn_noalloc(int type, FfnArgs args, cudaStream_t s);

}  // namespace mmvq
