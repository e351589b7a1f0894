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

}  // namespace mmvq
