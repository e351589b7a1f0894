// C ABI of libmmvq.so (declared in include/mmvq.h).  Every entry point
// checks its arguments on the host before any CUDA call, then launches
// asynchronously on the caller's stream.  Nothing is allocated here.
#include <cstdint>

#include "common.cuh"
#include "ffn_args.cuh"

namespace mmvq {
int launch_quantize_q8_1(const float* x, int K, int ncols, int64_t ldx, void* xq, cudaStream_t s);
int launch_silu_mul_quantize(const float* gu, int F, int n, void* xq, float* h_out, cudaStream_t s);
int launch_quantize_route(const float* x, int K, int ncols, int64_t ldx, void* xq,
                          const int32_t* topk, int T, int k, int n_experts, int32_t* expert_ids,
                          int32_t* token_offsets, int32_t* act_index, int32_t* slot_of,
                          int32_t* status, cudaStream_t stream);
int launch_rmsnorm_quantize(const float* x, const float* w, float eps, int K, int ncols,
                            int64_t ldx, void* xq, float* y_out, cudaStream_t s);
int launch_dense(int type, const void* W, int64_t rows, int K, const void* xq, int ncols, float* y,
                 int32_t* sumi, uint32_t flags, cudaStream_t s);
int launch_grouped(int type, const void* W, int n_experts, int64_t rows, int K,
                   const int32_t* expert_ids, const int32_t* offsets, int n_groups,
                   const int32_t* act_index, const void* xq, int n_xq_cols, float* y,
                   int32_t* status, cudaStream_t s);
int launch_repack_planar(int type, const void* W, int64_t rows, int K, void* P, cudaStream_t s);
int launch_gather_planar(const void* P, int64_t rows, int K, const int32_t* row_ids, int n,
                         void* out, int32_t* status, cudaStream_t s);
int read_device_fault(int* fault, cudaStream_t stream);
int launch_wait_timeout_selftest(uint32_t limit_us, cudaStream_t stream);
int dense_shape(int type, int64_t rows, int K, int ncols, int32_t* info);
int launch_gemv_f32(int type, const void* W, int64_t rows, int K, const float* x, int64_t ldx,
                    int ncols, void* xq, float* y, uint32_t flags, cudaStream_t s);
int gemv_f32_fused(int type, int64_t rows, int K, int ncols, int* fused);
int launch_route_groups(const int32_t* topk, int T, int k, int n_experts, int32_t* expert_ids,
                        int32_t* offsets, int32_t* act_index, int32_t* slot_of, int32_t* status,
                        cudaStream_t s);
}  // namespace mmvq

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_weights_shape(int64_t rows, int K) {
  if (rows < 1 || rows > 0x7fffffffLL) return MMVQ_ERR_SHAPE;
  if (K < mmvq::kQK || K > mmvq::kMaxK || K % mmvq::kQK != 0) return MMVQ_ERR_SHAPE;
  return MMVQ_OK;
}

}  // namespace

extern "C" {

int mmvq_version(void) { return 10000; }

const char* mmvq_strerror(int code) {
  switch (code) {
    case MMVQ_OK: return "ok";
    case MMVQ_ERR_TYPE: return "unsupported weight type for this call";
    case MMVQ_ERR_SHAPE: return "bad shape (K must be a multiple of 256, at most 16384; sizes >= 1)";
    case MMVQ_ERR_NCOLS: return "ncols must be in 1..8";
    case MMVQ_ERR_NULL: return "a required pointer is NULL";
    case MMVQ_ERR_ALIGN: return "a pointer breaks its alignment rule (16 B for W/xq/out, 4 B otherwise)";
    case MMVQ_ERR_ROUTING: return "routing lists rejected";
    case MMVQ_ERR_CUDA: return "CUDA launch failed (no usable sm_103a device?)";
    case MMVQ_ERR_SCRATCH:
      return "the layer's intermediates exceed the fixed scratch of mmvq_expert_ffn_noalloc "
             "(MMVQ_NOALLOC_SCRATCH_BYTES)";
  }
  return "unknown mmvq status";
}

int mmvq_quantize_q8_1(const float* x, int K, int ncols, int64_t ldx, void* xq,
                       mmvq_stream_t stream) {
  if (!x || !xq) return MMVQ_ERR_NULL;
  if (K <= 0 || K % mmvq::kQK8 != 0 || ldx < K || ncols < 1 || ncols > 65535) return MMVQ_ERR_SHAPE;
  if (!aligned(x, 4) || !aligned(xq, 16)) return MMVQ_ERR_ALIGN;
  return mmvq::launch_quantize_q8_1(x, K, ncols, ldx, xq, (cudaStream_t)stream);
}

int mmvq_quantize_route_groups(const float* x, int K, int ncols, int64_t ldx, void* xq,
                               const int32_t* topk, int T, int k, int n_experts,
                               int32_t* expert_ids, int32_t* token_offsets, int32_t* act_index,
                               int32_t* slot_of, int32_t* status, mmvq_stream_t stream) {
  if (!x || !xq || !expert_ids || !token_offsets || !act_index || !slot_of) return MMVQ_ERR_NULL;
  if (T > 0 && !topk) return MMVQ_ERR_NULL;
  if (K <= 0 || K % mmvq::kQK8 != 0 || ldx < K || ncols < 1 || ncols > 65535) return MMVQ_ERR_SHAPE;
  if (n_experts < 1 || n_experts > 4096 || T < 0 || k < 1 || (int64_t)T * k > 65536)
    return MMVQ_ERR_SHAPE;
  if (!aligned(x, 4) || !aligned(xq, 16) || (topk && !aligned(topk, 4)) ||
      !aligned(expert_ids, 4) || !aligned(token_offsets, 4) || !aligned(act_index, 4) ||
      !aligned(slot_of, 4) || (status && !aligned(status, 4)))
    return MMVQ_ERR_ALIGN;
  return mmvq::launch_quantize_route(x, K, ncols, ldx, xq, topk, T, k, n_experts, expert_ids,
                                     token_offsets, act_index, slot_of, status,
                                     (cudaStream_t)stream);
}

static bool dense_type(int type) {
  return type == MMVQ_Q4_K || type == MMVQ_Q6_K || type == MMVQ_Q4_K_PLANAR ||
         type == MMVQ_Q6_K_PLANAR || type == MMVQ_Q5_K_PLANAR;
}

static bool grouped_type(int type) {
  return type == MMVQ_Q4_K || type == MMVQ_Q6_K || type == MMVQ_Q4_K_PLANAR ||
         type == MMVQ_Q6_K_PLANAR;
}

static bool repack_source_type(int type) {
  return type == MMVQ_Q6_K || type == MMVQ_Q4_K || type == MMVQ_Q5_K;
}

static int tile_bytes_of_source(int type) {
  return type == MMVQ_Q4_K ? mmvq::kTileBytesQ4
                           : type == MMVQ_Q5_K ? mmvq::kTileBytesQ5 : mmvq::kTileBytes;
}

static int gemv_checks(int type, const void* W, int64_t rows, int K, const void* xq, int ncols,
                       const void* out) {
  if (!dense_type(type)) return MMVQ_ERR_TYPE;
  if (!W || !xq || !out) return MMVQ_ERR_NULL;
  const int rc = check_weights_shape(rows, K);
  if (rc) return rc;
  if (ncols < 1 || ncols > mmvq::kMaxCols) return MMVQ_ERR_NCOLS;
  if (!aligned(W, 16) || !aligned(xq, 16) || !aligned(out, 4)) return MMVQ_ERR_ALIGN;
  return MMVQ_OK;
}

int mmvq_gemv(int type, const void* W, int64_t rows, int K, const void* xq, int ncols, float* y,
              mmvq_stream_t stream) {
  const int rc = gemv_checks(type, W, rows, K, xq, ncols, y);
  if (rc) return rc;
  return mmvq::launch_dense(type, W, rows, K, xq, ncols, y, nullptr, 0u, (cudaStream_t)stream);
}

int mmvq_gemv_ex(int type, const void* W, int64_t rows, int K, const void* xq, int ncols, float* y,
                 unsigned int flags, mmvq_stream_t stream) {
  const int rc = gemv_checks(type, W, rows, K, xq, ncols, y);
  if (rc) return rc;
  if (flags & ~(unsigned int)(MMVQ_FLAG_XQ_STABLE | MMVQ_FLAG_TENSOR_CORE)) return MMVQ_ERR_SHAPE;
  return mmvq::launch_dense(type, W, rows, K, xq, ncols, y, nullptr, flags, (cudaStream_t)stream);
}

static bool planar_type(int type) {
  return type == MMVQ_Q4_K_PLANAR || type == MMVQ_Q5_K_PLANAR || type == MMVQ_Q6_K_PLANAR;
}

int mmvq_gemv_f32(int type, const void* W, int64_t rows, int K, const float* x, int64_t ldx,
                  int ncols, void* xq, float* y, unsigned int flags, mmvq_stream_t stream) {
  if (!planar_type(type)) return MMVQ_ERR_TYPE;
  if (!W || !x || !xq || !y) return MMVQ_ERR_NULL;
  const int rc = check_weights_shape(rows, K);
  if (rc) return rc;
  if (ncols < 1 || ncols > mmvq::kMaxCols) return MMVQ_ERR_NCOLS;
  if (ldx < K) return MMVQ_ERR_SHAPE;
  if (flags & ~(unsigned int)(MMVQ_FLAG_XQ_STABLE | MMVQ_FLAG_TENSOR_CORE)) return MMVQ_ERR_SHAPE;
  if (!aligned(W, 16) || !aligned(xq, 16) || !aligned(x, 4) || !aligned(y, 4)) return MMVQ_ERR_ALIGN;
  return mmvq::launch_gemv_f32(type, W, rows, K, x, ldx, ncols, xq, y, flags, (cudaStream_t)stream);
}

int mmvq_gemv_f32_fused(int type, int64_t rows, int K, int ncols, int32_t* fused) {
  if (!planar_type(type)) return MMVQ_ERR_TYPE;
  if (!fused) return MMVQ_ERR_NULL;
  const int rc = check_weights_shape(rows, K);
  if (rc) return rc;
  if (ncols < 1 || ncols > mmvq::kMaxCols) return MMVQ_ERR_NCOLS;
  int f = 0;
  const int r2 = mmvq::gemv_f32_fused(type, rows, K, ncols, &f);
  if (r2) return r2;
  *fused = f;
  return MMVQ_OK;
}

int mmvq_debug_block_sums(int type, const void* W, int64_t rows, int K, const void* xq, int ncols,
                          int32_t* sumi, float* y, mmvq_stream_t stream) {
  return mmvq_debug_block_sums_ex(type, W, rows, K, xq, ncols, sumi, y, 0u, stream);
}

int mmvq_debug_block_sums_ex(int type, const void* W, int64_t rows, int K, const void* xq,
                             int ncols, int32_t* sumi, float* y, unsigned int flags,
                             mmvq_stream_t stream) {
  const int rc = gemv_checks(type, W, rows, K, xq, ncols, sumi);
  if (rc) return rc;
  if (!y) return MMVQ_ERR_NULL;
  if (!aligned(y, 4)) return MMVQ_ERR_ALIGN;
  if (flags & ~(unsigned int)(MMVQ_FLAG_XQ_STABLE | MMVQ_FLAG_TENSOR_CORE)) return MMVQ_ERR_SHAPE;
  return mmvq::launch_dense(type, W, rows, K, xq, ncols, y, sumi, flags, (cudaStream_t)stream);
}

int mmvq_grouped(int type, const void* W_experts, int n_experts, int64_t rows, int K,
                 const int32_t* expert_ids, const int32_t* token_offsets, int n_groups,
                 const int32_t* act_index, const void* xq, int n_xq_cols, float* y,
                 int32_t* status, mmvq_stream_t stream) {
  if (!grouped_type(type)) return MMVQ_ERR_TYPE;
  if (!W_experts || !expert_ids || !token_offsets || !xq || !y) return MMVQ_ERR_NULL;
  int rc = check_weights_shape(rows, K);
  if (rc) return rc;
  if ((type == MMVQ_Q4_K_PLANAR || type == MMVQ_Q6_K_PLANAR) && rows % mmvq::kTileRows != 0)
    return MMVQ_ERR_SHAPE;
  if (n_experts < 1 || n_xq_cols < 1) return MMVQ_ERR_SHAPE;
  if (n_groups < 1 || n_groups > 4096) return MMVQ_ERR_ROUTING;
  if (!aligned(W_experts, 16) || !aligned(xq, 16) || !aligned(y, 4) || !aligned(expert_ids, 4) ||
      !aligned(token_offsets, 4) || (act_index && !aligned(act_index, 4)) ||
      (status && !aligned(status, 4)))
    return MMVQ_ERR_ALIGN;
  return mmvq::launch_grouped(type, W_experts, n_experts, rows, K, expert_ids, token_offsets,
                              n_groups, act_index, xq, n_xq_cols, y, status, (cudaStream_t)stream);
}

static int check_expert_ffn(int type, const void* W_gate_up, const void* W_down, int n_experts,
                            int H, int F, const float* x, int64_t ldx, int T, const int32_t* topk,
                            int k) {
  if (type != MMVQ_Q4_K_PLANAR && type != MMVQ_Q6_K_PLANAR) return MMVQ_ERR_TYPE;
  if (!W_gate_up || !W_down || !x || !topk) return MMVQ_ERR_NULL;
  if (H < mmvq::kQK || H > mmvq::kMaxK || H % mmvq::kQK != 0 || F < mmvq::kQK ||
      F > mmvq::kMaxK || F % mmvq::kQK != 0 || ldx < H)
    return MMVQ_ERR_SHAPE;
  if (T < 1 || T > mmvq::kMaxCols) return MMVQ_ERR_NCOLS;
  if (k < 1 || k > 256 || T * k > 256) return MMVQ_ERR_SHAPE;
  if (n_experts < 1 || n_experts > 1024) return MMVQ_ERR_ROUTING;
  return MMVQ_OK;
}

int mmvq_expert_ffn(int type, const void* W_gate_up, const void* W_down, int n_experts, int H,
                    int F, const float* x, int64_t ldx, int T, const int32_t* topk, int k,
                    float* gu, void* hq, float* y, int32_t* expert_ids, int32_t* token_offsets,
                    int32_t* act_index, int32_t* slot_of, void* xq, int32_t* status,
                    uint32_t* sync, mmvq_stream_t stream) {
  int rc = check_expert_ffn(type, W_gate_up, W_down, n_experts, H, F, x, ldx, T, topk, k);
  if (rc) return rc;
  if (!gu || !hq || !y || !xq || !sync) return MMVQ_ERR_NULL;
  if (!aligned(W_gate_up, 16) || !aligned(W_down, 16) || !aligned(hq, 16) || !aligned(xq, 16) || !aligned(x, 4) || !aligned(topk, 4) || !aligned(gu, 4) ||
      !aligned(y, 4) || !aligned(sync, 4) || (expert_ids && !aligned(expert_ids, 4)) ||
      (token_offsets && !aligned(token_offsets, 4)) || (act_index && !aligned(act_index, 4)) ||
      (slot_of && !aligned(slot_of, 4)) || (status && !aligned(status, 4)))
    return MMVQ_ERR_ALIGN;
  mmvq::FfnArgs a = {};
  a.w_gu = static_cast<const uint8_t*>(W_gate_up);
  a.w_dn = static_cast<const uint8_t*>(W_down);
  a.n_experts = n_experts;
  a.H = H;
  a.F = F;
  a.x = x;
  a.ldx = ldx;
  a.T = T;
  a.topk = topk;
  a.k = k;
  a.gu = gu;
  a.hq = static_cast<uint8_t*>(hq);
  a.y = y;
  a.expert_ids = expert_ids;
  a.offsets = token_offsets;
  a.act_index = act_index;
  a.slot_of = slot_of;
  a.xq = static_cast<uint8_t*>(xq);
  a.status = status;
  a.sync = sync;
  return mmvq::launch_expert_ffn(type, a, (cudaStream_t)stream, nullptr);
}

int mmvq_expert_ffn_noalloc(int type, const void* W_gate_up, const void* W_down, int n_experts,
                            int H, int F, const float* x, int64_t ldx, int T,
                            const int32_t* topk, int k, float* y, int32_t* expert_ids,
                            int32_t* token_offsets, int32_t* act_index, int32_t* slot_of,
                            int32_t* status, mmvq_stream_t stream) {
  int rc = check_expert_ffn(type, W_gate_up, W_down, n_experts, H, F, x, ldx, T, topk, k);
  if (rc) return rc;
  if (!y) return MMVQ_ERR_NULL;
  if (!aligned(W_gate_up, 16) || !aligned(W_down, 16) || !aligned(x, 4) || !aligned(topk, 4) ||
      !aligned(y, 4) || (expert_ids && !aligned(expert_ids, 4)) ||
      (token_offsets && !aligned(token_offsets, 4)) || (act_index && !aligned(act_index, 4)) ||
      (slot_of && !aligned(slot_of, 4)) || (status && !aligned(status, 4)))
    return MMVQ_ERR_ALIGN;
  static_assert(mmvq::kFfnScratchBytes == MMVQ_NOALLOC_SCRATCH_BYTES, "scratch size");
  if (mmvq::ffn_scratch_layout(H, F, T, k).end > mmvq::kFfnScratchBytes) return MMVQ_ERR_SCRATCH;
  mmvq::FfnArgs a = {};
  a.w_gu = static_cast<const uint8_t*>(W_gate_up);
  a.w_dn = static_cast<const uint8_t*>(W_down);
  a.n_experts = n_experts;
  a.H = H;
  a.F = F;
  a.x = x;
  a.ldx = ldx;
  a.T = T;
  a.topk = topk;
  a.k = k;
  a.y = y;
  a.expert_ids = expert_ids;
  a.offsets = token_offsets;
  a.act_index = act_index;
  a.slot_of = slot_of;
  a.status = status;
  return mmvq::launch_expert_ffn_noalloc(type, a, (cudaStream_t)stream);
}

int mmvq_expert_ffn_shape(int type, int n_experts, int H, int F, int T, int k, int32_t* info) {
  // any non-null, aligned pointers: only the shape rules are checked here
  static const uint64_t dummy[2] = {0, 0};
  int rc = check_expert_ffn(type, dummy, dummy, n_experts, H, F,
                            reinterpret_cast<const float*>(dummy), H, T,
                            reinterpret_cast<const int32_t*>(dummy), k);
  if (rc) return rc;
  if (!info) return MMVQ_ERR_NULL;
  mmvq::FfnArgs a = {};
  a.n_experts = n_experts;
  a.H = H;
  a.F = F;
  a.T = T;
  a.k = k;
  return mmvq::launch_expert_ffn(type, a, nullptr, info);
}

int mmvq_route_groups(const int32_t* topk, int T, int k, int n_experts, int32_t* expert_ids,
                      int32_t* token_offsets, int32_t* act_index, int32_t* slot_of,
                      int32_t* status, mmvq_stream_t stream) {
  if (!expert_ids || !token_offsets || !act_index || !slot_of) return MMVQ_ERR_NULL;
  if (T > 0 && !topk) return MMVQ_ERR_NULL;
  if (n_experts < 1 || n_experts > 4096 || T < 0 || k < 1 || (int64_t)T * k > 65536)
    return MMVQ_ERR_SHAPE;
  if ((topk && !aligned(topk, 4)) || !aligned(expert_ids, 4) || !aligned(token_offsets, 4) ||
      !aligned(act_index, 4) || !aligned(slot_of, 4) || (status && !aligned(status, 4)))
    return MMVQ_ERR_ALIGN;
  return mmvq::launch_route_groups(topk, T, k, n_experts, expert_ids, token_offsets, act_index,
                                   slot_of, status, (cudaStream_t)stream);
}

int mmvq_silu_mul_quantize_q8_1(const float* gu, int F, int n, void* xq, float* h_out,
                                mmvq_stream_t stream) {
  if (!gu || !xq) return MMVQ_ERR_NULL;
  if (F <= 0 || F % mmvq::kQK8 != 0 || n < 1) return MMVQ_ERR_SHAPE;
  if (!aligned(gu, 4) || !aligned(xq, 16) || (h_out && !aligned(h_out, 4))) return MMVQ_ERR_ALIGN;
  return mmvq::launch_silu_mul_quantize(gu, F, n, xq, h_out, (cudaStream_t)stream);
}

int64_t mmvq_planar_bytes(int type, int64_t rows, int K) {
  if (!repack_source_type(type)) return -1;
  if (check_weights_shape(rows, K) != MMVQ_OK) return -1;
  const int64_t groups = (rows + mmvq::kTileRows - 1) / mmvq::kTileRows;
  return groups * (K / mmvq::kQK) * tile_bytes_of_source(type);
}

int mmvq_repack_planar(int type, const void* W_gguf, int64_t rows, int K, void* W_planar,
                       mmvq_stream_t stream) {
  if (!repack_source_type(type)) return MMVQ_ERR_TYPE;
  if (!W_gguf || !W_planar) return MMVQ_ERR_NULL;
  const int rc = check_weights_shape(rows, K);
  if (rc) return rc;
  if (!aligned(W_gguf, type == MMVQ_Q6_K ? 2 : 16) || !aligned(W_planar, 16)) return MMVQ_ERR_ALIGN;
  return mmvq::launch_repack_planar(type, W_gguf, rows, K, W_planar, (cudaStream_t)stream);
}

int mmvq_gather_planar_rows(const void* W_planar, int64_t rows, int K, const int32_t* row_ids,
                            int n, void* out, int32_t* status, mmvq_stream_t stream) {
  if (!W_planar || !row_ids || !out) return MMVQ_ERR_NULL;
  int rc = check_weights_shape(rows, K);
  if (rc) return rc;
  if (n < 1) return MMVQ_ERR_SHAPE;
  if (!aligned(W_planar, 16) || !aligned(out, 16) || !aligned(row_ids, 4) ||
      (status && !aligned(status, 4)))
    return MMVQ_ERR_ALIGN;
  return mmvq::launch_gather_planar(W_planar, rows, K, row_ids, n, out, status,
                                    (cudaStream_t)stream);
}

int mmvq_launch_shape_ex(int type, int64_t rows, int K, int ncols, int32_t* info, int n_info) {
  if (!dense_type(type)) return MMVQ_ERR_TYPE;
  if (!info) return MMVQ_ERR_NULL;
  if (n_info < 1) return MMVQ_ERR_SHAPE;
  const int rc = check_weights_shape(rows, K);
  if (rc) return rc;
  if (ncols < 1 || ncols > mmvq::kMaxCols) return MMVQ_ERR_NCOLS;
  int32_t all[7];
  const int r2 = mmvq::dense_shape(type, rows, K, ncols, all);
  if (r2) return r2;
  for (int i = 0; i < n_info && i < 7; ++i) info[i] = all[i];
  return MMVQ_OK;
}

int mmvq_launch_shape(int type, int64_t rows, int K, int ncols, int32_t* info) {
  return mmvq_launch_shape_ex(type, rows, K, ncols, info, 6);
}

int mmvq_selftest_wait_timeout(unsigned int limit_us, mmvq_stream_t stream) {
  if (limit_us < 1 || limit_us > 100000) return MMVQ_ERR_SHAPE;
  return mmvq::launch_wait_timeout_selftest(limit_us, (cudaStream_t)stream);
}

int mmvq_selftest_grid_barrier_timeout(uint32_t* sync, unsigned int limit_us,
                                       mmvq_stream_t stream) {
  if (!sync) return MMVQ_ERR_NULL;
  if (!aligned(sync, 4)) return MMVQ_ERR_ALIGN;
  if (limit_us < 1 || limit_us > 100000) return MMVQ_ERR_SHAPE;
  return mmvq::launch_grid_barrier_selftest(sync, limit_us, (cudaStream_t)stream);
}

int mmvq_rmsnorm_quantize_q8_1(const float* x, const float* w, float eps, int K, int ncols,
                               int64_t ldx, void* xq, float* y_out, mmvq_stream_t stream) {
  if (!x || !w || !xq) return MMVQ_ERR_NULL;
  if (K <= 0 || K % mmvq::kQK8 != 0 || K > (1 << 24) || ncols < 1 || ncols > 65535 || ldx < K)
    return MMVQ_ERR_SHAPE;
  if (!(eps >= 0.0f) || !(eps < INFINITY)) return MMVQ_ERR_SHAPE;
  if (!aligned(x, 4) || !aligned(w, 4) || !aligned(xq, 16) || (y_out && !aligned(y_out, 4)))
    return MMVQ_ERR_ALIGN;
  return mmvq::launch_rmsnorm_quantize(x, w, eps, K, ncols, ldx, xq, y_out, (cudaStream_t)stream);
}

int mmvq_read_device_fault(int* fault, mmvq_stream_t stream) {
  if (!fault) return MMVQ_ERR_NULL;
  return mmvq::read_device_fault(fault, (cudaStream_t)stream);
}

}  // extern "C"
