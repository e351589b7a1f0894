/*
 * mmvq.h: C ABI of libmmvq.so, block-quantized weight x Q8_1 activation
 * matrix-vector products (MMVQ) at 1-8 columns, for NVIDIA GB300 (sm_103a).
 *
 * Conventions for every entry point:
 *  - Pointers named W (W_*), xq, hq, x, y, gu, sumi, row_ids, topk,
 *    expert_ids, token_offsets, act_index, slot_of, status, sync and out are
 *    DEVICE pointers, owned by the caller, who allocates and frees them.  The library allocates no
 *    device or host memory and never synchronises the stream (its one
 *    device buffer is the fixed array of mmvq_expert_ffn_noalloc).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  Launch failures are reported by the return
 *    value; faults inside a kernel surface at the caller's next sync.
 *  - Return value: MMVQ_OK (0) or a negative mmvq_status.  Arguments are
 *    checked on the host before any CUDA call, so a rejected call launches
 *    nothing and leaves every buffer untouched.
 *  - Alignment: W, xq and out must be 16-byte aligned; x, y, gu and the
 *    int32 arrays 4-byte aligned.
 *  - There is no CPU fallback: without a usable sm_103a device a launch
 *    fails with MMVQ_ERR_CUDA.
 *  - Launch shapes are chosen on the first call for a shape and cached; the
 *    caches are guarded, so calls may come from several host threads.  A
 *    process may drive several GPUs of the same model (the cached shapes
 *    assume one SM count); kernel attributes are set per device.
 *
 * Formats (the pages are the Strata engine's SYCL port: PRs #2746, #2340,
 * #2207, #1774 and issue #2801; the byte arrangement inside each block is
 * the GGUF one):
 *  - Q8_1 block, 36 bytes per 32 activations: fp16 d, fp16 s, int8 q[32];
 *    d = amax/127, q = round-half-away(x/d), s = d * sum(q) (PR #2340,
 *    "int4 activation loads": quants 4-byte aligned behind the header).
 *  - Q6_K block, 210 bytes per 256 weights: ql[128] low nibbles, qh[64]
 *    2-bit high fields, int8 scales[16] (one per 16 weights), fp16 d.
 *    Weight = d * scale * (q - 32), q in 0..63 (PR #2340, "Q6_K six-bit
 *    offset as SWAR").
 *  - Q4_K block, 144 bytes per 256 weights: fp16 d, fp16 dmin, 12 bytes of
 *    packed 6-bit scales and mins for 8 sub-blocks of 32, qs[128] nibbles.
 *    Weight = d * sc * q - dmin * m.
 *  - Dense matrices are row-major: row r holds K/256 consecutive blocks.
 *  - Planar Q6_K (MMVQ_Q6_K_PLANAR), this library's load-time layout after
 *    PR #2340 "STRATA_Q6_PLANAR" (the same bytes, as ql/qh/scales/d planes,
 *    so every load is an aligned 16-byte load).  Rows are taken in groups
 *    of 16 (the last group padded with zero rows).  The matrix is a
 *    sequence of 3360-byte tiles T(g, b), g = row group (major), b = 256-block
 *    (minor).  Inside a tile, lane L = 16*h + i, where i = row in the group
 *    and h = half of the block:
 *      bytes [512*j + 16*L, +16)         j = 0..3 : ql[64*h + 16*j .. +15]
 *      bytes [2048 + 512*j + 16*L, +16)  j = 0..1 : qh[32*h + 16*j .. +15]
 *      bytes [3072 + 8*L, +8)                     : scales[8*h .. 8*h+7]
 *      bytes [3328 + 2*i, +2)                     : d
 *    so each warp-wide 16-byte load reads one contiguous 512-byte segment.
 *    Size: mmvq_planar_bytes(MMVQ_Q6_K, rows, K).
 *  - Planar Q4_K (MMVQ_Q4_K_PLANAR), the same idea for Q4_K: 2304-byte
 *    tiles T(g, b) in the same order; lane L = 16*u + i (u = half of the
 *    block, i.e. sub-blocks 4u..4u+3):
 *      bytes [512*j + 16*L, +16)  j = 0..3 : qs[64*u + 16*j .. +15]
 *      bytes [2048 + 16*i, +16)            : d, dmin, scales[12] of row i
 *    Size: mmvq_planar_bytes(MMVQ_Q4_K, rows, K).
 *  - Q5_K block, 176 bytes per 256 weights (the pages run Q5_K matrices in
 *    the same wide kernels, PR #2340 "ld_i4_a4", without giving the block;
 *    this is the GGUF Q5_K arrangement): fp16 d, fp16 dmin, the Q4_K scale
 *    and min bytes, qh[32], qs[128] as in Q4_K; weight l of sub-block j
 *    takes its fifth bit from bit j of qh[l]; code q in 0..31,
 *    weight = d * sc * q - dmin * m.  Products run from planar tiles only.
 *  - Planar Q5_K (MMVQ_Q5_K_PLANAR): 2816-byte tiles, the Q4_K tile plus
 *      bytes [2304 + 32*i, +32)            : qh[0..31] of row i
 *    Size: mmvq_planar_bytes(MMVQ_Q5_K, rows, K).
 *
 * Results: y is fp32, [ncols][rows] (column-major over the activation
 * columns).  Block sums are exact integers; the FP32 output of a row is
 * sum over 32-blocks of d_w*d_a*sumi (Q4_K: minus dmin*m*s_a), summed in an
 * order that differs from plain index order only in rounding (PR #1774,
 * "What changed": only the sub-block summation order differs, so the last
 * bits can differ).
 */
#ifndef MMVQ_H_
#define MMVQ_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mmvq_stream_t; /* == cudaStream_t */

/* Symbols of this ABI are the only ones the library exports. */
#if defined(__GNUC__)
#define MMVQ_API __attribute__((visibility("default")))
#else
#define MMVQ_API
#endif

enum mmvq_type {
  MMVQ_Q4_K = 12,          /* GGUF Q4_K blocks, 144 B / 256 weights */
  MMVQ_Q5_K = 13,          /* GGUF Q5_K blocks, 176 B / 256 weights (repack source) */
  MMVQ_Q6_K = 14,          /* GGUF Q6_K blocks, 210 B / 256 weights */
  MMVQ_Q4_K_PLANAR = 1012, /* Q4_K in 16-row planar tiles (see above) */
  MMVQ_Q5_K_PLANAR = 1013, /* Q5_K in 16-row planar tiles (see above) */
  MMVQ_Q6_K_PLANAR = 1014  /* Q6_K in 16-row planar tiles (see above) */
};

/* Flags of mmvq_gemv_ex. */
enum mmvq_flags {
  /* xq is stable: no kernel that may still be running when this call starts
   * writes it (true when xq came from mmvq_quantize_q8_1 or
   * mmvq_silu_mul_quantize_q8_1, or earlier work, and nothing launched
   * since writes it; those quantisers never let their successor start
   * early).  The product then runs before waiting for the preceding kernel,
   * and only the stores of y wait for it. */
  MMVQ_FLAG_XQ_STABLE = 1,
  /* Planar types, 4-8 columns: form the integer sums with warp-level f16
   * tensor-core MMAs (one per 16-weight sub-block, exact) instead of dp4a,
   * in the same launch shape; the per-block sums and y are the same, bit
   * for bit.  Measured on GB300 it is no faster than dp4a at 8 columns and
   * slower below, so the default stays dp4a (the calls are latency-bound,
   * not bound by the dp4a issue rate).  Ignored where the extra 4 bytes of
   * shared memory per value of K do not fit, and by the GGUF types. */
  MMVQ_FLAG_TENSOR_CORE = 2
};

enum mmvq_status {
  MMVQ_OK = 0,
  MMVQ_ERR_TYPE = -1,    /* type not supported by this entry point */
  MMVQ_ERR_SHAPE = -2,   /* K % 256 (K % 32 for Q8_1), rows/n <= 0, sizes too large */
  MMVQ_ERR_NCOLS = -3,   /* ncols outside 1..8 */
  MMVQ_ERR_NULL = -4,    /* a required pointer is NULL */
  MMVQ_ERR_ALIGN = -5,   /* a pointer breaks its alignment rule */
  MMVQ_ERR_ROUTING = -6, /* routing lists rejected (host-side limits) */
  MMVQ_ERR_CUDA = -7,    /* a CUDA launch or attribute call failed */
  MMVQ_ERR_SCRATCH = -8  /* mmvq_expert_ffn_noalloc: intermediates exceed its fixed scratch */
};

/* Version of this ABI (major*10000 + minor*100 + patch). */
MMVQ_API int mmvq_version(void);

/* Human-readable text for a status code (static storage). */
MMVQ_API const char* mmvq_strerror(int code);

/*
 * Q8_1 activation quantisation (PR #2340 "int4 activation loads"; PR #1774
 * "d * ds * sumi").  x: fp32 [ncols][ldx]; the first K values of each column
 * are quantised in blocks of 32 into xq: [ncols][K/32] Q8_1 blocks (36 B).
 * Bit-exact: d = fp16(amax/127), q = roundf(x/d) (0 when amax = 0),
 * s = fp16(d*sum q) with d unrounded; fp16 conversions round to nearest even.
 * Requires K % 32 == 0, K > 0, ldx >= K, 1 <= ncols <= 65535.
 */
MMVQ_API int mmvq_quantize_q8_1(const float* x, int K, int ncols, int64_t ldx, void* xq,
                       mmvq_stream_t stream);

/*
 * Dense MMVQ (PR #2207 wide kernels, PR #1774 iq3s_wide_kernel: weights read
 * once for all 1-8 columns).  W: rows x K/256 blocks of `type` (MMVQ_Q4_K,
 * MMVQ_Q6_K, MMVQ_Q4_K_PLANAR, MMVQ_Q5_K_PLANAR or MMVQ_Q6_K_PLANAR); xq:
 * [ncols][K/32] Q8_1 blocks;
 * y: fp32 [ncols][rows].  Requires K % 256 == 0 (PR #1774: the row length a
 * multiple of 256), 1 <= ncols <= 8 (PR #2207: 1 to 8 columns),
 * K <= 16384, 1 <= rows <= 2^31 - 1.
 * Speed: the GGUF types are a compatibility path for matrices used as
 * stored (their 2-byte aligned 210-byte Q6_K blocks and 144-byte Q4_K rows
 * do not stream as whole tiles).  On GB300 they reach about a tenth of HBM
 * bandwidth against 0.4-0.9 for the planar tiles, so a hot-path caller
 * repacks once at load with mmvq_repack_planar and passes the *_PLANAR type
 * (PR #2340 "STRATA_Q6_PLANAR": the head is repacked at load for the same
 * reason).
 */
MMVQ_API int mmvq_gemv(int type, const void* W, int64_t rows, int K, const void* xq, int ncols, float* y,
              mmvq_stream_t stream);

/*
 * mmvq_gemv with launch flags (mmvq_flags; 0 gives mmvq_gemv).  With
 * MMVQ_FLAG_XQ_STABLE, consecutive calls that share one quantised
 * activation (several matrices reading one input, like q/k/v or gate/up)
 * overlap on the GPU: each call streams its weights and computes while the
 * previous call is still finishing.  Weights are always streamed before the
 * wait; no kernel of this library that writes weights (repack, gather)
 * lets its successor start early.  Unknown flag bits: MMVQ_ERR_SHAPE.  The
 * flag changes the schedule of the three planar types (MMVQ_Q4_K_PLANAR,
 * MMVQ_Q5_K_PLANAR, MMVQ_Q6_K_PLANAR): their activations are staged before
 * the wait, so the hazard it waives applies to all three.  The GGUF types
 * (MMVQ_Q4_K, MMVQ_Q6_K) ignore it.
 */
MMVQ_API int mmvq_gemv_ex(int type, const void* W, int64_t rows, int K, const void* xq, int ncols,
                          float* y, unsigned int flags, mmvq_stream_t stream);

/*
 * Dense MMVQ from fp32 activation columns: Q8_1 of x, then the product, as
 * mmvq_quantize_q8_1 followed by mmvq_gemv_ex, with the same results (xq
 * gets the same bytes, y the same bits).  Where the columns are small
 * enough (a round or two of 32-blocks for the CTA's warps: one column of K
 * up to about 5120 on the common launch shapes), it is one launch whose CTAs
 * each quantise the columns into their own staging while their first weight
 * stages stream in, so a decode step needs no separate quantisation launch;
 * otherwise it issues the two launches.  x: fp32 [ncols][ldx], ldx >= K;
 * xq: Q8_1 [ncols][K/32], written (the quantised columns); y: fp32
 * [ncols][rows].  type: a planar type.  flags as mmvq_gemv_ex, where
 * MMVQ_FLAG_XQ_STABLE promises that x is stable.  Other rules as mmvq_gemv.
 * No counterpart on the pages (their engine quantises in its own launch).
 */
MMVQ_API int mmvq_gemv_f32(int type, const void* W, int64_t rows, int K, const float* x,
                           int64_t ldx, int ncols, void* xq, float* y, unsigned int flags,
                           mmvq_stream_t stream);

/* Whether mmvq_gemv_f32 runs this call as one launch (*fused = 1) or as the
 * quantiser and the product (0).  Host-only. */
MMVQ_API int mmvq_gemv_f32_fused(int type, int64_t rows, int K, int ncols, int32_t* fused);

/*
 * The per-32-block integer sums the dense product forms, for parity checks:
 * sumi: int32 [ncols][rows][K/32], sumi = sc0*sum16 + sc1*sum16 (Q6_K) or
 * sc*sum32 (Q4_K).  Runs mmvq_gemv's kernel code in the same launch shape,
 * in an instance that also stores the sums (the product instance carries no
 * such store); y, when y != NULL, gets the same bits as mmvq_gemv gives.
 * Same argument rules as mmvq_gemv.
 */
MMVQ_API int mmvq_debug_block_sums(int type, const void* W, int64_t rows, int K, const void* xq, int ncols,
                          int32_t* sumi, float* y, mmvq_stream_t stream);

/* mmvq_debug_block_sums with the flags of mmvq_gemv_ex (MMVQ_FLAG_TENSOR_CORE:
 * the sums as the tensor-core consumer forms them). */
MMVQ_API int mmvq_debug_block_sums_ex(int type, const void* W, int64_t rows, int K,
                                      const void* xq, int ncols, int32_t* sumi, float* y,
                                      unsigned int flags, mmvq_stream_t stream);

/*
 * Grouped expert MMVQ over per-expert token lists (PR #2746 "B70
 * validation": grouped calls with empty groups; issue #2801: the grouped
 * gate/up and down kernels).  W_experts: n_experts matrices of rows x K,
 * one after another, of `type` (MMVQ_Q4_K, MMVQ_Q6_K, or a planar type
 * with each expert repacked on its own and rows a multiple of 16).  Group g (0 <= g < n_groups) multiplies
 * expert expert_ids[g] with the activation columns of positions
 * p in [token_offsets[g], token_offsets[g+1]); column act_index[p] of xq
 * (column p when act_index == NULL).  Output row p: y[p][0..rows); rows of
 * positions outside every group are not written.
 * xq: [n_xq_cols][K/32] Q8_1 blocks.  Empty groups are legal and cost
 * nothing.  Groups may hold any number of positions (processed 8 at a time).
 * Device-side checks: an expert id outside [0, n_experts), decreasing
 * offsets or an activation index outside [0, n_xq_cols) skip that group or
 * position and set *status to MMVQ_ERR_ROUTING when status != NULL (the
 * caller clears *status beforehand).  Host limits: 1 <= n_groups <= 4096,
 * K % 256 == 0, K <= 16384, rows >= 1, n_experts >= 1.
 */
MMVQ_API int mmvq_grouped(int type, const void* W_experts, int n_experts, int64_t rows, int K,
                 const int32_t* expert_ids, const int32_t* token_offsets, int n_groups,
                 const int32_t* act_index, const void* xq, int n_xq_cols, float* y,
                 int32_t* status, mmvq_stream_t stream);

/*
 * Per-expert token lists from top-k routing: all n_experts groups in id order
 * (expert_ids[e] = e, token_offsets [n_experts+1]), positions inside a group
 * in token order; act_index[p] = token of position p, slot_of[p] = t*k + j
 * for routing entry topk[t][j].  topk: int32 [T][k].  Out-of-range expert ids
 * are dropped and set *status to MMVQ_ERR_ROUTING when status != NULL.
 * Requires 1 <= n_experts <= 4096, T >= 0, 1 <= k, T*k <= 65536.
 */
MMVQ_API int mmvq_route_groups(const int32_t* topk, int T, int k, int n_experts, int32_t* expert_ids,
                      int32_t* token_offsets, int32_t* act_index, int32_t* slot_of,
                      int32_t* status, mmvq_stream_t stream);

/*
 * The first step of an expert layer in one launch: mmvq_quantize_q8_1 of the
 * hidden states x and mmvq_route_groups of topk (the two are independent;
 * every output is the same bits as the two calls give).  Arguments and
 * limits are those of the two calls.  With n_experts > 1024 it issues the two
 * kernels one after the other.  No counterpart on the pages (their engine
 * launches them separately).
 */
MMVQ_API int mmvq_quantize_route_groups(const float* x, int K, int ncols, int64_t ldx, void* xq,
                                        const int32_t* topk, int T, int k, int n_experts,
                                        int32_t* expert_ids, int32_t* token_offsets,
                                        int32_t* act_index, int32_t* slot_of, int32_t* status,
                                        mmvq_stream_t stream);

/*
 * SiLU(gate) * up, requantised to Q8_1 between the grouped gate/up and down
 * calls.  gu: fp32 [n][2F] rows laid out [gate F | up F] (the grouped
 * gate/up output when the expert's first F rows are gate and the next F
 * rows up).  h = gate/(1+exp(-gate)) * up in fp32, then Q8_1 as
 * mmvq_quantize_q8_1 into xq: [n][F/32].  h_out (may be NULL): fp32 [n][F].
 * Requires F % 32 == 0, F > 0, n >= 1.
 */
MMVQ_API int mmvq_silu_mul_quantize_q8_1(const float* gu, int F, int n, void* xq, float* h_out,
                                mmvq_stream_t stream);

/*
 * The routed-expert FFN of one MoE layer in one launch (issue #2801: the
 * grouped gate/up and down kernels with the activation between them; PR
 * #2746: grouped calls over per-expert token groups).  For T tokens (1..8)
 * routed to k experts each by topk (int32 [T][k]) it computes:
 *  - the token lists of mmvq_route_groups (position p runs over the valid
 *    routing entries in expert order, tokens in order inside an expert);
 *  - gu[p][0..2F) = the gate|up matrix of expert e(p) (W_gate_up: n_experts
 *    planar matrices of 2F x H, one after another, gate rows first) times
 *    Q8_1(x[token(p)]), as mmvq_grouped;
 *  - hq[p] = Q8_1(SiLU(gate) * up) as mmvq_silu_mul_quantize_q8_1;
 *  - y[p][0..H) = the down matrix of expert e(p) (W_down: n_experts planar
 *    matrices of H x F) times hq[p], as mmvq_grouped.
 * Each step uses the arithmetic of its separate entry point: Q8_1 bytes and
 * per-32-block integer sums are the same, fp32 sums may be added in another
 * order.
 *   type: MMVQ_Q4_K_PLANAR or MMVQ_Q6_K_PLANAR (both matrices).
 *   x: fp32 [T][ldx], ldx >= H.  xq: Q8_1 [T][H/32], the quantised hidden
 *   states (written, then read by the gate|up step).  gu: fp32 [T*k][2F];
 *   hq: Q8_1 [T*k][F/32]; y: fp32 [T*k][H]; rows p >= the number of valid
 *   entries are not written.  expert_ids [n_experts], token_offsets
 *   [n_experts+1], act_index [T*k] and slot_of [T*k] are optional outputs
 *   (NULL: not written) holding what mmvq_quantize_route_groups gives.
 *   status (optional): set to MMVQ_ERR_ROUTING when an expert id lies
 *   outside [0, n_experts) (that entry is dropped).
 *   sync: one uint32 word, zero before the first call.  The launch uses it
 *   as its grid-barrier counter and leaves its low 31 bits zero (the top bit
 *   alternates); launches that may run at the same time need separate
 *   words.  A grid barrier that does not open within about a second sets
 *   bit 2 of the device fault word (outputs then undefined); zero the word
 *   again before the next launch.
 * One cooperative launch (one CTA per SM for T <= 2, three from T = 3 on);
 * every wait in it is bounded.
 * Requires 1 <= T <= 8 (else MMVQ_ERR_NCOLS), 1 <= k, T*k <= 256,
 * 1 <= n_experts <= 1024 (else MMVQ_ERR_ROUTING), H and F multiples of 256
 * in [256, 16384], and a CTA's ring of at least two stages plus the staged
 * columns of one group (up to 8 x max(H, F) quants) within shared memory,
 * else MMVQ_ERR_SHAPE (mmvq_expert_ffn_shape tells).  No counterpart on the pages (their engine launches the
 * steps one by one).
 */
MMVQ_API int mmvq_expert_ffn(int type, const void* W_gate_up, const void* W_down, int n_experts,
                             int H, int F, const float* x, int64_t ldx, int T,
                             const int32_t* topk, int k, float* gu, void* hq, float* y,
                             int32_t* expert_ids, int32_t* token_offsets, int32_t* act_index,
                             int32_t* slot_of, void* xq, int32_t* status, uint32_t* sync,
                             mmvq_stream_t stream);

/*
 * mmvq_expert_ffn for callers that cannot allocate device memory.  Some
 * callers only ever hold the buffers of their own tensors: a plugin inside
 * an inference engine whose memory pool owns the whole device, or a C
 * caller that was handed device pointers and has no allocator of its own.
 * Others must keep cudaMalloc, which can synchronise the device, out of a
 * decode step.  For them the layer's intermediates (the grid-barrier word,
 * the Q8_1 hidden states xq, the gate|up rows gu and the requantised hq)
 * live in one fixed device array of MMVQ_NOALLOC_SCRATCH_BYTES inside the
 * library; the caller passes only inputs and outputs.  The pages have no
 * counterpart (their engine allocates its buffers).
 *   Arguments, limits and results are those of mmvq_expert_ffn, without
 *   gu, hq, xq and sync.  y gets the same bits as mmvq_expert_ffn gives for
 *   the same inputs.
 *   Size limit: the parts, each rounded up to 256 bytes, must fit:
 *   256 + T*(H/32)*36 + T*k*(F/32)*36 + T*k*2F*4 <= MMVQ_NOALLOC_SCRATCH_BYTES
 *   (2 MiB; the pages' layer, H = 2560, F = 768, T = 8, k = 8, takes
 *   about 0.5 MiB), else MMVQ_ERR_SCRATCH before any CUDA call.
 *   Memory: every GPU that loads the library holds the array until the
 *   process exits.  The call allocates nothing and frees nothing; it clears
 *   the barrier word with cudaMemsetAsync on `stream` before the launch.
 *   Set-up: the first call on a device, with that device current, looks up
 *   the array's device address (cudaGetSymbolAddress) and caches it; make
 *   that first call before any stream capture.
 *   Sharing: every call on a device uses the same array, which keeps the
 *   last call's intermediates.  Calls that may run at the same time on one
 *   device (other streams, other host threads) race on it and give
 *   undefined results; calls in order on one stream are safe.
 */
MMVQ_API int mmvq_expert_ffn_noalloc(int type, const void* W_gate_up, const void* W_down,
                                     int n_experts, int H, int F, const float* x, int64_t ldx,
                                     int T, const int32_t* topk, int k, float* y,
                                     int32_t* expert_ids, int32_t* token_offsets,
                                     int32_t* act_index, int32_t* slot_of, int32_t* status,
                                     mmvq_stream_t stream);

/* Size of the fixed scratch array of mmvq_expert_ffn_noalloc, per device. */
#define MMVQ_NOALLOC_SCRATCH_BYTES (2u << 20)

/*
 * The launch shape mmvq_expert_ffn picks (host-only; no kernel runs).
 * info[8] (HOST memory): grid, threads per CTA, dynamic shared bytes, ring
 * stages, then G (row groups per item) and P (K-slices) of the gate|up
 * phase and of the down phase.  Same shape rules as mmvq_expert_ffn.
 */
MMVQ_API int mmvq_expert_ffn_shape(int type, int n_experts, int H, int F, int T, int k,
                                   int32_t* info);

/*
 * RMSNorm folded into the Q8_1 quantiser (the opt-in fused norm named in
 * PR #1774 "How it was checked"; the pages give no formula, so the plain RMS
 * norm with a weight vector).  Per column c of x (fp32 [ncols][ldx], ldx >= K):
 * ms = (sum of x_i^2 in fp64) / K, scale = fp32(1 / sqrt(ms + eps)) computed
 * in fp64, y_i = (x_i * scale) * w_i in fp32 (w: fp32 [K]), then Q8_1 of y
 * into xq ([ncols][K/32] blocks) exactly as mmvq_quantize_q8_1.  y_out (may
 * be NULL): fp32 [ncols][K].  Requires K % 32 == 0, 0 < K <= 2^24,
 * 1 <= ncols <= 65535, 0 <= eps < inf; x, w, y_out 4-byte and xq 16-byte
 * aligned.
 */
MMVQ_API int mmvq_rmsnorm_quantize_q8_1(const float* x, const float* w, float eps, int K, int ncols,
                                        int64_t ldx, void* xq, float* y_out,
                                        mmvq_stream_t stream);

/* Bytes of the planar form of a rows x K matrix of `type` (MMVQ_Q6_K,
 * MMVQ_Q5_K or MMVQ_Q4_K); -1 on a bad type or shape. */
MMVQ_API int64_t mmvq_planar_bytes(int type, int64_t rows, int K);

/*
 * Load-time repack of GGUF Q6_K blocks into planar tiles (PR #2340
 * "STRATA_Q6_PLANAR": same bytes, the GGUF copy can then be freed).
 * Out-of-place; W_planar holds mmvq_planar_bytes(type, rows, K) bytes; pad
 * rows are written as zeros.  type: MMVQ_Q6_K (-> MMVQ_Q6_K_PLANAR),
 * MMVQ_Q5_K (-> MMVQ_Q5_K_PLANAR) or MMVQ_Q4_K (-> MMVQ_Q4_K_PLANAR).
 * K % 256 == 0; W_gguf 16-byte aligned (2-byte for Q6_K).
 */
MMVQ_API int mmvq_repack_planar(int type, const void* W_gguf, int64_t rows, int K, void* W_planar,
                       mmvq_stream_t stream);

/*
 * Draft-head gather (PR #2340: "the draft head's subset is gathered from the
 * planar head"): out = planar matrix of n rows whose row k is row
 * row_ids[k] of the planar matrix W_planar (rows x K).  out holds
 * mmvq_planar_bytes(MMVQ_Q6_K, n, K) bytes.  Row ids outside [0, rows) give zero rows
 * and set *status to MMVQ_ERR_ROUTING when status != NULL.
 */
MMVQ_API int mmvq_gather_planar_rows(const void* W_planar, int64_t rows, int K, const int32_t* row_ids,
                            int n, void* out, int32_t* status, mmvq_stream_t stream);

/*
 * The launch shape mmvq_gemv picks for this matrix and column count, on the
 * current device (host-only; no kernel runs).  info[6] (HOST memory):
 * grid, threads per CTA, dynamic shared bytes, then for MMVQ_Q6_K_PLANAR
 * G (row groups per batch), P (warps per row group), ring stages; for the
 * GGUF types WR (row groups per CTA), WK (warps per row group), 0.
 * Same argument rules as mmvq_gemv.  No counterpart on the pages.
 */
MMVQ_API int mmvq_launch_shape(int type, int64_t rows, int K, int ncols, int32_t* info);

/*
 * mmvq_launch_shape writing n_info (1..7) values; the seventh is the
 * number of CTAs per thread-block cluster of the planar kernel (1: no
 * cluster; 2: each row group's K split over a pair of CTAs that add their
 * partial sums through distributed shared memory).  No counterpart on the
 * pages.
 */
MMVQ_API int mmvq_launch_shape_ex(int type, int64_t rows, int K, int ncols, int32_t* info,
                                  int n_info);

/*
 * Device fault word of the bulk-copy kernels.  Every wait of those kernels
 * on a shared-memory barrier, and of mmvq_expert_ffn on its grid barriers,
 * is bounded (about one second); a wait that runs out sets a bit here (1: a
 * shared-memory barrier wait timed out; 2: a grid barrier timed out) instead
 * of hanging, and the kernel returns with its outputs undefined.  In the
 * debug build (libmmvq_checked.so, compiled with MMVQ_CHECKED) bit 4 reports
 * a failed device-side index check (the access was skipped).  Synchronises
 * `stream`, stores the word in *fault and clears it.  This HOST-pointer
 * call blocks; it is not part of the hot path.  No counterpart on the
 * pages (their kernels have no such waits).
 */
MMVQ_API int mmvq_read_device_fault(int* fault, mmvq_stream_t stream);

/*
 * Self-test of the bounded waits above: launches one warp that waits, with
 * the kernels' own wait routine and a limit of limit_us microseconds
 * (1..100000), on a shared-memory barrier that nothing completes.  The wait
 * runs out and sets bit 1 of the device fault word, read afterwards with
 * mmvq_read_device_fault; nothing faults and the context stays usable.  For
 * checking the failure path on a live GPU; no counterpart on the pages.
 */
MMVQ_API int mmvq_selftest_wait_timeout(unsigned int limit_us, mmvq_stream_t stream);

/*
 * Self-test of the grid barrier's bound in mmvq_expert_ffn: one CTA enters
 * that barrier, on the counter word *sync, as the first of two blocks whose
 * second is never launched, with a limit of limit_us microseconds
 * (1..100000).  The wait runs out and sets bit 2 of the device fault word;
 * nothing faults.  *sync is left changed (use a word of its own).  No
 * counterpart on the pages.
 */
MMVQ_API int mmvq_selftest_grid_barrier_timeout(uint32_t* sync, unsigned int limit_us,
                                                mmvq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MMVQ_H_ */
