/*
 * moe_nvfp4.h - C ABI of the GB300 (sm_103a) routed-MoE forward with online
 * per-token NVFP4 activation quantization.
 *
 * One call of moe_forward runs, on one CUDA stream, with no host
 * synchronisation and no allocation:
 *   router logits -> top-k -> expert permutation (expand) -> per-token NVFP4
 *   quantization -> block-scaled FP4 grouped GEMM on w13 with SwiGLU and
 *   per-row requantization in its epilogue -> block-scaled FP4 grouped GEMM on
 *   w2 -> top-k weighted finalize -> bf16 output.  Up to 64 tokens the w2
 *   epilogue adds the weighted rows into an FP32 accumulator; in
 *   deterministic mode and above 64 tokens it stores one bf16 row per
 *   (token, slot), summed in slot order by the finalize.  An optional shared
 *   expert runs on a second stream forked from and joined back into the
 *   caller's.
 *
 * Where each operation is defined (the pages' titles and sections):
 *   - "CuTe DSL backend gets per-token NVFP4 online quantization and reload",
 *     Implementation items 1-3 and the code snippets: per-token FP32 global
 *     scale, E4M3 block scales over 16-element blocks, E2M1 codes; online
 *     NVFP4 weight conversion; in-place scale refresh after a weight reload
 *     that keeps every captured address valid and fails loudly when scale
 *     metadata changed; deterministic inference forces the non-fused
 *     (fixed-order) finalize.
 *   - "size CuteDSL MoE allgather buffers for the worst-case forward",
 *     Motivation and Implementation: buffers are sized once from the
 *     worst-case token count of one forward; a larger forward is an error.
 *   - "SM10X Command-A-Plus decode 2.3x faster, BCG capture memory -78%",
 *     Motivation and Implementation item 2: routing, expandInputRows,
 *     activation and finalize fused around the expert GEMMs; the routed
 *     output must not alias its input.  Its code snippets (the Cohere2MoE
 *     sparse block): shared experts on an alternate stream next to the
 *     routed experts, outputs added, halved under the 'average' strategy.
 *
 * Numeric rules (the pages print no formula; these are the library's stated
 * readings):
 *   gs   = fl32(2688 / amax) per token (activations), per expanded row (the
 *          intermediate) or per expert (weights); 1 when amax == 0.
 *   sf   = E4M3_rne_satfinite(fl32(fl32(amax_16 * gs) / 6)).
 *   code = E2M1_rne_satfinite(fl32(x * fl32(gs / dec(sf)))), +0 if dec(sf)==0.
 *   Router logits are FP32 in a canonical order (8-element chunks, partial
 *   p sums chunks p, p+32, ... with fused multiply-adds, then a pairwise tree
 *   over the 32 partials); top-k by logit (ties to the lower expert id);
 *   weights = softmax over all experts, chosen ones renormalised.
 *   Requires hidden % 256 == 0, inter % 128 == 0, num_experts % 8 == 0,
 *   num_experts <= 256, 1 <= top_k <= min(num_experts, 16), and a router
 *   tile within one CTA's shared memory (hidden x 8..32 experts of the
 *   router weight in bf16 plus 48 KB of activation rings: hidden <= 11264 on
 *   sm_103a).
 *
 * Memory and ownership: every pointer argument is a device pointer on the
 * handle's device unless stated otherwise.  Inputs are borrowed and read in
 * stream order; the caller keeps them alive until the stream reaches the
 * work.  The handle owns the quantized weights and all workspace.
 *
 * Errors: every entry point returns a moe_status and never aborts; the text
 * of the last error on a handle is available from moe_get_last_error.
 * Kernel-side waits are bounded: a wait that runs out records
 * MOE_ERR_DEVICE_TIMEOUT in a host-visible status word, which the next
 * moe_forward and moe_get_status report.
 */
#ifndef MOE_NVFP4_H
#define MOE_NVFP4_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_handle moe_handle; /* opaque; owns all device memory */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,       /* bad pointer, size, shape or dtype */
  MOE_ERR_TOO_MANY_TOKENS = 2,   /* num_tokens > max_num_tokens */
  MOE_ERR_NOT_LOADED = 3,        /* forward / refresh before moe_load_weights */
  MOE_ERR_METADATA_CHANGED = 4,  /* refresh with a different shape/dtype/device */
  MOE_ERR_ALIAS = 5,             /* out overlaps x */
  MOE_ERR_CUDA = 6,              /* a CUDA runtime call failed */
  MOE_ERR_DEVICE_TIMEOUT = 7,    /* a bounded device-side wait ran out */
  MOE_ERR_UNSUPPORTED = 8        /* shape outside the supported set, or no sm_103a device */
} moe_status;

/* Deterministic mode: the top-k weighted reduction runs in a fixed order
 * (slot 0, 1, ..., K-1 per token) with no floating-point atomics, so the
 * output is bitwise identical across runs.  The w2 GEMM stores each
 * (token, slot) expert output row rounded to bf16, and a finalize kernel sums
 * a token's K rows in slot order in FP32.  Without the flag, forwards of at
 * most 64 tokens accumulate the expert rows with FP32 atomic adds in the w2
 * epilogue (the fused finalize); larger forwards take the ordered path in
 * either mode, since there the atomic traffic (top_k x the output) bounds
 * the w2 GEMM. */
#define MOE_FLAG_DETERMINISTIC 1u

/* Static per-tensor activation scales: the contract "CuTe DSL backend gets
 * per-token NVFP4 online quantization and reload" (Summary; Implementation
 * item 2) keeps apart from per-token quantization.  With this flag the
 * forward quantizes every token of x with one calibrated FP32 global scale,
 * and each expert's SwiGLU output with that expert's calibrated global
 * scale, both set with moe_set_static_scales, instead of scales derived from
 * each token's and each expanded row's maximum.  Blocks whose maximum times
 * the scale exceeds 2688 saturate (block scale 448, codes +-6). */
#define MOE_FLAG_STATIC_ACT_SCALES 2u

/* Shared-expert combination: with a shared expert (moe_config.shared_inter
 * > 0) the layer output is routed + shared by default; with this flag it is
 * (routed + shared) / 2, the 'average' combination strategy of the
 * Cohere2MoE sparse block in "SM10X Command-A-Plus decode 2.3x faster, BCG
 * capture memory -78%" (its key source listing). */
#define MOE_FLAG_SHARED_AVERAGE 4u

/* SwiGLU sigmoid form.  The pages do not fix how the activation between the
 * expert GEMMs is evaluated.  By default the w13 epilogue forms
 * sigmoid(g) = 1/2 + tanh(g/2)/2 with the hardware tanh approximation (one
 * special-function operation per element, relative error about 2^-11);
 * with this flag it forms sigmoid(g) = 1 / (1 + expf(-g)) with an IEEE
 * division.  Either way the requantized intermediate is not a bit-exact
 * target: its codes depend on FP32 accumulation in the tensor cores.  The
 * accurate form moves fewer of its near-tie rounding decisions away from an
 * FP64 evaluation. */
#define MOE_FLAG_ACCURATE_SIGMOID 8u

typedef struct {
  int hidden;          /* H: model width (K dim of w13, N dim of w2) */
  int inter;           /* I: expert intermediate width */
  int num_experts;     /* E */
  int top_k;           /* K: experts per token */
  int max_num_tokens;  /* worst-case tokens of one forward; fixes all buffer sizes */
  int device;          /* CUDA device ordinal */
  unsigned flags;      /* MOE_FLAG_* */
  int shared_inter;    /* Is: intermediate width of the shared expert, 0 = none
                          (a multiple of 128, at most 2048; not with
                          MOE_FLAG_STATIC_ACT_SCALES) */
} moe_config;

typedef enum { MOE_DTYPE_BF16 = 1 } moe_dtype;

/* Shape of an expert weight tensor as the caller holds it: a contiguous,
 * row-major [dims[0], dims[1], dims[2]] array of dtype on device `device`. */
typedef struct {
  int64_t dims[3];
  int dtype;           /* moe_dtype */
  int device;          /* CUDA ordinal the data lives on */
} moe_weight_desc;

/* Create a handle and allocate every device buffer for the worst-case forward
 * (max_num_tokens tokens).  Nothing is allocated afterwards.  *out is set to
 * NULL on failure. */
MOE_API moe_status moe_create(const moe_config* cfg, moe_handle** out);

/* Release all device memory of the handle.  Waits for the device.  NULL is
 * accepted. */
MOE_API moe_status moe_destroy(moe_handle* h);

/* Online NVFP4 conversion of bf16 expert weights.
 *   w13: [E, 2I, H] bf16; rows [0, I) of expert e are the gate projection,
 *        rows [I, 2I) the up projection.
 *   w2:  [E, H, I] bf16.
 * One FP32 global scale per expert and tensor (2688 / amax over the expert's
 * whole matrix), E4M3 block scales along the reduction dimension.  Enqueued
 * on `stream` (a cudaStream_t; NULL = legacy default stream).  The bf16
 * inputs may be freed once the stream has passed this call. */
MOE_API moe_status moe_load_weights(moe_handle* h, const void* w13, const moe_weight_desc* w13_desc,
                            const void* w2, const moe_weight_desc* w2_desc, void* stream);

/* Weight reload: re-quantize new bf16 weights into the SAME device buffers
 * (codes, block scales, global scales), so a CUDA graph captured around
 * moe_forward stays valid and replays with the new weights.  Fails with
 * MOE_ERR_NOT_LOADED before the first load and with MOE_ERR_METADATA_CHANGED
 * if any shape, dtype or device differs from the loaded weights (a captured
 * graph would then need to be recaptured).  Never reallocates. */
MOE_API moe_status moe_refresh_scales_inplace(moe_handle* h, const void* w13, const moe_weight_desc* w13_desc,
                                      const void* w2, const moe_weight_desc* w2_desc, void* stream);

/* Shared expert ("SM10X Command-A-Plus decode 2.3x faster, BCG capture
 * memory -78%", the Cohere2MoE sparse block of its key source listing: the
 * shared experts read the same input as the routed experts, on a second
 * stream while the routed experts run, and their output is added to the
 * routed output).  Online NVFP4 conversion of its bf16 weights, as
 * moe_load_weights does for one expert:
 *   w13s: [1, 2*Is, H] bf16 (gate rows [0, Is), up rows [Is, 2*Is));
 *   w2s:  [1, H, Is] bf16.
 * Calling it again requantizes into the same buffers (a captured graph stays
 * valid).  MOE_ERR_INVALID_ARG if the handle has no shared expert or a shape
 * differs.  With a shared expert, moe_forward returns MOE_ERR_NOT_LOADED
 * until this has been called.  Every forward then quantizes x per token once
 * more on the handle's second stream (forked from and joined back into the
 * caller's stream, so capture works as for moe_forward), runs the shared
 * expert's two GEMMs there, and the finalize adds (or averages, with
 * MOE_FLAG_SHARED_AVERAGE) its bf16 output rows into the routed sum in FP32
 * before the single bf16 rounding of the output. */
MOE_API moe_status moe_load_shared_weights(moe_handle* h, const void* w13s, const moe_weight_desc* w13s_desc,
                                           const void* w2s, const moe_weight_desc* w2s_desc, void* stream);

/* Calibrated global scales of the static contract, copied on `stream` into
 * handle-owned buffers (the same buffers every time, so a captured graph
 * replays with new values):
 *   x_gs: device pointer to 1 float, the w13 input's scale (all tokens);
 *   h_gs: device pointer to E floats, expert e's w2 input scale.
 * Scales follow gs = 2688 / calibrated maximum and must be positive and
 * finite.  MOE_ERR_INVALID_ARG unless the handle was created with
 * MOE_FLAG_STATIC_ACT_SCALES; a forward of such a handle before the first
 * call returns MOE_ERR_NOT_LOADED. */
MOE_API moe_status moe_set_static_scales(moe_handle* h, const float* x_gs, const float* h_gs, void* stream);

/* One forward of the routed MoE layer.
 *   x:      [num_tokens, H] bf16 activations (read only).
 *   gate_w: [H, E] bf16 router weight.
 *   out:    [num_tokens, H] bf16, written; must not overlap x.
 * 0 <= num_tokens <= max_num_tokens (0 is a no-op).  Enqueued on `stream`
 * with no host synchronisation, no allocation and no host read of device
 * results, so the call may be captured into a CUDA graph. */
MOE_API moe_status moe_forward(moe_handle* h, const void* x, const void* gate_w, void* out,
                       int num_tokens, void* stream);

/* moe_forward with an optional FP32 [E] bias added to the router logits
 * (NULL = none).  The bias moves both the top-k choice and the softmax. */
MOE_API moe_status moe_forward_ex(moe_handle* h, const void* x, const void* gate_w, const float* gate_bias,
                          void* out, int num_tokens, void* stream);

/* Same forward, but x, gate_w, gate_bias and out are HOST pointers: the call
 * copies the inputs into handle-owned device staging buffers, runs the
 * forward and copies the result back, all on `stream`, and returns after the
 * stream has finished (so it is not capturable). */
MOE_API moe_status moe_forward_host(moe_handle* h, const void* x_host, const void* gate_w_host,
                            const float* gate_bias_host, void* out_host, int num_tokens,
                            void* stream);

/* Device bytes owned by the handle (weights + workspace + staging). */
MOE_API size_t moe_get_workspace_bytes(const moe_handle* h);

/* Text of the last error on this handle ("" if none).  The pointer stays
 * valid until the next call on the handle. */
MOE_API const char* moe_get_last_error(const moe_handle* h);

/* Human-readable name of a status code. */
MOE_API const char* moe_status_string(moe_status s);

/* Reads the host-visible device status word without synchronising: MOE_OK,
 * or MOE_ERR_DEVICE_TIMEOUT if a kernel of this handle gave up a bounded
 * wait.  Call after synchronising the stream to see the latest state. */
MOE_API moe_status moe_get_status(const moe_handle* h);

/* ---------------------------------------------------------------------------
 * Stage timing (tracing).  When enabled, moe_forward records a CUDA event
 * before its first kernel and after each of its MOE_NUM_STAGES stages; inside
 * a stream capture the records become event nodes of the graph, so every
 * replay re-records them.  moe_get_stage_times returns the durations of the
 * last completed forward or replay (synchronise first).  Enabling allocates
 * the events; call it before any capture.
 * ------------------------------------------------------------------------ */
#define MOE_NUM_STAGES 7  /* router, top-k, permute, quantize, gemm_w13, gemm_w2, finalize */

MOE_API moe_status moe_set_stage_timing(moe_handle* h, int enable);

/* ms[i] = duration of stage i in milliseconds; on entry *n is the capacity of
 * ms, on return the number of stages written. */
MOE_API moe_status moe_get_stage_times(const moe_handle* h, float* ms, int* n);

/* Name of stage i ("router", "topk", ...), or NULL. */
MOE_API const char* moe_stage_name(int i);

/* ---------------------------------------------------------------------------
 * Routing without a handle and without allocation.  The method described on
 * the pages has no counterpart: this is a library convenience.
 *
 * For callers that must not allocate device memory when they route: a
 * runtime whose memory pool already holds all free device memory (a
 * cudaMalloc there fails), or a step that cannot afford the device-wide
 * synchronisation a cudaMalloc/cudaFree implies.  Such callers have no
 * moe_handle to hold a workspace, so the intermediate router logits live in
 * one fixed array in the library's device code: MOE_ROUTE_NOALLOC_MAX_LOGITS
 * floats (4 MiB per device, reserved when the library's device code is loaded
 * on that device).  After the first call on a device, nothing is allocated by
 * a call, by CUDA or otherwise.  Under CUDA's default lazy module loading the
 * device code (and with it the array) is loaded on a device by the first call
 * there, so that first call reserves the 4 MiB: make it before a memory pool
 * takes the device's free memory, as well as before any stream capture.
 *
 * Computes exactly the routing of moe_forward_ex on the same inputs (the same
 * kernels): FP32 router logits in the canonical order, plus gate_bias if not
 * NULL; top-k by logit, ties to the lower expert id; softmax over all
 * experts, chosen weights renormalised.
 *   x:         [num_tokens, hidden] bf16, device, 16-byte aligned.
 *   gate_w:    [hidden, num_experts] bf16, device, 16-byte aligned.
 *   gate_bias: [num_experts] f32, device, 16-byte aligned, or NULL.
 *   topk_ids:  [num_tokens, top_k] int32, written (slot order = descending
 *              logit).
 *   topk_w:    [num_tokens, top_k] f32, written.
 * Runs on the calling thread's current device, which must hold every
 * pointer; enqueued on `stream` (NULL = legacy default stream) with no host
 * synchronisation.  All buffers are the caller's.
 *
 * Limits and errors: hidden % 256 == 0, hidden <= 11264 (the router tile's
 * shared memory), num_experts % 8 == 0, num_experts <= 256,
 * 1 <= top_k <= min(num_experts, 16), otherwise MOE_ERR_UNSUPPORTED;
 * num_tokens * num_experts above MOE_ROUTE_NOALLOC_MAX_LOGITS returns
 * MOE_ERR_TOO_MANY_TOKENS (split the batch); NULL or misaligned pointers MOE_ERR_INVALID_ARG; a device other
 * than sm_103 MOE_ERR_UNSUPPORTED; num_tokens == 0 does nothing.
 *
 * The first call on each device does that device's set-up (loads the device
 * code there if it is not loaded yet, looks up the array's device address and
 * raises the router kernel's launch limits), so make one call on each device
 * before any stream capture and before a pool reserves its free memory.  The array is
 * shared by every call on the device: calls whose device work overlaps
 * (different streams, or threads without ordering between them) race on it
 * and corrupt each other's results; order them on one stream.
 * ------------------------------------------------------------------------ */
#define MOE_ROUTE_NOALLOC_MAX_LOGITS (1 << 20) /* num_tokens * num_experts, e.g. 8192 x 128 */

MOE_API moe_status moe_route_noalloc(const void* x, const void* gate_w, const float* gate_bias, int num_tokens,
                                     int hidden, int num_experts, int top_k, int32_t* topk_ids, float* topk_w,
                                     void* stream);

/* ---------------------------------------------------------------------------
 * Parity exports.  Each copies state left by the LAST moe_forward on the
 * handle (or by the last load/refresh for the weights) into caller device
 * buffers, in canonical row-major layouts, on `stream`.  T below is that
 * forward's num_tokens, R = T*K.
 * ------------------------------------------------------------------------ */

/* topk_ids int32 [T,K] (slot order), topk_w f32 [T,K], src_of_row int32 [R]
 * (row r of the expert-grouped order is slot src%K of token src/K),
 * expert_offsets int32 [E+1] (unpadded exclusive prefix sum). Any pointer may
 * be NULL to skip it. */
MOE_API moe_status moe_debug_routing(moe_handle* h, int32_t* topk_ids, float* topk_w, int32_t* src_of_row,
                             int32_t* expert_offsets, void* stream);

/* Router logits f32 [T,E] (bias included). */
MOE_API moe_status moe_debug_logits(moe_handle* h, float* logits, void* stream);

/* Per-token activation quantization: codes uint8 [T, H/2] (element 2i in the
 * low nibble), block scales uint8 [T, H/16] (E4M3), gs f32 [T]. */
MOE_API moe_status moe_debug_act_quant(moe_handle* h, uint8_t* codes, uint8_t* sf, float* gs, void* stream);

/* Quantized weights. which = 0: w13 -> codes [E, 2I, H/2], sf [E, 2I, H/16];
 * which = 1: w2 -> codes [E, H, I/2], sf [E, H, I/16]; gs f32 [E]. Rows in the
 * caller's order (gate rows first for w13). */
MOE_API moe_status moe_debug_weight_quant(moe_handle* h, int which, uint8_t* codes, uint8_t* sf, float* gs,
                                  void* stream);

/* Requantized intermediate of the last forward: h_codes uint8 [R, I/2],
 * h_sf uint8 [R, I/16], h_gs f32 [R], indexed by src = t*K + j. */
MOE_API moe_status moe_debug_intermediate(moe_handle* h, uint8_t* h_codes, uint8_t* h_sf, float* h_gs,
                                  void* stream);

/* The shared expert's part of the last forward (handles with a shared expert
 * only): rows bf16 [T, H], its w2 output for token t before the combination;
 * h_codes uint8 [T, Is/2], h_sf uint8 [T, Is/16], h_gs f32 [T], its
 * requantized intermediate.  Device pointers; rows may be NULL, and the
 * other three are all given or all NULL.  MOE_ERR_INVALID_ARG without a
 * shared expert, MOE_ERR_NOT_LOADED before the first forward. */
MOE_API moe_status moe_debug_shared(moe_handle* h, uint16_t* rows, uint8_t* h_codes, uint8_t* h_sf, float* h_gs,
                                    void* stream);

/* The shared expert's own per-token quantization of x in the last forward
 * (its second stream quantizes the tokens into token-ordered rows, with the
 * same per-token rules as the routed experts' input): codes uint8 [T, H/2],
 * sf uint8 [T, H/16], gs f32 [T], device pointers, all three required.
 * Errors as moe_debug_shared. */
MOE_API moe_status moe_debug_shared_act_quant(moe_handle* h, uint8_t* codes, uint8_t* sf, float* gs, void* stream);

/* Addresses of every device buffer the handle owns (weights, scales,
 * workspace), for checking that load/refresh never moves them.  On entry *n
 * is the capacity of ptrs; on return it is the number of buffers. */
MOE_API moe_status moe_debug_buffer_ptrs(const moe_handle* h, const void** ptrs, int* n);

/* Hardware conversion check: for n FP32 inputs, e2m1[i] = E2M1 code of in[i]
 * (round to nearest even, satfinite) and e4m3[i] = E4M3 byte of in[i], using
 * the same conversion instructions as the quantizer. Inputs must be finite. */
MOE_API moe_status moe_debug_convert(const float* in, uint8_t* e2m1, uint8_t* e4m3, int64_t n, void* stream);

/* Block-scaled FP4 GEMM through the same tcgen05 main loop as the expert
 * GEMMs: d[m][n] = sum_k dec(a)*dec(sfa)*dec(b)*dec(sfb) in FP32, for
 * a_codes [M, K/2], a_sf [M, K/16], b_codes [N, K/2], b_sf [N, K/16]
 * (canonical layouts), d f32 [M, N].  M % 128 == 0, N % 128 == 0,
 * K % 256 == 0.  Allocates and frees temporary buffers and synchronises the
 * stream; for tests only. */
MOE_API moe_status moe_debug_block_scaled_gemm(const uint8_t* a_codes, const uint8_t* a_sf,
                                       const uint8_t* b_codes, const uint8_t* b_sf,
                                       float* d, int M, int N, int K, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_NVFP4_H */
