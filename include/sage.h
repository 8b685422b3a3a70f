/*
 * sage.h -- C ABI of the GB300 (sm_103a) SageAttention-style quantized
 * attention forward.
 *
 * The method (diffusers issue #15014 "gfx1201 (RDNA4) SageAttention attention
 * backend: aiter package or Hub kernel?", section "Is your feature request
 * related to a problem?", kernel contract bullets):
 *   - INT8 QK^T and FP8 PV with FP32 accumulation;
 *   - Q and K quantized per 32-row block, V per channel;
 *   - inputs BF16 [B, S, H, 128], Q/K/V of equal shape, no mask, non-causal.
 * diffusers PR #15060 "Add aiter_sage_hub attention backend for AMD RDNA4
 * (gfx1201)", "What does this PR do?": head dim 128 only; inference only; the
 * kernel returns no LSE.  The same issue, "Describe the solution you'd
 * like": unsupported inputs are rejected with a clear error.
 *
 * Conventions for every entry point:
 *   - Pointers are device pointers unless stated otherwise; the caller owns
 *     every buffer.  Tensors are dense and row-major in the layouts given.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are stream-ordered and asynchronous; none synchronises
 *     the host except sage_sync_status().
 *   - All argument checks run on the host before any launch; a failed check
 *     launches nothing.  On failure the call returns a non-zero sage_status
 *     and sage_last_error() describes it (thread-local text).
 *   - Nothing traps on the device.  A device-side wait that runs past its
 *     limit records SAGE_ERR_TIMEOUT in a per-device error word, which
 *     sage_sync_status() reports.
 *   - Pointers are 16-byte aligned; the `out` of every entry point that
 *     runs the attention kernel is 32-byte aligned (the kernel writes each
 *     output row as 32-byte vectors).  Otherwise SAGE_ERR_MISALIGNED.
 *   - Shapes: B, S, H >= 1; D must be 128.  B*H <= 2^31-1.
 *     S_pad = ceil(S / 128) * 128, nb = ceil(S / 32).
 */
#ifndef SAGE_H_
#define SAGE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sage_status {
  SAGE_OK = 0,
  SAGE_ERR_INVALID_ARG = 1, /* a size < 1, a NULL pointer, a non-finite or non-positive scale */
  SAGE_ERR_UNSUPPORTED = 2, /* head dimension other than 128; a plan option not offered */
  SAGE_ERR_MISALIGNED = 3,  /* a pointer not 16-byte aligned (an attention `out` not 32-byte aligned) */
  SAGE_ERR_CUDA = 4,        /* a CUDA runtime or launch error (message kept) */
  SAGE_ERR_NO_MEMORY = 5,   /* workspace allocation failed */
  SAGE_ERR_TIMEOUT = 6,     /* a device wait gave up (reported by sage_sync_status) */
  SAGE_ERR_WORKSPACE = 7    /* caller workspace smaller than sage_workspace_bytes() */
} sage_status;

/* Head dimension, Q/K quantisation block and tile sizes of this library. */
#define SAGE_HEAD_DIM 128
#define SAGE_QK_BLOCK 32
#define SAGE_TILE 128

/* S rounded up to a multiple of 128 (the token extent of the quantised
 * layouts).  Returns 0 for S < 1. */
int64_t sage_padded_len(int S);

/* Number of kernels one call of sage_attn_fwd, _ws, _lse, _cross or _fused_q
 * launches for this shape (Sq = Skv for self-attention), or of
 * sage_attn_fwd_smooth_k when smooth_k is non-zero: zeroing of the V maxima,
 * Q/K quantisation with the V maxima, V encoding, attention (and for
 * smooth_k the K channel sums and means).  Returns -1 for an invalid shape.
 * No device work. */
int sage_attn_fwd_launches(int B, int Sq, int Skv, int H, int smooth_k);

/* Bytes of device workspace sage_attn_fwd_ws() / sage_attn_fwd_quantized()
 * need for this shape (0 if the shape is invalid).  Layout is private. */
size_t sage_workspace_bytes(int B, int S, int H, int D);

/*
 * sage_quantize_qkv -- quantise BF16 Q, K, V.
 * Passage: the issue's contract bullet "Q/K are quantized per 32-row block
 * and V per channel"; "FP8 PV" (PR #15060, "What does this PR do?").
 *
 *   q, k, v   in : bf16 [B, S, H, D]
 *   q_i8      out: int8 [B, H, S_pad, D]; rows >= S are 0
 *   q_scale   out: fp32 [B, H, nb]; block j covers tokens [32j, 32j+32) of
 *                  one (batch, head): scale = amax / 127,
 *                  code = clamp(rint(x / scale), -127, 127) (fp32 RNE
 *                  divisions); an all-zero block has scale 0 and codes 0
 *   k_i8, k_scale out: same for K
 *   vt_fp8    out: E4M3FN codes of V transposed, [B, H, D, S_pad];
 *                  columns >= S are 0
 *   v_scale   out: fp32 [B, H, D]: sv = amax over all S tokens of the
 *                  channel / 448, code = e4m3_rn_satfinite(v / sv)
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED (every pointer 16-byte
 * aligned), CUDA.  Uses 4*B*H*D bytes of scratch allocated from a private
 * stream-ordered pool (NO_MEMORY if that fails).
 */
sage_status sage_quantize_qkv(const void* q, const void* k, const void* v, int B, int S, int H, int D,
                              int8_t* q_i8, float* q_scale, int8_t* k_i8, float* k_scale,
                              uint8_t* vt_fp8, float* v_scale, void* stream);

/*
 * sage_quantize_qkv_noalloc -- sage_quantize_qkv for callers that cannot
 * allocate device memory.  No counterpart on the pages.
 *
 * Some callers cannot call cudaMalloc or any allocating routine where they
 * quantise: code running under a framework that owns every device
 * allocation, a real-time loop that must not take the driver's allocation
 * locks, or a device whose memory was reserved up front.  sage_quantize_qkv
 * takes its scratch (the per-channel |V| maxima, 4 * B * H * 128 bytes) from
 * a stream-ordered pool; this entry point uses a fixed 4 MiB array in device
 * memory instead and allocates nothing (it calls no cudaMalloc, no pool
 * allocation, no allocating library routine).
 *
 * Same arguments, outputs, layouts and results as sage_quantize_qkv.  Limit:
 * B * H <= 8192, else SAGE_ERR_INVALID_ARG with a message.  The array lives in
 * every GPU that loads this library until the process exits.  The first call
 * on a device looks up the array's device address (cudaGetSymbolAddress, with
 * that device current); make that first call before any stream capture.
 * Every call shares the array, which keeps the last call's contents; each call
 * zeroes the part it uses first.  Calls whose work overlaps on the GPU (on
 * different streams, or on other host threads) race on the array: order them.
 */
sage_status sage_quantize_qkv_noalloc(const void* q, const void* k, const void* v, int B, int S,
                                      int H, int D, int8_t* q_i8, float* q_scale, int8_t* k_i8,
                                      float* k_scale, uint8_t* vt_fp8, float* v_scale, void* stream);

/*
 * sage_attn_fwd -- the whole path: quantise Q/K/V, then fused quantized
 * attention.  Passage: the issue's contract bullets (INT8 QK^T, FP8 PV,
 * FP32 accumulation; BF16 [B, S, H, 128]; no mask, non-causal) and
 * aiter.gfx1201_sage_attention(q, k, v, softmax_scale) as named there.
 *
 *   q, k, v        in : bf16 [B, S, H, D]
 *   out            out: bf16 [B, S, H, D] = softmax(QK^T * softmax_scale) V
 *                       computed by the quantised algorithm; no LSE
 *   softmax_scale  in : finite, > 0 (typically 1/sqrt(D))
 * The workspace (sage_workspace_bytes) is taken from a private
 * stream-ordered memory pool on `stream` and released in stream order, so
 * concurrent calls on different streams do not share it.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, NO_MEMORY, CUDA.
 */
sage_status sage_attn_fwd(const void* q, const void* k, const void* v, void* out, int B, int S, int H,
                          int D, float softmax_scale, void* stream);

/* As sage_attn_fwd, with caller-owned workspace of at least
 * sage_workspace_bytes(B, S, H, D) bytes (256-byte aligned).  Calls that
 * share a workspace must not overlap on the GPU.  Extra error: WORKSPACE. */
sage_status sage_attn_fwd_ws(const void* q, const void* k, const void* v, void* out, int B, int S,
                             int H, int D, float softmax_scale, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * sage_attn_fwd_lse -- sage_attn_fwd that also writes each query row's
 * log-sum-exp.  Passage: PR #15060, "What does this PR do?" (the pages' kernel
 * returns no LSE; the LSE is what merging partial attentions of one query,
 * e.g. over sequence shards, needs).
 *
 *   lse  out: fp32 [B, H, S] (device, 16-byte aligned), row (b, h, i) =
 *             ln 2 * (m + log2 L - log2 448): m the row's final running max
 *             of the base-2 scores, L its accumulated E4M3 weights (the
 *             normaliser of `out`).  This is log sum_j exp(scale q_i . k_j)
 *             as the quantised computation estimates it.
 * Everything else, including errors, as sage_attn_fwd; `out` is identical.
 */
sage_status sage_attn_fwd_lse(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                              int S, int H, int D, float softmax_scale, void* stream);

/*
 * sage_attn_fwd_cross -- quantised cross-attention: Q has Sq rows, K and V
 * have Skv rows (Skv != Sq allowed; Skv == Sq gives sage_attn_fwd exactly).
 * Passage: the pages' second workload, shorter K/V, which the gfx1201 kernel
 * sends to its fallback (issue #15014, "Describe the solution you'd like";
 * SageAttention 2.2 results in InvokeAI PR #9657, "Summary").
 *
 *   q         in : bf16 [B, Sq, H, D]; k, v in: bf16 [B, Skv, H, D]
 *   out       out: bf16 [B, Sq, H, D]
 *   lse       out: fp32 [B, H, Sq] as sage_attn_fwd_lse, or NULL for none
 * Q and K are quantised over their own 32-row blocks, V per channel over
 * its own Skv tokens.  Shape limits (D = 128, lengths >= 1) apply to both
 * lengths; errors as sage_attn_fwd.
 */
sage_status sage_attn_fwd_cross(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                                int Sq, int Skv, int H, int D, float softmax_scale, void* stream);

/*
 * sage_plan -- one sage_attn_fwd_cross call (sage_attn_fwd when Sq == Skv
 * and lse is NULL) fixed to its pointers and shape, recorded once as a CUDA
 * graph and replayed by sage_plan_launch.  What it computes is that call's
 * (issue #15014 and PR #15060, as sage_attn_fwd: Q/K per-32-row-block INT8,
 * V per-channel FP8, attend); the plan only removes the per-call host work
 * (argument checks, workspace allocation, tensor-map encoding and the
 * separate launches) for shapes too small to hide it.  No counterpart on
 * the pages.
 *
 * sage_plan_create: arguments as sage_attn_fwd_cross (device pointers,
 *   layouts, lse optional), checked the same way; *plan receives the plan
 *   (host object owned by the caller) or NULL on failure.  The plan owns
 *   the workspace the call would otherwise take from the library's pool
 *   (sage_workspace_bytes(B, S, H, D) bytes when Sq == Skv == S), allocated
 *   here with cudaMalloc on the current device, and records the
 *   launches on a private stream: nothing runs on the device during
 *   creation.  The wait limit in force (sage_set_wait_timeout_ns) is the
 *   one the plan's kernels use; the timing hook (sage_set_attention_events)
 *   is not recorded.  Errors: INVALID_ARG (plan NULL, bad shape or scale),
 *   MISALIGNED, NO_MEMORY (workspace), CUDA (capture or instantiation).
 * sage_plan_launch: runs the recorded call on `stream` (a cudaStream_t as
 *   void*; NULL = legacy default stream), reading q, k and v as they are at
 *   that point of the stream and writing out (and lse).  The current device
 *   must be the plan's.  Launches of one plan share its workspace, so they
 *   must not overlap: issue them on one stream or order them.  Allocates
 *   nothing.  Errors: INVALID_ARG (plan NULL, other device), CUDA.
 * sage_plan_destroy: frees the plan and its workspace (cudaFree, which waits
 *   for the device's outstanding work).  NULL is a no-op.  Errors: CUDA.
 * sage_plan_create_ex: sage_plan_create recording one of the variant calls
 *   instead, chosen by `flags`: SAGE_PLAN_SMOOTH_K records
 *   sage_attn_fwd_smooth_k (K smoothing before the attention step),
 *   SAGE_PLAN_FUSED_Q records sage_attn_fwd_fused_q (Q quantised inside the
 *   attention kernel); 0 is sage_plan_create.  The results are those calls'
 *   (bit for bit).  Both variants are self-attention without LSE, so a flag
 *   needs Sq == Skv and lse NULL (INVALID_ARG otherwise); both flags at once
 *   or an unknown bit: UNSUPPORTED.  Everything else as sage_plan_create.
 */
typedef struct sage_plan sage_plan;
#define SAGE_PLAN_SMOOTH_K 1u
#define SAGE_PLAN_FUSED_Q 2u
sage_status sage_plan_create(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Sq,
                             int Skv, int H, int D, float softmax_scale, sage_plan** plan);
sage_status sage_plan_create_ex(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Sq,
                                int Skv, int H, int D, float softmax_scale, unsigned flags, sage_plan** plan);
sage_status sage_plan_launch(sage_plan* plan, void* stream);
sage_status sage_plan_destroy(sage_plan* plan);

/*
 * sage_quantize_qkv_smooth_k -- sage_quantize_qkv with K smoothing: before K
 * is quantised, each (batch, head, channel) loses its mean over the S
 * tokens.  Passage: InvokeAI PR #9657, "Summary" / "How it works"
 * (SageAttention's smooth_k; softmax-invariant, since every score of a query
 * row moves by the same q . mean).
 *   k_mean  out: fp32 [B, H, D]: fp32(sum_s k / S), the sum exact in double
 *   k_i8, k_scale: codes and block scales of fp32(k - mean); other outputs,
 *   layouts and errors as sage_quantize_qkv.
 */
sage_status sage_quantize_qkv_smooth_k(const void* q, const void* k, const void* v, int B, int S, int H, int D,
                                       int8_t* q_i8, float* q_scale, int8_t* k_i8, float* k_scale, uint8_t* vt_fp8,
                                       float* v_scale, float* k_mean, void* stream);

/*
 * sage_attn_fwd_smooth_k -- sage_attn_fwd with K smoothing (as
 * sage_quantize_qkv_smooth_k) before the attention step.  The pages measure
 * it helping typical heads and hurting outlier heads, so it is opt-in.
 * Arguments and errors as sage_attn_fwd.
 */
sage_status sage_attn_fwd_smooth_k(const void* q, const void* k, const void* v, void* out, int B, int S, int H,
                                   int D, float softmax_scale, void* stream);

/*
 * sage_attn_fwd_fused_q -- sage_attn_fwd with Q quantised inside the
 * attention kernel, as the pages' kernel does (issue #15014, contract
 * bullet "quantized per 32-row block ... inside the kernel"): the kernel
 * loads bf16 Q and each softmax warp quantises its own 32-row block before
 * the first QK^T; only K and V go through the separate quantisation pass.
 * Same arguments, results (bit for bit) and errors as sage_attn_fwd.  On
 * GB300 it is slower than sage_attn_fwd: the in-kernel quantisation sits on
 * every CTA's critical path ahead of its first MMA.
 */
sage_status sage_attn_fwd_fused_q(const void* q, const void* k, const void* v, void* out, int B, int S,
                                  int H, int D, float softmax_scale, void* stream);

/*
 * sage_debug_fused_q -- sage_attn_fwd_fused_q that also writes out the Q
 * codes and block scales its attention kernel computed.
 *   q_i8     out: int8 [B, H, S_pad, D] (rows >= S are 0)
 *   q_scale  out: fp32 [B, H, nb]
 * Same values sage_quantize_qkv writes for Q; for tests.  Errors as
 * sage_attn_fwd.
 */
sage_status sage_debug_fused_q(const void* q, const void* k, const void* v, void* out, int B, int S, int H,
                               int D, float softmax_scale, int8_t* q_i8, float* q_scale, void* stream);

/*
 * sage_attn_fwd_quantized -- the attention step alone, from operands in the
 * layouts sage_quantize_qkv() writes (same passage as sage_attn_fwd).
 * `workspace` (caller-owned, >= sage_workspace_bytes) receives fp16 copies of
 * the INT8 codes that feed the tensor cores.  Extra error: WORKSPACE.
 */
sage_status sage_attn_fwd_quantized(const int8_t* q_i8, const float* q_scale, const int8_t* k_i8,
                                    const float* k_scale, const uint8_t* vt_fp8,
                                    const float* v_scale, void* out, int B, int S, int H, int D,
                                    float softmax_scale, void* workspace, size_t workspace_bytes,
                                    void* stream);

/*
 * sage_debug_qk_int32 -- test entry: runs sage_attn_fwd_quantized and also
 * writes the exact integer Q K^T accumulators the tensor cores produced,
 * s_out int32 [B, H, S, S] (device, caller-owned; B*H*S*S*4 bytes).
 * Passage: "INT8 QK^T ... with FP32 accumulation" (issue #15014); the
 * accumulators are integers below 2^24 and equal the INT32 dot products.
 */
sage_status sage_debug_qk_int32(const int8_t* q_i8, const float* q_scale, const int8_t* k_i8,
                                const float* k_scale, const uint8_t* vt_fp8, const float* v_scale,
                                void* out, int32_t* s_out, int B, int S, int H, int D,
                                float softmax_scale, void* workspace, size_t workspace_bytes,
                                void* stream);

/*
 * sage_debug_staging_codes -- test entry: the Q/K quantisation exactly as
 * sage_attn_fwd runs it before the attention kernel (the same launch), into
 * caller buffers.  The codes are the INT8 values of sage_quantize_qkv stored
 * as fp16 (the tensor-core operand type of QK^T; every code is an integer in
 * [-127, 127], exact in fp16).  Passage: the issue's contract bullet "Q/K are
 * quantized per 32-row block".
 *
 *   q, k       in : bf16 [B, S, H, D]
 *   q16, k16   out: fp16 [B, H, S_pad, D]; rows >= S are 0
 *   q_scale, k_scale out: fp32 [B, H, nb], as sage_quantize_qkv
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, CUDA.
 */
sage_status sage_debug_staging_codes(const void* q, const void* k, int B, int S, int H, int D, void* q16,
                                     float* q_scale, void* k16, float* k_scale, void* stream);

/* Fault sites of sage_debug_inject_fault. */
enum {
  SAGE_FAULT_NONE = 0,          /* disarm */
  SAGE_FAULT_POOL_ALLOC = 1,    /* a workspace / scratch allocation (the library's pool, or a plan's workspace) */
  SAGE_FAULT_QUANT_LAUNCH = 2,  /* the Q/K quantisation launch of the attention entry points */
  SAGE_FAULT_ATTN_LAUNCH = 3    /* the attention kernel launch */
};

/*
 * sage_debug_inject_fault -- host-side fault injection for tests (no
 * counterpart on the pages; off by default).  Arms one site: the site's
 * (skip+1)-th next event, in any thread, fails without doing its work (no
 * allocation, no launch) and reports what a real failure there reports --
 * SAGE_ERR_NO_MEMORY for the pool, SAGE_ERR_CUDA for a launch -- with
 * "injected fault" in sage_last_error(); then the hook disarms.  Work the
 * call had already enqueued stays valid, and its workspace is released in
 * stream order as on every other failure.  Nothing faults on the device, and
 * the CUDA context stays usable.  Returns INVALID_ARG for an unknown site or
 * a negative skip.
 */
sage_status sage_debug_inject_fault(int site, int skip);

/*
 * sage_debug_pool_state -- test query (no counterpart on the pages): whether
 * this library has created its private stream-ordered memory pool on the
 * current device (*created, 0 or 1), and the bytes currently allocated from
 * it (*used_bytes; 0 if none).  Host pointers.  Errors: INVALID_ARG, CUDA.
 */
sage_status sage_debug_pool_state(int* created, uint64_t* used_bytes);

/*
 * sage_debug_wait_timeout -- test entry for failure detection without a GPU
 * fault: launches one warp that waits on an mbarrier nothing arrives on,
 * with a limit of timeout_ns (1..10^10).  The wait gives up, records
 * SAGE_ERR_TIMEOUT in the device error word and the kernel returns;
 * sage_sync_status() then reports it.  No counterpart on the pages.
 */
sage_status sage_debug_wait_timeout(uint64_t timeout_ns, void* stream);

/* Synchronise `stream`, then report (and clear) the device error word of the
 * current device: SAGE_OK, SAGE_ERR_TIMEOUT, or SAGE_ERR_CUDA if the stream
 * itself failed. */
sage_status sage_sync_status(void* stream);

/* Limit, in nanoseconds, of every device-side wait in later launches from
 * this process (default 2 s; 0 restores the default). */
void sage_set_wait_timeout_ns(uint64_t ns);

/* Timing hook (no counterpart on the pages): while set, every
 * sage_attn_fwd / _ws / _lse / _cross call made by this thread records `before`
 * on its stream immediately before launching its attention kernel and
 * `after` immediately after, so that the kernel's own duration can be read
 * with cudaEventElapsedTime.  Both are cudaEvent_t passed as void*, owned by
 * the caller; (NULL, NULL) clears the hook. */
void sage_set_attention_events(void* before, void* after);

/* Thread-local text of the last failure on this thread ("" if none). */
const char* sage_last_error(void);

/* Static name of a status code. */
const char* sage_status_string(sage_status s);

#ifdef __cplusplus
}
#endif

#endif /* SAGE_H_ */
