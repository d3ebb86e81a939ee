/*
 * moe.h — C ABI of libmoe_b300.so, the gpt-oss Mixture-of-Experts MLP block on
 * one NVIDIA B300 (sm_103a).
 *
 * What is computed (pages about the gpt-oss architecture, cited by title and
 * section):
 *   "OpenAI 最新开源模型 gpt-oss 架构与训练解析", section 模型架构, MoE bullet:
 *     a router over E experts (32 for 20b, 128 for 120b), top-4 routing, softmax
 *     weighting over the selected experts only, and experts that are gated
 *     SwiGLU FFNs with clamping and a residual-style term;
 *   same page, weight-quantisation bullet: expert weights in MXFP4 (4.25 bits);
 *   same page, section 更深对比更宽: d_model = expert width = 2880;
 *   "【LLM】GPT-OSS架构变化详解", section 2.4: the MoE replaces the single FFN
 *     and a router picks the experts of each token.
 *
 * For token t with input x[t] (already normalised; moe_block_forward below
 * adds the RMSNorm before the block and the residual add after it):
 *   logits[e] = x[t]·router_w[e] + router_b[e]                    (fp32)
 *   S         = the k largest logits, ordered by (logit desc, index asc)
 *   w_j       = exp(l_j - l_max) / Σ_{j'∈S} exp(l_j' - l_max)
 *   z         = W_gu[e_j]·x[t] + b_gu[e_j]        (rows [0,W) gate, [W,2W) up)
 *   g = min(z_gate, limit);  u = clamp(z_up, -limit, limit)
 *   h         = g·σ(alpha·g)·(u + 1)
 *   y_j       = W_dn[e_j]·h + b_dn[e_j]
 *   out[t]    = bf16( Σ_j w_j·y_j )          (fp32 sum in slot order j = 0..k-1)
 * No shared expert is added.  Plain SwiGLU is limit = +inf, alpha = 1 with the
 * +1 absorbed into the up bias.
 *
 * MXFP4 weights: each row of a weight matrix is split along K (the reduction
 * axis) into blocks of 32 elements; a block holds 32 E2M1 codes (sign bit 3,
 * magnitude {0,0.5,1,1.5,2,3,4,6}[code&7]) and one E8M0 scale byte s meaning
 * 2^(s-127) (s = 255 is NaN and must not occur).  Codes are packed two per byte,
 * the even K index in the low nibble.
 *
 * Conventions common to every entry point
 *   - Every data pointer is DEVICE memory owned by the caller; the library
 *     allocates nothing and frees nothing.  Scratch comes from the caller's
 *     `workspace` of at least moe_workspace_bytes(...) bytes.
 *   - All work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is
 *     the legacy default stream).  No entry point synchronises, except
 *     moe_poll_status.
 *   - Pointers must be 16-byte aligned (the kernels move tiles with TMA and
 *     16-byte vector loads); violations return MOE_ERR_ALIGN.
 *   - Argument errors are detected on the host before anything is enqueued
 *     and leave every output untouched.  A failed launch returns MOE_ERR_CUDA.
 *     The message of the last failure on the calling thread is returned by
 *     moe_last_error().
 *   - Device-side failures (a bounded wait that ran out, an index out of range)
 *     do not trap: the kernel records a code in the workspace status word and
 *     returns; read it with moe_poll_status.
 *   - T = 0 returns MOE_OK and enqueues nothing.
 *   - Shape limits: d % 32 == 0, W % 32 == 0 (whole MX blocks), 1 <= E <= 256,
 *     1 <= k <= min(E, 8), 1 <= T, T·k < 2^31.
 *   - Determinism: for fixed inputs every output is bitwise reproducible run to
 *     run (no floating-point atomics; fixed reduction orders).
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_NULL = 1,        /* a required pointer is NULL */
  MOE_ERR_SHAPE = 2,       /* a size violates the limits above */
  MOE_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
  MOE_ERR_WORKSPACE = 4,   /* workspace smaller than moe_workspace_bytes() */
  MOE_ERR_UNSUPPORTED = 5, /* no sm_103a device, or a feature this build lacks */
  MOE_ERR_CUDA = 6,        /* a CUDA runtime/driver call failed */
  MOE_ERR_TIMEOUT = 7,     /* device: a bounded wait ran out (status word) */
  MOE_ERR_DEVICE_BOUNDS = 8 /* device: an index was out of range (status word) */
} moe_status;

/*
 * Bytes of scratch moe_forward / moe_route need for this shape (0 for T = 0).
 * The workspace holds the routing tables, the permuted activations, the hidden
 * activations h and the per-row expert outputs y; its first 256 bytes are the
 * device status word.  Returns 0 and sets moe_last_error() for invalid shapes.
 */
size_t moe_workspace_bytes(int64_t T, int d, int W, int E, int k);

/*
 * The whole MoE block: router, top-k, selected softmax, permutation, grouped
 * gate_up GEMM with the clamped SwiGLU, grouped down GEMM, weighted combine.
 *
 *   x_bf16      [T, d]        bf16, row-major
 *   router_w    [E, d]        fp32
 *   router_b    [E]           fp32
 *   w_gu_fp4    [E, 2W, d/2]  packed E2M1 (gate rows then up rows)
 *   w_gu_scale  [E, 2W, d/32] E8M0
 *   b_gu_bf16   [E, 2W]       bf16
 *   w_dn_fp4    [E, d, W/2]   packed E2M1
 *   w_dn_scale  [E, d, W/32]  E8M0
 *   b_dn_bf16   [E, d]        bf16
 *   limit       clamp bound (7.0 for gpt-oss; +inf disables the clamp)
 *   alpha       sigmoid slope (1.702 for gpt-oss)
 *   out_bf16    [T, d]        bf16, written completely
 * Precision: router logits, softmax and all accumulation in fp32.  The
 * weights enter the products exactly (code x 2^(scale - 127)).  Two number
 * formats carry the activations, chosen per call (moe_hidden_format says which):
 *  - decode-sized loads (at most 8 routed rows per expert on average) with a
 *    clamp 0 < limit <= 16, weight buffers 32-byte aligned: x and h as sums
 *    of E4M3 terms fed to the tensor cores' block-scaled MXFP4 x MXFP8
 *    products: x = hi + lo/16 with a power-of-two scale per 32-element block
 *    (exact for bf16 x within 2^-7 of its block's largest |x|, else within
 *    2^-13 of it), h = t0 + t1/16 + t2/256 + t3/4096 with one fixed
 *    scale 2^e that keeps |h| <= limit·(limit+1) inside the E4M3 range
 *    (about 16 significant bits);
 *  - otherwise x exactly (f16 after a per-token power-of-two scaling) and h
 *    as a pair of 16-bit terms, hi + lo: f16 (about 22 significant bits) when
 *    limit·(limit+1) < 16384, else bf16 (about 16 bits).
 * y is fp32; out is rounded once, to nearest even.
 */
moe_status moe_forward(const void* x_bf16, int64_t T, int d, int W,
                       const float* router_w, const float* router_b,
                       const uint8_t* w_gu_fp4, const uint8_t* w_gu_scale, const void* b_gu_bf16,
                       const uint8_t* w_dn_fp4, const uint8_t* w_dn_scale, const void* b_dn_bf16,
                       int E, int k, float limit, float alpha,
                       void* out_bf16, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The MoE sub-layer of a pre-norm transformer block, with the step before it
 * and the residual add after it:
 *   out = x + MoE(RMSNorm(x)),   RMSNorm(x) = x / sqrt(mean(x²) + eps) · norm_w
 * x is the un-normalised residual stream.  RMSNorm divides each token by its
 * root mean square, with no mean subtracted and no bias ("【LLM】GPT-OSS架构变化详解"
 * 2.7.1; "OpenAI 最新开源模型 gpt-oss 架构与训练解析", section RMSNorm 替换
 * LayerNorm); the residual connection is the one the latter page names in
 * section 更深对比更宽.  The learned per-feature scale norm_w and eps are not on
 * the pages (gpt-oss uses eps = 1e-5).
 *   norm_w   [d]  fp32
 *   eps      >= 0, finite
 * Every other argument is as for moe_forward.  The MoE's input is bf16, so it
 * reads RMSNorm(x) rounded to the nearest bf16 (ties to even); 1/rms is kept in
 * fp64 so that rounding is decided as for the exact value.  The normalisation
 * runs in the router kernel at decode sizes (a separate pass over x for more
 * than 256 tokens); the residual add runs in the combine, which rounds
 * x + Σ_j w_j·y_j once to bf16.  out may be the same buffer as x (an in-place
 * residual update).
 */
moe_status moe_block_forward(const void* x_bf16, int64_t T, int d, int W, const float* norm_w,
                             float eps, const float* router_w, const float* router_b,
                             const uint8_t* w_gu_fp4, const uint8_t* w_gu_scale,
                             const void* b_gu_bf16, const uint8_t* w_dn_fp4,
                             const uint8_t* w_dn_scale, const void* b_dn_bf16, int E, int k,
                             float limit, float alpha, void* out_bf16, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * Routing only (the first two stages of moe_forward), with its tables returned:
 *   topk_idx  [T, k]  int32   selected experts, slot order (logit desc, index asc)
 *   topk_w    [T, k]  fp32    softmax over the selected logits
 *   offsets   [E + 1] int32   offsets[e] = first permuted row of expert e,
 *                             offsets[E] = T·k
 *   perm      [T·k]   int32   permuted row -> t·k + j; rows sorted by
 *                             (expert, token, slot)
 *   inv       [T, k]  int32   (t, j) -> permuted row
 * Any of the five output pointers may be NULL to skip that table.  The
 * workspace is the same as moe_forward's.
 */
moe_status moe_route(const void* x_bf16, int64_t T, int d,
                     const float* router_w, const float* router_b, int E, int k,
                     int32_t* topk_idx, float* topk_w, int32_t* offsets,
                     int32_t* perm, int32_t* inv,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * Synchronises `stream`, then reads and returns the device status word of
 * `workspace` (MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_BOUNDS) left by the
 * last call that used this workspace.  Returns MOE_ERR_CUDA if the stream
 * itself reports an error.
 */
moe_status moe_poll_status(const void* workspace, void* stream);

/* Message describing the last failure on the calling thread ("" if none). */
const char* moe_last_error(void);

/*
 * Where an intermediate table lives inside the workspace, for inspection in
 * tests: writes its byte offset and size.  Contents are valid after a
 * moe_forward (or, for the routing tables, moe_route) on that workspace.
 *   which: 0 topk_idx int32[T,k]   1 topk_w fp32[T,k]     2 offsets int32[E+1]
 *          3 perm int32[T·k]       4 inv int32[T,k]       5 x_perm f16[T·k,d]
 *          6 h_hi [T·k,W]          7 h_lo [T·k,W]         8 y fp32[T·k,d]
 * h_hi and h_lo are f16 or bf16 as moe_hidden_format reports; in the E4M3
 * terms format the four E4M3 tables start at region 6 and run into region 7.
 * x_perm holds each routed row's token scaled by 2^e_t (e_t puts the token's
 * largest |x| in [2^14, 2^15), so the f16 value is exact); in the E4M3 terms
 * format it holds the two E4M3 tables of x (hi [T·k,d] then lo [T·k,d]).
 * Returns MOE_ERR_SHAPE for an invalid shape or `which`.
 */
moe_status moe_workspace_region(int64_t T, int d, int W, int E, int k, int which,
                                size_t* offset, size_t* bytes);

/*
 * The number format moe_forward uses for h between the two GEMMs on this shape
 * and clamp (for weight buffers aligned to 32 bytes):
 *   *format = MOE_HIDDEN_BF16_PAIR   h = hi + lo, two bf16 tables
 *             MOE_HIDDEN_F16_PAIR    h = hi + lo, two f16 tables
 *             MOE_HIDDEN_E4M3_TERMS  h = (t0 + t1/16 + t2/256 + t3/4096) · 2^(*exponent),
 *                                    four E4M3 tables [T·k,W] one after another
 * `exponent` may be NULL.  This only describes the intermediate tables inside
 * the workspace (for inspection); the results do not depend on it beyond
 * rounding.  Returns MOE_ERR_SHAPE / MOE_ERR_NULL like the other calls.  The
 * pages have no counterpart: this is an inspection aid.
 */
#define MOE_HIDDEN_BF16_PAIR 0
#define MOE_HIDDEN_F16_PAIR 1
#define MOE_HIDDEN_E4M3_TERMS 2
moe_status moe_hidden_format(int64_t T, int d, int W, int E, int k, float limit, int* format,
                             int* exponent);

/*
 * Tracing aid: make moe_forward / moe_block_forward calls from the calling
 * thread record CUDA events at its stage boundaries, on the call's stream.
 * `events` holds n = 7 cudaEvent_t handles (as void*) created by the caller:
 *   [0] before the router   [1] after router/top-k   [2] after the scan
 *   [3] after the permute   [4] after gate_up        [5] after down and the
 *   combine (which runs in the down kernel's epilogue)   [6] = [5]
 * The block-scaled design (MOE_HIDDEN_E4M3_TERMS) runs gate_up, down and the
 * combine in one kernel: [4] = [5] = [6] follow it.
 * n = 0 (or events = NULL) turns tracing off.  The handles are used by every
 * later moe_forward on this thread until replaced; the caller keeps them alive.
 * Returns MOE_ERR_SHAPE for any other n.
 */
moe_status moe_set_trace_events(void* const* events, int n);

/*
 * Failure detection.  Every wait inside the grouped GEMMs is bounded: after
 * the wait limit (2 s by default) the waiting role records MOE_ERR_TIMEOUT in
 * the status word, the CTA's other roles stop at their next wait, copies and
 * tensor-core work already issued are waited for (up to about 2 s more), and
 * the kernel returns; moe_poll_status then reports the timeout.
 * moe_set_wait_limit sets the limit, in seconds within [1e-4, 60], for later
 * calls from the calling thread; 0 restores the default.  Returns
 * MOE_ERR_SHAPE otherwise.  No counterpart on the pages.
 */
moe_status moe_set_wait_limit(double seconds);

/*
 * Test hooks for the failure paths (no counterpart on the pages; not for
 * production use).
 * moe_set_fault_injection(mode), per calling thread, for later calls:
 *   0  none (the default)
 *   1  the gate_up GEMM's weight producer issues nothing, so the MMA's wait
 *      for its first stage runs out: the call completes with MOE_ERR_TIMEOUT
 *      in the status word and out holding no meaningful values.
 * moe_debug_combine runs the weighted combine that the down GEMM runs in its
 * epilogue on caller tables (device memory): y [T·k, d] fp32, perm [T·k]
 * (permuted row -> t·k + j), inv [T, k], topk_w [T, k]; out [T, d] bf16.  The
 * workspace needs 256 + 4·T·ceil(d/128) bytes; its first word is the status
 * word (read it with moe_poll_status).  An inv entry outside [0, T·k) is left
 * out of its token's sum and recorded as MOE_ERR_DEVICE_BOUNDS.  perm must be
 * a permutation of [0, T·k).
 */
moe_status moe_set_fault_injection(int mode);
moe_status moe_debug_combine(const float* y, const int32_t* perm, const int32_t* inv,
                             const float* topk_w, int64_t T, int d, int k, void* out_bf16,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * Measurement aid: the dense rate, in TFLOP/s, of the tensor-core MMA forms
 * the grouped GEMMs issue (M = 128, fp32 accumulators in tensor memory):
 *   kind 0   tcgen05.mma kind::f16 on bf16 operands in shared memory, N = 256
 *   kind 1   tcgen05.mma kind::mxf8f6f4.block_scale, E2M1 x E4M3 with UE8M0
 *            scales, operands in shared memory, N = 256 (the block-scaled
 *            design's kind)
 *   kind 2   kind::f16 with A read from tensor memory, N = 128 (the TMEM
 *            design's form; its chunks are up to 192 tokens)
 *   kind 3   kind::f16 with A read from tensor memory, N = 256
 * One CTA per SM issues iters x 4 MMAs back to back; the launch is timed with
 * CUDA events on `stream` (synchronises it).  workspace: 4 bytes of device
 * memory for a status word.  Returns MOE_ERR_SHAPE for another kind or iters
 * outside [1, 2^24].  No counterpart on the pages.
 */
moe_status moe_mma_peak(int kind, int iters, double* tflops, void* workspace, void* stream);

/*
 * Size of the scratch array built into the library for moe_forward_noalloc:
 * 16 MiB, enough for up to 144 tokens at d = W = 2880 with k = 4 (E <= 128).
 */
#define MOE_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * moe_forward without a workspace argument, for callers that cannot allocate
 * device memory while they run the block (an engine plugin whose host forbids
 * allocation while serving, a real-time loop with a no-allocation rule, code
 * that is handed only its input and output buffers).  It computes exactly
 * what moe_forward computes, through the same kernels; the scratch is a
 * device array of MOE_NOALLOC_SCRATCH_BYTES inside the library, which every
 * GPU that loads the library keeps until the process exits.  This is a
 * convenience of this library; the pages the block follows have no
 * counterpart.
 *   - Arguments, layouts and results are those of moe_forward.
 *   - Shapes whose moe_workspace_bytes() exceeds MOE_NOALLOC_SCRATCH_BYTES are
 *     rejected with MOE_ERR_WORKSPACE and a message from moe_last_error();
 *     nothing is enqueued.
 *   - No cudaMalloc, cudaFree or other allocation happens.  The first call on
 *     a device looks up the array's device address (cudaGetSymbolAddress) with
 *     that device current; make that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents.
 *     Every call rewrites all of it that it reads, so nothing needs clearing,
 *     but calls that overlap on the GPU (two streams, two threads) race on it:
 *     issue them one after another.  Errors from argument checks are returned
 *     as usual (T = 0 included); device-side failures of the last call are
 *     read with moe_poll_status_noalloc.
 *   - The array's address is looked up once per device and kept: do not call
 *     this entry point again on a device after cudaDeviceReset.
 */
moe_status moe_forward_noalloc(const void* x_bf16, int64_t T, int d, int W,
                               const float* router_w, const float* router_b,
                               const uint8_t* w_gu_fp4, const uint8_t* w_gu_scale,
                               const void* b_gu_bf16, const uint8_t* w_dn_fp4,
                               const uint8_t* w_dn_scale, const void* b_dn_bf16, int E, int k,
                               float limit, float alpha, void* out_bf16, void* stream);

/*
 * moe_poll_status for moe_forward_noalloc: synchronises `stream`, then reads
 * the status word at the start of the built-in scratch array on the current
 * device (MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_BOUNDS from the last
 * no-alloc call there).  Allocates nothing.  No counterpart on the pages.
 */
moe_status moe_poll_status_noalloc(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
