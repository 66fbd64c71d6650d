/*
 * linattn — C ABI of the GB300 (sm_103a) chunked gated-delta-rule prefill library.
 *
 * The path (metrale engine documentation pages "split_prefill.rs", trait
 * LayerSplitPrefill, and "glm5next_kda/prefill.rs", Glm5NextKdaLayer::prefill_with_pad_fill):
 *
 *   x --conv1d+SiLU (carried conv state)--> [q | k | v] --L2 per q|k head--> gated delta rule
 *   S_t = S_{t-1} diag(alpha_t) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,  o_t = scale S_t q_t,
 *   alpha_t = exp(g_t) (scalar per v-head: GDN; one value per k-channel: KDA),
 *
 * evaluated chunk by chunk (64 tokens) with the WY form: per chunk the cumulative gate gc,
 * A = strictly-lower(diag(beta) (K K^T (.) decay)), U' = (I + A)^{-1} (diag(beta) V -
 * diag(beta) (K (.) e^gc) H), O = scale ((Q (.) e^gc) H + P U'), and the carried state
 * H <- diag(e^gc_L) H + (K (.) e^{gc_L - gc})^T U'.
 *
 * Conventions shared by every call
 *  - Pointers are raw DEVICE pointers owned by the caller, unless stated otherwise. The library
 *    allocates no device memory and keeps no per-call state; all work is enqueued on `stream`
 *    (a cudaStream_t passed as uint64_t; 0 = legacy default stream) and is asynchronous. Two
 *    fixed arrays live in the library's own device image for the life of the process: the
 *    status word of la_device_status and the scratch of la_gdn_prefill_varlen_noalloc. Their
 *    device addresses are looked up once per device and cached, so a cudaDeviceReset (or any
 *    other teardown of the primary context) invalidates them: do not call the library on a
 *    device after resetting it in the same process.
 *  - Host-side fault injection (testing): with the environment variable LA_FAULT_INJECT set to
 *    "launch", every call that passes its checks returns LA_ERR_CUDA ("injected launch
 *    failure") instead of launching; set to "alloc", every call that needs one of the library's
 *    device arrays (the status word, the no-allocation scratch) returns LA_ERR_CUDA as if its
 *    address lookup had failed. Nothing is launched and no buffer is touched in either case.
 *    The variable is read at every call.
 *  - Every check runs on the host BEFORE any launch; on error nothing is launched and no buffer
 *    is touched. Return value: LA_OK or one of the LA_ERR_* codes; la_last_error() then gives a
 *    thread-local message.
 *  - dtype selects the activation type (x, conv weights/state, q, k, v, out): LA_F32 or LA_BF16.
 *    Gates g, beta and the recurrent state are always fp32.
 *  - Vector access: every activation pointer must be 16-byte aligned and every activation row
 *    stride / channel count a multiple of 16 bytes (8 bf16 or 4 fp32 elements).
 *  - Token counts: a call covers 1..max_tokens tokens; 0 or more than max_tokens is refused with
 *    LA_ERR_COUNT before any launch ("glm5next_kda/prefill.rs", module invariant and the
 *    t == 0 || t > ws.max_tokens check of prefill_with_pad_fill).
 *  - States are updated in place: the conv state and the recurrent state carry a stream from one
 *    call to the next ("split_prefill.rs", prefill_phase1_conv1d_one advancing the conv state;
 *    "glm5next_kda/prefill.rs", prefill starting from the carried state).
 *  - Varlen streams: cu_seqlens is a DEVICE int32 array of B+1 token offsets, cu_seqlens[0] = 0,
 *    nondecreasing, cu_seqlens[B] = total_tokens, each length <= max_seqlen. A zero-length
 *    stream is a no-op for its state. The kernels check these bounds on the device; a violation
 *    skips the offending stream and raises a flag that la_device_status() reports.
 */
#ifndef LINATTN_H
#define LINATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---- */
#define LA_OK 0
#define LA_ERR_ARG 1         /* null / misaligned pointer, bad stride, inconsistent dims */
#define LA_ERR_COUNT 2       /* token count 0 or above max_tokens: refused before any launch */
#define LA_ERR_UNSUPPORTED 3 /* dims outside the compiled instances (cf. the pages' Ok(false)) */
#define LA_ERR_CUDA 4        /* the CUDA runtime reported an error at launch */

/* ---- activation dtypes ---- */
#define LA_F32 0
#define LA_BF16 1

/* ---- device status flags (la_device_status) ---- */
#define LA_DEV_BAD_SEQLENS 1 /* cu_seqlens not monotone, out of range, or a length > max_seqlen */
#define LA_DEV_TIMEOUT 2     /* a bounded wait inside a kernel gave up; that kernel's results are
                                incomplete (never expected; reported instead of hanging) */
/* Every wait of the tensor-core kernels on an mbarrier (MMA or copy completion) gives up after
 * 2 s; the block then drains its own MMAs and copies, frees its tensor memory, raises
 * LA_DEV_TIMEOUT and exits, so the context stays usable. Two environment variables, read at
 * every call, exist to test that path: LA_WAIT_LIMIT_NS (a positive integer, raised to at least
 * 1 ms) replaces the 2 s limit, and LA_DEBUG_STALL=1 makes each block of those kernels wait once on a barrier that
 * nothing completes, so that the wait runs out. Neither is meant for production use. */

/* ABI version of this header (bumped on any signature change). */
#define LA_ABI_VERSION 1
int la_abi_version(void);

/* Thread-local description of the last error returned on this host thread ("" if none). */
const char *la_last_error(void);

/* Synchronises `stream`, then returns and clears the device status flags (LA_DEV_*) raised by
 * kernels of this library on the current device since the last call. Returns a negative value
 * if the synchronisation itself failed. Debug/test use: it blocks the host. */
int la_device_status(uint64_t stream);

/* ---------------------------------------------------------------------------------------------
 * Causal depthwise conv1d + SiLU over one stream, advancing its conv state.
 * "glm5next_kda/prefill.rs", conv_prefill launch (conv + SiLU only, bias slot NULL);
 * "split_prefill.rs", prefill_phase1_conv1d_one.
 *
 *   xh = [conv_state (kernel-1 rows, oldest first) ; x (t rows)]
 *   out[tau][c] = SiLU(bias[c] + sum_{j<kernel} w[c][j] * xh[tau + j][c])   (tap kernel-1 = current)
 *   conv_state <- xh[t .. t+kernel-2]
 *
 * conv_state [kernel-1][channels] (dtype, contiguous, in/out; may be NULL when kernel == 1)
 * x          [t][x_stride]      (dtype; the first `channels` entries of each row are read)
 * w          [channels][kernel] (dtype, contiguous)
 * bias       [channels] (dtype) or NULL for none
 * out        [t][out_stride]    (dtype; may not alias x)
 * kernel in 1..4.  Errors: LA_ERR_COUNT (t), LA_ERR_ARG, LA_ERR_UNSUPPORTED (kernel).
 * ------------------------------------------------------------------------------------------- */
int la_conv1d_silu_prefill(void *conv_state, const void *x, const void *w, const void *bias,
                           void *out, int t, int max_tokens, int channels, int kernel,
                           int64_t x_stride, int64_t out_stride, int dtype, uint64_t stream);

/* Same over B packed streams (cu_seqlens), each with its own conv state: conv_state_ptrs is a
 * DEVICE array of B device pointers, each to a [kernel-1][channels] state of dtype. */
int la_conv1d_silu_prefill_varlen(const uint64_t *conv_state_ptrs, const void *x, const void *w,
                                  const void *bias, void *out, const int32_t *cu_seqlens, int B,
                                  int total_tokens, int max_tokens, int channels, int kernel,
                                  int64_t x_stride, int64_t out_stride, int dtype,
                                  uint64_t stream);

/* Fused front end: conv1d + SiLU as above (single stream when cu_seqlens is NULL and B == 1,
 * else varlen), then the per-(token, head) L2 norm of la_l2norm_heads over the first
 * l2_heads*head_dim output channels, in one pass: x is read once and out written once. The conv
 * output is rounded to dtype before it is normalised, exactly as the two separate calls store
 * and re-read it, so the results are bitwise identical to la_conv1d_silu_prefill[_varlen]
 * followed by la_l2norm_heads ("glm5next_kda/prefill.rs": conv_prefill then l2 on conv_out).
 * conv_state_ptrs: DEVICE array of B device pointers to [kernel-1][channels] states.
 * head_dim in {64, 128}; l2_heads*head_dim <= channels. */
int la_conv1d_silu_l2_prefill(const uint64_t *conv_state_ptrs, const void *x, const void *w,
                              const void *bias, void *out, const int32_t *cu_seqlens, int B,
                              int total_tokens, int max_tokens, int channels, int kernel,
                              int l2_heads, int head_dim, float eps, int64_t x_stride,
                              int64_t out_stride, int dtype, uint64_t stream);

/* ---------------------------------------------------------------------------------------------
 * Per-(token, head) L2 norm, in place, over the first n_heads*head_dim channels of each row.
 * "glm5next_kda/prefill.rs", l2 launch (grid q|k heads x tokens, eps = cfg.l2_eps);
 * "split_prefill.rs", prefill_phase1_l2_batched (over all stacked tokens).
 *   x[tau][h*head_dim + c] <- x / sqrt(sum_c x^2 + eps)
 * x [t][row_stride] (dtype). head_dim in {64, 128}. t >= 1.
 * ------------------------------------------------------------------------------------------- */
int la_l2norm_heads(void *x, int t, int n_heads, int head_dim, int64_t row_stride, float eps,
                    int dtype, uint64_t stream);

/* ---------------------------------------------------------------------------------------------
 * Recurrence arguments shared by the three prefill calls below.
 *
 * h_state_ptrs  DEVICE array of B device pointers; pointer s -> fp32 state of stream s laid out
 *               [Hv][dk][dv] (H = S^T, H[c][d] = S[d][c]); read and updated in place.
 *               ("split_prefill.rs", prefill_gdn_full_batched: one h-state pointer per stream.)
 * q, k          [tokens][q_stride], [tokens][k_stride] (dtype): head h at columns h*dk..h*dk+dk-1,
 *               h < Hk. They may point into one packed [q | k | v] buffer (the split of the
 *               pages' split_widen becomes pointer arithmetic).
 * v             [tokens][v_stride] (dtype): v-head j at columns j*dv..j*dv+dv-1, j < Hv.
 * beta          [tokens][Hv] fp32.
 * out           [tokens][Hv][dv] (dtype, contiguous). Rows of padding are never written.
 * GQA           v-head j reads q/k head floor(j*Hk/Hv); Hv must be a multiple of Hk.
 * scale         output scale (the pages pass 1/sqrt(head_dim) to chunk_scan).
 * dk, dv        in {64, 128}.
 * workspace     device scratch of at least la_prefill_workspace_bytes(...) bytes (16-byte
 *               aligned); may be NULL when that size is 0.
 * ------------------------------------------------------------------------------------------- */

/* Bytes of device workspace the prefill calls need for these sizes (0 if none). */
size_t la_prefill_workspace_bytes(int B, int total_tokens, int Hk, int Hv, int dk, int dv,
                                  int dtype);

/* GDN, B streams of equal length T back to back (tokens s*T .. s*T+T-1 belong to stream s).
 * "split_prefill.rs", prefill_gdn_full_batched (h_state_ptrs, batch_size, chunk_len).
 * g [B*T][Hv] fp32 log-decay (alpha = exp(g)). Count rule: 1 <= B*T <= max_tokens. */
int la_gdn_prefill_batched(const uint64_t *h_state_ptrs, const void *q, const void *k,
                           const void *v, const float *g, const float *beta, void *out, int B,
                           int T, int max_tokens, int Hk, int Hv, int dk, int dv,
                           int64_t q_stride, int64_t k_stride, int64_t v_stride, float scale,
                           int dtype, void *workspace, size_t workspace_bytes, uint64_t stream);

/* GDN over B streams of different lengths driven by cu_seqlens (device) and max_seqlen.
 * "split_prefill.rs", prefill_gdn_full_batched_fla_varlen (cu_seqlens, total_nt, max_seqlen).
 * g [total_tokens][Hv] fp32. Count rule: 1 <= total_tokens <= max_tokens. */
int la_gdn_prefill_varlen(const uint64_t *h_state_ptrs, const void *q, const void *k,
                          const void *v, const float *g, const float *beta, void *out,
                          const int32_t *cu_seqlens, int B, int total_tokens, int max_seqlen,
                          int max_tokens, int Hk, int Hv, int dk, int dv, int64_t q_stride,
                          int64_t k_stride, int64_t v_stride, float scale, int dtype,
                          void *workspace, size_t workspace_bytes, uint64_t stream);

/* GDN varlen like la_gdn_prefill_varlen, for callers that cannot allocate device memory: it
 * takes no workspace and allocates nothing. Some callers cannot call cudaMalloc or grow a pool
 * at the moment they run this layer (an engine whose device memory is fully carved up by its
 * own allocator, a plugin with a fixed call signature that has nowhere to pass a workspace,
 * code that must not allocate while other work is being captured or replayed); this call lets
 * them still use the tensor-core path. The paper has no counterpart: it is a library service.
 *  - Scratch: a fixed array inside the library's device image (about 17 KB), held on every GPU
 *    that loads the library until the process exits. It serves at most 4096 streams per call;
 *    more is refused with LA_ERR_UNSUPPORTED before any launch.
 *  - Covers bf16 activations with dk = dv = 128 (the tensor-core kernel), else
 *    LA_ERR_UNSUPPORTED. All other arguments and errors are those of la_gdn_prefill_varlen.
 *  - Shared state: every call on a device uses the same scratch; the call re-initialises what
 *    must start at zero, but two calls whose work overlaps on the GPU (different streams, no
 *    ordering between them) race and give wrong results. Order them on one stream or by events.
 *  - The first call on each device looks up the scratch address (a host-side query, no
 *    allocation); make that first call before any stream capture on that device. */
int la_gdn_prefill_varlen_noalloc(const uint64_t *h_state_ptrs, const void *q, const void *k,
                                  const void *v, const float *g, const float *beta, void *out,
                                  const int32_t *cu_seqlens, int B, int total_tokens,
                                  int max_seqlen, int max_tokens, int Hk, int Hv, int dk, int dv,
                                  int64_t q_stride, int64_t k_stride, int64_t v_stride,
                                  float scale, uint64_t stream);

/* KDA (per-channel gate) over one stream (cu_seqlens == NULL: tokens 0..total_tokens-1, B = 1)
 * or B varlen streams. "glm5next_kda/prefill.rs", Glm5NextKdaLayer::prefill_with_pad_fill.
 * gate [total_tokens][Hv][dk] fp32 log-decay per k-channel.
 * pad_fill: the value the kernels place in the q/k tile rows at or past a stream's end before
 *   masking them (the pages fill the padded q/k/v tails with it). Outputs and states do not
 *   depend on it: positions past the end are removed in-kernel by select, never by a zero
 *   multiply, so NaN works too. Tiles that a kernel contracts over tokens keep zeros there.
 * Count rule: 1 <= total_tokens <= max_tokens. */
int la_kda_prefill(const uint64_t *h_state_ptrs, const void *q, const void *k, const void *v,
                   const float *gate, const float *beta, void *out, const int32_t *cu_seqlens,
                   int B, int total_tokens, int max_seqlen, int max_tokens, int Hk, int Hv,
                   int dk, int dv, int64_t q_stride, int64_t k_stride, int64_t v_stride,
                   float scale, float pad_fill, int dtype, void *workspace,
                   size_t workspace_bytes, uint64_t stream);

/* The whole prefill of one GDN or KDA layer in one call: causal depthwise conv1d + SiLU over
 * the carried conv state, L2 norm of every q and k head row, then the chunked recurrence, with
 * the conv output kept on chip (it never reaches HBM). Results are those of
 * la_conv1d_silu_l2_prefill followed by la_gdn_prefill_batched / la_gdn_prefill_varlen /
 * la_kda_prefill on the same inputs (bit for bit: the same arithmetic in the same order).
 * "glm5next_kda/prefill.rs", Glm5NextKdaLayer::prefill_with_pad_fill (conv_prefill, l2,
 * chunk_prepare and chunk_scan launches); "split_prefill.rs", prefill_phase1_conv1d_one,
 * prefill_phase1_l2_batched and prefill_gdn_full_batched(_fla_varlen).
 *
 * conv_state_ptrs DEVICE array of B device pointers (each 16-byte aligned); pointer s -> conv
 *               state of stream s, [conv_kernel - 1][cd] in x's dtype, oldest row first; read
 *               and advanced in place. May be NULL when conv_kernel == 1.
 * h_state_ptrs  as for the recurrence calls ([Hv][dk][dv] fp32 per stream, in place).
 * x             [total_tokens][x_stride] pre-conv rows, cd = 2*Hk*dk + Hv*dv channels packed
 *               [q heads | k heads | v heads]; 16-byte aligned, x_stride a multiple of 16 bytes.
 * conv_w        [cd][conv_kernel] (x's dtype), tap conv_kernel-1 multiplies the current token.
 * conv_bias     [cd] (x's dtype) or NULL.
 * g, beta       GDN (kda == 0): g [total_tokens][Hv]; KDA (kda == 1): g [total_tokens][Hv][dk];
 *               beta [total_tokens][Hv]; fp32.
 * out           [total_tokens][Hv][dv] (x's dtype, contiguous).
 * cu_seqlens    DEVICE int32 [B + 1], or NULL for B streams of total_tokens / B tokens each
 *               (total_tokens must then be a multiple of B).
 * l2_eps        x / sqrt(sum x^2 + l2_eps) per q/k head row.
 * pad_fill      KDA: value of the q/k tile rows past a stream's end before masking (as
 *               la_kda_prefill); results do not depend on it. GDN ignores it (zeros there).
 * z, norm_w, norm_eps  optional gated RMSNorm in the output store ("split_prefill.rs",
 *               prefill_phase3: the gated RMSNorm of the GDN output with Z): z NULL -> out = o;
 *               else z [total_tokens][Hv][dv] and norm_w [dv] (x's dtype, 16-byte aligned) and
 *               out = o / sqrt(mean(o^2) + norm_eps) * norm_w * SiLU(z) per (token, v-head) row,
 *               computed from o as stored (bf16), bit for bit as la_gated_rmsnorm on that o.
 * workspace     at least la_prefill_workspace_bytes(B, total_tokens, Hk, Hv, dk, dv, dtype).
 * Covers bf16 activations with dk = dv = 128 (the tensor-core kernel) and conv_kernel 1..4;
 * anything else is LA_ERR_UNSUPPORTED (use the separate calls). Count rule:
 * 1 <= total_tokens <= max_tokens. A zero-length stream leaves both of its states unchanged. */
int la_prefill_front(const uint64_t *conv_state_ptrs, const uint64_t *h_state_ptrs,
                     const void *x, const void *conv_w, const void *conv_bias, int conv_kernel,
                     const float *g, const float *beta, void *out, const int32_t *cu_seqlens,
                     int B, int total_tokens, int max_seqlen, int max_tokens, int Hk, int Hv,
                     int dk, int dv, int64_t x_stride, float l2_eps, float scale, float pad_fill,
                     const void *z, const void *norm_w, float norm_eps, int kda, int dtype,
                     void *workspace, size_t workspace_bytes, uint64_t stream);

/* Gated RMSNorm of a recurrence output, per (token, v-head) row of dv channels:
 *   y = o / sqrt(mean(o^2) + eps) * w * SiLU(z),   SiLU(z) = z / (1 + e^-z).
 * "split_prefill.rs", LayerSplitPrefill::prefill_phase3 (the gated RMSNorm of the GDN output
 * with Z that starts phase 3); the pages name the step only, this is its plain reading.
 * o, z, y [t][Hv][dv] contiguous (dtype; y may equal o), w [dv] (dtype); 16-byte aligned.
 * dv in {64, 128}. Count rule: t >= 1. */
int la_gated_rmsnorm(const void *o, const void *z, const void *w, void *y, int t, int Hv, int dv,
                     float eps, int dtype, uint64_t stream);

/* ------------------------------------------------------------------------------------------
 * Decode step: one new token for each of B streams, on the carried conv and h states (the step
 * that follows a prefill). "glm5next_kda/prefill.rs", Glm5NextKdaLayer::prefill_with_pad_fill:
 * the layer's decode_k shares the prefill's front-end and recurrence buckets, i.e. it is the same
 * layer applied to one token per stream: conv1d + SiLU over the conv state (which shifts by one
 * row), L2 of each q and k head, then one step of the recurrence on H = S^T.
 *
 * x             [B][x_stride] (dtype): row s is stream s's new token, cd = 2*Hk*dk + Hv*dv
 *               channels packed [q heads | k heads | v heads].
 * conv_state_ptrs, h_state_ptrs  as for la_prefill_front (one conv and one h state per stream,
 *               updated in place); each h state 16-byte aligned.
 * conv_w, conv_bias, conv_kernel, l2_eps, scale  as for la_prefill_front.
 * g, beta       GDN (kda == 0): g [B][Hv]; KDA (kda == 1): g [B][Hv][dk]; beta [B][Hv]; fp32.
 * out           [B][Hv][dv] (dtype, contiguous).
 * workspace     at least la_decode_workspace_bytes(...) bytes (holds the conv output).
 * dtype LA_F32 or LA_BF16; dk = dv in {64, 128}; conv_kernel 1..4. Two launches (front end,
 * recurrence), CUDA cores, fp32 arithmetic. Count rule: 1 <= B <= max_streams. */
size_t la_decode_workspace_bytes(int B, int Hk, int Hv, int dk, int dv, int dtype);
int la_decode_step(const uint64_t *conv_state_ptrs, const uint64_t *h_state_ptrs,
                   const void *x, const void *conv_w, const void *conv_bias, int conv_kernel,
                   const float *g, const float *beta, void *out, int B, int max_streams, int Hk,
                   int Hv, int dk, int dv, int64_t x_stride, float l2_eps, float scale, int kda,
                   int dtype, void *workspace, size_t workspace_bytes, uint64_t stream);

/* Phase-1 projection GEMM: C[M][N] = A[M][K] W[N][K]^T. "split_prefill.rs",
 * LayerSplitPrefill::prefill_phase1_proj_batched (the QKVZ and gate projections of all stacked
 * tokens of a batched prefill, on the normalised hidden rows).
 * a, w, c       bf16, row-major with row strides lda, ldw, ldc (elements, multiples of 8, at
 *               least K, K, N); 16-byte aligned; c may not overlap a or w. w is a linear layer's
 *               weight in its [out][in] layout.
 * Tensor cores (tcgen05, TMA), fp32 accumulation, the output rounded to bf16 once.
 * Count rule: M, N, K >= 1. */
int la_gemm_bf16(const void *a, const void *w, void *c, int M, int N, int K, int64_t lda,
                 int64_t ldw, int64_t ldc, uint64_t stream);

/* The norm of phase 1: y = x / sqrt(mean(x^2) + eps) * w per row of `width` channels (bf16).
 * "split_prefill.rs", prefill_phase1_proj_batched ("projections (norm, QKVZ, gates)"): the
 * norm of the hidden rows that the projection GEMM reads. x [rows][ldx], y [rows][ldy] (may be
 * x), w [width]; 16-byte aligned; width a multiple of 8 up to 8192; strides multiples of 8.
 * Count rule: rows >= 1. */
int la_rmsnorm_rows(const void *x, const void *w, void *y, int rows, int width, int64_t ldx,
                    int64_t ldy, float eps, uint64_t stream);

/* The gates of phase 1 from the gate projection rows ab [t][ld] (bf16, columns a | b):
 * g = -softplus(a) [t][na] and beta = sigmoid(b) [t][nb], fp32 (na = Hv for GDN, Hv*dk for KDA;
 * nb = Hv). "split_prefill.rs", prefill_phase1_proj_batched ("gates"). Count rule: t >= 1. */
int la_gate_activations(const void *ab, int64_t ld, int t, int na, int nb, float *g,
                        float *beta, uint64_t stream);

/* Chunk-parallel prefill of ONE long stream: the recurrence (GDN, kda == 0, or KDA, kda == 1;
 * q, k, v, g, beta, out as for la_gdn_prefill_varlen / la_kda_prefill with B = 1) with the
 * stream cut into `segments` pieces (at multiples of 64 tokens, at most 8) that run side by
 * side on the tensor cores and are then joined through each piece's state transition
 * (H_end = M H_0 + N; o_t = o_t(0) + H_0^T p_t). Not on the pages (their chunk_scan walks a
 * head's chunks in one block): it is for calls with too few (stream, v-head) units to fill the
 * GPU. Worth it while Hv * (2 * segments - 1) stays within the SM count. segments = 1 is the
 * plain call. Covers bf16 with dk = dv = 128 (else LA_ERR_UNSUPPORTED).
 * workspace  at least la_prefill_segmented_workspace_bytes(total_tokens, Hv, segments) bytes.
 * Count rule: 1 <= total_tokens <= max_tokens. */
size_t la_prefill_segmented_workspace_bytes(int total_tokens, int Hv, int segments);
int la_prefill_segmented(const uint64_t *h_state_ptrs, const void *q, const void *k,
                         const void *v, const float *g, const float *beta, void *out,
                         int total_tokens, int max_tokens, int Hk, int Hv, int dk, int dv,
                         int64_t q_stride, int64_t k_stride, int64_t v_stride, float scale,
                         int kda, int segments, int dtype, void *workspace,
                         size_t workspace_bytes, uint64_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LINATTN_H */
