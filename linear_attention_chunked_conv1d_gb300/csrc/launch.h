// Internal launcher interface between the C ABI (abi.cu) and the kernels. Not exported.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace la {

struct ConvArgs {
    const uint64_t *state_ptrs;  // varlen: device array of B state pointers; else nullptr
    void *single_state;          // single stream: the state
    const void *x, *w, *bias;
    void *out;
    const int32_t *cu;  // nullptr: one stream of `total` tokens
    int B, total, channels, kernel;
    int64_t x_stride, out_stride;
    int dtype;
    int l2_heads, head_dim;  // l2_heads > 0: fused L2 over the first l2_heads * head_dim channels
    float eps;
    int *status;
    bool one_per_stream;  // decode: B streams of one token, token s = row s (cu unused)
};
cudaError_t launch_conv1d_silu(const ConvArgs &a, cudaStream_t st);

struct L2Args {
    void *x;
    int t, n_heads, head_dim;
    int64_t row_stride;
    float eps;
    int dtype;
};
cudaError_t launch_l2norm_heads(const L2Args &a, cudaStream_t st);

struct RecArgs {
    const uint64_t *h_ptrs;
    const void *q, *k, *v;
    const float *g;  // GDN [tok][Hv]; KDA [tok][Hv][dk]
    const float *beta;
    void *out;
    const int32_t *cu;  // nullptr: batched, stream s = tokens s*T_each ..
    int B, T_each, total, max_seqlen;
    int Hk, Hv, dk, dv;
    int64_t q_stride, k_stride, v_stride;
    float scale, pad_fill;
    int dtype;
    bool kda;
    void *workspace;
    size_t workspace_bytes;
    int *status;
    uint64_t wait_ns;  // tensor-core kernel: limit of its bounded waits (0: the 2 s default)
    int debug_stall;   // tensor-core kernel, test knob: one wait on a barrier nothing completes
    // Fused front end (tensor-core kernel only): q, k and v are not read; each block computes
    // them per chunk from the pre-conv rows x [tok][cd] (cd = 2 Hk dk + Hv dv, packed
    // q | k | v heads), the depthwise conv weights [cd][conv_k] (+ optional bias [cd]) and
    // the carried conv states [conv_k - 1][cd] (one per stream, advanced in place).
    bool front;
    const void *x, *conv_w, *conv_bias;
    const uint64_t *conv_state_ptrs;
    int64_t x_stride;
    int conv_k;
    float l2_eps;
    // Segmented scan (tensor-core kernel, not with the fused front end): streams s >= alt_from
    // read v as zero (v_alt: one zero row, stride 0) and write their outputs to out_alt.
    // Their token ranges come from cu_alt (index s - alt_from).
    bool use_alt;
    int alt_from;
    const int32_t *cu_alt;
    const void *v_alt;
    void *out_alt;
    // Gated RMSNorm in the output store (tensor-core kernel only): when z is set, out receives
    // o / sqrt(mean(o^2) + norm_eps) * norm_w * SiLU(z) per (token, v-head) row, from the bf16 o.
    const void *z, *norm_w;
    float norm_eps;
};
// CUDA-core chunked kernel (fp32 and bf16 activations, head dims 64 and 128).
cudaError_t launch_chunk_simt(const RecArgs &a, cudaStream_t st);

// Tensor-core (tcgen05) chunked kernel: bf16 activations, dk = dv = 128. Needs a workspace of
// chunk_tc_workspace_bytes(B, Hk) bytes (stream order, unit counter and, for the fused front
// end, one conv-state reader count per (stream, k-head)); Hk = 0 sizes it without the counts.
bool chunk_tc_supported(const RecArgs &a);
size_t chunk_tc_workspace_bytes(int B, int Hk);
cudaError_t launch_chunk_tc(const RecArgs &a, cudaStream_t st);
// Library-owned scratch usable in place of a workspace by the tensor-core kernel (at most
// chunk_tc_static_scratch_max_streams() streams per call).
int chunk_tc_static_scratch_max_streams();
cudaError_t chunk_tc_static_scratch(void **ptr, size_t *bytes);

// Decode step of the recurrence: one token per stream, q|k|v rows [B][qkv_stride] (the conv
// output), states through h_ptrs, out [B][Hv][dv]. CUDA cores, fp32 arithmetic.
struct DecArgs {
    const uint64_t *h_ptrs;
    const void *qkv;
    int64_t qkv_stride;
    const float *g, *beta;  // GDN g [B][Hv]; KDA g [B][Hv][dk]; beta [B][Hv]
    void *out;
    int B, Hk, Hv, d;
    float scale;
    int dtype;
    bool kda;
};
cudaError_t launch_decode_recurrence(const DecArgs &a, cudaStream_t st);

// Gated RMSNorm y = o / sqrt(mean(o^2) + eps) * w * SiLU(z) per row of dv channels; o, z, y
// [t][Hv][dv] contiguous (y may be o), w [dv].
struct GatedNormArgs {
    const void *o, *z, *w;
    void *y;
    int t, Hv, dv;
    float eps;
    int dtype;
};
cudaError_t launch_gated_rmsnorm(const GatedNormArgs &a, cudaStream_t st);

// Projection GEMM C[M][N] = A[M][K] W[N][K]^T, bf16 in and out, fp32 accumulation (tcgen05).
struct GemmArgs {
    const void *a, *w;
    void *c;
    int M, N, K;
    int64_t lda, ldw, ldc;
    int *status;
    uint64_t wait_ns;  // limit of the kernel's bounded waits (0: the 2 s default)
    int debug_stall;   // test knob: one wait on a barrier that nothing completes
};
cudaError_t launch_gemm_bf16(const GemmArgs &a, cudaStream_t st);

// Row RMSNorm y = x / sqrt(mean(x^2) + eps) * w (bf16; width a multiple of 8, at most
// rmsnorm_rows_max_width()).
struct RowNormArgs {
    const void *x, *w;
    void *y;
    int rows, width;
    int64_t ldx, ldy;
    float eps;
};
cudaError_t launch_rmsnorm_rows(const RowNormArgs &a, cudaStream_t st);
int rmsnorm_rows_max_width();

// Gate activations: g = -softplus(a) [t][na], beta = sigmoid(b) [t][nb] (fp32) from the bf16
// gate projection rows [t][ld] holding a | b.
struct GateArgs {
    const void *ab;
    int64_t ld;
    int t, na, nb;
    float *g, *beta;
};
cudaError_t launch_gate_activations(const GateArgs &a, cudaStream_t st);

// Chunk-parallel scan of one long stream (tensor-core path): the stream's tokens cut into up to
// kMaxSegments segments run side by side, then joined (segscan.cu). `a` describes one stream
// (cu == nullptr, B == 1); its workspace must hold segmented_workspace_bytes(...).
constexpr int kMaxSegments = 8;
int segmented_plan_segments(int total, int requested);
size_t segmented_workspace_bytes(int total, int Hv, int segments);
cudaError_t launch_segmented(const RecArgs &a, int segments, cudaStream_t st);

// Encodes a 2-D tiled TMA map (a CUtensorMap, 64-byte aligned storage of 128 bytes) of a
// row-major bf16 matrix [rows][cols] with row stride ld elements, boxes of box_rows x box_cols,
// optional 128-byte swizzle; out-of-range elements of a box read as zero. False on failure.
bool make_map_bf16_2d(void *map, const void *base, int64_t rows, int64_t cols, int64_t ld,
                      uint32_t box_cols, uint32_t box_rows, bool swizzle128);

}  // namespace la
