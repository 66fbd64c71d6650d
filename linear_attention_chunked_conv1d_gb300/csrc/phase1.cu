// Phase-1 elementwise steps around the projection GEMM: the row RMSNorm of the hidden rows
// before it, and the gate activations after it.
//
// Page: "split_prefill.rs", LayerSplitPrefill::prefill_phase1_proj_batched — "projections
// (norm, QKVZ, gates) over all stacked tokens". The pages name the steps only; read plainly:
//   norm:  y = x / sqrt(mean(x^2) + eps) * w per hidden row;
//   gates: g = -softplus(a) (the log-decay, one per v-head for GDN or per (v-head, k-channel)
//          for KDA) and beta = sigmoid(b), from the gate projections a and b.
//
// GB300 design: both are HBM-bound elementwise passes. The norm takes one 256-thread block per
// row (16-byte accesses, up to 4 per thread kept in registers between the reduction and the
// scaling; warp shuffles then one shared-memory step); the gates take one thread per output.
#include "common.cuh"
#include "launch.h"

namespace la {

namespace {

constexpr int RN_THREADS = 256;
constexpr int RN_MAX_PER_THREAD = 4;  // 16-byte pieces: widths up to 256 x 8 x 4 = 8192

__global__ void __launch_bounds__(RN_THREADS)
rmsnorm_rows_kernel(const __nv_bfloat16 *__restrict__ x, const __nv_bfloat16 *__restrict__ w,
                    __nv_bfloat16 *__restrict__ y, int width, int64_t ldx, int64_t ldy,
                    float eps) {
    __shared__ float part[RN_THREADS / 32];
    const int64_t r = blockIdx.x;
    const int t = threadIdx.x;
    const int pieces = width / 8;
    float v[RN_MAX_PER_THREAD][8];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < RN_MAX_PER_THREAD; ++i) {
        const int p = t + RN_THREADS * i;
        if (p < pieces) {
            Vec16<__nv_bfloat16>::load(x + r * ldx + p * 8, v[i]);
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = fmaf(v[i][e], v[i][e], ss);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((t & 31) == 0) part[t >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < RN_THREADS / 32; ++i) tot += part[i];
    const float inv = rsqrtf(tot / width + eps);
#pragma unroll
    for (int i = 0; i < RN_MAX_PER_THREAD; ++i) {
        const int p = t + RN_THREADS * i;
        if (p < pieces) {
            float wv[8];
            Vec16<__nv_bfloat16>::load(w + p * 8, wv);
#pragma unroll
            for (int e = 0; e < 8; ++e) v[i][e] = v[i][e] * inv * wv[e];
            Vec16<__nv_bfloat16>::store(y + r * ldy + p * 8, v[i]);
        }
    }
}

// a [t][na] and b [t][nb] are column ranges of the gate projection rows (row stride ld).
__global__ void gate_act_kernel(const __nv_bfloat16 *__restrict__ ab, int64_t ld, int t, int na,
                                int nb, float *__restrict__ g, float *__restrict__ beta) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t n = (int64_t)t * (na + nb);
    if (i >= n) return;
    const int64_t row = i / (na + nb);
    const int col = (int)(i % (na + nb));
    const float v = __bfloat162float(ab[row * ld + col]);
    if (col < na) {
        // -softplus(v) = -(max(v, 0) + log1p(e^-|v|)), without overflow
        g[row * na + col] = -(fmaxf(v, 0.f) + log1pf(expf(-fabsf(v))));
    } else {
        beta[row * nb + col - na] = 1.f / (1.f + expf(-v));
    }
}

}  // namespace

cudaError_t launch_rmsnorm_rows(const RowNormArgs &a, cudaStream_t st) {
    rmsnorm_rows_kernel<<<a.rows, RN_THREADS, 0, st>>>(
        (const __nv_bfloat16 *)a.x, (const __nv_bfloat16 *)a.w, (__nv_bfloat16 *)a.y, a.width,
        a.ldx, a.ldy, a.eps);
    return cudaGetLastError();
}

cudaError_t launch_gate_activations(const GateArgs &a, cudaStream_t st) {
    const int64_t n = (int64_t)a.t * (a.na + a.nb);
    const unsigned blocks = (unsigned)((n + 255) / 256);
    gate_act_kernel<<<blocks, 256, 0, st>>>((const __nv_bfloat16 *)a.ab, a.ld, a.t, a.na, a.nb,
                                            a.g, a.beta);
    return cudaGetLastError();
}

int rmsnorm_rows_max_width() { return RN_THREADS * 8 * RN_MAX_PER_THREAD; }

}  // namespace la
