// Per-(token, head) L2 norm in place over the q|k heads of the conv output.
//
// Page: "glm5next_kda/prefill.rs", Glm5NextKdaLayer::prefill_with_pad_fill, l2 launch (grid
// q|k heads x tokens, one head_dim vector per block there, eps = cfg.l2_eps, row stride = conv
// dim); "split_prefill.rs", LayerSplitPrefill::prefill_phase1_l2_batched.
//
// GB300 design: HBM-bound. A group of head_dim/4 lanes (32 lanes for d = 128) owns one
// (token, head) vector, each lane 4 channels; the sum of squares is reduced with xor-shuffles
// inside the group (the same order as the fused conv + L2 kernel, which gives identical bits),
// with coalesced reads and writes and no shared memory.
#include "common.cuh"
#include "launch.h"

namespace la {

constexpr int L2_THREADS = 256;

template <typename T, int HD>
__global__ void __launch_bounds__(L2_THREADS)
l2norm_heads_kernel(T *__restrict__ x, int t, int n_heads, int64_t rs, float eps) {
    using V = Vec4<T>;
    constexpr int N = V::N;
    constexpr int LPH = HD / N;  // lanes per head vector (power of two, <= 32)
    static_assert(LPH >= 1 && LPH <= 32 && (LPH & (LPH - 1)) == 0, "lanes per head");
    const int64_t gid = (int64_t)blockIdx.x * (L2_THREADS / LPH) + threadIdx.x / LPH;
    const int lane = threadIdx.x % LPH;
    const bool active = gid < (int64_t)t * n_heads;
    const int64_t tok = active ? gid / n_heads : 0;
    const int h = active ? (int)(gid % n_heads) : 0;
    T *p = x + tok * rs + (int64_t)h * HD + lane * N;
    float f[N];
    float ss = 0.f;
    if (active) {
        V::load(p, f);
#pragma unroll
        for (int e = 0; e < N; ++e) ss = fmaf(f[e], f[e], ss);
    }
#pragma unroll
    for (int off = LPH / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (!active) return;
    const float inv = rsqrtf(ss + eps);
#pragma unroll
    for (int e = 0; e < N; ++e) f[e] *= inv;
    V::store(p, f);
}

template <typename T, int HD>
static cudaError_t launch_l2_t(const L2Args &a, cudaStream_t st) {
    constexpr int LPH = HD / Vec4<T>::N;
    constexpr int per_block = L2_THREADS / LPH;
    int64_t groups = (int64_t)a.t * a.n_heads;
    unsigned blocks = (unsigned)((groups + per_block - 1) / per_block);
    l2norm_heads_kernel<T, HD><<<blocks, L2_THREADS, 0, st>>>((T *)a.x, a.t, a.n_heads,
                                                              a.row_stride, a.eps);
    return cudaGetLastError();
}

cudaError_t launch_l2norm_heads(const L2Args &a, cudaStream_t st) {
    if (a.dtype == LA_BF16) {
        return a.head_dim == 64 ? launch_l2_t<__nv_bfloat16, 64>(a, st)
                                : launch_l2_t<__nv_bfloat16, 128>(a, st);
    }
    return a.head_dim == 64 ? launch_l2_t<float, 64>(a, st) : launch_l2_t<float, 128>(a, st);
}

}  // namespace la
