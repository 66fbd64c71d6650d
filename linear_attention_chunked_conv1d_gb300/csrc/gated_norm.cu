// Gated RMSNorm of the recurrence output, per (token, v-head) row of dv channels:
//   y = o / sqrt(mean(o^2) + eps) * w * SiLU(z)
//
// Page: "split_prefill.rs", LayerSplitPrefill::prefill_phase3 — phase 3 of the split prefill
// starts with the gated RMSNorm of the GDN output with Z (then the output projection, which is
// out of this library's scope). The pages name the step only; the formula above is its plain
// reading: RMS over the head's dv channels, one weight per channel shared by the heads.
//
// GB300 design: HBM-bound elementwise work with a 128-channel reduction. dv/8 lanes own one row
// (8 channels each, 16-byte bf16 accesses); the sum of squares is reduced with xor-shuffles. The
// tensor-core recurrence applies the same arithmetic, in the same order, in its output store
// when it is given z (la_prefill_front), so the fused and separate paths give identical bits.
#include "common.cuh"
#include "launch.h"

namespace la {

namespace {

constexpr int GN_THREADS = 256;

template <typename T> struct Vec8;
template <> struct Vec8<__nv_bfloat16> {
    __device__ __forceinline__ static void load(const __nv_bfloat16 *p, float *f) {
        Vec16<__nv_bfloat16>::load(p, f);
    }
    __device__ __forceinline__ static void store(__nv_bfloat16 *p, const float *f) {
        Vec16<__nv_bfloat16>::store(p, f);
    }
};
template <> struct Vec8<float> {
    __device__ __forceinline__ static void load(const float *p, float *f) {
        Vec16<float>::load(p, f);
        Vec16<float>::load(p + 4, f + 4);
    }
    __device__ __forceinline__ static void store(float *p, const float *f) {
        Vec16<float>::store(p, f);
        Vec16<float>::store(p + 4, f + 4);
    }
};

template <typename T, int HD>
__global__ void __launch_bounds__(GN_THREADS)
gated_rmsnorm_kernel(const T *__restrict__ o, const T *__restrict__ z, const T *__restrict__ w,
                     T *y, int64_t rows, float eps) {
    constexpr int LPR = HD / 8;  // lanes per row
    const int64_t r = (int64_t)blockIdx.x * (GN_THREADS / LPR) + threadIdx.x / LPR;
    const int lane = threadIdx.x % LPR;
    const bool active = r < rows;
    float ov[8], zv[8], wv[8];
    float ss = 0.f;
    if (active) {
        Vec8<T>::load(o + r * HD + lane * 8, ov);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(ov[e], ov[e], ss);
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (!active) return;
    Vec8<T>::load(z + r * HD + lane * 8, zv);
    Vec8<T>::load(w + lane * 8, wv);
    const float inv = rsqrtf(ss * (1.f / HD) + eps);
#pragma unroll
    for (int e = 0; e < 8; ++e) ov[e] = ov[e] * inv * wv[e] * silu(zv[e]);
    Vec8<T>::store(y + r * HD + lane * 8, ov);
}

template <typename T, int HD>
cudaError_t launch_gn_t(const GatedNormArgs &a, cudaStream_t st) {
    constexpr int per_block = GN_THREADS / (HD / 8);
    const int64_t rows = (int64_t)a.t * a.Hv;
    const unsigned blocks = (unsigned)((rows + per_block - 1) / per_block);
    gated_rmsnorm_kernel<T, HD><<<blocks, GN_THREADS, 0, st>>>(
        (const T *)a.o, (const T *)a.z, (const T *)a.w, (T *)a.y, rows, a.eps);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gated_rmsnorm(const GatedNormArgs &a, cudaStream_t st) {
    if (a.dtype == LA_BF16)
        return a.dv == 64 ? launch_gn_t<__nv_bfloat16, 64>(a, st) : launch_gn_t<__nv_bfloat16, 128>(a, st);
    return a.dv == 64 ? launch_gn_t<float, 64>(a, st) : launch_gn_t<float, 128>(a, st);
}

}  // namespace la
