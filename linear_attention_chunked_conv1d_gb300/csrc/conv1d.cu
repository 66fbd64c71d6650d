// Causal depthwise conv1d + SiLU with a carried conv state, single stream or varlen.
//
// Page: "glm5next_kda/prefill.rs", Glm5NextKdaLayer::prefill_with_pad_fill, conv_prefill launch
// (conv + SiLU only; the fourth pointer slot, read here as an optional bias, is NULL there);
// "split_prefill.rs", LayerSplitPrefill::prefill_phase1_conv1d_one (conv over one request's
// tokens of a batched prefill, advancing that request's conv state).
//
// GB300 design: the op is HBM-bound elementwise work, so each thread owns one 16-byte vector
// of channels (8 bf16 / 4 fp32) and a run of up to ROWS consecutive tokens of ONE stream,
// keeping the kernel-1 previous rows in registers as a sliding window: x is read once (plus
// kernel-1 halo rows per run, served by L2) and out written once, with coalesced 16-byte
// accesses. Runs are aligned to stream starts (stream s owns run slots floor(cu[s]/ROWS) + s
// onwards, found by binary search), so the first run of a stream is the only one that reads
// its conv state, and that same thread advances the state in place afterwards: no race, no
// second pass.
#include "common.cuh"
#include "launch.h"

namespace la {

constexpr int CONV_THREADS = 128;
constexpr int CONV_ROWS = 64;

// First run slot of stream s.
__device__ __forceinline__ int conv_run_base(const int32_t *cu, int s) {
    return cu[s] / CONV_ROWS + s;
}

template <typename T, int K>
__global__ void __launch_bounds__(CONV_THREADS)
conv1d_silu_kernel(const uint64_t *__restrict__ state_ptrs, T *single_state,
                   const T *__restrict__ x, const T *__restrict__ w,
                   const T *__restrict__ bias, T *__restrict__ out,
                   const int32_t *__restrict__ cu, int B, int total, int C, int64_t xs,
                   int64_t os, int *status) {
    using V = Vec16<T>;
    constexpr int N = V::N;
    const int cv = blockIdx.y * CONV_THREADS + threadIdx.x;
    const int c0 = cv * N;
    if (c0 >= C) return;

    // Which stream and which run of it this block covers.
    int s = 0, sb = 0, se = total, run = blockIdx.x;
    if (cu) {
        if (cu[0] != 0 || cu[B] != total) {
            raise_status(status, LA_DEV_BAD_SEQLENS);
            return;
        }
        const int y = blockIdx.x;
        int lo = 0, hi = B - 1;  // last s with base(s) <= y
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (conv_run_base(cu, mid) <= y) lo = mid; else hi = mid - 1;
        }
        s = lo;
        sb = cu[s];
        se = cu[s + 1];
        if (se < sb || se > total) {
            raise_status(status, LA_DEV_BAD_SEQLENS);
            return;
        }
        run = y - conv_run_base(cu, s);
    }
    const int r0 = sb + run * CONV_ROWS;
    if (run < 0 || r0 >= se) return;  // slot past this stream's runs
    const int r1 = min(r0 + CONV_ROWS, se);

    float wr[N][K];
#pragma unroll
    for (int e = 0; e < N; ++e)
#pragma unroll
        for (int j = 0; j < K; ++j) wr[e][j] = to_f(w[(int64_t)(c0 + e) * K + j]);
    float br[N];
    if (bias) {
        V::load(bias + c0, br);
    } else {
#pragma unroll
        for (int e = 0; e < N; ++e) br[e] = 0.f;
    }

    // win[m] = row (tau - (K-1) + m) of xh = [state ; x] for the current tau.
    float win[K > 1 ? K - 1 : 1][N];
    if constexpr (K > 1) {
        if (run == 0) {
            // Only reader of this stream's state: read it, fill the window, then advance it.
            T *st = state_ptrs ? reinterpret_cast<T *>(state_ptrs[s]) : single_state;
            float old[K - 1][N];
#pragma unroll
            for (int m = 0; m < K - 1; ++m) V::load(st + (int64_t)m * C + c0, old[m]);
#pragma unroll
            for (int m = 0; m < K - 1; ++m)
#pragma unroll
                for (int e = 0; e < N; ++e) win[m][e] = old[m][e];
            const int len = se - sb;
#pragma unroll
            for (int m = 0; m < K - 1; ++m) {
                const int idx = len + m;  // row of xh
                float nv[N];
                if (idx >= K - 1) {
                    V::load(x + (int64_t)(sb + idx - (K - 1)) * xs + c0, nv);
                } else {
                    // idx is a runtime value: select among the registers, no local memory
#pragma unroll
                    for (int mm = 0; mm < K - 1; ++mm)
                        if (mm == idx)
#pragma unroll
                            for (int e = 0; e < N; ++e) nv[e] = old[mm][e];
                }
                V::store(st + (int64_t)m * C + c0, nv);
            }
        } else {
#pragma unroll
            for (int m = 0; m < K - 1; ++m)
                V::load(x + (int64_t)(r0 - (K - 1) + m) * xs + c0, win[m]);
        }
    }

    for (int tau = r0; tau < r1; ++tau) {
        float cur[N];
        V::load(x + (int64_t)tau * xs + c0, cur);
        float y[N];
#pragma unroll
        for (int e = 0; e < N; ++e) {
            float acc = br[e];
#pragma unroll
            for (int m = 0; m < K - 1; ++m) acc = fmaf(wr[e][m], win[m][e], acc);
            acc = fmaf(wr[e][K - 1], cur[e], acc);
            y[e] = acc / (1.f + expf(-acc));
        }
        V::store(out + (int64_t)tau * os + c0, y);
        if constexpr (K > 1) {
#pragma unroll
            for (int m = 0; m < K - 2; ++m)
#pragma unroll
                for (int e = 0; e < N; ++e) win[m][e] = win[m + 1][e];
#pragma unroll
            for (int e = 0; e < N; ++e) win[K - 2][e] = cur[e];
        }
    }
}

template <typename T, int K>
static cudaError_t launch_conv_t(const ConvArgs &a, cudaStream_t st) {
    constexpr int N = Vec16<T>::N;
    int nvec = a.channels / N;
    // Run slots: single stream ceil(total/ROWS); varlen floor(total/ROWS) + B covers every
    // stream's runs (stream s starts at slot floor(cu[s]/ROWS) + s).
    int slots = a.cu ? a.total / CONV_ROWS + a.B : (a.total + CONV_ROWS - 1) / CONV_ROWS;
    dim3 grid(slots, (nvec + CONV_THREADS - 1) / CONV_THREADS);
    conv1d_silu_kernel<T, K><<<grid, CONV_THREADS, 0, st>>>(
        a.state_ptrs, (T *)a.single_state, (const T *)a.x, (const T *)a.w, (const T *)a.bias,
        (T *)a.out, a.cu, a.B, a.total, a.channels, a.x_stride, a.out_stride, a.status);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_conv_k(const ConvArgs &a, cudaStream_t st) {
    switch (a.kernel) {
        case 1: return launch_conv_t<T, 1>(a, st);
        case 2: return launch_conv_t<T, 2>(a, st);
        case 3: return launch_conv_t<T, 3>(a, st);
        case 4: return launch_conv_t<T, 4>(a, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_conv1d_silu(const ConvArgs &a, cudaStream_t st) {
    return a.dtype == LA_BF16 ? launch_conv_k<__nv_bfloat16>(a, st) : launch_conv_k<float>(a, st);
}

}  // namespace la
