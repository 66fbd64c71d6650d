// Causal depthwise conv1d + SiLU with a carried conv state, single stream or varlen, optionally
// fused with the per-head L2 norm of the q|k channels.
//
// Page: "glm5next_kda/prefill.rs", Glm5NextKdaLayer::prefill_with_pad_fill, conv_prefill launch
// (conv + SiLU only; the fourth pointer slot, read here as an optional bias, is NULL there);
// "split_prefill.rs", LayerSplitPrefill::prefill_phase1_conv1d_one (conv over one request's
// tokens of a batched prefill, advancing that request's conv state).
//
// GB300 design: the op is HBM-bound elementwise work, so each thread owns 4 channels (an 8-byte
// bf16 / 16-byte fp32 vector) and a run of up to ROWS (64, 128 or 256: conv_rows) consecutive
// tokens of ONE stream, keeping the kernel-1 previous rows in registers as a sliding window:
// x is read once (plus kernel-1 halo rows per run, served by L2) and out written once, with
// coalesced 16-byte accesses. Runs are aligned to stream starts (stream s owns run slots floor(cu[s]/ROWS) + s
// onwards, found by binary search), so the first run of a stream is the only one that reads
// its conv state, and that same thread advances the state in place afterwards: no race, no
// second pass.
#include "common.cuh"
#include "launch.h"

namespace la {

constexpr int CONV_THREADS = 128;
constexpr int CONV_ROWS = 64;  // the shortest run; a launch takes 64, 128 or 256 (conv_rows)
constexpr int CONV_G_BF16 = 8;  // bf16 rows in flight per thread

// First run slot of stream s (runs of `rows` tokens).
__device__ __forceinline__ int conv_run_base(const int32_t *cu, int s, int rows) {
    return cu[s] / rows + s;
}

// One output row of a thread's 4 channels: y = SiLU(b + sum_m w_m xh_m) over the K-1 window
// rows and the current row, then (HD > 0, in a warp that holds normalised channels) rounded to
// T and scaled by 1/sqrt(sum of squares of the head + eps). Every lane of the warp calls it.
template <typename T, int K, int HD>
__device__ __forceinline__ void conv_row(const uint64_t (&wp)[K][2], const uint64_t (&bp)[2],
                                         const float (&win)[K > 1 ? K - 1 : 1][4],
                                         const float (&cur)[4], bool l2_warp, bool do_l2,
                                         float eps, float (&y)[4]) {
    constexpr int LPH = HD > 0 ? HD / 4 : 1;  // lanes per head
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint64_t acc = bp[h];
#pragma unroll
        for (int m = 0; m < K - 1; ++m)
            acc = fma2(wp[m][h], pk2(win[m][2 * h], win[m][2 * h + 1]), acc);
        acc = fma2(wp[K - 1][h], pk2(cur[2 * h], cur[2 * h + 1]), acc);
        upk2(silu2(acc), y[2 * h], y[2 * h + 1]);
    }
    if (HD > 0 && l2_warp) {
        // round to the stored type, then the same reduction as the l2 launch
        round_to_2<T>(y[0], y[1]);
        round_to_2<T>(y[2], y[3]);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) ss = fmaf(y[e], y[e], ss);
#pragma unroll
        for (int off = LPH / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (do_l2) {
            const float inv = rsqrtf(ss + eps);
#pragma unroll
            for (int e = 0; e < 4; ++e) y[e] *= inv;
        }
    }
}

// Taps and bias of a thread's 4 channels as packed pairs (e0, e1), (e2, e3).
template <typename T, int K>
__device__ __forceinline__ void load_taps(const T *w, const T *bias, int c0, bool active,
                                          uint64_t (&wp)[K][2], uint64_t (&bp)[2]) {
    float wr[4][K], br[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int j = 0; j < K; ++j) wr[e][j] = active ? to_f(w[(int64_t)(c0 + e) * K + j]) : 0.f;
    if (bias && active) Vec4<T>::load(bias + c0, br);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        bp[h] = pk2(br[2 * h], br[2 * h + 1]);
#pragma unroll
        for (int m = 0; m < K; ++m) wp[m][h] = pk2(wr[2 * h][m], wr[2 * h + 1][m]);
    }
}

// HD > 0: also L2-normalise, per (token, head), the first n_l2 channels (whole heads of HD
// channels). The conv output is rounded to T first, exactly as the separate l2 launch would
// read it back, and the sum of squares is reduced in the same order as that launch, so the
// fused and the two-launch paths give identical bits.
template <typename T, int K, int HD>
__global__ void __launch_bounds__(CONV_THREADS, 8)
conv1d_silu_kernel(const uint64_t *__restrict__ state_ptrs, T *single_state,
                   const T *__restrict__ x, const T *__restrict__ w,
                   const T *__restrict__ bias, T *__restrict__ out,
                   const int32_t *__restrict__ cu, int B, int total, int C, int64_t xs,
                   int64_t os, int n_l2, float eps, int rows, int *status) {
    using V = Vec4<T>;
    constexpr int N = V::N;
    const int cv = blockIdx.y * CONV_THREADS + threadIdx.x;
    const int c0 = cv * N;
    const bool active = c0 < C;  // inactive lanes still take part in the head reductions
    const bool do_l2 = HD > 0 && c0 < n_l2;

    // Which stream and which run of it this block covers.
    int s = 0, sb = 0, se = total, run = blockIdx.x;
    if (cu) {
        if (cu[0] != 0 || cu[B] != total) {
            if (threadIdx.x == 0) raise_status(status, LA_DEV_BAD_SEQLENS);
            return;
        }
        const int y = blockIdx.x;
        int lo = 0, hi = B - 1;  // last s with base(s) <= y
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (conv_run_base(cu, mid, rows) <= y) lo = mid; else hi = mid - 1;
        }
        s = lo;
        sb = cu[s];
        se = cu[s + 1];
        if (se < sb || se > total) {
            if (threadIdx.x == 0) raise_status(status, LA_DEV_BAD_SEQLENS);
            return;
        }
        run = y - conv_run_base(cu, s, rows);
    }
    const int r0 = sb + run * rows;
    if (run < 0 || r0 >= se) return;  // slot past this stream's runs (uniform per block)
    const int r1 = min(r0 + rows, se);

    uint64_t wp[K][2], bp[2];
    load_taps<T, K>(w, bias, c0, active, wp, bp);

    // win[m] = row (tau - (K-1) + m) of xh = [state ; x] for the current tau.
    float win[K > 1 ? K - 1 : 1][N];
#pragma unroll
    for (int m = 0; m < (K > 1 ? K - 1 : 1); ++m)
#pragma unroll
        for (int e = 0; e < N; ++e) win[m][e] = 0.f;
    if constexpr (K > 1) {
        if (active && run == 0) {
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
        } else if (active) {
#pragma unroll
            for (int m = 0; m < K - 1; ++m)
                V::load(x + (int64_t)(r0 - (K - 1) + m) * xs + c0, win[m]);
        }
    }

    // warps whose channels all lie past the normalised heads (v) skip the L2 work entirely
    const bool l2_warp = HD > 0 && __any_sync(0xffffffffu, do_l2);

    const T *xp = x + (int64_t)r0 * xs + c0;
    T *op = out + (int64_t)r0 * os + c0;
    // rows in groups of G: the G loads are issued before any of them is used, and held as
    // loaded (bf16: two registers a row) until their row is computed, so that more rows are in
    // flight within the 64 registers that 8 blocks of 128 threads per SM allow
    constexpr int G = sizeof(T) == 2 ? CONV_G_BF16 : 6;
    for (int g0 = r0; g0 < r1; g0 += G, xp += G * xs, op += G * os) {
        typename V::Raw raw[G];
#pragma unroll
        for (int q = 0; q < G; ++q)
            raw[q] = (active && g0 + q < r1) ? V::load_raw(xp + q * xs) : V::zero_raw();
#pragma unroll
        for (int q = 0; q < G; ++q) {
            float cur[N];
            V::widen(raw[q], cur);
            float y[N];
            conv_row<T, K, HD>(wp, bp, win, cur, l2_warp, do_l2, eps, y);
            if (active && g0 + q < r1) V::store(op + q * os, y);
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
}

// One new token per stream (decode): row s of x is the token of stream s. A block takes
// STEP_STREAMS streams for its 128 x 4 channels, so the taps are read once per 8 streams; each
// stream's state is read, the row computed by the same conv_row as above, and the state
// advanced by that one row.
constexpr int STEP_STREAMS = 8;

template <typename T, int K, int HD>
__global__ void __launch_bounds__(CONV_THREADS)
conv1d_silu_step_kernel(const uint64_t *__restrict__ state_ptrs, const T *__restrict__ x,
                        const T *__restrict__ w, const T *__restrict__ bias, T *__restrict__ out,
                        int B, int C, int64_t xs, int64_t os, int n_l2, float eps) {
    using V = Vec4<T>;
    const int c0 = (blockIdx.y * CONV_THREADS + threadIdx.x) * 4;
    const bool active = c0 < C;
    const bool do_l2 = HD > 0 && c0 < n_l2;
    const bool l2_warp = HD > 0 && __any_sync(0xffffffffu, do_l2);
    uint64_t wp[K][2], bp[2];
    load_taps<T, K>(w, bias, c0, active, wp, bp);
    const int s_end = min(B, (int)(blockIdx.x + 1) * STEP_STREAMS);
    for (int s = blockIdx.x * STEP_STREAMS; s < s_end; ++s) {  // uniform over the block
        float win[K > 1 ? K - 1 : 1][4] = {};
        float cur[4] = {0.f, 0.f, 0.f, 0.f};
        T *st = K > 1 ? reinterpret_cast<T *>(state_ptrs[s]) : nullptr;
        if (active) {
            if constexpr (K > 1) {
#pragma unroll
                for (int m = 0; m < K - 1; ++m) V::load(st + (int64_t)m * C + c0, win[m]);
            }
            V::load(x + (int64_t)s * xs + c0, cur);
        }
        float y[4];
        conv_row<T, K, HD>(wp, bp, win, cur, l2_warp, do_l2, eps, y);
        if (active) {
            V::store(out + (int64_t)s * os + c0, y);
            if constexpr (K > 1) {
#pragma unroll
                for (int m = 0; m < K - 2; ++m) V::store(st + (int64_t)m * C + c0, win[m + 1]);
                V::store(st + (int64_t)(K - 2) * C + c0, cur);
            }
        }
    }
}

// Rows per run: longer runs read fewer halo rows and repeat less per-block setup, but make
// fewer blocks. Take the longest of 256, 128 and 64 that still gives six waves of the resident
// blocks (8 per SM); the small workloads keep 64.
static int conv_rows(const ConvArgs &a, int col_blocks) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
    const int64_t target = 6LL * 8 * sms;
    for (int rows = 4 * CONV_ROWS; rows > CONV_ROWS; rows >>= 1) {
        const int64_t slots = a.cu ? a.total / rows + a.B : (a.total + rows - 1) / rows;
        if (slots * col_blocks >= target) return rows;
    }
    return CONV_ROWS;
}

template <typename T, int K, int HD>
static cudaError_t launch_conv_t(const ConvArgs &a, cudaStream_t st) {
    if (a.one_per_stream) {
        const int nvec = a.channels / 4;
        dim3 grid((a.B + STEP_STREAMS - 1) / STEP_STREAMS, (nvec + CONV_THREADS - 1) / CONV_THREADS);
        conv1d_silu_step_kernel<T, K, HD><<<grid, CONV_THREADS, 0, st>>>(
            a.state_ptrs, (const T *)a.x, (const T *)a.w, (const T *)a.bias, (T *)a.out, a.B,
            a.channels, a.x_stride, a.out_stride, a.l2_heads * a.head_dim, a.eps);
        return cudaGetLastError();
    }
    constexpr int N = Vec4<T>::N;
    int nvec = a.channels / N;
    // Run slots: single stream ceil(total/rows); varlen floor(total/rows) + B covers every
    // stream's runs (stream s starts at slot floor(cu[s]/rows) + s).
    const int col_blocks = (nvec + CONV_THREADS - 1) / CONV_THREADS;
    const int rows = conv_rows(a, col_blocks);
    int slots = a.cu ? a.total / rows + a.B : (a.total + rows - 1) / rows;
    dim3 grid(slots, col_blocks);
    conv1d_silu_kernel<T, K, HD><<<grid, CONV_THREADS, 0, st>>>(
        a.state_ptrs, (T *)a.single_state, (const T *)a.x, (const T *)a.w, (const T *)a.bias,
        (T *)a.out, a.cu, a.B, a.total, a.channels, a.x_stride, a.out_stride,
        a.l2_heads * a.head_dim, a.eps, rows, a.status);
    return cudaGetLastError();
}

template <typename T, int HD>
static cudaError_t launch_conv_k(const ConvArgs &a, cudaStream_t st) {
    switch (a.kernel) {
        case 1: return launch_conv_t<T, 1, HD>(a, st);
        case 2: return launch_conv_t<T, 2, HD>(a, st);
        case 3: return launch_conv_t<T, 3, HD>(a, st);
        case 4: return launch_conv_t<T, 4, HD>(a, st);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
static cudaError_t launch_conv_h(const ConvArgs &a, cudaStream_t st) {
    if (a.l2_heads <= 0) return launch_conv_k<T, 0>(a, st);
    return a.head_dim == 64 ? launch_conv_k<T, 64>(a, st) : launch_conv_k<T, 128>(a, st);
}

cudaError_t launch_conv1d_silu(const ConvArgs &a, cudaStream_t st) {
    return a.dtype == LA_BF16 ? launch_conv_h<__nv_bfloat16>(a, st) : launch_conv_h<float>(a, st);
}

}  // namespace la
