// Chunked gated delta rule on CUDA cores (fp32 arithmetic; fp32 or bf16 activations).
//
// Pages: "glm5next_kda/prefill.rs", Glm5NextKdaLayer::prefill_with_pad_fill — chunk_prepare
// (grid nchunks x heads: cumulative gate gc and the WY factors u, w per chunk) followed by
// chunk_scan (grid heads, one block per head walking the chunks in order, the recurrent state
// updated in place, scale 1/sqrt(head_dim)); "split_prefill.rs", prefill_gdn_full_batched
// (B equal-length streams, device array of h-state pointers) and
// prefill_gdn_full_batched_fla_varlen (streams of different lengths via cu_seqlens).
//
// This kernel fuses prepare and scan: one block per (stream, v-head) unit walks the unit's
// chunks of C = 64 tokens with the state H = S^T [dk][dv] resident in shared memory (fp32).
// Per chunk, with gc the inclusive cumulative log-gate (per channel for KDA, pad rows g = 0):
//   A[t][i] = beta_t sum_c K[t][c] K[i][c] e^{gc[t][c]-gc[i][c]}   (i < t)
//   P[t][i] =        sum_c Q[t][c] K[i][c] e^{gc[t][c]-gc[i][c]}   (i <= t)
//   R       = diag(beta) (V - (K (.) e^{gc}) H)
//   U'      = (I + A)^{-1} R            (forward substitution, one column per thread)
//   O       = scale ((Q (.) e^{gc}) H + P U')
//   H      <- diag(e^{gc_L}) H + (K (.) e^{gc_L - gc})^T U'
// which is the token recurrence S_t = S_{t-1} diag(a_t)(I - b_t k_t k_t^T) + b_t v_t k_t^T
// unrolled over the chunk (every exponent above is <= 0 except e^{gc} of the chunk start
// reference, so nothing overflows). Rows at or past the stream's end are loaded as pad_fill
// and removed by selects, never by multiplying with zero.
//
// It is the arithmetic baseline that the tensor-core kernel is checked against and the path
// for fp32 activations (whose 1e-5 bar rules out tf32/bf16 tensor-core operands).
#include "common.cuh"
#include "launch.h"

namespace la {

constexpr int SIMT_C = 64;        // chunk length
constexpr int SIMT_THREADS = 256;  // 16 x 16 thread grid for the 64-row tiles

template <int DK, int DV> struct SimtSmem {
    static constexpr int LK = DK + 4;  // padded row of K and gc/Kdec: conflict-free row gathers
    static constexpr int H = 0;                      // [DK][DV]   state
    static constexpr int K = H + DK * DV;            // [C][LK]    K -> K (.) e^gc
    static constexpr int Q = K + SIMT_C * LK;        // [C][DK]    Q -> Q (.) e^gc
    static constexpr int V = Q + SIMT_C * DK;        // [C][DV]    V -> R -> U'
    static constexpr int G = V + SIMT_C * DV;        // [C][LK]    gc -> K (.) e^{gc_L - gc}
    static constexpr int A = G + SIMT_C * LK;        // [C][C]     A (strictly lower)
    static constexpr int P = A + SIMT_C * SIMT_C;    // [C][C]     P (lower incl. diagonal)
    static constexpr int BETA = P + SIMT_C * SIMT_C; // [C]
    static constexpr int GL = BETA + SIMT_C;         // [DK]       gc of the chunk's last row
    static constexpr int TOTAL = GL + DK;
    static constexpr size_t BYTES = sizeof(float) * TOTAL;
};

template <typename T, int DK, int DV, bool KDA>
__global__ void __launch_bounds__(SIMT_THREADS, 1) chunk_simt_kernel(RecArgs p) {
    using L = SimtSmem<DK, DV>;
    using VT = Vec16<T>;
    constexpr int C = SIMT_C;
    constexpr int LK = L::LK;
    constexpr int NG = DV / 64;  // float4 column groups per thread in the [.][DV] tiles
    static_assert(DV % 64 == 0 && DK % 16 == 0, "dims");
    extern __shared__ __align__(16) float sm[];
    float *Hs = sm + L::H, *Ks = sm + L::K, *Qs = sm + L::Q, *Vs = sm + L::V, *Gs = sm + L::G;
    float *As = sm + L::A, *Ps = sm + L::P, *bs = sm + L::BETA, *gL = sm + L::GL;

    const int j = blockIdx.x;  // v-head
    const int s = blockIdx.y;  // stream
    const int kh = j / (p.Hv / p.Hk);
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;

    int t0, len;
    if (!stream_range(p.cu, s, p.T_each, p.total, p.max_seqlen, p.status, t0, len)) return;
    if (len <= 0) return;

    const T *qg = reinterpret_cast<const T *>(p.q) + (int64_t)kh * DK;
    const T *kg = reinterpret_cast<const T *>(p.k) + (int64_t)kh * DK;
    const T *vg = reinterpret_cast<const T *>(p.v) + (int64_t)j * DV;
    T *og = reinterpret_cast<T *>(p.out) + (int64_t)j * DV;
    float *hg = reinterpret_cast<float *>(p.h_ptrs[s]) + (int64_t)j * DK * DV;

    for (int i = tid * 4; i < DK * DV; i += SIMT_THREADS * 4)
        *reinterpret_cast<float4 *>(Hs + i) = *reinterpret_cast<const float4 *>(hg + i);

    const int nchunks = (len + C - 1) / C;
    for (int ch = 0; ch < nchunks; ++ch) {
        const int tok0 = t0 + ch * C;
        const int n = min(C, len - ch * C);

        // ---- load K, Q, V (rows >= n hold pad_fill), beta, cumulative gate ----
        {
            constexpr int VPR = DK / VT::N;  // vectors per K/Q row
            for (int idx = tid; idx < C * VPR; idx += SIMT_THREADS) {
                const int r = idx / VPR, cv = (idx % VPR) * VT::N;
                float fk[VT::N], fq[VT::N];
                if (r < n) {
                    VT::load(kg + (int64_t)(tok0 + r) * p.k_stride + cv, fk);
                    VT::load(qg + (int64_t)(tok0 + r) * p.q_stride + cv, fq);
                } else {
#pragma unroll
                    for (int e = 0; e < VT::N; ++e) fk[e] = fq[e] = p.pad_fill;
                }
#pragma unroll
                for (int e = 0; e < VT::N; ++e) {
                    Ks[r * LK + cv + e] = fk[e];
                    Qs[r * DK + cv + e] = fq[e];
                }
            }
            constexpr int VPRV = DV / VT::N;
            for (int idx = tid; idx < C * VPRV; idx += SIMT_THREADS) {
                const int r = idx / VPRV, cv = (idx % VPRV) * VT::N;
                float fv[VT::N];
                if (r < n) {
                    VT::load(vg + (int64_t)(tok0 + r) * p.v_stride + cv, fv);
                } else {
#pragma unroll
                    for (int e = 0; e < VT::N; ++e) fv[e] = p.pad_fill;
                }
#pragma unroll
                for (int e = 0; e < VT::N; ++e) Vs[r * DV + cv + e] = fv[e];
            }
            if (tid < C) bs[tid] = tid < n ? p.beta[(int64_t)(tok0 + tid) * p.Hv + j] : 0.f;
            if (tid < DK) {
                // inclusive cumulative log-gate; pad rows contribute g = 0 (the pages zero the
                // gate tail), so gc of the last row equals gc of the last valid row
                float acc = 0.f;
#pragma unroll 8
                for (int r = 0; r < C; ++r) {
                    float gv = 0.f;
                    if (r < n) {
                        gv = KDA ? p.g[((int64_t)(tok0 + r) * p.Hv + j) * DK + tid]
                                 : p.g[(int64_t)(tok0 + r) * p.Hv + j];
                    }
                    acc += gv;
                    Gs[r * LK + tid] = acc;
                }
                gL[tid] = acc;
            }
        }
        __syncthreads();

        // ---- A and P (rows t = ty + 16a, columns i = tx + 16b; only b <= a can be nonzero) ----
        {
            float accA[4][4], accP[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) accA[a][b] = accP[a][b] = 0.f;
#pragma unroll 2
            for (int c = 0; c < DK; c += 4) {
                float4 kt[4], qt[4], ki[4], gt[4], gi[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    kt[a] = *reinterpret_cast<const float4 *>(Ks + (ty + 16 * a) * LK + c);
                    qt[a] = *reinterpret_cast<const float4 *>(Qs + (ty + 16 * a) * DK + c);
                    ki[a] = *reinterpret_cast<const float4 *>(Ks + (tx + 16 * a) * LK + c);
                    if (KDA) {
                        gt[a] = *reinterpret_cast<const float4 *>(Gs + (ty + 16 * a) * LK + c);
                        gi[a] = *reinterpret_cast<const float4 *>(Gs + (tx + 16 * a) * LK + c);
                    }
                }
#pragma unroll
                for (int a = 0; a < 4; ++a) {
#pragma unroll
                    for (int b = 0; b <= a; ++b) {
                        if (KDA) {
                            const float e0 = __expf(gt[a].x - gi[b].x);
                            const float e1 = __expf(gt[a].y - gi[b].y);
                            const float e2 = __expf(gt[a].z - gi[b].z);
                            const float e3 = __expf(gt[a].w - gi[b].w);
                            accA[a][b] = fmaf(kt[a].x * ki[b].x, e0, accA[a][b]);
                            accA[a][b] = fmaf(kt[a].y * ki[b].y, e1, accA[a][b]);
                            accA[a][b] = fmaf(kt[a].z * ki[b].z, e2, accA[a][b]);
                            accA[a][b] = fmaf(kt[a].w * ki[b].w, e3, accA[a][b]);
                            accP[a][b] = fmaf(qt[a].x * ki[b].x, e0, accP[a][b]);
                            accP[a][b] = fmaf(qt[a].y * ki[b].y, e1, accP[a][b]);
                            accP[a][b] = fmaf(qt[a].z * ki[b].z, e2, accP[a][b]);
                            accP[a][b] = fmaf(qt[a].w * ki[b].w, e3, accP[a][b]);
                        } else {
                            accA[a][b] = fmaf(kt[a].x, ki[b].x, accA[a][b]);
                            accA[a][b] = fmaf(kt[a].y, ki[b].y, accA[a][b]);
                            accA[a][b] = fmaf(kt[a].z, ki[b].z, accA[a][b]);
                            accA[a][b] = fmaf(kt[a].w, ki[b].w, accA[a][b]);
                            accP[a][b] = fmaf(qt[a].x, ki[b].x, accP[a][b]);
                            accP[a][b] = fmaf(qt[a].y, ki[b].y, accP[a][b]);
                            accP[a][b] = fmaf(qt[a].z, ki[b].z, accP[a][b]);
                            accP[a][b] = fmaf(qt[a].w, ki[b].w, accP[a][b]);
                        }
                    }
                }
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int t = ty + 16 * a, i = tx + 16 * b;
                    float av = 0.f, pv = 0.f;
                    if (b <= a && i <= t && t < n) {  // i <= t < n implies i < n
                        float dec = 1.f;
                        if (!KDA) dec = __expf(Gs[t * LK] - Gs[i * LK]);
                        pv = accP[a][b] * dec;
                        if (i < t) av = bs[t] * accA[a][b] * dec;
                    }
                    As[t * C + i] = av;
                    Ps[t * C + i] = pv;
                }
            }
        }
        __syncthreads();

        // ---- Q <- Q (.) e^gc, K <- K (.) e^gc, G <- K (.) e^{gc_L - gc} (pad rows -> 0) ----
        for (int idx = tid; idx < C * DK; idx += SIMT_THREADS) {
            const int t = idx / DK, c = idx % DK;
            const float gct = Gs[t * LK + c];
            const float kv = Ks[t * LK + c];
            const bool valid = t < n;
            Qs[t * DK + c] *= __expf(gct);
            Ks[t * LK + c] = valid ? kv * __expf(gct) : 0.f;
            Gs[t * LK + c] = valid ? kv * __expf(gL[c] - gct) : 0.f;
        }
        __syncthreads();

        // ---- R = diag(beta) (V - Kg H), in place in V ----
        {
            float acc[4][NG][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int gI = 0; gI < NG; ++gI)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[a][gI][e] = 0.f;
#pragma unroll 4
            for (int c = 0; c < DK; ++c) {
                float ka[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) ka[a] = Ks[(ty + 16 * a) * LK + c];
#pragma unroll
                for (int gI = 0; gI < NG; ++gI) {
                    const float4 h = *reinterpret_cast<const float4 *>(Hs + c * DV + gI * 64 + tx * 4);
#pragma unroll
                    for (int a = 0; a < 4; ++a) {
                        acc[a][gI][0] = fmaf(ka[a], h.x, acc[a][gI][0]);
                        acc[a][gI][1] = fmaf(ka[a], h.y, acc[a][gI][1]);
                        acc[a][gI][2] = fmaf(ka[a], h.z, acc[a][gI][2]);
                        acc[a][gI][3] = fmaf(ka[a], h.w, acc[a][gI][3]);
                    }
                }
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int t = ty + 16 * a;
                const float b = bs[t];
#pragma unroll
                for (int gI = 0; gI < NG; ++gI) {
                    float *vp = Vs + t * DV + gI * 64 + tx * 4;
                    float4 v = *reinterpret_cast<float4 *>(vp);
                    float4 r;
                    const bool valid = t < n;
                    r.x = valid ? b * (v.x - acc[a][gI][0]) : 0.f;
                    r.y = valid ? b * (v.y - acc[a][gI][1]) : 0.f;
                    r.z = valid ? b * (v.z - acc[a][gI][2]) : 0.f;
                    r.w = valid ? b * (v.w - acc[a][gI][3]) : 0.f;
                    *reinterpret_cast<float4 *>(vp) = r;
                }
            }
        }
        __syncthreads();

        // ---- U' = (I + A)^{-1} R: forward substitution, one column per thread ----
        if (tid < DV) {
            float u[C];
#pragma unroll
            for (int t = 0; t < C; ++t) u[t] = Vs[t * DV + tid];
#pragma unroll
            for (int t = 1; t < C; ++t) {
                float acc = u[t];
#pragma unroll
                for (int i = 0; i < t; ++i) acc = fmaf(-As[t * C + i], u[i], acc);
                u[t] = acc;
            }
#pragma unroll
            for (int t = 0; t < C; ++t) Vs[t * DV + tid] = u[t];
        }
        __syncthreads();

        // ---- O = scale (Qg H + P U'), rows < n stored ----
        {
            float acc[4][NG][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int gI = 0; gI < NG; ++gI)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[a][gI][e] = 0.f;
#pragma unroll 4
            for (int c = 0; c < DK; ++c) {
                float qa[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) qa[a] = Qs[(ty + 16 * a) * DK + c];
#pragma unroll
                for (int gI = 0; gI < NG; ++gI) {
                    const float4 h = *reinterpret_cast<const float4 *>(Hs + c * DV + gI * 64 + tx * 4);
#pragma unroll
                    for (int a = 0; a < 4; ++a) {
                        acc[a][gI][0] = fmaf(qa[a], h.x, acc[a][gI][0]);
                        acc[a][gI][1] = fmaf(qa[a], h.y, acc[a][gI][1]);
                        acc[a][gI][2] = fmaf(qa[a], h.z, acc[a][gI][2]);
                        acc[a][gI][3] = fmaf(qa[a], h.w, acc[a][gI][3]);
                    }
                }
            }
#pragma unroll 4
            for (int i = 0; i < C; ++i) {
                float pa[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) pa[a] = Ps[(ty + 16 * a) * C + i];
#pragma unroll
                for (int gI = 0; gI < NG; ++gI) {
                    const float4 u = *reinterpret_cast<const float4 *>(Vs + i * DV + gI * 64 + tx * 4);
#pragma unroll
                    for (int a = 0; a < 4; ++a) {
                        acc[a][gI][0] = fmaf(pa[a], u.x, acc[a][gI][0]);
                        acc[a][gI][1] = fmaf(pa[a], u.y, acc[a][gI][1]);
                        acc[a][gI][2] = fmaf(pa[a], u.z, acc[a][gI][2]);
                        acc[a][gI][3] = fmaf(pa[a], u.w, acc[a][gI][3]);
                    }
                }
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int t = ty + 16 * a;
                if (t < n) {
                    T *orow = og + (int64_t)(tok0 + t) * p.Hv * DV;
#pragma unroll
                    for (int gI = 0; gI < NG; ++gI)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            orow[gI * 64 + tx * 4 + e] = from_f<T>(p.scale * acc[a][gI][e]);
                }
            }
        }
        __syncthreads();

        // ---- H <- diag(e^{gc_L}) H + Kdec^T U' ----
        {
            constexpr int RA = DK / 16;
            float acc[RA][NG][4];
#pragma unroll
            for (int a = 0; a < RA; ++a) {
                const int c = ty + 16 * a;
                const float dec = __expf(gL[c]);
#pragma unroll
                for (int gI = 0; gI < NG; ++gI) {
                    const float4 h = *reinterpret_cast<const float4 *>(Hs + c * DV + gI * 64 + tx * 4);
                    acc[a][gI][0] = dec * h.x;
                    acc[a][gI][1] = dec * h.y;
                    acc[a][gI][2] = dec * h.z;
                    acc[a][gI][3] = dec * h.w;
                }
            }
            for (int t = 0; t < n; ++t) {
                float kd[RA];
#pragma unroll
                for (int a = 0; a < RA; ++a) kd[a] = Gs[t * LK + ty + 16 * a];
#pragma unroll
                for (int gI = 0; gI < NG; ++gI) {
                    const float4 u = *reinterpret_cast<const float4 *>(Vs + t * DV + gI * 64 + tx * 4);
#pragma unroll
                    for (int a = 0; a < RA; ++a) {
                        acc[a][gI][0] = fmaf(kd[a], u.x, acc[a][gI][0]);
                        acc[a][gI][1] = fmaf(kd[a], u.y, acc[a][gI][1]);
                        acc[a][gI][2] = fmaf(kd[a], u.z, acc[a][gI][2]);
                        acc[a][gI][3] = fmaf(kd[a], u.w, acc[a][gI][3]);
                    }
                }
            }
#pragma unroll
            for (int a = 0; a < RA; ++a) {
                const int c = ty + 16 * a;
#pragma unroll
                for (int gI = 0; gI < NG; ++gI)
                    *reinterpret_cast<float4 *>(Hs + c * DV + gI * 64 + tx * 4) =
                        make_float4(acc[a][gI][0], acc[a][gI][1], acc[a][gI][2], acc[a][gI][3]);
            }
        }
        __syncthreads();
    }

    for (int i = tid * 4; i < DK * DV; i += SIMT_THREADS * 4)
        *reinterpret_cast<float4 *>(hg + i) = *reinterpret_cast<const float4 *>(Hs + i);
}

template <typename T, int DK, int DV, bool KDA>
static cudaError_t launch_simt_t(const RecArgs &a, cudaStream_t st) {
    auto kern = chunk_simt_kernel<T, DK, DV, KDA>;
    constexpr size_t bytes = SimtSmem<DK, DV>::BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bytes);
    if (e != cudaSuccess) return e;
    dim3 grid(a.Hv, a.B);
    kern<<<grid, SIMT_THREADS, bytes, st>>>(a);
    return cudaGetLastError();
}

template <typename T, bool KDA>
static cudaError_t launch_simt_d(const RecArgs &a, cudaStream_t st) {
    if (a.dk == 64) return launch_simt_t<T, 64, 64, KDA>(a, st);
    return launch_simt_t<T, 128, 128, KDA>(a, st);
}

cudaError_t launch_chunk_simt(const RecArgs &a, cudaStream_t st) {
    if (a.dtype == LA_BF16)
        return a.kda ? launch_simt_d<__nv_bfloat16, true>(a, st)
                     : launch_simt_d<__nv_bfloat16, false>(a, st);
    return a.kda ? launch_simt_d<float, true>(a, st) : launch_simt_d<float, false>(a, st);
}

}  // namespace la
