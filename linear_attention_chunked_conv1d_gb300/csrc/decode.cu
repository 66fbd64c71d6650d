// Decode step of the gated delta rule: one new token per stream, on the states a prefill
// leaves behind.
//
// Page: "glm5next_kda/prefill.rs", Glm5NextKdaLayer::prefill_with_pad_fill — the layer's decode
// step (decode_k) is profiled in the same buckets as the prefill (front end, recurrence), i.e. it
// is the same layer applied to a single token: conv1d + SiLU over the carried conv state, L2 of
// the q and k heads, then one step of S <- S diag(alpha) (I - beta k k^T) + beta v k^T,
// o = scale S q, with S = H^T kept as H [dk][dv] fp32 per (stream, v-head).
//
// GB300 design: the step reads and rewrites every state once (64 KB each way per (stream,
// v-head) at d = 128) and does ~6 flops per state element, so it is HBM-bound; tensor cores have
// nothing to contract (a matrix-vector product per state). One block per (stream, v-head): each
// thread keeps a 16 x 4 slab of H in registers (coalesced 16-byte loads, one row of H per warp
// instruction), so H crosses HBM exactly twice; the two reductions over k-channels (r = S k and
// o = S q) go through shared memory. Grid = B x Hv blocks, two resident per SM.
//
//   H[c][d] <- alpha_c H[c][d]                         (decay; alpha scalar for GDN)
//   r_d      = sum_c H[c][d] k_c                        (S k after the decay)
//   u_d      = beta (v_d - r_d)
//   H[c][d] <- H[c][d] + k_c u_d                        (delta-rule write)
//   o_d      = scale sum_c H[c][d] q_c
#include "common.cuh"
#include "launch.h"

namespace la {

namespace {

template <int D> struct DecShape {
    static constexpr int NT = D == 128 ? 256 : 128;  // threads per block
    static constexpr int DV4 = D / 4;                 // float4 columns of a row of H
    static constexpr int CG = NT / DV4;               // k-channel groups (8)
    static constexpr int CPER = D / CG;               // k-channels per thread (16 or 8)
};

template <typename T, int D, bool KDA>
__global__ void __launch_bounds__(DecShape<D>::NT)
decode_rec_kernel(const DecArgs a) {
    using S = DecShape<D>;
    __shared__ float qs[D], ks[D], al[D], us[D];
    __shared__ float red[S::CG][D];
    const int u = blockIdx.x;
    const int s = u / a.Hv, j = u % a.Hv;
    const int kh = j / (a.Hv / a.Hk);
    const int t = threadIdx.x;
    const int d4 = t % S::DV4, cg = t / S::DV4;
    const int c0 = cg * S::CPER;

    float *h = reinterpret_cast<float *>(a.h_ptrs[s]) + (int64_t)j * D * D;
    float4 hv[S::CPER];
#pragma unroll
    for (int i = 0; i < S::CPER; ++i)
        hv[i] = *reinterpret_cast<const float4 *>(h + (int64_t)(c0 + i) * D + 4 * d4);

    const T *row = reinterpret_cast<const T *>(a.qkv) + (int64_t)s * a.qkv_stride;
    const float beta = a.beta[(int64_t)s * a.Hv + j];
    for (int i = t; i < D; i += S::NT) {
        qs[i] = to_f(row[kh * D + i]);
        ks[i] = to_f(row[(a.Hk + kh) * D + i]);
        us[i] = to_f(row[(2 * a.Hk + j) * D + i]);  // v, replaced by u below
        al[i] = __expf(KDA ? a.g[((int64_t)s * a.Hv + j) * D + i] : a.g[(int64_t)s * a.Hv + j]);
    }
    __syncthreads();

    // decay, then this thread's part of r = S k
    float4 rp = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < S::CPER; ++i) {
        const float ac = al[c0 + i], kc = ks[c0 + i];
        hv[i].x *= ac; hv[i].y *= ac; hv[i].z *= ac; hv[i].w *= ac;
        rp.x = fmaf(hv[i].x, kc, rp.x);
        rp.y = fmaf(hv[i].y, kc, rp.y);
        rp.z = fmaf(hv[i].z, kc, rp.z);
        rp.w = fmaf(hv[i].w, kc, rp.w);
    }
    *reinterpret_cast<float4 *>(&red[cg][4 * d4]) = rp;
    __syncthreads();
    if (t < D) {
        float r = 0.f;
#pragma unroll
        for (int g = 0; g < S::CG; ++g) r += red[g][t];
        us[t] = beta * (us[t] - r);
    }
    __syncthreads();

    // delta-rule write, state back to HBM, and this thread's part of o = S q
    const float4 uv = *reinterpret_cast<const float4 *>(&us[4 * d4]);
    float4 op = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < S::CPER; ++i) {
        const float kc = ks[c0 + i], qc = qs[c0 + i];
        hv[i].x = fmaf(kc, uv.x, hv[i].x);
        hv[i].y = fmaf(kc, uv.y, hv[i].y);
        hv[i].z = fmaf(kc, uv.z, hv[i].z);
        hv[i].w = fmaf(kc, uv.w, hv[i].w);
        *reinterpret_cast<float4 *>(h + (int64_t)(c0 + i) * D + 4 * d4) = hv[i];
        op.x = fmaf(hv[i].x, qc, op.x);
        op.y = fmaf(hv[i].y, qc, op.y);
        op.z = fmaf(hv[i].z, qc, op.z);
        op.w = fmaf(hv[i].w, qc, op.w);
    }
    *reinterpret_cast<float4 *>(&red[cg][4 * d4]) = op;
    __syncthreads();
    if (t < D) {
        float o = 0.f;
#pragma unroll
        for (int g = 0; g < S::CG; ++g) o += red[g][t];
        reinterpret_cast<T *>(a.out)[((int64_t)s * a.Hv + j) * D + t] = from_f<T>(a.scale * o);
    }
}

template <typename T, int D>
cudaError_t launch_dec_t(const DecArgs &a, cudaStream_t st) {
    const unsigned grid = (unsigned)a.B * (unsigned)a.Hv;
    if (a.kda) decode_rec_kernel<T, D, true><<<grid, DecShape<D>::NT, 0, st>>>(a);
    else decode_rec_kernel<T, D, false><<<grid, DecShape<D>::NT, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_recurrence(const DecArgs &a, cudaStream_t st) {
    if (a.dtype == LA_BF16)
        return a.d == 64 ? launch_dec_t<__nv_bfloat16, 64>(a, st) : launch_dec_t<__nv_bfloat16, 128>(a, st);
    return a.d == 64 ? launch_dec_t<float, 64>(a, st) : launch_dec_t<float, 128>(a, st);
}

}  // namespace la
