// Chunk-parallel scan of one long stream: the stream is cut into S segments (at multiples of the
// 64-token chunk) that the tensor-core recurrence runs side by side, then joined.
//
// The recurrence is affine in its state: over a segment, H_end = M H_0 + N and every output is
// o_t = o_t(H_0 = 0) + H_0^T p_t, where M (dk x dk) is the segment's transition, N its end state
// from H_0 = 0, and p_t = scale (transition up to t)^T q_t. Both come out of the same kernel:
//   - segment 0 runs from the true state (its outputs and end state are final);
//   - segment j >= 1 runs twice in the same launch: from H_0 = 0 with the real v (outputs
//     o_t(0) into `out`, end state N_j), and from H_0 = I with v = 0 (outputs p_t into a
//     workspace, end state M_j);
//   - then, for j = 1 .. S-1, one launch whose blocks do two independent things from
//     H_start(j): join blocks compute H_start(j+1) = M_j H_start(j) + N_j (the last one is the
//     stream's final state), correction blocks add H_start(j)^T p_t to the outputs of segment j.
//     Segment 0 runs on a copy of the true state, so the caller's state is written only by
//     the last join.
// This is not on the pages (they walk the chunks of a head in one block); it costs the
// transition runs (about 2x the work for segments >= 1) and wins when a call has too few
// (stream, v-head) units to fill the GPU, as a single long stream does.
#include "common.cuh"
#include "launch.h"

namespace la {

namespace {

constexpr int SD = 128;  // dk = dv of the tensor-core path

struct SegPlan {
    int S;                      // segments
    int b[kMaxSegments + 1];    // boundaries (token offsets), b[0] = 0, b[S] = total
};

// Pseudo-stream tables and the initial states of the segment runs.
__global__ void seg_setup_kernel(SegPlan plan, int Hv, const uint64_t *h_real, int32_t *cu_p,
                                 int32_t *cu_alt, uint64_t *ptrs, float *Nb, float *Mb,
                                 float *Hs, __nv_bfloat16 *zero_v) {
    const int S = plan.S, P = 2 * S - 1;
    const int64_t per = (int64_t)Hv * SD * SD;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        for (int i = 0; i <= S; ++i) cu_p[i] = plan.b[i];
        for (int i = S + 1; i <= P; ++i) cu_p[i] = plan.b[S];  // transition runs: see cu_alt
        for (int i = 0; i < S; ++i) cu_alt[i] = plan.b[i + 1];
        ptrs[0] = reinterpret_cast<uint64_t>(Hs);  // segment 0 runs on a copy of the state
        for (int j = 1; j < S; ++j) {
            ptrs[j] = reinterpret_cast<uint64_t>(Nb + (j - 1) * per);
            ptrs[S + j - 1] = reinterpret_cast<uint64_t>(Mb + (j - 1) * per);
        }
    }
    const int64_t n = (S - 1) * per;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        Nb[i] = 0.f;
        const int64_t e = i % (SD * SD);
        Mb[i] = (e / SD == e % SD) ? 1.f : 0.f;
    }
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < Hv * SD; i += gridDim.x * blockDim.x)
        zero_v[i] = __float2bfloat16_rn(0.f);
    const float4 *src = reinterpret_cast<const float4 *>(h_real[0]);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < per / 4;
         i += (int64_t)gridDim.x * blockDim.x)
        reinterpret_cast<float4 *>(Hs)[i] = src[i];
}

constexpr int JB = 32;                 // rows of H_start(j+1) per join block
constexpr int JOIN_BLOCKS = SD / JB;   // join blocks per v-head
constexpr int P_LD = SD + 4;           // padded row of the p tile (fp32)
constexpr size_t FIN_SMEM = (size_t)SD * SD * 4 + (size_t)64 * P_LD * 4;

// Step j of the join and the correction of segment j, both from H_start(j) = Hs[j-1]:
//  - blocks [0, Hv * JOIN_BLOCKS): rows 32 r .. of H_start(j+1) = M_j H_start(j) + N_j, written
//    to Hs[j], or to the stream's state for the last step; thread (row pair, 8 columns);
//  - the rest: a 64-token tile of segment j for one v-head, out[t] += H_start(j)^T p_t
//    (thread: 4 tokens x 8 channels).
__global__ void __launch_bounds__(256) seg_finish_kernel(SegPlan plan, int j, int Hv,
                                                         const float *Nb, const float *Mb,
                                                         float *Hs, const uint64_t *h_state,
                                                         const __nv_bfloat16 *pbuf,
                                                         __nv_bfloat16 *out) {
    extern __shared__ float fs[];
    const int tid = threadIdx.x;
    const int64_t per = (int64_t)Hv * SD * SD;
    const int nj = Hv * JOIN_BLOCKS;  // every step has a join (the last writes the final state)
    float *h = fs;  // H_start(j) [k][d]
    if ((int)blockIdx.x < nj) {
        const int head = blockIdx.x / JOIN_BLOCKS, rb = blockIdx.x % JOIN_BLOCKS;
        const int64_t hoff = (int64_t)head * SD * SD;
        const float *H = Hs + (j - 1) * per + hoff;
        const float *M = Mb + (j - 1) * per + hoff;
        const float *N = Nb + (j - 1) * per + hoff;
        float *mrow = fs + SD * SD;  // rows 32 rb .. of M_j [32][P_LD]
        for (int i = tid; i < SD * SD / 4; i += 256)
            reinterpret_cast<float4 *>(h)[i] = reinterpret_cast<const float4 *>(H)[i];
        for (int i = tid; i < JB * SD / 4; i += 256) {
            const int r = i / (SD / 4), c4 = i % (SD / 4);
            *reinterpret_cast<float4 *>(mrow + r * P_LD + 4 * c4) =
                *reinterpret_cast<const float4 *>(M + (int64_t)(JB * rb + r) * SD + 4 * c4);
        }
        __syncthreads();
        const int r2 = tid >> 4, c8 = tid & 15;  // rows 2 r2, 2 r2 + 1; columns 8 c8 ..
        float acc[2][8];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int c = 0; c < 8; ++c)
                acc[r][c] = N[(int64_t)(JB * rb + 2 * r2 + r) * SD + 8 * c8 + c];
        for (int k = 0; k < SD; ++k) {
            const float m0 = mrow[(2 * r2) * P_LD + k], m1 = mrow[(2 * r2 + 1) * P_LD + k];
            const float4 b0 = *reinterpret_cast<const float4 *>(h + k * SD + 8 * c8);
            const float4 b1 = *reinterpret_cast<const float4 *>(h + k * SD + 8 * c8 + 4);
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                acc[0][c] = fmaf(m0, bv[c], acc[0][c]);
                acc[1][c] = fmaf(m1, bv[c], acc[1][c]);
            }
        }
        float *dst = (j + 1 < plan.S) ? Hs + j * per + hoff
                                      : reinterpret_cast<float *>(h_state[0]) + hoff;
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int c = 0; c < 8; c += 4)
                *reinterpret_cast<float4 *>(dst + (int64_t)(JB * rb + 2 * r2 + r) * SD + 8 * c8 + c) =
                    make_float4(acc[r][c], acc[r][c + 1], acc[r][c + 2], acc[r][c + 3]);
        return;
    }
    // correction of segment j
    const int cb = blockIdx.x - nj;
    const int seg_len = plan.b[j + 1] - plan.b[j];
    const int ntile = (seg_len + 63) / 64;
    const int head = cb / ntile, tile = cb % ntile;
    const int t_tile = plan.b[j] + 64 * tile;
    const float *H = Hs + (j - 1) * per + (int64_t)head * SD * SD;
    float *pt = fs + SD * SD;  // p tile [64][P_LD]
    for (int i = tid; i < SD * SD / 4; i += 256)
        reinterpret_cast<float4 *>(h)[i] = reinterpret_cast<const float4 *>(H)[i];
    for (int i = tid; i < 64 * SD / 8; i += 256) {
        const int t = i / (SD / 8), c8 = (i % (SD / 8)) * 8;
        float v[8];
        if (t_tile + t < plan.b[j + 1]) {
            Vec16<__nv_bfloat16>::load(pbuf + ((int64_t)(t_tile + t) * Hv + head) * SD + c8, v);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.f;
        }
        *reinterpret_cast<float4 *>(pt + t * P_LD + c8) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4 *>(pt + t * P_LD + c8 + 4) = make_float4(v[4], v[5], v[6], v[7]);
    }
    __syncthreads();
    const int tg = tid >> 4, dg = tid & 15;
    float acc[4][8];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[r][c] = 0.f;
    for (int c4 = 0; c4 < SD; c4 += 4) {
        float pv[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float4 q = *reinterpret_cast<const float4 *>(pt + (4 * tg + r) * P_LD + c4);
            pv[r][0] = q.x; pv[r][1] = q.y; pv[r][2] = q.z; pv[r][3] = q.w;
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const float4 h0 = *reinterpret_cast<const float4 *>(h + (c4 + cc) * SD + 8 * dg);
            const float4 h1 = *reinterpret_cast<const float4 *>(h + (c4 + cc) * SD + 8 * dg + 4);
            const float h8[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int d = 0; d < 8; ++d) acc[r][d] = fmaf(h8[d], pv[r][cc], acc[r][d]);
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int t = t_tile + 4 * tg + r;
        if (t >= plan.b[j + 1]) continue;
        __nv_bfloat16 *o = out + ((int64_t)t * Hv + head) * SD + 8 * dg;
        float ov[8];
        Vec16<__nv_bfloat16>::load(o, ov);
#pragma unroll
        for (int d = 0; d < 8; ++d) ov[d] += acc[r][d];
        Vec16<__nv_bfloat16>::store(o, ov);
    }
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct SegLayout {
    size_t cu_p, cu_alt, ptrs, zero_v, N, M, Hs, P, tc, total;
};

SegLayout seg_layout(int total, int Hv, int S) {
    SegLayout l{};
    const int P = 2 * S - 1;
    const size_t st = (size_t)(S - 1) * Hv * SD * SD * 4;
    size_t o = 0;
    l.cu_p = o;   o += align256((size_t)(P + 1) * 4);
    l.cu_alt = o; o += align256((size_t)S * 4);
    l.ptrs = o;   o += align256((size_t)P * 8);
    l.zero_v = o; o += align256((size_t)Hv * SD * 2);
    l.N = o;      o += align256(st);
    l.M = o;      o += align256(st);
    l.Hs = o;     o += align256(st);
    l.P = o;      o += align256((size_t)total * Hv * SD * 2);
    l.tc = o;     o += align256(chunk_tc_workspace_bytes(P, 0));
    l.total = o;
    return l;
}

}  // namespace

int segmented_plan_segments(int total, int requested) {
    const int nch = (total + 63) / 64;
    int S = requested < 1 ? 1 : requested;
    if (S > kMaxSegments) S = kMaxSegments;
    if (S > nch) S = nch;
    return S;
}

size_t segmented_workspace_bytes(int total, int Hv, int segments) {
    const int S = segmented_plan_segments(total, segments);
    if (S <= 1) return chunk_tc_workspace_bytes(1, 0);
    return seg_layout(total, Hv, S).total;
}

cudaError_t launch_segmented(const RecArgs &a0, int segments, cudaStream_t st) {
    const int total = a0.total, Hv = a0.Hv;
    const int S = segmented_plan_segments(total, segments);
    if (S <= 1) return launch_chunk_tc(a0, st);
    SegPlan plan{};
    plan.S = S;
    const int nch = (total + 63) / 64;
    for (int i = 0; i <= S; ++i) plan.b[i] = (int)((int64_t)nch * i / S) * 64;
    plan.b[S] = total;
    int max_len = 0;
    for (int i = 0; i < S; ++i) max_len = plan.b[i + 1] - plan.b[i] > max_len ? plan.b[i + 1] - plan.b[i] : max_len;
    const SegLayout l = seg_layout(total, Hv, S);
    unsigned char *ws = reinterpret_cast<unsigned char *>(a0.workspace);
    int32_t *cu_p = reinterpret_cast<int32_t *>(ws + l.cu_p);
    int32_t *cu_alt = reinterpret_cast<int32_t *>(ws + l.cu_alt);
    uint64_t *ptrs = reinterpret_cast<uint64_t *>(ws + l.ptrs);
    __nv_bfloat16 *zero_v = reinterpret_cast<__nv_bfloat16 *>(ws + l.zero_v);
    float *Nb = reinterpret_cast<float *>(ws + l.N), *Mb = reinterpret_cast<float *>(ws + l.M);
    float *Hs = reinterpret_cast<float *>(ws + l.Hs);
    __nv_bfloat16 *pbuf = reinterpret_cast<__nv_bfloat16 *>(ws + l.P);

    seg_setup_kernel<<<256, 256, 0, st>>>(plan, Hv, a0.h_ptrs, cu_p, cu_alt, ptrs, Nb, Mb, Hs,
                                          zero_v);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    RecArgs a = a0;
    a.h_ptrs = ptrs;
    a.cu = cu_p;
    a.B = 2 * S - 1;
    a.T_each = 0;
    a.max_seqlen = max_len;
    a.use_alt = true;
    a.alt_from = S;
    a.cu_alt = cu_alt;
    a.v_alt = zero_v;
    a.out_alt = pbuf;
    a.workspace = ws + l.tc;
    a.workspace_bytes = chunk_tc_workspace_bytes(a.B, 0);
    e = launch_chunk_tc(a, st);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(seg_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)FIN_SMEM);
    if (e != cudaSuccess) return e;
    for (int j = 1; j < S; ++j) {
        const int ntile = (plan.b[j + 1] - plan.b[j] + 63) / 64;
        seg_finish_kernel<<<Hv * JOIN_BLOCKS + Hv * ntile, 256, FIN_SMEM, st>>>(
            plan, j, Hv, Nb, Mb, Hs, a0.h_ptrs, pbuf, reinterpret_cast<__nv_bfloat16 *>(a0.out));
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace la
