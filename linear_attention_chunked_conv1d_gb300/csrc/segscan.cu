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
//   - a join kernel walks the segments: H_start(j+1) = M_j H_start(j) + N_j (H_start(1) = the end
//     state of segment 0), ending with the stream's final state;
//   - a correction kernel adds H_start(j)^T p_t to the outputs of segment j.
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
                                 __nv_bfloat16 *zero_v) {
    const int S = plan.S, P = 2 * S - 1;
    const int64_t per = (int64_t)Hv * SD * SD;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        for (int i = 0; i <= S; ++i) cu_p[i] = plan.b[i];
        for (int i = S + 1; i <= P; ++i) cu_p[i] = plan.b[S];  // transition runs: see cu_alt
        for (int i = 0; i < S; ++i) cu_alt[i] = plan.b[i + 1];
        ptrs[0] = h_real[0];
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
}

constexpr int MT_LD = SD + 4;  // padded row of the transposed transition in shared memory
constexpr size_t JOIN_SMEM = (size_t)SD * MT_LD * 4 + (size_t)SD * SD * 4;

// One block per v-head: H_start(1) = the real state (segment 0's end), H_start(j+1) =
// M_j H_start(j) + N_j; H_start(j) kept for the correction, the last one written back as the
// stream's final state. Thread (tr, tc) computes rows 8tr.. and columns 8tc.. of each product.
__global__ void __launch_bounds__(256) seg_join_kernel(int S, const uint64_t *ptrs, const float *Nb,
                                                       const float *Mb, float *Hs) {
    float *h_real = reinterpret_cast<float *>(ptrs[0]);  // the stream's own state
    extern __shared__ float js[];
    float *mt = js;               // M^T [k][c], row MT_LD
    float *hc = js + SD * MT_LD;  // H_start(j) [k][d]
    const int j_head = blockIdx.x;
    const int64_t per = (int64_t)gridDim.x * SD * SD;
    const int64_t hoff = (int64_t)j_head * SD * SD;
    const int tid = threadIdx.x, tr = tid >> 4, tcol = tid & 15;
    float *hreal = h_real + hoff;
    for (int i = tid; i < SD * SD; i += 256) {
        const float v = hreal[i];
        hc[i] = v;
        Hs[hoff + i] = v;  // H_start(1)
    }
    for (int j = 1; j < S; ++j) {
        const float *M = Mb + (j - 1) * per + hoff;
        const float *N = Nb + (j - 1) * per + hoff;
        for (int i = tid; i < SD * SD; i += 256) mt[(i % SD) * MT_LD + i / SD] = M[i];
        __syncthreads();
        float acc[8][8];
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[r][c] = N[(int64_t)(8 * tr + r) * SD + 8 * tcol + c];
        for (int k = 0; k < SD; ++k) {
            const float4 a0 = *reinterpret_cast<const float4 *>(mt + k * MT_LD + 8 * tr);
            const float4 a1 = *reinterpret_cast<const float4 *>(mt + k * MT_LD + 8 * tr + 4);
            const float4 b0 = *reinterpret_cast<const float4 *>(hc + k * SD + 8 * tcol);
            const float4 b1 = *reinterpret_cast<const float4 *>(hc + k * SD + 8 * tcol + 4);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
        }
        __syncthreads();  // every thread is done reading hc and mt
        float *dst = (j + 1 < S) ? Hs + j * per + hoff : hreal;
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int idx = (8 * tr + r) * SD + 8 * tcol + c;
                hc[idx] = acc[r][c];
                dst[idx] = acc[r][c];
            }
        __syncthreads();
    }
}

constexpr int PT_LD = 68;  // padded row of the transposed p tile
constexpr size_t CORR_SMEM = (size_t)SD * SD * 4 + (size_t)SD * PT_LD * 4;

// out[t][j] += H_start(seg)^T p_t for the 64-token tile blockIdx.x of the tokens past segment 0
// (tiles never straddle a boundary: boundaries are multiples of 64), v-head blockIdx.y. Thread
// (tg, dg) computes tokens 4tg.. and channels 8dg.. of the tile.
__global__ void __launch_bounds__(256) seg_correct_kernel(SegPlan plan, int Hv, int total,
                                                          const float *Hs,
                                                          const __nv_bfloat16 *pbuf,
                                                          __nv_bfloat16 *out) {
    extern __shared__ float cs[];
    float *h = cs;             // H_start [c][d]
    float *pt = cs + SD * SD;  // p^T [c][t], row PT_LD
    const int j = blockIdx.y;
    const int t_tile = plan.b[1] + 64 * blockIdx.x;
    if (t_tile >= total) return;
    int seg = 1;
    while (seg + 1 < plan.S && t_tile >= plan.b[seg + 1]) ++seg;
    const int64_t per = (int64_t)Hv * SD * SD;
    const float *H = Hs + (seg - 1) * per + (int64_t)j * SD * SD;
    const int tid = threadIdx.x;
    for (int i = tid; i < SD * SD / 4; i += 256)
        reinterpret_cast<float4 *>(h)[i] = reinterpret_cast<const float4 *>(H)[i];
    for (int i = tid; i < 64 * SD; i += 256) {
        const int t = i / SD, c = i % SD;
        pt[c * PT_LD + t] = t_tile + t < total
            ? __bfloat162float(pbuf[((int64_t)(t_tile + t) * Hv + j) * SD + c]) : 0.f;
    }
    __syncthreads();
    const int tg = tid >> 4, dg = tid & 15;
    float acc[4][8];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[r][c] = 0.f;
    for (int c = 0; c < SD; ++c) {
        const float4 pv = *reinterpret_cast<const float4 *>(pt + c * PT_LD + 4 * tg);
        const float4 h0 = *reinterpret_cast<const float4 *>(h + c * SD + 8 * dg);
        const float4 h1 = *reinterpret_cast<const float4 *>(h + c * SD + 8 * dg + 4);
        const float p4[4] = {pv.x, pv.y, pv.z, pv.w};
        const float h8[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int d = 0; d < 8; ++d) acc[r][d] = fmaf(h8[d], p4[r], acc[r][d]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int t = t_tile + 4 * tg + r;
        if (t >= total) continue;
        __nv_bfloat16 *o = out + ((int64_t)t * Hv + j) * SD + 8 * dg;
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

    seg_setup_kernel<<<256, 256, 0, st>>>(plan, Hv, a0.h_ptrs, cu_p, cu_alt, ptrs, Nb, Mb, zero_v);
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
    e = cudaFuncSetAttribute(seg_join_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)JOIN_SMEM);
    if (e != cudaSuccess) return e;
    // the real state pointer lives in device memory: the join reads it from the table the
    // setup kernel filled (ptrs[0])
    seg_join_kernel<<<Hv, 256, JOIN_SMEM, st>>>(S, ptrs, Nb, Mb, Hs);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(seg_correct_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CORR_SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid((total - plan.b[1] + 63) / 64, Hv);
    seg_correct_kernel<<<grid, 256, CORR_SMEM, st>>>(plan, Hv, total, Hs, pbuf,
                                                     reinterpret_cast<__nv_bfloat16 *>(a0.out));
    return cudaGetLastError();
}

}  // namespace la
