// Phase-1 projection GEMM on the 5th-generation tensor cores: C = A W^T, bf16 operands, fp32
// accumulation in TMEM, bf16 output.
//
// Page: "split_prefill.rs", LayerSplitPrefill::prefill_phase1_proj_batched — the QKVZ and gate
// projections of the normalised hidden rows of all stacked tokens of a batched prefill, the step
// before the conv. A [M][K] are those rows, W [N][K] a linear layer's weight ([out][in]).
//
// GB300 design: a persistent, warp-specialised kernel, one 192-thread block per SM.
//  - warp 0: one elected lane streams 128 x 64 tiles of A and 256 x 64 tiles of W into a
//    4-stage ring of 48 KB stages with TMA (cp.async.bulk.tensor, 128-byte swizzle, the layout
//    the MMA descriptors read), completion on per-stage mbarriers (expect_tx);
//  - warp 1: one elected lane issues tcgen05.mma kind::f16 (M = 128, N = 256, K = 16, four per
//    stage) into one of two 256-column TMEM accumulators, frees each stage with tcgen05.commit;
//  - warps 2-5: the epilogue (one TMEM lane quadrant each) drains the other accumulator to bf16
//    while the next tile accumulates.
// Tiles are walked n-fastest: a wave covers a few 128-row bands of A against all of W, so W
// stays in L2 and A is read from HBM about once. Every
// wait is bounded (2 s): on timeout the block records LA_DEV_TIMEOUT, stops issuing, drains its
// own copies and MMAs, frees TMEM and returns. Tails in M, N and K come from TMA's zero fill;
// stores are guarded.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace la {

namespace {

constexpr int GM = 128, GN = 256, GK = 64, STAGES = 4;
constexpr uint32_t A_BYTES = GM * GK * 2;   // 16 KB
constexpr uint32_t B_BYTES = GN * GK * 2;   // 32 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t G_BAR = STAGES * STAGE_BYTES;  // 192 KB of tiles, then the barriers
constexpr size_t G_SMEM = G_BAR + 256 + 1024;     // + barriers + alignment slack
constexpr int G_THREADS = 192;
constexpr uint32_t ACC_COLS = 2 * GN;             // two accumulators
constexpr uint64_t G_WAIT_NS = 2000000000ull;
constexpr uint32_t G_SLEEP_NS = 1000000u;  // a waiting thread sleeps up to 1 ms between tests

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

__global__ void __launch_bounds__(G_THREADS, 1)
gemm_bf16_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_w,
                 __nv_bfloat16 *__restrict__ C, int M, int N, int K, int64_t ldc, int *status,
                 uint64_t wait_ns, int debug_stall) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + G_BAR);
    uint64_t *empty = full + STAGES;
    uint64_t *accf = empty + STAGES;  // accumulator ready (MMA -> epilogue)
    uint64_t *acce = accf + 2;        // accumulator drained (epilogue -> MMA)
    uint64_t *fin = acce + 2;         // the MMA thread's last commit
    uint32_t *tmem_sh = reinterpret_cast<uint32_t *>(fin + 1);
    volatile int *err = reinterpret_cast<volatile int *>(tmem_sh + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(full + s, 1);
            tc::mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(accf + b, 1);
            tc::mbar_init(acce + b, 128);
        }
        tc::mbar_init(fin, 1);
        *err = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_sh, ACC_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = *tmem_sh;
    const int mt = (M + GM - 1) / GM, nt = (N + GN - 1) / GN;
    const int ntiles = mt * nt, kb = (K + GK - 1) / GK;
    const uint32_t sbase = tc::smem_u32(sm);

    if (warp == 0) {
        if (tc::elect_one()) {  // ---- TMA producer
            uint32_t it = 0;  // copies issued so far
            for (int tile = blockIdx.x; tile < ntiles && !*err; tile += gridDim.x) {
                const int m0 = (tile / nt) * GM, n0 = (tile % nt) * GN;
                for (int k = 0; k < kb; ++k, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                    if (!tc::mbar_wait(empty + s, ph ^ 1u, wait_ns, G_SLEEP_NS) || *err) {
                        *err = 1;
                        break;
                    }
                    tc::mbar_expect_tx(full + s, STAGE_BYTES);
                    tc::tma_load_2d(sbase + s * STAGE_BYTES, &map_a, k * GK, m0, full + s);
                    tc::tma_load_2d(sbase + s * STAGE_BYTES + A_BYTES, &map_w, k * GK, n0, full + s);
                }
            }
            // every copy this thread issued must have landed before the block exits: the last
            // one on stage s was copy number it - 1 - ((it - 1 - s) mod STAGES)
            for (uint32_t s = 0; s < STAGES && s < it; ++s) {
                const uint32_t last = it - 1 - ((it - 1 - s) % STAGES);
                if (!tc::mbar_wait(full + s, (last / STAGES) & 1u, G_WAIT_NS, G_SLEEP_NS)) *err = 1;
            }
        }
    } else if (warp == 1) {
        if (tc::elect_one()) {  // ---- MMA issuer
            constexpr uint32_t id = tc::idesc(GM, GN, tc::FMT_BF16);
            uint32_t it = 0, tcnt = 0;
            // test knob: a wait on a barrier nothing has completed yet (its first phase ends
            // with the final commit below) runs out, and the block unwinds
            if (debug_stall && !tc::mbar_wait(fin, 0, wait_ns, G_SLEEP_NS)) *err = 1;
            for (int tile = blockIdx.x; tile < ntiles && !*err; tile += gridDim.x, ++tcnt) {
                const uint32_t acc = tcnt & 1u, aph = (tcnt >> 1) & 1u;
                if (!tc::mbar_wait(acce + acc, aph ^ 1u, wait_ns, G_SLEEP_NS)) {
                    *err = 1;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t d = tm + acc * GN;
                bool ok = true;
                for (int k = 0; k < kb; ++k, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                    if (!tc::mbar_wait(full + s, ph, wait_ns, G_SLEEP_NS) || *err) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t a_addr = sbase + s * STAGE_BYTES, b_addr = a_addr + A_BYTES;
#pragma unroll
                    for (uint32_t kk = 0; kk < GK / 16; ++kk)
                        tc::mma_bf16_ss(d, tc::sdesc_sw128(a_addr + kk * 32u),
                                        tc::sdesc_sw128(b_addr + kk * 32u), id, (k | kk) != 0);
                    tc::mma_commit(empty + s);
                }
                if (!ok) {
                    *err = 1;
                    break;
                }
                tc::mma_commit(accf + acc);
            }
            // every MMA this thread issued must have completed before the block exits
            tc::mma_commit(fin);
            if (!tc::mbar_wait(fin, 0, G_WAIT_NS, G_SLEEP_NS)) *err = 1;
        }
    } else {  // ---- epilogue: warps 2-5, TMEM lane quadrant warp % 4
        const uint32_t q = warp & 3;
        uint32_t tcnt = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++tcnt) {
            // every decision to stop is made per warp: the TMEM loads below are warp-collective
            if (__any_sync(0xffffffffu, *err != 0)) break;
            const uint32_t acc = tcnt & 1u, aph = (tcnt >> 1) & 1u;
            if (!__all_sync(0xffffffffu, tc::mbar_wait(accf + acc, aph, wait_ns, G_SLEEP_NS))) {
                *err = 1;
                break;
            }
            tc::fence_after_sync();
            const int m0 = (tile / nt) * GM, n0 = (tile % nt) * GN;
            const int row = m0 + 32 * (int)q + lane;
            __nv_bfloat16 *crow = C + (int64_t)row * ldc + n0;
#pragma unroll 1
            for (int c = 0; c < GN; c += 16) {
                float v[16];
                tc::tmem_ld16(tc::tmem_addr(tm + acc * GN, 32 * q, c), v);
                tc::tmem_wait_ld();
                if (row < M && n0 + c < N) {
                    if (n0 + c + 16 <= N) {
                        Vec16<__nv_bfloat16>::store(crow + c, v);
                        Vec16<__nv_bfloat16>::store(crow + c + 8, v + 8);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (n0 + c + e < N) crow[c + e] = __float2bfloat16_rn(v[e]);
                    }
                }
            }
            tc::fence_before_sync();
            mbar_arrive(acce + acc);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tm, ACC_COLS);
    if (*err && threadIdx.x == 0) raise_status(status, LA_DEV_TIMEOUT);
}

int device_sms() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

}  // namespace

cudaError_t launch_gemm_bf16(const GemmArgs &a, cudaStream_t st) {
    CUtensorMap ma, mw;
    if (!make_map_bf16_2d(&ma, a.a, a.M, a.K, a.lda, GK, GM, true) ||
        !make_map_bf16_2d(&mw, a.w, a.N, a.K, a.ldw, GK, GN, true))
        return cudaErrorInvalidValue;
    const int64_t ntiles = (int64_t)((a.M + GM - 1) / GM) * ((a.N + GN - 1) / GN);
    const int grid = (int)(ntiles < device_sms() ? ntiles : device_sms());
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)G_SMEM);
    if (e != cudaSuccess) return e;
    gemm_bf16_kernel<<<grid, G_THREADS, G_SMEM, st>>>(ma, mw, reinterpret_cast<__nv_bfloat16 *>(a.c),
                                                      a.M, a.N, a.K, a.ldc, a.status,
                                                      a.wait_ns ? a.wait_ns : G_WAIT_NS,
                                                      a.debug_stall);
    return cudaGetLastError();
}

}  // namespace la
