// GPU unit check of how the tf32 MMA reads fp32 operands: D[128][16] = A[128][8] . B[16][8]^T
// with B rows 0..7 the identity, so D[:, 0:8] is A as the tensor core interprets it (A from
// shared memory, or from tensor memory). Test-only.
#include <cuda_runtime.h>
#include <cstdint>
#include "tc.cuh"
using namespace la::tc;

__global__ void __launch_bounds__(128, 1)
trunc_kernel(const float *A, float *D, int ts, int *err) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base_sh;
    unsigned char *sm = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5;
    unsigned char *As = sm;            // 128 rows x 8 fp32 in a 128-byte swizzle atom (32 wide)
    unsigned char *Bs = sm + 128 * 128; // 16 rows
    for (int i = tid; i < (128 + 16) * 32; i += 128) ((float *)sm)[i] = 0.f;
    __syncthreads();
    for (int i = tid; i < 128 * 8; i += 128) {
        const int r = i / 8, k = i % 8;
        *(float *)(As + sw128_offset(r, k, 128, 4)) = A[i];  // raw bits, no rounding
    }
    if (tid < 8) *(float *)(Bs + sw128_offset(tid, tid, 16, 4)) = 1.0f;
    if (tid == 0) { mbar_init(&bar, 1); fence_mbar_init(); }
    if (warp == 0) { tmem_alloc(&tmem_base_sh, 64); tmem_relinquish(); }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = tmem_base_sh;
    const uint32_t lane = tmem_lane_base(warp);
    if (ts) {  // A row tid -> TMEM lane tid, columns 32..39
        float v[16];
        for (int i = 0; i < 16; ++i) v[i] = i < 8 ? A[tid * 8 + i] : 0.f;
        tmem_st16(tmem_addr(tbase, lane, 32), v);
        tmem_wait_st();
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    if (warp == 0 && elect_one()) {
        fence_after_sync();
        const uint32_t id = idesc(128, 16, FMT_TF32);
        const uint64_t bd = sdesc_sw128(smem_u32(Bs));
        if (ts) mma_tf32_ts(tbase, tbase + 32, bd, id, 0);
        else mma_tf32_ss(tbase, sdesc_sw128(smem_u32(As)), bd, id, 0);
        mma_commit(&bar);
    }
    __syncwarp();
    const bool ok = mbar_wait(&bar, 0, 1000000000ull);
    if (!ok && (tid & 31) == 0) atomicExch(err, 1);
    fence_after_sync();
    if (ok) {
        float v[16];
        tmem_ld16(tmem_addr(tbase, lane, 0), v);
        tmem_wait_ld();
        for (int i = 0; i < 8; ++i) D[tid * 8 + i] = v[i];
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 64);
}

extern "C" int trunc_run(const float *A, float *D, int ts, int *err) {
    const size_t smem = (128 + 16) * 128 + 1024;
    if (cudaFuncSetAttribute(trunc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return -1;
    trunc_kernel<<<1, 128, smem>>>(A, D, ts, err);
    if (cudaGetLastError() != cudaSuccess) return -2;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : -3;
}
