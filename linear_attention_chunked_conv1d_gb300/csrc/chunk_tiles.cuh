// Tile helpers of the tensor-core recurrence kernel: async copies, column walks down swizzled
// tiles, scalar shared-memory conversions, named barriers and mbarrier arrivals.
#pragma once
#include <cuda_bf16.h>

#include "tc.cuh"

namespace la {
namespace tiles {

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
// 4-byte async copy (gate scalars); `valid` false writes zero without reading the source.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 4 : 0)
                 : "memory");
}
// Wait until at most the most recent committed group of this thread is still in flight.
__device__ __forceinline__ void cp_async_wait_but_last() {
    asm volatile("cp.async.wait_group 1;" ::: "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Asks the memory system to bring `bytes` (a multiple of 16, 16-byte aligned) into L2 without
// touching shared memory; the later copy of the same rows then hits L2.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Barrier over `count` threads (a multiple of 32) on hardware barrier `id` (1..15; 0 is the
// block-wide __syncthreads barrier).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Arrival on hardware barrier `id` without waiting (the threads that sync on it see this
// thread's earlier shared-memory writes once it completes).
__device__ __forceinline__ void named_arrive(uint32_t id, uint32_t count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// One arrival on an mbarrier (release at CTA scope: the caller's earlier shared-memory writes
// are visible to a thread whose wait on this phase succeeds).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

// Byte offsets of one column (element k) of a K-major SW128 tile with R rows: row t sits at
// off[t % 8] + (t / 8) * 1024, so fully unrolled walks down a column need no address math.
struct ColWalk {
    uint32_t off[8];
    __device__ __forceinline__ void init(uint32_t base, uint32_t k, uint32_t R, uint32_t es) {
#pragma unroll
        for (uint32_t r = 0; r < 8; ++r) off[r] = base + tc::sw128_offset(r, k, R, es);
    }
    __device__ __forceinline__ uint32_t at(int t) const {
        return off[t & 7] + static_cast<uint32_t>(t >> 3) * 1024u;
    }
};

// bf16 element widened to fp32 (exact: the bf16 bits are the top half of the fp32 pattern).
__device__ __forceinline__ float ld_bf16(const unsigned char *sm, uint32_t off) {
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(sm + off)) << 16);
}
// A tf32 MMA operand element (see tc::to_tf32_operand).
__device__ __forceinline__ void st_tf32(unsigned char *sm, uint32_t off, float v) {
    *reinterpret_cast<float *>(sm + off) = tc::to_tf32_operand(v);
}

}  // namespace tiles
}  // namespace la
