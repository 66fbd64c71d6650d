// Shared device helpers of the linattn library (not part of the C ABI).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "linattn.h"

namespace la {

// 16-byte vector of activations, widened to fp32.
template <typename T> struct Vec16;

template <> struct Vec16<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void load(const float *p, float *f) {
        float4 v = *reinterpret_cast<const float4 *>(p);
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    }
    __device__ __forceinline__ static void store(float *p, const float *f) {
        *reinterpret_cast<float4 *>(p) = make_float4(f[0], f[1], f[2], f[3]);
    }
};

template <> struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void load(const __nv_bfloat16 *p, float *f) {
        uint4 v = *reinterpret_cast<const uint4 *>(p);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 t = __bfloat1622float2(h[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
    __device__ __forceinline__ static void store(__nv_bfloat16 *p, const float *f) {
        uint4 v;
        __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        *reinterpret_cast<uint4 *>(p) = v;
    }
};

// 4 activations per access (16 bytes of fp32, 8 bytes of bf16), widened to fp32. The
// elementwise front-end kernels use it so that both dtypes reduce in the same order.
template <typename T> struct Vec4;

template <> struct Vec4<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void load(const float *p, float *f) { Vec16<float>::load(p, f); }
    __device__ __forceinline__ static void store(float *p, const float *f) { Vec16<float>::store(p, f); }
    // the access as loaded (kept in this form while in flight), and its widening
    using Raw = float4;
    __device__ __forceinline__ static Raw load_raw(const float *p) { return *reinterpret_cast<const float4 *>(p); }
    __device__ __forceinline__ static Raw zero_raw() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ __forceinline__ static void widen(const Raw &v, float *f) {
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    }
};

template <> struct Vec4<__nv_bfloat16> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void load(const __nv_bfloat16 *p, float *f) {
        widen(load_raw(p), f);
    }
    // the access as loaded (two registers while in flight), and its exact widening
    using Raw = uint2;
    __device__ __forceinline__ static Raw load_raw(const __nv_bfloat16 *p) {
        return *reinterpret_cast<const uint2 *>(p);
    }
    __device__ __forceinline__ static Raw zero_raw() { return make_uint2(0u, 0u); }
    __device__ __forceinline__ static void widen(const Raw &v, float *f) {
        f[0] = __uint_as_float(v.x << 16);
        f[1] = __uint_as_float(v.x & 0xFFFF0000u);
        f[2] = __uint_as_float(v.y << 16);
        f[3] = __uint_as_float(v.y & 0xFFFF0000u);
    }
    __device__ __forceinline__ static void store(__nv_bfloat16 *p, const float *f) {
        uint2 v;
        __nv_bfloat162 a = __floats2bfloat162_rn(f[0], f[1]);
        __nv_bfloat162 b = __floats2bfloat162_rn(f[2], f[3]);
        v.x = *reinterpret_cast<uint32_t *>(&a);
        v.y = *reinterpret_cast<uint32_t *>(&b);
        *reinterpret_cast<uint2 *>(p) = v;
    }
};

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) {  // exact widening
    return __uint_as_float(static_cast<uint32_t>(__bfloat16_as_ushort(x)) << 16);
}
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}
// Two values rounded to T and widened back to fp32 (T = bf16: one paired conversion).
template <typename T> __device__ __forceinline__ void round_to_2(float &a, float &b);
template <> __device__ __forceinline__ void round_to_2<float>(float &, float &) {}
template <> __device__ __forceinline__ void round_to_2<__nv_bfloat16>(float &a, float &b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const uint32_t u = *reinterpret_cast<const uint32_t *>(&h);
    a = __uint_as_float(u << 16);
    b = __uint_as_float(u & 0xFFFF0000u);
}

// Packed pairs of fp32 (Blackwell f32x2 ALU ops; each lane rounds like the scalar op, so a
// packed chain gives the bits of the scalar one).
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Hardware base-2 exponential and reciprocal (approximate, subnormals flushed).
__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// SiLU(y) = y sigmoid(y) = y / (1 + e^-y), with e^-y = 2^(-y log2 e) and the reciprocal from
// the hardware approximations. silu2 applies it to a packed pair with the same roundings, so
// every caller (the conv kernel, the fused front end and the gated epilogues) gets the bits of
// the scalar form.
constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float silu(float y) {
    const float e = ex2_approx(__fmul_rn(y, -kLog2e));
    return __fmul_rn(y, rcp_approx(__fadd_rn(1.f, e)));
}
__device__ __forceinline__ uint64_t silu2(uint64_t y) {
    float t0, t1;
    upk2(mul2(y, pk2(-kLog2e, -kLog2e)), t0, t1);
    float d0, d1;
    upk2(add2(pk2(1.f, 1.f), pk2(ex2_approx(t0), ex2_approx(t1))), d0, d1);
    return mul2(y, pk2(rcp_approx(d0), rcp_approx(d1)));
}

// Raises a device status flag (LA_DEV_*). `status` points at the library's per-device word.
__device__ __forceinline__ void raise_status(int *status, int flag) {
    if (status) atomicOr(status, flag);
}

// Token range of stream s: explicit cu_seqlens (varlen) or s*T_each (batched / single).
// Returns false (and raises LA_DEV_BAD_SEQLENS) if the offsets are out of bounds.
__device__ __forceinline__ bool stream_range(const int32_t *cu, int s, int T_each, int total,
                                             int max_seqlen, int *status, int &t0, int &len) {
    if (!cu) {
        t0 = s * T_each;
        len = T_each;
        return true;
    }
    int a = cu[s], b = cu[s + 1];
    if (a < 0 || b < a || b > total || (b - a) > max_seqlen) {
        raise_status(status, LA_DEV_BAD_SEQLENS);
        return false;
    }
    t0 = a;
    len = b - a;
    return true;
}

}  // namespace la
