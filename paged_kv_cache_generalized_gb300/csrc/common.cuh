// Device helpers shared by the libpagedkv kernels (sm_103a): element conversion, mbarrier and
// bulk-copy PTX wrappers, bounded waits, the device status word.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

// A bounded wait gives up after this many nanoseconds of %globaltimer and reports
// PA_DEV_TIMEOUT instead of spinning forever.
constexpr uint64_t kWaitTimeoutNs = 1000000000ull;

__device__ __forceinline__ void report(unsigned *status, unsigned bits) {
    if (status) atomicOr(status, bits);
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- element conversion -------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float to_f(float x) { return x; }
    static __device__ __forceinline__ float from_f(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};
template <> struct Elem<__half> {
    static __device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
    static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
};

// Loads N consecutive elements (N * sizeof(T) a multiple of 8 bytes, naturally aligned to the
// vector width) from shared or global memory and widens them to float.  16-byte multiples use
// 128-bit accesses.
template <typename T, int N>
__device__ __forceinline__ void load_f(const T *p, float (&out)[N]) {
    constexpr int kBytes = N * sizeof(T);
    static_assert(kBytes % 8 == 0, "vector width");
    if constexpr (kBytes % 16 == 0) {
        uint4 raw[kBytes / 16];
#pragma unroll
        for (int w = 0; w < kBytes / 16; ++w) raw[w] = reinterpret_cast<const uint4 *>(p)[w];
        const T *e = reinterpret_cast<const T *>(raw);
#pragma unroll
        for (int i = 0; i < N; ++i) out[i] = Elem<T>::to_f(e[i]);
    } else {
        uint2 raw[kBytes / 8];
#pragma unroll
        for (int w = 0; w < kBytes / 8; ++w) raw[w] = reinterpret_cast<const uint2 *>(p)[w];
        const T *e = reinterpret_cast<const T *>(raw);
#pragma unroll
        for (int i = 0; i < N; ++i) out[i] = Elem<T>::to_f(e[i]);
    }
}

template <typename T, int N>
__device__ __forceinline__ void store_f(T *p, const float (&in)[N]) {
    constexpr int kBytes = N * sizeof(T);
    static_assert(kBytes % 8 == 0, "vector width");
    if constexpr (kBytes % 16 == 0) {
        uint4 raw[kBytes / 16];
        T *e = reinterpret_cast<T *>(raw);
#pragma unroll
        for (int i = 0; i < N; ++i) e[i] = Elem<T>::from_f(in[i]);
#pragma unroll
        for (int w = 0; w < kBytes / 16; ++w) reinterpret_cast<uint4 *>(p)[w] = raw[w];
    } else {
        uint2 raw[kBytes / 8];
        T *e = reinterpret_cast<T *>(raw);
#pragma unroll
        for (int i = 0; i < N; ++i) e[i] = Elem<T>::from_f(in[i]);
#pragma unroll
        for (int w = 0; w < kBytes / 8; ++w) reinterpret_cast<uint2 *>(p)[w] = raw[w];
    }
}

// ---- fast exp2 and packed two-lane fp32 arithmetic ------------------------------------------
// 2^x by the special-function unit (relative error about 2^-22; -inf -> +0; subnormal results
// flush to zero).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two fp32 values in one 64-bit register pair, for the packed fp32 instructions.
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Widens 2*NP consecutive 16-bit, fp32 or E4M3 elements to NP packed fp32 pairs (even, odd),
// ready for the packed fp32 instructions.  bf16 -> fp32 is exact by moving the 16 bits into the high
// half of a word (a shift for the even element, a mask for the odd one); f16 uses the hardware
// conversion; fp32 pairs are the loaded words themselves.  16-byte aligned, 16-byte multiples.
template <typename T> __device__ __forceinline__ uint64_t widen2(uint32_t w);
template <> __device__ __forceinline__ uint64_t widen2<__nv_bfloat16>(uint32_t w) {
    uint64_t r;
    asm("{\n\t.reg .b32 lo, hi;\n\tshl.b32 lo, %1, 16;\n\tand.b32 hi, %1, 0xffff0000;\n\t"
        "mov.b64 %0, {lo, hi};\n\t}"
        : "=l"(r)
        : "r"(w));
    return r;
}
template <> __device__ __forceinline__ uint64_t widen2<__half>(uint32_t w) {
    uint64_t r;
    asm("{\n\t.reg .b16 h0, h1;\n\t.reg .f32 lo, hi;\n\tmov.b32 {h0, h1}, %1;\n\t"
        "cvt.f32.f16 lo, h0;\n\tcvt.f32.f16 hi, h1;\n\tmov.b64 %0, {lo, hi};\n\t}"
        : "=l"(r)
        : "r"(w));
    return r;
}

// One FP8 E4M3 code (1 sign, 4 exponent bits with bias 7, 3 fraction bits), the storage element
// of 8-bit K/V caches.
struct e4m3 {
    uint8_t bits;
};

// Four E4M3 codes (bytes 0..3 of w, element order) -> two packed fp32 pairs, exactly: the
// hardware conversion to f16 pairs (every E4M3 value is an f16 value), then f16 -> f32.
__device__ __forceinline__ void widen4_e4m3(uint32_t w, uint64_t &p01, uint64_t &p23) {
    asm("{\n\t.reg .b16 lo, hi, a0, a1, a2, a3;\n\t.reg .b32 h0, h1;\n\t.reg .f32 f0, f1, f2, f3;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 h0, lo;\n\tcvt.rn.f16x2.e4m3x2 h1, hi;\n\t"
        "mov.b32 {a0, a1}, h0;\n\tmov.b32 {a2, a3}, h1;\n\t"
        "cvt.f32.f16 f0, a0;\n\tcvt.f32.f16 f1, a1;\n\tcvt.f32.f16 f2, a2;\n\tcvt.f32.f16 f3, a3;\n\t"
        "mov.b64 %0, {f0, f1};\n\tmov.b64 %1, {f2, f3};\n\t}"
        : "=l"(p01), "=l"(p23)
        : "r"(w));
}

// Four E4M3 codes (bytes 0..3 of w) -> two f16 pairs (elements 0, 1 and 2, 3), exactly.
__device__ __forceinline__ void e4m3x4_to_h2(uint32_t w, uint32_t &h01, uint32_t &h23) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(h01), "=r"(h23)
        : "r"(w));
}

// Mixed-precision FMAs with f16 operands and fp32 accumulators (products of f16 values are exact
// in fp32, so each step rounds once): d0 += a.lo * b.lo and d1 += a.hi * b.hi.
__device__ __forceinline__ void fma_h2(uint32_t a, uint32_t b, float &d0, float &d1) {
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %2;\n\tmov.b32 {b0, b1}, %3;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %0;\n\tfma.rn.f32.f16 %1, a1, b1, %1;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "r"(a), "r"(b));
}
// d0 += a.lo * s and d1 += a.hi * s for an f16 scalar s.
__device__ __forceinline__ void fma_h2s(uint32_t a, uint16_t s, float &d0, float &d1) {
    asm("{\n\t.reg .b16 a0, a1;\n\tmov.b32 {a0, a1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, %3, %0;\n\tfma.rn.f32.f16 %1, a1, %3, %1;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "r"(a), "h"(s));
}
// The same with bf16 operands: d0 += a.lo * b.lo and d1 += a.hi * b.hi (products exact in fp32).
__device__ __forceinline__ void fma_bf2(uint32_t a, uint32_t b, float &d0, float &d1) {
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %2;\n\tmov.b32 {b0, b1}, %3;\n\t"
        "fma.rn.f32.bf16 %0, a0, b0, %0;\n\tfma.rn.f32.bf16 %1, a1, b1, %1;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "r"(a), "r"(b));
}
// fp32 -> f16 (round to nearest even) and two fp32 -> one f16 pair (a in the low half).
__device__ __forceinline__ uint16_t f16_from_f32(float a) {
    uint16_t r;
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(r) : "f"(a));
    return r;
}
__device__ __forceinline__ uint32_t h2_from_f32(float a, float b) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}

// Two fp32 values -> two E4M3 codes (a in the low byte), rounded to nearest even with the
// magnitude saturated at 448.
__device__ __forceinline__ uint16_t e4m3x2_from_f32(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}

template <typename T, int NP>
__device__ __forceinline__ void load_pairs(const T *p, uint64_t (&out)[NP]) {
    if constexpr (sizeof(T) == 1) {            // E4M3 codes: 8-byte or 16-byte vectors
        static_assert((2 * NP) % 8 == 0, "8-byte vectors");
        if constexpr ((2 * NP) % 16 == 0) {
#pragma unroll
            for (int w = 0; w < NP / 8; ++w) {
                const uint4 v = reinterpret_cast<const uint4 *>(p)[w];
                widen4_e4m3(v.x, out[8 * w], out[8 * w + 1]);
                widen4_e4m3(v.y, out[8 * w + 2], out[8 * w + 3]);
                widen4_e4m3(v.z, out[8 * w + 4], out[8 * w + 5]);
                widen4_e4m3(v.w, out[8 * w + 6], out[8 * w + 7]);
            }
        } else {
#pragma unroll
            for (int w = 0; w < NP / 4; ++w) {
                const uint2 v = reinterpret_cast<const uint2 *>(p)[w];
                widen4_e4m3(v.x, out[4 * w], out[4 * w + 1]);
                widen4_e4m3(v.y, out[4 * w + 2], out[4 * w + 3]);
            }
        }
    } else if constexpr (sizeof(T) == 4) {
        static_assert((2 * NP * sizeof(T)) % 16 == 0, "16-byte vectors");
#pragma unroll
        for (int w = 0; w < NP / 2; ++w) {
            const uint4 v = reinterpret_cast<const uint4 *>(p)[w];
            out[2 * w] = (uint64_t)v.x | ((uint64_t)v.y << 32);
            out[2 * w + 1] = (uint64_t)v.z | ((uint64_t)v.w << 32);
        }
    } else {
        static_assert((2 * NP * sizeof(T)) % 16 == 0, "16-byte vectors");
#pragma unroll
        for (int w = 0; w < NP / 4; ++w) {
            const uint4 v = reinterpret_cast<const uint4 *>(p)[w];
            out[4 * w] = widen2<T>(v.x);
            out[4 * w + 1] = widen2<T>(v.y);
            out[4 * w + 2] = widen2<T>(v.z);
            out[4 * w + 3] = widen2<T>(v.w);
        }
    }
}

// ---- mbarrier ---------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete; false after kWaitTimeoutNs.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > kWaitTimeoutNs) return false;
    }
}

// ---- bulk (non-tensor) async copy global -> shared, completion on an mbarrier -------------------
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// ---- tiled tensor copy (TMA) global -> shared, completion on an mbarrier -----------------------
// `map` is a __grid_constant__ kernel parameter; c0 is the innermost coordinate (elements).
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
        : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before later async-proxy
// (bulk copy / tensor core) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

}  // namespace pkv
