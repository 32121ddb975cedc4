// Widening of E4M3 cache blocks for the tensor-core kernel.
//
// "KVキャッシュ管理の教科書" (第3章, 第22章) keeps the cache in fewer bits per element; a tcgen05
// MMA takes both operands in one 16-bit type, so the blocks of the sequences the planner gave the
// tensor-core kernel are widened first, once per call, into scratch blocks of the query dtype.
// Every E4M3 value is a bf16 and an f16 value, so the copy is exact and the scales stay outside
// it: the K scale joins the softmax scale and the V scale the output normalisation.
//
// Scratch block b belongs to the candidate sequence i with wid_cu[i] <= b < wid_cu[i+1] (block
// j = b - wid_cu[i] of its table); the kernel also writes the remapped table entry, so the
// tensor-core kernel reads block j of sequence i at scratch block b.  Persistent grid: CTAs
// stride over the scratch blocks, 16 codes per thread and step (16 bytes in, 32 out).
#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kWidenThreads = 256;

struct WidenParams {
    const uint8_t *k, *v;          // E4M3 caches
    char *wk, *wv;                 // widened blocks [cap][Hkv * B * d] of the query dtype
    const int32_t *bt;
    int32_t *wbt;                  // remapped block table [S, max_blocks]
    const int32_t *wid_cu;         // [S + 1]
    const int32_t *groups;         // planner: 0 marks a tensor-core sequence
    const uint32_t *counters;
    unsigned *status;
    int64_t num_blocks;            // physical blocks of the E4M3 caches
    int64_t bstride;               // codes between physical blocks
    int64_t blk_codes;             // Hkv * B * d
    int num_seqs, max_blocks;
};

// 16 E4M3 codes -> 16 elements of T (two 16-byte vectors), exactly.
template <typename T>
__device__ __forceinline__ void widen16(uint4 c, uint4 &lo, uint4 &hi);

template <>
__device__ __forceinline__ void widen16<__half>(uint4 c, uint4 &lo, uint4 &hi) {
    uint32_t h[8];
    e4m3x4_to_h2(c.x, h[0], h[1]);
    e4m3x4_to_h2(c.y, h[2], h[3]);
    e4m3x4_to_h2(c.z, h[4], h[5]);
    e4m3x4_to_h2(c.w, h[6], h[7]);
    lo = make_uint4(h[0], h[1], h[2], h[3]);
    hi = make_uint4(h[4], h[5], h[6], h[7]);
}

// E4M3 -> fp32 (exact, through f16) -> bf16 pairs (exact: at most 4 significant bits, exponents
// from 2^-9 to 2^8).
__device__ __forceinline__ uint32_t bf2_from_pair(uint64_t f01) {
    float a, b;
    f2unpack(f01, a, b);
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}

template <>
__device__ __forceinline__ void widen16<__nv_bfloat16>(uint4 c, uint4 &lo, uint4 &hi) {
    uint64_t p[8];
    widen4_e4m3(c.x, p[0], p[1]);
    widen4_e4m3(c.y, p[2], p[3]);
    widen4_e4m3(c.z, p[4], p[5]);
    widen4_e4m3(c.w, p[6], p[7]);
    lo = make_uint4(bf2_from_pair(p[0]), bf2_from_pair(p[1]), bf2_from_pair(p[2]), bf2_from_pair(p[3]));
    hi = make_uint4(bf2_from_pair(p[4]), bf2_from_pair(p[5]), bf2_from_pair(p[6]), bf2_from_pair(p[7]));
}

template <typename T>
__global__ void __launch_bounds__(kWidenThreads) widen_kernel(WidenParams p) {
    __shared__ int64_t s_src;
    const int64_t used = p.counters[kWidTotal];
    const int64_t vecs = p.blk_codes / 16;
    for (int64_t b = blockIdx.x; b < used; b += gridDim.x) {
        if (threadIdx.x == 0) {
            // owner: the last sequence i with wid_cu[i] <= b
            int lo = 0, hi = p.num_seqs - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if ((int64_t)__ldg(p.wid_cu + mid) <= b) lo = mid;
                else hi = mid - 1;
            }
            const int j = (int)(b - __ldg(p.wid_cu + lo));
            int64_t src = -1;
            if (__ldg(p.groups + lo) == 0) {   // a tensor-core sequence (its blocks all fit)
                src = __ldg(p.bt + (int64_t)lo * p.max_blocks + j);
                const bool bad = src < 0 || src >= p.num_blocks;
                if (bad) report(p.status, PA_DEV_BAD_BLOCK_ID);
                p.wbt[(int64_t)lo * p.max_blocks + j] = bad ? -1 : (int32_t)b;
                if (bad) src = -1;
            }
            s_src = src;
        }
        __syncthreads();
        const int64_t src = s_src;
        __syncthreads();   // s_src is rewritten by the next block's owner search
        if (src < 0) continue;
        const uint4 *ks = reinterpret_cast<const uint4 *>(p.k + src * p.bstride);
        const uint4 *vs = reinterpret_cast<const uint4 *>(p.v + src * p.bstride);
        uint4 *kd = reinterpret_cast<uint4 *>(p.wk + b * p.blk_codes * (int64_t)sizeof(T));
        uint4 *vd = reinterpret_cast<uint4 *>(p.wv + b * p.blk_codes * (int64_t)sizeof(T));
        for (int64_t e = threadIdx.x; e < vecs; e += kWidenThreads) {
            const uint4 kc = __ldg(ks + e), vc = __ldg(vs + e);
            uint4 lo, hi;
            widen16<T>(kc, lo, hi);
            kd[2 * e] = lo;
            kd[2 * e + 1] = hi;
            widen16<T>(vc, lo, hi);
            vd[2 * e] = lo;
            vd[2 * e + 1] = hi;
        }
    }
}

}  // namespace

cudaError_t launch_widen(const FwdArgs &a, cudaStream_t s) {
    const pa_dims &d = a.dims;
    WidenParams p;
    p.k = static_cast<const uint8_t *>(a.k);
    p.v = static_cast<const uint8_t *>(a.v);
    p.wk = static_cast<char *>(a.wid_k);
    p.wv = static_cast<char *>(a.wid_v);
    p.bt = a.bt;
    p.wbt = a.wid_bt;
    p.wid_cu = a.wid_cu;
    p.groups = reinterpret_cast<const int32_t *>(a.ws + a.lay.groups);
    p.counters = reinterpret_cast<const uint32_t *>(a.ws + a.lay.counters);
    p.status = a.status;
    p.num_blocks = d.num_blocks;
    p.blk_codes = (int64_t)d.num_kv_heads * d.block_size * d.head_dim;
    p.bstride = d.kv_block_stride ? d.kv_block_stride : p.blk_codes;
    p.num_seqs = d.num_seqs;
    p.max_blocks = d.max_blocks_per_seq;
    // blocks are 16 x 16 x 128 codes at least: a few CTAs per SM keep the copy streaming
    const unsigned grid = (unsigned)a.num_sms * 4;
    if (d.dtype == PA_F16) widen_kernel<__half><<<grid, kWidenThreads, 0, s>>>(p);
    else widen_kernel<__nv_bfloat16><<<grid, kWidenThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv
