// 2-bit paged KV cache with promoted 4-bit key channels ("KVキャッシュ管理の教科書", 第22章, on
// Kitty): the page quantiser and decode attention over quantised pages.  The record format and
// the readings taken where the chapter leaves a step open are in include/pagedkv.h.
//
// kitty_quantize_kernel: one CTA of 512 threads per (pair, KV head), the page's K and V staged in
// shared memory.  Thread x < 128 owns channel x for the statistics -- float32 magnitude sum over
// the tokens in order, min, max; the promoted set is the P channels of largest sum (rank by
// comparison with every other channel, ties to the lower id).  Codes by float32 subtract, divide
// and round-half-even, four threads per channel (a quarter of the tokens each); 16 channels' low
// bits meet in one word through shuffles, high bits through shared-memory ORs.  V: one warp per
// token, a lane per 4 channels, min/max by shuffles; the codes by a thread per (half page,
// channel, 16 tokens), packed channel-major per half page.
//
// kitty_decode_kernel: persistent, 16 warps per CTA (128 registers each), one CTA per SM.  Phase 1
// streams the quantised pages: a work item is (sequence, query head, up to kChunkPages pages);
// each warp runs a 2-stage ring of half pages (64 keys of one (page, KV head) record: the half's
// codes, V scales and minimums, and on the first half the K scales, minimums and promoted ids),
// filled by bulk copies with mbarrier completion, and claims its next item while the current one
// computes, so the ring runs across items.  Per page the warp folds each channel's scale into the
// query (a_x = scale * q_x * s_x, and b = scale * sum_x q_x min_x), so a key's score is
// b + sum_x a_x code_x, and puts a_x on a 16-bit integer grid (the page's largest |a_x| at
// 2^13..2^14).  The codes are never unpacked to floats: masking field j of a 32-bit word of codes
// in place leaves four bytes code * 4^j (<= 192), and dp2a multiplies two of them by two 16-bit
// weights and adds both to an int32 -- one AND per four codes and one instruction per two codes,
// exact sums, the 4^j divided out once per field.  QK^T: one lane per key, the weights as pairs in
// shared memory in the order of the masked bytes (channels j, 4 + j, 8 + j, 12 + j of a word); the
// promoted channels' high bits the same way, times 4 after the sum.  After one online-softmax
// step over the half's 64 keys, P times the token's V scale goes on the half's 16-bit grid (its
// largest at 2^13..2^14) in shared memory, in the order of the channel-major V words' bytes, and
// PV takes one lane per 4 channels the same way; the V minimum
// contributes sum_t p_t min_t.  Phase 2 runs each sequence's residual page (fewer than 128
// unquantised tokens) as one more item with plain loads.  Items of one row merge by the
// logsumexp rule: the last split to finish reads the others' (m, l, o) records through L2.  Every
// warp streams pages first and takes residual items when no page item is left.
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kPageTokens = 128;
constexpr int kDim = 128;
constexpr int kOffKs = 0, kOffKm = 512, kOffVs = 1024, kOffVm = 1536, kOffPid = 2048, kOffKlo = 2080;
constexpr int kOffKhi = kOffKlo + 32 * kPageTokens;               // 6176
constexpr int kChunkPages = 8;                                    // pages per decode work item
constexpr int kDecWarps = 16;
constexpr int kStages = 2;
constexpr int kPartFloats = 132;                                  // m, l, 2 pad, o[128]
constexpr int kMaxSeqs = 4096;
constexpr int kScratchBytes = 512 + 64 * 4 + 16 * 4;              // a_x fp32, f16 pairs lo, hi

__host__ __device__ constexpr int record_bytes(int P) { return 10272 + 32 * P; }
__host__ __device__ constexpr int off_vc(int P) { return kOffKhi + 32 * P; }
// A decode ring stage holds half a page (64 keys) of one record: K scales and minimums and the
// promoted ids (first half only), then the half's V scales, V minimums, K low bits, K high bits
// and V codes.
constexpr int kHsKs = 0, kHsKm = 512, kHsVs = 1024, kHsVm = 1280, kHsPid = 1536, kHsKlo = 1568, kHsKhi = 3616;
__host__ __device__ constexpr int hs_vc(int P) { return kHsKhi + 16 * P; }
__host__ __device__ constexpr int half_stage_bytes(int P) { return hs_vc(P) + 2048; }

// ---- quantiser ---------------------------------------------------------------------------------
struct QuantParams {
    const void *res_k, *res_v;
    const int64_t *pairs;
    uint8_t *pages;
    int64_t num_pairs, num_pages, num_res;
    int kv_heads;
    unsigned *status;
};

constexpr int kQThreads = 512;
constexpr int kQSmem = 2 * kPageTokens * kDim * 2;                // the page's K and V (16-bit)

template <typename T, int P>
__global__ void __launch_bounds__(kQThreads) kitty_quantize_kernel(QuantParams p) {
    constexpr int kHiWords = P / 16;                 // 32-bit words of high bits per token
    extern __shared__ __align__(16) unsigned char qsm[];
    T *s_k = reinterpret_cast<T *>(qsm);
    T *s_v = s_k + kPageTokens * kDim;
    __shared__ float s_mag[kDim], s_min[kDim], s_step[kDim];
    __shared__ int s_slot[kDim];                     // promoted slot of a channel, or -1
    __shared__ int s_cnt[4];
    __shared__ uint32_t s_hi[kPageTokens * kHiWords];
    __shared__ float s_vlo[kPageTokens], s_vsc[kPageTokens];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t pair = blockIdx.x;
    const int h = blockIdx.y;
    const int64_t src = p.pairs[2 * pair], dst = p.pairs[2 * pair + 1];
    if (src < 0 || src >= p.num_res || dst < 0 || dst >= p.num_pages) {
        if (tid == 0) report(p.status, PA_DEV_BAD_PAIR);
        return;
    }
    const size_t plane = (size_t)kPageTokens * kDim;
    const T *rk = reinterpret_cast<const T *>(p.res_k) + ((size_t)src * p.kv_heads + h) * plane;
    const T *rv = reinterpret_cast<const T *>(p.res_v) + ((size_t)src * p.kv_heads + h) * plane;
    uint8_t *rec = p.pages + ((size_t)dst * p.kv_heads + h) * record_bytes(P);
    for (int i = tid; i < kPageTokens * kHiWords; i += kQThreads) s_hi[i] = 0u;
    {
        constexpr int kVecs = kPageTokens * kDim * (int)sizeof(T) / 16;
        const uint4 *k4 = reinterpret_cast<const uint4 *>(rk), *v4 = reinterpret_cast<const uint4 *>(rv);
        uint4 *dk = reinterpret_cast<uint4 *>(s_k), *dv = reinterpret_cast<uint4 *>(s_v);
#pragma unroll
        for (int i = tid; i < kVecs; i += kQThreads) {
            dk[i] = __ldg(k4 + i);
            dv[i] = __ldg(v4 + i);
        }
    }
    __syncthreads();

    // K, one thread per channel x: magnitude sum (tokens in order), minimum and maximum in float32
    float mag = 0.f, mn = INFINITY, mx = -INFINITY;
    if (tid < kDim) {
        for (int t = 0; t < kPageTokens; ++t) {
            const float v = Elem<T>::to_f(s_k[t * kDim + tid]);
            mag = __fadd_rn(mag, fabsf(v));
            mn = fminf(mn, v);
            mx = fmaxf(mx, v);
        }
        s_mag[tid] = mag;
    }
    __syncthreads();
    if (tid < kDim) {
        // rank = channels ahead of this one (larger sum, or equal sum and lower id)
        int rank = 0;
        for (int y = 0; y < kDim; ++y) {
            const float my = s_mag[y];
            rank += (my > mag) || (my == mag && y < tid);
        }
        const bool prom = rank < P;
        const unsigned ball = __ballot_sync(0xffffffffu, prom);
        if (lane == 0) s_cnt[warp] = __popc(ball);
        s_slot[tid] = prom ? __popc(ball & ((1u << lane) - 1u)) : -1;
        const float L = prom ? 15.f : 3.f;
        const float st = __fdiv_rn(__fsub_rn(mx, mn), L);
        s_min[tid] = mn;
        s_step[tid] = st;
        reinterpret_cast<float *>(rec + kOffKs)[tid] = st;
        reinterpret_cast<float *>(rec + kOffKm)[tid] = mn;
    }
    __syncthreads();
    if (tid < kDim) {
        if (s_slot[tid] >= 0) {
            int slot = s_slot[tid];
            for (int w = 0; w < warp; ++w) slot += s_cnt[w];
            s_slot[tid] = slot;
            rec[kOffPid + slot] = (uint8_t)tid;
        }
        if (tid >= P && tid < 32) rec[kOffPid + tid] = 0;
    }
    __syncthreads();

    // K codes: thread (channel x, token quarter g); 16 channels' low bits form one word
    {
        const int x = tid & (kDim - 1), g = tid >> 7;
        const float mnx = s_min[x], sx = s_step[x];
        const int slot = s_slot[x];
        const float L = slot >= 0 ? 15.f : 3.f;
        for (int t = g * 32; t < g * 32 + 32; ++t) {
            const float v = Elem<T>::to_f(s_k[t * kDim + x]);
            uint32_t c = 0;
            if (sx != 0.f) c = (uint32_t)fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(v, mnx), sx)), 0.f), L);
            uint32_t w = (c & 3u) << (2 * (x & 15));
            w |= __shfl_xor_sync(0xffffffffu, w, 1);
            w |= __shfl_xor_sync(0xffffffffu, w, 2);
            w |= __shfl_xor_sync(0xffffffffu, w, 4);
            w |= __shfl_xor_sync(0xffffffffu, w, 8);
            if ((x & 15) == 0) reinterpret_cast<uint32_t *>(rec + kOffKlo + t * 32)[x >> 4] = w;
            if (slot >= 0) atomicOr(&s_hi[t * kHiWords + (slot >> 4)], (c >> 2) << (2 * (slot & 15)));
        }
    }

    // V scale and minimum: one warp per token, lane l reads channels 4l..4l+3
    for (int t = warp; t < kPageTokens; t += kQThreads / 32) {
        float v[4];
        load_f<T, 4>(s_v + t * kDim + 4 * lane, v);
        float lo = fminf(fminf(v[0], v[1]), fminf(v[2], v[3]));
        float hi = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        if (lane == 0) {
            const float sv = __fdiv_rn(__fsub_rn(hi, lo), 3.f);
            s_vlo[t] = lo;
            s_vsc[t] = sv;
            reinterpret_cast<float *>(rec + kOffVs)[t] = sv;
            reinterpret_cast<float *>(rec + kOffVm)[t] = lo;
        }
    }
    __syncthreads();
    // V codes, channel-major per half page: thread (half hf, channel x, word w) packs tokens
    // 64 hf + 16 w + i (i = 0..15) of channel x at bits 2 i of one 32-bit word
    for (int i = tid; i < 2 * kDim * 4; i += kQThreads) {
        const int w = i & 3, x = (i >> 2) & (kDim - 1), hf = i >> 9;
        uint32_t word = 0;
#pragma unroll 4
        for (int k = 0; k < 16; ++k) {
            const int t = 64 * hf + 16 * w + k;
            const float sv = s_vsc[t];
            uint32_t c = 0;
            if (sv != 0.f)
                c = (uint32_t)fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(Elem<T>::to_f(s_v[t * kDim + x]), s_vlo[t]), sv)),
                                          0.f), 3.f);
            word |= c << (2 * k);
        }
        reinterpret_cast<uint32_t *>(rec + off_vc(P) + 2048 * hf + 16 * x)[w] = word;
    }
    __syncthreads();
    for (int i = tid; i < kPageTokens * kHiWords; i += kQThreads)
        reinterpret_cast<uint32_t *>(rec + kOffKhi)[i] = s_hi[i];
}

// ---- decode attention ----------------------------------------------------------------------
struct DecParams {
    const void *q;
    const uint8_t *pages;
    const void *res_k, *res_v;
    const int32_t *bt, *ctx, *qlen;
    void *out;
    float scale_log2;                  // scale * log2(e): scores in log2 units
    int num_seqs, q_heads, kv_heads, group, max_pages, max_chunks;
    int64_t num_pages, num_res;
    uint32_t *counters;                // [0] next quantised item, [1] next residual item
    uint32_t *arrive;                  // [num_seqs * q_heads] splits finished per row
    float *parts;                      // [rows * max_chunks * kPartFloats] split records
    unsigned *status;
};

__device__ __forceinline__ float wsum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// 2^e for e in [-126, 127].
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

// The binary exponent of a positive finite float (its value in [2^e, 2^(e+1))), or -127 for 0
// and subnormals.
__device__ __forceinline__ int exponent_of(float a) { return ((__float_as_int(a) >> 23) & 0xff) - 127; }

// Tokens of sequence s (cached + the new one), or -1 when its lengths are invalid.
__device__ __forceinline__ int seq_tokens(const DecParams &p, int s) {
    const int c = __ldg(p.ctx + s), ql = __ldg(p.qlen + s);
    if (ql != 1 || c < 0 || (int64_t)c + 1 > (int64_t)p.max_pages * kPageTokens) return -1;
    return c + 1;
}

__device__ __forceinline__ int quant_chunks(int n) {
    return n <= 0 ? 0 : (n / kPageTokens + kChunkPages - 1) / kChunkPages;
}

struct Item {
    int seq, h, kvh, k, p0, p1, nch;
    bool valid;
};

// Claims the next quantised-page item: items are numbered sequence by sequence (prefix s_cu),
// within a sequence head-major, so the chunks of one row are claimed back to back.
__device__ __forceinline__ Item claim_quant(const DecParams &p, const int *s_cu, int lane) {
    Item it;
    it.valid = false;
    uint32_t i = 0;
    if (lane == 0) i = atomicAdd(p.counters, 1u);
    i = __shfl_sync(0xffffffffu, i, 0);
    if (i >= (uint32_t)s_cu[p.num_seqs]) return it;
    int lo = 0, hi = p.num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((uint32_t)s_cu[mid] <= i) lo = mid;
        else hi = mid - 1;
    }
    const int n = seq_tokens(p, lo);
    const int nq = quant_chunks(n);
    const int w = (int)i - s_cu[lo];
    it.seq = lo;
    it.h = w / nq;
    it.k = w - it.h * nq;
    it.kvh = it.h / p.group;
    it.p0 = it.k * kChunkPages;
    it.p1 = min(it.p0 + kChunkPages, n / kPageTokens);
    it.nch = nq + (n % kPageTokens != 0);
    it.valid = true;
    return it;
}

// Called by a whole warp after it wrote split k's record of `row`.  The last of the row's nch
// splits to arrive merges them, out = sum_k 2^(m_k - M) o_k / sum_k 2^(m_k - M) l_k, and writes
// the output row (lane l: channels 4l..4l+3).
template <typename T>
__device__ void merge_row(const DecParams &p, int row, int nch, int lane) {
    __threadfence();
    __syncwarp();
    uint32_t before = 0;
    if (lane == 0) before = atomicAdd(p.arrive + row, 1u);
    before = __shfl_sync(0xffffffffu, before, 0);
    if (before != (uint32_t)(nch - 1)) return;
    __threadfence();
    const float *base = p.parts + (size_t)row * p.max_chunks * kPartFloats;
    float M = -INFINITY;
    for (int k = lane; k < nch; k += 32) M = fmaxf(M, __ldcg(base + (size_t)k * kPartFloats));
    M = warp_max(M);
    float L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int k = 0; k < nch; ++k) {
        const float *r = base + (size_t)k * kPartFloats;
        const float m = __ldcg(r), l = __ldcg(r + 1);
        const float4 o = __ldcg(reinterpret_cast<const float4 *>(r + 4) + lane);
        const float w = m == -INFINITY ? 0.f : exp2f(m - M);
        L = fmaf(w, l, L);
        acc[0] = fmaf(w, o.x, acc[0]);
        acc[1] = fmaf(w, o.y, acc[1]);
        acc[2] = fmaf(w, o.z, acc[2]);
        acc[3] = fmaf(w, o.w, acc[3]);
    }
    const float inv = 1.f / L;
    float v[4] = {acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv};
    store_f<T, 4>(reinterpret_cast<T *>(p.out) + (size_t)row * kDim + 4 * lane, v);
}

// Mixed-precision FMA on a pair of 16-bit elements of the query's type.
template <typename T> __device__ __forceinline__ void fma_pair(uint32_t a, uint32_t b, float &d0, float &d1);
template <> __device__ __forceinline__ void fma_pair<__nv_bfloat16>(uint32_t a, uint32_t b, float &d0, float &d1) {
    fma_bf2(a, b, d0, d1);
}
template <> __device__ __forceinline__ void fma_pair<__half>(uint32_t a, uint32_t b, float &d0, float &d1) {
    fma_h2(a, b, d0, d1);
}

// Residual-page items, one per (sequence, query head) whose length is not a multiple of 128: the
// last n % 128 tokens, unquantised, with plain loads (one lane per key for QK^T, one lane per 4
// channels for PV, 8 keys' V rows in flight).
template <typename T>
__device__ void tail_items(const DecParams &p, int lane) {
    const uint32_t rows = (uint32_t)p.num_seqs * p.q_heads;
    while (true) {
        uint32_t j = 0;
        if (lane == 0) j = atomicAdd(p.counters + 1, 1u);
        j = __shfl_sync(0xffffffffu, j, 0);
        if (j >= rows) break;
        const int seq = j / p.q_heads, h = j - seq * p.q_heads;
        const int n = seq_tokens(p, seq);
        if (n < 0 || n % kPageTokens == 0) continue;
        const int nt = n % kPageTokens, nfull = n / kPageTokens;
        const int nch = quant_chunks(n) + 1;
        const int32_t rid = __ldg(p.bt + (int64_t)seq * p.max_pages + nfull);
        float m_run = -INFINITY, l_l = 0.f;
        uint64_t o2[2] = {0ull, 0ull};               // channels 4 lane .. 4 lane + 3
        if (rid < 0 || rid >= p.num_res) {
            if (lane == 0) report(p.status, PA_DEV_BAD_BLOCK_ID);
        } else {
            const size_t plane = (size_t)kPageTokens * kDim;
            const T *rk = reinterpret_cast<const T *>(p.res_k) + ((size_t)rid * p.kv_heads + h / p.group) * plane;
            const T *rv = reinterpret_cast<const T *>(p.res_v) + ((size_t)rid * p.kv_heads + h / p.group) * plane;
            uint32_t qp[64];
            const uint4 *qsrc = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(p.q) + (size_t)j * kDim);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint4 w = __ldg(qsrc + i);
                qp[4 * i] = w.x, qp[4 * i + 1] = w.y, qp[4 * i + 2] = w.z, qp[4 * i + 3] = w.w;
            }
            for (int t0 = 0; t0 < nt; t0 += 32) {
                const int t = t0 + lane;
                float z = -INFINITY;
                if (t < nt) {
                    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                    const uint4 *kr = reinterpret_cast<const uint4 *>(rk + (size_t)t * kDim);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint4 w = __ldg(kr + i);
                        fma_pair<T>(qp[4 * i], w.x, acc[0], acc[1]);
                        fma_pair<T>(qp[4 * i + 1], w.y, acc[2], acc[3]);
                        fma_pair<T>(qp[4 * i + 2], w.z, acc[4], acc[5]);
                        fma_pair<T>(qp[4 * i + 3], w.w, acc[6], acc[7]);
                    }
                    z = (((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]))) * p.scale_log2;
                }
                const float mloc = warp_max(z);
                if (mloc > m_run) {
                    const float al = fast_exp2(m_run - mloc);
                    l_l *= al;
                    const uint64_t al2 = f2pack(al, al);
                    o2[0] = mul2(o2[0], al2);
                    o2[1] = mul2(o2[1], al2);
                    m_run = mloc;
                }
                const float pz = t < nt ? fast_exp2(z - m_run) : 0.f;
                l_l += pz;
                const int cnt = min(32, nt - t0);
                const T *vb = rv + (size_t)t0 * kDim + 4 * lane;
                // 8 keys' V rows in flight at once; rows past the tail (never read) may hold NaN
                for (int k0 = 0; k0 < cnt; k0 += 8) {
                    uint2 w[8];
                    float pk[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        pk[u] = __shfl_sync(0xffffffffu, pz, k0 + u);
                        w[u] = k0 + u < cnt ? __ldg(reinterpret_cast<const uint2 *>(vb + (size_t)(k0 + u) * kDim))
                                            : make_uint2(0u, 0u);
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint64_t pk2 = f2pack(pk[u], pk[u]);
                        o2[0] = fma2(widen2<T>(w[u].x), pk2, o2[0]);
                        o2[1] = fma2(widen2<T>(w[u].y), pk2, o2[1]);
                    }
                }
            }
        }
        const float l = wsum(l_l);
        float res[4];
        f2unpack(o2[0], res[0], res[1]);
        f2unpack(o2[1], res[2], res[3]);
        if (nch == 1) {
            if (rid >= 0 && rid < p.num_res) {
                const float inv = 1.f / l;
                float v[4] = {res[0] * inv, res[1] * inv, res[2] * inv, res[3] * inv};
                store_f<T, 4>(reinterpret_cast<T *>(p.out) + (size_t)j * kDim + 4 * lane, v);
            }
        } else {
            float *rec = p.parts + ((size_t)j * p.max_chunks + (nch - 1)) * kPartFloats;
            reinterpret_cast<float4 *>(rec + 4)[lane] = make_float4(res[0], res[1], res[2], res[3]);
            if (lane == 0) {
                rec[0] = m_run;
                rec[1] = l;
            }
            merge_row<T>(p, (int)j, nch, lane);
        }
    }
}

// 16-byte shared-memory load kept in place (volatile), so that the compiler does not hoist the
// a_x pairs of every word into registers across the passes.
__device__ __forceinline__ void lds128(uint32_t addr, uint32_t &a, uint32_t &b, uint32_t &c, uint32_t &d) {
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr));
}

// d = c + a.lo * b.byte0 + a.hi * b.byte1 (dp2a_lo) or with bytes 2, 3 (dp2a_hi): two signed 16-bit
// weights times two unsigned 8-bit codes, exact in int32.
__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Shared memory of the decode kernel: per warp kStages half-page stages and a scratch area, the
// ring's mbarriers, then the per-sequence item prefix.
__host__ __device__ constexpr size_t dec_smem_bytes(int P, int num_seqs) {
    return (size_t)kDecWarps * (kStages * half_stage_bytes(P) + kScratchBytes) + kDecWarps * kStages * 8 +
           (size_t)(num_seqs + 1) * 4;
}

template <typename T, int P>
__global__ void __launch_bounds__(kDecWarps * 32, 1) kitty_decode_kernel(DecParams p) {
    constexpr int REC = record_bytes(P);
    constexpr int HS = half_stage_bytes(P);
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_part[kDecWarps * 32];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned char *ring = smem + (size_t)warp * kStages * HS;
    unsigned char *scratch = smem + (size_t)kDecWarps * kStages * HS + warp * kScratchBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)kDecWarps * (kStages * HS + kScratchBytes)) +
                     warp * kStages;
    int *s_cu = reinterpret_cast<int *>(smem + (size_t)kDecWarps * (kStages * HS + kScratchBytes) +
                                        kDecWarps * kStages * 8);
    // per warp: the page's query weights on a 16-bit grid (channel order), the same as dp2a
    // pairs in the order of the unpacked low-bit and high-bit code bytes, and the half page's P
    // on a 16-bit grid in the order of the unpacked V code bytes
    int16_t *s_q16 = reinterpret_cast<int16_t *>(scratch);                 // [128]
    int16_t *s_wlo = reinterpret_cast<int16_t *>(scratch + 256);           // [8 words][4 fields][2][2]
    int16_t *s_whi = reinterpret_cast<int16_t *>(scratch + 512);           // [P / 16][4][2][2]
    int16_t *s_p16 = reinterpret_cast<int16_t *>(scratch + 576);           // [4 words][4][2][2]

    // item prefix over sequences: sequence s has quant_chunks(n_s) * q_heads quantised items
    {
        const int S = p.num_seqs;
        const int per = (S + kDecWarps * 32 - 1) / (kDecWarps * 32);
        const int lo = min(S, tid * per), hi = min(S, lo + per);
        int sum = 0;
        for (int s = lo; s < hi; ++s) {
            const int n = seq_tokens(p, s);
            if (n < 0 && blockIdx.x == 0) report(p.status, PA_DEV_BAD_LENGTHS);
            sum += quant_chunks(n) * p.q_heads;
        }
        s_part[tid] = sum;
        if (lane == 0) {
#pragma unroll
            for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
            mbar_fence_init();
        }
        __syncthreads();
        if (warp == 0) {
            int v[kDecWarps], t = 0;
#pragma unroll
            for (int i = 0; i < kDecWarps; ++i) {
                v[i] = s_part[lane * kDecWarps + i];
                t += v[i];
            }
            int incl = t;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            int run = incl - t;
#pragma unroll
            for (int i = 0; i < kDecWarps; ++i) {
                s_part[lane * kDecWarps + i] = run;
                run += v[i];
            }
            if (lane == 31) s_cu[S] = run;
        }
        __syncthreads();
        int run = s_part[tid];
        for (int s = lo; s < hi; ++s) {
            s_cu[s] = run;
            run += quant_chunks(seq_tokens(p, s)) * p.q_heads;
        }
        __syncthreads();
    }


    // ---- phase 1: quantised pages, streamed as half pages ----
    Item cur = claim_quant(p, s_cu, lane), nxt;
    nxt.valid = false;
    bool have_nxt = false, iss_nxt = false, dead = false;
    int iss_pg = cur.p0, iss_h = 0;
    uint32_t issued = 0, done = 0;

    auto page_id = [&](const Item &it, int pg) -> int64_t {
        const int32_t id = __ldg(p.bt + (int64_t)it.seq * p.max_pages + pg);
        return (id < 0 || id >= p.num_pages) ? -1 : id;
    };
    // Issues the copies of the next half page (of the current item, else of the next one, which
    // it claims when needed); false when there is nothing to issue.
    auto issue = [&]() -> bool {
        if (!cur.valid) return false;
        if (iss_pg >= (iss_nxt ? nxt.p1 : cur.p1)) {
            if (iss_nxt) return false;
            if (!have_nxt) {
                nxt = claim_quant(p, s_cu, lane);
                have_nxt = true;
            }
            if (!nxt.valid) return false;
            iss_nxt = true;
            iss_pg = nxt.p0;
            iss_h = 0;
        }
        const Item &it = iss_nxt ? nxt : cur;
        int64_t id = page_id(it, iss_pg);
        if (id < 0) id = 0;      // a bad id still fills the stage (the ring stays in step); compute skips it
        const int slot = issued % kStages;
        if (lane == 0) {
            const uint8_t *rec = p.pages + ((size_t)id * p.kv_heads + it.kvh) * REC;
            unsigned char *dst = ring + slot * HS;
            const uint32_t bytes = (iss_h == 0 ? 1056u : 0u) + 512u + 2048u + 16u * P + 2048u;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bars[slot], bytes);
            if (iss_h == 0) {
                bulk_g2s(dst + kHsKs, rec + kOffKs, 1024, &bars[slot]);          // K scales, minimums
                bulk_g2s(dst + kHsPid, rec + kOffPid, 32, &bars[slot]);
            }
            bulk_g2s(dst + kHsVs, rec + kOffVs + 256 * iss_h, 256, &bars[slot]);
            bulk_g2s(dst + kHsVm, rec + kOffVm + 256 * iss_h, 256, &bars[slot]);
            bulk_g2s(dst + kHsKlo, rec + kOffKlo + 2048 * iss_h, 2048, &bars[slot]);
            bulk_g2s(dst + kHsKhi, rec + kOffKhi + 16 * P * iss_h, 16 * P, &bars[slot]);
            bulk_g2s(dst + hs_vc(P), rec + off_vc(P) + 2048 * iss_h, 2048, &bars[slot]);
        }
        ++issued;
        if (++iss_h == 2) {
            iss_h = 0;
            ++iss_pg;
        }
        return true;
    };

    while (issued - done < kStages && issue()) {
    }
    while (cur.valid) {
        const int row = cur.seq * p.q_heads + cur.h;
        float qs[4];
        load_f<T, 4>(reinterpret_cast<const T *>(p.q) + (size_t)row * kDim + 4 * lane, qs);
#pragma unroll
        for (int e = 0; e < 4; ++e) qs[e] *= p.scale_log2;
        float m_run = -INFINITY, l_l = 0.f, bv_l = 0.f;
        // o[c]: channel 4 lane + ((c + vrot) & 3), units of 2^-F
        float o[4] = {0.f, 0.f, 0.f, 0.f};
        const int vrot = (lane >> 1) & 3;
        int F_cur = 0;
        bool have_F = false;
        float b = 0.f, zmul = 0.f;                  // of the current page, set by its first half

        for (int pg = cur.p0; pg < cur.p1 && !dead; ++pg) {
            const bool page_ok = page_id(cur, pg) >= 0;
            if (!page_ok && lane == 0) report(p.status, PA_DEV_BAD_BLOCK_ID);
            for (int hh = 0; hh < 2; ++hh) {
                const int slot = done % kStages;
                if (!mbar_wait(&bars[slot], (done / kStages) & 1u)) {
                    report(p.status, PA_DEV_TIMEOUT);
                    dead = true;
                    break;
                }
                const unsigned char *st = ring + slot * HS;
                if (page_ok) {
                    if (hh == 0) {
                        // page prologue: a_x = scale q_x s_x on a 16-bit grid, qi_x = rint(a_x 2^E)
                        // with E putting max |a| in [2^13, 2^14); b = scale sum_x q_x min_x
                        const float4 ks = reinterpret_cast<const float4 *>(st + kHsKs)[lane];
                        const float4 km = reinterpret_cast<const float4 *>(st + kHsKm)[lane];
                        const float a[4] = {qs[0] * ks.x, qs[1] * ks.y, qs[2] * ks.z, qs[3] * ks.w};
                        b = wsum(qs[0] * km.x + qs[1] * km.y + qs[2] * km.z + qs[3] * km.w);
                        const float amax =
                            warp_max(fmaxf(fmaxf(fabsf(a[0]), fabsf(a[1])), fmaxf(fabsf(a[2]), fabsf(a[3]))));
                        const int E = amax > 0.f ? max(-100, min(100, 13 - exponent_of(amax))) : 0;
                        const float sE = pow2f(E);
                        __syncwarp();                     // the previous page's weights are read
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            // channel x = 4 lane + e = 16 w + 4 a + e: byte a of field e of word w
                            const int16_t qi = (int16_t)__float2int_rn(a[e] * sE);
                            const int w = lane >> 2, aa = lane & 3;
                            s_q16[4 * lane + e] = qi;
                            s_wlo[2 * ((w * 4 + e) * 2 + (aa >> 1)) + (aa & 1)] = qi;
                        }
                        __syncwarp();
                        if (lane < P) {
                            // promoted slot k = lane: its high-bit weight (x 4 after the sums)
                            const int w = lane >> 4, i = lane & 15, aa = i >> 2, e = i & 3;
                            s_whi[2 * ((w * 4 + e) * 2 + (aa >> 1)) + (aa & 1)] = s_q16[st[kHsPid + lane]];
                        }
                        __syncwarp();
                        zmul = pow2f(-E);
                    }
                    const float *vsc = reinterpret_cast<const float *>(st + kHsVs);
                    const float *vmn = reinterpret_cast<const float *>(st + kHsVm);
                    const uint32_t wlo_a = smem_addr(s_wlo), whi_a = smem_addr(s_whi);

                    float z0, z1;                           // keys lane and 32 + lane of the half
                    {
                        // QK^T, two keys per lane (lane, 32 + lane) in one pass, so each weight pair
                        // loaded serves both keys: the codes unpacked to bytes (field j of a word
                        // holds channels j, 4 + j, 8 + j, 12 + j) meet the weight pairs in dp2a
                        // (exact int32).  Field j is masked in place, leaving bytes code * 4^j (<=
                        // 192), one accumulator per field and key; the 4^j is divided out exactly
                        // at the end
                        const uint4 *kl0 = reinterpret_cast<const uint4 *>(st + kHsKlo + lane * 32);
                        const uint4 *kl1 = reinterpret_cast<const uint4 *>(st + kHsKlo + (32 + lane) * 32);
                        int a0[4] = {0, 0, 0, 0}, a1[4] = {0, 0, 0, 0};
#pragma unroll
                        for (int hw4 = 0; hw4 < 2; ++hw4) {
                            const uint4 x0 = kl0[hw4], x1 = kl1[hw4];
                            const uint32_t k0w[4] = {x0.x, x0.y, x0.z, x0.w}, k1w[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const int wd = hw4 * 4 + q;
                                uint32_t wp[8];
                                lds128(wlo_a + wd * 32, wp[0], wp[1], wp[2], wp[3]);
                                lds128(wlo_a + wd * 32 + 16, wp[4], wp[5], wp[6], wp[7]);
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    const uint32_t m = 0x03030303u << (2 * j);
                                    const uint32_t u0 = k0w[q] & m, u1 = k1w[q] & m;
                                    a0[j] = dp2a_lo(wp[2 * j], u0, a0[j]);
                                    a1[j] = dp2a_lo(wp[2 * j], u1, a1[j]);
                                    a0[j] = dp2a_hi(wp[2 * j + 1], u0, a0[j]);
                                    a1[j] = dp2a_hi(wp[2 * j + 1], u1, a1[j]);
                                }
                            }
                        }
                        int h0[4] = {0, 0, 0, 0}, h1[4] = {0, 0, 0, 0};
                        uint32_t hv0[P / 16], hv1[P / 16];
                        if constexpr (P == 32) {
                            const uint2 y0 = *reinterpret_cast<const uint2 *>(st + kHsKhi + lane * 8);
                            const uint2 y1 = *reinterpret_cast<const uint2 *>(st + kHsKhi + (32 + lane) * 8);
                            hv0[0] = y0.x; hv0[1] = y0.y; hv1[0] = y1.x; hv1[1] = y1.y;
                        } else {
                            hv0[0] = *reinterpret_cast<const uint32_t *>(st + kHsKhi + lane * 4);
                            hv1[0] = *reinterpret_cast<const uint32_t *>(st + kHsKhi + (32 + lane) * 4);
                        }
#pragma unroll
                        for (int wd = 0; wd < P / 16; ++wd) {
                            uint32_t wp[8];
                            lds128(whi_a + wd * 32, wp[0], wp[1], wp[2], wp[3]);
                            lds128(whi_a + wd * 32 + 16, wp[4], wp[5], wp[6], wp[7]);
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const uint32_t m = 0x03030303u << (2 * j);
                                const uint32_t u0 = hv0[wd] & m, u1 = hv1[wd] & m;
                                h0[j] = dp2a_lo(wp[2 * j], u0, h0[j]);
                                h1[j] = dp2a_lo(wp[2 * j], u1, h1[j]);
                                h0[j] = dp2a_hi(wp[2 * j + 1], u0, h0[j]);
                                h1[j] = dp2a_hi(wp[2 * j + 1], u1, h1[j]);
                            }
                        }
                        const int d0 = (a0[0] + (a0[1] >> 2)) + ((a0[2] >> 4) + (a0[3] >> 6)) +
                                       4 * ((h0[0] + (h0[1] >> 2)) + ((h0[2] >> 4) + (h0[3] >> 6)));
                        const int d1 = (a1[0] + (a1[1] >> 2)) + ((a1[2] >> 4) + (a1[3] >> 6)) +
                                       4 * ((h1[0] + (h1[1] >> 2)) + ((h1[2] >> 4) + (h1[3] >> 6)));
                        z0 = fmaf((float)d0, zmul, b);
                        z1 = fmaf((float)d1, zmul, b);
                    }
                    // online softmax over the half's 64 keys (one max, so every P of the half
                    // refers to the same m_run), reduced together with the half's largest V
                    // token scale: F puts it in [2^13, 2^14); o is kept in units of 2^-F
                    float mloc = fmaxf(z0, z1), vmax = fmaxf(vsc[lane], vsc[lane + 32]);
#pragma unroll
                    for (int sh = 16; sh > 0; sh >>= 1) {
                        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, sh));
                        vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, sh));
                    }
                    const int F = vmax > 0.f ? max(-60, min(60, 13 - exponent_of(vmax))) : 0;
                    if (!have_F) {
                        F_cur = F;
                        have_F = true;
                    } else if (F != F_cur) {
                        const float r = pow2f(F - F_cur);
#pragma unroll
                        for (int i = 0; i < 4; ++i) o[i] *= r;
                        F_cur = F;
                    }
                    const float psc = pow2f(F_cur);
                    if (mloc > m_run) {
                        const float al = fast_exp2(m_run - mloc);
                        l_l *= al;
                        bv_l *= al;
#pragma unroll
                        for (int i = 0; i < 4; ++i) o[i] *= al;
                        m_run = mloc;
                    }
#pragma unroll
                    for (int pass = 0; pass < 2; ++pass) {
                        const int t = pass * 32 + lane;
                        const float pz = fast_exp2((pass == 0 ? z0 : z1) - m_run);
                        l_l += pz;
                        bv_l = fmaf(pz, vmn[t], bv_l);
                        // P times the V scale on the half page's 16-bit grid, stored where the V
                        // pair products want it: token t = 16 w + 4 a + j -> field j of word w, byte a
                        const int w = t >> 4, aa = (t >> 2) & 3, j = t & 3;
                        s_p16[2 * ((w * 4 + j) * 2 + (aa >> 1)) + (aa & 1)] =
                            (int16_t)__float2int_rn(pz * vsc[t] * psc);
                    }
                    __syncwarp();
                    // P V: lane l takes channels 4 l .. 4 l + 3 over the half's 64 tokens; a V word
                    // holds 16 tokens of one channel, field j of it tokens j, 4 + j, 8 + j, 12 + j
                    {
                        const uint4 *vc = reinterpret_cast<const uint4 *>(st + hs_vc(P) + 64 * lane);
                        uint32_t pp[32];
                        const uint32_t p_a = smem_addr(s_p16);
#pragma unroll
                        for (int i = 0; i < 8; ++i) lds128(p_a + 16 * i, pp[4 * i], pp[4 * i + 1], pp[4 * i + 2], pp[4 * i + 3]);
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            // the lane's c-th load is its word (c + vrot) & 3: neighbouring lanes
                            // start on different 16-byte words, so a load touches every bank
                            // four times instead of half the banks sixteen times
                            const uint4 v = vc[(c + vrot) & 3];
                            const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
                            int af[4] = {0, 0, 0, 0};       // per field j, in units of 4^j
#pragma unroll
                            for (int w = 0; w < 4; ++w)
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    const uint32_t u = vw[w] & (0x03030303u << (2 * j));
                                    af[j] = dp2a_lo(pp[(w * 4 + j) * 2], u, af[j]);
                                    af[j] = dp2a_hi(pp[(w * 4 + j) * 2 + 1], u, af[j]);
                                }
                            o[c] += (float)((af[0] + (af[1] >> 2)) + ((af[2] >> 4) + (af[3] >> 6)));
                        }
                    }
                }
                __syncwarp();
                ++done;
                issue();
            }
        }
        if (dead) break;

        // item epilogue: out[x] = (o[x] 2^-F + sum_t p_t min_t) / l for this lane's 4 channels
        const float l = wsum(l_l), bv = wsum(bv_l);
        const float f = pow2f(-F_cur);
        float res[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = (i - vrot) & 3;
            const float oc = c == 0 ? o[0] : c == 1 ? o[1] : c == 2 ? o[2] : o[3];
            res[i] = fmaf(oc, f, bv);
        }
        if (cur.nch == 1) {
            const float inv = 1.f / l;
            float v[4] = {res[0] * inv, res[1] * inv, res[2] * inv, res[3] * inv};
            store_f<T, 4>(reinterpret_cast<T *>(p.out) + (size_t)row * kDim + 4 * lane, v);
        } else {
            float *rec = p.parts + ((size_t)row * p.max_chunks + cur.k) * kPartFloats;
            reinterpret_cast<float4 *>(rec + 4)[lane] = make_float4(res[0], res[1], res[2], res[3]);
            if (lane == 0) {
                rec[0] = m_run;
                rec[1] = l;
            }
            merge_row<T>(p, row, cur.nch, lane);
        }

        // next item (claimed already if the ring ran ahead into it)
        if (!have_nxt) {
            nxt = claim_quant(p, s_cu, lane);
            have_nxt = true;
        }
        cur = nxt;
        have_nxt = false;
        if (iss_nxt) {
            iss_nxt = false;
        } else {
            iss_pg = cur.p0;
            iss_h = 0;
        }
        while (issued - done < kStages && issue()) {
        }
    }
    if (dead) {
        // drain this warp's copies in flight (bounded) and stop
        for (; done < issued; ++done) mbar_wait(&bars[done % kStages], (done / kStages) & 1u);
        return;
    }

    tail_items<T>(p, lane);
}

// ---- launchers ---------------------------------------------------------------------------------
constexpr int kMaxDevs = 64;

template <typename T, int P>
cudaError_t launch_decode_t(const DecParams &d, int num_sms, cudaStream_t s) {
    static bool configured[kMaxDevs];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevs) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(kitty_decode_kernel<T, P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)dec_smem_bytes(P, kMaxSeqs));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    kitty_decode_kernel<T, P><<<num_sms, kDecWarps * 32, dec_smem_bytes(P, d.num_seqs), s>>>(d);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_decode(const DecParams &d, int P, int num_sms, cudaStream_t s) {
    return P == 16 ? launch_decode_t<T, 16>(d, num_sms, s) : launch_decode_t<T, 32>(d, num_sms, s);
}

template <typename T, int P>
cudaError_t launch_quantize_t(const QuantParams &q, cudaStream_t s) {
    static bool configured[kMaxDevs];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevs) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(kitty_quantize_kernel<T, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const dim3 grid((unsigned)q.num_pairs, (unsigned)q.kv_heads);
    kitty_quantize_kernel<T, P><<<grid, kQThreads, kQSmem, s>>>(q);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_quantize(const QuantParams &q, int P, cudaStream_t s) {
    return P == 16 ? launch_quantize_t<T, 16>(q, s) : launch_quantize_t<T, 32>(q, s);
}

bool is_aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

pa_status check_kitty_dims(const pa_kitty_dims *d) {
    if (!d) return PA_ERR_INVALID_ARG;
    if (d->dtype != PA_BF16 && d->dtype != PA_F16) return d->dtype == PA_F32 ? PA_ERR_UNSUPPORTED : PA_ERR_INVALID_ARG;
    if (d->num_seqs < 1 || d->num_q_heads < 1 || d->num_kv_heads < 1 || d->max_pages_per_seq < 1)
        return PA_ERR_INVALID_ARG;
    if (d->num_q_heads % d->num_kv_heads) return PA_ERR_INVALID_ARG;
    if (d->num_pages < 0 || d->num_res_pages < 0) return PA_ERR_INVALID_ARG;
    if (d->head_dim != kDim || (d->promoted != 16 && d->promoted != 32)) return PA_ERR_UNSUPPORTED;
    if (d->num_seqs > kMaxSeqs) return PA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)d->num_seqs * d->num_q_heads;
    const int64_t chunks = ((int64_t)d->max_pages_per_seq + kChunkPages - 1) / kChunkPages + 1;
    if (rows * chunks >= ((int64_t)1 << 31)) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

struct KittyWs {
    size_t arrive, parts, zero_bytes, total;
    int max_chunks;
};

KittyWs kitty_ws(const pa_kitty_dims &d) {
    KittyWs w;
    const size_t rows = (size_t)d.num_seqs * d.num_q_heads;
    w.max_chunks = (d.max_pages_per_seq + kChunkPages - 1) / kChunkPages + 1;
    w.arrive = 256;
    w.parts = w.arrive + align_up(rows * 4, 256);
    w.zero_bytes = w.parts;
    w.total = w.parts + rows * w.max_chunks * kPartFloats * sizeof(float);
    return w;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

size_t pa_kitty_record_bytes(int32_t head_dim, int32_t promoted) {
    if (head_dim != kDim || (promoted != 16 && promoted != 32)) return 0;
    return (size_t)record_bytes(promoted);
}

size_t pa_kitty_workspace_size(const pa_kitty_dims *dims) {
    if (check_kitty_dims(dims) != PA_OK) return 0;
    return kitty_ws(*dims).total;
}

pa_status kv_quantize_pages(const pa_kitty_dims *dims, const void *res_k, const void *res_v,
                            const int64_t *pairs, int64_t num_pairs, void *pages, pa_stream_t stream) {
    // only the page geometry matters here (the decode fields may hold anything)
    if (!dims) return PA_ERR_INVALID_ARG;
    if (dims->dtype != PA_BF16 && dims->dtype != PA_F16)
        return dims->dtype == PA_F32 ? PA_ERR_UNSUPPORTED : PA_ERR_INVALID_ARG;
    if (dims->num_kv_heads < 1 || dims->num_pages < 0 || dims->num_res_pages < 0) return PA_ERR_INVALID_ARG;
    if (dims->head_dim != kDim || (dims->promoted != 16 && dims->promoted != 32)) return PA_ERR_UNSUPPORTED;
    if (num_pairs < 0 || num_pairs > 0x7fffffff) return PA_ERR_INVALID_ARG;
    if (num_pairs == 0) return PA_OK;
    if (!res_k || !res_v || !pairs || !pages) return PA_ERR_INVALID_ARG;
    if (!is_aligned(res_k, 16) || !is_aligned(res_v, 16) || !is_aligned(pages, 16) || !is_aligned(pairs, 8))
        return PA_ERR_INVALID_ARG;
    QuantParams q;
    q.res_k = res_k;
    q.res_v = res_v;
    q.pairs = pairs;
    q.pages = static_cast<uint8_t *>(pages);
    q.num_pairs = num_pairs;
    q.num_pages = dims->num_pages;
    q.num_res = dims->num_res_pages;
    q.kv_heads = dims->num_kv_heads;
    q.status = status_ptr();
    if (!q.status) return PA_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = dims->dtype == PA_BF16 ? launch_quantize<__nv_bfloat16>(q, dims->promoted, s)
                                                 : launch_quantize<__half>(q, dims->promoted, s);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_forward_kitty(const pa_kitty_dims *dims, const void *q, const void *pages,
                           const void *res_k, const void *res_v, const int32_t *block_tables,
                           const int32_t *ctx_lens, const int32_t *q_lens, float scale, void *out,
                           void *workspace, size_t workspace_bytes, pa_stream_t stream) {
    const pa_status st = check_kitty_dims(dims);
    if (st != PA_OK) return st;
    const pa_kitty_dims &d = *dims;
    if (!q || !pages || !res_k || !res_v || !block_tables || !ctx_lens || !q_lens || !out)
        return PA_ERR_INVALID_ARG;
    if (!is_aligned(q, 16) || !is_aligned(out, 16) || !is_aligned(pages, 16) || !is_aligned(res_k, 16) ||
        !is_aligned(res_v, 16))
        return PA_ERR_INVALID_ARG;
    if (!is_aligned(block_tables, 4) || !is_aligned(ctx_lens, 4) || !is_aligned(q_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
    const size_t row_bytes = (size_t)d.num_seqs * d.num_q_heads * kDim * 2;
    const char *qc = static_cast<const char *>(q), *oc = static_cast<const char *>(out);
    if (qc < oc + row_bytes && oc < qc + row_bytes) return PA_ERR_INVALID_ARG;
    const KittyWs w = kitty_ws(d);
    if (!workspace || workspace_bytes < w.total || !is_aligned(workspace, 256)) return PA_ERR_WORKSPACE;
    DecParams p;
    p.q = q;
    p.pages = static_cast<const uint8_t *>(pages);
    p.res_k = res_k;
    p.res_v = res_v;
    p.bt = block_tables;
    p.ctx = ctx_lens;
    p.qlen = q_lens;
    p.out = out;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.num_seqs = d.num_seqs;
    p.q_heads = d.num_q_heads;
    p.kv_heads = d.num_kv_heads;
    p.group = d.num_q_heads / d.num_kv_heads;
    p.max_pages = d.max_pages_per_seq;
    p.max_chunks = w.max_chunks;
    p.num_pages = d.num_pages;
    p.num_res = d.num_res_pages;
    char *ws = static_cast<char *>(workspace);
    p.counters = reinterpret_cast<uint32_t *>(ws);
    p.arrive = reinterpret_cast<uint32_t *>(ws + w.arrive);
    p.parts = reinterpret_cast<float *>(ws + w.parts);
    p.status = status_ptr();
    const int sms = sm_count();
    if (!p.status || sms <= 0) return PA_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, w.zero_bytes, s) != cudaSuccess) return PA_ERR_CUDA;
    const cudaError_t e = d.dtype == PA_BF16 ? launch_decode<__nv_bfloat16>(p, d.promoted, sms, s)
                                             : launch_decode<__half>(p, d.promoted, sms, s);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"
