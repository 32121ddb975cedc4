// Generalized paged attention for multi-token turns on the 5th-generation tensor cores (tcgen05).
//
// Method: softmax(QK^T / sqrt(d_k)) V over each sequence's cached-plus-new keys with a causal
// mask ("SOSP 2023論文解説: PagedAttention", section "PagedAttentionアルゴリズム";
// "Stateful Large Language Model Serving with Pensieve", section "汎化PagedAttentionカーネル":
// ragged multi-token queries against non-contiguous KV blocks, masking fused so no score matrix
// is written out).  Scores are computed tile by tile with an online softmax
// ("KVキャッシュ管理の教科書" 第6章, FlashAttention's tiling in on-chip memory).
//
// One work item is a tile of 128 query rows of one sequence and one KV head.  Rows are
// (token, head-in-GQA-group) pairs, so the g query heads sharing a KV head are packed into the
// same tile (M = 128 even for short turns with GQA).  Per 128-key tile:
//   S = Q K^T   (tcgen05.mma, M=N=128, K=d=128, bf16/f16 -> fp32 in tensor memory)
//   P = exp2(S * scale * log2 e - m), rows masked causally on diagonal tiles only
//   O += P V    (tcgen05.mma, P from shared memory, V MN-major, O accumulates in tensor memory)
// The running max is only moved (and O rescaled in tensor memory) when it grows by more than
// 2^8, so most tiles skip the rescale; the final O / l is exact either way.
//
// Warp roles (192 threads, one CTA per SM, persistent over the tile list):
//   warp 0      TMA producer: Q tile once per item; K and V tiles gathered block by block through
//               the block table, one 3-D box (64 columns x B rows of one (block, head)) per copy,
//               128-byte swizzled, two stages each for K and V.
//   warp 1      MMA issuer (one lane) and tensor-memory owner; zeroes V rows past the last key of
//               a sequence's final tile (those slots may hold anything, NaN included).
//   warps 2-5   softmax: one thread per tile row (tensor-memory lane), P to shared memory in the
//               UMMA K-major 128-byte-swizzled layout, lazy O rescale, epilogue O / l -> out.
// Every wait is bounded; on a timeout the role reports PA_DEV_TIMEOUT and stops, the kernel
// drains what it issued, frees its tensor memory and returns.
#include <cuda.h>
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kRows = 128;          // query rows per tile (UMMA M)
constexpr int kKeys = 128;          // keys per KV tile (UMMA N of QK^T, K of PV)
constexpr int kDim = 128;           // head_dim
constexpr int kPanel = 128 * 128;   // bytes of one 64-column panel of a 128-row tile (16 KiB)
constexpr int kTile = 2 * kPanel;   // one 128 x 128 16-bit tile (32 KiB)
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS0 = 0, kTmemS1 = 128, kTmemO = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows > 2^8

// shared-memory map (offsets from a 1024-byte aligned base)
constexpr int kSmQ = 0;
constexpr int kSmK = kSmQ + kTile;          // 2 stages
constexpr int kSmV = kSmK + 2 * kTile;      // 2 stages
constexpr int kSmP = kSmV + 2 * kTile;
constexpr int kSmBar = kSmP + kTile;
constexpr int kSmBytes = kSmBar + 256 + 1024;   // barriers, tensor-memory slot, alignment slack

enum Bar {
    kQFull = 0, kQEmpty, kKFull0, kKFull1, kKEmpty0, kKEmpty1, kVFull0, kVFull1, kVEmpty0, kVEmpty1,
    kSFull0, kSFull1, kPFull, kOReady, kDrain, kNumBars
};

// ---- tcgen05 / TMA wrappers -----------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
        : "memory");
}

// Shared-memory matrix descriptor: 128-byte swizzle, version 1 (tcgen05).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate, A and B bf16 (or both f16), A K-major,
// B K-major or MN-major, M = N = 128.
__host__ __device__ constexpr uint32_t instr_desc(bool b_mn_major, bool f16) {
    return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) |
           ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(128 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                     uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

#define PKV_R32(x)                                                                               \
    "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]),         \
        "=r"(x[7]), "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]),  \
        "=r"(x[14]), "=r"(x[15]), "=r"(x[16]), "=r"(x[17]), "=r"(x[18]), "=r"(x[19]),            \
        "=r"(x[20]), "=r"(x[21]), "=r"(x[22]), "=r"(x[23]), "=r"(x[24]), "=r"(x[25]),            \
        "=r"(x[26]), "=r"(x[27]), "=r"(x[28]), "=r"(x[29]), "=r"(x[30]), "=r"(x[31])
#define PKV_W32(x)                                                                               \
    "r"(x[0]), "r"(x[1]), "r"(x[2]), "r"(x[3]), "r"(x[4]), "r"(x[5]), "r"(x[6]), "r"(x[7]),     \
        "r"(x[8]), "r"(x[9]), "r"(x[10]), "r"(x[11]), "r"(x[12]), "r"(x[13]), "r"(x[14]),        \
        "r"(x[15]), "r"(x[16]), "r"(x[17]), "r"(x[18]), "r"(x[19]), "r"(x[20]), "r"(x[21]),      \
        "r"(x[22]), "r"(x[23]), "r"(x[24]), "r"(x[25]), "r"(x[26]), "r"(x[27]), "r"(x[28]),      \
        "r"(x[29]), "r"(x[30]), "r"(x[31])

// 32 consecutive fp32 columns of this thread's tensor-memory lane (load and wait in one asm so
// no use of the registers can be scheduled before the data has arrived).
__device__ __forceinline__ void tmem_load32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "{\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
        "%30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t}"
        : PKV_R32(r)
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_store32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "{\n\t"
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
        "%29, %30, %31, %32};\n\t"
        "tcgen05.wait::st.sync.aligned;\n\t}" ::"r"(taddr),
        PKV_W32(r)
        : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename T> __device__ __forceinline__ uint32_t pack2(float a, float b);
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}
template <> __device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Bounded wait by a whole warp; the outcome is made warp-uniform so that no warp-collective
// tcgen05 instruction can run with part of the warp after a timeout.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) {
    const bool ok = mbar_wait(bar, parity);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ int find_rank(const int32_t *a, int n, int key) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(a + mid) <= key) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

struct TcParams {
    char *out;
    const int32_t *bt, *ctx, *qlen;
    const int32_t *cu_q, *tc_cu, *tc_seq;
    const uint32_t *counters;
    unsigned *status;
    int64_t num_blocks;
    float scale_log2;
    int num_seqs, q_heads, kv_heads, group, block_size, max_blocks;
};

struct Item {
    int seq, kvh, j0, rows_valid, ntiles;
    int64_t tok0, pmin, pmax;
};

__device__ __forceinline__ Item decode_item(const TcParams &p, int it) {
    Item t;
    const int rank = find_rank(p.tc_cu, p.num_seqs, it);
    t.seq = __ldg(p.tc_seq + rank);
    const int local = it - __ldg(p.tc_cu + rank);
    const int rows = __ldg(p.qlen + t.seq) * p.group;
    const int tph = (rows + kRows - 1) / kRows;
    const int qt = tph - 1 - (local % tph);  // a sequence's last (longest) query tile first
    t.kvh = local / tph;
    t.j0 = qt * (kRows / p.group);
    t.rows_valid = min(kRows, rows - qt * kRows);
    t.tok0 = __ldg(p.cu_q + t.seq);
    const int64_t c = __ldg(p.ctx + t.seq);
    t.pmin = c + t.j0;
    t.pmax = c + t.j0 + (t.rows_valid - 1) / p.group;
    t.ntiles = (int)((t.pmax + kKeys) / kKeys);
    return t;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    tc_attention_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, TcParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kSmBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kSmBar + kNumBars * 8);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr bool kF16 = std::is_same<T, __half>::value;
    const uint32_t idesc_qk = instr_desc(false, kF16);
    const uint32_t idesc_pv = instr_desc(true, kF16);

    if (threadIdx.x == 0) {
        for (int b = 0; b < kNumBars; ++b) mbar_init(&bars[b], b == kPFull ? 4 : 1);
        mbar_fence_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int total = (int)p.counters[kTcTotal];
    const int B = p.block_size;
    const int bpt = kKeys / B;   // blocks per KV tile

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        uint32_t kv_iter = 0, items = 0;
        uint32_t armed_k[2] = {0, 0}, armed_v[2] = {0, 0}, armed_q = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < total && ok; it += gridDim.x, ++items) {
            const Item t = decode_item(p, it);
            if (items > 0 && !warp_wait(&bars[kQEmpty], (items - 1) & 1)) { ok = false; break; }
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars[kQFull], kTile);
                const int y = t.kvh * p.group;
                const int z = (int)(t.tok0 + t.j0);
                tma_load_3d(smem + kSmQ, &qmap, 0, y, z, &bars[kQFull]);
                tma_load_3d(smem + kSmQ + kPanel, &qmap, 64, y, z, &bars[kQFull]);
            }
            ++armed_q;
            const int32_t *bt_row = p.bt + (int64_t)t.seq * p.max_blocks;
            for (int kt = 0; kt < t.ntiles; ++kt, ++kv_iter) {
                const int s = kv_iter & 1;
                const int64_t key0 = (int64_t)kt * kKeys;
                const int64_t keys = min((int64_t)kKeys, t.pmax + 1 - key0);
                const int nblk = (int)((keys + B - 1) / B);
                int phys = 0;
                if (lane < nblk) {
                    phys = __ldg(bt_row + (int64_t)kt * bpt + lane);
                    if (phys < 0 || (int64_t)phys >= p.num_blocks) {
                        report(p.status, PA_DEV_BAD_BLOCK_ID);
                        phys = (int)p.num_blocks;   // out of the tensor map: the copy fills zeros
                    }
                }
                const uint32_t bytes = (uint32_t)nblk * B * 128 * 2;
                if (kv_iter >= 2 && !warp_wait(&bars[kKEmpty0 + s], ((kv_iter >> 1) - 1) & 1)) { ok = false; break; }
                if (lane == 0) mbar_arrive_expect_tx(&bars[kKFull0 + s], bytes);
                __syncwarp();
                if (lane < nblk) {
                    unsigned char *dst = smem + kSmK + s * kTile + lane * B * 128;
                    tma_load_3d(dst, &kmap, 0, t.kvh * B, phys, &bars[kKFull0 + s]);
                    tma_load_3d(dst + kPanel, &kmap, 64, t.kvh * B, phys, &bars[kKFull0 + s]);
                }
                ++armed_k[s];
                if (kv_iter >= 2 && !warp_wait(&bars[kVEmpty0 + s], ((kv_iter >> 1) - 1) & 1)) { ok = false; break; }
                if (lane == 0) mbar_arrive_expect_tx(&bars[kVFull0 + s], bytes);
                __syncwarp();
                if (lane < nblk) {
                    unsigned char *dst = smem + kSmV + s * kTile + lane * B * 128;
                    tma_load_3d(dst, &vmap, 0, t.kvh * B, phys, &bars[kVFull0 + s]);
                    tma_load_3d(dst + kPanel, &vmap, 64, t.kvh * B, phys, &bars[kVFull0 + s]);
                }
                ++armed_v[s];
            }
        }
        if (!ok && lane == 0) report(p.status, PA_DEV_TIMEOUT);
        // every copy this warp issued lands before the CTA can exit
        for (int s = 0; s < 2; ++s) {
            if (armed_k[s]) mbar_wait(&bars[kKFull0 + s], (armed_k[s] - 1) & 1);
            if (armed_v[s]) mbar_wait(&bars[kVFull0 + s], (armed_v[s] - 1) & 1);
        }
        if (armed_q) mbar_wait(&bars[kQFull], (armed_q - 1) & 1);
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        uint32_t kv_iter = 0, items = 0;
        bool ok = true;
        const uint32_t q_addr = smem_addr(smem + kSmQ);
        const uint32_t p_addr = smem_addr(smem + kSmP);
        auto issue_s = [&](uint32_t g) -> bool {
            const int s = g & 1;
            if (!warp_wait(&bars[kKFull0 + s], (g >> 1) & 1)) return false;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t k_addr = smem_addr(smem + kSmK + s * kTile);
                const uint32_t d_tmem = tmem + (s ? kTmemS1 : kTmemS0);
#pragma unroll
                for (int k = 0; k < kDim / 16; ++k) {
                    const uint32_t off = (k >> 2) * kPanel + (k & 3) * 32;
                    umma(d_tmem, smem_desc(q_addr + off, 16, 1024), smem_desc(k_addr + off, 16, 1024),
                         idesc_qk, k > 0);
                }
                umma_commit(&bars[kSFull0 + s]);
                umma_commit(&bars[kKEmpty0 + s]);
            }
            __syncwarp();
            return true;
        };
        for (int it = blockIdx.x; it < total && ok; it += gridDim.x, ++items) {
            const Item t = decode_item(p, it);
            if (!warp_wait(&bars[kQFull], items & 1)) { ok = false; break; }
            tc_fence_after();
            if (!issue_s(kv_iter)) { ok = false; break; }
            for (int kt = 0; kt < t.ntiles; ++kt) {
                const uint32_t g = kv_iter + kt;
                if (kt + 1 < t.ntiles) {
                    if (!issue_s(g + 1)) { ok = false; break; }
                } else if (lane == 0) {
                    umma_commit(&bars[kQEmpty]);      // Q is free once every S of the item is done
                }
                __syncwarp();
                if (!warp_wait(&bars[kPFull], g & 1)) { ok = false; break; }
                const int s = g & 1;
                if (!warp_wait(&bars[kVFull0 + s], (g >> 1) & 1)) { ok = false; break; }
                // zero V rows past the last key any row of this tile sees (free or stale slots)
                const int64_t valid = t.pmax + 1 - (int64_t)kt * kKeys;
                if (valid < kKeys) {
                    unsigned char *vb = smem + kSmV + s * kTile;
                    const int first = (int)valid;
                    const int n16 = (kKeys - first) * 8;            // 16-byte chunks per panel
                    for (int i = lane; i < 2 * n16; i += 32) {
                        const int panel = i / n16, rem = i - panel * n16;
                        *reinterpret_cast<uint4 *>(vb + panel * kPanel + first * 128 + rem * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t v_addr = smem_addr(smem + kSmV + s * kTile);
#pragma unroll
                    for (int k = 0; k < kKeys / 16; ++k) {
                        const uint32_t a_off = (k >> 2) * kPanel + (k & 3) * 32;
                        umma(tmem + kTmemO, smem_desc(p_addr + a_off, 16, 1024),
                             smem_desc(v_addr + k * 16 * 128, kPanel, 1024), idesc_pv,
                             (kt > 0 || k > 0) ? 1u : 0u);
                    }
                    umma_commit(&bars[kOReady]);
                    umma_commit(&bars[kVEmpty0 + s]);
                }
                __syncwarp();
            }
            kv_iter += t.ntiles;
        }
        if (!ok && lane == 0) report(p.status, PA_DEV_TIMEOUT);
        // no tensor-core work of this CTA may be in flight when its tensor memory is freed
        if (lane == 0) umma_commit(&bars[kDrain]);
        __syncwarp();
        mbar_wait(&bars[kDrain], 0);
    } else {
        // ------------------------------------------------------------------ softmax warps
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        unsigned char *pbase = smem + kSmP;
        uint32_t kv_iter = 0, pv_seen = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
            const Item t = decode_item(p, it);
            int64_t prow = t.pmin + row / p.group;
            if (prow > t.pmax) prow = t.pmax;             // padding rows: finite, never stored
            float m = -INFINITY, l = 0.f;
            for (int kt = 0; kt < t.ntiles; ++kt) {
                const uint32_t g = kv_iter + kt;
                const int s = g & 1;
                if (!warp_wait(&bars[kSFull0 + s], (g >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                float x[kKeys];
#pragma unroll
                for (int c = 0; c < kKeys / 32; ++c) {
                    uint32_t r[32];
                    tmem_load32(lane_base + (s ? kTmemS1 : kTmemS0) + c * 32, r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(r[i]) * p.scale_log2;
                }
                const int64_t key0 = (int64_t)kt * kKeys;
                if (key0 + kKeys - 1 > t.pmin) {           // diagonal tile: causal mask
                    const int64_t lim = prow - key0;       // visible columns: 0 .. lim
#pragma unroll
                    for (int i = 0; i < kKeys; ++i)
                        if (i > lim) x[i] = -INFINITY;
                }
                float mt = x[0];
#pragma unroll
                for (int i = 1; i < kKeys; ++i) mt = fmaxf(mt, x[i]);
                const float mnew = fmaxf(m, mt);
                const bool rescale = mnew > m + kRescaleThreshold;
                const float muse = rescale ? mnew : m;
                if (kt > 0) {
                    // PV of the previous tile must be done: it reads P, and O may be rescaled
                    if (!warp_wait(&bars[kOReady], pv_seen & 1)) { ok = false; break; }
                    ++pv_seen;
                    tc_fence_after();
                    // tensor-memory loads/stores are warp-collective: the whole warp rescales
                    // when any of its rows must (alpha = 1 for the others)
                    if (__any_sync(0xffffffffu, rescale)) {
                        const float alpha = rescale ? fast_exp2(m - muse) : 1.f;
                        l *= alpha;
#pragma unroll 1
                        for (int c = 0; c < kDim / 32; ++c) {
                            uint32_t r[32];
                            tmem_load32(lane_base + kTmemO + c * 32, r);
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                            tmem_store32(lane_base + kTmemO + c * 32, r);
                        }
                    }
                }
                m = muse;
                // P = exp2(x - m) -> 16-bit, into the K-major swizzled A tile of the PV product
#pragma unroll
                for (int c16 = 0; c16 < kKeys / 8; ++c16) {
                    float e[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        e[i] = fast_exp2(x[c16 * 8 + i] - m);
                        l += e[i];
                    }
                    uint4 v;
                    v.x = pack2<T>(e[0], e[1]);
                    v.y = pack2<T>(e[2], e[3]);
                    v.z = pack2<T>(e[4], e[5]);
                    v.w = pack2<T>(e[6], e[7]);
                    const int panel = c16 >> 3, chunk = (c16 & 7) ^ (row & 7);
                    *reinterpret_cast<uint4 *>(pbase + panel * kPanel + row * 128 + chunk * 16) = v;
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kPFull]);
            }
            if (!ok) break;
            // epilogue: O / l -> out
            if (!warp_wait(&bars[kOReady], pv_seen & 1)) { ok = false; break; }
            ++pv_seen;
            tc_fence_after();
            const float inv = 1.f / l;
            const bool store = row < t.rows_valid;
            const int j = t.j0 + row / p.group, hh = row % p.group;
            T *orow = reinterpret_cast<T *>(p.out) +
                      ((t.tok0 + j) * p.q_heads + (int64_t)t.kvh * p.group + hh) * kDim;
#pragma unroll 1
            for (int c = 0; c < kDim / 32; ++c) {
                uint32_t r[32];
                tmem_load32(lane_base + kTmemO + c * 32, r);
                if (store) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 v;
                        v.x = pack2<T>(__uint_as_float(r[q4 * 8 + 0]) * inv, __uint_as_float(r[q4 * 8 + 1]) * inv);
                        v.y = pack2<T>(__uint_as_float(r[q4 * 8 + 2]) * inv, __uint_as_float(r[q4 * 8 + 3]) * inv);
                        v.z = pack2<T>(__uint_as_float(r[q4 * 8 + 4]) * inv, __uint_as_float(r[q4 * 8 + 5]) * inv);
                        v.w = pack2<T>(__uint_as_float(r[q4 * 8 + 6]) * inv, __uint_as_float(r[q4 * 8 + 7]) * inv);
                        *reinterpret_cast<uint4 *>(orow + c * 32 + q4 * 8) = v;
                    }
                }
            }
            tc_fence_before();
            kv_iter += t.ntiles;
        }
        if (!ok && lane == 0) report(p.status, PA_DEV_TIMEOUT);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

// ---- host: tensor maps ----------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

bool make_map(CUtensorMap *map, int dtype, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
              uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b1, uint32_t b2) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {s1_bytes, s2_bytes};
    const cuuint32_t box[3] = {64, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(map, dtype == PA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                           3, const_cast<void *>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool tc_shape_supported(const pa_dims &d) {
    if (d.dtype != PA_BF16 && d.dtype != PA_F16) return false;
    if (d.head_dim != kDim) return false;
    const int g = d.num_q_heads / d.num_kv_heads;
    if (g < 1 || g > kRows || (kRows % g) != 0) return false;
    if (d.block_size < 16 || d.block_size > kKeys) return false;
    if (d.num_blocks >= (int64_t(1) << 31) - 1 || d.total_q >= (int64_t(1) << 31)) return false;
    return encode_fn() != nullptr;
}

cudaError_t launch_tc(const FwdArgs &a, cudaStream_t s) {
    const pa_dims &d = a.dims;
    const int g = d.num_q_heads / d.num_kv_heads;
    const uint64_t es = 2;
    const int64_t bstride = d.kv_block_stride ? d.kv_block_stride
                                              : (int64_t)d.num_kv_heads * d.block_size * d.head_dim;
    CUtensorMap qmap, kmap, vmap;
    if (!make_map(&qmap, d.dtype, a.q, kDim, d.num_q_heads, d.total_q, kDim * es,
                  (uint64_t)d.num_q_heads * kDim * es, g, kRows / g) ||
        !make_map(&kmap, d.dtype, a.k, kDim, (uint64_t)d.num_kv_heads * d.block_size, d.num_blocks,
                  kDim * es, bstride * es, d.block_size, 1) ||
        !make_map(&vmap, d.dtype, a.v, kDim, (uint64_t)d.num_kv_heads * d.block_size, d.num_blocks,
                  kDim * es, bstride * es, d.block_size, 1))
        return cudaErrorInvalidValue;
    TcParams p;
    const WsLayout &L = a.lay;
    p.out = static_cast<char *>(a.out);
    p.bt = a.bt;
    p.ctx = a.ctx;
    p.qlen = a.qlen;
    p.cu_q = reinterpret_cast<const int32_t *>(a.ws + L.cu_q);
    p.tc_cu = reinterpret_cast<const int32_t *>(a.ws + L.tc_cu);
    p.tc_seq = reinterpret_cast<const int32_t *>(a.ws + L.tc_seq);
    p.counters = reinterpret_cast<const uint32_t *>(a.ws + L.counters);
    p.status = a.status;
    p.num_blocks = d.num_blocks;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.num_seqs = d.num_seqs;
    p.q_heads = d.num_q_heads;
    p.kv_heads = d.num_kv_heads;
    p.group = g;
    p.block_size = d.block_size;
    p.max_blocks = d.max_blocks_per_seq;
    cudaError_t e;
    if (d.dtype == PA_F16) {
        e = cudaFuncSetAttribute(tc_attention_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmBytes);
        if (e != cudaSuccess) return e;
        tc_attention_kernel<__half><<<a.num_sms, kThreads, kSmBytes, s>>>(qmap, kmap, vmap, p);
    } else {
        e = cudaFuncSetAttribute(tc_attention_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmBytes);
        if (e != cudaSuccess) return e;
        tc_attention_kernel<__nv_bfloat16><<<a.num_sms, kThreads, kSmBytes, s>>>(qmap, kmap, vmap, p);
    }
    return cudaGetLastError();
}

}  // namespace pkv
