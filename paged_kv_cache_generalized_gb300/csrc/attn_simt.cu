// Generalized paged attention on CUDA cores: the device-side planner and the split-KV work-item
// kernels (the last split of a row group to finish merges the group's partial results).
//
// Method: softmax(QK^T / sqrt(d_k)) V evaluated block by block through the block table
// ("SOSP 2023論文解説: PagedAttention", section "PagedAttentionアルゴリズム", blockwise A_j and
// o = sum_j A_j V_j), for ragged multi-token queries with a causal mask over cached-plus-new
// positions ("Stateful Large Language Model Serving with Pensieve", section
// "汎化PagedAttentionカーネル").  The softmax is computed online with a running max and sum,
// and a sequence's KV range may be split across work items whose partial (max, sum, weighted V)
// triples are merged with the logsumexp rule L = m + log(l) ("KVキャッシュ管理の教科書", 第6章,
// FlashAttention-2's statistics).
//
// GB300 design: one warp owns one work item (a KV head, up to R query rows of one sequence that
// share it, and a range of KV blocks).  The warp streams its K/V through a private ring of
// shared-memory stages filled by asynchronous copies with mbarrier completion, so each SM keeps
// ~200 KB of HBM reads in flight.  Work items are taken from a global counter (persistent grid).
// Three kernels: simt_attention_kernel for one query row per KV head (MHA decode; half-warps
// take alternate keys, each lane holds d/16 dimensions, reductions are warp shuffles, one bulk
// copy per 16-token run of a (block, head)), simt_gqa_kernel for 2 or 4 rows (below), and
// gqa_mma_kernel, which takes those GQA rows instead for 16-bit caches with head_dim 128
// (tensor-core fragments).  The CUDA-core kernels read K/V caches of the query's dtype or of
// one-byte E4M3 codes (the scales fold into the query scale and into o).  On E4M3 caches the one-row kernel converts the codes to f16 pairs in hardware and
// feeds them, with an f16 copy of the query (scaled by a power of two) or of P, to mixed-precision
// FMAs with fp32 accumulators: no f16 -> fp32 widening per element.
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "kv_append.cuh"

namespace pkv {
namespace {

constexpr int kStageTokens = 16;       // keys per pipeline stage
constexpr int kSimtMaxWarps = 8;

// ----------------------------------------------------------------------------------------------
// Planner (one CTA).  Reads q_lens/ctx_lens on the device, so no host round trip is needed.
// ----------------------------------------------------------------------------------------------
struct PlanParams {
    const int32_t *ctx;
    const int32_t *qlen;
    uint32_t *counters;
    int32_t *cu_q, *simt_cu, *parts_cu, *comb_cu, *groups, *nchunk, *tc_cu, *tc_seq;
    uint32_t *unit_cnt;
    uint32_t *tc_arrive;               // chunk arrival counters (when the workspace holds them)
    int32_t *wid_cu;                   // E4M3 widening: prefix of candidate sequences' blocks
    unsigned *status;
    int64_t total_q;
    int64_t max_parts;
    int64_t wid_cap;                   // widened blocks the scratch holds; -1: no widening (16-bit caches)
    int num_seqs, kv_heads, group, block_size, max_blocks, rows, tc, total_warps, tc_chunk_ok;
};

constexpr int kPlanThreads = 1024;
constexpr int kPlanAppendUnroll = 2;

// In-place exclusive scan of a[0..n) (a[n] receives the total), one CTA.
__device__ int64_t block_exclusive_scan(int32_t *a, int n) {
    __shared__ int64_t warp_sums[32];
    __shared__ int64_t carry_sh;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry_sh = 0;
    __syncthreads();
    for (int base = 0; base < n; base += kPlanThreads) {
        const int i = base + tid;
        int64_t v = i < n ? a[i] : 0;
        int64_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int64_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int64_t w = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int64_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_sums[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const int64_t carry = carry_sh;
        const int64_t before = (warp ? warp_sums[warp - 1] : 0) + x - v;
        if (i < n) a[i] = (int32_t)(carry + before);
        __syncthreads();
        if (tid == 0) carry_sh = carry + warp_sums[31];
        __syncthreads();
    }
    const int64_t total = carry_sh;
    if (tid == 0) a[n] = (int32_t)total;
    __syncthreads();
    return total;
}

// Block 0 plans; with a fused append (pa_forward_append) the other blocks write the step's new
// tokens into the caches meanwhile, so the attention kernels launched after this one read them.
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanParams p, AppendParams ap) {
    if (blockIdx.x > 0) {   // the fused cache append (two units per thread fit 64 registers)
        append_loop<kPlanAppendUnroll>(ap, blockIdx.x - 1, gridDim.x - 1);
        return;
    }
    __shared__ int64_t red[32];
    const int tid = threadIdx.x;
    const int S = p.num_seqs;
    if (tid < kNumCounters) p.counters[tid] = 0;
    // pass A: exclusive prefix of q_lens (the caller's packing of q and out)
    for (int i = tid; i < S; i += kPlanThreads) p.cu_q[i] = max(p.qlen[i], 0);
    __syncthreads();
    const int64_t total = block_exclusive_scan(p.cu_q, S);
    const bool packing_ok = (total == p.total_q);
    if (!packing_ok && tid == 0) report(p.status, PA_DEV_BAD_LENGTHS);

    // pass B0 (E4M3 caches): the blocks each tensor-core candidate would widen, in sequence
    // order; a candidate takes the tensor-core kernel when all of its blocks fit the scratch
    if (p.wid_cap >= 0) {
        for (int i = tid; i < S; i += kPlanThreads) {
            const int c = p.ctx[i], q = p.qlen[i];
            const int64_t n = (int64_t)c + q;
            const int64_t nb = (n + p.block_size - 1) / p.block_size;
            const bool valid = packing_ok && q >= 1 && c >= 0 && nb <= p.max_blocks && n <= kMaxSeqTokens;
            p.wid_cu[i] = (valid && p.tc && (int64_t)q * p.group >= kTcMinRows) ? (int32_t)nb : 0;
        }
        __syncthreads();
        const int64_t wtotal = block_exclusive_scan(p.wid_cu, S);
        if (tid == 0) p.counters[kWidTotal] = (uint32_t)(wtotal < p.wid_cap ? wtotal : p.wid_cap);
    }

    // pass B: classify sequences, total CUDA-core work (block-heads) for the split size
    int64_t work = 0;
    for (int i = tid; i < S; i += kPlanThreads) {
        const int c = p.ctx[i], q = p.qlen[i];
        const int64_t n = (int64_t)c + q;
        const int64_t nb = (n + p.block_size - 1) / p.block_size;
        const bool valid = packing_ok && q >= 1 && c >= 0 && nb <= p.max_blocks && n <= kMaxSeqTokens;
        if (packing_ok && !valid) report(p.status, PA_DEV_BAD_LENGTHS);
        int path = 0;
        if (valid) {
            const bool fits = p.wid_cap < 0 || (int64_t)p.wid_cu[i] + nb <= p.wid_cap;
            path = (p.tc && (int64_t)q * p.group >= kTcMinRows && fits) ? 2 : 1;
        }
        const int64_t rows = (int64_t)q * p.group;
        const int G = path == 1 ? (int)((rows + p.rows - 1) / p.rows) : 0;
        p.groups[i] = path == 0 ? -1 : G;    // -1 marks an invalid sequence
        p.nchunk[i] = path == 2 ? 0 : 1;
        if (path == 1) work += (int64_t)p.kv_heads * G * nb;
    }
    // block reduce of work
    {
        int64_t w = work;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
        if ((tid & 31) == 0) red[tid >> 5] = w;
        __syncthreads();
        if (tid < 32) {
            w = red[tid];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
            if (tid == 0) red[0] = w;
        }
        __syncthreads();
        work = red[0];
        __syncthreads();
    }
    // about 16 work items per warp slot of the persistent grid
    int64_t target = (int64_t)p.total_warps * 16;
    if (target > kMaxTargetItems) target = kMaxTargetItems;
    int64_t chunk = (work + target - 1) / (target > 0 ? target : 1);
    // at least kMinSplitTokens keys per split, so a warp's pipeline fill and its partial record
    // stay small next to the keys it streams
    const int64_t min_chunk = (kMinSplitTokens + p.block_size - 1) / p.block_size;
    if (chunk < min_chunk) chunk = min_chunk;
    if (tid == 0) p.counters[kChunkBlocks] = (uint32_t)chunk;

    // pass C: per-sequence counts
    for (int i = tid; i < S; i += kPlanThreads) {
        const int G = p.groups[i];
        int32_t items = 0, parts = 0, comb = 0;
        if (G > 0) {
            const int64_t n = (int64_t)p.ctx[i] + p.qlen[i];
            const int64_t nb = (n + p.block_size - 1) / p.block_size;
            // only sequences whose rows fit one row group are split (decode steps); longer
            // turns already spread over their row groups
            int K = 1;
            if (G == 1) {
                int64_t c_i = chunk;
                const int64_t min_c = (nb + kMaxSplits - 1) / kMaxSplits;
                if (c_i < min_c) c_i = min_c;
                K = (int)((nb + c_i - 1) / c_i);
            }
            p.nchunk[i] = K;
            items = p.kv_heads * G * K;
            if (K > 1) {
                parts = items;
                comb = p.kv_heads * G * p.rows;
            }
        }
        p.simt_cu[i] = items;
        p.parts_cu[i] = parts;
        p.comb_cu[i] = comb;
    }
    __syncthreads();
    const int64_t n_items = block_exclusive_scan(p.simt_cu, S);
    const int64_t n_parts = block_exclusive_scan(p.parts_cu, S);
    const int64_t n_comb = block_exclusive_scan(p.comb_cu, S);
    if (n_parts > p.max_parts) {
        // cannot happen with the workspace bound; refuse rather than overflow
        if (tid == 0) report(p.status, PA_DEV_BAD_LENGTHS);
        if (tid == 0) {
            p.counters[kSimtTotal] = 0;
            p.counters[kCombTotal] = 0;
        }
    } else {
        if (tid == 0) {
            p.counters[kSimtTotal] = (uint32_t)n_items;
            p.counters[kCombTotal] = (uint32_t)n_comb;
        }
        // arrival counters of the split row groups
        const int64_t n_units = n_comb / p.rows;
        for (int64_t u = tid; u < n_units; u += kPlanThreads) p.unit_cnt[u] = 0;
    }

    // tensor-core tiles: sequences ranked by descending length (longest first), ties by index
    if (p.tc) {
        for (int i = tid; i < S; i += kPlanThreads) p.tc_seq[i] = -1;
        __syncthreads();
        const bool rank_by_len = S <= 4096;
        for (int i = tid; i < S; i += kPlanThreads) {
            if (p.groups[i] < 0 || p.nchunk[i] != 0) continue;   // not a tensor-core sequence
            const int64_t ni = (int64_t)p.ctx[i] + p.qlen[i];
            int rank = 0;
            for (int k = 0; k < S; ++k) {
                if (p.groups[k] < 0 || p.nchunk[k] != 0) continue;
                if (rank_by_len) {
                    const int64_t nk = (int64_t)p.ctx[k] + p.qlen[k];
                    if (nk > ni || (nk == ni && k < i)) ++rank;
                } else if (k < i) {
                    ++rank;
                }
            }
            p.tc_seq[rank] = i;
        }
        __syncthreads();
        // pair items (one per KV head and pair of query tiles) of each ranked sequence
        for (int r = tid; r < S; r += kPlanThreads) {
            const int i = p.tc_seq[r];
            int32_t pairs = 0;
            if (i >= 0) {
                const int64_t rows = (int64_t)p.qlen[i] * p.group;
                const int64_t tph = (rows + kTcTileRows - 1) / kTcTileRows;
                pairs = p.kv_heads * (int32_t)((tph + kTcTilesPerItem - 1) / kTcTilesPerItem);
            }
            p.tc_cu[r] = pairs;
        }
        __syncthreads();
        int64_t n_items = block_exclusive_scan(p.tc_cu, S);
        // Fewer pair items than CTAs: split each pair's key range into chunks of about lc KV
        // tiles, so that the chunks fill the grid (at most one per CTA and kMaxTcChunkItems in
        // all).  The KV tile count of every distinct pair (the same for each KV head) goes to
        // shared memory, then warp 0 searches the chunk length.
        __shared__ int s_lc;
        __shared__ int s_nt[kMaxTcChunkItems];
        const int ctas = p.total_warps / 8;   // the tensor-core grid: one CTA per SM
        const int cap = ctas < kMaxTcChunkItems ? ctas : kMaxTcChunkItems;
        const bool few = p.tc_chunk_ok && n_items > 0 && n_items < cap;   // block-uniform
        if (tid == 0) s_lc = 0;
        if (few) {
            for (int r = tid; r < S; r += kPlanThreads) {
                const int i = p.tc_seq[r];
                if (i < 0) continue;
                const int rows = p.qlen[i] * p.group;
                const int pph = ((rows + kTcTileRows - 1) / kTcTileRows + 1) / 2;
                const int at = p.tc_cu[r] / p.kv_heads;             // the sequence's first pair
                for (int pi = 0; pi < pph; ++pi) s_nt[at + pi] = tc_pair_tiles(p.ctx[i], rows, p.group, pi);
            }
        }
        __syncthreads();
        if (few && tid < 32) {
            const int npairs = (int)(n_items / p.kv_heads);
            auto items_for = [&](int len) -> int64_t {   // items with chunk length len (0: KV tiles)
                int64_t n = 0;
                for (int k = tid; k < npairs; k += 32) n += len > 0 ? tc_pair_chunks(s_nt[k], len) : s_nt[k];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
                return n * p.kv_heads;
            };
            const int64_t tiles = items_for(0);
            int64_t lo = (tiles + cap - 1) / cap;
            if (lo < kTcMinChunkTiles) lo = kTcMinChunkTiles;
            // the shortest chunk length whose items fit (items never grow with the length; long
            // enough, every pair is one chunk and fits)
            int64_t hi = lo;
            while (items_for((int)hi) > cap) hi *= 2;
            if (hi > lo) {
                lo = hi / 2;                              // items_for(lo) > cap >= items_for(hi)
                while (hi - lo > 1) {
                    const int64_t mid = (lo + hi) / 2;
                    if (items_for((int)mid) > cap) lo = mid;
                    else hi = mid;
                }
            }
            const int64_t chunked = items_for((int)hi);   // every lane takes part in the sums
            if (tid == 0 && chunked > n_items) s_lc = (int)hi;
        }
        __syncthreads();
        if (tid == 0) p.counters[kTcChunk] = (uint32_t)s_lc;
        const int lc = s_lc;
        if (lc > 0) {
            for (int r = tid; r < S; r += kPlanThreads) {
                const int i = p.tc_seq[r];
                int32_t items = 0;
                if (i >= 0) {
                    const int rows = p.qlen[i] * p.group;
                    const int pph = ((rows + kTcTileRows - 1) / kTcTileRows + 1) / 2;
                    for (int pi = 0; pi < pph; ++pi)
                        items += tc_pair_chunks(tc_pair_tiles(p.ctx[i], rows, p.group, pi), lc);
                    items *= p.kv_heads;
                }
                p.tc_cu[r] = items;
            }
            for (int k = tid; k < kMaxTcChunkItems * 8; k += kPlanThreads) p.tc_arrive[k] = 0u;
            __syncthreads();
            n_items = block_exclusive_scan(p.tc_cu, S);
        }
        if (tid == 0) p.counters[kTcTotal] = (uint32_t)n_items;
    }
}

// Last index k in [0, n) with a[k] <= key (a is a non-decreasing prefix array of n+1 entries
// and key < a[n]).
__device__ __forceinline__ int find_owner(const int32_t *a, int n, int key) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(a + mid) <= key) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// ----------------------------------------------------------------------------------------------
// Work-item kernel
// ----------------------------------------------------------------------------------------------
struct SimtParams {
    const char *q;
    const char *k;
    const char *v;
    char *out;
    const int32_t *bt, *ctx, *qlen;
    const int32_t *cu_q, *simt_cu, *parts_cu, *comb_cu, *groups, *nchunk;
    uint32_t *counters;
    uint32_t *unit_cnt;
    float2 *parts_ml;
    float *parts_o;
    unsigned *status;
    int64_t num_blocks, block_stride;   // elements
    float scale_log2;                   // scale * log2(e) (* k_scale for E4M3 caches)
    float v_scale;                      // 1, or the V scale of E4M3 caches
    int num_seqs, q_heads, kv_heads, group, block_size, max_blocks, nst, bar_bytes;
};

// A split whose partial records are written but not yet counted in: a warp counts itself in (and
// merges, if it is the group's last) only after it has issued the first copies of its next item,
// so that the merge's latency overlaps them.
struct PendingSplit {
    int seq, kvh, grp, G, K, r0, nrows;
    int64_t tok0;
    bool on;
};

// Called by a whole warp after it wrote the partial records (m, l, o) of its split of row group
// (seq, kvh, grp).  The last of the group's K splits to get here merges the K records of every
// row with the logsumexp rule, out = sum_k 2^(m_k - M) o_k / sum_k 2^(m_k - M) l_k,
// M = max_k m_k, and writes the output rows; the others return at once.  Each writer fences its
// records before it counts itself in; the merger fences after it and reads through L2.
template <typename T, int D, int R>
__device__ __forceinline__ void finish_split(const SimtParams &p, int seq, int kvh, int grp, int G, int K,
                                             int r0, int nrows, int64_t tok0, int lane) {
    constexpr int EO = D / 32;                     // output dims per lane
    const int64_t unit = (int64_t)__ldg(p.comb_cu + seq) / R + (int64_t)kvh * G + grp;
    __threadfence();
    __syncwarp();
    uint32_t before = 0;
    if (lane == 0) before = atomicAdd(p.unit_cnt + unit, 1u);
    before = __shfl_sync(0xffffffffu, before, 0);
    if (before != (uint32_t)(K - 1)) return;
    __threadfence();
    const int64_t part0 = (int64_t)__ldg(p.parts_cu + seq) + ((int64_t)kvh * G + grp) * K;
    // lane k (and k + 32) reads split k's (m, l) of every row, then every row's weights and
    // denominators follow from warp reductions; the rows' o records of one split are read in the
    // same step, so R loads (times the unroll) are in flight at once
    float w0[R], w1[R], inv[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const bool ok = r < nrows;
        const float2 a0 = ok && lane < K ? __ldcg(p.parts_ml + (part0 + lane) * R + r)
                                         : make_float2(-INFINITY, 0.f);
        const float2 a1 = ok && lane + 32 < K ? __ldcg(p.parts_ml + (part0 + lane + 32) * R + r)
                                              : make_float2(-INFINITY, 0.f);
        const float M = warp_max(fmaxf(a0.x, a1.x));
        w0[r] = a0.x == -INFINITY ? 0.f : exp2f(a0.x - M);
        w1[r] = a1.x == -INFINITY ? 0.f : exp2f(a1.x - M);
        float L = w0[r] * a0.y + w1[r] * a1.y;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        inv[r] = 1.f / L;
    }
    float acc[R][EO];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int e = 0; e < EO; ++e) acc[r][e] = 0.f;
    const float *po = p.parts_o + part0 * R * D + lane * EO;
#pragma unroll 4
    for (int k = 0; k < K; ++k) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float w = __shfl_sync(0xffffffffu, k < 32 ? w0[r] : w1[r], k & 31);
            float x[EO];
            if (r < nrows) {
                const float *src = po + ((int64_t)k * R + r) * D;
                if constexpr (EO == 4) {
                    const float4 v = __ldcg(reinterpret_cast<const float4 *>(src));
                    x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
                } else {
                    const float2 v = __ldcg(reinterpret_cast<const float2 *>(src));
                    x[0] = v.x, x[1] = v.y;
                }
            } else {
#pragma unroll
                for (int e = 0; e < EO; ++e) x[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < EO; ++e) acc[r][e] = fmaf(w, x[e], acc[r][e]);
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (r >= nrows) continue;
        const int row = r0 + r;
        const int j = row / p.group, hh = row - j * p.group;
        T *op = reinterpret_cast<T *>(p.out) + ((tok0 + j) * p.q_heads + (int64_t)kvh * p.group + hh) * D +
                lane * EO;
#pragma unroll
        for (int e = 0; e < EO; ++e) op[e] = Elem<T>::from_f(acc[r][e] * inv[r]);
    }
}

template <typename T, typename TK, int D, int R>
__global__ void __launch_bounds__(kSimtMaxWarps * 32) simt_attention_kernel(SimtParams p) {
    constexpr int E = D / 16;                       // dims per lane
    // E4M3 caches: codes become f16 pairs in hardware and meet the query (as f16) in
    // mixed-precision FMAs with fp32 accumulators; no f16 -> fp32 conversion per element
    constexpr bool kE4 = sizeof(TK) == 1;
    static_assert(!kE4 || E == 8, "E4M3 caches: head_dim 128");
    constexpr uint32_t kRunBytes = kStageTokens * D * sizeof(TK);
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = lane >> 4, sub = lane & 15;
    const int NST = p.nst;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem) + warp * NST;
    unsigned char *ring = smem + p.bar_bytes + (size_t)warp * NST * 2 * kRunBytes;
    if (lane == 0) {
        for (int s = 0; s < NST; ++s) mbar_init(&bars[s], 1);
        mbar_fence_init();
    }
    __syncwarp();

    const int B = p.block_size;
    const int spb = B / kStageTokens;               // stages per block
    uint32_t issued = 0, consumed = 0;               // ring positions (persist across items)
    const uint32_t total_items = p.counters[kSimtTotal];
    PendingSplit pend;
    pend.on = false;

    while (true) {
        int item = 0;
        if (lane == 0) item = (int)atomicAdd(&p.counters[kSimtNext], 1u);
        item = __shfl_sync(0xffffffffu, item, 0);
        if ((uint32_t)item >= total_items) break;

        const int seq = find_owner(p.simt_cu, p.num_seqs, item);
        const int local = item - __ldg(p.simt_cu + seq);
        const int K = __ldg(p.nchunk + seq);
        const int G = __ldg(p.groups + seq);
        const int chunk = local % K;
        const int rest = local / K;
        const int grp = rest % G;
        const int kvh = rest / G;
        const int c = __ldg(p.ctx + seq), qn = __ldg(p.qlen + seq);
        const int64_t tok0 = __ldg(p.cu_q + seq);
        const int rows_total = qn * p.group;
        const int r0 = grp * R;
        const int nrows = min(R, rows_total - r0);
        const int64_t n = (int64_t)c + qn;
        const int64_t nb = (n + B - 1) / B;
        const int64_t cblocks = (nb + K - 1) / K;     // blocks per split of this sequence

        // query rows -> registers, pre-scaled into log2 units
        float qf[R][E];
        int64_t Pr[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (r < nrows) {
                const int row = r0 + r;
                const int j = row / p.group, hh = row - (row / p.group) * p.group;
                Pr[r] = (int64_t)c + j;
                const T *qp = reinterpret_cast<const T *>(p.q) +
                              ((tok0 + j) * p.q_heads + (int64_t)kvh * p.group + hh) * D + sub * E;
                load_f<T, E>(qp, qf[r]);
#pragma unroll
                for (int e = 0; e < E; ++e) qf[r][e] *= p.scale_log2;
            } else {
                Pr[r] = -1;
#pragma unroll
                for (int e = 0; e < E; ++e) qf[r][e] = 0.f;
            }
        }
        // packed (even, odd) dimension pairs for the two-lane fp32 instructions
        uint64_t q2[R][E / 2];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int e = 0; e < E / 2; ++e) q2[r][e] = f2pack(qf[r][2 * e], qf[r][2 * e + 1]);
        // E4M3 caches: each query row as f16 pairs, scaled by the power of two that puts its
        // largest component in [2^14, 2^15) (far from f16 overflow and underflow); qmul undoes it
        uint32_t qh[R][E / 2];
        float qmul[R];
        if constexpr (kE4) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float mx = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) mx = fmaxf(mx, fabsf(qf[r][e]));
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                int ex = ((__float_as_int(mx) >> 23) & 0xff) - 127 - 14;
                ex = max(-100, min(100, ex));
                const float down = __int_as_float((127 - ex) << 23);
                qmul[r] = __int_as_float((127 + ex) << 23);
#pragma unroll
                for (int e = 0; e < E / 2; ++e) qh[r][e] = h2_from_f32(qf[r][2 * e] * down, qf[r][2 * e + 1] * down);
            }
        }
        const int64_t Pmax = (int64_t)c + (r0 + nrows - 1) / p.group;
        const int64_t nb_lim = (Pmax + B) / B;                  // blocks holding keys 0..Pmax
        const int64_t st_lo = (int64_t)chunk * cblocks * spb;
        int64_t st_hi = (int64_t)(chunk + 1) * cblocks * spb;
        const int64_t st_need = (Pmax + kStageTokens) / kStageTokens;
        if (st_hi > st_need) st_hi = st_need;

        float m[R], l[R];
        uint64_t acc2[R][E / 2];                      // (even, odd) dimension pairs of O
#pragma unroll
        for (int r = 0; r < R; ++r) {
            m[r] = -INFINITY;
            l[r] = 0.f;
#pragma unroll
            for (int e = 0; e < E / 2; ++e) acc2[r][e] = 0ull;
        }

        const int32_t *bt_row = p.bt + (int64_t)seq * p.max_blocks;
        int64_t wbase = -1000000;
        int32_t win = 0;
        bool timed_out = false;
        int64_t st_issue = st_lo;

        auto issue = [&](int64_t st) {
            const int64_t b = st / spb;
            if (b >= wbase + 32 || b < wbase) {
                wbase = b;
                win = (wbase + lane < nb_lim) ? __ldg(bt_row + wbase + lane) : 0;
            }
            int32_t phys = __shfl_sync(0xffffffffu, win, (int)(b - wbase));
            if (phys < 0 || (int64_t)phys >= p.num_blocks) {
                if (lane == 0) report(p.status, PA_DEV_BAD_BLOCK_ID);
                phys = 0;
            }
            if (lane == 0) {
                const uint32_t slot = issued % NST;
                const int64_t off =
                    (int64_t)phys * p.block_stride +
                    ((int64_t)kvh * B + (int64_t)(st - b * spb) * kStageTokens) * D;
                unsigned char *dst = ring + (size_t)slot * 2 * kRunBytes;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&bars[slot], 2 * kRunBytes);
                bulk_g2s(dst, p.k + off * sizeof(TK), kRunBytes, &bars[slot]);
                bulk_g2s(dst + kRunBytes, p.v + off * sizeof(TK), kRunBytes, &bars[slot]);
            }
            ++issued;
        };

        while (st_issue < st_hi && issued - consumed < (uint32_t)NST) issue(st_issue++);
        if (pend.on) {
            finish_split<T, D, R>(p, pend.seq, pend.kvh, pend.grp, pend.G, pend.K, pend.r0, pend.nrows,
                                  pend.tok0, lane);
            pend.on = false;
        }

        for (int64_t st = st_lo; st < st_hi; ++st) {
            const uint32_t slot = consumed % NST;
            if (!mbar_wait(&bars[slot], (consumed / NST) & 1u)) {
                timed_out = true;
                break;
            }
            const TK *sk = reinterpret_cast<const TK *>(ring + (size_t)slot * 2 * kRunBytes);
            const TK *sv = reinterpret_cast<const TK *>(ring + (size_t)slot * 2 * kRunBytes + kRunBytes);
            const int64_t p0 = st * kStageTokens;

            float s[R][kStageTokens / 2];
#pragma unroll
            for (int i = 0; i < kStageTokens / 2; ++i) {
                const int key = 2 * i + half;
                if constexpr (kE4) {
                    const uint2 kw = *reinterpret_cast<const uint2 *>(sk + key * D + sub * E);
                    uint32_t kh[4];
                    e4m3x4_to_h2(kw.x, kh[0], kh[1]);
                    e4m3x4_to_h2(kw.y, kh[2], kh[3]);
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        float d0 = 0.f, d1 = 0.f;
#pragma unroll
                        for (int e = 0; e < 4; ++e) fma_h2(qh[r][e], kh[e], d0, d1);
                        float dot = d0 + d1;
                        dot += __shfl_xor_sync(0xffffffffu, dot, 8);
                        dot += __shfl_xor_sync(0xffffffffu, dot, 4);
                        dot += __shfl_xor_sync(0xffffffffu, dot, 2);
                        dot += __shfl_xor_sync(0xffffffffu, dot, 1);
                        s[r][i] = (p0 + key <= Pr[r]) ? dot * qmul[r] : -INFINITY;
                    }
                    continue;
                }
                uint64_t k2[E / 2];
                if constexpr (E * sizeof(TK) >= 16 || sizeof(TK) == 1) {
                    load_pairs<TK, E / 2>(sk + key * D + sub * E, k2);
                } else {
                    float kf[E];
                    load_f<TK, E>(sk + key * D + sub * E, kf);
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) k2[e] = f2pack(kf[2 * e], kf[2 * e + 1]);
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    uint64_t d2 = 0ull;
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) d2 = fma2(q2[r][e], k2[e], d2);
                    float d0, d1;
                    f2unpack(d2, d0, d1);
                    float dot = d0 + d1;
                    dot += __shfl_xor_sync(0xffffffffu, dot, 8);
                    dot += __shfl_xor_sync(0xffffffffu, dot, 4);
                    dot += __shfl_xor_sync(0xffffffffu, dot, 2);
                    dot += __shfl_xor_sync(0xffffffffu, dot, 1);
                    s[r][i] = (p0 + key <= Pr[r]) ? dot : -INFINITY;
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < kStageTokens / 2; ++i) mx = fmaxf(mx, s[r][i]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float mnew = fmaxf(m[r], mx);
                const float mref = (mnew == -INFINITY) ? 0.f : mnew;
                const float alpha = fast_exp2(m[r] - mref);
                float ps = 0.f;
#pragma unroll
                for (int i = 0; i < kStageTokens / 2; ++i) {
                    s[r][i] = fast_exp2(s[r][i] - mref);
                    ps += s[r][i];
                }
                l[r] = l[r] * alpha + ps;
                const uint64_t a2 = f2pack(alpha, alpha);
#pragma unroll
                for (int e = 0; e < E / 2; ++e) acc2[r][e] = mul2(acc2[r][e], a2);
                m[r] = mnew;
            }
            // O += p V; slots past the last query's key are never read (only a sequence's last
            // stage can hold such keys, so full stages skip the test)
            auto pv_key = [&](int i) {
                const int key = 2 * i + half;
                if constexpr (kE4) {
                    const uint2 vw = *reinterpret_cast<const uint2 *>(sv + key * D + sub * E);
                    uint32_t vh[4];
                    e4m3x4_to_h2(vw.x, vh[0], vh[1]);
                    e4m3x4_to_h2(vw.y, vh[2], vh[3]);
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint16_t ph = f16_from_f32(s[r][i]);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float a, b;
                            f2unpack(acc2[r][e], a, b);
                            fma_h2s(vh[e], ph, a, b);
                            acc2[r][e] = f2pack(a, b);
                        }
                    }
                    return;
                }
                uint64_t v2[E / 2];
                if constexpr (E * sizeof(TK) >= 16 || sizeof(TK) == 1) {
                    load_pairs<TK, E / 2>(sv + key * D + sub * E, v2);
                } else {
                    float vf[E];
                    load_f<TK, E>(sv + key * D + sub * E, vf);
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) v2[e] = f2pack(vf[2 * e], vf[2 * e + 1]);
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint64_t p2 = f2pack(s[r][i], s[r][i]);
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) acc2[r][e] = fma2(v2[e], p2, acc2[r][e]);
                }
            };
            if (p0 + kStageTokens - 1 <= Pmax) {
#pragma unroll
                for (int i = 0; i < kStageTokens / 2; ++i) pv_key(i);
            } else {
#pragma unroll
                for (int i = 0; i < kStageTokens / 2; ++i)
                    if (p0 + 2 * i + half <= Pmax) pv_key(i);
            }
            __syncwarp();
            ++consumed;
            if (st_issue < st_hi) issue(st_issue++);
        }

        if (timed_out) {
            if (lane == 0) report(p.status, PA_DEV_TIMEOUT);
            // let the copies already in flight land before the warp leaves
            while (consumed < issued) {
                mbar_wait(&bars[consumed % NST], (consumed / NST) & 1u);
                ++consumed;
            }
            return;
        }

        float acc[R][E];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int e = 0; e < E / 2; ++e) f2unpack(acc2[r][e], acc[r][2 * e], acc[r][2 * e + 1]);
        // merge the two half-warps (alternate keys); V's scale (E4M3 caches) applies to o
#pragma unroll
        for (int r = 0; r < R; ++r) {
            l[r] += __shfl_xor_sync(0xffffffffu, l[r], 16);
#pragma unroll
            for (int e = 0; e < E; ++e)
                acc[r][e] = (acc[r][e] + __shfl_xor_sync(0xffffffffu, acc[r][e], 16)) * p.v_scale;
        }
        if (K == 1) {
            if (half == 0) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (r >= nrows) continue;
                    const int row = r0 + r;
                    const int j = row / p.group, hh = row - (row / p.group) * p.group;
                    const float inv = 1.f / l[r];
                    float o[E];
#pragma unroll
                    for (int e = 0; e < E; ++e) o[e] = acc[r][e] * inv;
                    T *op = reinterpret_cast<T *>(p.out) +
                            ((tok0 + j) * p.q_heads + (int64_t)kvh * p.group + hh) * D + sub * E;
                    store_f<T, E>(op, o);
                }
            }
        } else {
            const int64_t part = (int64_t)__ldg(p.parts_cu + seq) + local;
            if (half == 0) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (r >= nrows) continue;
                    float *po = p.parts_o + ((part * R + r) * D + sub * E);
#pragma unroll
                    for (int e = 0; e < E; e += 4)
                        *reinterpret_cast<float4 *>(po + e) =
                            make_float4(acc[r][e], acc[r][e + 1], acc[r][e + 2], acc[r][e + 3]);
                    if (sub == 0) p.parts_ml[part * R + r] = make_float2(m[r], l[r]);
                }
            }
            pend = PendingSplit{seq, kvh, grp, G, K, r0, nrows, tok0, true};
        }
    }
    if (pend.on)
        finish_split<T, D, R>(p, pend.seq, pend.kvh, pend.grp, pend.G, pend.K, pend.r0, pend.nrows, pend.tok0,
                              lane);
}

// ----------------------------------------------------------------------------------------------
// GQA work-item kernel: R = 2 or 4 query rows of one KV head share every K/V stage.
//
// QK^T: four lanes per key, each holding a quarter of the head dimension of all R query rows, so
// one pass covers eight keys.  The R partial dot products of a lane are summed over its four
// quarter lanes by a transpose-reduce (each shuffle level hands half of the rows still held to
// the partner lane), which leaves lane (quarter r, key k) with the full score of row r (R = 4;
// rows r/2 for R = 2) in three (two) shuffles per eight keys, where a reduce of every row on
// every lane would take sixteen.  K arrives by TMA as 128-byte panels with the 128-byte swizzle
// (16-byte chunk c of row t stored at chunk c ^ (t mod 8)), so the eight lanes of one quarter
// read chunks of eight different rows without a bank conflict; V arrives by one bulk copy.
// The softmax runs on the score owners; the probabilities go through a small shared-memory
// table to the PV lanes: half-warps take alternate keys and each lane holds D/16 dimensions of
// the R output rows.  The rescale of the R accumulators is skipped when no row's max moved.
// ----------------------------------------------------------------------------------------------
template <typename T, int D>
struct GqaStage {
    static constexpr int kRow = D * (int)sizeof(T);         // bytes of one key row
    static constexpr int kPanels = kRow / 128;               // 128-byte TMA panels per row
    static constexpr int kPanelBytes = kStageTokens * 128;   // one panel of the stage's 16 rows
    static constexpr uint32_t kK = kStageTokens * kRow;      // swizzled K panels
    static constexpr uint32_t kV = kStageTokens * kRow;      // V rows, as in global memory
    static constexpr uint32_t kBytes = kK + kV;              // a multiple of 1024
};

template <typename T, typename TK, int D, int R>
__global__ void __launch_bounds__(kSimtMaxWarps * 32, 1)
    simt_gqa_kernel(const __grid_constant__ CUtensorMap kmap, SimtParams p) {
    static_assert(R == 2 || R == 4, "two or four rows per item");
    using S = GqaStage<TK, D>;
    constexpr int QD = D / 4;                       // dims per quarter lane (QK^T)
    constexpr int E = D / 16;                       // dims per lane (PV)
    constexpr int EC = 16 / (int)sizeof(TK);        // elements per 16-byte chunk
    constexpr int NJ = QD / EC;                     // chunks per quarter lane and key
    constexpr int kPs = (kStageTokens + 1) * R;     // (p, p) pairs of a warp: 16 keys + alpha
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qd = lane >> 3, kk = lane & 7;        // QK^T roles: quarter, key
    const int half = lane >> 4, sub = lane & 15;    // PV roles: key parity, dims
    const int rrow = R == 4 ? qd : (qd >> 1);       // the score row this lane owns
    const bool owner = R == 4 || (qd & 1) == 0;     // one writer per (row, key)
    const int NST = p.nst;
    const int nwarps = blockDim.x >> 5;
    // shared memory: rings [warp][stage], probability tables [warp], barriers [warp][stage]
    unsigned char *ring = smem + (size_t)warp * NST * S::kBytes;
    float2 *ps = reinterpret_cast<float2 *>(smem + (size_t)nwarps * NST * S::kBytes) + warp * kPs;
    float2 *alpha_s = ps + kStageTokens * R;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)nwarps * (NST * S::kBytes + kPs * 8)) +
                     warp * NST;
    // byte offsets (within a key row of the swizzled panels) of this lane's NJ chunks
    int koff[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const int ob = qd * QD * (int)sizeof(TK) + j * 16;
        koff[j] = (ob >> 7) * S::kPanelBytes + ((((ob >> 4) & 7) ^ kk) << 4);
    }
    if (lane == 0) {
        for (int s = 0; s < NST; ++s) mbar_init(&bars[s], 1);
        mbar_fence_init();
    }
    __syncwarp();

    const int B = p.block_size;
    const int spb = B / kStageTokens;
    // ring state, continuous across items: issue slot, consume slot and its phase, stages in flight
    int slot_i = 0, slot_c = 0, inflight = 0;
    uint32_t phase_c = 0;
    const uint32_t total_items = p.counters[kSimtTotal];
    PendingSplit pend;
    pend.on = false;

    while (true) {
        int item = 0;
        if (lane == 0) item = (int)atomicAdd(&p.counters[kSimtNext], 1u);
        item = __shfl_sync(0xffffffffu, item, 0);
        if ((uint32_t)item >= total_items) break;

        const int seq = find_owner(p.simt_cu, p.num_seqs, item);
        const int local = item - __ldg(p.simt_cu + seq);
        const int K = __ldg(p.nchunk + seq);
        const int G = __ldg(p.groups + seq);
        const int chunk = local % K;
        const int rest = local / K;
        const int grp = rest % G;
        const int kvh = rest / G;
        const int c = __ldg(p.ctx + seq), qn = __ldg(p.qlen + seq);
        const int64_t tok0 = __ldg(p.cu_q + seq);
        const int rows_total = qn * p.group;
        const int r0 = grp * R;
        const int nrows = min(R, rows_total - r0);
        const int n = c + qn;                        // < 2^31 (checked by the planner)
        const int nb = (n + B - 1) / B;
        const int cblocks = (nb + K - 1) / K;

        // causal limit of the row this lane scores (-1: a padding row, every key masked)
        const int Pmine = rrow < nrows ? c + (r0 + rrow) / p.group : -1;
        const int Pmax = c + (r0 + nrows - 1) / p.group;
        const int st_lo = chunk * cblocks * spb;
        const int st_hi = min((chunk + 1) * cblocks * spb, (Pmax + kStageTokens) / kStageTokens);
        const int nb_lim = (Pmax + B) / B;

        float m = -INFINITY, lsum = 0.f;             // of row rrow, over this lane's keys
        uint64_t acc2[R][E / 2];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int e = 0; e < E / 2; ++e) acc2[r][e] = 0ull;

        const int32_t *bt_row = p.bt + (int64_t)seq * p.max_blocks;
        int wbase = -1000000;
        int32_t win = 0;
        bool timed_out = false;
        // issue cursor: next stage, its logical block and its 16-token part within the block
        int st_issue = st_lo, ib = st_lo / spb, isub = st_lo - (st_lo / spb) * spb;

        auto issue = [&]() {
            if (ib >= wbase + 32 || ib < wbase) {
                wbase = ib;
                win = (wbase + lane < nb_lim) ? __ldg(bt_row + wbase + lane) : 0;
            }
            int32_t phys = __shfl_sync(0xffffffffu, win, ib - wbase);
            if (phys < 0 || (int64_t)phys >= p.num_blocks) {
                if (lane == 0) report(p.status, PA_DEV_BAD_BLOCK_ID);
                phys = 0;
            }
            if (lane == 0) {
                unsigned char *dst = ring + (size_t)slot_i * S::kBytes;
                const int row = kvh * B + isub * kStageTokens;     // of the block's [Hkv * B] rows
                const int64_t off = (int64_t)phys * p.block_stride + (int64_t)row * D;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&bars[slot_i], S::kK + S::kV);
#pragma unroll
                for (int pn = 0; pn < S::kPanels; ++pn)
                    tma_load_3d(dst + pn * S::kPanelBytes, &kmap, pn * (128 / (int)sizeof(TK)), row, phys,
                                &bars[slot_i]);
                bulk_g2s(dst + S::kK, p.v + off * sizeof(TK), S::kV, &bars[slot_i]);
            }
            slot_i = slot_i + 1 == NST ? 0 : slot_i + 1;
            ++inflight;
            ++st_issue;
            if (++isub == spb) {
                isub = 0;
                ++ib;
            }
        };

        while (st_issue < st_hi && inflight < NST) issue();
        if (pend.on) {
            finish_split<T, D, R>(p, pend.seq, pend.kvh, pend.grp, pend.G, pend.K, pend.r0, pend.nrows,
                                  pend.tok0, lane);
            pend.on = false;
        }
        // the queries are loaded after the merge, which then has their registers for its loads
        // this lane's quarter of every query row, pre-scaled into log2 units, in the lane's own row
        // order: slot sl holds row rrow ^ sl, so the transpose-reduce below keeps slots 0 (and 1)
        // and sends the others without selecting
        uint64_t q2[R][QD / 2];
#pragma unroll
        for (int sl = 0; sl < R; ++sl) {
            const int r = rrow ^ sl;
            float qf[QD];
            if (r < nrows) {
                const int row = r0 + r;
                const int j = row / p.group, hh = row - j * p.group;
                const T *qp = reinterpret_cast<const T *>(p.q) +
                              ((tok0 + j) * p.q_heads + (int64_t)kvh * p.group + hh) * D + qd * QD;
                load_f<T, QD>(qp, qf);
            } else {
#pragma unroll
                for (int e = 0; e < QD; ++e) qf[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < QD / 2; ++e)
                q2[sl][e] = f2pack(qf[2 * e] * p.scale_log2, qf[2 * e + 1] * p.scale_log2);
        }

        for (int st = st_lo; st < st_hi; ++st) {
            if (!mbar_wait(&bars[slot_c], phase_c)) {
                timed_out = true;
                break;
            }
            const unsigned char *sk = ring + (size_t)slot_c * S::kBytes;
            const TK *sv = reinterpret_cast<const TK *>(sk + S::kK);
            const int p0 = st * kStageTokens;

            // scores: lane (qd, kk) ends with row rrow's score of keys kk and 8 + kk
            float sc[2];
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                const int key = it * 8 + kk;
                const unsigned char *kr = sk + key * 128;
                uint64_t d2[R];
#pragma unroll
                for (int r = 0; r < R; ++r) d2[r] = 0ull;
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    uint64_t k2[EC / 2];
                    load_pairs<TK, EC / 2>(reinterpret_cast<const TK *>(kr + koff[j]), k2);
#pragma unroll
                    for (int e = 0; e < EC / 2; ++e)
#pragma unroll
                        for (int r = 0; r < R; ++r) d2[r] = fma2(q2[r][j * (EC / 2) + e], k2[e], d2[r]);
                }
                float d[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float a, b2;
                    f2unpack(d2[r], a, b2);
                    d[r] = a + b2;
                }
                // d[sl] is row rrow ^ sl.  R = 4: the partner across lane bit 4 (rows rrow ^ 2, ^3)
                // sends its slots 2, 3 = this lane's rows rrow, rrow ^ 1; across bit 3 the partner
                // (row rrow ^ 1) sends its slot 1 = row rrow.  R = 2: across bit 4 the other row's
                // lanes send slot 1 = row rrow; across bit 3 both lanes hold the same row.
                float s;
                if constexpr (R == 4) {
                    const float keep0 = d[0] + __shfl_xor_sync(0xffffffffu, d[2], 16);
                    const float keep1 = d[1] + __shfl_xor_sync(0xffffffffu, d[3], 16);
                    s = keep0 + __shfl_xor_sync(0xffffffffu, keep1, 8);
                } else {
                    const float keep = d[0] + __shfl_xor_sync(0xffffffffu, d[1], 16);
                    s = keep + __shfl_xor_sync(0xffffffffu, keep, 8);
                }
                sc[it] = (p0 + key <= Pmine) ? s : -INFINITY;
            }
            // online softmax of row rrow over this stage's 16 keys
            float mx = fmaxf(sc[0], sc[1]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            const float mnew = fmaxf(m, mx);
            const float mref = (mnew == -INFINITY) ? 0.f : mnew;
            const float alpha = fast_exp2(m - mref);
            const float pe0 = fast_exp2(sc[0] - mref), pe1 = fast_exp2(sc[1] - mref);
            lsum = lsum * alpha + (pe0 + pe1);
            m = mnew;
            if (owner) {
                ps[kk * R + rrow] = make_float2(pe0, pe0);
                ps[(8 + kk) * R + rrow] = make_float2(pe1, pe1);
                if (kk == 0) alpha_s[rrow] = make_float2(alpha, alpha);
            }
            const bool rescale = __any_sync(0xffffffffu, alpha != 1.f);
            __syncwarp();
            if (rescale) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint64_t a2 = *reinterpret_cast<const uint64_t *>(alpha_s + r);
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) acc2[r][e] = mul2(acc2[r][e], a2);
                }
            }
            // O += P V over the stage's keys; slots past the last query's key are never read
            auto pv_key = [&](int key) {
                uint64_t pr[R];
#pragma unroll
                for (int r = 0; r < R; r += 2) {
                    const uint4 t = *reinterpret_cast<const uint4 *>(ps + key * R + r);
                    pr[r] = (uint64_t)t.x | ((uint64_t)t.y << 32);
                    pr[r + 1] = (uint64_t)t.z | ((uint64_t)t.w << 32);
                }
                uint64_t v2[E / 2];
                if constexpr (E * sizeof(TK) >= 16 || sizeof(TK) == 1) {
                    load_pairs<TK, E / 2>(sv + key * D + sub * E, v2);
                } else {
                    float vf[E];
                    load_f<TK, E>(sv + key * D + sub * E, vf);
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) v2[e] = f2pack(vf[2 * e], vf[2 * e + 1]);
                }
#pragma unroll
                for (int e = 0; e < E / 2; ++e)
#pragma unroll
                    for (int r = 0; r < R; ++r) acc2[r][e] = fma2(v2[e], pr[r], acc2[r][e]);
            };
            if (p0 + kStageTokens - 1 <= Pmax) {
#pragma unroll
                for (int i = 0; i < kStageTokens / 2; ++i) pv_key(2 * i + half);
            } else {
#pragma unroll 1
                for (int key = half; p0 + key <= Pmax; key += 2) pv_key(key);
            }
            __syncwarp();
            slot_c = slot_c + 1 == NST ? 0 : slot_c + 1;
            phase_c ^= slot_c == 0 ? 1u : 0u;
            --inflight;
            if (st_issue < st_hi) issue();
        }

        if (timed_out) {
            if (lane == 0) report(p.status, PA_DEV_TIMEOUT);
            // let the copies already in flight land before the warp leaves
            while (inflight > 0) {
                mbar_wait(&bars[slot_c], phase_c);
                slot_c = slot_c + 1 == NST ? 0 : slot_c + 1;
                phase_c ^= slot_c == 0 ? 1u : 0u;
                --inflight;
            }
            return;
        }

        // row statistics: sum the key lanes' partial sums, then hand (m, l) of every row to
        // every lane; merge the two half-warps' accumulators
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 4);
        float mr[R], lr[R], acc[R][E];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int src = (R == 4 ? r : 2 * r) * 8;
            mr[r] = __shfl_sync(0xffffffffu, m, src);
            lr[r] = __shfl_sync(0xffffffffu, lsum, src);
#pragma unroll
            for (int e = 0; e < E / 2; ++e) f2unpack(acc2[r][e], acc[r][2 * e], acc[r][2 * e + 1]);
#pragma unroll
            for (int e = 0; e < E; ++e)
                acc[r][e] = (acc[r][e] + __shfl_xor_sync(0xffffffffu, acc[r][e], 16)) * p.v_scale;
        }
        if (half == 0) {
            if (K == 1) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (r >= nrows) continue;
                    const int row = r0 + r;
                    const int j = row / p.group, hh = row - j * p.group;
                    const float inv = 1.f / lr[r];
                    float o[E];
#pragma unroll
                    for (int e = 0; e < E; ++e) o[e] = acc[r][e] * inv;
                    T *op = reinterpret_cast<T *>(p.out) +
                            ((tok0 + j) * p.q_heads + (int64_t)kvh * p.group + hh) * D + sub * E;
                    store_f<T, E>(op, o);
                }
            } else {
                const int64_t part = (int64_t)__ldg(p.parts_cu + seq) + local;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (r >= nrows) continue;
                    float *po = p.parts_o + ((part * R + r) * D + sub * E);
#pragma unroll
                    for (int e = 0; e < E; e += 4)
                        *reinterpret_cast<float4 *>(po + e) =
                            make_float4(acc[r][e], acc[r][e + 1], acc[r][e + 2], acc[r][e + 3]);
                    if (sub == 0) p.parts_ml[part * R + r] = make_float2(mr[r], lr[r]);
                }
            }
        }
        if (K > 1) pend = PendingSplit{seq, kvh, grp, G, K, r0, nrows, tok0, true};
    }
    if (pend.on)
        finish_split<T, D, R>(p, pend.seq, pend.kvh, pend.grp, pend.G, pend.K, pend.r0, pend.nrows, pend.tok0,
                              lane);
}

// ----------------------------------------------------------------------------------------------
// GQA decode on tensor cores (16-bit caches, head_dim 128; mma.m16n8k16, fp32 accumulators).  The
// item structure, the ring and the split merge are those of simt_gqa_kernel; the arithmetic runs
// as FlashAttention-2 style fragments: the item's R query rows are rows 0..R-1 of a 16-row A
// operand (the other rows zero), S = Q K^T takes K as B fragments straight from the swizzled TMA
// panels (ldmatrix), P stays in registers as the A operand of O += P V, and V arrives through TMA
// with the same swizzle and is read transposed (ldmatrix.trans).  Lane (g, c) owns row g: scores
// of keys 2c, 2c+1 (+8) of each 16-key stage, and output columns 8 n + 2c, +1.  P is rounded to the
// query's 16-bit type before PV, as in the tensor-core prefill kernel.
// ----------------------------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// D += A B, m16n8k16 with A rows 8..15 zero (a1 = a3 = 0): a0 = A[g][2c..2c+1], a2 = A[g][2c+8..2c+9].
template <typename T>
__device__ __forceinline__ void mma_rows8(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
    if constexpr (sizeof(T) == 2 && std::is_same<T, __nv_bfloat16>::value)
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
    else
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
// Two fp32 values -> one pair of the 16-bit type (a in the low half), rounded to nearest even.
template <typename T> __device__ __forceinline__ uint32_t pack16(float a, float b);
template <> __device__ __forceinline__ uint32_t pack16<__nv_bfloat16>(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}
template <> __device__ __forceinline__ uint32_t pack16<__half>(float a, float b) { return h2_from_f32(a, b); }

template <typename T, int R>
__global__ void __launch_bounds__(kSimtMaxWarps * 32, 1)
    gqa_mma_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap, SimtParams p) {
    constexpr int D = 128;
    static_assert(R == 2 || R == 4, "two or four rows per item");
    using S = GqaStage<T, D>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c4 = lane & 3;
    const int NST = p.nst;
    const int nwarps = blockDim.x >> 5;
    unsigned char *ring = smem + (size_t)warp * NST * S::kBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)nwarps * NST * S::kBytes) + warp * NST;
    // ldmatrix row addresses within a stage.  S: matrix i = lane / 8 covers keys 8 (i / 2) .. +7 and
    // channels 8 (i % 2) .. +7 of the 16-channel step; PV: keys 8 (i % 2) .. +7, channels 8 (i / 2)
    // .. +7 of the 16-channel pair of n-blocks.  Row t of a 128-byte panel holds 16-byte chunk q
    // at chunk q ^ (t mod 8).
    const int mi = lane >> 3, mr = lane & 7;
    const int kkey = (mi >> 1) * 8 + mr, kch = mi & 1;
    const int vkey = (mi & 1) * 8 + mr, vch = mi >> 1;
    if (lane == 0) {
        for (int s = 0; s < NST; ++s) mbar_init(&bars[s], 1);
        mbar_fence_init();
    }
    __syncwarp();

    const int B = p.block_size;
    const int spb = B / kStageTokens;
    int slot_i = 0, slot_c = 0, inflight = 0;
    uint32_t phase_c = 0;
    const uint32_t total_items = p.counters[kSimtTotal];
    PendingSplit pend;
    pend.on = false;

    while (true) {
        int item = 0;
        if (lane == 0) item = (int)atomicAdd(&p.counters[kSimtNext], 1u);
        item = __shfl_sync(0xffffffffu, item, 0);
        if ((uint32_t)item >= total_items) break;

        const int seq = find_owner(p.simt_cu, p.num_seqs, item);
        const int local = item - __ldg(p.simt_cu + seq);
        const int K = __ldg(p.nchunk + seq);
        const int G = __ldg(p.groups + seq);
        const int chunk = local % K;
        const int rest = local / K;
        const int grp = rest % G;
        const int kvh = rest / G;
        const int c = __ldg(p.ctx + seq), qn = __ldg(p.qlen + seq);
        const int64_t tok0 = __ldg(p.cu_q + seq);
        const int rows_total = qn * p.group;
        const int r0 = grp * R;
        const int nrows = min(R, rows_total - r0);
        const int n = c + qn;
        const int nb = (n + B - 1) / B;
        const int cblocks = (nb + K - 1) / K;
        // causal limit of this lane's row g (-1: a padding row, every key masked)
        const int Pmine = g < nrows ? c + (r0 + g) / p.group : -1;
        const int Pmax = c + (r0 + nrows - 1) / p.group;
        const int st_lo = chunk * cblocks * spb;
        const int st_hi = min((chunk + 1) * cblocks * spb, (Pmax + kStageTokens) / kStageTokens);
        const int nb_lim = (Pmax + B) / B;

        float m = -INFINITY, lsum = 0.f;
        float o[16][4];
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

        const int32_t *bt_row = p.bt + (int64_t)seq * p.max_blocks;
        int wbase = -1000000;
        int32_t win = 0;
        bool timed_out = false;
        int st_issue = st_lo, ib = st_lo / spb, isub = st_lo - (st_lo / spb) * spb;

        auto issue = [&]() {
            if (ib >= wbase + 32 || ib < wbase) {
                wbase = ib;
                win = (wbase + lane < nb_lim) ? __ldg(bt_row + wbase + lane) : 0;
            }
            int32_t phys = __shfl_sync(0xffffffffu, win, ib - wbase);
            if (phys < 0 || (int64_t)phys >= p.num_blocks) {
                if (lane == 0) report(p.status, PA_DEV_BAD_BLOCK_ID);
                phys = 0;
            }
            if (lane == 0) {
                unsigned char *dst = ring + (size_t)slot_i * S::kBytes;
                const int row = kvh * B + isub * kStageTokens;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&bars[slot_i], S::kK + S::kV);
#pragma unroll
                for (int pn = 0; pn < S::kPanels; ++pn) {
                    tma_load_3d(dst + pn * S::kPanelBytes, &kmap, pn * (128 / (int)sizeof(T)), row, phys, &bars[slot_i]);
                    tma_load_3d(dst + S::kK + pn * S::kPanelBytes, &vmap, pn * (128 / (int)sizeof(T)), row, phys,
                                &bars[slot_i]);
                }
            }
            slot_i = slot_i + 1 == NST ? 0 : slot_i + 1;
            ++inflight;
            ++st_issue;
            if (++isub == spb) {
                isub = 0;
                ++ib;
            }
        };

        while (st_issue < st_hi && inflight < NST) issue();
        if (pend.on) {
            finish_split<T, D, R>(p, pend.seq, pend.kvh, pend.grp, pend.G, pend.K, pend.r0, pend.nrows,
                                  pend.tok0, lane);
            pend.on = false;
        }
        // A fragments of the query rows (rows >= nrows and 8..15 zero): channels 16 ks + 2c, +1 and
        // 16 ks + 8 + 2c, +1 of row g
        uint32_t qa[8][2];
        {
            const T *qp = nullptr;
            if (g < nrows) {
                const int row = r0 + g;
                const int j = row / p.group, hh = row - j * p.group;
                qp = reinterpret_cast<const T *>(p.q) + ((tok0 + j) * p.q_heads + (int64_t)kvh * p.group + hh) * D;
            }
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                qa[ks][0] = qp ? __ldg(reinterpret_cast<const uint32_t *>(qp + 16 * ks + 2 * c4)) : 0u;
                qa[ks][1] = qp ? __ldg(reinterpret_cast<const uint32_t *>(qp + 16 * ks + 8 + 2 * c4)) : 0u;
            }
        }

        for (int st = st_lo; st < st_hi; ++st) {
            if (!mbar_wait(&bars[slot_c], phase_c)) {
                timed_out = true;
                break;
            }
            unsigned char *sk = ring + (size_t)slot_c * S::kBytes;
            unsigned char *sv = sk + S::kK;
            const int p0 = st * kStageTokens;
            // V rows past the last key any row sees hold stale or unread data (possibly NaN): zero
            // them, so that P = 0 times them stays 0 in the MMA
            if (p0 + kStageTokens - 1 > Pmax) {
                const int first = Pmax - p0 + 1;           // >= 1
                for (int i = lane; i < (kStageTokens - first) * (S::kRow / 16); i += 32) {
                    const int key = first + i / (S::kRow / 16), ch = i % (S::kRow / 16);
                    *reinterpret_cast<uint4 *>(sv + (ch >> 3) * S::kPanelBytes + key * 128 + ((ch & 7) << 4)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
            }
            // S = Q K^T: n-block 0 = keys 0..7, n-block 1 = keys 8..15 of the stage
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            const uint32_t kbase = smem_addr(sk);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int q = 2 * ks + kch;                    // 16-byte chunk of the key row
                const uint32_t addr = kbase + (q >> 3) * S::kPanelBytes + kkey * 128 + (((q & 7) ^ (kkey & 7)) << 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(addr, b0, b1, b2, b3);
                mma_rows8<T>(sc[0], qa[ks][0], qa[ks][1], b0, b1);
                mma_rows8<T>(sc[1], qa[ks][0], qa[ks][1], b2, b3);
            }
            // scores of keys 8 nb + 2c + e of row g, in log2 units, causally masked
            float z[2][2];
            float mx = -INFINITY;
#pragma unroll
            for (int nb2 = 0; nb2 < 2; ++nb2)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = 8 * nb2 + 2 * c4 + e;
                    z[nb2][e] = (p0 + key <= Pmine) ? sc[nb2][e] * p.scale_log2 : -INFINITY;
                    mx = fmaxf(mx, z[nb2][e]);
                }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mnew = fmaxf(m, mx);
            const float mref = (mnew == -INFINITY) ? 0.f : mnew;
            const float alpha = fast_exp2(m - mref);
            float pe[2][2];
#pragma unroll
            for (int nb2 = 0; nb2 < 2; ++nb2)
#pragma unroll
                for (int e = 0; e < 2; ++e) pe[nb2][e] = fast_exp2(z[nb2][e] - mref);
            lsum = lsum * alpha + ((pe[0][0] + pe[0][1]) + (pe[1][0] + pe[1][1]));
            m = mnew;
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    o[i][0] *= alpha;
                    o[i][1] *= alpha;
                }
            }
            // O += P V: P as the A operand (keys 2c, 2c+1 and 8 + 2c, +1 of row g), V by ldmatrix.trans
            const uint32_t pa0 = pack16<T>(pe[0][0], pe[0][1]), pa2 = pack16<T>(pe[1][0], pe[1][1]);
            const uint32_t vbase = smem_addr(sv);
#pragma unroll
            for (int np = 0; np < 8; ++np) {
                const int q = 2 * np + vch;
                const uint32_t addr = vbase + (q >> 3) * S::kPanelBytes + vkey * 128 + (((q & 7) ^ (vkey & 7)) << 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(addr, b0, b1, b2, b3);
                mma_rows8<T>(o[2 * np], pa0, pa2, b0, b1);
                mma_rows8<T>(o[2 * np + 1], pa0, pa2, b2, b3);
            }
            __syncwarp();
            slot_c = slot_c + 1 == NST ? 0 : slot_c + 1;
            phase_c ^= slot_c == 0 ? 1u : 0u;
            --inflight;
            if (st_issue < st_hi) issue();
        }

        if (timed_out) {
            if (lane == 0) report(p.status, PA_DEV_TIMEOUT);
            while (inflight > 0) {
                mbar_wait(&bars[slot_c], phase_c);
                slot_c = slot_c + 1 == NST ? 0 : slot_c + 1;
                phase_c ^= slot_c == 0 ? 1u : 0u;
                --inflight;
            }
            return;
        }

        // row g's sum over the four lanes of the row; lane (g, c) holds columns 8 i + 2c, +1
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
        if (g < nrows) {
            const int row = r0 + g;
            if (K == 1) {
                const int j = row / p.group, hh = row - j * p.group;
                const float inv = 1.f / lsum;
                T *op = reinterpret_cast<T *>(p.out) + ((tok0 + j) * p.q_heads + (int64_t)kvh * p.group + hh) * D;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    *reinterpret_cast<uint32_t *>(op + 8 * i + 2 * c4) = pack16<T>(o[i][0] * inv, o[i][1] * inv);
            } else {
                const int64_t part = (int64_t)__ldg(p.parts_cu + seq) + local;
                float *po = p.parts_o + (part * R + g) * D;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    *reinterpret_cast<float2 *>(po + 8 * i + 2 * c4) = make_float2(o[i][0], o[i][1]);
                if (c4 == 0) p.parts_ml[part * R + g] = make_float2(m, lsum);
            }
        }
        if (K > 1) pend = PendingSplit{seq, kvh, grp, G, K, r0, nrows, tok0, true};
    }
    if (pend.on)
        finish_split<T, D, R>(p, pend.seq, pend.kvh, pend.grp, pend.G, pend.K, pend.r0, pend.nrows, pend.tok0,
                              lane);
}

template <typename T, int R>
cudaError_t launch_gqa_mma_t(const FwdArgs &a, const SimtParams &p0, cudaStream_t s) {
    constexpr int D = 128;
    SimtParams p = p0;
    using S = GqaStage<T, D>;
    // K and V as [num_blocks][Hkv * B rows][D]; one TMA box = one 128-byte panel of 16 rows
    CUtensorMap kmap, vmap;
    const uint64_t es = sizeof(T);
    if (!make_map_3d(&kmap, a.dims.dtype, a.k, D, (uint64_t)a.dims.num_kv_heads * a.dims.block_size,
                     a.dims.num_blocks, D * es, (uint64_t)p.block_stride * es, (uint32_t)(128 / es), kStageTokens, 1) ||
        !make_map_3d(&vmap, a.dims.dtype, a.v, D, (uint64_t)a.dims.num_kv_heads * a.dims.block_size,
                     a.dims.num_blocks, D * es, (uint64_t)p.block_stride * es, (uint32_t)(128 / es), kStageTokens, 1))
        return cudaErrorInvalidValue;
    const int nst = 3, warps = kSimtMaxWarps;
    p.nst = nst;
    p.bar_bytes = 0;
    const size_t smem = 1024 + (size_t)warps * nst * (S::kBytes + sizeof(uint64_t));
    auto kern = gqa_mma_kernel<T, R>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<a.num_sms, warps * 32, smem, s>>>(kmap, vmap, p);
    return cudaGetLastError();
}

template <typename T, typename TK, int D, int R>
cudaError_t launch_simt_t(const FwdArgs &a, const SimtParams &p0, cudaStream_t s) {
    SimtParams p = p0;
    const size_t run = (size_t)kStageTokens * D * sizeof(TK);
    const size_t stage = 2 * run;
    const size_t budget = 200 * 1024;
    int nst = stage <= 8192 ? 3 : 2;
    int warps = (int)(budget / (nst * stage));
    if (warps > 8) warps = 8;
    if (warps < 1) {
        nst = 2;
        warps = 1;
    }
    p.nst = nst;
    p.bar_bytes = (int)align_up((size_t)warps * nst * sizeof(uint64_t), 128);
    const size_t smem = p.bar_bytes + (size_t)warps * nst * stage;
    auto kern = simt_attention_kernel<T, TK, D, R>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, warps * 32, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    kern<<<a.num_sms * per_sm, warps * 32, smem, s>>>(p);
    return cudaGetLastError();
}

template <typename T, typename TK, int D, int R>
cudaError_t launch_gqa_t(const FwdArgs &a, const SimtParams &p0, cudaStream_t s) {
    SimtParams p = p0;
    using S = GqaStage<TK, D>;
    // K as [num_blocks][Hkv * B rows][D], one TMA box = one 128-byte panel of 16 rows
    CUtensorMap kmap;
    const uint64_t es = sizeof(TK);
    if (!make_map_3d(&kmap, sizeof(TK) == 1 ? kMapBytes : a.dims.dtype, a.k, D, (uint64_t)a.dims.num_kv_heads * a.dims.block_size,
                     a.dims.num_blocks, D * es, (uint64_t)p.block_stride * es, (uint32_t)(128 / es),
                     kStageTokens, 1))
        return cudaErrorInvalidValue;
    const size_t per_stage = S::kBytes + sizeof(uint64_t);
    const size_t ps_bytes = (size_t)(kStageTokens + 1) * R * sizeof(float2);
    const size_t budget = 210 * 1024;
    int nst = 3;
    int warps = (int)(budget / (nst * per_stage + ps_bytes));
    const int warps2 = (int)(budget / (2 * per_stage + ps_bytes));
    if (warps < kSimtMaxWarps && warps2 > warps) {
        nst = 2;
        warps = warps2;
    }
    if (warps > kSimtMaxWarps) warps = kSimtMaxWarps;
    p.nst = nst;
    p.bar_bytes = 0;
    const size_t smem = 1024 + (size_t)warps * (nst * per_stage + ps_bytes);
    auto kern = simt_gqa_kernel<T, TK, D, R>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<a.num_sms, warps * 32, smem, s>>>(kmap, p);
    return cudaGetLastError();
}

template <typename T, typename TK, int D>
cudaError_t launch_simt_rows(const FwdArgs &a, const SimtParams &p, cudaStream_t s) {
    // GQA rows of 16-bit caches with head_dim 128 run on tensor cores
    constexpr bool kMma = std::is_same<T, TK>::value && sizeof(T) == 2 && D == 128;
    switch (a.lay.rows_per_item) {
    case 1: return launch_simt_t<T, TK, D, 1>(a, p, s);
    case 2:
        if constexpr (kMma) return launch_gqa_mma_t<T, 2>(a, p, s);
        else return launch_gqa_t<T, TK, D, 2>(a, p, s);
    default:
        if constexpr (kMma) return launch_gqa_mma_t<T, 4>(a, p, s);
        else return launch_gqa_t<T, TK, D, 4>(a, p, s);
    }
}

template <typename T>
cudaError_t launch_simt_dim(const FwdArgs &a, const SimtParams &p, cudaStream_t s) {
    if (a.dims.kv_dtype == PA_KV_E4M3) {
        if constexpr (sizeof(T) == 2) return launch_simt_rows<T, e4m3, 128>(a, p, s);
        return cudaErrorInvalidValue;
    }
    return a.dims.head_dim == 64 ? launch_simt_rows<T, T, 64>(a, p, s) : launch_simt_rows<T, T, 128>(a, p, s);
}

}  // namespace

cudaError_t launch_plan(const FwdArgs &a, cudaStream_t s) {
    PlanParams p;
    const WsLayout &L = a.lay;
    p.ctx = a.ctx;
    p.qlen = a.qlen;
    p.counters = reinterpret_cast<uint32_t *>(a.ws + L.counters);
    p.cu_q = reinterpret_cast<int32_t *>(a.ws + L.cu_q);
    p.simt_cu = reinterpret_cast<int32_t *>(a.ws + L.simt_cu);
    p.parts_cu = reinterpret_cast<int32_t *>(a.ws + L.parts_cu);
    p.comb_cu = reinterpret_cast<int32_t *>(a.ws + L.comb_cu);
    p.groups = reinterpret_cast<int32_t *>(a.ws + L.groups);
    p.nchunk = reinterpret_cast<int32_t *>(a.ws + L.nchunk);
    p.tc_cu = reinterpret_cast<int32_t *>(a.ws + L.tc_cu);
    p.tc_seq = reinterpret_cast<int32_t *>(a.ws + L.tc_seq);
    p.unit_cnt = reinterpret_cast<uint32_t *>(a.ws + L.unit_cnt);
    p.status = a.status;
    p.total_q = a.dims.total_q;
    p.max_parts = L.max_parts;
    p.num_seqs = a.dims.num_seqs;
    p.kv_heads = a.dims.num_kv_heads;
    p.group = a.dims.num_q_heads / a.dims.num_kv_heads;
    p.block_size = a.dims.block_size;
    p.max_blocks = a.dims.max_blocks_per_seq;
    p.rows = L.rows_per_item;
    p.tc = a.tc ? 1 : 0;
    p.tc_chunk_ok = a.lay.tc_chunks ? 1 : 0;
    p.tc_arrive = a.lay.tc_chunks ? reinterpret_cast<uint32_t *>(a.ws + L.tc_arrive) : nullptr;
    p.wid_cu = a.wid_cu;
    p.wid_cap = a.wid_cap > 0 ? a.wid_cap : -1;
    p.total_warps = a.num_sms * 8;
    AppendParams ap{};
    int64_t grid = 1;
    if (a.append && a.append->total_units > 0) {
        ap = *a.append;
        const int64_t per_cta = (int64_t)kPlanThreads * kPlanAppendUnroll;
        int64_t n = (ap.total_units + per_cta - 1) / per_cta;
        n = n < (int64_t)a.num_sms * 2 ? n : (int64_t)a.num_sms * 2;
        grid += n;
    }
    plan_kernel<<<(unsigned)grid, kPlanThreads, 0, s>>>(p, ap);
    return cudaGetLastError();
}

cudaError_t launch_simt(const FwdArgs &a, cudaStream_t s) {
    const WsLayout &L = a.lay;
    SimtParams p;
    p.q = static_cast<const char *>(a.q);
    p.k = static_cast<const char *>(a.k);
    p.v = static_cast<const char *>(a.v);
    p.out = static_cast<char *>(a.out);
    p.bt = a.bt;
    p.ctx = a.ctx;
    p.qlen = a.qlen;
    p.cu_q = reinterpret_cast<const int32_t *>(a.ws + L.cu_q);
    p.simt_cu = reinterpret_cast<const int32_t *>(a.ws + L.simt_cu);
    p.parts_cu = reinterpret_cast<const int32_t *>(a.ws + L.parts_cu);
    p.comb_cu = reinterpret_cast<const int32_t *>(a.ws + L.comb_cu);
    p.groups = reinterpret_cast<const int32_t *>(a.ws + L.groups);
    p.nchunk = reinterpret_cast<const int32_t *>(a.ws + L.nchunk);
    p.counters = reinterpret_cast<uint32_t *>(a.ws + L.counters);
    p.unit_cnt = reinterpret_cast<uint32_t *>(a.ws + L.unit_cnt);
    p.parts_ml = reinterpret_cast<float2 *>(a.ws + L.parts_ml);
    p.parts_o = reinterpret_cast<float *>(a.ws + L.parts_o);
    p.status = a.status;
    p.num_blocks = a.dims.num_blocks;
    const int64_t dflt = (int64_t)a.dims.num_kv_heads * a.dims.block_size * a.dims.head_dim;
    p.block_stride = a.dims.kv_block_stride ? a.dims.kv_block_stride : dflt;
    const bool e4 = a.dims.kv_dtype == PA_KV_E4M3;
    p.scale_log2 = a.scale * 1.4426950408889634f * (e4 ? a.dims.k_scale : 1.f);
    p.v_scale = e4 ? a.dims.v_scale : 1.f;
    p.num_seqs = a.dims.num_seqs;
    p.q_heads = a.dims.num_q_heads;
    p.kv_heads = a.dims.num_kv_heads;
    p.group = a.dims.num_q_heads / a.dims.num_kv_heads;
    p.block_size = a.dims.block_size;
    p.max_blocks = a.dims.max_blocks_per_seq;
    switch (a.dims.dtype) {
    case PA_F32: return launch_simt_dim<float>(a, p, s);
    case PA_BF16: return launch_simt_dim<__nv_bfloat16>(a, p, s);
    default: return launch_simt_dim<__half>(a, p, s);
    }
}

}  // namespace pkv
