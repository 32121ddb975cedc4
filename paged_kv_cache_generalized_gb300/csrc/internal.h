// Internal interface between the C-ABI entry points (api.cu) and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

// Query rows handled by one CUDA-core work item: (token, head-in-group) pairs of one KV head.
// Chosen per call from the GQA group size.
constexpr int kMaxRowsPerItem = 4;
// Multi-token sequences with at least this many query rows per KV head (q_len * g) go to the
// tensor-core kernel when it supports the dtype and head_dim.
constexpr int kTcMinRows = 16;
// Rows of one tensor-core tile (UMMA M).
constexpr int kTcTileRows = 128;
// Query tiles of one (sequence, KV head) processed together by one tensor-core work item (they
// share every K/V tile load).
constexpr int kTcTilesPerItem = 2;
// Launches with fewer tensor-core pair items than CTAs split each pair's key range into chunks
// run by separate CTAs and merged by the logsumexp rule; at most this many items then (each
// chunk item has a partial-result slot of 2 x 128 rows in the workspace), each chunk at least
// kTcMinChunkTiles KV tiles and at least 2 tiles.
constexpr int kMaxTcChunkItems = 120;
constexpr int kTcMinChunkTiles = 4;
// At most this many chunks per pair: the warps that merge a pair read every chunk's partial rows
// (528 bytes each), so the merge grows with the chunk count while the chunks' work shrinks.
constexpr int kTcMaxChunksPerPair = 16;
constexpr int kTcPartFloats = 4 + 128;   // per row: running max (log2 units), sum, 2 pad, o[128]
constexpr int kTcPartO = 4;               // o starts 16 bytes into the row (rows are 528 bytes)

// KV tiles (128 keys) of tensor-core pair pi of a sequence with c cached tokens and `rows` query
// rows per KV head (q_len * g): through the causal position of the pair's last row.
__host__ __device__ inline int tc_pair_tiles(int64_t c, int rows, int g, int pi) {
    const int tph = (rows + kTcTileRows - 1) / kTcTileRows;
    const int qt = 2 * pi + 1 < tph ? 2 * pi + 1 : 2 * pi;
    const int valid = rows - qt * kTcTileRows < kTcTileRows ? rows - qt * kTcTileRows : kTcTileRows;
    const int64_t pmax = c + (int64_t)qt * (kTcTileRows / g) + (valid - 1) / g;
    return (int)((pmax + 128) / 128);
}
// Chunks of a pair of nt KV tiles for chunk length lc (0: no chunking): at most nt / 2, so that
// every chunk holds at least 2 tiles, and at most kTcMaxChunksPerPair.
__host__ __device__ inline int tc_pair_chunks(int nt, int lc) {
    if (lc <= 0) return 1;
    int c = (nt + lc - 1) / lc;
    const int cap = nt / 2 < kTcMaxChunksPerPair ? nt / 2 : kTcMaxChunksPerPair;
    if (c > cap) c = cap;
    return c > 1 ? c : 1;
}

// Upper bound on the KV splits of one CUDA-core work item's rows.
constexpr int kMaxSplits = 64;
// The planner sizes splits for about 16 work items per warp of the persistent grid, capped here
// (enough for 256 SMs x 8 warps); the workspace bound on split partials follows from it.
constexpr int64_t kMaxTargetItems = 32768;
// Smallest KV split of a CUDA-core work item, in keys.
constexpr int kMinSplitTokens = 256;
// Longest sequence (cached + new tokens) a call accepts, so that token positions fit int32.
constexpr int64_t kMaxSeqTokens = (int64_t)1 << 30;

// Counters at the start of the workspace.
enum Counter : int {
    kSimtNext = 0,    // next CUDA-core item to take
    kSimtTotal = 1,   // number of CUDA-core items
    kTcNext = 2,      // next tensor-core tile to take
    kTcTotal = 3,     // number of tensor-core tiles
    kCombTotal = 4,   // number of split-KV rows to combine (row groups x rows)
    kChunkBlocks = 5, // KV blocks per CUDA-core split
    kTcChunk = 6,     // KV tiles per tensor-core chunk (0: pair items are not chunked)
    kWidTotal = 7,    // widened blocks to write (E4M3 caches on the tensor-core kernel)
    kNumCounters = 16
};

// Byte offsets of the workspace regions (all 256-byte aligned).
struct WsLayout {
    size_t counters;   // uint32 [kNumCounters]
    size_t cu_q;       // int32 [S+1]  exclusive prefix of q_lens
    size_t simt_cu;    // int32 [S+1]  prefix of CUDA-core items
    size_t parts_cu;   // int32 [S+1]  prefix of split partial records
    size_t comb_cu;    // int32 [S+1]  prefix of rows to combine
    size_t groups;     // int32 [S]    row groups per KV head (CUDA-core sequences)
    size_t nchunk;     // int32 [S]    KV splits per row group (CUDA-core sequences)
    size_t tc_cu;      // int32 [S+1]  prefix of tensor-core tiles over sequences in rank order
    size_t tc_seq;     // int32 [S]    sequence at each rank
    size_t parts_ml;   // float2 [max_parts * R]  (running max in log2 units, sum)
    size_t parts_o;    // float  [max_parts * R * d]
    size_t unit_cnt;   // uint32 [max_parts]  splits finished per split row group (zeroed by the planner)
    size_t tc_arrive;  // uint32 [kMaxTcChunkItems * 8]  chunks finished per (pair, tile, warp)
    size_t tc_part;    // float [kMaxTcChunkItems * 2 * 128 * kTcPartFloats]  chunk partial rows
    bool tc_chunks;    // the two regions above exist (dims the tensor-core kernel may take)
    size_t total;
    int64_t max_parts;
    int rows_per_item; // R
};

WsLayout ws_layout(const pa_dims &d);

// E4M3 caches on the tensor-core kernel.  The blocks of the sequences it takes are widened
// (exactly) to the query dtype into scratch past the workspace layout: the candidate-block prefix,
// a remapped block table, then `cap` widened K blocks and `cap` V blocks.  `cap` is what the
// caller's workspace holds, at most the bound for the dims; sequences whose blocks do not fit run
// on the CUDA-core kernels.  A workspace that holds the bound's blocks also holds, after them, the
// tensor-core kernel's chunk regions (16-bit caches keep those in the required layout).
struct WidenLayout {
    size_t cu;         // int32 [S+1]  prefix of candidate sequences' blocks (planner)
    size_t bt;         // int32 [S * max_blocks_per_seq]  block table of the widened blocks
    size_t k, v;       // [cap, Hkv, B, d] in the query dtype
    size_t arrive;     // chunk arrival counters, as WsLayout::tc_arrive (when `chunks`)
    size_t part;       // chunk partial rows, as WsLayout::tc_part (when `chunks`)
    size_t end;        // first byte past the chunk regions for the bound (the size to ask for)
    int64_t cap;       // widened blocks the caller's workspace holds (0: no widening)
    bool chunks;       // the workspace holds the bound's blocks and the chunk regions
};
// Whether E4M3 dims may widen at all (total_q > num_seqs and a shape the tensor-core kernel takes).
bool widen_eligible(const pa_dims &d);
// Widened blocks that cover every sequence the tensor-core kernel may take for these dims.
int64_t widen_bound_blocks(const pa_dims &d);
WidenLayout widen_layout(const pa_dims &d, size_t base, size_t workspace_bytes);
int rows_per_item(const pa_dims &d);
bool tc_supported(const pa_dims &d);
bool tc_shape_supported(const pa_dims &d);  // attn_tc.cu

struct AppendParams;    // kv_append.cuh

struct FwdArgs {
    pa_dims dims;
    const void *q;
    const void *k;
    const void *v;
    void *out;
    const int32_t *bt;
    const int32_t *ctx;
    const int32_t *qlen;
    float scale;
    char *ws;
    WsLayout lay;
    unsigned *status;
    int num_sms;
    bool tc;            // tensor-core kernel available for this call
    bool maybe_prefill; // some sequence may have q_len > 1
    const AppendParams *append = nullptr;   // new tokens written by the planner's launch (or none)
    // E4M3 caches on the tensor-core kernel (wid_cap > 0): the widening scratch
    int64_t wid_cap = 0;
    int32_t *wid_cu = nullptr;
    int32_t *wid_bt = nullptr;
    void *wid_k = nullptr;
    void *wid_v = nullptr;
};

cudaError_t launch_plan(const FwdArgs &a, cudaStream_t s);
cudaError_t launch_simt(const FwdArgs &a, cudaStream_t s);
cudaError_t launch_tc(const FwdArgs &a, cudaStream_t s);
// The widening of the planned sequences' E4M3 blocks (widen.cu), after the planner.
cudaError_t launch_widen(const FwdArgs &a, cudaStream_t s);

cudaError_t launch_kv_append(const kv_append_dims &d, const void *k_new, const void *v_new,
                             const int64_t *slots, void *k_cache, void *v_cache, unsigned *status,
                             int num_sms, cudaStream_t s);
// The same-dtype append's parameters (kv_move.cu); d.kv_dtype must be PA_KV_SAME.
void fill_append_params(const kv_append_dims &d, const void *k_new, const void *v_new, const int64_t *slots,
                        void *k_cache, void *v_cache, unsigned *status, AppendParams &p);
cudaError_t launch_block_copy(const block_copy_dims &d, const void *src, void *dst,
                              const int64_t *pairs, unsigned *status, int num_sms,
                              cudaStream_t s);

// Tensor maps (tensor_map.cu): a 3-D tiled map (dims d0 innermost, d1, d2; byte strides of d1 and
// d2; box b0 x b1 x b2 elements, b0 * element size = 128 bytes) with 128-byte swizzle.
// dtype code of make_map_3d for one-byte elements (E4M3 caches)
constexpr int kMapBytes = 100;
bool tensor_maps_available();
bool make_map_3d(CUtensorMap *map, int dtype, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                 uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2);

// The current device's status word (device address) and SM count; nullptr / 0 on failure.
unsigned *status_ptr();
int sm_count();

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int elem_bytes(int dtype) { return dtype == PA_F32 ? 4 : 2; }

}  // namespace pkv
