// The cache append of tokens whose K/V have the caches' element type, as a device loop shared by
// kv_append_kernel and by the first launch of pa_forward_append.  A new token goes into its
// sequence's current block while it has room, else into a fresh block
// ("SOSP 2023論文解説: PagedAttention", section "ブロックテーブルによるメモリ管理"); the caller's
// allocator encodes that choice as slot = physical block * B + offset.  Bits only: 16-byte
// vectors, no float arithmetic, so NaN payloads survive.
#pragma once

#include "common.cuh"

namespace pkv {

struct AppendParams {
    const uint4 *k_new;
    const uint4 *v_new;
    const int64_t *slots;
    uint4 *k_cache;
    uint4 *v_cache;
    unsigned *status;
    int64_t num_tokens;
    int64_t units_per_layer;   // num_tokens * Hkv * chunks
    int64_t total_units;       // * num_layers
    int64_t num_blocks;
    int64_t block_stride16;    // 16-byte units between physical blocks
    int64_t new_layer16;       // 16-byte units between layers of k_new / v_new
    int64_t cache_layer16;     // 16-byte units between layers of the caches
    int32_t kv_heads;
    int32_t chunks;            // 16-byte units per (token, head) row: d * elem / 16
    int32_t block_size;
};

constexpr int kAppendUnroll = 4;

// Units of the append done by block `blk` of `nblk` blocks (of blockDim.x threads each).  One
// thread moves U 16-byte units of K and of V per iteration (all loads issued before the stores).
// Unit u -> (layer, token, head, chunk) with chunk fastest, so consecutive threads read
// consecutive bytes of k_new and write one contiguous row of a cache block.
template <int U = kAppendUnroll>
__device__ __forceinline__ void append_loop(const AppendParams &p, int64_t blk, int64_t nblk) {
    const int64_t stride = nblk * blockDim.x * U;
    for (int64_t base = (blk * blockDim.x) * U + threadIdx.x; base < p.total_units; base += stride) {
        uint4 kv[U], vv[U];
        int64_t dst[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t u = base + (int64_t)k * blockDim.x;
            dst[k] = -1;
            if (u >= p.total_units) continue;
            const int64_t layer = u / p.units_per_layer;
            const int64_t in_layer = u - layer * p.units_per_layer;
            const int64_t row = in_layer / p.chunks;           // token * Hkv + head
            const int c = (int)(in_layer - row * p.chunks);
            const int64_t t = row / p.kv_heads;
            const int h = (int)(row - t * p.kv_heads);
            const int64_t slot = __ldg(p.slots + t);
            if (slot < 0) continue;                             // padding
            const int64_t blk_id = slot / p.block_size;
            if (blk_id >= p.num_blocks) {
                if (c == 0 && h == 0 && layer == 0) report(p.status, PA_DEV_BAD_SLOT);
                continue;
            }
            const int off = (int)(slot - blk_id * p.block_size);
            const int64_t src = layer * p.new_layer16 + row * p.chunks + c;
            dst[k] = layer * p.cache_layer16 + blk_id * p.block_stride16 +
                     ((int64_t)h * p.block_size + off) * p.chunks + c;
            kv[k] = __ldcs(p.k_new + src);
            vv[k] = __ldcs(p.v_new + src);
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (dst[k] < 0) continue;
            p.k_cache[dst[k]] = kv[k];
            p.v_cache[dst[k]] = vv[k];
        }
    }
}

}  // namespace pkv
