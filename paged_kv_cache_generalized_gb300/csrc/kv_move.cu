// Cache append (scatter of new tokens into their slots) and whole-block copy (copy-on-write,
// swap-in, swap-out).  Both move bits only: 16-byte vectors, no float arithmetic, so NaN payloads
// survive.  Grids are persistent (a multiple of the SM count) and stride over the work.
//
// Append: "SOSP 2023論文解説: PagedAttention", section "ブロックテーブルによるメモリ管理" -- a
// new token goes into its sequence's current block while it has room, else into a fresh block;
// the caller's allocator encodes that choice as slot = physical block * B + offset.
// Copy: same page, section "Copy-on-Writeによるメモリ共有"; "Stateful Large Language Model
// Serving with Pensieve", sections "GPU-CPU 2層キャッシュ構造" / "パイプライン化されたswap-in".
#include "common.cuh"
#include "internal.h"
#include "kv_append.cuh"

namespace pkv {
namespace {

// The same-dtype append (kv_append.cuh's loop over the whole grid).
__global__ void __launch_bounds__(256) kv_append_kernel(AppendParams p) { append_loop(p, blockIdx.x, gridDim.x); }

// E4M3 caches: the new tokens (bf16 / f16 / f32) are quantised on the way in.  One unit is 16
// consecutive elements of one (layer, token, head) row: read, widened to fp32, multiplied by the
// fp32 reciprocal of the scale, rounded to E4M3 (nearest even, saturating at 448), 16 bytes out.
struct AppendE4Params {
    const char *k_new;
    const char *v_new;
    const int64_t *slots;
    uint8_t *k_cache;
    uint8_t *v_cache;
    unsigned *status;
    int64_t units_per_layer;   // num_tokens * Hkv * (d / 16)
    int64_t total_units;       // * num_layers
    int64_t num_blocks;
    int64_t block_stride;      // codes between physical blocks
    int64_t new_layer;         // elements between layers of k_new / v_new
    int64_t cache_layer;       // codes between layers of the caches
    float inv_k, inv_v;
    int32_t kv_heads, head_dim, chunks, block_size;
};

template <typename T>
__device__ __forceinline__ uint4 quantize16(const T *src, float inv) {
    float f[16];
    load_f<T, 16>(src, f);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = (uint32_t)e4m3x2_from_f32(f[4 * i] * inv, f[4 * i + 1] * inv) |
               ((uint32_t)e4m3x2_from_f32(f[4 * i + 2] * inv, f[4 * i + 3] * inv) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename T>
__global__ void __launch_bounds__(256) kv_append_e4m3_kernel(AppendE4Params p) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < p.total_units; u += stride) {
        const int64_t layer = u / p.units_per_layer;
        const int64_t in_layer = u - layer * p.units_per_layer;
        const int64_t row = in_layer / p.chunks;               // token * Hkv + head
        const int c = (int)(in_layer - row * p.chunks);
        const int64_t t = row / p.kv_heads;
        const int h = (int)(row - t * p.kv_heads);
        const int64_t slot = __ldg(p.slots + t);
        if (slot < 0) continue;                                 // padding
        const int64_t blk = slot / p.block_size;
        if (blk >= p.num_blocks) {
            if (c == 0 && h == 0 && layer == 0) report(p.status, PA_DEV_BAD_SLOT);
            continue;
        }
        const int off = (int)(slot - blk * p.block_size);
        const int64_t src = (layer * p.new_layer + row * p.head_dim + (int64_t)c * 16) * (int64_t)sizeof(T);
        const int64_t dst = layer * p.cache_layer + blk * p.block_stride +
                            ((int64_t)h * p.block_size + off) * p.head_dim + (int64_t)c * 16;
        const uint4 kq = quantize16(reinterpret_cast<const T *>(p.k_new + src), p.inv_k);
        const uint4 vq = quantize16(reinterpret_cast<const T *>(p.v_new + src), p.inv_v);
        *reinterpret_cast<uint4 *>(p.k_cache + dst) = kq;
        *reinterpret_cast<uint4 *>(p.v_cache + dst) = vq;
    }
}

struct CopyParams {
    const uint4 *src;
    uint4 *dst;
    const int64_t *pairs;
    unsigned *status;
    int64_t num_pairs;
    int64_t units;             // 16-byte units per block
    int64_t tiles_per_block;   // ceil(units / kCopyTileUnits)
    int64_t total_tiles;       // pairs * planes * tiles_per_block
    int64_t src_plane16, dst_plane16, src_block16, dst_block16;
    int64_t src_blocks, dst_blocks;
    int32_t planes;
};

constexpr int kCopyThreads = 256;
constexpr int kCopyPerThread = 4;
constexpr int kCopyTileUnits = kCopyThreads * kCopyPerThread;   // 16 KiB per tile

// One CTA moves one 16 KiB tile of one (pair, plane) per iteration: every thread issues its
// four 16-byte loads before its stores.  Tile index -> (pair, plane, tile) with the tile fastest.
__global__ void __launch_bounds__(kCopyThreads) block_copy_kernel(CopyParams p) {
    for (int64_t tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x) {
        const int64_t pp = tile / p.tiles_per_block;           // pair * planes + plane
        const int64_t part = tile - pp * p.tiles_per_block;
        const int64_t pair = pp / p.planes;
        const int64_t plane = pp - pair * p.planes;
        const int64_t s = __ldg(p.pairs + 2 * pair);
        const int64_t t = __ldg(p.pairs + 2 * pair + 1);
        if (s < 0 || s >= p.src_blocks || t < 0 || t >= p.dst_blocks) {
            if (threadIdx.x == 0 && plane == 0 && part == 0) report(p.status, PA_DEV_BAD_PAIR);
            continue;
        }
        const uint4 *src = p.src + plane * p.src_plane16 + s * p.src_block16;
        uint4 *dst = p.dst + plane * p.dst_plane16 + t * p.dst_block16;
        const int64_t u0 = part * kCopyTileUnits + threadIdx.x;
        uint4 v[kCopyPerThread];
#pragma unroll
        for (int k = 0; k < kCopyPerThread; ++k) {
            const int64_t u = u0 + k * kCopyThreads;
            if (u < p.units) v[k] = __ldcs(src + u);
        }
#pragma unroll
        for (int k = 0; k < kCopyPerThread; ++k) {
            const int64_t u = u0 + k * kCopyThreads;
            if (u < p.units) __stcs(dst + u, v[k]);
        }
    }
}

}  // namespace

namespace {

cudaError_t launch_kv_append_e4m3(const kv_append_dims &d, const void *k_new, const void *v_new,
                                  const int64_t *slots, void *k_cache, void *v_cache, unsigned *status,
                                  int num_sms, cudaStream_t s) {
    AppendE4Params p;
    p.k_new = static_cast<const char *>(k_new);
    p.v_new = static_cast<const char *>(v_new);
    p.slots = slots;
    p.k_cache = static_cast<uint8_t *>(k_cache);
    p.v_cache = static_cast<uint8_t *>(v_cache);
    p.status = status;
    p.kv_heads = d.num_kv_heads;
    p.head_dim = d.head_dim;
    p.chunks = d.head_dim / 16;
    p.block_size = d.block_size;
    p.num_blocks = d.num_blocks;
    const int64_t row_elems = (int64_t)d.num_kv_heads * d.head_dim;
    p.block_stride = d.kv_block_stride ? d.kv_block_stride : row_elems * d.block_size;
    p.new_layer = d.new_layer_stride ? d.new_layer_stride : d.num_tokens * row_elems;
    p.cache_layer = d.cache_layer_stride ? d.cache_layer_stride : d.num_blocks * p.block_stride;
    p.inv_k = 1.0f / d.k_scale;
    p.inv_v = 1.0f / d.v_scale;
    p.units_per_layer = d.num_tokens * d.num_kv_heads * (int64_t)p.chunks;
    p.total_units = p.units_per_layer * d.num_layers;
    if (p.total_units == 0) return cudaSuccess;
    int64_t grid = (p.total_units + 255) / 256;
    grid = grid < (int64_t)num_sms * 8 ? grid : (int64_t)num_sms * 8;
    switch (d.dtype) {
    case PA_F32: kv_append_e4m3_kernel<float><<<(unsigned)grid, 256, 0, s>>>(p); break;
    case PA_BF16: kv_append_e4m3_kernel<__nv_bfloat16><<<(unsigned)grid, 256, 0, s>>>(p); break;
    default: kv_append_e4m3_kernel<__half><<<(unsigned)grid, 256, 0, s>>>(p); break;
    }
    return cudaGetLastError();
}

}  // namespace

void fill_append_params(const kv_append_dims &d, const void *k_new, const void *v_new, const int64_t *slots,
                        void *k_cache, void *v_cache, unsigned *status, AppendParams &p) {
    const int eb = elem_bytes(d.dtype);
    p.k_new = static_cast<const uint4 *>(k_new);
    p.v_new = static_cast<const uint4 *>(v_new);
    p.slots = slots;
    p.k_cache = static_cast<uint4 *>(k_cache);
    p.v_cache = static_cast<uint4 *>(v_cache);
    p.status = status;
    p.num_tokens = d.num_tokens;
    p.kv_heads = d.num_kv_heads;
    p.chunks = d.head_dim * eb / 16;
    p.block_size = d.block_size;
    p.num_blocks = d.num_blocks;
    const int64_t row_elems = (int64_t)d.num_kv_heads * d.head_dim;
    const int64_t bstride = d.kv_block_stride ? d.kv_block_stride : row_elems * d.block_size;
    const int64_t nls = d.new_layer_stride ? d.new_layer_stride : d.num_tokens * row_elems;
    const int64_t cls = d.cache_layer_stride ? d.cache_layer_stride : d.num_blocks * bstride;
    p.block_stride16 = bstride * eb / 16;
    p.new_layer16 = nls * eb / 16;
    p.cache_layer16 = cls * eb / 16;
    p.units_per_layer = d.num_tokens * d.num_kv_heads * (int64_t)p.chunks;
    p.total_units = p.units_per_layer * d.num_layers;
}

cudaError_t launch_kv_append(const kv_append_dims &d, const void *k_new, const void *v_new,
                             const int64_t *slots, void *k_cache, void *v_cache, unsigned *status,
                             int num_sms, cudaStream_t s) {
    if (d.kv_dtype == PA_KV_E4M3)
        return launch_kv_append_e4m3(d, k_new, v_new, slots, k_cache, v_cache, status, num_sms, s);
    AppendParams p;
    fill_append_params(d, k_new, v_new, slots, k_cache, v_cache, status, p);
    if (p.total_units == 0) return cudaSuccess;
    const int64_t per_cta = 256LL * kAppendUnroll;
    int64_t grid = (p.total_units + per_cta - 1) / per_cta;
    grid = grid < (int64_t)num_sms * 8 ? grid : (int64_t)num_sms * 8;
    kv_append_kernel<<<(unsigned)grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_block_copy(const block_copy_dims &d, const void *src, void *dst,
                              const int64_t *pairs, unsigned *status, int num_sms,
                              cudaStream_t s) {
    CopyParams p;
    p.src = static_cast<const uint4 *>(src);
    p.dst = static_cast<uint4 *>(dst);
    p.pairs = pairs;
    p.status = status;
    p.num_pairs = d.num_pairs;
    p.planes = d.num_planes;
    p.units = d.block_bytes / 16;
    p.tiles_per_block = (p.units + kCopyTileUnits - 1) / kCopyTileUnits;
    p.total_tiles = d.num_pairs * d.num_planes * p.tiles_per_block;
    p.src_plane16 = d.src_plane_stride / 16;
    p.dst_plane16 = d.dst_plane_stride / 16;
    p.src_block16 = (d.src_block_stride ? d.src_block_stride : d.block_bytes) / 16;
    p.dst_block16 = (d.dst_block_stride ? d.dst_block_stride : d.block_bytes) / 16;
    p.src_blocks = d.src_num_blocks;
    p.dst_blocks = d.dst_num_blocks;
    if (p.total_tiles == 0) return cudaSuccess;
    int64_t grid = p.total_tiles < (int64_t)num_sms * 8 ? p.total_tiles : (int64_t)num_sms * 8;
    if (d.max_ctas > 0 && grid > d.max_ctas) grid = d.max_ctas;
    block_copy_kernel<<<(unsigned)grid, kCopyThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv
