// C-ABI entry points of libpagedkv.so: argument validation, workspace layout and the launch
// sequence.  The declarations, with the meaning of every argument, are in include/pagedkv.h.
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "kv_append.cuh"

namespace pkv {
namespace {

// Device status word (PA_DEV_* bits), one per device that loads the library.
__device__ unsigned g_device_status;

constexpr int kMaxDevices = 64;

}  // namespace

// The status word's device address for the current device (looked up once per device; host
// code must not use the symbol itself as an address).
unsigned *status_ptr() {
    static unsigned *ptrs[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<unsigned *>(p);
    }
    return ptrs[dev];
}

int sm_count() {
    static int cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

namespace {

// A high-priority stream per device on which a call's decode kernel runs beside its tensor-core
// kernel, with the events that fork it from and join it back to the caller's stream.  Created on
// first use and kept until exit; the fork/join enqueue is serialised across host threads.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;

// Caller-owned CUDA events recorded around the attention kernels of later calls
// (pa_set_timing_events): tensor-core kernel start / stop, CUDA-core kernel start / stop.
std::atomic<void *> g_timing[4];

bool record_timing(int which, cudaStream_t st) {
    void *e = g_timing[which].load(std::memory_order_relaxed);
    return !e || cudaEventRecord(static_cast<cudaEvent_t>(e), st) == cudaSuccess;
}

SideStream *side_stream() {
    static SideStream side[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    SideStream &x = side[dev];
    if (!x.join) {
        int least = 0, greatest = 0;
        if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return nullptr;
        if (!x.stream && cudaStreamCreateWithPriority(&x.stream, cudaStreamNonBlocking, greatest) != cudaSuccess) {
            x.stream = nullptr;
            return nullptr;
        }
        if (!x.fork && cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming) != cudaSuccess) {
            x.fork = nullptr;
            return nullptr;
        }
        if (cudaEventCreateWithFlags(&x.join, cudaEventDisableTiming) != cudaSuccess) {
            x.join = nullptr;
            return nullptr;
        }
    }
    return &x;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_dtype(int32_t t) { return t == PA_F32 || t == PA_BF16 || t == PA_F16; }

bool valid_scale(float x) { return x > 0.f && x <= 3.4e38f; }   // finite and positive (NaN fails)

// Bytes of one cached element.
int kv_elem_bytes(int32_t dtype, int32_t kv_dtype) { return kv_dtype == PA_KV_E4M3 ? 1 : elem_bytes(dtype); }

bool overlap(const void *a, size_t an, const void *b, size_t bn) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bn && y < x + an;
}

// Whether the blocks of a pool's planes occupy disjoint bytes: either every plane lies past the
// previous plane's last block (planes outside one another, e.g. layer-first), or the planes sit
// side by side inside each block's stride (e.g. block-first, all layers of a block together).
// Anything else (a zero or short plane stride) lets one plane's copy overwrite another plane.
bool planes_disjoint(int32_t planes, int64_t plane_stride, int64_t block_stride, int64_t blocks,
                     int64_t block_bytes) {
    if (planes <= 1) return true;
    const int64_t bs = block_stride ? block_stride : block_bytes;
    if (plane_stride <= 0) return false;
    if (plane_stride >= blocks * bs) return true;
    return plane_stride >= block_bytes && bs >= (int64_t)planes * plane_stride;
}

pa_status check_dims(const pa_dims *d) {
    if (!d) return PA_ERR_INVALID_ARG;
    if (!valid_dtype(d->dtype)) return PA_ERR_INVALID_ARG;
    if (d->num_seqs < 1 || d->num_seqs > (1 << 20)) return PA_ERR_INVALID_ARG;
    if (d->total_q < d->num_seqs || d->total_q > (int64_t(1) << 30)) return PA_ERR_INVALID_ARG;
    if (d->num_q_heads < 1 || d->num_kv_heads < 1 || d->num_q_heads > 1024) return PA_ERR_INVALID_ARG;
    if (d->num_q_heads % d->num_kv_heads) return PA_ERR_INVALID_ARG;
    if (d->num_blocks < 1 || d->max_blocks_per_seq < 1) return PA_ERR_INVALID_ARG;
    if (d->head_dim != 64 && d->head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (d->block_size != 16 && d->block_size != 32 && d->block_size != 64 && d->block_size != 128)
        return PA_ERR_UNSUPPORTED;
    if (d->kv_dtype != PA_KV_SAME && d->kv_dtype != PA_KV_E4M3) return PA_ERR_INVALID_ARG;
    if (d->kv_dtype == PA_KV_E4M3) {
        if (!valid_scale(d->k_scale) || !valid_scale(d->v_scale)) return PA_ERR_INVALID_ARG;
        if (d->dtype == PA_F32 || d->head_dim != 128) return PA_ERR_UNSUPPORTED;
    }
    const int64_t dense = (int64_t)d->num_kv_heads * d->block_size * d->head_dim;
    if (d->kv_block_stride != 0) {
        if (d->kv_block_stride < dense) return PA_ERR_INVALID_ARG;
        if ((d->kv_block_stride * kv_elem_bytes(d->dtype, d->kv_dtype)) % 16) return PA_ERR_INVALID_ARG;
    }
    if ((int64_t)d->max_blocks_per_seq * d->block_size > (int64_t(1) << 30)) return PA_ERR_INVALID_ARG;
    return PA_OK;
}

}  // namespace

int rows_per_item(const pa_dims &d) {
    const int g = d.num_q_heads / d.num_kv_heads;
    return g >= 4 ? 4 : (g >= 2 ? 2 : 1);
}

WsLayout ws_layout(const pa_dims &d) {
    WsLayout L;
    const size_t S = (size_t)d.num_seqs;
    const int R = rows_per_item(d);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    L.counters = take(kNumCounters * sizeof(uint32_t));
    L.cu_q = take((S + 1) * 4);
    L.simt_cu = take((S + 1) * 4);
    L.parts_cu = take((S + 1) * 4);
    L.comb_cu = take((S + 1) * 4);
    L.groups = take(S * 4);
    L.nchunk = take(S * 4);
    L.tc_cu = take((S + 1) * 4);
    L.tc_seq = take(S * 4);
    // Only sequences whose rows fit one row group are split, into at most kMaxSplits parts of at
    // least C = ceil(work / target) blocks each, so the partial records number at most
    // sum_i Hkv * ceil(nb_i / C) <= target + Hkv * S.
    const int64_t splits = d.max_blocks_per_seq < kMaxSplits ? d.max_blocks_per_seq : kMaxSplits;
    int64_t parts = splits > 1 ? (int64_t)d.num_kv_heads * (int64_t)S * splits : 0;
    const int64_t by_target = kMaxTargetItems + (int64_t)d.num_kv_heads * (int64_t)S;
    L.max_parts = parts < by_target ? parts : by_target;
    L.rows_per_item = R;
    L.parts_ml = take((size_t)L.max_parts * R * sizeof(float) * 2);
    L.parts_o = take((size_t)L.max_parts * R * d.head_dim * sizeof(float));
    L.unit_cnt = take((size_t)L.max_parts * sizeof(uint32_t));
    // chunk partials of the tensor-core kernel, for dims it may take: some sequence may have
    // several query tokens, and the shape is one it supports (decided from the dims alone, so
    // that the size does not depend on the device)
    const int g = d.num_kv_heads > 0 ? d.num_q_heads / d.num_kv_heads : 0;
    L.tc_chunks = d.total_q > d.num_seqs && (d.dtype == PA_BF16 || d.dtype == PA_F16) &&
                  d.kv_dtype == PA_KV_SAME && d.head_dim == 128 &&
                  g >= 1 && g <= kTcTileRows && kTcTileRows % g == 0 && d.block_size >= 16 && d.block_size <= 128;
    L.tc_arrive = take(L.tc_chunks ? (size_t)kMaxTcChunkItems * 8 * sizeof(uint32_t) : 0);
    L.tc_part = take(L.tc_chunks ? (size_t)kMaxTcChunkItems * 2 * kTcTileRows * kTcPartFloats * sizeof(float) : 0);
    L.total = off;
    return L;
}

bool tc_supported(const pa_dims &d) { return tc_shape_supported(d); }

bool widen_eligible(const pa_dims &d) {
    // the tensor-core kernel's shapes, from the dims alone (the call also needs the driver's
    // tensor-map encoder); the planner's prefix of candidate blocks is int32
    const int g = d.num_kv_heads > 0 ? d.num_q_heads / d.num_kv_heads : 0;
    return d.kv_dtype == PA_KV_E4M3 && d.total_q > d.num_seqs && (d.dtype == PA_BF16 || d.dtype == PA_F16) &&
           d.head_dim == 128 && g >= 1 && g <= kTcTileRows && kTcTileRows % g == 0 && d.block_size >= 16 &&
           d.block_size <= 128 && d.total_q < (int64_t(1) << 31) &&
           (int64_t)d.num_seqs * d.max_blocks_per_seq < (int64_t(1) << 31) - 1;
}

int64_t widen_bound_blocks(const pa_dims &d) {
    // a tensor-core sequence has q_len * g >= kTcMinRows, so at most total_q / ceil(16 / g) of them
    const int g = d.num_q_heads / d.num_kv_heads;
    const int64_t qmin = (kTcMinRows + g - 1) / g;
    int64_t n = d.total_q / qmin;
    if (n > d.num_seqs) n = d.num_seqs;
    return n * d.max_blocks_per_seq;
}

WidenLayout widen_layout(const pa_dims &d, size_t base, size_t workspace_bytes) {
    WidenLayout w;
    const size_t S = (size_t)d.num_seqs;
    const size_t blk = (size_t)d.num_kv_heads * d.block_size * d.head_dim * elem_bytes(d.dtype);
    const int64_t bound = widen_bound_blocks(d);
    w.cu = base;
    w.bt = align_up(w.cu + (S + 1) * 4, 256);
    w.k = align_up(w.bt + S * (size_t)d.max_blocks_per_seq * 4, 256);
    w.arrive = align_up(w.k + (size_t)bound * 2 * blk, 256);
    w.part = align_up(w.arrive + (size_t)kMaxTcChunkItems * 8 * sizeof(uint32_t), 256);
    w.end = w.part + (size_t)kMaxTcChunkItems * 2 * kTcTileRows * kTcPartFloats * sizeof(float);
    // the bound's blocks and the chunk regions, else as many blocks as fit and no chunks
    w.chunks = workspace_bytes >= w.end;
    int64_t cap = w.chunks ? bound : (workspace_bytes > w.k ? (int64_t)((workspace_bytes - w.k) / (2 * blk)) : 0);
    if (cap > bound) cap = bound;
    if (cap >= (int64_t(1) << 31) - 1) {   // block ids of the tensor map
        cap = (int64_t(1) << 31) - 2;
        w.chunks = false;
    }
    w.cap = cap;
    w.v = w.k + (size_t)cap * blk;
    return w;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

const char *pa_version(void) { return "pagedkv 0.3 sm_103a"; }

const char *pa_status_string(pa_status s) {
    switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_DEVICE: return "PA_ERR_DEVICE";
    }
    return "PA_ERR_UNKNOWN";
}

size_t pa_forward_workspace_size(const pa_dims *dims) {
    if (check_dims(dims) != PA_OK) return 0;
    return ws_layout(*dims).total;
}

size_t pa_forward_widen_bytes(const pa_dims *dims) {
    if (check_dims(dims) != PA_OK || !widen_eligible(*dims)) return 0;
    const size_t base = ws_layout(*dims).total;
    return widen_layout(*dims, base, 0).end - base;
}

}  // extern "C"

namespace {

// The argument checks of pa_forward, before any device work.
pa_status forward_checks(const pa_dims *dims, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, const int32_t *ctx_lens, const int32_t *q_lens,
                         float scale, const void *out, const void *workspace, size_t workspace_bytes) {
    const pa_status st = check_dims(dims);
    if (st != PA_OK) return st;
    const pa_dims &d = *dims;
    if (!q || !k_cache || !v_cache || !block_tables || !ctx_lens || !q_lens || !out)
        return PA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return PA_ERR_INVALID_ARG;
    if (!aligned(block_tables, 4) || !aligned(ctx_lens, 4) || !aligned(q_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (!(scale == scale)) return PA_ERR_INVALID_ARG;  // NaN scale
    const size_t rows_bytes = (size_t)d.total_q * d.num_q_heads * d.head_dim * elem_bytes(d.dtype);
    if (overlap(q, rows_bytes, out, rows_bytes)) return PA_ERR_INVALID_ARG;
    const WsLayout lay = ws_layout(d);
    if (!workspace || workspace_bytes < lay.total || !aligned(workspace, 256)) return PA_ERR_WORKSPACE;
    return PA_OK;
}

// pa_forward, with the step's new tokens optionally written by the planner's launch (`append`,
// same-dtype caches) before the attention kernels run.
pa_status forward_impl(const pa_dims *dims, const void *q, const void *k_cache, const void *v_cache,
                       const int32_t *block_tables, const int32_t *ctx_lens, const int32_t *q_lens,
                       float scale, void *out, void *workspace, size_t workspace_bytes, pa_stream_t stream,
                       const AppendParams *append) {
    const pa_status st = forward_checks(dims, q, k_cache, v_cache, block_tables, ctx_lens, q_lens, scale, out,
                                        workspace, workspace_bytes);
    if (st != PA_OK) return st;
    const pa_dims &d = *dims;
    const WsLayout lay = ws_layout(d);
    FwdArgs a;
    a.dims = d;
    a.q = q;
    a.k = k_cache;
    a.v = v_cache;
    a.out = out;
    a.bt = block_tables;
    a.ctx = ctx_lens;
    a.qlen = q_lens;
    a.scale = scale;
    a.ws = static_cast<char *>(workspace);
    a.lay = lay;
    a.status = status_ptr();
    a.num_sms = sm_count();
    if (!a.status || a.num_sms <= 0) return PA_ERR_CUDA;
    a.maybe_prefill = d.total_q > d.num_seqs;
    a.tc = a.maybe_prefill && scale > 0.f && d.kv_dtype == PA_KV_SAME && tc_supported(d);
    if (a.maybe_prefill && scale * d.k_scale > 0.f && widen_eligible(d) && tc_supported(d)) {
        // E4M3 caches: the tensor-core kernel reads widened copies of its sequences' blocks
        const WidenLayout w = widen_layout(d, lay.total, workspace_bytes);
        if (w.cap > 0) {
            a.tc = true;
            a.wid_cap = w.cap;
            a.wid_cu = reinterpret_cast<int32_t *>(a.ws + w.cu);
            a.wid_bt = reinterpret_cast<int32_t *>(a.ws + w.bt);
            a.wid_k = a.ws + w.k;
            a.wid_v = a.ws + w.v;
            if (w.chunks) {   // few pair items: their key ranges may run as chunks
                a.lay.tc_chunks = true;
                a.lay.tc_arrive = w.arrive;
                a.lay.tc_part = w.part;
            }
        }
    }
    AppendParams ap;
    if (append) {
        ap = *append;
        ap.status = a.status;
        a.append = &ap;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_plan(a, s) != cudaSuccess) return PA_ERR_CUDA;
    if (a.wid_cap > 0 && launch_widen(a, s) != cudaSuccess) return PA_ERR_CUDA;
    if (a.tc) {
        // the tensor-core kernel right after the planner on the caller's stream, so that its CTAs
        // (one per SM, each holding the SM's whole register file) are dispatched first; the decode
        // kernel, forked onto the side stream, takes each SM as its tensor-core CTA finishes.  Both
        // only read the plan and write disjoint output rows.
        std::lock_guard<std::mutex> lock(g_side_mu);
        SideStream *x = side_stream();
        if (!x) return PA_ERR_CUDA;
        if (cudaEventRecord(x->fork, s) != cudaSuccess || cudaStreamWaitEvent(x->stream, x->fork, 0) != cudaSuccess)
            return PA_ERR_CUDA;
        if (!record_timing(0, s) || launch_tc(a, s) != cudaSuccess || !record_timing(1, s)) return PA_ERR_CUDA;
        if (!record_timing(2, x->stream) || launch_simt(a, x->stream) != cudaSuccess || !record_timing(3, x->stream))
            return PA_ERR_CUDA;
        if (cudaEventRecord(x->join, x->stream) != cudaSuccess || cudaStreamWaitEvent(s, x->join, 0) != cudaSuccess)
            return PA_ERR_CUDA;
    } else if (!record_timing(2, s) || launch_simt(a, s) != cudaSuccess || !record_timing(3, s)) {
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

}  // namespace

extern "C" {

pa_status pa_set_timing_events(void *tc_start, void *tc_stop, void *cc_start, void *cc_stop) {
    if (!tc_start != !tc_stop || !cc_start != !cc_stop) return PA_ERR_INVALID_ARG;
    g_timing[0].store(tc_start);
    g_timing[1].store(tc_stop);
    g_timing[2].store(cc_start);
    g_timing[3].store(cc_stop);
    return PA_OK;
}

pa_status pa_forward(const pa_dims *dims, const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_tables, const int32_t *ctx_lens, const int32_t *q_lens,
                     float scale, void *out, void *workspace, size_t workspace_bytes,
                     pa_stream_t stream) {
    return forward_impl(dims, q, k_cache, v_cache, block_tables, ctx_lens, q_lens, scale, out, workspace,
                        workspace_bytes, stream, nullptr);
}

pa_status pa_forward_append(const pa_dims *dims, const void *q, const void *k_new, const void *v_new,
                            const int64_t *slot_mapping, void *k_cache, void *v_cache,
                            const int32_t *block_tables, const int32_t *ctx_lens, const int32_t *q_lens,
                            float scale, void *out, void *workspace, size_t workspace_bytes,
                            pa_stream_t stream) {
    const pa_status st = forward_checks(dims, q, k_cache, v_cache, block_tables, ctx_lens, q_lens, scale, out,
                                        workspace, workspace_bytes);
    if (st != PA_OK) return st;
    const pa_dims &d = *dims;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(slot_mapping, 8)) return PA_ERR_INVALID_ARG;
    // the new tokens are the call's query tokens: [total_q, Hkv, d] of dims->dtype
    kv_append_dims ad;
    ad.dtype = d.dtype;
    ad.num_tokens = d.total_q;
    ad.num_kv_heads = d.num_kv_heads;
    ad.head_dim = d.head_dim;
    ad.block_size = d.block_size;
    ad.num_blocks = d.num_blocks;
    ad.kv_block_stride = d.kv_block_stride;
    ad.num_layers = 1;
    ad.new_layer_stride = 0;
    ad.cache_layer_stride = 0;
    ad.kv_dtype = d.kv_dtype;
    ad.k_scale = d.k_scale;
    ad.v_scale = d.v_scale;
    if (d.kv_dtype == PA_KV_E4M3) {
        // quantising append: its own launch, then the attention call
        const pa_status sa = kv_append(&ad, k_new, v_new, slot_mapping, k_cache, v_cache, stream);
        if (sa != PA_OK) return sa;
        return forward_impl(dims, q, k_cache, v_cache, block_tables, ctx_lens, q_lens, scale, out, workspace,
                            workspace_bytes, stream, nullptr);
    }
    AppendParams ap;
    fill_append_params(ad, k_new, v_new, slot_mapping, k_cache, v_cache, nullptr, ap);
    return forward_impl(dims, q, k_cache, v_cache, block_tables, ctx_lens, q_lens, scale, out, workspace,
                        workspace_bytes, stream, &ap);
}

pa_status kv_append(const kv_append_dims *dims, const void *k_new, const void *v_new,
                    const int64_t *slot_mapping, void *k_cache, void *v_cache, pa_stream_t stream) {
    if (!dims) return PA_ERR_INVALID_ARG;
    const kv_append_dims &d = *dims;
    if (!valid_dtype(d.dtype) || d.num_tokens < 0 || d.num_kv_heads < 1 || d.head_dim < 1 ||
        d.block_size < 1 || d.num_blocks < 1 || d.num_layers < 1)
        return PA_ERR_INVALID_ARG;
    if (d.kv_dtype != PA_KV_SAME && d.kv_dtype != PA_KV_E4M3) return PA_ERR_INVALID_ARG;
    if (d.kv_dtype == PA_KV_E4M3 && (!valid_scale(d.k_scale) || !valid_scale(d.v_scale)))
        return PA_ERR_INVALID_ARG;
    if (d.num_tokens == 0) return PA_OK;
    const int eb = elem_bytes(d.dtype);                 // new tokens
    const int cb = kv_elem_bytes(d.dtype, d.kv_dtype);  // caches
    if ((d.head_dim * eb) % 16 || (d.head_dim * cb) % 16) return PA_ERR_UNSUPPORTED;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(slot_mapping, 8))
        return PA_ERR_INVALID_ARG;
    const int64_t dense = (int64_t)d.num_kv_heads * d.block_size * d.head_dim;
    if (d.kv_block_stride && (d.kv_block_stride < dense || (d.kv_block_stride * cb) % 16))
        return PA_ERR_INVALID_ARG;
    if ((d.new_layer_stride * eb) % 16 || (d.cache_layer_stride * cb) % 16) return PA_ERR_INVALID_ARG;
    if (d.num_layers > 1) {
        const int64_t bs = d.kv_block_stride ? d.kv_block_stride : dense;
        if (d.new_layer_stride && d.new_layer_stride < d.num_tokens * d.num_kv_heads * d.head_dim)
            return PA_ERR_INVALID_ARG;
        if (d.cache_layer_stride && d.cache_layer_stride < d.num_blocks * bs) return PA_ERR_INVALID_ARG;
    }
    unsigned *status = status_ptr();
    const int sms = sm_count();
    if (!status || sms <= 0) return PA_ERR_CUDA;
    if (launch_kv_append(d, k_new, v_new, slot_mapping, k_cache, v_cache, status, sms,
                         reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}

pa_status block_copy(const block_copy_dims *dims, const void *src, void *dst, const int64_t *pairs,
                     pa_stream_t stream) {
    if (!dims) return PA_ERR_INVALID_ARG;
    const block_copy_dims &d = *dims;
    if (d.num_pairs < 0 || d.num_planes < 1 || d.block_bytes <= 0 || d.src_num_blocks < 1 ||
        d.dst_num_blocks < 1 || d.max_ctas < 0)
        return PA_ERR_INVALID_ARG;
    if (d.num_pairs == 0) return PA_OK;
    if (!src || !dst || !pairs) return PA_ERR_INVALID_ARG;
    if (d.block_bytes % 16 || d.src_plane_stride % 16 || d.dst_plane_stride % 16 ||
        d.src_block_stride % 16 || d.dst_block_stride % 16)
        return PA_ERR_INVALID_ARG;
    if (d.src_block_stride && d.src_block_stride < d.block_bytes) return PA_ERR_INVALID_ARG;
    if (d.dst_block_stride && d.dst_block_stride < d.block_bytes) return PA_ERR_INVALID_ARG;
    if (!planes_disjoint(d.num_planes, d.src_plane_stride, d.src_block_stride, d.src_num_blocks, d.block_bytes) ||
        !planes_disjoint(d.num_planes, d.dst_plane_stride, d.dst_block_stride, d.dst_num_blocks, d.block_bytes))
        return PA_ERR_INVALID_ARG;
    if (!aligned(src, 16) || !aligned(dst, 16) || !aligned(pairs, 8)) return PA_ERR_INVALID_ARG;
    unsigned *status = status_ptr();
    const int sms = sm_count();
    if (!status || sms <= 0) return PA_ERR_CUDA;
    if (launch_block_copy(d, src, dst, pairs, status, sms, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}

pa_status pa_get_device_status(uint32_t *flags, pa_stream_t stream) {
    if (!flags) return PA_ERR_INVALID_ARG;
    *flags = 0;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return PA_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof v) != cudaSuccess) return PA_ERR_CUDA;
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero) != cudaSuccess) return PA_ERR_CUDA;
    *flags = v;
    return v ? PA_ERR_DEVICE : PA_OK;
}

}  // extern "C"
