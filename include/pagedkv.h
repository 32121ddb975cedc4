/*
 * pagedkv.h -- C ABI of libpagedkv.so: generalized paged attention, cache append and block
 * copy on one GB300 (sm_103a).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All tensors are caller-owned, plain pointers; the library never allocates, never frees and
 *    never copies between host and device on the caller's behalf.  Device pointers must belong to
 *    the current CUDA device.  Host pointers are accepted only where a call says so (and must be
 *    page-locked, e.g. cudaHostAlloc / torch pin_memory, so the GPU can address them).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream)
 *    and never synchronises, except pa_get_device_status.  No call falls back to the CPU.
 *  - Shapes are described by small structs passed by pointer; element strides are given in
 *    elements of the tensor's dtype, byte strides say so.
 *  - Host-side validation (shapes, dtypes, alignment, supported sizes, workspace size) returns a
 *    pa_status != PA_OK and launches nothing.  Data-dependent faults that only the device can see
 *    (an out-of-range block id or slot, inconsistent lengths) are never trapped: the offending
 *    work is skipped, and a bit is set in a per-device status word that pa_get_device_status
 *    reads and clears.
 *  - Calls that share a workspace must not run concurrently.
 *
 * Notation (as on the pages): B = block size in tokens; Hq / Hkv = query / KV heads,
 * g = Hq / Hkv (GQA group); d = head_dim.  Sequence i has c_i = ctx_lens[i] tokens cached before
 * this step and q_i = q_lens[i] >= 1 new tokens; n_i = c_i + q_i; T = sum_i q_i.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *pa_stream_t; /* same type as cudaStream_t */

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,  /* a NULL pointer, a bad shape, stride or alignment */
    PA_ERR_UNSUPPORTED = 2,  /* a valid request the library does not implement (e.g. head_dim) */
    PA_ERR_WORKSPACE = 3,    /* workspace missing, too small or misaligned */
    PA_ERR_CUDA = 4,         /* a CUDA runtime call (launch, attribute query) failed */
    PA_ERR_DEVICE = 5        /* pa_get_device_status found device-side error bits */
} pa_status;

typedef enum { PA_F32 = 0, PA_BF16 = 1, PA_F16 = 2 } pa_dtype;

/* Storage of the K/V caches.  PA_KV_SAME: elements of the call's `dtype`.  PA_KV_E4M3: one-byte
 * FP8 E4M3 codes (1 sign, 4 exponent bits with bias 7, 3 fraction bits; no infinities;
 * S.1111.111 is NaN) with one float scale for K and one for V: a cached element's value is its
 * code's value times k_scale (v_scale).  The pages name fewer bits per element as the third way
 * to shrink the cache ("KVキャッシュ管理の教科書" 第3章) and quantise KV before decoding
 * (第22章); E4M3 with per-tensor scales is the plainest such format with conversions in
 * hardware, and halves the bytes decode streams. */
typedef enum { PA_KV_SAME = 0, PA_KV_E4M3 = 1 } pa_kv_dtype;

/* Bits of the device status word (pa_get_device_status). */
#define PA_DEV_BAD_BLOCK_ID 0x1u  /* a block-table entry that had to be read was outside the pool */
#define PA_DEV_BAD_LENGTHS 0x2u   /* q_len < 1, ctx_len < 0, n_i > max_blocks_per_seq * B, or
                                     sum(q_lens) != total_q; that sequence's rows are not written */
#define PA_DEV_BAD_SLOT 0x4u      /* kv_append: slot_mapping entry >= num_blocks * B (skipped) */
#define PA_DEV_BAD_PAIR 0x8u      /* block_copy: a src or dst block id outside its pool (skipped) */
#define PA_DEV_TIMEOUT 0x10u      /* a bounded wait inside a kernel gave up (internal error) */

/* ------------------------------------------------------------------------------------------
 * pa_forward: generalized paged attention.
 *
 * For every sequence i, new token j < q_i and query head h, with P = c_i + j the token's
 * absolute position and kh = h / g its KV head:
 *     out[cu_i + j, h, :] = sum_{p <= P} softmax_p(scale * q[cu_i + j, h, :] . K_i[p, kh, :]) V_i[p, kh, :]
 * where K_i[p] lives in physical block block_tables[i][p / B] at slot p % B, and cu_i is the
 * exclusive prefix sum of q_lens.  This is softmax(QK^T / sqrt(d_k)) V in the blockwise form
 * A_j / o = sum_j A_j V_j of "SOSP 2023論文解説: PagedAttention" (section
 * "PagedAttentionアルゴリズム"), generalized to ragged multi-token queries with a fused causal
 * mask over cached-plus-new positions as in "Stateful Large Language Model Serving with
 * Pensieve" (section "汎化PagedAttentionカーネル"); prefill turns (q_i > 1) and decode steps
 * (q_i = 1) share one call.  GQA groups are contiguous ("KVキャッシュ管理の教科書" 第19章).
 * The new tokens' K/V must already be in the cache (kv_append first).
 *
 * Layouts (all device memory):
 *   q, out        [T, Hq, d], row-major, dtype `dims->dtype`.  `out` must not alias q or caches.
 *   k_cache, v_cache  element (block b, kv head kh, slot s, dim x) at
 *                 b * kv_block_stride + (kh * B + s) * d + x  (dtype `dims->dtype`).
 *                 Physical blocks may be shared by several sequences (prefix sharing).
 *   block_tables  int32 [num_seqs, max_blocks_per_seq]; entries past ceil(n_i / B) are never read.
 *   ctx_lens, q_lens  int32 [num_seqs].
 *   scale         the softmax scale, normally 1/sqrt(d).
 *   workspace     device scratch of at least pa_forward_workspace_size(dims) bytes, 256-byte
 *                 aligned; contents need no initialisation and are clobbered.
 * Supported: dtype f32 / bf16 / f16; d in {64, 128}; B in {16, 32, 64, 128}; Hq % Hkv == 0;
 * 16-byte aligned q, out and caches; kv_block_stride * element size a multiple of 16 bytes.
 * E4M3 caches (kv_dtype = PA_KV_E4M3): dtype bf16 or f16, d = 128, finite k_scale, v_scale > 0;
 * kv_block_stride counts codes (bytes).  Decode rows run on the CUDA-core kernels, which read the
 * codes.  A tcgen05 MMA takes both operands in one 16-bit type, so the blocks of the sequences
 * the tensor-core kernel takes (the rule below, with scale * k_scale > 0) are first widened,
 * exactly, into scratch blocks of the query dtype in the workspace past its required part; the K
 * scale joins the softmax scale and the V scale the output normalisation.  The scratch holds as
 * many blocks as the caller's workspace has room for (pa_forward_widen_bytes: enough for every
 * sequence the kernel may take); such sequences are admitted in sequence order while all of their
 * blocks fit, and the others run on the CUDA-core kernels, so any workspace of at least
 * pa_forward_workspace_size bytes is valid.  Their key ranges are cut into chunks (as below) only
 * when the workspace holds all of pa_forward_widen_bytes, whose last 16 MB hold the chunks.
 * Sequences with q_len * g >= 16 query rows per KV head run on the tcgen05 tensor-core kernel when
 * the dtype is bf16/f16, d = 128, g divides 128 and scale > 0 (one work item per KV head and pair
 * of 128-row query tiles; when a call has fewer such items than SMs, each item's key range is
 * cut into chunks run by separate CTAs and merged by the logsumexp rule of the split-KV merge, at
 * most 120 chunk items; the workspace of dims with total_q > num_seqs holds their 15.5 MiB of
 * partial rows); decode steps, short turns and
 * everything else run on the split-KV decode kernels: 2-4 query rows per KV head of bf16/f16
 * caches with d = 128 as mma.m16n8k16 tensor-core fragments (P rounded to the 16-bit type before
 * P V), one row per KV head, E4M3 caches, fp32 and d = 64 on CUDA cores.
 * Streams: when some sequence takes the tensor-core kernel, that kernel runs on `stream` right
 * after the planner, and the decode kernel runs on a library-owned high-priority stream of the
 * current device, forked from `stream` after the planner and joined back at the end of the call,
 * so that the decode work fills the SMs the tensor-core kernel's CTAs leave as they finish.  To the
 * caller the call stays ordered on `stream` (also under stream capture, as a fork/join); host
 * threads that call pa_forward at the same time serialise briefly on the fork/join enqueue, and
 * their decode kernels of such calls run one after another on that device's side stream.
 * ---------------------------------------------------------------------------------------- */
typedef struct {
    int32_t dtype;              /* pa_dtype of q, out, k_cache and v_cache */
    int32_t num_seqs;           /* >= 1 */
    int64_t total_q;            /* T: rows of q and out; must equal sum(q_lens) */
    int32_t num_q_heads;        /* Hq */
    int32_t num_kv_heads;       /* Hkv, divides Hq */
    int32_t head_dim;           /* d */
    int32_t block_size;         /* B */
    int64_t num_blocks;         /* physical blocks addressable through k_cache / v_cache */
    int32_t max_blocks_per_seq; /* row length of block_tables */
    int64_t kv_block_stride;    /* elements between physical blocks b and b+1; 0 = Hkv * B * d */
    int32_t kv_dtype;           /* pa_kv_dtype of k_cache and v_cache (0 = `dtype`) */
    float k_scale;              /* PA_KV_E4M3: value of a cached K element = code value * k_scale */
    float v_scale;              /* PA_KV_E4M3: the same for V */
} pa_dims;

size_t pa_forward_workspace_size(const pa_dims *dims);

/* Extra workspace, past pa_forward_workspace_size(dims), that lets every sequence the tensor-core
 * kernel may take of an E4M3 call (dims with total_q > num_seqs and a shape that kernel supports)
 * run on it: a candidate-block prefix ([num_seqs + 1] int32) and a block table ([num_seqs,
 * max_blocks_per_seq] int32), each padded to 256 bytes; widened K and V blocks for
 * min(num_seqs, total_q / ceil(16 / g)) * max_blocks_per_seq blocks; then the tensor-core
 * kernel's chunk counters and partial rows (3840 and 120 * 2 * 128 * 528 bytes).  0 for other
 * dims or invalid dims.  The bound is from the dims alone; a smaller extra (down to none) is valid:
 * it holds fewer widened blocks (the sequences that do not fit run on the CUDA-core kernels) and
 * no chunk regions. */
size_t pa_forward_widen_bytes(const pa_dims *dims);

pa_status pa_forward(const pa_dims *dims, const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_tables, const int32_t *ctx_lens, const int32_t *q_lens,
                     float scale, void *out, void *workspace, size_t workspace_bytes,
                     pa_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * pa_set_timing_events: time the attention kernels of later pa_forward calls with CUDA events.
 *
 * Not part of the method: a measurement hook, because the call's kernels run on two streams and
 * overlap, so events the caller records around the call cannot bracket one kernel.
 * Each later pa_forward / pa_forward_append / pa_forward_no_alloc call (on any thread, until the
 * next pa_set_timing_events) records
 *   tc_start, tc_stop  right before and after the tcgen05 kernel's launch, on the stream it runs
 *                      on (the caller's; only calls that launch it);
 *   cc_start, cc_stop  right before and after the launch of the decode kernel (tensor-core GQA
 *                      or CUDA-core split-KV; every call launches it, after the planner), on the
 *                      stream it runs on (the side stream when the call also launches the
 *                      tcgen05 kernel, else the caller's).
 * cudaEventElapsedTime(start, stop) is then that kernel's device time (plus launch gaps).
 * Arguments are cudaEvent_t handles created by the caller (timing enabled) on the device of the
 * later calls, owned by the caller; NULL for both of a pair records nothing.  Returns
 * PA_ERR_INVALID_ARG (and changes nothing) if only one of a pair is NULL.  A pair re-recorded by
 * a later call holds the later call's times.
 * ---------------------------------------------------------------------------------------- */
pa_status pa_set_timing_events(void *tc_start, void *tc_stop, void *cc_start, void *cc_stop);

/* ------------------------------------------------------------------------------------------
 * pa_forward_no_alloc: pa_forward without a caller-provided workspace.
 *
 * The pages have no counterpart for this call; it exists for callers that cannot allocate
 * device memory where they run attention -- for example a plug-in inside an engine whose own
 * allocator owns every byte of device memory, or a latency-critical loop that must not call
 * cudaMalloc / cudaFree (which can synchronise the whole device).  Same arguments, semantics and
 * results as pa_forward, minus `workspace` / `workspace_bytes`.
 *
 *  - Scratch: a library-owned device array of PA_NO_ALLOC_WORKSPACE_BYTES (32 MiB), held by every
 *    GPU that loads the library until the process exits.  The call allocates nothing (no
 *    cudaMalloc, cudaFree or allocating library routine).
 *  - Dims whose pa_forward_workspace_size exceeds PA_NO_ALLOC_WORKSPACE_BYTES are rejected with
 *    PA_ERR_WORKSPACE before any device work (use pa_forward with your own workspace instead).
 *  - E4M3 calls widen their tensor-core turns into the part of the array past
 *    pa_forward_workspace_size (see pa_forward): turns that do not fit there run on the CUDA-core
 *    kernels.
 *  - The first call on a device looks up the array's device address (cudaGetSymbolAddress, with
 *    that device current); make that first call before any stream capture.
 *  - Every call on a device shares the one array, which keeps the last call's contents (nothing
 *    in it needs to start at zero).  Calls whose work overlaps on the GPU -- on different streams,
 *    or from different host threads -- race on it and give undefined results: serialise them.
 * ---------------------------------------------------------------------------------------- */
#define PA_NO_ALLOC_WORKSPACE_BYTES (32u * 1024u * 1024u)

pa_status pa_forward_no_alloc(const pa_dims *dims, const void *q, const void *k_cache,
                              const void *v_cache, const int32_t *block_tables,
                              const int32_t *ctx_lens, const int32_t *q_lens, float scale,
                              void *out, pa_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * kv_append: write the new tokens' K/V into the paged cache.
 *
 * For every new token t with slot_mapping[t] >= 0, every layer l and KV head h:
 *   k_cache[l][slot / B][h][slot % B][:] = k_new[l][t][h][:]   (and the same for V)
 * A slot is physical_block * B + offset; the caller's allocator picks it so that a sequence fills
 * its partially filled last block before a fresh one ("SOSP 2023論文解説: PagedAttention",
 * section "ブロックテーブルによるメモリ管理").  slot < 0 marks padding and is skipped; a slot
 * >= num_blocks * B is skipped and flagged PA_DEV_BAD_SLOT.  Two tokens with the same slot in
 * one call give an unspecified one of the two.  The copy is bit-exact.
 *
 * E4M3 caches (kv_dtype = PA_KV_E4M3; k_new/v_new in bf16, f16 or f32): each new element is
 * widened to fp32, multiplied by the fp32 reciprocal 1/k_scale (1/v_scale), and rounded to the
 * nearest E4M3 value, ties to the even code, magnitudes beyond 448 saturating to +-448 (the sign
 * is kept, also when the result rounds to zero).  Non-finite inputs give unspecified codes.
 *
 * Layouts (device memory): k_new/v_new element (l, t, h, x) at l*new_layer_stride +
 * (t*Hkv + h)*d + x; caches element (l, b, h, s, x) at l*cache_layer_stride +
 * b*kv_block_stride + (h*B + s)*d + x (cache strides count codes for E4M3 caches);
 * slot_mapping int64 [num_tokens].  Rows must be 16-byte aligned (d * element size a multiple
 * of 16, for the new tokens and for the caches).
 * ---------------------------------------------------------------------------------------- */
typedef struct {
    int32_t dtype;              /* pa_dtype (only the element size matters) */
    int64_t num_tokens;         /* T_new */
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t block_size;
    int64_t num_blocks;
    int64_t kv_block_stride;    /* 0 = Hkv * B * d */
    int32_t num_layers;         /* >= 1 */
    int64_t new_layer_stride;   /* 0 = num_tokens * Hkv * d */
    int64_t cache_layer_stride; /* 0 = num_blocks * kv_block_stride */
    int32_t kv_dtype;           /* pa_kv_dtype of the caches (0 = `dtype`) */
    float k_scale;              /* PA_KV_E4M3: > 0; K is stored as code(k / k_scale) */
    float v_scale;              /* PA_KV_E4M3: > 0 */
} kv_append_dims;

pa_status kv_append(const kv_append_dims *dims, const void *k_new, const void *v_new,
                    const int64_t *slot_mapping, void *k_cache, void *v_cache,
                    pa_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * pa_forward_append: kv_append of the step's new tokens, then pa_forward, in one call.
 *
 * The decode or prefill step of "SOSP 2023論文解説: PagedAttention" (sections
 * "ブロックテーブルによるメモリ管理" and "PagedAttentionアルゴリズム"): the new tokens' K/V go
 * into their slots, then every new token attends over its sequence's cached-plus-new positions.
 * Same result as kv_append (one layer, num_tokens = dims->total_q) followed by pa_forward with
 * the same arguments, bit for bit.  For same-dtype caches the writes are done by extra blocks of
 * pa_forward's first launch (its planner), so the step costs no launch of its own; E4M3 caches
 * take a separate quantising kv_append launch first.
 *
 *   k_new, v_new  [T, Hkv, d] device arrays of dtype `dims->dtype` (T = dims->total_q: the new
 *                 tokens are the call's query tokens, in q's order), 16-byte aligned.
 *   slot_mapping  int64 [T] device array: the token's slot (physical block * B + offset); < 0
 *                 skips the token; >= num_blocks * B is skipped and flagged PA_DEV_BAD_SLOT.
 *   k_cache, v_cache  written (the slots) and then read (the attention); other arguments,
 *                 layouts, supported shapes and the stream behaviour as for pa_forward and
 *                 kv_append.  The caller's block tables and ctx_lens must already count the new
 *                 tokens' blocks, as for pa_forward.
 * Errors: every argument check of kv_append and pa_forward, before any device work.
 * ---------------------------------------------------------------------------------------- */
pa_status pa_forward_append(const pa_dims *dims, const void *q, const void *k_new, const void *v_new,
                            const int64_t *slot_mapping, void *k_cache, void *v_cache,
                            const int32_t *block_tables, const int32_t *ctx_lens, const int32_t *q_lens,
                            float scale, void *out, void *workspace, size_t workspace_bytes,
                            pa_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * block_copy: copy whole blocks, every plane, bit for bit.
 *
 * For every pair (s, t) = (pairs[2k], pairs[2k+1]) and every plane p < num_planes:
 *   dst[p*dst_plane_stride + t*dst_block_stride .. + block_bytes) =
 *   src[p*src_plane_stride + s*src_block_stride .. + block_bytes)
 * Copy-on-write of a shared block before it is written ("SOSP 2023論文解説: PagedAttention",
 * section "Copy-on-Writeによるメモリ共有") when src and dst are the same device pool; swap-in
 * (src a page-locked host pool) and swap-out (dst a page-locked host pool) of blocks between the
 * CPU and GPU tiers ("Stateful Large Language Model Serving with Pensieve", sections
 * "GPU-CPU 2層キャッシュ構造" and "パイプライン化されたswap-in").  A plane is e.g. one
 * (layer, K|V) slice of a pool.
 *
 * pairs is int64 [num_pairs, 2] in device memory.  All destination ids must be distinct and no
 * destination may also be a source in the same call (pairs then act simultaneously); a violated
 * precondition gives unspecified bytes in the affected blocks, nothing else.  Ids outside
 * [0, src_num_blocks) / [0, dst_num_blocks) are skipped and flagged PA_DEV_BAD_PAIR.
 * src and dst may be device memory or page-locked host memory.  block_bytes, strides and both
 * base pointers must be multiples of 16 bytes.  With num_planes > 1 the planes of each pool must
 * not overlap: either plane_stride >= num_blocks * block stride (planes one after another), or
 * block_bytes <= plane_stride and num_planes * plane_stride <= block stride (planes side by side
 * inside every block); any other plane stride (0 included) is refused with PA_ERR_INVALID_ARG.
 *
 * max_ctas bounds the copy's grid (256-thread CTAs, no shared memory).  0 takes the default, a
 * persistent grid of 8 CTAs per SM, for a copy that has the GPU to itself.  A small value (a few
 * dozen CTAs move a host-memory swap at the link's full rate) leaves the other SMs to kernels
 * that run beside the copy on another stream, such as a layer's attention during a layer-by-layer
 * swap-in.  Negative values are refused with PA_ERR_INVALID_ARG.
 * ---------------------------------------------------------------------------------------- */
typedef struct {
    int64_t block_bytes;        /* bytes of one block in one plane */
    int32_t num_planes;         /* >= 1 */
    int64_t src_plane_stride;   /* bytes */
    int64_t dst_plane_stride;   /* bytes */
    int64_t src_block_stride;   /* bytes between blocks; 0 = block_bytes */
    int64_t dst_block_stride;   /* bytes between blocks; 0 = block_bytes */
    int64_t src_num_blocks;
    int64_t dst_num_blocks;
    int64_t num_pairs;          /* 0 is a no-op */
    int32_t max_ctas;           /* 0 = 8 CTAs per SM; > 0 = at most this many CTAs */
} block_copy_dims;

pa_status block_copy(const block_copy_dims *dims, const void *src, void *dst,
                     const int64_t *pairs, pa_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * 2-bit paged KV cache with promoted 4-bit key channels ("KVキャッシュ管理の教科書", 第22章, on
 * Kitty; 第3章 names fewer bits per element as the third way to shrink the cache).
 *
 * What the chapter fixes: K and V at 2 bits per element; the key channels whose mean magnitude
 * along the token direction is in the top 12.5-25 % promoted to 4 bits; a dense tensor of every
 * channel's low 2 bits plus a sparse tensor of only the promoted channels' high 2 bits; one
 * quantisation group of 128 tokens, which is one page of the paged cache, quantised once per 128
 * decode steps.  Readings taken for what it leaves open:
 *   - asymmetric min/max quantisation: K per channel over the page's 128 tokens, V per token over
 *     the head's d channels; code(x) = round-half-even((x - min) / s) clamped to [0, L] with
 *     s = (max - min) / L, L = 3, or 15 on a promoted key channel; s = 0 codes every element 0;
 *     a cached element's value is code * s + min (promoted key code = low + 4 * high);
 *   - the decisions that produce integers are taken in float32: the subtraction, the division and
 *     the magnitude sum (|k| added over the page's tokens in token order) round to nearest;
 *   - the P promoted channels are those with the largest magnitude sums, ties going to the lower
 *     channel index; P = 16 (12.5 %) or 32 (25 %) of d = 128;
 *   - a sequence of n tokens has floor(n / 128) quantised pages; its last n % 128 tokens stay in a
 *     residual page of the query's dtype (an ordinary 128-token cache block, written by kv_append
 *     with block_size 128) until it fills and kv_quantize_pages turns it into a quantised page.
 *
 * Record of one (page, KV head): pa_kitty_record_bytes(128, P) = 10272 + 32 P bytes (10784 or
 * 11296; 2.76 bits per cached element at P = 32), little-endian, at these byte offsets:
 *   [0, 512)          K scale s_x, float32, channel x = 0..127
 *   [512, 1024)       K minimum, float32 per channel
 *   [1024, 1536)      V scale, float32 per token t = 0..127
 *   [1536, 2048)      V minimum, float32 per token
 *   [2048, 2080)      promoted channel ids, uint8, ascending in slots 0..P-1, later slots 0
 *   [2080, 6176)      K low 2 bits: token t, channel x at byte 2080 + 32 t + x / 4, bits 2 (x % 4)
 *   [6176, 6176+32P)  K high 2 bits of promoted slot k: byte 6176 + (P/4) t + k / 4, bits 2 (k % 4)
 *   [6176+32P, +4096) V codes: token t, channel x at byte 2048 (t / 64) + 16 x + (t % 64) / 4,
 *                     bits 2 (t % 4) (channel-major within each half page of 64 tokens)
 * The byte order is the library's own: K codes token-major (a 32-bit word holds 16 channels of
 * one key) and V codes channel-major per half page (a word holds 16 tokens of one channel), the
 * orders in which decode feeds them to the tensor cores.
 * A page pool is [num_pages, Hkv, record] (record-major, 16-byte aligned); residual pools are
 * [num_res_pages, Hkv, 128, 128] of `dtype`.
 * ---------------------------------------------------------------------------------------- */
#define PA_KITTY_PAGE_TOKENS 128

typedef struct {
    int32_t dtype;              /* PA_BF16 or PA_F16: q, out and the residual pages */
    int32_t num_seqs;           /* >= 1; q and out are [num_seqs, Hq, d] (decode: q_len = 1) */
    int32_t num_q_heads;        /* Hq */
    int32_t num_kv_heads;       /* Hkv, divides Hq */
    int32_t head_dim;           /* d = 128 */
    int32_t promoted;           /* P = 16 or 32 */
    int64_t num_pages;          /* records in the page pool (per KV head) */
    int64_t num_res_pages;      /* blocks in the residual pools */
    int32_t max_pages_per_seq;  /* row length of block_tables */
} pa_kitty_dims;

/* Bytes of one (page, KV head) record, or 0 for an unsupported (head_dim, promoted). */
size_t pa_kitty_record_bytes(int32_t head_dim, int32_t promoted);

/* kv_quantize_pages: for every pair (s, t) = (pairs[2k], pairs[2k+1]) and every KV head h,
 * quantise the 128 tokens of residual page s (res_k / res_v [s][h]) into record t of `pages`, by
 * the rules above (bit-exact: same bytes on every run).  pairs is int64 device memory; ids
 * outside [0, num_res_pages) / [0, num_pages) are skipped and flagged PA_DEV_BAD_PAIR.
 * Destinations must be distinct.  Non-finite inputs give unspecified records.  Of `dims` only
 * dtype, num_kv_heads, head_dim, promoted, num_pages and num_res_pages are read. */
pa_status kv_quantize_pages(const pa_kitty_dims *dims, const void *res_k, const void *res_v,
                            const int64_t *pairs, int64_t num_pairs, void *pages,
                            pa_stream_t stream);

size_t pa_kitty_workspace_size(const pa_kitty_dims *dims);

/* pa_forward_kitty: decode attention (q_len = 1 for every sequence) over quantised pages.
 * Sequence i has n_i = ctx_lens[i] + 1 tokens, the new token's K/V already written (into its
 * residual page, or quantised with it when it filled the page).  block_tables[i][p] for
 * p < floor(n_i / 128) is a record id in `pages`; when n_i % 128 > 0, block_tables[i][floor(n_i /
 * 128)] is a residual page id in res_k / res_v.  For query head h (KV head h / g):
 *     out[i, h, :] = sum_{p < n_i} softmax_p(scale * q[i, h, :] . K_i[p]) V_i[p]
 * with K_i[p], V_i[p] the dequantised values (or the residual page's values).  Arithmetic: per
 * page, the query times each channel's scale is rounded to a 16-bit integer grid whose largest
 * magnitude lies in [2^13, 2^14), and its products with the codes are summed exactly (int32); per
 * half page (64 tokens), P times the token's V scale is rounded to a 16-bit grid the same way and
 * its products with the V codes are summed exactly; the page's partial sums are scaled back to
 * fp32.  The residual page runs in fp32 on the 16-bit values.
 * Workspace: pa_kitty_workspace_size(dims) bytes, 256-byte aligned, contents clobbered.
 * q_lens[i] != 1, ctx_lens[i] < 0 or n_i > max_pages_per_seq * 128 -> that sequence's rows are
 * not written, PA_DEV_BAD_LENGTHS; a page or residual id outside its pool -> that page is
 * skipped, PA_DEV_BAD_BLOCK_ID.  num_seqs <= 4096. */
pa_status pa_forward_kitty(const pa_kitty_dims *dims, const void *q, const void *pages,
                           const void *res_k, const void *res_v, const int32_t *block_tables,
                           const int32_t *ctx_lens, const int32_t *q_lens, float scale, void *out,
                           void *workspace, size_t workspace_bytes, pa_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * pa_get_device_status: synchronise `stream`, return the current device's status bits
 * (PA_DEV_*) accumulated since the last call in *flags, and clear them.  Returns PA_ERR_DEVICE
 * when any bit was set, PA_ERR_CUDA when the synchronisation failed, else PA_OK.
 * ---------------------------------------------------------------------------------------- */
pa_status pa_get_device_status(uint32_t *flags, pa_stream_t stream);

/* A static, human-readable name for a status code. */
const char *pa_status_string(pa_status status);

/* Library build identification: "pagedkv <version> sm_103a". */
const char *pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
