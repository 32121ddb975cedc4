// Generalized paged attention for multi-token turns on the 5th-generation tensor cores (tcgen05).
//
// Method: softmax(QK^T / sqrt(d_k)) V over each sequence's cached-plus-new keys with a causal
// mask ("SOSP 2023論文解説: PagedAttention", section "PagedAttentionアルゴリズム";
// "Stateful Large Language Model Serving with Pensieve", section "汎化PagedAttentionカーネル":
// ragged multi-token queries against non-contiguous KV blocks, masking fused so no score matrix
// is written out).  Scores are computed tile by tile with an online softmax
// ("KVキャッシュ管理の教科書" 第6章, FlashAttention's tiling in on-chip memory).
//
// A work item is a pair of 128-row query tiles of one sequence and one KV head (rows are
// (token, head-in-GQA-group) pairs, so the g query heads sharing a KV head fill the tiles even for
// short turns).  Both tiles walk the same 128-key K/V tiles, which are loaded once per pair:
//   S_t = Q_t K^T   (tcgen05.mma, M=N=128, K=d=128, Q_t and K from shared memory)
//   P_t = exp2(S_t * scale * log2 e - m_t), causal mask on diagonal tiles only, 16-bit
//   O_t += P_t V    (tcgen05.mma, P_t from tensor memory (over S_t), V from shared memory)
// The tensor core receives the two tiles' groups interleaved -- PV_0(j), S_0(j+1), PV_1(j),
// S_1(j+1) -- so it works on one tile while the other tile's softmax runs.  Each tile's groups
// come from their own issuing thread, the two taking turns: an issuer's mbarrier checks queue
// behind the MMAs it has issued, so one issuer for both tiles left the tensor core idle at every
// check, while with two, one thread's checks overlap the other's MMAs.  A turn commits once.
// The running max is only moved (and O_t rescaled in tensor memory) when it grows by more than
// 2^8; the final O / l is exact anyway.  Tiles below the diagonal take the row max from the
// reduction form of the tensor-memory load.
// A lone tile (odd tile count per KV head) runs in slot 0 alone; slot 1 passes its turns.
//
// Warp roles (384 threads, one CTA per SM, persistent; items claimed from a global counter):
//   warp 0      TMA producer for Q (both tiles, once per item) and K: per 128-key tile one 3-D
//               box (64 columns x B rows of one (block, head)) per block and panel, 128-byte
//               swizzled, 3 stages; block-table entries of the next tile fetched ahead.
//   warp 1      MMA issuer of tile 0 (one lane) and tensor-memory owner.
//   warp 11     MMA issuer of tile 1 (one lane).  Each issuer zeroes the V rows past the last
//               key of an item's final tile that its PV reads (those slots may hold anything,
//               NaN included).
//   warp 2      TMA producer for V (2 stages).
//   warps 3-6   softmax of tile 0, warps 7-10 softmax of tile 1: one thread per row
//               (tensor-memory lane), S -> P per KV tile, epilogue O / l -> out; one warp per
//               tile also releases the K/V stages and Q tiles its tile's MMAs have finished with.
// Tensor memory (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,384), O_1 [384,512).
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
constexpr int kThreads = 384;
constexpr int kKWarp = 0, kMmaWarp = 1, kVWarp = 2, kSoftmax0 = 3, kMma1Warp = 11;
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns of S_u and O_u for query tile u of the pair
__host__ __device__ constexpr uint32_t tmem_s(int u) { return u ? 128u : 0u; }
__host__ __device__ constexpr uint32_t tmem_o(int u) { return u ? 384u : 256u; }
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows > 2^8

constexpr int kKStages = 3;   // K(j) is freed once both S(j) are done and needed one step later
constexpr int kVStages = 2;   // V(j) is freed once both PV(j) are done and needed two steps later

// shared-memory map (offsets from a 1024-byte aligned base)
constexpr int kSmQ = 0;                          // two Q tiles
constexpr int kSmK = kSmQ + 2 * kTile;
constexpr int kSmV = kSmK + kKStages * kTile;
constexpr int kSmBar = kSmV + kVStages * kTile;
constexpr int kSmBytes = kSmBar + 256 + 1024;   // + alignment slack

enum Bar {
    kKFull0 = 0, kKEmpty0 = kKFull0 + kKStages, kVFull0 = kKEmpty0 + kKStages,
    kVEmpty0 = kVFull0 + kVStages, kSFull0 = kVEmpty0 + kVStages, kPFull0 = kSFull0 + 2,
    kOReady0 = kPFull0 + 2, kQFull = kOReady0 + 2, kQEmpty, kDrain, kItemFull0, kItemEmpty0 = kItemFull0 + 2,
    kTurn0 = kItemEmpty0 + 2, kNumBars = kTurn0 + 2
};
// Items are claimed by the K producer and handed to the other eleven warps through a two-slot ring.
constexpr int kItemConsumers = 3 + 8;
static_assert(kNumBars * 8 + 4 + 8 <= 256, "barrier area");

// ---- tcgen05 / TMA wrappers -----------------------------------------------------------------

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

// D (tensor memory) (+)= A (shared-memory descriptor) * B (shared-memory descriptor).
__device__ __forceinline__ void umma_ss(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D (tensor memory) (+)= A (tensor memory) * B (shared-memory descriptor).
__device__ __forceinline__ void umma_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(b), "r"(idesc), "r"(accumulate)
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

// All 128 fp32 columns of this thread's tensor-memory lane in one load (+ wait).
__device__ __forceinline__ void tmem_load128(uint32_t taddr, uint32_t (&r)[128]) {
    asm volatile(
        "{\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t}"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
        : "r"(taddr)
        : "memory");
}

// All 128 fp32 columns of this thread's tensor-memory lane and their maximum, in one load (+ wait):
// the reduction form of tcgen05.ld (sm_103a) returns the lane's maximum over the loaded columns
// beside the values, so a row whose columns are all visible needs no max pass of its own.  NaN
// columns do not take part in the maximum (the IEEE maxNum rule of max.f32).
__device__ __forceinline__ void tmem_load128_max(uint32_t taddr, uint32_t (&r)[128], float &mx) {
    asm volatile(
        "{\n\t"
        "tcgen05.ld.red.sync.aligned.32x32b.x128.max.f32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, %128, [%129];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t}"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127]), "=f"(mx)
        : "r"(taddr)
        : "memory");
}

// 64 32-bit columns (128 packed 16-bit values) into this thread's tensor-memory lane (+ wait).
__device__ __forceinline__ void tmem_store64(uint32_t taddr, const uint32_t (&r)[64]) {
    asm volatile(
        "{\n\t"
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};\n\t"
        "tcgen05.wait::st.sync.aligned;\n\t}"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
        : "memory");
}

// Maximum of three floats in one instruction.
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
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
    float *part;                  // chunk partial rows: [item][tile][row][kTcPartFloats]
    uint32_t *arrive;             // chunks finished: [first item of the pair][tile][warp]
    unsigned *status;
    int64_t num_blocks;
    float scale_log2;
    float v_scale;                // 1, or the V scale of E4M3 caches (their widened codes)
    int num_seqs, q_heads, kv_heads, group, block_size, max_blocks;
};

// One work item: query tiles qt0 = 2*pi and qt1 = 2*pi + 1 (if it exists) of one (sequence,
// KV head), over one chunk of the pair's key range.  Tile 1 holds later rows, so its causal range
// (and KV tile count) covers tile 0's.  The item loads KV tiles k0 .. k0 + ntiles - 1 once, in
// order; slot u reads them from k0 up to its own last tile nt[u] - 1.  Without chunking (the
// launch has at least one pair per CTA) every pair is one chunk, k0 = 0.
struct Item {
    int seq, kvh, ntiles;         // ntiles: KV tiles loaded = MMA steps (the longer slot's count)
    int k0, nchunk, chunk, first; // first KV tile; chunks of the pair, this one; item of chunk 0
    int64_t tok0;
    bool two;                     // tile 1 exists
    int j0[2], rows_valid[2], nt[2];
    int64_t pmin[2], pmax[2];
};

// (KV head, pair, chunk, chunks of the pair) of item `local` of a sequence whose pairs run as
// chunks of about lc KV tiles.  Out of line: only launches with few pairs take it.
__device__ __noinline__ int4 chunk_walk(int64_t c, int rows, int g, int pph, int lc, int local) {
    int per = 0;                                  // items per KV head
    for (int q = 0; q < pph; ++q) per += tc_pair_chunks(tc_pair_tiles(c, rows, g, q), lc);
    const int kvh = local / per;
    int rem = local - kvh * per, pi = pph - 1, nchunk = 1;
    for (; pi > 0; --pi) {
        nchunk = tc_pair_chunks(tc_pair_tiles(c, rows, g, pi), lc);
        if (rem < nchunk) break;
        rem -= nchunk;
    }
    if (pi == 0) nchunk = tc_pair_chunks(tc_pair_tiles(c, rows, g, 0), lc);
    return make_int4(kvh, pi, rem, nchunk);
}

// Item `it` of the launch; lc = KV tiles per chunk (0: pairs are not chunked).  Items are numbered
// by sequence rank, then KV head, then pair (a sequence's last, longest pair first), then chunk,
// so the chunks of one pair are consecutive items.
__device__ __forceinline__ Item decode_item(const TcParams &p, int it, int lc) {
    Item t;
    const int rank = find_rank(p.tc_cu, p.num_seqs, it);
    t.seq = __ldg(p.tc_seq + rank);
    const int local = it - __ldg(p.tc_cu + rank);
    const int rows = __ldg(p.qlen + t.seq) * p.group;
    const int tph = (rows + kRows - 1) / kRows;   // query tiles per KV head
    const int pph = (tph + 1) / 2;                // tile pairs per KV head
    const int64_t c = __ldg(p.ctx + t.seq);
    int pi, chunk = 0, nchunk = 1;
    if (lc <= 0) {
        pi = pph - 1 - (local % pph);
        t.kvh = local / pph;
    } else {
        const int4 w = chunk_walk(c, rows, p.group, pph, lc, local);
        t.kvh = w.x;
        pi = w.y;
        chunk = w.z;
        nchunk = w.w;
    }
    t.tok0 = __ldg(p.cu_q + t.seq);
    t.two = 2 * pi + 1 < tph;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int qt = 2 * pi + (u == 1 && t.two ? 1 : 0);
        t.j0[u] = qt * (kRows / p.group);
        t.rows_valid[u] = min(kRows, rows - qt * kRows);
        t.pmin[u] = c + t.j0[u];
        t.pmax[u] = c + t.j0[u] + (t.rows_valid[u] - 1) / p.group;
        t.nt[u] = (int)((t.pmax[u] + kKeys) / kKeys);
    }
    // chunk `chunk` of nchunk: KV tiles [k0, k1) of the pair's whole range (at least 2 each)
    const int ntot = t.two ? t.nt[1] : t.nt[0];
    t.k0 = (int)((int64_t)chunk * ntot / nchunk);
    t.ntiles = (int)((int64_t)(chunk + 1) * ntot / nchunk) - t.k0;
    t.nchunk = nchunk;
    t.chunk = chunk;
    t.first = it - chunk;
    return t;
}

// Physical block of each lane's block in KV tile kt (lanes < blocks of the tile), clamped.
__device__ __forceinline__ int tile_block(const TcParams &p, const int32_t *bt_row, int64_t pmax,
                                          int kt, int bpt, int lane, int &nblk) {
    const int64_t key0 = (int64_t)kt * kKeys;
    const int64_t keys = min((int64_t)kKeys, pmax + 1 - key0);
    nblk = (int)((keys + p.block_size - 1) / p.block_size);
    int phys = 0;
    if (lane < nblk) {
        phys = __ldg(bt_row + (int64_t)kt * bpt + lane);
        if (phys < 0 || (int64_t)phys >= p.num_blocks) {
            report(p.status, PA_DEV_BAD_BLOCK_ID);
            phys = (int)p.num_blocks;   // outside the tensor map: the copy fills zeros
        }
    }
    return phys;
}

// Epilogue of a chunk item (a pair whose key range runs as several items).  The warp's 32 rows
// write (m, l, O) -- running max in log2 units, sum, unnormalised O from tensor memory, O 16-byte
// aligned in a 528-byte row -- to the item's partial slot; after a device-scope fence, the warp arrives on its (pair, tile, warp)
// counter, and the warp that arrives last merges the pair's chunks row by row by the logsumexp
// rule, out = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c, M = max_c m_c (every row sees key 0
// in the first chunk, so M is a real score; a chunk in which a row saw no key has l = 0, O = 0 and
// m = -3e38, weight 0), and writes the row (orow, if stored).
template <typename T>
__device__ __noinline__ void chunk_epilogue(const TcParams &p, int it, const Item &t, int u, int quad, int row,
                                            int lane, uint32_t o_tmem, float m, float l, float v_scale, T *orow) {
    float *mine = p.part + ((size_t)(it * 2 + u) * kRows + row) * kTcPartFloats;
    mine[0] = m;
    mine[1] = l;
#pragma unroll 1
    for (int c = 0; c < kDim / 32; ++c) {
        uint32_t r[32];
        tmem_load32(o_tmem + c * 32, r);
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
            reinterpret_cast<float4 *>(mine + kTcPartO + c * 32)[q4] =
                make_float4(__uint_as_float(r[4 * q4]), __uint_as_float(r[4 * q4 + 1]),
                            __uint_as_float(r[4 * q4 + 2]), __uint_as_float(r[4 * q4 + 3]));
    }
    __threadfence();
    __syncwarp();
    uint32_t before = 0;
    if (lane == 0) before = atomicAdd(p.arrive + ((size_t)t.first * 2 + u) * 4 + quad, 1u);
    before = __shfl_sync(0xffffffffu, before, 0);
    if (before != (uint32_t)(t.nchunk - 1)) return;
    __threadfence();
    auto slot = [&](int c) -> const float * {
        return p.part + ((size_t)((t.first + c) * 2 + u) * kRows + row) * kTcPartFloats;
    };
    float M = -INFINITY;
    for (int c = 0; c < t.nchunk; ++c) M = fmaxf(M, __ldcg(slot(c)));
    float L = 0.f;
    for (int c = 0; c < t.nchunk; ++c) {
        const float mc = __ldcg(slot(c));
        L += mc == -INFINITY ? 0.f : fast_exp2(mc - M) * __ldcg(slot(c) + 1);
    }
    const float inv = (1.f / L) * v_scale;
#pragma unroll 1
    for (int b = 0; b < kDim / 32; ++b) {
        float acc[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = 0.f;
        for (int c = 0; c < t.nchunk; ++c) {
            const float *sc = slot(c);
            const float mc = __ldcg(sc);
            if (mc == -INFINITY) continue;
            const float w = fast_exp2(mc - M) * inv;
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(sc + kTcPartO + b * 32) + q4);
                acc[4 * q4] = fmaf(w, v.x, acc[4 * q4]);
                acc[4 * q4 + 1] = fmaf(w, v.y, acc[4 * q4 + 1]);
                acc[4 * q4 + 2] = fmaf(w, v.z, acc[4 * q4 + 2]);
                acc[4 * q4 + 3] = fmaf(w, v.w, acc[4 * q4 + 3]);
            }
        }
        if (orow) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint4 v;
                v.x = pack2<T>(acc[q4 * 8 + 0], acc[q4 * 8 + 1]);
                v.y = pack2<T>(acc[q4 * 8 + 2], acc[q4 * 8 + 3]);
                v.z = pack2<T>(acc[q4 * 8 + 4], acc[q4 * 8 + 5]);
                v.w = pack2<T>(acc[q4 * 8 + 6], acc[q4 * 8 + 7]);
                *reinterpret_cast<uint4 *>(orow + b * 32 + q4 * 8) = v;
            }
        }
    }
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
    volatile int *item_ring = reinterpret_cast<volatile int *>(smem + kSmBar + kNumBars * 8 + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr bool kF16 = std::is_same<T, __half>::value;
    const uint32_t idesc_qk = instr_desc(false, kF16);
    const uint32_t idesc_pv = instr_desc(true, kF16);

    if (threadIdx.x == 0) {
        for (int b = 0; b < kNumBars; ++b) {
            uint32_t count = 1;
            if (b == kPFull0 || b == kPFull0 + 1) count = 4;
            if (b == kItemEmpty0 || b == kItemEmpty0 + 1) count = kItemConsumers;
            // released by both MMA issuers
            if ((b >= kKEmpty0 && b < kKEmpty0 + kKStages) || (b >= kVEmpty0 && b < kVEmpty0 + kVStages) ||
                b == kQEmpty || b == kDrain)
                count = 2;
            mbar_init(&bars[b], count);
        }
        mbar_fence_init();
    }
    if (warp == kMmaWarp) {
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
    const int lc = (int)p.counters[kTcChunk];
    uint32_t *next_item = const_cast<uint32_t *>(p.counters) + kTcNext;
    const int B = p.block_size;
    const int bpt = kKeys / B;   // blocks per KV tile
    // next item for every warp but the K producer: -1 = no more work, -2 = the wait timed out
    auto receive_item = [&](uint32_t n) -> int {
        const int slot = n & 1;
        if (!warp_wait(&bars[kItemFull0 + slot], (n >> 1) & 1)) return -2;
        const int it = item_ring[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kItemEmpty0 + slot]);
        return it;
    };

    if (warp == kKWarp || warp == kVWarp) {
        // ------------------------------------------------------------ TMA producers (Q+K or V)
        const bool is_k = warp == kKWarp;
        const CUtensorMap *map = is_k ? &kmap : &vmap;
        const int full0 = is_k ? kKFull0 : kVFull0, empty0 = is_k ? kKEmpty0 : kVEmpty0;
        const int nst = is_k ? kKStages : kVStages;
        unsigned char *stage0 = smem + (is_k ? kSmK : kSmV);
        uint32_t iter = 0, items = 0;
        uint32_t armed[3] = {0, 0, 0}, armed_q = 0;
        bool ok = true;
        for (uint32_t n = 0; ok; ++n) {
            int it;
            if (is_k) {
                const int slot = n & 1;
                if (n >= 2 && !warp_wait(&bars[kItemEmpty0 + slot], ((n >> 1) - 1) & 1)) { ok = false; break; }
                if (lane == 0) {
                    const uint32_t claimed = atomicAdd(next_item, 1u);
                    item_ring[slot] = claimed < (uint32_t)total ? (int)claimed : -1;
                    mbar_arrive(&bars[kItemFull0 + slot]);
                }
                __syncwarp();
                it = item_ring[slot];
            } else {
                it = receive_item(n);
                if (it == -2) { ok = false; break; }
            }
            if (it < 0) break;
            const Item t = decode_item(p, it, lc);
            if (is_k) {
                // both query tiles of the pair (the previous pair's S MMAs are done with Q)
                if (items > 0 && !warp_wait(&bars[kQEmpty], (items - 1) & 1)) { ok = false; break; }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bars[kQFull], (t.two ? 2 : 1) * kTile);
                    const int y = t.kvh * p.group;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        if (u == 1 && !t.two) break;
                        const int z = (int)(t.tok0 + t.j0[u]);
                        tma_load_3d(smem + kSmQ + u * kTile, &qmap, 0, y, z, &bars[kQFull]);
                        tma_load_3d(smem + kSmQ + u * kTile + kPanel, &qmap, 64, y, z, &bars[kQFull]);
                    }
                }
                ++armed_q;
            }
            ++items;
            const int64_t pmax = t.two ? t.pmax[1] : t.pmax[0];
            const int32_t *bt_row = p.bt + (int64_t)t.seq * p.max_blocks;
            int nblk_next = 0;
            int phys_next = tile_block(p, bt_row, pmax, t.k0, bpt, lane, nblk_next);
            for (int ld = 0; ld < t.ntiles; ++ld, ++iter) {
                const int phys = phys_next, nblk = nblk_next;
                if (ld + 1 < t.ntiles)
                    phys_next = tile_block(p, bt_row, pmax, t.k0 + ld + 1, bpt, lane, nblk_next);
                const int s = iter % nst;
                const uint32_t use = iter / nst;
                if (use > 0 && !warp_wait(&bars[empty0 + s], (use - 1) & 1)) { ok = false; break; }
                if (lane == 0) mbar_arrive_expect_tx(&bars[full0 + s], (uint32_t)nblk * B * 128 * 2);
                __syncwarp();
                if (lane < nblk) {
                    unsigned char *dst = stage0 + s * kTile + lane * B * 128;
                    tma_load_3d(dst, map, 0, t.kvh * B, phys, &bars[full0 + s]);
                    tma_load_3d(dst + kPanel, map, 64, t.kvh * B, phys, &bars[full0 + s]);
                }
                if (s == 0) ++armed[0];
                else if (s == 1) ++armed[1];
                else ++armed[2];
            }
        }
        if (!ok && lane == 0) report(p.status, PA_DEV_TIMEOUT);
        // every copy this warp issued lands before the CTA can exit
        for (int s = 0; s < nst; ++s)
            if (armed[s]) mbar_wait(&bars[full0 + s], (armed[s] - 1) & 1);
        if (armed_q) mbar_wait(&bars[kQFull], (armed_q - 1) & 1);
    } else if (warp == kMmaWarp || warp == kMma1Warp) {
        // ------------------------------------------------------------------ MMA issuers
        // One thread per query-tile slot u issues that slot's MMAs (lane 0 of warp 1: slot 0, lane 0
        // of warp 11: slot 1); the two streams share the tensor core.  A thread's mbarrier check is
        // ordered behind the MMAs it has issued but the tensor core has not yet accepted, so a lone
        // issuer leaves the pipe idle at every check; with two, one thread's checks overlap the
        // other's queued MMAs.  Per 128-key step a thread waits for everything its next two groups
        // need (V(j), K(j+1), P_u(j)) in a row, then issues PV_u(j) and S_u(j+1) back to back.
        // S_u(j+1) overwrites the columns PV_u(j) reads P from; both come from the same thread, in
        // that order, and the tensor core keeps that order.  A commit takes a slot in the tensor
        // core's queue, so a turn commits once, after S_u(j+1): its completion also means PV_u(j) is
        // done (a commit tracks every earlier MMA of its thread).  The slot's softmax warps, which
        // wait for that barrier anyway, release the K stage S_u(j+1) read, the V stage PV_u(j) read
        // and, after the slot's last S of an item, the Q tiles; the slot's last PV of an item
        // commits O-ready.  K and V stages are released once per slot (empty barriers of count 2):
        // for a load its slot does not read, the issuing thread arrives once the load has landed
        // (so no slot can arrive twice on one stage before the other has arrived once).
        const int u = warp == kMmaWarp ? 0 : 1;
        if (lane == 0) {
            uint32_t iter = 0, items = 0, pcount = 0;
            bool ok = true;
            const uint32_t q_base = smem_addr(smem + kSmQ), k_base = smem_addr(smem + kSmK),
                           v_base = smem_addr(smem + kSmV);
            auto wait_bar = [&](int b, uint32_t parity) -> bool {
                if (!mbar_wait(&bars[b], parity)) return false;
                tc_fence_after();
                return true;
            };
            auto wait_k = [&](uint32_t g) -> bool { return wait_bar(kKFull0 + g % kKStages, (g / kKStages) & 1); };
            auto wait_v = [&](uint32_t g) -> bool { return wait_bar(kVFull0 + g % kVStages, (g / kVStages) & 1); };
            // Descriptors are built once; a tile, stage or k-step moves only the start-address
            // field (address / 16, below 2^14 for any shared-memory address).
            const uint64_t dq = smem_desc(q_base, 16, 1024), dk = smem_desc(k_base, 16, 1024),
                           dv = smem_desc(v_base, kPanel, 1024);
            auto issue_s = [&](uint32_t g, int qs) {   // S_u = Q_qs K(g)^T
                const uint64_t a = dq + (uint64_t)(qs * (kTile >> 4)),
                               b = dk + (uint64_t)((g % kKStages) * (kTile >> 4));
                const uint32_t d = tmem + tmem_s(u);
#pragma unroll
                for (int k = 0; k < kDim / 16; ++k) {
                    const uint64_t off = (uint64_t)(((k >> 2) * kPanel + (k & 3) * 32) >> 4);
                    umma_ss(d, a + off, b + off, idesc_qk, k > 0);
                }
                umma_commit(&bars[kSFull0 + u]);
            };
            // O_u += P_u V(g) over the first `ksteps` 16-key steps (P is zero past them)
            auto issue_pv = [&](uint32_t g, bool first, int ksteps) {
                const uint64_t b = dv + (uint64_t)((g % kVStages) * (kTile >> 4));
                const uint32_t d = tmem + tmem_o(u), a = tmem + tmem_s(u);
                if (ksteps == kKeys / 16) {
#pragma unroll
                    for (int k = 0; k < kKeys / 16; ++k)
                        umma_ts(d, a + k * 8, b + (uint64_t)(k * 128), idesc_pv, (!first || k > 0) ? 1u : 0u);
                } else {
#pragma unroll 1
                    for (int k = 0; k < ksteps; ++k)
                        umma_ts(d, a + k * 8, b + (uint64_t)(k * 128), idesc_pv, (!first || k > 0) ? 1u : 0u);
                }
            };
            // The 16-key steps of V stage vs this slot reads when `valid` of its keys are visible, and
            // the zeroed V rows [first_stale, 16 * steps) under them (slots past the item's last key:
            // free or stale, possibly NaN; P = 0 times them must stay 0).  Both threads may zero the
            // same rows; both write zeros.
            auto v_steps = [&](int vs, int64_t valid, int64_t first_stale) -> int {
                if (valid >= kKeys) return kKeys / 16;
                const int ksteps = (int)((valid + 15) / 16);
                const int end = ksteps * 16;
                if (first_stale < end) {
                    unsigned char *vb = smem + kSmV + vs * kTile;
                    for (int r = (int)first_stale; r < end; ++r)
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            *reinterpret_cast<uint4 *>(vb + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
                            *reinterpret_cast<uint4 *>(vb + kPanel + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
                        }
                    fence_proxy_async_smem();
                }
                return ksteps;
            };
            // Turns alternate strictly, slot 0 first: a thread's k-th turn starts once the other
            // thread has ended its turn before it (turn barrier u is arrived by thread 1 - u).  The
            // arrive is ordered after the thread's MMAs, so the tensor core receives the groups in
            // turn order, as from one issuer: PV_0(j), S_0(j+1), PV_1(j), S_1(j+1).
            uint32_t turns = 0;
            auto take_turn = [&]() -> bool {
                if (u == 0 && turns == 0) return true;
                return wait_bar(kTurn0 + u, (u == 0 ? turns - 1 : turns) & 1);
            };
            auto end_turn = [&]() {
                mbar_arrive(&bars[kTurn0 + (1 - u)]);
                ++turns;
            };
            for (uint32_t n = 0; ok; ++n, ++items) {
                const int slot = n & 1;
                if (!mbar_wait(&bars[kItemFull0 + slot], (n >> 1) & 1)) { ok = false; break; }
                const int it = item_ring[slot];
                mbar_arrive(&bars[kItemEmpty0 + slot]);
                if (it < 0) break;
                const Item t = decode_item(p, it, lc);
                // KV tiles this slot walks in the item: from k0 to its own last tile
                const int cnt = (u == 0 || t.two) ? max(0, min(t.k0 + t.ntiles, t.nt[u]) - t.k0) : 0;
                const int nload = t.ntiles;
                // last key any row of this slot sees, and past which V rows of a load are stale
                const int64_t last_key = t.pmax[u];
                const int64_t item_last = t.two ? t.pmax[1] : t.pmax[0];
                // Releases of the loads this slot does not read: wait for the K (or V) tile to land,
                // then arrive on its empty barrier.  K and V have their own cursors: the K tile of a
                // load is released by the step in which some slot's S reads it, the V tile by the
                // step in which some slot's PV reads it (a V tile released with its K tile would wait
                // for a PV of the other slot that comes after this thread's turn).
                int relk = 0, relv = 0;
                auto mine = [&](int L) -> bool { return L < cnt; };   // a slot reads loads 0 .. cnt - 1
                auto release_others = [&](int kupto, int vupto) -> bool {
                    for (; relk < kupto; ++relk) {
                        if (mine(relk)) continue;
                        const uint32_t g = iter + (uint32_t)relk;
                        if (!wait_k(g)) return false;
                        mbar_arrive(&bars[kKEmpty0 + g % kKStages]);
                    }
                    for (; relv < vupto; ++relv) {
                        if (mine(relv)) continue;
                        const uint32_t g = iter + (uint32_t)relv;
                        if (!wait_v(g)) return false;
                        mbar_arrive(&bars[kVEmpty0 + g % kVStages]);
                    }
                    return true;
                };
                // The item's groups in turns: the initial S, then per step PV(i) + S(i + 1); both
                // threads take 1 + nsteps turns (nsteps = the longer slot's tile count), passing a
                // turn when their slot has nothing in it.
                const int nsteps = t.ntiles;
                // Loads of the other slot are released step by step, up to the loads any slot reads
                // in the step: a thread that held them back would keep the producers from refilling
                // the stages the other thread waits for.  Exclusive bounds; step -1 is the first S.
                auto kbound = [&](int i) -> int { return min(i + 2, nload); };   // K of S(i + 1)
                auto vbound = [&](int i) -> int { return min(i + 1, nload); };   // V of PV(i)
                if (!wait_bar(kQFull, items & 1)) { ok = false; break; }
                if (!release_others(kbound(-1), vbound(-1))) { ok = false; break; }
                if (cnt > 0 && !wait_k(iter)) { ok = false; break; }
                if (!take_turn()) { ok = false; break; }
                if (cnt > 0) issue_s(iter, u);
                end_turn();
                for (int i = 0; i < nsteps && ok; ++i) {
                    const bool has = i < cnt, more = i + 1 < cnt;
                    const uint32_t g = iter + (uint32_t)(has ? i : 0);
                    const uint32_t gn = more ? iter + (uint32_t)(i + 1) : 0u;
                    // everything PV_u(i) and S_u(i+1) need, checked before the turn
                    if (!release_others(kbound(i), vbound(i))) { ok = false; break; }
                    if (has) {
                        if (!wait_v(g)) { ok = false; break; }
                        if (more && !wait_k(gn)) { ok = false; break; }
                        if (!wait_bar(kPFull0 + u, pcount & 1)) { ok = false; break; }
                        ++pcount;
                    }
                    if (!take_turn()) { ok = false; break; }
                    if (has) {
                        const int vs = g % kVStages;
                        const int64_t key0 = (int64_t)(t.k0 + i) * kKeys;
                        const int ksteps = v_steps(vs, last_key + 1 - key0, item_last + 1 - key0);
                        issue_pv(g, i == 0, ksteps);
                        if (more) issue_s(gn, u);
                        else umma_commit(&bars[kOReady0 + u]);   // the slot's last PV of the item
                    }
                    end_turn();
                }
                if (!ok) break;
                if (!release_others(nload, nload)) { ok = false; break; }
                if (cnt == 0) mbar_arrive(&bars[kQEmpty]);
                iter += nload;
            }
            if (!ok) report(p.status, PA_DEV_TIMEOUT);
            // no tensor-core work of this CTA may be in flight when its tensor memory is freed
            umma_commit(&bars[kDrain]);
            mbar_wait(&bars[kDrain], 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ softmax warps
        const int u = (warp - kSoftmax0) >> 2;          // query tile of the pair this warp serves
        const int quad = warp & 3;                      // tensor-memory lanes this warp may access
        const int row = quad * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        const uint32_t s_tmem = lane_base + tmem_s(u), o_tmem = lane_base + tmem_o(u);
        const float c_log2 = p.scale_log2;            // > 0 (other scales use CUDA cores)
        uint32_t scount = 0;                           // S / PV tiles of this query tile so far
        uint32_t ocount = 0;                           // items of this slot so far (O-ready phases)
        uint32_t iter = 0;                             // K/V loads of the items so far
        // one thread per slot releases the K/V stages and the Q tiles the slot's MMAs have read
        const bool releaser = warp == kSoftmax0 + 4 * u && lane == 0;
        bool ok = true;
        for (uint32_t n = 0; ok; ++n) {
            const int it = receive_item(n);
            if (it == -2) { ok = false; break; }
            if (it < 0) break;
            const Item t = decode_item(p, it, lc);
            const uint32_t item_iter = iter;
            iter += t.ntiles;
            if (u == 1 && !t.two) continue;
            const int64_t pmin = t.pmin[u], pmax = t.pmax[u];
            const int kt_end = min(t.k0 + t.ntiles, t.nt[u]);   // this slot's tiles: k0 .. kt_end - 1
            const int j = t.j0[u] + row / p.group, hh = row % p.group;
            int64_t prow = pmin + row / p.group;
            if (prow > pmax) prow = pmax;               // padding rows: finite, never stored
            // a finite start: in a chunk, a row may see no key in its first tiles (all scores
            // -inf), and -inf - m must stay -inf (P = 0), not NaN
            float m = -3.0e38f, l = 0.f;
            for (int kt = t.k0; kt < kt_end; ++kt, ++scount) {
                if (!warp_wait(&bars[kSFull0 + u], scount & 1)) { ok = false; break; }
                tc_fence_after();
                if (releaser) {
                    // S_u(s) is complete, and with it PV_u(s - 1): their K and V stages are free
                    const uint32_t ld = item_iter + (uint32_t)(kt - t.k0);   // the item's load of tile kt
                    mbar_arrive(&bars[kKEmpty0 + ld % kKStages]);
                    if (kt > t.k0) mbar_arrive(&bars[kVEmpty0 + (ld - 1) % kVStages]);
                    if (kt + 1 == kt_end) mbar_arrive(&bars[kQEmpty]);   // the slot's last S
                }
                uint32_t raw[kKeys];
                float *x = reinterpret_cast<float *>(raw);   // raw scores q.k (unscaled)
                const int64_t key0 = (int64_t)kt * kKeys;
                const bool diag = key0 + kKeys - 1 > pmin;   // tile crosses some row's diagonal (warp-uniform)
                const int64_t lim = prow - key0;             // visible columns: 0 .. lim
                float mraw;                                  // row max of the raw scores (scale > 0 keeps the order)
                if (!diag) {
                    // every column is a visible key: the load returns the row max with the scores
                    tmem_load128_max(s_tmem, raw, mraw);
                } else {
                    tmem_load128(s_tmem, raw);
                    // masked scores become -inf, so their exp2 below is exactly 0 (scale > 0 here); the
                    // columns past the last key may hold anything, so the max is taken after the mask
#pragma unroll
                    for (int i = 0; i < kKeys; ++i)
                        if (i > lim) x[i] = -INFINITY;
                    float mx[8];                             // 8 chains of 3-input max
#pragma unroll
                    for (int k = 0; k < 8; ++k) mx[k] = x[k];
#pragma unroll
                    for (int i = 8; i + 16 <= kKeys; i += 16)       // columns 8 .. 119
#pragma unroll
                        for (int k = 0; k < 8; ++k) mx[k] = max3(mx[k], x[i + k], x[i + 8 + k]);
#pragma unroll
                    for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], x[kKeys - 8 + k]);   // 120 .. 127
                    mraw = max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
                }
                const float mt = (mraw == -INFINITY) ? -INFINITY : mraw * c_log2;
                const float mnew = fmaxf(m, mt);
                const bool rescale = mnew > m + kRescaleThreshold;
                const float muse = rescale ? mnew : m;
                // P = exp2(scale*log2e*s - m), packed to 16 bits; the argument and the partial row
                // sums (4 chains) use the packed two-lane fp32 instructions
                uint32_t pk[kKeys / 2];
                const uint64_t c2 = f2pack(c_log2, c_log2), nm2 = f2pack(-muse, -muse);
                uint64_t ls[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) ls[k] = 0ull;
#pragma unroll
                for (int i = 0; i < kKeys / 2; ++i) {
                    float y0, y1;
                    f2unpack(fma2(f2pack(x[2 * i], x[2 * i + 1]), c2, nm2), y0, y1);
                    const float e0 = fast_exp2(y0), e1 = fast_exp2(y1);
                    ls[i & 3] = add2(ls[i & 3], f2pack(e0, e1));
                    pk[i] = pack2<T>(e0, e1);
                }
                float lsum = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float a0, a1;
                    f2unpack(ls[k], a0, a1);
                    lsum += a0 + a1;
                }
                // tensor-memory loads/stores are warp-collective: the whole warp rescales when any
                // of its rows with a key seen so far (l > 0) must, after the previous PV is complete
                // (alpha = 1 for rows that need not; a row with l = 0 has O = 0, and its alpha is
                // 2^-inf = 0)
                if (__any_sync(0xffffffffu, rescale && l > 0.f)) {
                    // PV_u(s - 1) is complete: it came before S_u(s) from the same issuer
                    const float alpha = rescale ? fast_exp2(m - muse) : 1.f;
                    l *= alpha;
#pragma unroll 1
                    for (int c = 0; c < kDim / 32; ++c) {
                        uint32_t r[32];
                        tmem_load32(o_tmem + c * 32, r);
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        tmem_store32(o_tmem + c * 32, r);
                    }
                }
                m = muse;
                l += lsum;
                // P over the first 64 columns of the S buffer it came from
                tmem_store64(s_tmem, pk);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kPFull0 + u]);
            }
            if (!ok) break;
            // epilogue: O / l -> out, after this tile's last PV
            if (!warp_wait(&bars[kOReady0 + u], ocount & 1)) { ok = false; break; }
            ++ocount;
            tc_fence_after();
            if (releaser) mbar_arrive(&bars[kVEmpty0 + (item_iter + (uint32_t)(kt_end - 1 - t.k0)) % kVStages]);
            const bool store = row < t.rows_valid[u];
            T *orow = reinterpret_cast<T *>(p.out) +
                      ((t.tok0 + j) * p.q_heads + (int64_t)t.kvh * p.group + hh) * kDim;
            if (t.nchunk > 1) {
                // one chunk of the pair's key range: this row's (m, l, O) to the item's partial
                // slot; the last of the pair's chunks to finish (per warp of rows) merges them
                chunk_epilogue<T>(p, it, t, u, quad, row, lane, o_tmem, m, l, p.v_scale, store ? orow : nullptr);
                tc_fence_before();
                continue;
            }
            const float inv = (1.f / l) * p.v_scale;
#pragma unroll 1
            for (int c = 0; c < kDim / 32; ++c) {
                uint32_t r[32];
                tmem_load32(o_tmem + c * 32, r);
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
        }
        if (!ok && lane == 0) report(p.status, PA_DEV_TIMEOUT);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

}  // namespace

bool tc_shape_supported(const pa_dims &d) {
    if (d.dtype != PA_BF16 && d.dtype != PA_F16) return false;
    if (d.head_dim != kDim) return false;
    const int g = d.num_q_heads / d.num_kv_heads;
    if (g < 1 || g > kRows || (kRows % g) != 0) return false;
    if (d.block_size < 16 || d.block_size > kKeys) return false;
    if (d.num_blocks >= (int64_t(1) << 31) - 1 || d.total_q >= (int64_t(1) << 31)) return false;
    return tensor_maps_available();
}

cudaError_t launch_tc(const FwdArgs &a, cudaStream_t s) {
    const pa_dims &d = a.dims;
    const int g = d.num_q_heads / d.num_kv_heads;
    const uint64_t es = 2;
    // E4M3 caches: the widened scratch blocks (dense, `wid_cap` of them) and their block table
    const bool wide = a.wid_cap > 0;
    const int64_t dense = (int64_t)d.num_kv_heads * d.block_size * d.head_dim;
    const int64_t bstride = wide ? dense : (d.kv_block_stride ? d.kv_block_stride : dense);
    const int64_t nblocks = wide ? a.wid_cap : d.num_blocks;
    const void *kbase = wide ? a.wid_k : a.k, *vbase = wide ? a.wid_v : a.v;
    CUtensorMap qmap, kmap, vmap;
    if (!make_map_3d(&qmap, d.dtype, a.q, kDim, d.num_q_heads, d.total_q, kDim * es,
                     (uint64_t)d.num_q_heads * kDim * es, 64, g, kRows / g) ||
        !make_map_3d(&kmap, d.dtype, kbase, kDim, (uint64_t)d.num_kv_heads * d.block_size, nblocks,
                     kDim * es, bstride * es, 64, d.block_size, 1) ||
        !make_map_3d(&vmap, d.dtype, vbase, kDim, (uint64_t)d.num_kv_heads * d.block_size, nblocks,
                     kDim * es, bstride * es, 64, d.block_size, 1))
        return cudaErrorInvalidValue;
    TcParams p;
    const WsLayout &L = a.lay;
    p.out = static_cast<char *>(a.out);
    p.bt = wide ? a.wid_bt : a.bt;
    p.ctx = a.ctx;
    p.qlen = a.qlen;
    p.cu_q = reinterpret_cast<const int32_t *>(a.ws + L.cu_q);
    p.tc_cu = reinterpret_cast<const int32_t *>(a.ws + L.tc_cu);
    p.tc_seq = reinterpret_cast<const int32_t *>(a.ws + L.tc_seq);
    p.counters = reinterpret_cast<const uint32_t *>(a.ws + L.counters);
    p.part = L.tc_chunks ? reinterpret_cast<float *>(a.ws + L.tc_part) : nullptr;
    p.arrive = L.tc_chunks ? reinterpret_cast<uint32_t *>(a.ws + L.tc_arrive) : nullptr;
    p.status = a.status;
    p.num_blocks = nblocks;
    p.scale_log2 = a.scale * 1.4426950408889634f * (wide ? d.k_scale : 1.f);
    p.v_scale = wide ? d.v_scale : 1.f;
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
