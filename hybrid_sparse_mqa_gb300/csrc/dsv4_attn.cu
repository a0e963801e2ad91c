// dsv4_attn.cu - hybrid sparse MQA attention step (DeepSeek-V4 decode and
// target-verify) for GB300, sm_103a.
//
// What is computed is stated in include/dsv4attn.h.  How:
//
// * A CTA owns one query token, one group of up to 64 of its heads and one
//   slice of its key list.  The key list (window slots, then C4 / C128 extra
//   slots) is cut into Sc x Sg slices: the Sc slices of a token share a
//   thread-block cluster and merge their partial results inside the kernel
//   (through L2); Sg groups of clusters merge through the workspace and the
//   combine kernel.  With H = 128 the two head groups of a slice read the
//   same rows.
// * Per 48-key tile: eight loader warps resolve key slots to pool rows (SWA
//   page table, C4 index list, C128 range) one 192-slot chunk ahead of use and
//   gather the 1 KB rows with 16-byte cp.async into a 128-byte-swizzled shared
//   tile (packed FP8 rows: two of the warps bulk-copy the 608-byte rows two
//   tiles ahead into the top of the stage, six dequantise them in place).
//   Four MMA issuer warps each compute one quarter of S = Q K^T on tcgen05
//   (128 of the 512 dims, M = 64 heads, N = 48 keys) into its own fp32 TMEM
//   accumulator, and one 128-dim block of O^T += V^T P^T (M = 128 value dims,
//   N = 64 heads, K = 48 keys) into 4 x 64 TMEM columns; V is the same shared
//   tile read MN-major (K and V are the same row).  Each tcgen05.mma costs its
//   issuing thread about as long as a small MMA takes to run, so the products
//   are issued from four warps and overlap.  Four softmax warps read the four
//   score quarters with the 16-lane TMEM access shape and add them: the two
//   threads t and t ^ 2 hold the even and odd key columns of one head, so the
//   online softmax (lazily updated running max, fp32 denominator) needs one
//   shuffle per reduction; the bf16 probabilities go into the head's 128-byte
//   line.
// * At the end the sink adds exp(sink - M) to each head's denominator, the
//   slices are merged with log-sum-exp weights and the bf16 output written.
//
// Sources (page title, section): "SGLang DeepSeek-V4 Attention Test
// Capability Matrix" - "Input And Config Coverage", "Reference Implementation
// Notes"; "DeepSeek-V4 Attention: Query, Cache Write and History Addressing"
// - sections 1, 3, 4, 5; "DeepSeek-V4 and SGLang Day-0" - "What V4 changed".
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "dsv4attn.h"
#include "dsv4_device.cuh"
#include "dsv4_internal.h"

namespace dsv4 {

// ------------------------------------------------------------------ shape
constexpr int kDim = 512;
constexpr int kPageSize = 256;
constexpr int kTileN = 48;           // keys per tile
constexpr int kStages = 3;           // gather pipeline depth (48 KB each)
constexpr int kHG = 64;              // heads per CTA (MMA M of S = Q K^T)
constexpr int kRingHalf = 192;       // key slots resolved per chunk (four tiles; two chunks held)
constexpr int kPtCache = 4096;       // extra page-table entries kept for the first chunk (the P area)
constexpr int kRing = 2 * kRingHalf;
constexpr int kSoftmaxWarps = 4;
constexpr int kLoadWarps = 8;
constexpr int kLoadThreads = kLoadWarps * 32;
constexpr int kMmaWarp0 = kSoftmaxWarps + kLoadWarps; // four MMA issuer warps: warp kMmaWarp0 + q issues
                                                      // S over dims 128 q .. 128 q + 127 and O^T for
                                                      // value dims 128 q .. (warp kMmaWarp0 owns TMEM)
constexpr int kMmaWarps = 4;
constexpr int kQkWarp = kMmaWarp0;                    // the TMEM owner / dealloc warp
constexpr int kWarps = kMmaWarp0 + kMmaWarps;
constexpr int kThreads = kWarps * 32;
// packed FP8: loader warps 0..5 dequantise (8 key rows each), 6 and 7 issue the row copies
constexpr int kFp8DqWarps = 6;
constexpr int kFp8DqThreads = kFp8DqWarps * 32;
static_assert(kWarps == 16, "one O^T read-out job (TMEM quadrant, value tile) per warp");
constexpr int kMaxCluster = 8;
constexpr float kRescaleLog2 = 8.0f; // lazy rescale threshold (factor 256)
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;       // scores, one partial sum per dim quarter q at column 48 q
constexpr uint32_t kTmemO = 256;     // O^T: 4 x 64 columns, value dim 128*m + lane
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// packed FP8 row: [448 e4m3 nope][64 bf16 rope][7 fp32 scales][pad], 608 bytes
constexpr int kFp8NopeBytes = 448;
constexpr int kFp8ScaleOff = 448 + 128;
constexpr int kFp8RowBytes = 608;

// ------------------------------------------------------------------ smem
constexpr int kChunkQ = kHG * 128;             // 64 head rows x 128 B: one 64-dim chunk of Q
constexpr int kChunkKV = kTileN * 128;         // 48 key rows x 128 B: one 64-dim chunk of a stage
constexpr int kQBytes = 8 * kChunkQ;           // 64 heads x 512 dims
constexpr int kStageBytes = 8 * kChunkKV;      // 48 keys x 512 dims
constexpr int kPBytes = kHG * 128;             // 64 heads x 128-byte lines (48 keys bf16 used)
constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + kQBytes;
constexpr int OFF_P = OFF_KV + kStages * kStageBytes;
constexpr int OFF_RING = OFF_P + 2 * kPBytes;  // int32 pool rows of resolved slots
constexpr int OFF_ML = OFF_RING + kRing * 4;   // float2 (m, l) per head
constexpr int OFF_W = OFF_ML + kHG * 8;        // float per head: rescale factors
constexpr int OFF_MASK = OFF_W + kHG * 4;      // 64-bit key validity mask per stage
constexpr int OFF_BAR = OFF_MASK + kStages * 8;
enum Bar {
    B_Q_FULL = 0,
    B_KV_FULL = 1,
    B_KV_EMPTY = B_KV_FULL + kStages,
    B_MASK_FULL = B_KV_EMPTY + kStages,
    B_RAW_FULL = B_MASK_FULL + kStages,        // packed FP8: a tile's raw rows landed
    B_S_FULL = B_RAW_FULL + kStages,
    B_S_FREE = B_S_FULL + 1,
    B_P_FULL = B_S_FREE + 1,
    B_P_FREE = B_P_FULL + 2,
    B_O_FINAL = B_P_FREE + 2,
    B_MERGE,                                   // peers' partials staged by bulk copy
    B_COUNT
};
constexpr int OFF_MISC = OFF_BAR + B_COUNT * 8;
constexpr int OFF_MERGE = OFF_KV;              // [owned dim][64 heads] fp32, reuses the KV stages,
                                               // followed by the outgoing bf16 rows of the other dims;
                                               // peers' bf16 blocks and every slice's (m, l) are
                                               // staged in the Q area, the merge weights in the P area
constexpr int kSmemUsed = OFF_MISC + 16;
constexpr int kSmemAlloc = kSmemUsed;          // the dynamic shared base is checked to be 1024-aligned
// merge workspace per (token, grid split, head group): [Sc][512 dims][64 heads]
// bf16 partial accumulators, then [Sc][64 heads] float2 (m, l)
constexpr size_t kMergeRowsElems = (size_t)kDim * kHG;
static_assert(kDim * kHG * 4 + 0 <= kStages * kStageBytes, "owned fp32 rows + outgoing bf16 rows fit in the KV stages");
static_assert(kSmemAlloc <= 232448, "shared memory budget");
static_assert(kRingHalf <= kLoadThreads, "one slot per loader thread per chunk");
static_assert(kRingHalf % kTileN == 0 && kRingHalf / kTileN == 4, "four tiles per ring chunk");
static_assert(6 * 80 * 128 + 7 * 512 <= kQBytes, "staged peer blocks and (m, l) (Sc = 7) must fit in the Q area");
static_assert(7 * 64 * 128 + 8 * 512 <= kQBytes, "staged peer blocks and (m, l) (Sc = 8) must fit in the Q area");
static_assert(kMaxCluster * kHG * 4 <= 2 * kPBytes, "merge weights must fit in the P area");
static_assert(kHG * 4 <= kRing * 4, "single-slice merge weights must fit in the ring");
static_assert(kPtCache * 4 <= 2 * kPBytes, "first-chunk page-table entries fit in the P area");
static_assert(kTileN % 16 == 0 && kTileN <= 64, "tile keys: whole K16 steps, one 64-bit mask");

__device__ unsigned int g_dev_error;

// Optional per-CTA phase timestamps (globaltimer ns), compiled in only with
// -DDSV4_TRACE; read back with dsv4_attn_trace_read().
#ifdef DSV4_TRACE
constexpr int kTraceSlots = 64;
constexpr int kTraceCtas = 2048;
__device__ unsigned long long g_trace[kTraceCtas * kTraceSlots];
// slots hold clock64() (SM cycles); slot 62 / 63 hold globaltimer at the first
// and last mark of slot 0 / 57 so cycles can be converted to time per CTA
__device__ __forceinline__ void trace_mark(int slot) {
    const int cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    if (cta < kTraceCtas && slot < kTraceSlots) {
        g_trace[cta * kTraceSlots + slot] = static_cast<unsigned long long>(clock64());
        if (slot == 0) g_trace[cta * kTraceSlots + 62] = globaltimer_ns();
        if (slot == 57) g_trace[cta * kTraceSlots + 63] = globaltimer_ns();
    }
}
#define DSV4_TR(slot) trace_mark(slot)
#else
#define DSV4_TR(slot) ((void)0)
#endif

struct Params {
    const __nv_bfloat16* q;
    int T, H, batch;
    int groups;              // head groups of 64 (1 or 2)
    const int* seq_lens;
    const int* cu_seqlens;   // nullable (decode)
    const int* rpi;          // nullable
    const uint8_t* swa_rows;
    long long swa_pages;
    int swa_row_bytes;
    const int* swa_pt;
    int swa_pt_rows, swa_pt_stride;
    int window, ratio;
    const uint8_t* ex_rows;
    long long ex_pages;
    int ex_row_bytes;
    const int* ex_pt;
    int ex_pt_rows, ex_pt_stride;
    const int* topk_idx;
    int topk;
    const float* sink;
    float scale_log2;        // scale * log2(e)
    int cw, ce;              // window / extra slots per slice
    int csplits, gsplits;
    __nv_bfloat16* out;
    float* lse;
    float* part_o;           // [T, Sg, H, 512] fp32 when gsplits > 1
    float2* part_ml;         // [T, Sg, H]
    uint16_t* merge;         // [T, Sg, G, Sc, 512, 64] bf16 when csplits > 1
    int* debug_rows;
    int debug_stride;
};

// A token's key list is its window slots 0 .. n_swa-1 (positions pos-n_swa+1
// .. pos) followed by its extra slots 0 .. n_extra-1 (C4 indices or C128
// compressed-row numbers).  Slice `split` of S takes window slots
// [w0, w0 + nw) and extra slots [e0, e0 + ne), as equal shares of each part;
// within the slice its extra slots come first (virtual slots 0 .. ne-1), so
// the first tiles need only the index list and the extra page table, and the
// window slots (which need the position first) come last.
struct TokenInfo {
    int trow, pos, n_swa, n_c, n_extra, e0, ne, w0, nw, ntiles;
};

__device__ __forceinline__ bool wait_spin(uint32_t bar, uint32_t parity, int* abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
            if (globaltimer_ns() - t0 > kTimeoutNs) {
                atomicOr(&g_dev_error, DSV4_DEV_ERR_TIMEOUT);
                *reinterpret_cast<volatile int*>(abort_flag) = 1;
                return false;
            }
        }
    }
}
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, int* abort_flag) {
    return wait_spin(bar, parity, abort_flag);
}
// Bounded wait on an mbarrier phase.  On time-out it records the error, marks
// the CTA aborted and returns; callers carry on (and keep arriving on the
// barriers others wait for), so every role reaches the end of the kernel.
// The spin is one shared out-of-line function (less code to fetch) or, where
// the caller keeps many values live across the wait and a call would make it
// save them, inlined.
template <bool kOutOfLine>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, int* abort_flag) {
    if (mbar_try(bar, parity)) return true;
    if constexpr (kOutOfLine) return wait_slow(bar, parity, abort_flag);
    else return wait_spin(bar, parity, abort_flag);
}

// The request of packed query token t (verify / extend): the largest
// b < batch with cu_seqlens[b] <= t (the entries <= t are a prefix, cu being
// non-decreasing).  The warp loads 256 entries at a time, every load issued
// before any vote, so a batch of up to 256 costs one round trip instead of a
// binary search's chain of loads.  Every lane of the warp calls this.
__device__ __forceinline__ int request_of(const Params& p, int t) {
    const int lane = threadIdx.x & 31;
    int b = 0;
    for (int base = 0; base < p.batch; base += 256) {
        int v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int i = base + 32 * j + lane;
            v[j] = i < p.batch ? __ldg(p.cu_seqlens + i) : INT_MAX;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const unsigned m = __ballot_sync(0xffffffffu, v[j] <= t);
            if (m) b = base + 32 * j + 31 - __clz(m);
        }
    }
    return b;
}

// Token t (of request b, found by request_of in verify / extend) -> request
// row, position and the slots of slice `split`.  In decode the request row
// does not depend on the position, so its load is issued together with the
// sequence length.
__device__ void token_info(const Params& p, int t, int b, int split, TokenInfo& ti, unsigned& err) {
    int pos, trow;
    bool ok = true;
    if (p.cu_seqlens == nullptr) {
        trow = p.rpi ? __ldg(p.rpi + b) : b;
        pos = __ldg(p.seq_lens + b) - 1;
    } else {
        trow = p.rpi ? __ldg(p.rpi + b) : b;
        const int c0 = __ldg(p.cu_seqlens + b), c1 = __ldg(p.cu_seqlens + b + 1);
        if (t < c0 || t >= c1) ok = false;
        pos = __ldg(p.seq_lens + b) - (c1 - c0) + (t - c0);
    }
    if (!ok || pos < 0) {
        err |= DSV4_DEV_ERR_POSITION;
        ok = false;
    }
    if (ok && (trow < 0 || trow >= p.swa_pt_rows || (p.ratio != 0 && trow >= p.ex_pt_rows))) {
        err |= DSV4_DEV_ERR_REQ_ROW;
        ok = false;
    }
    ti.trow = trow;
    ti.pos = pos;
    if (!ok) {
        ti.n_swa = ti.n_c = ti.n_extra = ti.e0 = ti.ne = ti.w0 = ti.nw = ti.ntiles = 0;
        return;
    }
    ti.n_swa = min(pos + 1, p.window);
    ti.n_c = p.ratio ? (pos + 1) / p.ratio : 0;
    ti.n_extra = p.ratio == 4 ? p.topk : (p.ratio == 128 ? ti.n_c : 0);
    const int S = p.csplits * p.gsplits;
    if (ti.n_swa > p.cw * S || ti.n_extra > p.ce * S) err |= DSV4_DEV_ERR_PLAN;
    ti.e0 = min(split * p.ce, ti.n_extra);
    ti.ne = min(ti.e0 + p.ce, ti.n_extra) - ti.e0;
    ti.w0 = min(split * p.cw, ti.n_swa);
    ti.nw = min(ti.w0 + p.cw, ti.n_swa) - ti.w0;
    ti.ntiles = (ti.ne + ti.nw + kTileN - 1) / kTileN;
}

// Window slot w -> physical SWA pool row (-1 = skipped).
__device__ __forceinline__ int resolve_window(const Params& p, const TokenInfo& ti, int w, unsigned& err) {
    const int j = ti.pos - ti.n_swa + 1 + w;
    const int lp = j / kPageSize;
    if (lp >= p.swa_pt_stride) { err |= DSV4_DEV_ERR_SWA_PAGE; return -1; }
    const int page = __ldg(p.swa_pt + (size_t)ti.trow * p.swa_pt_stride + lp);
    if (page < 0 || page >= p.swa_pages) { err |= DSV4_DEV_ERR_SWA_PAGE; return -1; }
    return page * kPageSize + (j % kPageSize);
}

// Extra slot with C4 index (or C128 compressed-row number) idx -> physical
// extra pool row (-1 = skipped).  `cache` (nullable) holds the request's
// extra page-table entries for logical pages lp_lo .. lp_lo + ncache - 1.
__device__ __forceinline__ int resolve_extra(const Params& p, const TokenInfo& ti, int idx, const int* cache,
                                             int lp_lo, int ncache, unsigned& err) {
    if (p.ratio == 4) {
        if (idx < 0) return -1;
        if (idx >= ti.n_c) { err |= DSV4_DEV_ERR_INDEX_RANGE; return -1; }
    }
    const int lp = idx / kPageSize;
    if (lp >= p.ex_pt_stride) { err |= DSV4_DEV_ERR_EXTRA_PAGE; return -1; }
    const int page = (cache != nullptr && lp >= lp_lo && lp < lp_lo + ncache)
                         ? cache[lp - lp_lo]
                         : __ldg(p.ex_pt + (size_t)ti.trow * p.ex_pt_stride + lp);
    if (page < 0 || page >= p.ex_pages) { err |= DSV4_DEV_ERR_EXTRA_PAGE; return -1; }
    return page * kPageSize + (idx % kPageSize);
}

// Key slot (position in the token's list) -> physical row, for the debug dump.
__device__ __forceinline__ int resolve_key_slot(const Params& p, int t, const TokenInfo& ti, int slot, unsigned& err) {
    if (slot < ti.n_swa) return resolve_window(p, ti, slot, err);
    const int e = slot - ti.n_swa;
    const int idx = p.ratio == 4 ? __ldg(p.topk_idx + (size_t)t * p.topk + e) : e;
    return resolve_extra(p, ti, idx, nullptr, 0, 0, err);
}

// Source row of the slice's virtual slot v (extra slots first) in its pool.
__device__ __forceinline__ const uint8_t* slot_row_ptr(const Params& p, const TokenInfo& ti, int v, int row) {
    return v < ti.ne ? p.ex_rows + (size_t)row * p.ex_row_bytes : p.swa_rows + (size_t)row * p.swa_row_bytes;
}

// Byte offset of 16-byte piece `piece` (0..7) of the 128-byte line `line` in
// a 1024-byte-aligned 128B-swizzled buffer.
__device__ __forceinline__ uint32_t sw128(uint32_t line, uint32_t piece) {
    return line * 128u + ((piece ^ (line & 7u)) << 4);
}

// OR of `pred` over the `count` threads taking part in named barrier `id`.
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n"
        " bar.red.or.pred p, %2, %3, q;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void prefetch_l2(const void* ptr, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}

template <int KV_FORMAT>
__global__ void __launch_bounds__(kThreads, 1) dsv4_attn_kernel(const __grid_constant__ Params p) {
    constexpr bool kOutOfLineWait = KV_FORMAT == DSV4_KV_BF16;   // the FP8 loader inlines its waits
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_u32(smem_raw);
    uint8_t* smem = smem_raw;
    if (base & 1023u) {
        // the 128-byte swizzle atoms need a 1024-byte-aligned base (uniform
        // over the grid, so every CTA of a cluster leaves here together)
        if (threadIdx.x == 0) atomicOr(&g_dev_error, DSV4_DEV_ERR_PLAN);
        return;
    }

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int G = p.groups;
    const int Sc = p.csplits;
    const int cs = static_cast<int>(cluster_ctarank());   // slice within the cluster (= blockIdx.x % Sc)
    const int grp = (blockIdx.x / Sc) % G;                 // head group (one cluster per group)
    const int t = blockIdx.x / (Sc * G);                   // query token
    const int gsplit = blockIdx.y;
    const int split = gsplit * Sc + cs;
    const int head0 = grp * kHG;
    const int hcount = min(kHG, p.H - head0);
    const bool is_loader = warp >= kSoftmaxWarps && warp < kQkWarp;
    const int lt = tid - kSoftmaxWarps * 32;           // loader thread (when is_loader)

    const uint32_t sQ = base + OFF_Q, sKV = base + OFF_KV, sP = base + OFF_P;
    int* ring = reinterpret_cast<int*>(smem + OFF_RING);
    float2* ml = reinterpret_cast<float2*>(smem + OFF_ML);
    float* wsm = reinterpret_cast<float*>(smem + OFF_W);
    const uint32_t bars = base + OFF_BAR;
    auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    int* abort_flag = reinterpret_cast<int*>(smem + OFF_MISC + 4);

    unsigned err = 0;
    if (tid == 0) DSV4_TR(0);
    // Launched as a programmatic dependent of the previous kernel in the
    // stream: barrier set-up and the TMEM allocation overlap its tail; every
    // read of an input waits for its completion.  The barriers are set up by
    // an MMA issuer warp, idle until the first tile lands, so that the
    // threads whose loads start the gather are not delayed by it.
    if (tid == (kMmaWarp0 + 2) * 32) {
        mbar_init(bar(B_Q_FULL), kSoftmaxWarps * 32);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(B_KV_FULL + s), KV_FORMAT == DSV4_KV_BF16 ? kLoadThreads : kFp8DqThreads);
            mbar_init(bar(B_KV_EMPTY + s), kMmaWarps);     // every value tile's PV
            mbar_init(bar(B_MASK_FULL + s), KV_FORMAT == DSV4_KV_BF16 ? 1 : 2);   // FP8: one per copier warp
            mbar_init(bar(B_RAW_FULL + s), 2);
        }
        mbar_init(bar(B_S_FULL), kMmaWarps);                // every dim quarter of S
        mbar_init(bar(B_S_FREE), kSoftmaxWarps * 32);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_P_FULL + s), kSoftmaxWarps * 32);
            mbar_init(bar(B_P_FREE + s), kMmaWarps);
        }
        mbar_init(bar(B_O_FINAL), kMmaWarps);
        mbar_init(bar(B_MERGE), 1);
        fence_mbar_init_cluster();
        *abort_flag = 0;
    }
    if (warp == kQkWarp) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the merge-weight threads (warps 0..3, lanes 0..15: head 16 * warp + lane)
    // fetch their head's sink logit now, off the epilogue's critical path
    float sink_l2 = -INFINITY;
    if (warp < 4 && lane < 16 && 16 * warp + lane < hcount) sink_l2 = __ldg(p.sink + head0 + 16 * warp + lane) * kLog2e;

    // ------------------------------------------------------------ set-up
    // Loads that need no position, issued together with the position's: the
    // C4 index of this loader thread's first extra slot, and (when the
    // request row is the token's own) the slice's entries of the extra page
    // table, kept for the first 192 slots in the P area (free until the first
    // probabilities).  C4 indices can point anywhere in the request, so C4
    // keeps the row's first kPtCache entries; a C128 slice reads its own
    // contiguous range.
    int* pt_cache = reinterpret_cast<int*>(smem + OFF_P);
    const int e0n = split * p.ce;                        // the slice's first extra slot
    int lp_lo = 0, ncache = 0;
    if (p.ratio == 4) {
        ncache = min(p.ex_pt_stride, kPtCache);
    } else if (p.ratio == 128) {
        lp_lo = e0n / kPageSize;
        ncache = max(0, min(p.ex_pt_stride - lp_lo, (min(p.ce, kRingHalf) + kPageSize - 1) / kPageSize + 1));
    }
    // the token's request (verify / extend: one warp-wide lookup); without
    // req_pool_indices it is also the page-table row
    const int b_req = p.cu_seqlens == nullptr ? t : request_of(p, t);
    const bool early_row = p.rpi == nullptr && p.ratio != 0 && b_req < p.ex_pt_rows;
    int pre_idx = -1;
    if (is_loader) {
        if (p.ratio == 4 && lt < min(p.ce, kRingHalf) && e0n + lt < p.topk)
            pre_idx = __ldg(p.topk_idx + (size_t)t * p.topk + e0n + lt);
        if (early_row)
            for (int k = lt; k < ncache; k += kLoadThreads)
                pt_cache[k] = __ldg(p.ex_pt + (size_t)b_req * p.ex_pt_stride + lp_lo + k);
    }
    // every thread derives the token's coordinates itself (same addresses; the
    // loads overlap the barrier set-up); thread 0 reports the errors
    TokenInfo ti;
    {
        unsigned e0 = 0;
        token_info(p, t, b_req, split, ti, e0);
        if (tid == 0) err |= e0;
    }
    if (is_loader && !early_row && p.ratio != 0 && ti.ntiles > 0)
        for (int k = lt; k < ncache; k += kLoadThreads)
            pt_cache[k] = __ldg(p.ex_pt + (size_t)ti.trow * p.ex_pt_stride + lp_lo + k);
    // the early C4 indices by extra slot (the thread that resolves slot e0 + v
    // depends on the padding, known only now), in ring half 1 until chunk 1
    if (is_loader && lt < kRingHalf) ring[kRingHalf + lt] = pre_idx;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int ntiles = ti.ntiles;
    if (tid == 0) DSV4_TR(1);
    if (is_loader) {
        // ============================================================ loader
        const int lw = lt >> 5;
        if (p.debug_rows != nullptr && grp == 0) {
            // this slice's key slots (slice 0 also marks the unused tail)
            int* dbg = p.debug_rows + (size_t)t * p.debug_stride;
            for (int w = lt; w < ti.nw; w += kLoadThreads)
                dbg[ti.w0 + w] = resolve_window(p, ti, ti.w0 + w, err);
            for (int e = lt; e < ti.ne; e += kLoadThreads)
                dbg[ti.n_swa + ti.e0 + e] = resolve_key_slot(p, t, ti, ti.n_swa + ti.e0 + e, err);
            if (split == 0)
                for (int k = ti.n_swa + ti.n_extra + lt; k < p.debug_stride; k += kLoadThreads) dbg[k] = -1;
        }
        const int nv = ti.ne + ti.nw;                    // the slice's slots
        // Tile i holds the tile positions 48 i .. 48 i + 47; position u is the
        // slice's virtual slot u - shift (extra slots first, then window
        // slots), and u < shift are padding.  The short tile of a slice is its
        // first one: it finishes early and frees a stage while the full tiles
        // are still landing.
        const int shift = ntiles * kTileN - nv;
        // Chunk c of the slice (kRingHalf positions) goes to ring half c & 1.
        // In chunk 0 the extra slots resolve from the loads issued with the
        // position; a window slot's page-table load is issued then too, and
        // its row is entered only before the first tile that holds a window
        // slot, so the extra-only tiles start one round trip earlier.
        const int u_win = ti.ne + shift;                 // tile position of the first window slot
        const int win_tile = (u_win < kRingHalf && ti.nw > 0) ? u_win / kTileN : -1;   // in chunk 0
        int win_j = -1, win_page = -1;                   // a deferred window slot: position, raw page id
        auto resolve_chunk = [&](int c) {
            if (lt >= kRingHalf) return;
            const int v = c * kRingHalf + lt - shift;
            int row = -1;
            if (v >= 0 && v < nv) {
                if (v < ti.ne) {
                    const int e = ti.e0 + v;
                    const int idx = p.ratio == 4 ? (c == 0 ? ring[kRingHalf + v] : __ldg(p.topk_idx + (size_t)t * p.topk + e)) : e;
                    row = resolve_extra(p, ti, idx, pt_cache, lp_lo, c == 0 ? ncache : 0, err);
                } else if (c == 0 && win_tile >= 0) {
                    // only issue the page-table load here; its value is used
                    // before tile win_tile, so this thread does not wait on it now
                    win_j = ti.pos - ti.n_swa + 1 + ti.w0 + v - ti.ne;
                    const int lp = win_j / kPageSize;
                    if (lp < p.swa_pt_stride) win_page = __ldg(p.swa_pt + (size_t)ti.trow * p.swa_pt_stride + lp);
                    else win_j = -2;
                } else {
                    row = resolve_window(p, ti, ti.w0 + v - ti.ne, err);
                }
            }
            ring[(c & 1) * kRingHalf + lt] = row;
        };
        if (ntiles > 0) {
            resolve_chunk(0);
            named_barrier_sync(1, kLoadThreads);
            if (lt == 0) DSV4_TR(3);
        }
        constexpr int kR = kTileN / kLoadWarps;          // rows per loader warp
        // before tile i's ring entries are read: chunk c's barrier, and chunk
        // 0's deferred window rows
        auto ring_ready = [&](int i) {
            if ((i & 3) == 0 && i > 0) named_barrier_sync(1, kLoadThreads);   // chunk i / 4 resolved
            if (i == win_tile) {
                const int v = lt - shift;
                if (lt < kRingHalf && v >= ti.ne && v < nv) {
                    int row = -1;
                    if (win_j == -2 || win_page < 0 || win_page >= p.swa_pages) err |= DSV4_DEV_ERR_SWA_PAGE;
                    else row = win_page * kPageSize + (win_j % kPageSize);
                    ring[lt] = row;
                }
                named_barrier_sync(1, kLoadThreads);
            }
        };
        auto tile_rows = [&](int i) { return ring + ((i >> 2) & 1) * kRingHalf + (i & 3) * kTileN; };
        // validity of tile i's key slots as a 64-bit mask (warp 0's lanes:
        // lane l checks rows l and 32 + l); read from the ring together with
        // the tile's rows
        auto tile_mask = [&](int i) -> uint64_t {
            const int v0 = i * kTileN - shift;
            const int* rg = tile_rows(i);
            const bool ok0 = v0 + lane >= 0 && v0 + lane < nv && rg[lane] >= 0;
            const bool ok1 = lane + 32 < kTileN && v0 + lane + 32 >= 0 && v0 + lane + 32 < nv && rg[lane + 32] >= 0;
            const unsigned b0 = __ballot_sync(0xffffffffu, ok0);
            const unsigned b1 = __ballot_sync(0xffffffffu, ok1);
            return static_cast<uint64_t>(b0) | (static_cast<uint64_t>(b1) << 32);
        };
        // warp 0 publishes tile i's mask once the tile is on its way; then
        // the next chunk's rows are resolved once this chunk's first two
        // tiles are issued (ring half (c + 1) & 1 was last read by chunk
        // c - 1, whose rows and masks every loader has read before the
        // barrier that opens chunk c)
        auto publish_mask = [&](int i, uint64_t mask) {
            if (lane == 0) {
                const int stage = i % kStages;
                *reinterpret_cast<volatile uint64_t*>(smem + OFF_MASK + stage * 8) = mask;
                mbar_arrive(bar(B_MASK_FULL + stage));
            }
        };
        auto tile_tail = [&](int i) {
            if (lt == 0 && i < 8) DSV4_TR(4 + i);
            const int c = i >> 2;
            if ((i & 3) == 1 && (c + 1) * kRingHalf < nv + shift) resolve_chunk(c + 1);
        };
        if constexpr (KV_FORMAT == DSV4_KV_BF16) {
            for (int i = 0; i < ntiles; ++i) {
                const int stage = i % kStages, use = i / kStages;
                ring_ready(i);
                const int v0 = i * kTileN - shift;                                // virtual slot of row 0 (may be padding)
                const int* rg = tile_rows(i);
                const uint32_t dst_stage = sKV + stage * kStageBytes;
                if (i >= kStages) {
                    wait_bar<kOutOfLineWait>(bar(B_KV_EMPTY + stage), (use - 1) & 1, abort_flag);
                    fence_proxy_async();
                }
#pragma unroll
                for (int k = 0; k < kR; ++k) {
                    const int r = lw * kR + k;
                    const int v = v0 + r;
                    const int row = (v >= 0 && v < nv) ? rg[r] : -1;
                    const uint8_t* src = row >= 0 ? slot_row_ptr(p, ti, v, row) : p.swa_rows;
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int piece = lane + 32 * h2;       // 16-byte piece of the 1 KB row
                        const uint32_t dst = dst_stage + (piece >> 3) * kChunkKV + sw128(r, piece & 7);
                        cp_async_16(dst, src + (row >= 0 ? piece * 16 : 0), row >= 0 ? 16u : 0u);
                    }
                }
                cp_async_arrive_noinc(bar(B_KV_FULL + stage));
                if (lw == 0) publish_mask(i, tile_mask(i));
                tile_tail(i);
            }
        } else {
            // Packed FP8 rows.  Loader warps 6 and 7 copy them, two tiles
            // ahead: each 608-byte row by one bulk copy into the top of its
            // tile's stage (rows 0..31 by warp 6, 32..47 by warp 7, which
            // also publish the tile's key mask, one 32-bit half each).  Warps
            // 0..5 dequantise: lane 4 k + q of warp w holds row 8 w + k,
            // dims 64 m + 16 q .. + 15 of every 64-dim block m (e4m3 x the
            // block's fp32 scale, rounded to bf16) and rope dims 16 q .. + 15
            // (already bf16).  The bf16 tile overwrites the raw rows, so the
            // six warps read all their raw bytes, meet, then write; every
            // shared access spreads its 16-byte pieces evenly over the banks.
            // A padded or masked row is written as zeros.
            static_assert(kFp8DqWarps * 8 == kTileN && kLoadWarps == kFp8DqWarps + 2, "FP8 loader roles");
            constexpr uint32_t kRawOff = kStageBytes - kTileN * kFp8RowBytes;
            static_assert(kRawOff % 16 == 0 && kFp8RowBytes % 16 == 0, "bulk copies move 16-byte units");
            if (lw >= kFp8DqWarps) {
                // ---------------------------------------------- row copies
                const int r = (lw - kFp8DqWarps) * 32 + lane;   // this lane's row of every tile
                for (int j = 0; j < ntiles; ++j) {
                    const int stage = j % kStages;
                    if ((j & 3) == 0 && j > 0) named_barrier_sync(1, kLoadThreads);   // chunk j / 4 resolved
                    if (j == win_tile) named_barrier_sync(1, kLoadThreads);          // deferred window rows
                    if (j >= kStages) {
                        // stage j % 3 held tile j - 3 (and its mask) until its PV finished
                        wait_bar<kOutOfLineWait>(bar(B_KV_EMPTY + stage), (j / kStages - 1) & 1, abort_flag);
                        fence_proxy_async();
                    }
                    const int v = j * kTileN - shift + r;
                    const int row = (r < kTileN && v >= 0 && v < nv) ? tile_rows(j)[r] : -1;
                    const unsigned valid = __ballot_sync(0xffffffffu, row >= 0);
                    if (lane == 0) {
                        reinterpret_cast<volatile uint32_t*>(smem + OFF_MASK + stage * 8)[lw - kFp8DqWarps] = valid;
                        mbar_arrive(bar(B_MASK_FULL + stage));
                        mbar_arrive_expect_tx(bar(B_RAW_FULL + stage), __popc(valid) * kFp8RowBytes);
                    }
                    __syncwarp();
                    if (row >= 0)
                        bulk_copy_g2s(sKV + stage * kStageBytes + kRawOff + r * kFp8RowBytes,
                                      slot_row_ptr(p, ti, v, row), kFp8RowBytes, bar(B_RAW_FULL + stage));
                }
            } else {
                // ---------------------------------------------- dequantisation
                if (win_tile >= 0) {
                    ring_ready(win_tile);           // enters the deferred window rows, then waits with the copiers
                }
                const int k = lane >> 2, q = lane & 3;
                const int r = lw * 8 + k;
                for (int i = 0; i < ntiles; ++i) {
                    const int stage = i % kStages;
                    const uint32_t dst_stage = sKV + stage * kStageBytes;
                    const uint32_t src = dst_stage + kRawOff + r * kFp8RowBytes;
                    wait_bar<kOutOfLineWait>(bar(B_RAW_FULL + stage), (i / kStages) & 1, abort_flag);
                    const bool ok = (*reinterpret_cast<volatile uint64_t*>(smem + OFF_MASK + stage * 8) >> r) & 1ull;
                    uint4 nope[7], rope[2];
                    float scl[7];
                    if (ok) {
#pragma unroll
                        for (int m = 0; m < 7; ++m) nope[m] = ld_shared_u4(src + (4 * m + q) * 16);
                        rope[0] = ld_shared_u4(src + kFp8NopeBytes + q * 32);
                        rope[1] = ld_shared_u4(src + kFp8NopeBytes + q * 32 + 16);
                        const float4 s03 = ld_shared_v4(src + kFp8ScaleOff);
                        const float4 s46 = ld_shared_v4(src + kFp8ScaleOff + 16);
                        scl[0] = s03.x; scl[1] = s03.y; scl[2] = s03.z; scl[3] = s03.w;
                        scl[4] = s46.x; scl[5] = s46.y; scl[6] = s46.z;
                    } else {
#pragma unroll
                        for (int m = 0; m < 7; ++m) { nope[m] = make_uint4(0, 0, 0, 0); scl[m] = 0.f; }
                        rope[0] = rope[1] = make_uint4(0, 0, 0, 0);
                    }
                    named_barrier_sync(4, kFp8DqThreads);       // every raw row of the stage is read
#pragma unroll
                    for (int m = 0; m < 7; ++m) {
                        const uint32_t w[4] = {nope[m].x, nope[m].y, nope[m].z, nope[m].w};
                        uint32_t o[8];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float f[4];
                            e4m3x4_to_f32(w[e], f);
                            o[2 * e] = pack_bf16x2(f[0] * scl[m], f[1] * scl[m]);
                            o[2 * e + 1] = pack_bf16x2(f[2] * scl[m], f[3] * scl[m]);
                        }
                        const uint32_t cb = dst_stage + m * kChunkKV;
                        st_shared_v4(cb + sw128(r, 2 * q), o[0], o[1], o[2], o[3]);
                        st_shared_v4(cb + sw128(r, 2 * q + 1), o[4], o[5], o[6], o[7]);
                    }
                    {
                        const uint32_t cb = dst_stage + 7 * kChunkKV;
                        st_shared_v4(cb + sw128(r, 2 * q), rope[0].x, rope[0].y, rope[0].z, rope[0].w);
                        st_shared_v4(cb + sw128(r, 2 * q + 1), rope[1].x, rope[1].y, rope[1].z, rope[1].w);
                    }
                    fence_proxy_async();
                    mbar_arrive(bar(B_KV_FULL + stage));
                    if (lt == 0 && i < 8) DSV4_TR(4 + i);
                    // the next chunk's rows once this chunk's first two tiles
                    // are in: ring half (c + 1) & 1 last held chunk c - 1, whose
                    // tiles were all copied before this tile's rows were
                    const int c = i >> 2;
                    if ((i & 3) == 1 && (c + 1) * kRingHalf < nv + shift) {
                        resolve_chunk(c + 1);
                        named_barrier_arrive(1, kLoadThreads);
                    }
                }
                // after an abort the waits above may have returned early: let
                // the last copies land (bounded) before the stages are reused
                // or the CTA exits
                for (int j = ntiles - 1; j >= 0 && j >= ntiles - kStages; --j) {
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try(bar(B_RAW_FULL + j % kStages), (j / kStages) & 1))
                        if (globaltimer_ns() - t0 > kTimeoutNs) break;
                }
            }
        }
        cp_async_wait_all();
    } else if (warp >= kMmaWarp0) {
        // ============================================================ MMA issuers
        // Warp kMmaWarp0 + q issues, for every tile, S = Q K^T over dims
        // 128 q .. 128 q + 127 into its own partial score sum (the softmax adds
        // the four), and O^T += V^T P^T for value dims 128 q .. 128 q + 127
        // (M = 128 value dims, N = 64 heads, K = 48 keys; A = the same KV
        // stage read MN-major).  A tcgen05.mma costs its issuing thread about
        // as long as a small MMA runs, so four issuers keep the tensor pipe fed.
        // S of tile i needs the tile's rows and the softmax to have read S of
        // tile i - 1 (one score buffer); PV of tile j needs its probabilities.
        const int mq = warp - kMmaWarp0;
        if (lane == 0 && ntiles > 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(kHG, kTileN, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, kHG, true, false);
            wait_bar<kOutOfLineWait>(bar(B_Q_FULL), 0, abort_flag);
            fence_proxy_async();
            tc_fence_after();
            // S of tile i and PV of tile i - 1 are issued in whichever order
            // their inputs are ready (PV must not wait for the next tile's rows)
            auto issue_s = [&](int i) {
                const int stage = i % kStages;
                if (mq == 0 && i < 8) DSV4_TR(12 + i);
                fence_proxy_async();
                tc_fence_after();
                const uint32_t stg = sKV + stage * kStageBytes;
                const uint32_t dcol = tmem + kTmemS + mq * kTileN;
#pragma unroll
                for (int kq = 0; kq < 8; ++kq) {
                    const int k = 8 * mq + kq;
                    const uint64_t a = smem_desc_sw128(sQ + (k >> 2) * kChunkQ + (k & 3) * 32, 16, 1024);
                    const uint64_t b = smem_desc_sw128(stg + (k >> 2) * kChunkKV + (k & 3) * 32, 16, 1024);
                    mma_bf16_ss(dcol, a, b, idesc_qk, kq > 0 ? 1u : 0u);
                }
                mma_commit(bar(B_S_FULL));
            };
            auto issue_pv = [&](int j) {
                const int stage = j % kStages;
                if (j < 8 && mq == 0) DSV4_TR(20 + j);
                tc_fence_after();
                const uint32_t stg = sKV + stage * kStageBytes;
                const uint32_t pbuf = sP + (j & 1) * kPBytes;
#pragma unroll
                for (int kk = 0; kk < kTileN / 16; ++kk) {
                    // A = V^T (dims 128*mq.., keys 16*kk..): MN-major, 64-dim atoms one chunk apart
                    const uint64_t a = smem_desc_sw128(stg + 2 * mq * kChunkKV + kk * 2048, kChunkKV, 1024);
                    // B = P (heads x keys), K-major
                    const uint64_t b = smem_desc_sw128(pbuf + kk * 32, 16, 1024);
                    mma_bf16_ss(tmem + kTmemO + mq * kHG, a, b, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar(B_P_FREE + (j & 1)));
                mma_commit(bar(B_KV_EMPTY + stage));
            };
            int ns = 0, np = 0;                    // S issued for tiles < ns, PV for tiles < np
            const uint64_t t0 = globaltimer_ns();
            for (uint32_t it = 1; np < ntiles; ++it) {
                bool progress = false;
                if (ns < ntiles && mbar_test(bar(B_KV_FULL + ns % kStages), (ns / kStages) & 1) &&
                    (ns == 0 || mbar_test(bar(B_S_FREE), (ns - 1) & 1))) {
                    issue_s(ns++);
                    progress = true;
                }
                if (np < ns && mbar_test(bar(B_P_FULL + (np & 1)), (np >> 1) & 1)) {
                    issue_pv(np++);
                    progress = true;
                }
                if (!progress && (it & 63u) == 0) {
                    if (*reinterpret_cast<volatile int*>(abort_flag)) break;
                    if (globaltimer_ns() - t0 > kTimeoutNs) {
                        atomicOr(&g_dev_error, DSV4_DEV_ERR_TIMEOUT);
                        *reinterpret_cast<volatile int*>(abort_flag) = 1;
                        break;
                    }
                }
            }
            mma_commit(bar(B_O_FINAL));
        }
        __syncwarp();
    } else if (warp < kSoftmaxWarps) {
        // ============================================================ softmax
        // Q rows of this head group (1 KB each), zero past the last head
        {
            const uint8_t* qb = reinterpret_cast<const uint8_t*>(p.q) + ((size_t)t * p.H + head0) * 1024;
            for (int k = tid; k < kHG * 64; k += kSoftmaxWarps * 32) {
                const int r = k >> 6, piece = k & 63;
                const uint32_t dst = sQ + (piece >> 3) * kChunkQ + sw128(r, piece & 7);
                const bool on = r < hcount && ntiles > 0;
                cp_async_16(dst, on ? qb + (size_t)r * 1024 + piece * 16 : qb, on ? 16u : 0u);
            }
            cp_async_arrive_noinc(bar(B_Q_FULL));
        }
        // Head row h of S lives in TMEM lane 32*(h / 16) + h % 16 (M = 64).  The
        // 16x64b access shape gives thread t of warp h / 16 the columns of
        // parity (t >> 1) & 1 of lane (t >> 2) + 8 * (t & 1): threads t and
        // t ^ 2 share a head and hold its even and odd keys.
        const int qd = warp;
        const int par = (lane >> 1) & 1;
        const int h = qd * 16 + (lane >> 2) + 8 * (lane & 1);
        const bool live = h < hcount;
        const bool owner = par == 0;                 // writes the head's per-head values
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(qd * 32) << 16);
        constexpr int kJ = kTileN / 2;               // keys per thread
        constexpr int kW = kJ / 2;                   // bf16 words each thread of the pair writes
        float m_run = -INFINITY, l_run = 0.f;
        for (int i = 0; i < ntiles; ++i) {
            const int sb = i & 1;
            const int stage = i % kStages, use = i / kStages;
            float s[kJ];
            wait_bar<kOutOfLineWait>(bar(B_S_FULL), i & 1, abort_flag);
            if (tid == 0 && i < 8) DSV4_TR(28 + i);
            __syncwarp();
            tc_fence_after();
            tmem_ld16x64b_48_sum4(lane_addr + kTmemS, s);
            tc_fence_before();
            mbar_arrive(bar(B_S_FREE));
            wait_bar<kOutOfLineWait>(bar(B_MASK_FULL + stage), use & 1, abort_flag);
            const uint64_t mask = *reinterpret_cast<volatile uint64_t*>(smem + OFF_MASK + stage * 8) >> par;
            // four independent partial maxima and sums keep the dependent
            // chains short
            float tm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int j = 0; j < kJ; ++j) {
                s[j] = ((mask >> (2 * j)) & 1ull) ? s[j] * p.scale_log2 : -INFINITY;
                tm[j & 3] = fmaxf(tm[j & 3], s[j]);
            }
            float tmax = fmaxf(fmaxf(tm[0], tm[1]), fmaxf(tm[2], tm[3]));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
            const bool need = live && tmax > m_run + kRescaleLog2;
            float alpha = 1.f;
            if (need) {
                alpha = fast_exp2(m_run - tmax);
                m_run = tmax;
            }
            float pv[kJ];
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
            const bool any = live && m_run != -INFINITY;
#pragma unroll
            for (int j = 0; j < kJ; ++j) {
                // the denominator sums the fp32 probabilities; the bf16 copies
                // only feed the PV product
                pv[j] = any ? fast_exp2(s[j] - m_run) : 0.f;
                ls[j & 3] += pv[j];
            }
            l_run = l_run * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
            // bf16 words (key 2w, key 2w + 1) of the head's line: the even-key
            // thread builds words 0..kW-1, the odd-key thread words kW..2kW-1
            uint32_t wd[kW];
#pragma unroll
            for (int m = 0; m < kW / 2; ++m) {
                const uint32_t snd = par ? pack_bf16x2(pv[2 * m], pv[2 * m + 1])
                                         : pack_bf16x2(pv[kW + 2 * m], pv[kW + 2 * m + 1]);
                const uint32_t rcv = __shfl_xor_sync(0xffffffffu, snd, 2);
                const uint32_t own = par ? pack_bf16x2(pv[kW + 2 * m], pv[kW + 2 * m + 1])
                                         : pack_bf16x2(pv[2 * m], pv[2 * m + 1]);
                const uint32_t ev = par ? rcv : own;   // even keys of words 2m, 2m + 1 of this thread's range
                const uint32_t od = par ? own : rcv;   // odd keys
                wd[2 * m] = __byte_perm(ev, od, 0x5410);
                wd[2 * m + 1] = __byte_perm(ev, od, 0x7632);
            }
            if (i > 0) {
                // a head whose running max moved scales its O^T column; each
                // softmax warp scales the 32 value dims of its TMEM quadrant
                if (bar_red_or(2, kSoftmaxWarps * 32, need)) {
                    if (owner) wsm[h] = alpha;
                    named_barrier_sync(2, kSoftmaxWarps * 32);
                    wait_bar<kOutOfLineWait>(bar(B_P_FREE + ((i - 1) & 1)), ((i - 1) >> 1) & 1, abort_flag);
                    __syncwarp();
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) {
                        float o[32];
                        tmem_ld32(lane_addr + kTmemO + c * 32, o);
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] *= wsm[(c & 1) * 32 + j];
                        tmem_st32(lane_addr + kTmemO + c * 32, o);
                    }
                }
            }
            if (i >= 2) wait_bar<kOutOfLineWait>(bar(B_P_FREE + sb), ((i - 2) >> 1) & 1, abort_flag);
            {
                const uint32_t prow = sP + sb * kPBytes;
#pragma unroll
                for (int q = 0; q < kW / 4; ++q)
                    st_shared_v4(prow + sw128(h, (kW / 4) * par + q), wd[4 * q], wd[4 * q + 1], wd[4 * q + 2],
                                 wd[4 * q + 3]);
            }
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(bar(B_P_FULL + sb));
            if (tid == 0 && i < 8) DSV4_TR(44 + i);
        }
        // the head's denominator is the sum of its two halves
        const float l_all = l_run + __shfl_xor_sync(0xffffffffu, l_run, 2);
        if (owner) ml[h] = make_float2(live && ntiles > 0 ? m_run : -INFINITY, live && ntiles > 0 ? l_all : 0.f);
        fence_proxy_async();
    }

    // ------------------------------------------------------------ epilogue
    // Slice cs owns the 8-dim units [u_lo, u_hi) of the output (nd dims from
    // dbase).  Warp w reads value dims 128 (w / 4) + 32 (w % 4) + lane of O^T
    // (its TMEM lane quadrant) for all heads.  A thread whose dim is owned
    // keeps its 64 values in registers; the other dims go, as bf16 rows, to
    // the outgoing area (row order = dim order without the owned range, so
    // each peer's dims are one contiguous block), from where each warp
    // bulk-stores its rows to the workspace.  After the cluster barrier each
    // slice bulk-loads its dims from every peer and every slice's (m, l) (L2
    // and bulk copies move these far faster than distributed shared memory
    // does), and the owners add them to their registers.  Bf16 rows are 128 B
    // with 16-byte chunk q stored at q ^ (dim & 7).
    const int u_lo = (cs * 64) / Sc, u_hi = ((cs + 1) * 64) / Sc;
    const int nd = 8 * (u_hi - u_lo), dbase = 8 * u_lo;
    const uint32_t sOut = base + OFF_MERGE;                          // outgoing bf16 rows
    uint16_t* mrg_t = p.merge + (((size_t)t * p.gsplits + gsplit) * G + grp) * Sc * (kMergeRowsElems + 4 * kHG);
    float2* mrg_ml = reinterpret_cast<float2*>(mrg_t + Sc * kMergeRowsElems);
    const bool final_out = p.gsplits == 1;
    const uint32_t sIn = base + OFF_Q;                               // peers' bf16 rows [slot][dim]
    const float2* mlx = reinterpret_cast<const float2*>(smem + OFF_Q + (Sc - 1) * nd * 128);   // [slice][head]
    // [slice][head] merge weights: with Sc == 1 they are computed while the
    // last PV may still read P, so they go to the ring (no longer read once the
    // softmax has seen the last tile's mask); otherwise into P, after O_FINAL
    float* W = reinterpret_cast<float*>(smem + (Sc == 1 ? OFF_RING : OFF_P));
    // weights of every slice's accumulator for head h: exp(m_s - M) / L (the
    // sink enters M and L once); thread (warp < 4, lane < 16) owns head 16 warp + lane
    auto merge_weights = [&]() {
        const int h = warp * 16 + lane;
        const bool live = h < hcount;
        float2 mls[kMaxCluster];
#pragma unroll
        for (int s2 = 0; s2 < kMaxCluster; ++s2)
            mls[s2] = s2 < Sc ? (s2 == cs ? ml[h] : mlx[s2 * kHG + h]) : make_float2(-INFINITY, 0.f);
        float M = -INFINITY;
#pragma unroll
        for (int s2 = 0; s2 < kMaxCluster; ++s2) M = fmaxf(M, mls[s2].x);
        const float sk = sink_l2;
        if (final_out) M = fmaxf(M, sk);
        float Lsum = 0.f;
        float e[kMaxCluster];
#pragma unroll
        for (int s2 = 0; s2 < kMaxCluster; ++s2) {
            e[s2] = (M != -INFINITY && mls[s2].x != -INFINITY) ? fast_exp2(mls[s2].x - M) : 0.f;
            Lsum += mls[s2].y * e[s2];
        }
        if (final_out && M != -INFINITY && sk != -INFINITY) Lsum += fast_exp2(sk - M);
        const float inv = (live && Lsum > 0.f) ? 1.f / Lsum : 0.f;
#pragma unroll
        for (int s2 = 0; s2 < kMaxCluster; ++s2)
            if (s2 < Sc) W[s2 * kHG + h] = e[s2] * inv;
        if (live && cs == 0) {
            if (final_out) {
                if (p.lse) p.lse[(size_t)t * p.H + head0 + h] = (Lsum > 0.f ? M + log2f(Lsum) : -INFINITY) * kLn2;
            } else {
                p.part_ml[((size_t)t * p.gsplits + gsplit) * p.H + head0 + h] = make_float2(M, Lsum);
            }
        }
    };
    // the bf16 output (or the fp32 partial of a grid split) of value dim d for
    // all heads; consecutive lanes hold consecutive dims
    auto write_dim = [&](int d, const float (&acc)[kHG]) {
        if (final_out) {
            __nv_bfloat16* o = p.out + ((size_t)t * p.H + head0) * kDim + d;
#pragma unroll
            for (int h = 0; h < kHG; ++h)
                if (h < hcount) o[(size_t)h * kDim] = __float2bfloat16_rn(acc[h]);
        } else {
            float* o = p.part_o + (((size_t)t * p.gsplits + gsplit) * p.H + head0) * kDim + d;
#pragma unroll
            for (int h = 0; h < kHG; ++h)
                if (h < hcount) o[(size_t)h * kDim] = acc[h];
        }
    };
    if (warp < kSoftmaxWarps) {
        // (m, l) of this slice are complete once the four softmax warps are
        named_barrier_sync(3, kSoftmaxWarps * 32);
        if (Sc > 1 && tid == 0) {
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(mrg_ml + cs * kHG),
                         "r"(base + OFF_ML), "r"(static_cast<uint32_t>(kHG * 8))
                         : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        if (Sc == 1 && lane < 16) merge_weights();
    }
    if (Sc == 1) __syncthreads();   // the weights are ready before the read-out
    // ============================================================ O^T read-out
    const int qd = warp & 3, mt = warp >> 2;
    const int d = mt * 128 + qd * 32 + lane;                 // this thread's value dim
    const bool owned = d >= dbase && d < dbase + nd;
    float o[kHG];
    if (ntiles > 0) {
        wait_bar<kOutOfLineWait>(bar(B_O_FINAL), 0, abort_flag);
        if (tid == 0) DSV4_TR(52);
        tc_fence_after();
        fence_proxy_async();
        __syncwarp();
        const uint32_t la = tmem + (static_cast<uint32_t>(qd * 32) << 16) + kTmemO + mt * kHG;
        float a[32], b[32];
        tmem_ld32(la, a);
        tmem_ld32(la + 32, b);
#pragma unroll
        for (int j = 0; j < 32; ++j) { o[j] = a[j]; o[32 + j] = b[j]; }
        if (tid == 0) DSV4_TR(54);
    } else {
#pragma unroll
        for (int j = 0; j < kHG; ++j) o[j] = 0.f;
    }
    if (Sc == 1) {
        // the slice is the whole key list: scale by the weight and write
#pragma unroll
        for (int h = 0; h < kHG; ++h) o[h] *= W[h];
        write_dim(d, o);
    } else {
        if (!owned) {
            const int r = d < dbase ? d : d - nd;
            const uint32_t row = sOut + r * 128;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                st_shared_v4(row + ((q ^ (d & 7)) << 4), pack_bf16x2(o[8 * q], o[8 * q + 1]),
                             pack_bf16x2(o[8 * q + 2], o[8 * q + 3]), pack_bf16x2(o[8 * q + 4], o[8 * q + 5]),
                             pack_bf16x2(o[8 * q + 6], o[8 * q + 7]));
        }
        // the warp's 32 dims outside the owned range -> workspace rows [cs][dim][head]
        // (at most two runs of rows)
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
            const int d0 = mt * 128 + qd * 32, d1 = d0 + 32;
            const int runs[2][2] = {{d0, min(d1, dbase)}, {max(d0, dbase + nd), d1}};
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int a0 = runs[k][0], a1 = runs[k][1];
                if (a0 >= a1) continue;
                const int r0 = a0 < dbase ? a0 : a0 - nd;
                uint16_t* dst = mrg_t + ((size_t)cs * kDim + a0) * kHG;
                asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                             "r"(sOut + r0 * 128), "r"(static_cast<uint32_t>((a1 - a0) * 128))
                             : "memory");
            }
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
            asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        __syncwarp();
        if (tid == 0) DSV4_TR(60);
        tc_fence_before();
        cluster_sync();   // B: every slice's rows and (m, l) are published
        tc_fence_after();
        if (tid == 0) DSV4_TR(55);
        if (tid == kQkWarp * 32) {
            // this slice's dims from every other slice (one contiguous block
            // each) and every slice's (m, l)
            asm volatile("fence.proxy.async.global;" ::: "memory");
            const uint32_t mb = bar(B_MERGE);
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb),
                         "r"(static_cast<uint32_t>((Sc - 1) * nd * 128 + Sc * kHG * 8))
                         : "memory");
            int slot = 0;
            for (int s2 = 0; s2 < Sc; ++s2) {
                if (s2 == cs) continue;
                const uint16_t* src = mrg_t + ((size_t)s2 * kDim + dbase) * kHG;
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                        sIn + slot * nd * 128),
                    "l"(src), "r"(static_cast<uint32_t>(nd * 128)), "r"(mb)
                    : "memory");
                ++slot;
            }
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    sIn + (Sc - 1) * nd * 128),
                "l"(mrg_ml), "r"(static_cast<uint32_t>(Sc * kHG * 8)), "r"(mb)
                : "memory");
        }
        wait_bar<kOutOfLineWait>(bar(B_MERGE), 0, abort_flag);
        if (tid == 0) DSV4_TR(59);
        if (warp < 4 && lane < 16) merge_weights();
        __syncthreads();
        if (tid == 0) DSV4_TR(58);
        if (owned) {
            // own accumulator x own weight + every peer's bf16 row x its weight
            const int dl = d - dbase;
            {
                const float4* w4 = reinterpret_cast<const float4*>(W + cs * kHG);
#pragma unroll
                for (int q = 0; q < kHG / 4; ++q) {
                    const float4 w = w4[q];
                    o[4 * q] *= w.x;
                    o[4 * q + 1] *= w.y;
                    o[4 * q + 2] *= w.z;
                    o[4 * q + 3] *= w.w;
                }
            }
            int slot = 0;
            for (int s2 = 0; s2 < Sc; ++s2) {
                if (s2 == cs) continue;
                const float4* ws = reinterpret_cast<const float4*>(W + s2 * kHG);
                const uint32_t row = sIn + (slot * nd + dl) * 128;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 v = ld_shared_v4(row + ((q ^ (d & 7)) << 4));
                    const uint32_t w4[4] = {__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z),
                                            __float_as_uint(v.w)};
                    const float4 wa = ws[2 * q], wb = ws[2 * q + 1];
                    const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        o[8 * q + 2 * e] += wv[2 * e] * __uint_as_float(w4[e] << 16);
                        o[8 * q + 2 * e + 1] += wv[2 * e + 1] * __uint_as_float(w4[e] & 0xffff0000u);
                    }
                }
                ++slot;
            }
            write_dim(d, o);
        }
    }
    if (tid == 0) DSV4_TR(61);
    if (err) atomicOr(&g_dev_error, err);
    if (tid == 0) DSV4_TR(56);
    // no slice touches another's shared memory after barrier B
    tc_fence_before();
    __syncthreads();
    if (tid == 0) DSV4_TR(57);
    if (warp == kQkWarp) {
        tc_fence_after();
        if (*reinterpret_cast<volatile int*>(abort_flag)) {
            // a wait gave up: give in-flight tensor-core work time to drain
            for (int k = 0; k < 1000; ++k) __nanosleep(10000);
        }
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Merges Sg cluster results of each (token, head): the weights are
// L_g * exp(M_g - M) with M the largest of the M_g and the sink; the sink
// adds exp(sink - M) to the denominator and nothing to the numerator.  One
// thread per (token, head, 4 value dims).  Launched as a programmatic
// dependent of the attention launch: nothing is read before the wait.  The
// groups are taken eight at a time, every load of the eight issued before
// any is used (one memory round trip for Sg <= 8); the running maximum is
// moved between batches by rescaling what has been summed.
constexpr int kCombineUnits = kDim / 4;         // 4-dim units per head
constexpr int kCombineBatch = 8;
__global__ void __launch_bounds__(256) dsv4_combine_kernel(const __grid_constant__ Params p) {
    const int nb = (p.H * kCombineUnits + 255) / 256;          // blocks per token
    const int t = blockIdx.x / nb;
    const int it = (blockIdx.x % nb) * blockDim.x + threadIdx.x;   // (head, 4-dim unit)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (it >= p.H * kCombineUnits) return;
    const int h = it / kCombineUnits;
    const int u = it % kCombineUnits;
    const int Sg = p.gsplits;
    const float sk = p.sink[h] * kLog2e;
    const float2* mlp = p.part_ml + (size_t)t * Sg * p.H + h;
    const float* src = p.part_o + ((size_t)t * Sg * p.H + h) * kDim + u * 4;
    const size_t gstride = (size_t)p.H * kDim;
    float M = sk;                                   // running maximum (log2 units)
    float L = sk != -INFINITY ? 1.f : 0.f;          // exp2(sink - M)
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int g0 = 0; g0 < Sg; g0 += kCombineBatch) {
        float2 ml[kCombineBatch];
        float4 o[kCombineBatch];
#pragma unroll
        for (int k = 0; k < kCombineBatch; ++k) {
            const int g = g0 + k;
            ml[k] = make_float2(-INFINITY, 0.f);
            o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (g < Sg) {
                ml[k] = mlp[(size_t)g * p.H];
                o[k] = *reinterpret_cast<const float4*>(src + g * gstride);
            }
        }
        float mb = M;
#pragma unroll
        for (int k = 0; k < kCombineBatch; ++k)
            if (ml[k].y > 0.f) mb = fmaxf(mb, ml[k].x);
        if (mb == -INFINITY) continue;              // nothing in this batch, nor before it
        if (mb > M) {
            const float r = M == -INFINITY ? 0.f : exp2f(M - mb);
            L *= r;
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[j] *= r;
            M = mb;
        }
#pragma unroll
        for (int k = 0; k < kCombineBatch; ++k) {
            const float w = ml[k].y > 0.f ? ml[k].y * exp2f(ml[k].x - M) : 0.f;
            L += w;
            acc[0] += w * o[k].x;
            acc[1] += w * o[k].y;
            acc[2] += w * o[k].z;
            acc[3] += w * o[k].w;
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint2 v;
    v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(p.out + ((size_t)t * p.H + h) * kDim + u * 4) = v;
    if (u == 0 && p.lse) p.lse[(size_t)t * p.H + h] = (L > 0.f ? M + log2f(L) : -INFINITY) * kLn2;
}

// ------------------------------------------------------------------ host
struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int max_clusters[kMaxCluster + 1] = {0, 0, 0, 0, 0, 0, 0, 0, 0};   // by cluster size
};
constexpr int kMaxDevices = 64;
static DeviceInfo g_devinfo[kMaxDevices];
static std::mutex g_devinfo_mu;

static int device_info(DeviceInfo& out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSV4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_devinfo_mu);
    DeviceInfo& di = g_devinfo[dev];
    if (!di.ready) {
        if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DSV4_ERR_CUDA;
        auto kern = dsv4_attn_kernel<DSV4_KV_BF16>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc) != cudaSuccess)
            return DSV4_ERR_CUDA;
        if (cudaFuncSetAttribute(dsv4_attn_kernel<DSV4_KV_FP8_PACKED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemAlloc) != cudaSuccess)
            return DSV4_ERR_CUDA;
        for (int cl = 1; cl <= kMaxCluster; ++cl) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            cfg.gridDim = dim3(cl, 1, 1);
            cfg.blockDim = dim3(kThreads, 1, 1);
            cfg.dynamicSmemBytes = kSmemAlloc;
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = cl;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
                cudaGetLastError();
                n = di.sms / cl * 3 / 4;
            }
            di.max_clusters[cl] = n > 0 ? n : 1;
        }
        di.ready = true;
    }
    out = di;
    return DSV4_OK;
}

static int list_max(int ratio, int window, int topk, int max_seq_len) {
    const int extra = ratio == 4 ? topk : (ratio == 128 ? max_seq_len / 128 : 0);
    return window + extra;
}

// Split plan: Sc key slices merged inside the kernel (one cluster of Sc CTAs
// per token and head group) times Sg cluster groups merged by the combine
// kernel.  The cost is an estimate in microseconds from measured figures: a
// 48-key tile per CTA, a fixed start-up and epilogue per wave of CTAs, the
// in-cluster merge, and the combine kernel with its fp32 partials.
static int make_plan(int T, int G, int lmax, int num_splits, const DeviceInfo& di, int& sc, int& sg) {
    const int tiles_total = (lmax + kTileN - 1) / kTileN;
    const int max_sc = kMaxCluster;
    if (num_splits > 0) {
        sc = 1;
        for (int c = max_sc; c >= 1; --c)
            if (num_splits % c == 0) { sc = c; break; }
        sg = num_splits / sc;
        return DSV4_OK;
    }
    constexpr double kTileUs = 1.3, kWaveUs = 4.0, kMergeUs = 1.5, kMergeSliceUs = 0.2;
    constexpr double kCombineUs = 3.0, kCombineBytesPerUs = 5.0e6;
    const int H = G * kHG;
    double best = 1e30;
    sc = 1;
    sg = 1;
    for (int c = 1; c <= max_sc; ++c) {
        const int per_wave = di.max_clusters[c];
        for (int g = 1; g <= 64; ++g) {
            const int s = c * g;
            if (s > 1 && s > tiles_total) break;
            const long long clusters = (long long)T * G * g;
            if (g > 1 && clusters > 4LL * per_wave) break;
            const long long waves = (clusters + per_wave - 1) / per_wave;
            const double tiles = std::ceil((double)lmax / s / kTileN);
            double cost = (double)waves * (tiles * kTileUs + kWaveUs + (c > 1 ? kMergeUs + kMergeSliceUs * (c - 1) : 0.0));
            if (g > 1) cost += kCombineUs + (double)T * g * H * kDim * 4 / kCombineBytesPerUs;
            if (cost < best - 1e-9) { best = cost; sc = c; sg = g; }
        }
    }
    return DSV4_OK;
}

int check_pool(const dsv4_kv_pool* pool) {
    if (!pool || !pool->rows || !pool->page_table) return DSV4_ERR_INVALID;
    if (pool->page_size != kPageSize) return DSV4_ERR_UNSUPPORTED;
    if (pool->format == DSV4_KV_BF16) {
        if (pool->row_bytes != 1024) return DSV4_ERR_UNSUPPORTED;
    } else if (pool->format == DSV4_KV_FP8_PACKED) {
        if (pool->row_bytes != kFp8RowBytes) return DSV4_ERR_UNSUPPORTED;
    } else {
        return DSV4_ERR_UNSUPPORTED;
    }
    if (pool->num_pages < 1 || pool->num_pages * kPageSize >= (1LL << 31)) return DSV4_ERR_INVALID;
    if (pool->page_table_rows < 1 || pool->page_table_stride < 1) return DSV4_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(pool->rows) % 16) return DSV4_ERR_INVALID;
    return DSV4_OK;
}

static unsigned int* g_dev_error_addr[kMaxDevices];
static std::mutex g_dev_error_mu;

unsigned int* device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_dev_error_mu);
    if (g_dev_error_addr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_dev_error) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_dev_error_addr[dev] = static_cast<unsigned int*>(ptr);
    }
    return g_dev_error_addr[dev];
}

// Workspace: [fp32 partial outputs and (m, l) of each cluster group when
// Sg > 1][bf16 per-slice accumulators exchanged inside a cluster when Sc > 1].
static size_t ws_part_bytes(int T, int H, int sg) {
    if (sg <= 1) return 0;
    return ((size_t)T * sg * H * kDim * sizeof(float) + (size_t)T * sg * H * sizeof(float2) + 255) & ~size_t(255);
}
static size_t ws_merge_bytes(int T, int G, int sc, int sg) {
    if (sc <= 1) return 0;
    return (size_t)T * sg * G * sc * (kMergeRowsElems * sizeof(uint16_t) + kHG * sizeof(float2));
}
static size_t workspace_bytes_for(int T, int H, int sc, int sg) {
    const int G = (H + kHG - 1) / kHG;
    const size_t n = ws_part_bytes(T, H, sg) + ws_merge_bytes(T, G, sc, sg);
    return n ? n + 256 : 0;
}

struct Call {
    const void* q;
    int T, batch, H;
    const int* seq_lens;
    const int* cu;
    const int* rpi;
    const dsv4_kv_pool* swa;
    int window, ratio;
    const dsv4_kv_pool* extra;
    const int* topk_idx;
    int topk, max_seq_len;
    const float* sink;
    float scale;
    void* out;
    float* lse;
    int num_splits;
    void* ws;
    size_t ws_bytes;
    int* debug_rows;
    void* stream;
};

static int run(const Call& c) {
    if (!c.q || !c.out || !c.seq_lens || !c.sink) return DSV4_ERR_INVALID;
    if (c.T < 1 || c.batch < 1 || c.H < 1 || c.H > 2 * kHG || c.window < 1) return DSV4_ERR_INVALID;
    if (!std::isfinite(c.scale)) return DSV4_ERR_INVALID;
    if (c.ratio != 0 && c.ratio != 4 && c.ratio != 128) return DSV4_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(c.q) % 16 || reinterpret_cast<uintptr_t>(c.out) % 16) return DSV4_ERR_INVALID;
    int rc = check_pool(c.swa);
    if (rc) return rc;
    if (c.ratio != 0) {
        rc = check_pool(c.extra);
        if (rc) return rc;
        if (c.extra->format != c.swa->format) return DSV4_ERR_UNSUPPORTED;
    }
    if (c.ratio == 4 && (!c.topk_idx || c.topk < 1)) return DSV4_ERR_INVALID;
    if (c.ratio == 128 && c.max_seq_len < 1) return DSV4_ERR_INVALID;
    if (c.num_splits < 0) return DSV4_ERR_INVALID;

    DeviceInfo di;
    rc = device_info(di);
    if (rc) return rc;
    const int lmax = list_max(c.ratio, c.window, c.topk, c.max_seq_len);
    const int G = (c.H + kHG - 1) / kHG;
    int sc = 1, sg = 1;
    make_plan(c.T, G, lmax, c.num_splits, di, sc, sg);
    const int splits = sc * sg;
    // each slice takes an equal share of the window slots and of the extra slots
    const int cw = (c.window + splits - 1) / splits, ce = (lmax - c.window + splits - 1) / splits;
    if ((long long)c.T * sc * G > 0x7fffffffLL) return DSV4_ERR_UNSUPPORTED;
    const size_t need = workspace_bytes_for(c.T, c.H, sc, sg);
    if (need > 0 && (!c.ws || c.ws_bytes < need)) return DSV4_ERR_WORKSPACE;

    Params p;
    std::memset(&p, 0, sizeof(p));
    p.q = static_cast<const __nv_bfloat16*>(c.q);
    p.T = c.T;
    p.H = c.H;
    p.batch = c.batch;
    p.groups = G;
    p.seq_lens = c.seq_lens;
    p.cu_seqlens = c.cu;
    p.rpi = c.rpi;
    p.swa_rows = static_cast<const uint8_t*>(c.swa->rows);
    p.swa_pages = c.swa->num_pages;
    p.swa_row_bytes = c.swa->row_bytes;
    p.swa_pt = c.swa->page_table;
    p.swa_pt_rows = c.swa->page_table_rows;
    p.swa_pt_stride = c.swa->page_table_stride;
    p.window = c.window;
    p.ratio = c.ratio;
    if (c.ratio != 0) {
        p.ex_rows = static_cast<const uint8_t*>(c.extra->rows);
        p.ex_pages = c.extra->num_pages;
        p.ex_row_bytes = c.extra->row_bytes;
        p.ex_pt = c.extra->page_table;
        p.ex_pt_rows = c.extra->page_table_rows;
        p.ex_pt_stride = c.extra->page_table_stride;
    }
    p.topk_idx = c.topk_idx;
    p.topk = c.topk;
    p.sink = c.sink;
    p.scale_log2 = static_cast<float>(static_cast<double>(c.scale) * 1.4426950408889634);
    p.cw = cw;
    p.ce = ce;
    p.csplits = sc;
    p.gsplits = sg;
    p.out = static_cast<__nv_bfloat16*>(c.out);
    p.lse = c.lse;
    if (need > 0) {
        const uintptr_t w = (reinterpret_cast<uintptr_t>(c.ws) + 255) & ~uintptr_t(255);
        if (sg > 1) {
            p.part_o = reinterpret_cast<float*>(w);
            p.part_ml = reinterpret_cast<float2*>(w + (size_t)c.T * sg * c.H * kDim * sizeof(float));
        }
        if (sc > 1) p.merge = reinterpret_cast<uint16_t*>(w + ws_part_bytes(c.T, c.H, sg));
    }
    p.debug_rows = c.debug_rows;
    p.debug_stride = lmax;

    cudaStream_t st = static_cast<cudaStream_t>(c.stream);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3(static_cast<unsigned>(sc * G * c.T), sg, 1);   // x: (token, head group, slice)
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemAlloc;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = sc;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic dependent launch: the kernel waits for the previous
    // kernel in the stream (griddepcontrol.wait) before it reads any input
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const cudaError_t le = c.swa->format == DSV4_KV_BF16
                               ? cudaLaunchKernelEx(&cfg, dsv4_attn_kernel<DSV4_KV_BF16>, p)
                               : cudaLaunchKernelEx(&cfg, dsv4_attn_kernel<DSV4_KV_FP8_PACKED>, p);
    if (le != cudaSuccess) {
        cudaGetLastError();
        return DSV4_ERR_CUDA;
    }
    if (sg > 1) {
        cudaLaunchConfig_t ccfg = {};
        cudaLaunchAttribute cattr[1];
        ccfg.gridDim = dim3(static_cast<unsigned>((c.H * kCombineUnits + 255) / 256 * c.T), 1, 1);
        ccfg.blockDim = dim3(256, 1, 1);
        ccfg.dynamicSmemBytes = 0;
        ccfg.stream = st;
        cattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        cattr[0].val.programmaticStreamSerializationAllowed = 1;
        ccfg.attrs = cattr;
        ccfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&ccfg, dsv4_combine_kernel, p) != cudaSuccess) {
            cudaGetLastError();
            return DSV4_ERR_CUDA;
        }
    }
    return DSV4_OK;
}

// Scratch for dsv4_attn_c4_sparse_noalloc: a library-owned device buffer so
// that callers without an allocator can still run split plans.  Host code sees
// only a stand-in for this symbol; the device address is looked up per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DSV4_NOALLOC_SCRATCH_BYTES];
static void* g_noalloc_addr[kMaxDevices];
static std::mutex g_noalloc_mu;

static int noalloc_scratch(void** addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSV4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return DSV4_ERR_CUDA;
        }
        g_noalloc_addr[dev] = ptr;
    }
    *addr = g_noalloc_addr[dev];
    return DSV4_OK;
}

}  // namespace dsv4

using dsv4::Call;

extern "C" {

int dsv4_attn_swa(const void* q, int32_t batch, int32_t num_heads, const int32_t* seq_lens,
                  const int32_t* req_pool_indices, const dsv4_kv_pool* swa, int32_t window,
                  const float* sink, float scale, void* out, float* lse, int32_t num_splits,
                  void* workspace, size_t workspace_bytes, int32_t* debug_rows, void* stream) {
    Call c{q, batch, batch, num_heads, seq_lens, nullptr, req_pool_indices, swa, window, 0, nullptr,
           nullptr, 0, 0, sink, scale, out, lse, num_splits, workspace, workspace_bytes, debug_rows, stream};
    return dsv4::run(c);
}

int dsv4_attn_c4_sparse(const void* q, int32_t batch, int32_t num_heads, const int32_t* seq_lens,
                        const int32_t* req_pool_indices, const dsv4_kv_pool* swa, int32_t window,
                        const dsv4_kv_pool* extra, const int32_t* topk_idx, int32_t topk,
                        const float* sink, float scale, void* out, float* lse, int32_t num_splits,
                        void* workspace, size_t workspace_bytes, int32_t* debug_rows, void* stream) {
    Call c{q, batch, batch, num_heads, seq_lens, nullptr, req_pool_indices, swa, window, 4, extra,
           topk_idx, topk, 0, sink, scale, out, lse, num_splits, workspace, workspace_bytes, debug_rows, stream};
    return dsv4::run(c);
}

int dsv4_attn_c128_dense(const void* q, int32_t batch, int32_t num_heads, const int32_t* seq_lens,
                         const int32_t* req_pool_indices, const dsv4_kv_pool* swa, int32_t window,
                         const dsv4_kv_pool* extra, int32_t max_seq_len, const float* sink, float scale,
                         void* out, float* lse, int32_t num_splits, void* workspace,
                         size_t workspace_bytes, int32_t* debug_rows, void* stream) {
    Call c{q, batch, batch, num_heads, seq_lens, nullptr, req_pool_indices, swa, window, 128, extra,
           nullptr, 0, max_seq_len, sink, scale, out, lse, num_splits, workspace, workspace_bytes,
           debug_rows, stream};
    return dsv4::run(c);
}

int dsv4_attn_verify(const void* q, int32_t num_tokens, int32_t batch, int32_t num_heads,
                     const int32_t* seq_lens, const int32_t* cu_seqlens_q,
                     const int32_t* req_pool_indices, const dsv4_kv_pool* swa, int32_t window,
                     int32_t compress_ratio, const dsv4_kv_pool* extra, const int32_t* topk_idx,
                     int32_t topk, int32_t max_seq_len, const float* sink, float scale, void* out,
                     float* lse, int32_t num_splits, void* workspace, size_t workspace_bytes,
                     int32_t* debug_rows, void* stream) {
    if (!cu_seqlens_q) return DSV4_ERR_INVALID;
    Call c{q, num_tokens, batch, num_heads, seq_lens, cu_seqlens_q, req_pool_indices, swa, window,
           compress_ratio, extra, topk_idx, topk, max_seq_len, sink, scale, out, lse, num_splits,
           workspace, workspace_bytes, debug_rows, stream};
    return dsv4::run(c);
}

int dsv4_attn_plan(int32_t num_tokens, int32_t num_heads, int32_t compress_ratio, int32_t window,
                   int32_t topk, int32_t max_seq_len, int32_t num_splits, int32_t* cluster_splits,
                   int32_t* grid_splits) {
    if (num_tokens < 1 || num_heads < 1 || num_heads > 2 * dsv4::kHG || window < 1 || num_splits < 0 ||
        !cluster_splits || !grid_splits)
        return DSV4_ERR_INVALID;
    if (compress_ratio != 0 && compress_ratio != 4 && compress_ratio != 128) return DSV4_ERR_UNSUPPORTED;
    dsv4::DeviceInfo di;
    int rc = dsv4::device_info(di);
    if (rc) return rc;
    int sc = 1, sg = 1;
    dsv4::make_plan(num_tokens, (num_heads + dsv4::kHG - 1) / dsv4::kHG,
                    dsv4::list_max(compress_ratio, window, topk, max_seq_len), num_splits, di, sc, sg);
    *cluster_splits = sc;
    *grid_splits = sg;
    return DSV4_OK;
}

size_t dsv4_attn_workspace_size(int32_t num_tokens, int32_t num_heads, int32_t compress_ratio,
                                int32_t window, int32_t topk, int32_t max_seq_len, int32_t num_splits) {
    int32_t sc = 1, sg = 1;
    if (dsv4_attn_plan(num_tokens, num_heads, compress_ratio, window, topk, max_seq_len, num_splits, &sc, &sg))
        return 0;
    return dsv4::workspace_bytes_for(num_tokens, num_heads, sc, sg);
}

int dsv4_attn_get_device_error(uint32_t* flags, void* stream) {
    if (!flags) return DSV4_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned v = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return DSV4_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, dsv4::g_dev_error, sizeof(v)) != cudaSuccess) return DSV4_ERR_CUDA;
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(dsv4::g_dev_error, &zero, sizeof(zero)) != cudaSuccess) return DSV4_ERR_CUDA;
    *flags = v;
    return DSV4_OK;
}

int dsv4_attn_c4_sparse_noalloc(const void* q, int32_t batch, int32_t num_heads, const int32_t* seq_lens,
                                const int32_t* req_pool_indices, const dsv4_kv_pool* swa, int32_t window,
                                const dsv4_kv_pool* extra, const int32_t* topk_idx, int32_t topk,
                                const float* sink, float scale, void* out, float* lse, int32_t num_splits,
                                int32_t* debug_rows, void* stream) {
    if (batch < 1 || num_heads < 1 || num_heads > 2 * dsv4::kHG || window < 1 || topk < 1 || num_splits < 0)
        return DSV4_ERR_INVALID;
    // the plan query's own status (a device or argument error) is returned as
    // is, not mistaken for "needs no scratch"
    int32_t sc = 1, sg = 1;
    const int prc = dsv4_attn_plan(batch, num_heads, 4, window, topk, 0, num_splits, &sc, &sg);
    if (prc != DSV4_OK) return prc;
    const size_t need = dsv4::workspace_bytes_for(batch, num_heads, sc, sg);
    if (need > DSV4_NOALLOC_SCRATCH_BYTES) return DSV4_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    if (need > 0) {
        const int rc = dsv4::noalloc_scratch(&scratch);
        if (rc) return rc;
    }
    Call c{q, batch, batch, num_heads, seq_lens, nullptr, req_pool_indices, swa, window, 4, extra,
           topk_idx, topk, 0, sink, scale, out, lse, num_splits, scratch,
           need > 0 ? static_cast<size_t>(DSV4_NOALLOC_SCRATCH_BYTES) : 0, debug_rows, stream};
    return dsv4::run(c);
}

#ifdef DSV4_TRACE
int dsv4_attn_trace_read(void* host, size_t bytes) {
    if (bytes > sizeof(dsv4::g_trace)) bytes = sizeof(dsv4::g_trace);
    if (cudaDeviceSynchronize() != cudaSuccess) return DSV4_ERR_CUDA;
    if (cudaMemcpyFromSymbol(host, dsv4::g_trace, bytes) != cudaSuccess) return DSV4_ERR_CUDA;
    return DSV4_OK;
}
#endif

const char* dsv4_attn_strerror(int status) {
    switch (status) {
        case DSV4_OK: return "ok";
        case DSV4_ERR_INVALID: return "invalid argument";
        case DSV4_ERR_UNSUPPORTED: return "unsupported configuration";
        case DSV4_ERR_WORKSPACE: return "workspace too small";
        case DSV4_ERR_CUDA: return "CUDA error";
        case DSV4_ERR_SCRATCH_LIMIT: return "call needs more scratch than the library's built-in buffer";
        default: return "unknown status";
    }
}

}  // extern "C"
