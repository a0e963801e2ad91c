// dsv4_attn.cu - hybrid sparse MQA attention step (DeepSeek-V4 decode and
// target-verify) for GB300, sm_103a.
//
// What is computed is stated in include/dsv4attn.h.  How:
//
// * One thread-block cluster of 2*Sc CTAs handles one query token and one
//   of Sg slices of its key list; CTA (s, c) of the cluster takes piece s of
//   that slice and half c (dims c*256 .. c*256+255) of every 512-wide row.
//   Splitting the row dimension between the two CTAs of a pair keeps the
//   H x 512 fp32 output accumulator within one SM's tensor memory (256 of
//   its 512 columns) and halves every CTA's gather.
// * Per 64-key tile: four loader warps resolve key slots to pool rows (SWA
//   page table, C4 index list, C128 range) and gather their 512-byte row
//   halves with 16-byte cp.async into a 128-byte-swizzled shared tile; the
//   MMA warp computes the partial scores Q[:,half] K[:,half]^T on tcgen05
//   (heads padded to M=128, fp32 in TMEM); the four softmax warps add the
//   partner CTA's partial scores (exchanged through distributed shared
//   memory), run an online softmax in registers (thread h owns head h) and
//   write bf16 probabilities to shared memory; the MMA warp accumulates
//   O[:,half] += P V[:,half] (V is the same tile, read MN-major).
// * Splits are merged with their log-sum-exp weights, the sink's exp(sink)
//   is added to the denominator once, and the bf16 output is written; merges
//   inside a cluster go through distributed shared memory, merges across
//   clusters through the workspace and the combine kernel.
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

namespace dsv4 {

// ------------------------------------------------------------------ shape
constexpr int kDim = 512;
constexpr int kPageSize = 256;
constexpr int kTileN = 64;           // key rows per tile
constexpr int kStages = 3;           // gather pipeline depth
constexpr int kM = 128;              // MMA M: heads padded to 128
constexpr int kRing = 512;           // resolved key slots held at a time
constexpr int kSoftmaxWarps = 4;
constexpr int kLoadWarps = 4;
constexpr int kMmaWarp = kSoftmaxWarps + kLoadWarps;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr int kMaxClusterSplits = 4;
constexpr float kRescaleLog2 = 8.0f; // lazy rescale threshold (factor 256)
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;       // two 64-column score buffers
constexpr uint32_t kTmemO = 256;     // 256-column output accumulator
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ------------------------------------------------------------------ smem
constexpr int kQBytes = 4 * kM * 128;          // 4 chunks of 64 dims
constexpr int kStageBytes = 4 * kTileN * 128;  // 4 chunks of 64 dims
constexpr int kPBytes = kM * 128;              // 64 keys x 128 heads bf16
constexpr int kXBytes = kM * 64 * 4;           // partner's partial scores
constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + kQBytes;
constexpr int OFF_P = OFF_KV + kStages * kStageBytes;
constexpr int OFF_X = OFF_P + 2 * kPBytes;
constexpr int OFF_RING = OFF_X + kXBytes;      // int32 rows; (m, l) pairs after the loop
constexpr int OFF_MASK = OFF_RING + kRing * 4;
constexpr int OFF_BAR = OFF_MASK + kStages * 8;
enum Bar {
    B_Q_FULL = 0,
    B_KV_FULL = 1,
    B_KV_EMPTY = B_KV_FULL + kStages,
    B_MASK_FULL = B_KV_EMPTY + kStages,
    B_S_FULL = B_MASK_FULL + kStages,
    B_S_FREE = B_S_FULL + 2,
    B_P_FULL = B_S_FREE + 2,
    B_P_FREE = B_P_FULL + 2,
    B_O_FINAL = B_P_FREE + 2,
    B_X_FULL,
    B_X_FREE,
    B_COUNT
};
constexpr int OFF_MISC = OFF_BAR + B_COUNT * 8;
constexpr int OFF_MERGE = OFF_KV;              // 128 x 256 fp32, reuses KV + P
constexpr int kSmemUsed = OFF_MISC + 64;
constexpr int kSmemAlloc = 232448;             // per-block maximum on sm_100/103
static_assert(OFF_MERGE + kM * 1024 <= OFF_X, "merge buffer must fit in the KV and P buffers");
static_assert(kM * 8 <= kRing * 4, "(m, l) pairs must fit in the ring");
static_assert(kSmemUsed <= kSmemAlloc, "shared memory budget");

__device__ unsigned int g_dev_error;

struct Params {
    const __nv_bfloat16* q;
    int T, H, batch;
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
    int chunk;               // key slots per split (multiple of kTileN)
    int csplits, gsplits;
    __nv_bfloat16* out;
    float* lse;
    float* part_o;           // [T, Sg, H, 512] when gsplits > 1
    float2* part_ml;         // [T, Sg, H]
    int* debug_rows;
    int debug_stride;
};

struct TokenInfo {
    int trow, pos, n_swa, n_c, L, slot_begin, slot_end, ntiles;
};

__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, bool cluster_scope, int* abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (cluster_scope ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity)) return true;
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
// Bounded wait on an mbarrier phase.  On time-out it records the error, marks
// the CTA aborted and returns; callers carry on (and keep arriving on the
// barriers others wait for), so every role reaches the end of the kernel.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, int* abort_flag) {
    if (mbar_try(bar, parity)) return true;
    return wait_slow(bar, parity, false, abort_flag);
}
__device__ __forceinline__ bool wait_bar_cluster(uint32_t bar, uint32_t parity, int* abort_flag) {
    if (mbar_try_cluster(bar, parity)) return true;
    return wait_slow(bar, parity, true, abort_flag);
}

// Query token t -> request row, position and key-list extent of this split.
__device__ void token_info(const Params& p, int t, int split, TokenInfo& ti, unsigned& err) {
    int b, pos;
    bool ok = true;
    if (p.cu_seqlens == nullptr) {
        b = t;
        pos = __ldg(p.seq_lens + b) - 1;
    } else {
        int lo = 0, hi = p.batch - 1;        // largest b with cu[b] <= t
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (__ldg(p.cu_seqlens + mid) <= t) lo = mid; else hi = mid - 1;
        }
        b = lo;
        const int c0 = __ldg(p.cu_seqlens + b), c1 = __ldg(p.cu_seqlens + b + 1);
        if (t < c0 || t >= c1) ok = false;
        pos = __ldg(p.seq_lens + b) - (c1 - c0) + (t - c0);
    }
    if (!ok || pos < 0) {
        err |= DSV4_DEV_ERR_POSITION;
        ok = false;
    }
    int trow = p.rpi ? __ldg(p.rpi + b) : b;
    if (ok && (trow < 0 || trow >= p.swa_pt_rows || (p.ratio != 0 && trow >= p.ex_pt_rows))) {
        err |= DSV4_DEV_ERR_REQ_ROW;
        ok = false;
    }
    ti.trow = trow;
    ti.pos = pos;
    if (!ok) {
        ti.n_swa = ti.n_c = ti.L = ti.slot_begin = ti.slot_end = ti.ntiles = 0;
        return;
    }
    ti.n_swa = min(pos + 1, p.window);
    ti.n_c = p.ratio ? (pos + 1) / p.ratio : 0;
    const int n_extra = p.ratio == 4 ? p.topk : (p.ratio == 128 ? ti.n_c : 0);
    ti.L = ti.n_swa + n_extra;
    if (ti.L > p.chunk * p.csplits * p.gsplits) err |= DSV4_DEV_ERR_PLAN;
    ti.slot_begin = split * p.chunk;
    ti.slot_end = min(ti.slot_begin + p.chunk, ti.L);
    ti.ntiles = ti.slot_end > ti.slot_begin ? (ti.slot_end - ti.slot_begin + kTileN - 1) / kTileN : 0;
}

// Key slot -> physical pool row (-1 = skipped).  Window slots are positions
// pos-n_swa+1 .. pos in the SWA pool; extra slots are C4 indices or C128
// compressed-row numbers in the extra pool.
__device__ __forceinline__ int resolve_slot(const Params& p, int t, const TokenInfo& ti, int slot,
                                            unsigned& err) {
    if (slot < ti.n_swa) {
        const int j = ti.pos - ti.n_swa + 1 + slot;
        const int lp = j / kPageSize;
        if (lp >= p.swa_pt_stride) { err |= DSV4_DEV_ERR_SWA_PAGE; return -1; }
        const int page = __ldg(p.swa_pt + (size_t)ti.trow * p.swa_pt_stride + lp);
        if (page < 0 || page >= p.swa_pages) { err |= DSV4_DEV_ERR_SWA_PAGE; return -1; }
        return page * kPageSize + (j % kPageSize);
    }
    const int e = slot - ti.n_swa;
    int idx;
    if (p.ratio == 4) {
        idx = __ldg(p.topk_idx + (size_t)t * p.topk + e);
        if (idx < 0) return -1;
        if (idx >= ti.n_c) { err |= DSV4_DEV_ERR_INDEX_RANGE; return -1; }
    } else {
        idx = e;
    }
    const int lp = idx / kPageSize;
    if (lp >= p.ex_pt_stride) { err |= DSV4_DEV_ERR_EXTRA_PAGE; return -1; }
    const int page = __ldg(p.ex_pt + (size_t)ti.trow * p.ex_pt_stride + lp);
    if (page < 0 || page >= p.ex_pages) { err |= DSV4_DEV_ERR_EXTRA_PAGE; return -1; }
    return page * kPageSize + (idx % kPageSize);
}

// Byte offset of 16-byte piece `piece` (0..7) of the 128-byte line `line` in
// a 1024-byte-aligned 128B-swizzled buffer.
__device__ __forceinline__ uint32_t sw128(uint32_t line, uint32_t piece) {
    return line * 128u + ((piece ^ (line & 7u)) << 4);
}

template <int KV_FORMAT>
__global__ void __launch_bounds__(kThreads, 1) dsv4_attn_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_base);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t half = rank & 1u;
    const uint32_t csplit = rank >> 1;
    const uint32_t peer = rank ^ 1u;
    const int t = blockIdx.y;
    const int gsplit = blockIdx.z;
    const int split = gsplit * p.csplits + static_cast<int>(csplit);

    const uint32_t sQ = base + OFF_Q, sKV = base + OFF_KV, sP = base + OFF_P, sX = base + OFF_X;
    const uint32_t sMerge = base + OFF_MERGE;
    int* ring = reinterpret_cast<int*>(smem + OFF_RING);
    float2* ml = reinterpret_cast<float2*>(smem + OFF_RING);
    uint16_t* mask16 = reinterpret_cast<uint16_t*>(smem + OFF_MASK);
    const uint32_t bars = base + OFF_BAR;
    auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    int* abort_flag = reinterpret_cast<int*>(smem + OFF_MISC + 4);
    TokenInfo* tinfo = reinterpret_cast<TokenInfo*>(smem + OFF_MISC + 16);

    unsigned err = 0;
    if ((base - raw_base) + kSmemUsed > static_cast<uint32_t>(kSmemAlloc)) {
        // Same layout in every CTA of the cluster, so all of them leave here.
        if (threadIdx.x == 0) atomicOr(&g_dev_error, DSV4_DEV_ERR_TIMEOUT);
        return;
    }

    // ------------------------------------------------------------ set-up
    if (tid == 0) {
        mbar_init(bar(B_Q_FULL), kLoadWarps * 32);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(B_KV_FULL + s), kLoadWarps * 32);
            mbar_init(bar(B_KV_EMPTY + s), 1);
            mbar_init(bar(B_MASK_FULL + s), kLoadWarps);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_S_FULL + s), 1);
            mbar_init(bar(B_S_FREE + s), kSoftmaxWarps * 32);
            mbar_init(bar(B_P_FULL + s), kSoftmaxWarps * 32);
            mbar_init(bar(B_P_FREE + s), 1);
        }
        mbar_init(bar(B_O_FINAL), 1);
        mbar_init(bar(B_X_FULL), kSoftmaxWarps * 32);
        mbar_init(bar(B_X_FREE), kSoftmaxWarps * 32);
        fence_mbar_init_cluster();
        *abort_flag = 0;
        TokenInfo ti;
        token_info(p, t, split, ti, err);
        *tinfo = ti;
    }
    if (warp == kMmaWarp) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();   // every CTA's barriers are initialised before any remote arrival
    const uint32_t tmem = *tmem_slot;
    const TokenInfo ti = *tinfo;
    const int ntiles = ti.ntiles;

    if (warp >= kSoftmaxWarps && warp < kMmaWarp) {
        // ============================================================ loader
        const int lt = tid - kSoftmaxWarps * 32;
        const int lw = lt >> 5;
        // debug dump of this split's slots (pair half 0 only)
        if (p.debug_rows != nullptr && half == 0) {
            const int d0 = split * p.chunk;
            const int d1 = min(d0 + p.chunk, p.debug_stride);
            for (int s = d0 + lt; s < d1; s += kLoadWarps * 32) {
                const int row = (s < ti.L) ? resolve_slot(p, t, ti, s, err) : -1;
                p.debug_rows[(size_t)t * p.debug_stride + s] = row;
            }
        }
        // query rows of this half: 128 heads x 512 bytes, zero-filled past H
        {
            const uint8_t* qb = reinterpret_cast<const uint8_t*>(p.q) + ((size_t)t * p.H) * 1024 + half * 512;
            for (int k = lt; k < kM * 32; k += kLoadWarps * 32) {
                const int h = k >> 5, piece = k & 31;
                const uint32_t dst = sQ + (piece >> 3) * (kM * 128) + sw128(h, piece & 7);
                const bool on = h < p.H && ntiles > 0;
                cp_async_16(dst, on ? qb + (size_t)h * 1024 + piece * 16 : qb, on ? 16u : 0u);
            }
            cp_async_arrive_noinc(bar(B_Q_FULL));
        }
        int ring_base = -1;
        for (int i = 0; i < ntiles; ++i) {
            const int stage = i % kStages;
            if (i >= kStages) {
                wait_bar(bar(B_KV_EMPTY + stage), ((i / kStages) - 1) & 1, abort_flag);
                fence_proxy_async();
            }
            const int slot0 = ti.slot_begin + i * kTileN;
            if (ring_base < 0 || slot0 + kTileN > ring_base + kRing) {
                named_barrier_sync(1, kLoadWarps * 32);
                ring_base = slot0;
                const int lim = min(ring_base + kRing, ti.slot_end);
#pragma unroll 4
                for (int s = ring_base + lt; s < ring_base + kRing; s += kLoadWarps * 32)
                    ring[s - ring_base] = (s < lim) ? resolve_slot(p, t, ti, s, err) : -1;
                named_barrier_sync(1, kLoadWarps * 32);
            }
            // validity mask of this tile, 16 slots per loader warp
            {
                const int r = lw * 16 + (lane & 15);
                const int slot = slot0 + r;
                const bool valid = slot < ti.slot_end && ring[slot - ring_base] >= 0;
                const unsigned bal = __ballot_sync(0xffffffffu, lane < 16 && valid);
                if (lane == 0) mask16[stage * 4 + lw] = static_cast<uint16_t>(bal & 0xffffu);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_MASK_FULL + stage));
            }
            const uint32_t dst_stage = sKV + stage * kStageBytes;
#pragma unroll 4
            for (int k = 0; k < 16; ++k) {
                const int r = lw * 16 + k;
                const int slot = slot0 + r;
                const int row = slot < ti.slot_end ? ring[slot - ring_base] : -1;
                const bool from_swa = slot < ti.n_swa;
                const uint8_t* pool = from_swa ? p.swa_rows : p.ex_rows;
                const int rb = from_swa ? p.swa_row_bytes : p.ex_row_bytes;
                const uint8_t* src = row >= 0 ? pool + (size_t)row * rb + half * 512 + lane * 16 : p.swa_rows;
                const uint32_t dst = dst_stage + (lane >> 3) * (kTileN * 128) + sw128(r, lane & 7);
                cp_async_16(dst, src, row >= 0 ? 16u : 0u);
            }
            cp_async_arrive_noinc(bar(B_KV_FULL + stage));
        }
        cp_async_wait_all();
    } else if (warp == kMmaWarp) {
        // ============================================================ MMA issuer
        if (lane == 0 && ntiles > 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(kM, kTileN, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(kM, 256, false, true);
            wait_bar(bar(B_Q_FULL), 0, abort_flag);
            fence_proxy_async();
            tc_fence_after();
            auto issue_pv = [&](int j) {
                const int pb = j & 1;
                const int stage = j % kStages;
                wait_bar(bar(B_P_FULL + pb), (j >> 1) & 1, abort_flag);
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < kTileN / 16; ++k) {
                    const uint64_t a = smem_desc_sw128(sP + pb * kPBytes + k * 32, 16, 1024);
                    const uint64_t b = smem_desc_sw128(sKV + stage * kStageBytes + k * 2048, kTileN * 128, 1024);
                    mma_bf16_ss(tmem + kTmemO, a, b, idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(bar(B_P_FREE + pb));
                mma_commit(bar(B_KV_EMPTY + stage));
            };
            for (int i = 0; i < ntiles; ++i) {
                const int stage = i % kStages;
                const int sb = i & 1;
                wait_bar(bar(B_KV_FULL + stage), (i / kStages) & 1, abort_flag);
                fence_proxy_async();
                if (i >= 2) wait_bar(bar(B_S_FREE + sb), ((i - 2) >> 1) & 1, abort_flag);
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const uint64_t a = smem_desc_sw128(sQ + (k >> 2) * (kM * 128) + (k & 3) * 32, 16, 1024);
                    const uint64_t b = smem_desc_sw128(sKV + stage * kStageBytes + (k >> 2) * (kTileN * 128) + (k & 3) * 32, 16, 1024);
                    mma_bf16_ss(tmem + kTmemS + sb * kTileN, a, b, idesc_qk, k > 0 ? 1u : 0u);
                }
                mma_commit(bar(B_S_FULL + sb));
                if (i >= 1) issue_pv(i - 1);
            }
            issue_pv(ntiles - 1);
            mma_commit(bar(B_O_FINAL));
        }
        __syncwarp();
    } else {
        // ============================================================ softmax
        const int h = tid;   // head row == TMEM lane
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const uint32_t peer_x = mapa(sX, peer);
        const uint32_t peer_x_full = mapa(bar(B_X_FULL), peer);
        const uint32_t peer_x_free = mapa(bar(B_X_FREE), peer);
        const bool live = h < p.H;
        float m_run = -INFINITY, l_run = 0.f;
        for (int i = 0; i < ntiles; ++i) {
            const int sb = i & 1;
            const int stage = i % kStages;
            float s[64];
            wait_bar(bar(B_S_FULL + sb), (i >> 1) & 1, abort_flag);
            tc_fence_after();
            {
                float a[32], b[32];
                tmem_ld32(lane_addr + kTmemS + sb * kTileN, a);
                tmem_ld32(lane_addr + kTmemS + sb * kTileN + 32, b);
#pragma unroll
                for (int j = 0; j < 32; ++j) { s[j] = a[j]; s[32 + j] = b[j]; }
            }
            tc_fence_before();
            mbar_arrive(bar(B_S_FREE + sb));
            // exchange partial scores with the partner CTA (other row half)
            if (i >= 1) wait_bar_cluster(bar(B_X_FREE), (i - 1) & 1, abort_flag);
            if (live) {
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    st_cluster_v4(peer_x + h * 256 + ((q ^ (h & 15)) << 4), s[4 * q], s[4 * q + 1],
                                  s[4 * q + 2], s[4 * q + 3]);
            }
            mbar_arrive_cluster(peer_x_full);
            wait_bar_cluster(bar(B_X_FULL), i & 1, abort_flag);
            if (live) {
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const float4 x = ld_shared_v4(sX + h * 256 + ((q ^ (h & 15)) << 4));
                    s[4 * q] += x.x; s[4 * q + 1] += x.y; s[4 * q + 2] += x.z; s[4 * q + 3] += x.w;
                }
            }
            mbar_arrive_cluster(peer_x_free);
            // mask, scale to log2 units, online max with lazy rescaling
            wait_bar(bar(B_MASK_FULL + stage), (i / kStages) & 1, abort_flag);
            const uint64_t mask = *reinterpret_cast<volatile uint64_t*>(smem + OFF_MASK + stage * 8);
            float mt = -INFINITY;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                s[j] = ((mask >> j) & 1ull) ? s[j] * p.scale_log2 : -INFINITY;
                mt = fmaxf(mt, s[j]);
            }
            const float m_new = fmaxf(m_run, mt);
            const bool rescale = m_new > m_run + kRescaleLog2;
            float alpha = 1.f;
            if (rescale) {
                alpha = fast_exp2(m_run - m_new);
                m_run = m_new;
            }
            uint32_t pk[32];
            float lsum = 0.f;
            const bool any = m_run != -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float p0 = any ? fast_exp2(s[2 * j] - m_run) : 0.f;
                const float p1 = any ? fast_exp2(s[2 * j + 1] - m_run) : 0.f;
                __nv_bfloat162 v = __floats2bfloat162_rn(p0, p1);
                lsum += __low2float(v) + __high2float(v);
                pk[j] = *reinterpret_cast<uint32_t*>(&v);
            }
            l_run = l_run * alpha + lsum;
            if (rescale && i > 0) {
                wait_bar(bar(B_P_FREE + ((i - 1) & 1)), ((i - 1) >> 1) & 1, abort_flag);
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {
                    float o[32];
                    tmem_ld32(lane_addr + kTmemO + c * 32, o);
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] *= alpha;
                    tmem_st32(lane_addr + kTmemO + c * 32, o);
                }
            }
            if (i >= 2) wait_bar(bar(B_P_FREE + sb), ((i - 2) >> 1) & 1, abort_flag);
            const uint32_t prow = sP + sb * kPBytes;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                st_shared_v4(prow + sw128(h, q), pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(bar(B_P_FULL + sb));
        }
        if (ntiles > 0) {
            wait_bar(bar(B_O_FINAL), 0, abort_flag);
            tc_fence_after();
            fence_proxy_async();
        }
        ml[h] = make_float2(ntiles > 0 ? m_run : -INFINITY, ntiles > 0 ? l_run : 0.f);
    }

    // ------------------------------------------------------------ merge
    cluster_sync();   // A: every split of the cluster finished its key loop
    const bool final_out = p.gsplits == 1;
    if (warp < kSoftmaxWarps) {
        const int h = tid;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        if (h < p.H) {
            float M = -INFINITY;
            float2 mls[kMaxClusterSplits];
            for (int s = 0; s < p.csplits; ++s) {
                mls[s] = ld_cluster_v2(mapa(base + OFF_RING + h * 8, 2 * s + half));
                M = fmaxf(M, mls[s].x);
            }
            const float sk = __ldg(p.sink + h) * kLog2e;
            if (final_out) M = fmaxf(M, sk);
            float Lsum = 0.f;
            if (M != -INFINITY) {
                for (int s = 0; s < p.csplits; ++s)
                    if (mls[s].x != -INFINITY) Lsum += mls[s].y * exp2f(mls[s].x - M);
                if (final_out && sk != -INFINITY) Lsum += exp2f(sk - M);
            }
            const float mine = mls[csplit].x;
            const float alpha = (ntiles > 0 && Lsum > 0.f && mine != -INFINITY) ? exp2f(mine - M) / Lsum : 0.f;
            for (int c = 0; c < 8; ++c) {
                float o[32];
                if (ntiles > 0) {
                    tmem_ld32(lane_addr + kTmemO + c * 32, o);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = 0.f;
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    st_shared_v4(sMerge + h * 1024 + (((c * 8 + q) ^ (h & 7)) << 4),
                                 __float_as_uint(o[4 * q] * alpha), __float_as_uint(o[4 * q + 1] * alpha),
                                 __float_as_uint(o[4 * q + 2] * alpha), __float_as_uint(o[4 * q + 3] * alpha));
            }
            if (rank == 0) {
                if (final_out) {
                    if (p.lse) p.lse[(size_t)t * p.H + h] = (Lsum > 0.f ? M + log2f(Lsum) : -INFINITY) * kLn2;
                } else {
                    p.part_ml[((size_t)t * p.gsplits + gsplit) * p.H + h] = make_float2(M, Lsum);
                }
            }
        }
    }
    tc_fence_before();
    cluster_sync();   // B: every CTA's scaled accumulator is in its merge buffer
    tc_fence_after();
    {
        // CTA (csplit, half) writes 8-column units [u0, u1) of its half.
        const int u0 = (static_cast<int>(csplit) * 32) / p.csplits;
        const int u1 = ((static_cast<int>(csplit) + 1) * 32) / p.csplits;
        const int nu = u1 - u0;
        const int items = p.H * nu;
        for (int it = tid; it < items; it += kThreads) {
            const int h = it / nu;
            const int u = u0 + it % nu;
            float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            for (int s = 0; s < p.csplits; ++s) {
                const uint32_t rb = mapa(sMerge + h * 1024, 2 * s + half);
                const float4 a = ld_cluster_v4(rb + (((2 * u) ^ (h & 7)) << 4));
                const float4 b = ld_cluster_v4(rb + (((2 * u + 1) ^ (h & 7)) << 4));
                acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
                acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
            }
            const size_t col = (size_t)half * 256 + u * 8;
            if (final_out) {
                uint4 v;
                v.x = pack_bf16x2(acc[0], acc[1]);
                v.y = pack_bf16x2(acc[2], acc[3]);
                v.z = pack_bf16x2(acc[4], acc[5]);
                v.w = pack_bf16x2(acc[6], acc[7]);
                *reinterpret_cast<uint4*>(p.out + ((size_t)t * p.H + h) * kDim + col) = v;
            } else {
                float* dst = p.part_o + (((size_t)t * p.gsplits + gsplit) * p.H + h) * kDim + col;
                *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
            }
        }
    }
    if (err) atomicOr(&g_dev_error, err);
    cluster_sync();   // C: peers are done reading this CTA's shared memory
    if (warp == kMmaWarp) {
        if (*reinterpret_cast<volatile int*>(abort_flag)) {
            // a wait gave up: give in-flight tensor-core work time to drain
            for (int k = 0; k < 1000; ++k) __nanosleep(10000);
        }
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Merges Sg cluster results of each (token, head): the weights are
// L_g * exp(M_g - M) with M the largest of the M_g and the sink; the sink
// adds exp(sink - M) to the denominator and nothing to the numerator.
__global__ void __launch_bounds__(256) dsv4_combine_kernel(const __grid_constant__ Params p) {
    const int t = blockIdx.x;
    for (int it = threadIdx.x; it < p.H * 64; it += blockDim.x) {
        const int h = it >> 6;
        const int u = it & 63;
        const float sk = __ldg(p.sink + h) * kLog2e;
        const float2* mlp = p.part_ml + (size_t)t * p.gsplits * p.H + h;
        float M = sk;
        for (int g = 0; g < p.gsplits; ++g) M = fmaxf(M, mlp[(size_t)g * p.H].x);
        float L = 0.f;
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (M != -INFINITY) {
            if (sk != -INFINITY) L = exp2f(sk - M);
            for (int g = 0; g < p.gsplits; ++g) {
                const float2 v = mlp[(size_t)g * p.H];
                if (v.x == -INFINITY || v.y <= 0.f) continue;
                const float w = v.y * exp2f(v.x - M);
                L += w;
                const float* src = p.part_o + (((size_t)t * p.gsplits + g) * p.H + h) * kDim + u * 8;
                const float4 a = *reinterpret_cast<const float4*>(src);
                const float4 b = *reinterpret_cast<const float4*>(src + 4);
                acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
                acc[4] += w * b.x; acc[5] += w * b.y; acc[6] += w * b.z; acc[7] += w * b.w;
            }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        uint4 v;
        v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        v.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
        v.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
        *reinterpret_cast<uint4*>(p.out + ((size_t)t * p.H + h) * kDim + u * 8) = v;
        if (u == 0 && p.lse) p.lse[(size_t)t * p.H + h] = (L > 0.f ? M + log2f(L) : -INFINITY) * kLn2;
    }
}

// ------------------------------------------------------------------ host
struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int max_clusters[kMaxClusterSplits + 1] = {0, 0, 0, 0, 0};
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
        for (int sc = 1; sc <= kMaxClusterSplits; ++sc) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            cfg.gridDim = dim3(2 * sc, 1, 1);
            cfg.blockDim = dim3(kThreads, 1, 1);
            cfg.dynamicSmemBytes = kSmemAlloc;
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2 * sc;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
                cudaGetLastError();
                n = di.sms / (2 * sc) * 3 / 4;
            }
            di.max_clusters[sc] = n > 0 ? n : 1;
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

// Split plan: cluster splits sc (merged on chip) x grid splits sg (merged by
// the combine kernel), chosen to minimise waves x tiles per split.
static int make_plan(int T, int lmax, int num_splits, const DeviceInfo& di, int& sc, int& sg) {
    const int tiles_total = (lmax + kTileN - 1) / kTileN;
    if (num_splits > 0) {
        sc = 1;
        for (int c = kMaxClusterSplits; c >= 1; --c)
            if (num_splits % c == 0) { sc = c; break; }
        sg = num_splits / sc;
        return DSV4_OK;
    }
    double best = 1e30;
    sc = 1;
    sg = 1;
    for (int c = 1; c <= kMaxClusterSplits; ++c) {
        for (int g = 1; g <= 64; ++g) {
            const int s = c * g;
            if (s > 1 && s > tiles_total) break;
            const long long clusters = (long long)T * g;
            if (g > 1 && clusters > 4LL * di.max_clusters[c]) break;
            const long long waves = (clusters + di.max_clusters[c] - 1) / di.max_clusters[c];
            const int tiles = (tiles_total + s - 1) / s;
            const double cost = (double)waves * (tiles + 1) + (g > 1 ? 3.0 : 0.0) + 0.25 * (c - 1);
            if (cost < best - 1e-9) { best = cost; sc = c; sg = g; }
        }
    }
    return DSV4_OK;
}

static int check_pool(const dsv4_kv_pool* pool) {
    if (!pool || !pool->rows || !pool->page_table) return DSV4_ERR_INVALID;
    if (pool->page_size != kPageSize) return DSV4_ERR_UNSUPPORTED;
    if (pool->format == DSV4_KV_BF16) {
        if (pool->row_bytes != 1024) return DSV4_ERR_UNSUPPORTED;
    } else {
        return DSV4_ERR_UNSUPPORTED;
    }
    if (pool->num_pages < 1 || pool->num_pages * kPageSize >= (1LL << 31)) return DSV4_ERR_INVALID;
    if (pool->page_table_rows < 1 || pool->page_table_stride < 1) return DSV4_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(pool->rows) % 16) return DSV4_ERR_INVALID;
    return DSV4_OK;
}

static size_t workspace_bytes_for(int T, int H, int sg) {
    if (sg <= 1) return 0;
    return (size_t)T * sg * H * kDim * sizeof(float) + (size_t)T * sg * H * sizeof(float2) + 256;
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
    if (c.T < 1 || c.batch < 1 || c.H < 1 || c.H > kM || c.window < 1) return DSV4_ERR_INVALID;
    if (!std::isfinite(c.scale)) return DSV4_ERR_INVALID;
    if (c.T > 65535) return DSV4_ERR_UNSUPPORTED;
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
    int sc = 1, sg = 1;
    make_plan(c.T, lmax, c.num_splits, di, sc, sg);
    const int splits = sc * sg;
    const int chunk = ((lmax + splits - 1) / splits + kTileN - 1) / kTileN * kTileN;
    if (c.T * (long long)sg > 65535) return DSV4_ERR_UNSUPPORTED;
    const size_t need = workspace_bytes_for(c.T, c.H, sg);
    if (need > 0 && (!c.ws || c.ws_bytes < need)) return DSV4_ERR_WORKSPACE;

    Params p;
    std::memset(&p, 0, sizeof(p));
    p.q = static_cast<const __nv_bfloat16*>(c.q);
    p.T = c.T;
    p.H = c.H;
    p.batch = c.batch;
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
    p.chunk = chunk;
    p.csplits = sc;
    p.gsplits = sg;
    p.out = static_cast<__nv_bfloat16*>(c.out);
    p.lse = c.lse;
    if (sg > 1) {
        uintptr_t w = (reinterpret_cast<uintptr_t>(c.ws) + 255) & ~uintptr_t(255);
        p.part_o = reinterpret_cast<float*>(w);
        p.part_ml = reinterpret_cast<float2*>(w + (size_t)c.T * sg * c.H * kDim * sizeof(float));
    }
    p.debug_rows = c.debug_rows;
    p.debug_stride = lmax;

    cudaStream_t st = static_cast<cudaStream_t>(c.stream);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(2 * sc, c.T, sg);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemAlloc;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2 * sc;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, dsv4_attn_kernel<DSV4_KV_BF16>, p) != cudaSuccess) {
        cudaGetLastError();
        return DSV4_ERR_CUDA;
    }
    if (sg > 1) {
        dsv4_combine_kernel<<<c.T, 256, 0, st>>>(p);
        if (cudaGetLastError() != cudaSuccess) return DSV4_ERR_CUDA;
    }
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
    if (num_tokens < 1 || num_heads < 1 || num_heads > dsv4::kM || window < 1 || num_splits < 0 ||
        !cluster_splits || !grid_splits)
        return DSV4_ERR_INVALID;
    if (compress_ratio != 0 && compress_ratio != 4 && compress_ratio != 128) return DSV4_ERR_UNSUPPORTED;
    dsv4::DeviceInfo di;
    int rc = dsv4::device_info(di);
    if (rc) return rc;
    int sc = 1, sg = 1;
    dsv4::make_plan(num_tokens, dsv4::list_max(compress_ratio, window, topk, max_seq_len), num_splits, di, sc, sg);
    *cluster_splits = sc;
    *grid_splits = sg;
    return DSV4_OK;
}

size_t dsv4_attn_workspace_size(int32_t num_tokens, int32_t num_heads, int32_t compress_ratio,
                                int32_t window, int32_t topk, int32_t max_seq_len, int32_t num_splits) {
    int32_t sc = 1, sg = 1;
    if (dsv4_attn_plan(num_tokens, num_heads, compress_ratio, window, topk, max_seq_len, num_splits, &sc, &sg))
        return 0;
    return dsv4::workspace_bytes_for(num_tokens, num_heads, sg);
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

const char* dsv4_attn_strerror(int status) {
    switch (status) {
        case DSV4_OK: return "ok";
        case DSV4_ERR_INVALID: return "invalid argument";
        case DSV4_ERR_UNSUPPORTED: return "unsupported configuration";
        case DSV4_ERR_WORKSPACE: return "workspace too small";
        case DSV4_ERR_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}

}  // extern "C"
