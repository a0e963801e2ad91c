// dsv4_topk.cu - top-k index selection for the C4 index lists (the k best
// indexer scores of every query token).  What is computed is stated in
// include/dsv4topk.h.
//
// Sources (page title, section): "DeepSeek-V4 and SGLang Day-0" - kernel
// list (the indexer keeps the top 512 of 256K candidates at 1M context with
// a radix select over a cluster of thread blocks instead of a global sort);
// "DeepSeek-V4 Attention: Query, Cache Write and History Addressing" -
// section 5 (the top-k indices limit the C4 rows a token reads).
//
// How: a score's order-preserving 32-bit key (its fp32 bits with the sign
// folded) makes "higher score" plain integer order.  One thread-block
// cluster takes one row; CTA r of its C CTAs holds chunk r of the row on
// chip (read once from HBM, coalesced), and the cluster finds the row's k-th
// largest key by an exact radix select over digits of 12, 10 and 10 bits
// from the top.  For each digit every CTA counts its keys into its own
// shared histogram and adds the occupied bins into the totals of every CTA
// of the cluster (distributed shared memory), so each CTA finds the bin
// holding the k-th key by itself after one cluster barrier.  The select
// stops as soon as that bin holds exactly the keys still needed.  After the
// first digit the keys of its bin (few) go to a shared list that the later
// digits are counted over, and a last pass marks the keys above the
// threshold T and those equal to it; both passes look only inside groups of
// four keys whose largest reaches the bound.  Keys above T are selected,
// keys equal to it go to the lowest indices; per-warp counts, exchanged once
// across the cluster, and a bitmap of each warp's positions place every
// selected index at its rank in the row's ascending order, so nothing is
// merged afterwards.
//
// Work per key is what bounds a long row (65536 keys per SM), so the per-key
// passes are few and short: the count of the first digit, then passes that
// look only inside groups of four whose largest key reaches the bound.
// Warp-wide instructions are counted too: all 32 warps issue them at once.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "dsv4attn.h"
#include "dsv4topk.h"
#include "dsv4_device.cuh"
#include "dsv4_internal.h"

namespace dsv4 {
namespace {

constexpr int kTkThreads = 1024;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kMaxClusterCtas = 8;                        // portable cluster size
constexpr int kMaxKeys = 64;                              // scores per thread, longest chunk
constexpr int kMaxLength = kMaxClusterCtas * kTkThreads * kMaxKeys;   // 524288
constexpr int kMaxK = 1024;
constexpr int kBins1 = 4096;                              // first digit: 12 bits
constexpr int kBins2 = 1024;                              // second and third digits: 10 bits
constexpr int kListCap = 8192;                            // threshold-bin keys a CTA lists
constexpr int kAllEqual = 0x7fffffff;                     // every key equal to T is selected

struct TopkParams {
    const float* scores;
    long long stride;          // floats between rows
    const int* lengths;
    int max_len;
    int k;
    int* out;                  // [rows][k]
    unsigned int* err;
};

// Per digit: this CTA's own counts (hist) and the cluster's totals (tot),
// which every CTA of the cluster adds its occupied bins into.
struct SelectSmem {
    int hist1[kBins1];
    int hist2[kBins2];
    int hist3[kBins2];
    int tot1[kBins1];
    int tot2[kBins2];
    int tot3[kBins2];
    uint32_t list[kListCap];
    int cta_gt[kMaxClusterCtas];        // every CTA's count of keys above T
    int cta_eq[kMaxClusterCtas];        // every CTA's count of keys equal to T
    int warp_gt[kTkWarps];
    int warp_eq[kTkWarps];
    int ctrl[3];                        // threshold bin, entries above it, entries in it
    int nlist;
    int wsum[kTkWarps];
};

// The raw floats of the shared-memory key groups follow the select state:
// their 16-byte copies and loads need it to end on a 16-byte boundary, and
// the first digit's counts are read as int4.
static_assert(sizeof(SelectSmem) % 16 == 0, "key groups follow the select state on a 16-byte boundary");
static_assert(offsetof(SelectSmem, hist1) % 16 == 0 && offsetof(SelectSmem, tot1) % 16 == 0,
              "first-digit counts are read as int4");

__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return u ^ ((static_cast<uint32_t>(static_cast<int32_t>(u) >> 31)) | 0x80000000u);
}
// The float whose order key is k.
__device__ __forceinline__ float key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}
__device__ __forceinline__ void red_cluster_add(uint32_t addr, int v) {
    asm volatile("red.shared::cluster.add.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_s32(uint32_t addr, int v) {
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// After this CTA has counted a digit into `hist` (BPT * kTkThreads bins,
// thread t owning bins BPT*t .. BPT*t + BPT - 1): add its occupied bins into
// `tot` of every CTA of the cluster, wait for the other CTAs' counts, and
// find the bin holding the k_rem-th largest key of the row, leaving {bin,
// entries above it, entries in it} in ctrl.
template <int BPT>
__device__ void cluster_find_bin(const int* hist, int* tot, int k_rem, int C, SelectSmem& sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int c[BPT];
    if constexpr (BPT == 4) {
        const int4 v = *reinterpret_cast<const int4*>(hist + 4 * tid);
        c[0] = v.x;
        c[1] = v.y;
        c[2] = v.z;
        c[3] = v.w;
    } else {
        c[0] = hist[tid];
    }
    const uint32_t a = smem_u32(tot + BPT * tid);
#pragma unroll
    for (int b = 0; b < BPT; ++b)
        if (c[b])
            for (int q = 0; q < C; ++q) red_cluster_add(mapa(a + 4u * b, q), c[b]);
    cluster_sync();                                        // every CTA's counts are in tot
    if constexpr (BPT == 4) {
        const int4 v = *reinterpret_cast<const int4*>(tot + 4 * tid);
        c[0] = v.x;
        c[1] = v.y;
        c[2] = v.z;
        c[3] = v.w;
    } else {
        c[0] = tot[tid];
    }
    int mine = 0;
#pragma unroll
    for (int b = 0; b < BPT; ++b) mine += c[b];
    int suf = mine;                                        // this lane's bins and every higher lane's
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, suf, off);
        if (lane + off < 32) suf += y;
    }
    if (lane == 0) sm.wsum[warp] = suf;
    __syncthreads();
    // entries in the bins of the warps above: lane l holds warp l's total
    int ws = sm.wsum[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, ws, off);
        if (lane + off < 32) ws += y;
    }
    const int above_warps = __shfl_sync(0xffffffffu, ws, (warp + 1) & 31);
    int ab = suf - mine + (warp + 1 < kTkWarps ? above_warps : 0);   // entries in bins above this thread's
#pragma unroll
    for (int b = BPT - 1; b >= 0; --b) {
        if (ab < k_rem && ab + c[b] >= k_rem) {
            sm.ctrl[0] = BPT * tid + b;
            sm.ctrl[1] = ab;
            sm.ctrl[2] = c[b];
        }
        ab += c[b];
    }
    __syncthreads();
}

// The KPT scores one thread holds, in groups of four: group i of lane l in
// warp w is scores wbase + 128 i + 4 l + 0..3 of the row (wbase: the warp's
// first), so a warp reads 512 contiguous bytes per group.  Up to 8 groups
// live as keys in registers; the rest (KPT = 64) as raw floats in shared
// memory, group i of thread t at sk[(i - 8) * kTkThreads + t].  Groups
// i < ng hold scores of the row; a key past the row's end is 0, below every
// finite score's key.
template <int KPT>
struct Keys {
    static constexpr int G = KPT / 4;
    static constexpr int GR = G > 8 ? 8 : G;               // groups in registers
    static constexpr int W = (KPT + 31) / 32;              // words of a per-key bit mask
    uint32_t reg[4 * GR];
    const float4* sk;
    int ng;
    // f(i, v): v the four keys of group i, for every group i < ng
    template <class F>
    __device__ __forceinline__ void for_each_group(F&& f) const {
#pragma unroll
        for (int i = 0; i < G; ++i) {
            if (i < ng) {
                uint32_t v[4];
                if (i < GR) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) v[c] = reg[4 * i + c];
                } else {
                    const float4 f4 = sk[(i - GR) * kTkThreads];
                    v[0] = order_key(f4.x);
                    v[1] = order_key(f4.y);
                    v[2] = order_key(f4.z);
                    v[3] = order_key(f4.w);
                }
                f(i, v);
            }
        }
    }
    // f(i, v) for the groups i < ng whose largest key may reach t (a
    // superset of those that do: shared-memory groups are screened on their
    // raw floats against t_f, the float of key t, or let through when that
    // is not a number)
    template <class F>
    __device__ __forceinline__ void for_each_group_reaching(uint32_t t, float t_f, F&& f) const {
#pragma unroll
        for (int i = 0; i < G; ++i) {
            if (i < ng) {
                uint32_t v[4];
                if (i < GR) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) v[c] = reg[4 * i + c];
                    if (max(max(v[0], v[1]), max(v[2], v[3])) >= t) f(i, v);
                } else {
                    const float4 f4 = sk[(i - GR) * kTkThreads];
                    if (!(fmaxf(fmaxf(f4.x, f4.y), fmaxf(f4.z, f4.w)) < t_f)) {
                        v[0] = order_key(f4.x);
                        v[1] = order_key(f4.y);
                        v[2] = order_key(f4.z);
                        v[3] = order_key(f4.w);
                        f(i, v);
                    }
                }
            }
        }
    }
    __device__ __forceinline__ static uint32_t nib(const uint32_t (&m)[W], int i) {
        return (m[(4 * i) >> 5] >> ((4 * i) & 31)) & 0xfu;
    }
    __device__ __forceinline__ static void set_nib(uint32_t (&m)[W], int i, uint32_t x) {
        m[(4 * i) >> 5] |= x << ((4 * i) & 31);
    }
};

template <int KPT>
__global__ void __launch_bounds__(kTkThreads, 1) dsv4_topk_kernel(const __grid_constant__ TopkParams p) {
    using K = Keys<KPT>;
    constexpr int kCh = kTkThreads * KPT;                  // scores per CTA
    extern __shared__ __align__(16) uint8_t tk_smem[];
    SelectSmem& sm = *reinterpret_cast<SelectSmem*>(tk_smem);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int C = static_cast<int>(gridDim.x);             // CTAs per row = the cluster
    const int rank = static_cast<int>(cluster_ctarank());
    const int r = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k = p.k;
    int n = __ldg(p.lengths + r);
    if (n < 0 || n > p.max_len) {
        if (rank == 0 && tid == 0) atomicOr(p.err, DSV4_DEV_ERR_TOPK_LENGTH);
        n = n < 0 ? 0 : p.max_len;
    }
    int* out = p.out + (size_t)r * k;
    if (n <= k) {                                          // every candidate; the cluster leaves
        if (rank == 0)
            for (int i = tid; i < k; i += kTkThreads) out[i] = i < n ? i : -1;
        return;
    }
    // ---- this thread's scores: key (i, c) is row index wbase + 128 i + 4 lane + c
    const int wbase = rank * kCh + warp * 32 * KPT;
    const int lim = n - wbase - 4 * lane;                  // key (i, c) exists iff 128 i + c < lim
    K key;
    key.sk = reinterpret_cast<const float4*>(tk_smem + sizeof(SelectSmem)) + tid;
    key.ng = lim <= 0 ? 0 : min(K::G, (lim + 127) / 128);
    // a group's float4 never passes the row's stride (a multiple of 4 >= n)
    const float4* src = reinterpret_cast<const float4*>(p.scores + (size_t)r * p.stride + wbase) + lane;
    if constexpr (K::G > K::GR) {
        // the shared-memory groups first, as asynchronous copies that stay
        // in flight with the register loads below
        const uint32_t dst = smem_u32(key.sk);
#pragma unroll
        for (int i = K::GR; i < K::G; ++i)
            if (i < key.ng) cp_async_16(dst + 16u * (i - K::GR) * kTkThreads, src + 32 * i, 16u);
    }
#pragma unroll
    for (int i = 0; i < K::GR; ++i) {
        uint32_t v[4] = {0u, 0u, 0u, 0u};
        if (i < key.ng) {
            const float4 f = __ldcs(src + 32 * i);
            v[0] = order_key(f.x);
            v[1] = order_key(f.y);
            v[2] = order_key(f.z);
            v[3] = order_key(f.w);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (128 * i + c >= lim) v[c] = 0u;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) key.reg[4 * i + c] = v[c];
    }
    {
        int* z = sm.hist1;                                 // hist1 .. tot3 are contiguous
        for (int i = tid; i < 2 * (kBins1 + 2 * kBins2); i += kTkThreads) z[i] = 0;
        if (tid == 0) sm.nlist = 0;
    }
    // the other CTAs add into this CTA's totals only once it has cleared them
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    if constexpr (K::G > K::GR) {
        cp_async_wait_all();                               // this thread's own groups have landed
        const int last = key.ng - 1;                       // a group cut by the row's end
        if (last >= K::GR && 128 * last + 4 > lim) {
            float* f = reinterpret_cast<float*>(tk_smem + sizeof(SelectSmem)) +
                       4 * ((last - K::GR) * kTkThreads + tid);
            for (int c = 0; c < 4; ++c)
                if (128 * last + c >= lim) f[c] = __uint_as_float(0xffffffffu);   // key 0
        }
    }
    __syncthreads();

    // ---- first digit, bits 31..20, over every key
    key.for_each_group([&](int, const uint32_t(&v)[4]) {
#pragma unroll
        for (int c = 0; c < 4; ++c) atomicAdd(&sm.hist1[v[c] >> 20], 1);
    });
    __syncthreads();
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");   // every CTA's totals are cleared
    cluster_find_bin<kBins1 / kTkThreads>(sm.hist1, sm.tot1, k, C, sm);
    const uint32_t d1 = static_cast<uint32_t>(sm.ctrl[0]);
    int k_rem = k - sm.ctrl[1];
    const int inbin1 = sm.ctrl[2];
    uint32_t pval = d1 << 20, pmask = 0xfff00000u;
    uint32_t T = pval;
    int take_eq = kAllEqual;
    if (inbin1 != k_rem) {
        // ---- this CTA's keys of the threshold bin into the list (any order);
        // a bin too large for it (the same decision in every CTA) is counted
        // from the keys themselves
        const bool listed = inbin1 <= kListCap;
        if (listed) {
            uint32_t inm[K::W];
#pragma unroll
            for (int w = 0; w < K::W; ++w) inm[w] = 0u;
            int cnt = 0;
            key.for_each_group_reaching(pval, key_float(pval), [&](int i, const uint32_t(&v)[4]) {
                uint32_t b = 0;
#pragma unroll
                for (int c = 0; c < 4; ++c) b |= static_cast<uint32_t>((v[c] & pmask) == pval) << c;
                K::set_nib(inm, i, b);
                cnt += __popc(b);
            });
            int wt, o;
            {
                int incl = cnt;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += y;
                }
                wt = __shfl_sync(0xffffffffu, incl, 31);
                int wb = 0;
                if (lane == 0 && wt) wb = atomicAdd(&sm.nlist, wt);
                o = __shfl_sync(0xffffffffu, wb, 0) + incl - cnt;
            }
            if (cnt) {
#pragma unroll
                for (int i = 0; i < K::G; ++i) {
                    const uint32_t b = K::nib(inm, i);
                    if (b) {
                        const float4 f4 = i < K::GR ? make_float4(0.f, 0.f, 0.f, 0.f) : key.sk[(i - K::GR) * kTkThreads];
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            if ((b >> c) & 1u) {
                                const uint32_t v = i < K::GR ? key.reg[(4 * i + c) % (4 * K::GR)]
                                                             : order_key(c == 0 ? f4.x : c == 1 ? f4.y : c == 2 ? f4.z : f4.w);
                                if (o < kListCap) sm.list[o] = v;
                                ++o;
                            }
                    }
                }
            }
            __syncthreads();
        }
        const int nlist = min(sm.nlist, kListCap);
        // ---- digits 2 and 3: bits 19..10, then 9..0
#pragma unroll 1
        for (int d = 0; d < 2; ++d) {
            const int shift = d == 0 ? 10 : 0;
            int* hist = d == 0 ? sm.hist2 : sm.hist3;
            int* tot = d == 0 ? sm.tot2 : sm.tot3;
            if (listed) {
                for (int i = tid; i < nlist; i += kTkThreads) {
                    const uint32_t v = sm.list[i];
                    if ((v & pmask) == pval) atomicAdd(&hist[(v >> shift) & 1023u], 1);
                }
            } else {
                key.for_each_group_reaching(pval, key_float(pval), [&](int, const uint32_t(&v)[4]) {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        if ((v[c] & pmask) == pval) atomicAdd(&hist[(v[c] >> shift) & 1023u], 1);
                });
            }
            __syncthreads();
            cluster_find_bin<kBins2 / kTkThreads>(hist, tot, k_rem, C, sm);
            k_rem -= sm.ctrl[1];
            pval |= static_cast<uint32_t>(sm.ctrl[0]) << shift;
            pmask |= 1023u << shift;
            T = pval;
            if (sm.ctrl[2] == k_rem) break;                // the whole bin is selected
            if (d == 1) take_eq = k_rem;                   // T is a complete key
        }
    }
    // ---- selection: keys above T, and the first take_eq keys equal to T in
    // row order (kAllEqual: every key from T up); only groups whose largest
    // key reaches T are looked at
    uint32_t gt[K::W], eq[K::W];
#pragma unroll
    for (int w = 0; w < K::W; ++w) gt[w] = eq[w] = 0u;
    key.for_each_group_reaching(T, key_float(T), [&](int i, const uint32_t(&v)[4]) {
        uint32_t g = 0, e = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            g |= static_cast<uint32_t>(v[c] > T) << c;
            e |= static_cast<uint32_t>(v[c] == T) << c;
        }
        if (take_eq == kAllEqual) {
            g |= e;
            e = 0;
        }
        K::set_nib(gt, i, g);
        K::set_nib(eq, i, e);
    });
    // ---- counts per warp, per CTA, and across the cluster
    {
        int gc = 0, ec = 0;
#pragma unroll
        for (int w = 0; w < K::W; ++w) {
            gc += __popc(gt[w]);
            ec += __popc(eq[w]);
        }
        gc = __reduce_add_sync(0xffffffffu, gc);
        ec = __reduce_add_sync(0xffffffffu, ec);
        if (lane == 0) {
            sm.warp_gt[warp] = gc;
            sm.warp_eq[warp] = ec;
        }
    }
    __syncthreads();
    int gb, eb, gtot, etot;                                // before this warp; in the CTA
    {
        // lane l holds warp l's counts: inclusive scans, read at this warp
        int g = sm.warp_gt[lane], e = sm.warp_eq[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int yg = __shfl_up_sync(0xffffffffu, g, off), ye = __shfl_up_sync(0xffffffffu, e, off);
            if (lane >= off) {
                g += yg;
                e += ye;
            }
        }
        gtot = __shfl_sync(0xffffffffu, g, 31);
        etot = __shfl_sync(0xffffffffu, e, 31);
        const int gi = __shfl_sync(0xffffffffu, g, warp), ei = __shfl_sync(0xffffffffu, e, warp);
        gb = gi - __shfl_sync(0xffffffffu, sm.warp_gt[lane], warp);
        eb = ei - __shfl_sync(0xffffffffu, sm.warp_eq[lane], warp);
    }
    if (tid < C) {
        st_cluster_s32(mapa(smem_u32(&sm.cta_gt[rank]), tid), gtot);
        st_cluster_s32(mapa(smem_u32(&sm.cta_eq[rank]), tid), etot);
    }
    cluster_sync();                                        // every CTA's counts are everywhere
    for (int q = 0; q < rank; ++q) {
        gb += sm.cta_gt[q];
        eb += sm.cta_eq[q];
    }
    // gb, eb: keys above T / equal to T before this warp in the row
    const int out_o = gb + min(eb, take_eq);               // selected entries before this warp
    // ---- write: the warp's selected positions (128 i + 4 lane + c within
    // its region, which is row order) go to a bitmap of the region in the
    // free list area, bit b of word b / 32 for position b; lane l then owns
    // words 2l and 2l + 1 and one warp scan places every index.  With one
    // group per lane the positions are in lane order already.
    uint32_t a, b = 0u;                                    // the lane's selected positions, in order
    int any_eq = 0;
#pragma unroll
    for (int w = 0; w < K::W; ++w) any_eq |= eq[w];
    const bool weq = __any_sync(0xffffffffu, any_eq != 0);
    if constexpr (K::G == 1) {
        // one group: the lane's four positions 4 lane + c are already in row
        // order, so a is its nibble (positions counted from 4 lane, below)
        a = gt[0];
        if (weq) {
            uint32_t q = eq[0];
            const int ec = __popc(q);
            int incl = ec;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            int rk = eb + incl - ec;
            for (; q; q &= q - 1, ++rk)
                if (rk < take_eq) a |= q & (0u - q);
        }
    } else {
        uint32_t* bm = sm.list + warp * KPT;               // selected
        uint32_t* bq = sm.list + (kTkWarps + warp) * KPT;  // equal to T (only when the warp has any)
        for (int w = lane; w < KPT; w += 32) {
            bm[w] = 0u;
            if (weq) bq[w] = 0u;
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < K::G; ++i) {
            const uint32_t g = K::nib(gt, i), e = K::nib(eq, i);
            const int wd = 4 * i + (lane >> 3), sh = 4 * (lane & 7);
            if (g) atomicOr(&bm[wd], g << sh);
            if (e) atomicOr(&bq[wd], e << sh);
        }
        __syncwarp();
        const bool owns = 2 * lane < KPT;                  // words 2 lane, 2 lane + 1
        a = owns ? bm[2 * lane] : 0u;
        b = owns ? bm[2 * lane + 1] : 0u;
        if (weq) {
            // equal keys in row order take row ranks eb, eb + 1, ...: the
            // first take_eq of the row are selected
            uint32_t qa = owns ? bq[2 * lane] : 0u, qb = owns ? bq[2 * lane + 1] : 0u;
            const int ec = __popc(qa) + __popc(qb);
            int incl = ec;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            int rk = eb + incl - ec;
            for (; qa; qa &= qa - 1, ++rk)
                if (rk < take_eq) a |= qa & (0u - qa);
            for (; qb; qb &= qb - 1, ++rk)
                if (rk < take_eq) b |= qb & (0u - qb);
        }
    }
    const int sc = __popc(a) + __popc(b);
    int incl = sc;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    int o = out_o + incl - sc;
    const int pos0 = wbase + (K::G == 1 ? 4 : 64) * lane;
    for (; a; a &= a - 1, ++o)
        if (static_cast<unsigned>(o) < static_cast<unsigned>(k)) out[o] = pos0 + __ffs(a) - 1;
    for (; b; b &= b - 1, ++o)
        if (static_cast<unsigned>(o) < static_cast<unsigned>(k)) out[o] = pos0 + 32 + __ffs(b) - 1;
}

std::mutex g_topk_mu;
int g_topk_sms[64];            // SM count per device, 0 until prepared
int g_topk_clusters[64][5][kMaxClusterCtas + 1];   // clusters resident at once, per (device, KPT, size); 0 = not asked

constexpr int kKptCount = 5;                       // KPT = 4, 8, 16, 32, 64
constexpr size_t topk_smem_bytes(int kpt) {
    return sizeof(SelectSmem) + (kpt > 32 ? static_cast<size_t>(kpt - 32) * kTkThreads * 4 : 0);
}
static_assert(topk_smem_bytes(kMaxKeys) <= 227 * 1024, "top-k shared memory");
static_assert(2 * kTkWarps * kMaxKeys <= kListCap, "the output bitmaps reuse the list");

template <int KPT>
bool allow_smem() {
    return cudaFuncSetAttribute(dsv4_topk_kernel<KPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(topk_smem_bytes(KPT))) == cudaSuccess;
}

template <int KPT>
cudaError_t launch_kpt(cudaLaunchConfig_t& cfg, const TopkParams& p, int* max_clusters) {
    if (max_clusters) return cudaOccupancyMaxActiveClusters(max_clusters, dsv4_topk_kernel<KPT>, &cfg);
    return cudaLaunchKernelEx(&cfg, dsv4_topk_kernel<KPT>, p);
}

// Launches (or, with max_clusters, asks how many clusters of this shape the
// device holds at once).
cudaError_t launch_topk(int kpt, cudaLaunchConfig_t& cfg, const TopkParams& p, int* max_clusters) {
    switch (kpt) {
        case 4: return launch_kpt<4>(cfg, p, max_clusters);
        case 8: return launch_kpt<8>(cfg, p, max_clusters);
        case 16: return launch_kpt<16>(cfg, p, max_clusters);
        case 32: return launch_kpt<32>(cfg, p, max_clusters);
        default: return launch_kpt<64>(cfg, p, max_clusters);
    }
}

// The shared state exceeds the default 48 KB: allow it once per device.
int topk_prepare_device(int& dev) {
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DSV4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_topk_mu);
    if (!g_topk_sms[dev]) {
        int n = 0;
        if (!allow_smem<4>() || !allow_smem<8>() || !allow_smem<16>() || !allow_smem<32>() || !allow_smem<64>() ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
            cudaGetLastError();
            return DSV4_ERR_CUDA;
        }
        g_topk_sms[dev] = n;
    }
    return DSV4_OK;
}

void fill_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int kpt, int C, int rows, cudaStream_t stream) {
    cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(C), static_cast<unsigned>(rows), 1);
    cfg.blockDim = dim3(kTkThreads, 1, 1);
    cfg.dynamicSmemBytes = topk_smem_bytes(kpt);
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
}

// Clusters of C CTAs at KPT scores per thread the device holds at once.
int resident_clusters(int dev, int kpt_idx, int kpt, int C) {
    {
        std::lock_guard<std::mutex> lock(g_topk_mu);
        if (g_topk_clusters[dev][kpt_idx][C]) return g_topk_clusters[dev][kpt_idx][C];
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    fill_config(cfg, attr, kpt, C, 1, nullptr);
    cfg.numAttrs = 1;                                      // the cluster shape alone
    int n = 0;
    TopkParams none = {};
    if (launch_topk(kpt, cfg, none, &n) != cudaSuccess || n < 1) {
        cudaGetLastError();
        n = 1;
    }
    std::lock_guard<std::mutex> lock(g_topk_mu);
    g_topk_clusters[dev][kpt_idx][C] = n;
    return n;
}

}  // namespace
}  // namespace dsv4

extern "C" int32_t dsv4_topk_max_length(int32_t k) {
    return (k < 1 || k > dsv4::kMaxK) ? 0 : dsv4::kMaxLength;
}

extern "C" int dsv4_topk(const float* scores, int32_t num_rows, int64_t row_stride, const int32_t* lengths,
                         int32_t max_length, int32_t k, int32_t* out_idx, void* stream) {
    using namespace dsv4;
    if (num_rows < 1 || num_rows > 65535 || k < 1 || k > kMaxK || max_length < 0) return DSV4_ERR_INVALID;
    if (!scores || !lengths || !out_idx) return DSV4_ERR_INVALID;
    if (row_stride < max_length || row_stride % 4 || reinterpret_cast<uintptr_t>(scores) % 16) return DSV4_ERR_INVALID;
    if (max_length > kMaxLength) return DSV4_ERR_UNSUPPORTED;
    unsigned int* err = device_error_word();
    if (!err) return DSV4_ERR_CUDA;
    int dev = 0;
    if (topk_prepare_device(dev) != DSV4_OK) return DSV4_ERR_CUDA;
    // scores per thread: the fewest whose cluster (at most 8 CTAs) covers a
    // row while every row's cluster is resident at once; failing that, the
    // fewest that cover a row
    const int len = max(max_length, 1);
    int kpt = 0, C = 0;
    for (int i = 0, e = 4; i < kKptCount; ++i, e *= 2) {
        const int c = (len + kTkThreads * e - 1) / (kTkThreads * e);
        if (c > kMaxClusterCtas) continue;
        if (!kpt) {
            kpt = e;
            C = c;
        }
        if (num_rows <= resident_clusters(dev, i, e, c)) {
            kpt = e;
            C = c;
            break;
        }
    }
    TopkParams p;
    p.scores = scores;
    p.stride = row_stride;
    p.lengths = lengths;
    p.max_len = max_length;
    p.k = k;
    p.out = out_idx;
    p.err = err;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    fill_config(cfg, attr, kpt, C, num_rows, static_cast<cudaStream_t>(stream));
    if (launch_topk(kpt, cfg, p, nullptr) != cudaSuccess) {
        cudaGetLastError();
        return DSV4_ERR_CUDA;
    }
    return DSV4_OK;
}
