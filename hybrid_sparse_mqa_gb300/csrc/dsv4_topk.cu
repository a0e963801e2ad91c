// dsv4_topk.cu - top-k index selection for the C4 index lists (the k best
// indexer scores of every query token).  What is computed is stated in
// include/dsv4topk.h.
//
// Sources (page title, section): "DeepSeek-V4 and SGLang Day-0" - kernel
// list (the indexer keeps the top 512 of 256K candidates at 1M context with
// a radix select over a thread-block cluster instead of a global sort);
// "DeepSeek-V4 Attention: Query, Cache Write and History Addressing" -
// section 5 (the top-k indices limit the C4 rows a token reads).
//
// How: a score's order-preserving 32-bit key (its fp32 bits with the sign
// folded) makes "higher score" plain integer order.  A CTA takes a chunk of
// 16384 scores of one row, 32 consecutive scores per thread held in
// registers (one HBM read), and finds the k-th largest key by an exact radix
// select: digits of 12, 10 and 10 bits from the top, counted into one shared
// histogram (the first over the registers, the other two over a shared list
// of the keys in the first digit's threshold bin), stopping as soon as the
// k-th key's bin holds exactly the entries still needed.  Keys above the threshold are selected; when several
// keys equal it, the lowest indices among them are taken, found by a prefix
// count in index order (a thread's scores are consecutive, so thread order
// is index order).  Selected entries leave in ascending index order through
// one block-wide prefix sum.  A row of one chunk is done there; longer rows
// write each chunk's k best (key and index) to the workspace, and the last
// CTA of the row to finish (an atomic counter it resets) selects the final k
// from those candidates the same way.  The pages' design spreads one row
// over a cluster of 8 CTAs; here the chunks of a row need not be
// co-resident, so any number of rows fills the GPU.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "dsv4attn.h"
#include "dsv4topk.h"
#include "dsv4_internal.h"

namespace dsv4 {
namespace {

constexpr int kTkThreads = 512;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kKeysPerThread = 32;                        // scores per thread in a chunk
constexpr int kChunk = kTkThreads * kKeysPerThread;       // 16384 scores per CTA
constexpr int kMergePerThread = 16;                       // candidates per thread in a merge
constexpr int kMergeCap = kTkThreads * kMergePerThread;   // 8192 candidates per row
constexpr int kMaxK = 1024;
constexpr int kMaxChunks = 64;                            // chunks per row (size of the offset table)

struct TopkParams {
    const float* scores;
    long long stride;          // floats between rows
    const int* lengths;
    int rows;
    int max_len;
    int k;
    int chunks;                // chunks of the longest row (grid x)
    int* out;                  // [rows][k]
    unsigned long long* cand;  // [rows][chunks][k] composites of each chunk's k best
    int* cnt;                  // [rows][chunks] how many each chunk kept
    int* done;                 // [rows] chunks finished (zero between calls)
    unsigned int* err;
};

constexpr int kHistBins = 4096;                          // widest digit (12 bits)
constexpr int kListCap = 8192;                            // keys of the threshold bin after the first digit

struct SelectSmem {
    int hist[kHistBins];
    uint32_t list[kListCap];
    int ctrl[3];
    int wsum[kTkWarps];
    int flag;
};

// fp32 bits -> uint32 whose unsigned order is the value order (-0 below +0)
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum of x over the block (thread order) and the total.
__device__ int block_exclusive_scan(int x, int& total, SelectSmem& sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int v = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += y;
    }
    if (lane == 31) sm.wsum[warp] = v;
    __syncthreads();
    int before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kTkWarps; ++w) {
        const int s = sm.wsum[w];
        before += w < warp ? s : 0;
        tot += s;
    }
    total = tot;
    __syncthreads();
    return before + v - x;
}

// Histogram of digit (key >> shift) & (nb - 1) over the keys that match
// `pval` on `pmask`, then the bin d holding the k_rem-th largest of them:
// sets ctrl = {d, entries in bins above d, entries in bin d}.
__device__ __forceinline__ int hist_total(const SelectSmem& sm, int b) { return sm.hist[b]; }
__device__ __forceinline__ void hist_zero(SelectSmem& sm, int nb) {
    for (int i = threadIdx.x; i < nb; i += kTkThreads) sm.hist[i] = 0;
}

__device__ void find_digit_bin(int nb, int k_rem, SelectSmem& sm) {
    const int tid = threadIdx.x;
    const int per = nb / kTkThreads;                 // bins owned by each thread
    int own = 0;
    for (int b = 0; b < per; ++b) own += hist_total(sm, tid * per + b);
    int total;
    const int before = block_exclusive_scan(own, total, sm);
    int above = total - before - own;                // entries in the bins of later threads
    for (int b = per - 1; b >= 0; --b) {
        const int h = hist_total(sm, tid * per + b);
        if (above < k_rem && above + h >= k_rem) {
            sm.ctrl[0] = tid * per + b;
            sm.ctrl[1] = above;
            sm.ctrl[2] = h;
        }
        above += h;
    }
    __syncthreads();
}

// Threshold of the k largest keys among the block's valid entries (E per
// thread, bit j of `valid` for entry j; at least k valid): every key above T
// is selected, and `take_eq` of the keys equal to T (the lowest indices;
// INT_MAX when all of them).  The first digit (12 bits) is counted over the
// registers; the keys of its threshold bin are then gathered into a shared
// list and the remaining two digits (10 bits each) are counted over it.
template <int E>
__device__ void select_threshold(const uint32_t (&key)[E], uint32_t valid, int k, uint32_t& T, int& take_eq,
                                 SelectSmem& sm) {
    const int tid = threadIdx.x;
    int* hw = sm.hist;
    // ---- digit 1: bits 31..20, over every key
    hist_zero(sm, 4096);
    __syncthreads();
#pragma unroll
    for (int j = 0; j < E; ++j)
        if ((valid >> j) & 1u) atomicAdd(hw + (key[j] >> 20), 1);
    __syncthreads();
    find_digit_bin(4096, k, sm);
    const int d1 = sm.ctrl[0];
    int k_rem = k - sm.ctrl[1];
    const int inbin1 = sm.ctrl[2];
    uint32_t pval = static_cast<uint32_t>(d1) << 20;
    if (inbin1 == k_rem) {
        T = pval;
        take_eq = 0x7fffffff;
        return;
    }
    // ---- the bin's keys into the list (any order: only the threshold is
    // sought); a bin too large for it is counted from the registers instead
    const bool listed = inbin1 <= kListCap;
    if (listed) {
        uint32_t in = 0;
#pragma unroll
        for (int j = 0; j < E; ++j)
            if (((valid >> j) & 1u) && (key[j] >> 20) == static_cast<uint32_t>(d1)) in |= 1u << j;
        int total;
        int o = block_exclusive_scan(__popc(in), total, sm);
#pragma unroll
        for (int j = 0; j < E; ++j)
            if ((in >> j) & 1u) sm.list[o++] = key[j];
    }
    // ---- digits 2 and 3: bits 19..10, then 9..0
    uint32_t pmask = 0xfff00000u;
#pragma unroll 1
    for (int shift = 10; shift >= 0; shift -= 10) {
        hist_zero(sm, 1024);
        __syncthreads();
        if (listed) {
            for (int i = tid; i < inbin1; i += kTkThreads) {
                const uint32_t v = sm.list[i];
                if ((v & pmask) == pval) atomicAdd(hw + ((v >> shift) & 1023u), 1);
            }
        } else {
#pragma unroll
            for (int j = 0; j < E; ++j)
                if (((valid >> j) & 1u) && (key[j] & pmask) == pval) atomicAdd(hw + ((key[j] >> shift) & 1023u), 1);
        }
        __syncthreads();
        find_digit_bin(1024, k_rem, sm);
        const int d = sm.ctrl[0], a = sm.ctrl[1], inbin = sm.ctrl[2];
        k_rem -= a;
        pval |= static_cast<uint32_t>(d) << shift;
        pmask |= 1023u << shift;
        if (inbin == k_rem) {
            T = pval;
            take_eq = 0x7fffffff;
            return;
        }
    }
    T = pval;                                        // the key is fully decided
    take_eq = k_rem;
}

// Bit j set when entry j is among the k selected (threshold T, take_eq of
// the keys equal to T in index order = thread order, then j).
template <int E>
__device__ uint32_t selected_mask(const uint32_t (&key)[E], uint32_t valid, uint32_t T, int take_eq,
                                  SelectSmem& sm) {
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int j = 0; j < E; ++j) {
        if ((valid >> j) & 1u) {
            gt |= (key[j] > T) ? (1u << j) : 0u;
            eq |= (key[j] == T) ? (1u << j) : 0u;
        }
    }
    if (take_eq == 0x7fffffff) return gt | eq;
    int total;
    int rank = block_exclusive_scan(__popc(eq), total, sm);   // equal keys before this thread's
    uint32_t sel = gt;
#pragma unroll
    for (int j = 0; j < E; ++j)
        if ((eq >> j) & 1u) {
            if (rank < take_eq) sel |= 1u << j;
            ++rank;
        }
    return sel;
}

template <int KPT>
__global__ void __launch_bounds__(kTkThreads, 2) dsv4_topk_kernel(const __grid_constant__ TopkParams p) {
    constexpr int kCh = kTkThreads * KPT;                // scores per chunk
    extern __shared__ __align__(16) uint8_t tk_smem[];
    SelectSmem& sm = *reinterpret_cast<SelectSmem*>(tk_smem);
    __shared__ int chunk_off[kMaxChunks + 1];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int r = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
    const int k = p.k;
    int n = __ldg(p.lengths + r);
    if (n < 0 || n > p.max_len) {
        if (c == 0 && tid == 0) atomicOr(p.err, DSV4_DEV_ERR_TOPK_LENGTH);
        n = n < 0 ? 0 : p.max_len;
    }
    int* out = p.out + (size_t)r * k;
    if (n <= k) {
        // every candidate is selected
        if (c == 0)
            for (int i = tid; i < k; i += kTkThreads) out[i] = i < n ? i : -1;
        return;
    }
    const int nch = (n + kCh - 1) / kCh;
    if (c >= nch) return;
    const int base = c * kCh;
    const int m = min(kCh, n - base);
    const int first = KPT * tid;                 // this thread's scores: base + first + j
    const uint32_t gidx0 = static_cast<uint32_t>(base + first);
    const float* src = p.scores + (size_t)r * p.stride + base + first;
    uint32_t key[KPT];
    uint32_t valid = 0;
    if (first + KPT <= m) {
        const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
        for (int q = 0; q < KPT / 4; ++q) {
            const float4 v = __ldcs(s4 + q);
            key[4 * q] = order_key(v.x);
            key[4 * q + 1] = order_key(v.y);
            key[4 * q + 2] = order_key(v.z);
            key[4 * q + 3] = order_key(v.w);
        }
        valid = 0xffffffffu;
    } else {
#pragma unroll
        for (int j = 0; j < KPT; ++j) {
            key[j] = 0;
            if (first + j < m) {
                key[j] = order_key(__ldcs(src + j));
                valid |= 1u << j;
            }
        }
    }
    const int want = min(k, m);
    uint32_t sel = valid;
    if (m > want) {
        uint32_t T;
        int take_eq;
        select_threshold<KPT>(key, valid, want, T, take_eq, sm);
        sel = selected_mask<KPT>(key, valid, T, take_eq, sm);
    }
    int total;
    const int off = block_exclusive_scan(__popc(sel), total, sm);
    if (nch == 1) {
        // the whole row: its k indices, ascending
        int o = off;
#pragma unroll
        for (int j = 0; j < KPT; ++j)
            if ((sel >> j) & 1u) out[o++] = static_cast<int>(gidx0 + j);
        return;
    }
    // this chunk's k best as (key << 32 | index), in index order
    unsigned long long* cand = p.cand + ((size_t)r * p.chunks + c) * k;
    {
        int o = off;
#pragma unroll
        for (int j = 0; j < KPT; ++j)
            if ((sel >> j) & 1u) cand[o++] = (static_cast<unsigned long long>(key[j]) << 32) | (gidx0 + j);
    }
    if (tid == 0) p.cnt[(size_t)r * p.chunks + c] = total;
    // the last chunk of the row to finish selects among all chunks' candidates
    __threadfence();
    __syncthreads();
    if (tid == 0) sm.flag = atomicAdd(p.done + r, 1) == nch - 1;
    __syncthreads();
    if (!sm.flag) return;
    __threadfence();
    if (tid < 32) {
        // chunk counts loaded together (lanes l and l + 32), then prefix-summed
        const int* cr = p.cnt + (size_t)r * p.chunks;
        const int c0 = tid < nch ? __ldcg(cr + tid) : 0;
        const int c1 = tid + 32 < nch ? __ldcg(cr + tid + 32) : 0;
        int s0 = c0, s1 = c1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y0 = __shfl_up_sync(0xffffffffu, s0, off), y1 = __shfl_up_sync(0xffffffffu, s1, off);
            if (tid >= off) {
                s0 += y0;
                s1 += y1;
            }
        }
        const int tot0 = __shfl_sync(0xffffffffu, s0, 31);
        chunk_off[tid] = s0 - c0;                  // exclusive offsets
        chunk_off[tid + 32] = tot0 + s1 - c1;
        if (tid == 31) chunk_off[64] = tot0 + s1;
        if (tid == 0) p.done[r] = 0;             // ready for the next call
    }
    __syncthreads();
    const int ncand = chunk_off[nch];           // <= nch * k <= kMergeCap (host check on max_length)
    const unsigned long long* rc = p.cand + (size_t)r * p.chunks * k;
    uint32_t ck[kMergePerThread], ci[kMergePerThread];
    uint32_t v2 = 0;
    int cc = 0;
#pragma unroll
    for (int j = 0; j < kMergePerThread; ++j) {
        const int pos = kMergePerThread * tid + j;     // candidates in chunk order = ascending index
        ck[j] = 0;
        ci[j] = 0;
        if (pos < ncand) {
            while (chunk_off[cc + 1] <= pos) ++cc;
            const unsigned long long v = __ldcg(rc + (size_t)cc * k + (pos - chunk_off[cc]));
            ck[j] = static_cast<uint32_t>(v >> 32);
            ci[j] = static_cast<uint32_t>(v);
            v2 |= 1u << j;
        }
    }
    uint32_t sel2 = v2;
    if (ncand > k) {
        uint32_t T2;
        int take_eq2;
        select_threshold<kMergePerThread>(ck, v2, k, T2, take_eq2, sm);
        sel2 = selected_mask<kMergePerThread>(ck, v2, T2, take_eq2, sm);
    }
    const int off2 = block_exclusive_scan(__popc(sel2), total, sm);
    int o = off2;
#pragma unroll
    for (int j = 0; j < kMergePerThread; ++j)
        if ((sel2 >> j) & 1u) out[o++] = static_cast<int>(ci[j]);
}

std::mutex g_topk_mu;
int g_topk_sms[64];

// The kernel's shared state exceeds the default 48 KB: allow it once per
// device; returns the device's SM count (0 on failure).
int topk_prepare_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(g_topk_mu);
    if (!g_topk_sms[dev]) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaFuncSetAttribute(dsv4_topk_kernel<kKeysPerThread>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(sizeof(SelectSmem))) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        g_topk_sms[dev] = sms;
    }
    return g_topk_sms[dev];
}

size_t topk_ws_bytes(int rows, int max_len, int k) {
    const size_t chunks = max_len > 0 ? (static_cast<size_t>(max_len) + kChunk - 1) / kChunk : 1;
    return (static_cast<size_t>(rows) * chunks * k * 8 + 255) / 256 * 256 +
           (static_cast<size_t>(rows) * chunks * 4 + 255) / 256 * 256 + static_cast<size_t>(rows) * 4;
}

}  // namespace
}  // namespace dsv4

extern "C" int32_t dsv4_topk_max_length(int32_t k) {
    using namespace dsv4;
    if (k < 1 || k > kMaxK) return 0;
    const int chunks = kMergeCap / k < kMaxChunks ? kMergeCap / k : kMaxChunks;
    return chunks * kChunk;
}

extern "C" size_t dsv4_topk_workspace_size(int32_t num_rows, int32_t max_length, int32_t k) {
    if (num_rows < 1 || max_length < 0 || k < 1 || k > dsv4::kMaxK) return 0;
    return dsv4::topk_ws_bytes(num_rows, max_length, k);
}

extern "C" int dsv4_topk(const float* scores, int32_t num_rows, int64_t row_stride, const int32_t* lengths,
                         int32_t max_length, int32_t k, int32_t* out_idx, void* workspace, size_t workspace_bytes,
                         void* stream) {
    using namespace dsv4;
    if (num_rows < 1 || num_rows > 65535 || k < 1 || k > kMaxK || max_length < 0) return DSV4_ERR_INVALID;
    if (!scores || !lengths || !out_idx) return DSV4_ERR_INVALID;
    if (row_stride < max_length || row_stride % 4 || reinterpret_cast<uintptr_t>(scores) % 16) return DSV4_ERR_INVALID;
    if (max_length > dsv4_topk_max_length(k)) return DSV4_ERR_UNSUPPORTED;
    const size_t need = topk_ws_bytes(num_rows, max_length, k);
    if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256) return DSV4_ERR_WORKSPACE;
    unsigned int* err = device_error_word();
    if (!err) return DSV4_ERR_CUDA;
    if (!topk_prepare_device()) return DSV4_ERR_CUDA;
    const int chunks = max_length > 0 ? (max_length + kChunk - 1) / kChunk : 1;
    TopkParams p;
    p.scores = scores;
    p.stride = row_stride;
    p.lengths = lengths;
    p.rows = num_rows;
    p.max_len = max_length;
    p.k = k;
    p.chunks = chunks;
    p.out = out_idx;
    uint8_t* w = static_cast<uint8_t*>(workspace);
    p.cand = reinterpret_cast<unsigned long long*>(w);
    w += (static_cast<size_t>(num_rows) * chunks * k * 8 + 255) / 256 * 256;
    p.cnt = reinterpret_cast<int*>(w);
    w += (static_cast<size_t>(num_rows) * chunks * 4 + 255) / 256 * 256;
    p.done = reinterpret_cast<int*>(w);
    p.err = err;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>(chunks), static_cast<unsigned>(num_rows), 1);
    cfg.blockDim = dim3(kTkThreads, 1, 1);
    cfg.dynamicSmemBytes = sizeof(SelectSmem);
    cfg.stream = static_cast<cudaStream_t>(stream);
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t le = cudaLaunchKernelEx(&cfg, dsv4_topk_kernel<kKeysPerThread>, p);
    if (le != cudaSuccess) {
        cudaGetLastError();
        return DSV4_ERR_CUDA;
    }
    return DSV4_OK;
}
