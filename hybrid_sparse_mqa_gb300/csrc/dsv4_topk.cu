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
// How: every candidate gets a unique 64-bit composite key, (order-preserving
// bits of its fp32 score) << 32 | ~index, so "higher score, then lower index"
// is plain integer order and the k best form a unique set.  A CTA takes a
// chunk of 16384 scores of one row, 32 consecutive scores per thread held in
// registers (one HBM read), and finds the k-th largest composite by an exact
// radix select: one 8-bit digit per pass from the top, counted into
// warp-private shared histograms, stopping as soon as the k-th digit's bin
// holds exactly the entries still needed (four passes for distinct scores,
// up to eight when scores tie at the threshold).  Selected entries leave in
// ascending index order through one block-wide prefix sum.  A row of one
// chunk is done there; longer rows write each chunk's k best to the
// workspace, and the last CTA of the row to finish (an atomic counter it
// resets) selects the final k from those candidates the same way.  The
// pages' design spreads one row over a cluster of 8 CTAs; here the chunks
// of a row need not be co-resident, so any number of rows fills the GPU.
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

struct SelectSmem {
    int hist[kTkWarps][256];
    int ctrl[3];
    int wsum[kTkWarps];
    int flag;
};

// fp32 bits -> uint32 whose unsigned order is the value order (-0 below +0)
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The k_rem-th largest composite among this block's valid entries (E per
// thread, bit j of `valid` for entry j, comp(j) its composite; every
// composite distinct; at least k_rem valid): returns T such that exactly
// k_rem entries are >= T.
template <int E, typename Comp>
__device__ uint64_t select_threshold(Comp comp, uint32_t valid, int k_rem, SelectSmem& sm) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t pval = 0, pmask = 0;
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = tid; i < kTkWarps * 256; i += kTkThreads) (&sm.hist[0][0])[i] = 0;
        __syncthreads();
#pragma unroll
        for (int j = 0; j < E; ++j) {
            if ((valid >> j) & 1u) {
                const uint64_t c = comp(j);
                if ((c & pmask) == pval) atomicAdd(&sm.hist[warp][static_cast<int>((c >> shift) & 0xffu)], 1);
            }
        }
        __syncthreads();
        if (tid < 256) {
            // thread d: entries in bin d, and in bins d .. 255 (suffix sum)
            int tot = 0;
#pragma unroll
            for (int w = 0; w < kTkWarps; ++w) tot += sm.hist[w][tid];
            int v = tot;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int x = __shfl_down_sync(0xffffffffu, v, off);
                if (lane + off < 32) v += x;
            }
            if (lane == 0) sm.wsum[warp] = v;
            asm volatile("bar.sync 1, 256;" ::: "memory");
            int later = 0;
            for (int w = warp + 1; w < 256 / 32; ++w) later += sm.wsum[w];
            const int at_or_above = v + later, above = at_or_above - tot;
            if (at_or_above >= k_rem && above < k_rem) {
                sm.ctrl[0] = tid;
                sm.ctrl[1] = above;
                sm.ctrl[2] = tot;
            }
        }
        __syncthreads();
        const int d = sm.ctrl[0], above = sm.ctrl[1], inbin = sm.ctrl[2];
        k_rem -= above;
        pval |= static_cast<uint64_t>(d) << shift;
        pmask |= 0xffull << shift;
        if (inbin == k_rem) break;       // every entry of the bin is selected (uniform)
    }
    return pval;
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

__global__ void __launch_bounds__(kTkThreads) dsv4_topk_kernel(const __grid_constant__ TopkParams p) {
    __shared__ SelectSmem sm;
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
    const int nch = (n + kChunk - 1) / kChunk;
    if (c >= nch) return;
    const int base = c * kChunk;
    const int m = min(kChunk, n - base);
    const int first = kKeysPerThread * tid;                 // this thread's scores: base + first + j
    const uint32_t gidx0 = static_cast<uint32_t>(base + first);
    const float* src = p.scores + (size_t)r * p.stride + base + first;
    uint32_t key[kKeysPerThread];
    uint32_t valid = 0;
    if (first + kKeysPerThread <= m) {
        const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
        for (int q = 0; q < kKeysPerThread / 4; ++q) {
            const float4 v = __ldcs(s4 + q);
            key[4 * q] = order_key(v.x);
            key[4 * q + 1] = order_key(v.y);
            key[4 * q + 2] = order_key(v.z);
            key[4 * q + 3] = order_key(v.w);
        }
        valid = 0xffffffffu;
    } else {
#pragma unroll
        for (int j = 0; j < kKeysPerThread; ++j) {
            key[j] = 0;
            if (first + j < m) {
                key[j] = order_key(__ldcs(src + j));
                valid |= 1u << j;
            }
        }
    }
    auto comp = [&](int j) { return (static_cast<uint64_t>(key[j]) << 32) | static_cast<uint32_t>(~(gidx0 + j)); };
    const int want = min(k, m);
    const uint64_t T = m > want ? select_threshold<kKeysPerThread>(comp, valid, want, sm) : 0ull;
    uint32_t sel = 0;
#pragma unroll
    for (int j = 0; j < kKeysPerThread; ++j)
        if (((valid >> j) & 1u) && comp(j) >= T) sel |= 1u << j;
    int total;
    const int off = block_exclusive_scan(__popc(sel), total, sm);
    if (nch == 1) {
        // the whole row: its k indices, ascending
        int o = off;
#pragma unroll
        for (int j = 0; j < kKeysPerThread; ++j)
            if ((sel >> j) & 1u) out[o++] = static_cast<int>(gidx0 + j);
        return;
    }
    unsigned long long* cand = p.cand + ((size_t)r * p.chunks + c) * k;
    {
        int o = off;
#pragma unroll
        for (int j = 0; j < kKeysPerThread; ++j)
            if ((sel >> j) & 1u) cand[o++] = comp(j);
    }
    if (tid == 0) p.cnt[(size_t)r * p.chunks + c] = total;
    // the last chunk of the row to finish selects among all chunks' candidates
    __threadfence();
    __syncthreads();
    if (tid == 0) sm.flag = atomicAdd(p.done + r, 1) == nch - 1;
    __syncthreads();
    if (!sm.flag) return;
    __threadfence();
    if (tid == 0) {
        int acc = 0;
        for (int cc = 0; cc < nch; ++cc) {
            chunk_off[cc] = acc;
            acc += __ldcg(p.cnt + (size_t)r * p.chunks + cc);
        }
        chunk_off[nch] = acc;
        p.done[r] = 0;                          // ready for the next call
    }
    __syncthreads();
    const int ncand = chunk_off[nch];           // <= nch * k <= kMergeCap (host check on max_length)
    const unsigned long long* rc = p.cand + (size_t)r * p.chunks * k;
    uint64_t cv[kMergePerThread];
    uint32_t v2 = 0;
    int cc = 0;
#pragma unroll
    for (int j = 0; j < kMergePerThread; ++j) {
        const int pos = kMergePerThread * tid + j;     // candidates in chunk order = ascending index
        cv[j] = 0;
        if (pos < ncand) {
            while (chunk_off[cc + 1] <= pos) ++cc;
            cv[j] = __ldcg(rc + (size_t)cc * k + (pos - chunk_off[cc]));
            v2 |= 1u << j;
        }
    }
    auto comp2 = [&](int j) { return cv[j]; };
    const uint64_t T2 = ncand > k ? select_threshold<kMergePerThread>(comp2, v2, k, sm) : 0ull;
    uint32_t sel2 = 0;
#pragma unroll
    for (int j = 0; j < kMergePerThread; ++j)
        if (((v2 >> j) & 1u) && cv[j] >= T2) sel2 |= 1u << j;
    const int off2 = block_exclusive_scan(__popc(sel2), total, sm);
    int o = off2;
#pragma unroll
    for (int j = 0; j < kMergePerThread; ++j)
        if ((sel2 >> j) & 1u) out[o++] = static_cast<int>(~static_cast<uint32_t>(cv[j]));
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
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, dsv4_topk_kernel, p) != cudaSuccess) {
        cudaGetLastError();
        return DSV4_ERR_CUDA;
    }
    return DSV4_OK;
}
