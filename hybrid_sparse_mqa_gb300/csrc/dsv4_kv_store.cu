// dsv4_kv_store.cu - the KV cache write before the hybrid sparse MQA
// attention step (DeepSeek-V4): new key rows stored into a paged pool,
// packed to FP8 for packed pools.  What is computed is stated in
// include/dsv4kvstore.h.
//
// Sources (page title, section): "DeepSeek-V4 Attention: Query, Cache Write
// and History Addressing" - section 3 (the current token is written into its
// SWA slot before attention), section 4 (page table); "SGLang DeepSeek-V4
// Attention Test Capability Matrix" - "Input And Config Coverage" (packed
// FP8 nope + BF16 rope rows), "Reference Implementation Notes" (the
// production pack-and-store path fills the SWA and extra pools).
//
// How: a warp stores two consecutive rows, issuing all of their loads
// before packing the first, so their memory round trips overlap.  Lane l
// holds values 16 l .. 16 l + 15 of a row (two 16-byte loads of a contiguous
// 1 KB row).  For a packed pool, lanes 0..27 hold the
// nope values (4 lanes per 64-value block: the block amax is two xor
// shuffles away), lanes 28..31 the rope; each nope lane writes its 16 codes
// as one 16-byte store, the rope lanes copy their 32 bytes, and lanes 0 and
// 1 write the 7 scales and the zero padding, so a 608-byte row is 38
// aligned 16-byte stores.  The work is a gather-free scatter bound by HBM:
// 1024 bytes read and 608 (or 1024) written per row, plus 8 bytes of
// indices and one page-table entry.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "dsv4attn.h"
#include "dsv4kvstore.h"
#include "dsv4_internal.h"

namespace dsv4 {
namespace {

constexpr int kStoreWarps = 8;             // warps per block
constexpr int kStoreRowsPerWarp = 2;       // rows whose loads a warp issues together
constexpr int kStoreMinBlocks = 6;         // resident blocks per SM the register budget allows
constexpr int kStorePageSize = 256;
constexpr int kNopeBytes = 448;            // e4m3 codes of the 448 nope values
constexpr int kRopeOff = 448;              // 64 bf16 rope values
constexpr int kScaleOff = 448 + 128;       // 7 fp32 block scales, then 4 zero bytes

struct StoreParams {
    const uint4* k;          // [n][64] 16-byte pieces of the bf16 rows
    int n;
    const int* req_rows;
    const int* positions;
    uint8_t* rows;
    long long num_pages;
    int row_bytes;
    const int* page_table;
    int pt_rows, pt_stride;
    unsigned int* err;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// e4m3 codes of four fp32 values, nearest with ties to even, saturating at
// +-448; byte j of the result is the code of v[j]
__device__ __forceinline__ uint32_t e4m3x4(float v0, float v1, float v2, float v3) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(v0, v1), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(v2, v3), __NV_SATFINITE, __NV_E4M3);
    return (lo & 0xffffu) | (hi << 16);
}

// Two fp32 values in one 64-bit register and the packed f32x2 arithmetic
// (each lane of a packed operation rounds exactly as the scalar one does).
__device__ __forceinline__ uint64_t f32x2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float2 f32x2_split(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// e4m3 codes of 16 values of one 64-value block, given the block's amax and
// scale, as 16 bytes (byte j = code of v[j]).  The codes are those of the
// correctly rounded quotient v / scale, nearest e4m3 with ties to even,
// saturating.  For amax >= 2^-100 one Markstein correction of v * RN(1/scale)
// gives the same code for every bf16 v with |v| <= amax (checked
// exhaustively over all such pairs; it fails only below amax = 2^-104, where
// the residual underflows); the sign is copied so that -0 stays -0.  Smaller
// blocks divide.
__device__ __forceinline__ uint4 e4m3x16(const float (&v)[16], float amax, float scale) {
    float q[16];
    if (amax >= 0x1p-100f) {
        const float y = __frcp_rn(scale);
        const uint64_t y2 = f32x2(y, y), ns2 = f32x2(-scale, -scale);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint64_t x2 = f32x2(v[2 * j], v[2 * j + 1]);
            const uint64_t q0 = mul_f32x2(x2, y2);
            const float2 q1 = f32x2_split(fma_f32x2(fma_f32x2(q0, ns2, x2), y2, q0));
            q[2 * j] = copysignf(q1.x, v[2 * j]);
            q[2 * j + 1] = copysignf(q1.y, v[2 * j + 1]);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) q[j] = __fdiv_rn(v[j], scale);
    }
    uint32_t c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) c[j] = e4m3x4(q[4 * j], q[4 * j + 1], q[4 * j + 2], q[4 * j + 3]);
    return make_uint4(c[0], c[1], c[2], c[3]);
}

// One row: the lane's 16 values (a, b) into pool row `dst`.
template <int FORMAT>
__device__ __forceinline__ void store_row(uint8_t* dst, uint4 a, uint4 b, int lane) {
    if constexpr (FORMAT == DSV4_KV_BF16) {
        uint4* d = reinterpret_cast<uint4*>(dst) + 2 * lane;
        d[0] = a;
        d[1] = b;
    } else {
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        float f[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            f[2 * j] = bf16_lo(w[j]);
            f[2 * j + 1] = bf16_hi(w[j]);
        }
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(f[j]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        // block scale (lanes 28..31 compute one for the rope; it is not used)
        const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
        if (lane < kNopeBytes / 16) {
            *reinterpret_cast<uint4*>(dst + 16 * lane) = e4m3x16(f, amax, scale);
        } else {
            uint4* d = reinterpret_cast<uint4*>(dst + kRopeOff + 32 * (lane - kNopeBytes / 16));
            d[0] = a;
            d[1] = b;
        }
        // scale of block k is in lanes 4k .. 4k + 3
        float s[7];
#pragma unroll
        for (int k = 0; k < 7; ++k) s[k] = __shfl_sync(0xffffffffu, scale, 4 * k);
        if (lane == 0)
            *reinterpret_cast<float4*>(dst + kScaleOff) = make_float4(s[0], s[1], s[2], s[3]);
        else if (lane == 1)
            *reinterpret_cast<float4*>(dst + kScaleOff + 16) = make_float4(s[4], s[5], s[6], 0.f);
    }
}

// Warp w stores rows RPW w .. RPW w + RPW - 1: every load of those rows (the
// values, the request rows and positions, then the page-table entries) is
// issued before the first row is packed, so their memory round trips overlap.
template <int FORMAT, int RPW>
__global__ void __launch_bounds__(kStoreWarps * 32, kStoreMinBlocks) dsv4_kv_store_kernel(const __grid_constant__ StoreParams p) {
    // programmatic dependent launch: wait for the producer of k and the
    // indices; let a following attention launch start its set-up
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int i0 = (blockIdx.x * kStoreWarps + (threadIdx.x >> 5)) * RPW;
    if (i0 >= p.n) return;
    uint4 a[RPW], b[RPW];
    int r[RPW], l[RPW];
    bool have[RPW];                              // row i0 + j exists (uniform over the warp)
#pragma unroll
    for (int j = 0; j < RPW; ++j) {
        const int i = i0 + j;
        have[j] = i < p.n;
        r[j] = l[j] = -1;
        a[j] = b[j] = make_uint4(0u, 0u, 0u, 0u);
        if (have[j]) {
            // this lane's 16 values, read once (streaming)
            const uint4* src = p.k + (size_t)i * 64 + 2 * lane;
            a[j] = __ldcs(src);
            b[j] = __ldcs(src + 1);
            r[j] = __ldg(p.req_rows + i);
            l[j] = __ldg(p.positions + i);
        }
    }
    int page[RPW];
#pragma unroll
    for (int j = 0; j < RPW; ++j) {
        page[j] = -1;
        if (have[j] && r[j] >= 0 && r[j] < p.pt_rows && l[j] >= 0 && l[j] / kStorePageSize < p.pt_stride)
            page[j] = __ldg(p.page_table + (size_t)r[j] * p.pt_stride + l[j] / kStorePageSize);
    }
#pragma unroll
    for (int j = 0; j < RPW; ++j) {
        if (!have[j]) continue;
        if (page[j] < 0 || page[j] >= p.num_pages) {
            if (lane == 0) atomicOr(p.err, DSV4_DEV_ERR_STORE_ROW);
            continue;
        }
        const long long dst_row = (long long)page[j] * kStorePageSize + l[j] % kStorePageSize;
        store_row<FORMAT>(p.rows + dst_row * p.row_bytes, a[j], b[j], lane);
    }
}

}  // namespace
}  // namespace dsv4

extern "C" int dsv4_kv_store(const void* k, int32_t n, const int32_t* req_rows, const int32_t* positions,
                             const dsv4_kv_pool* pool, void* stream) {
    using namespace dsv4;
    if (n < 0) return DSV4_ERR_INVALID;
    const int rc = check_pool(pool);
    if (rc) return rc;
    if (n == 0) return DSV4_OK;
    if (!k || !req_rows || !positions) return DSV4_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(k) % 16) return DSV4_ERR_INVALID;
    unsigned int* err = device_error_word();
    if (!err) return DSV4_ERR_CUDA;
    StoreParams p;
    p.k = static_cast<const uint4*>(k);
    p.n = n;
    p.req_rows = req_rows;
    p.positions = positions;
    p.rows = static_cast<uint8_t*>(const_cast<void*>(pool->rows));
    p.num_pages = pool->num_pages;
    p.row_bytes = pool->row_bytes;
    p.page_table = pool->page_table;
    p.pt_rows = pool->page_table_rows;
    p.pt_stride = pool->page_table_stride;
    p.err = err;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    constexpr int kRowsPerBlock = kStoreWarps * kStoreRowsPerWarp;
    cfg.gridDim = dim3(static_cast<unsigned>((n + kRowsPerBlock - 1) / kRowsPerBlock), 1, 1);
    cfg.blockDim = dim3(kStoreWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t le = pool->format == DSV4_KV_BF16
                               ? cudaLaunchKernelEx(&cfg, dsv4_kv_store_kernel<DSV4_KV_BF16, kStoreRowsPerWarp>, p)
                               : cudaLaunchKernelEx(&cfg, dsv4_kv_store_kernel<DSV4_KV_FP8_PACKED, kStoreRowsPerWarp>, p);
    if (le != cudaSuccess) {
        cudaGetLastError();
        return DSV4_ERR_CUDA;
    }
    return DSV4_OK;
}
