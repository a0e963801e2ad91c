/*
 * dsv4kvstore.h - C ABI of the KV cache write that comes before the hybrid
 * sparse MQA attention step: new key rows (512 bf16 values each, after RoPE)
 * stored into a paged pool, packed to FP8 when the pool holds packed rows.
 *
 * Sources (page title, section):
 *   "DeepSeek-V4 Attention: Query, Cache Write and History Addressing" -
 *     section 3 (the current token's shared KV representation is written
 *     into its SWA slot before the attention backend reads the cache);
 *     section 4 (req_pool_indices and the page table locate each request's
 *     rows); section 5 (the C4 / C128 compressed rows live in their own
 *     pools).
 *   "SGLang DeepSeek-V4 Attention Test Capability Matrix" - "Input And
 *     Config Coverage" (the SWA cache holds packed FP8 nope + BF16 rope rows,
 *     584 bytes per token; page_size 256); "Reference Implementation Notes"
 *     (the production pack-and-store path fills the SWA and extra pools).
 *   The pages name the pack step but not its arithmetic; the one stated
 *   below (block scale amax / 448, e4m3 round to nearest even, fp32) is this
 *   library's reading of it.
 *
 * What one call does, for i = 0 .. n-1 with r = req_rows[i] and
 * l = positions[i]: row i of k goes to pool row
 *     page_table[r * page_table_stride + l / 256] * 256 + l % 256
 * (l is the token position for an SWA pool, the compressed-row number for a
 * C4 / C128 pool).
 *   DSV4_KV_BF16 pool: the 512 bf16 values, unchanged.
 *   DSV4_KV_FP8_PACKED pool: [448 e4m3 codes][64 bf16][7 fp32 scales][4 zero
 *     bytes].  For nope block b (values 64 b .. 64 b + 63): amax = max |x|,
 *     scale[b] = amax / 448 in fp32 (1 when amax is 0); code d = the e4m3
 *     value nearest to x_d / scale[d / 64] computed in fp32 (ties to even,
 *     saturating at +-448).  The 64 rope values keep their bf16 bits.
 *     Values must be finite.
 * Rows that no other index of the same call addresses are written exactly
 * once; when two indices address the same pool row, one of them wins.
 *
 * Arguments (all device memory owned by the caller; asynchronous on stream):
 *   k:         bf16 [n, 512], contiguous, 16-byte aligned.
 *   n:         number of rows (0 = nothing to do).
 *   req_rows:  int32 [n], page-table row of each row's request
 *              (req_pool_indices[b] of its request).
 *   positions: int32 [n], logical row number of each row.
 *   pool:      the destination; its rows are written through pool->rows.
 *   stream:    a cudaStream_t (NULL = legacy default stream).
 *
 * Errors: returns DSV4_OK, DSV4_ERR_INVALID (n < 0, a null or misaligned
 * pointer, a bad pool descriptor) or DSV4_ERR_UNSUPPORTED (page size other
 * than 256, row size that does not match the format) before launching
 * anything, or DSV4_ERR_CUDA.  On the device, a row whose request row,
 * logical page or page id falls outside the page table or the pool is not
 * written and sets DSV4_DEV_ERR_STORE_ROW in the error word that
 * dsv4_attn_get_device_error() reads and clears.
 */
#ifndef DSV4KVSTORE_H
#define DSV4KVSTORE_H

#include <stdint.h>

#include "dsv4attn.h"

#ifdef __cplusplus
extern "C" {
#endif

int dsv4_kv_store(const void* k, int32_t n, const int32_t* req_rows, const int32_t* positions,
                  const dsv4_kv_pool* pool, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSV4KVSTORE_H */
