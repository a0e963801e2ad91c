/*
 * dsv4topk.h - C ABI of the top-k index selection that produces the C4 index
 * lists of the hybrid sparse MQA attention step: for every query token, the
 * indices of the k best of its indexer scores.
 *
 * Sources (page title, section): "DeepSeek-V4 and SGLang Day-0" - kernel
 * list (at 1M context the indexer keeps the top 512 of 256K candidate
 * compressed rows; a radix select over a thread-block cluster replaces a
 * global sort); "DeepSeek-V4 Attention: Query, Cache Write and History
 * Addressing" - section 5 (the indexer's top-k indices limit which C4
 * compressed rows a token reads).  The pages do not fix the order of the
 * result or how equal scores are broken; the rules below are this library's
 * reading.
 *
 * What one call computes, for each row r (one query token) with
 * n = lengths[r] candidates scores[r * row_stride + 0 .. n - 1] (fp32):
 *   the k candidates ranked first by value (higher first; -0.0 ranks below
 *   +0.0; equal values: the lower index first), written to
 *   out_idx[r * k + 0 .. k - 1] as indices in ascending order, followed by
 *   -1 entries when n < k.  The result is unique.  Scores must be finite.
 *
 * Arguments (device memory owned by the caller; asynchronous on stream):
 *   scores:     fp32 [num_rows, row_stride], row_stride a multiple of 4,
 *               16-byte aligned.
 *   lengths:    int32 [num_rows], 0 <= lengths[r] <= max_length.
 *   max_length: bound on lengths (sizes the launch); at most
 *               dsv4_topk_max_length(k) (524288).
 *   k:          1 .. 1024.
 *   out_idx:    int32 [num_rows, k].
 *   stream:     a cudaStream_t (NULL = legacy default stream).
 * The call needs no scratch memory: each row is held on chip by one
 * thread-block cluster.
 *
 * Errors: DSV4_OK; DSV4_ERR_INVALID (null or misaligned pointer, num_rows
 * outside 1..65535, k outside 1..1024, max_length < 0, row_stride <
 * max_length or not a multiple of 4), DSV4_ERR_UNSUPPORTED (max_length above
 * dsv4_topk_max_length(k)), DSV4_ERR_CUDA.  On the device, a length outside
 * 0..max_length is clamped into it and sets DSV4_DEV_ERR_TOPK_LENGTH in the
 * error word read by dsv4_attn_get_device_error().
 */
#ifndef DSV4TOPK_H
#define DSV4TOPK_H

#include <stddef.h>
#include <stdint.h>

#include "dsv4attn.h"

#ifdef __cplusplus
extern "C" {
#endif

int32_t dsv4_topk_max_length(int32_t k);
int dsv4_topk(const float* scores, int32_t num_rows, int64_t row_stride, const int32_t* lengths,
              int32_t max_length, int32_t k, int32_t* out_idx, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSV4TOPK_H */
