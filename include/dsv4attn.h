/*
 * dsv4attn.h - C ABI of the GB300 (sm_103a) hybrid sparse MQA attention step
 * used by DeepSeek-V4 decode and target-verify.
 *
 * What one call computes, for every packed query token t with H query heads
 * that share one 512-wide KV head (K and V are the same row):
 *
 *   keys(t) = window(t) ++ extra(t)
 *   s_j     = scale * <q[t,h,:], k_j>
 *   L       = exp(sink[h]) + sum_j exp(s_j)
 *   out     = sum_j exp(s_j) k_j / L         lse = ln L
 *
 * window(t): positions max(0, p-window+1) .. p of the token's request, read
 *   from the paged SWA pool (the current token is already in the cache).
 * extra(t):  compress ratio 4 (C4): the token's given list of top-k
 *   compressed-row indices; ratio 128 (C128): every compressed row the token
 *   can see; ratio 0: none.  A token at position p sees n_c(p) = (p+1)/ratio
 *   compressed rows.
 *
 * Sources (page title, section):
 *   "SGLang DeepSeek-V4 Attention Test Capability Matrix" - "Input And Config
 *     Coverage" (head_dim 512 = 448 nope + 64 rope, page_size 256, SWA window
 *     128, packed FP8 nope + BF16 rope KV); "Reference Implementation Notes"
 *     (vanilla softmax over the gathered rows; the sink is a virtual key with
 *     a per-head score and a zero value); "Production-Unsupported" items 3-5
 *     (page_size must be 256, head_dim must be 512, compress_ratio must be
 *     one of 0, 4, 128).
 *   "DeepSeek-V4 Attention: Query, Cache Write and History Addressing" -
 *     section 1 (MQA, positions count from zero), section 3 (k is v, the
 *     current token is stored before attention), section 4 (req_pool_indices
 *     and the page table locate each request's history; cu_seqlens_q bounds
 *     the query rows of each request), section 5 (ratio 0 / 4 / 128).
 *   "DeepSeek-V4 and SGLang Day-0" - "What V4 changed" (SWA 128 + C4 top-512
 *     or C128 dense in every layer); kernel list (the FlashMLA interface
 *     that reads SWA and extra rows in one call).
 *
 * Conventions shared by every entry point
 *   Memory: every pointer is device memory owned by the caller (q, pools,
 *     page tables, index lists, sink, out, lse, workspace, debug_rows); the
 *     library allocates nothing and keeps no state besides a per-device
 *     cache of SM and occupancy figures.  Calls are asynchronous on `stream`
 *     (a cudaStream_t; NULL = legacy default stream).
 *   q:    bf16 [T, H, 512], row-major, contiguous.  1 <= H <= 128.
 *   out:  bf16 [T, H, 512], row-major, contiguous.
 *   lse:  fp32 [T, H] (natural log of the full denominator, sink included),
 *         may be NULL.
 *   sink: fp32 [H] raw logits (not multiplied by scale); -INFINITY disables.
 *   seq_lens: int32 [batch], length of each request including the newest
 *         token(s).  req_pool_indices: int32 [batch] page-table row of each
 *         request, or NULL for row b = request b.
 *   scale: softmax scale applied to q.k (1/sqrt(512) for DeepSeek-V4).
 *   num_splits: 0 lets the library choose; otherwise the key list of each
 *         token is cut into this many pieces (split-KV), merged by a
 *         log-sum-exp combine.  Results do not depend on it beyond rounding.
 *   workspace: device scratch of at least dsv4_attn_workspace_size(...)
 *         bytes for the chosen split plan (may be NULL when that size is 0).
 *   debug_rows: NULL, or int32 [T, debug_stride] that receives, for every
 *         token, the physical pool row read for each key slot in slot order
 *         (window slots, then extra slots), -1 for a skipped slot.
 *         debug_stride = window + (ratio 4: topk; ratio 128:
 *         max_seq_len/128; ratio 0: 0).
 *
 * Errors
 *   Return value: DSV4_OK, or a negative DSV4_ERR_* for a host-side check
 *   that failed (nothing was launched).  Device-side problems never trap: a
 *   page id outside the pool, an index past n_c(p), an inconsistent position
 *   or a list longer than the plan covers skips that key slot (or token) and
 *   ORs a DSV4_DEV_ERR_* bit into a per-device error word that
 *   dsv4_attn_get_device_error() reads and clears.
 */
#ifndef DSV4ATTN_H
#define DSV4ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (return values) ---- */
#define DSV4_OK                 0
#define DSV4_ERR_INVALID      (-1)  /* null pointer, H outside 1..128, T/batch < 1, bad stride */
#define DSV4_ERR_UNSUPPORTED  (-2)  /* page_size != 256, ratio not 0/4/128, row_bytes mis-sized, or
                                       more than 2^31 - 1 CTAs (tokens x key slices x 64-head groups) */
#define DSV4_ERR_WORKSPACE    (-3)  /* workspace smaller than dsv4_attn_workspace_size() */
#define DSV4_ERR_CUDA         (-4)  /* a CUDA runtime call or launch failed */
#define DSV4_ERR_SCRATCH_LIMIT (-5) /* dsv4_attn_c4_sparse_noalloc: the call needs more scratch than
                                       the library's built-in DSV4_NOALLOC_SCRATCH_BYTES */

/* ---- device error bits (dsv4_attn_get_device_error) ---- */
#define DSV4_DEV_ERR_SWA_PAGE     0x01u  /* window row on a page id outside the SWA pool */
#define DSV4_DEV_ERR_EXTRA_PAGE   0x02u  /* compressed row on a page id outside the extra pool */
#define DSV4_DEV_ERR_INDEX_RANGE  0x04u  /* C4 index >= n_c(p) (negative indices are absent slots) */
#define DSV4_DEV_ERR_POSITION     0x08u  /* token position < 0 or cu_seqlens_q inconsistent */
#define DSV4_DEV_ERR_PLAN         0x10u  /* key list longer than the split plan covers (max_seq_len too small) */
#define DSV4_DEV_ERR_TIMEOUT      0x20u  /* an internal pipeline wait gave up (library bug) */
#define DSV4_DEV_ERR_REQ_ROW      0x40u  /* req_pool_indices entry outside the page table */
#define DSV4_DEV_ERR_STORE_ROW    0x80u  /* dsv4_kv_store (dsv4kvstore.h): a row whose request row,
                                            logical page or page id is outside the tables or the pool */
#define DSV4_DEV_ERR_TOPK_LENGTH  0x100u /* dsv4_topk (dsv4topk.h): a length outside 0..max_length */

/* ---- KV pool formats ---- */
#define DSV4_KV_BF16        0   /* row = 512 bf16 (1024 bytes) */
#define DSV4_KV_FP8_PACKED  1   /* row = [448 e4m3][64 bf16][7 fp32 scales], stride 608 bytes:
                                   nope[d] = e4m3(byte d) * scale[d/64] */

/* A paged KV pool: num_pages pages of page_size rows each, rows stored
   back to back at row_bytes stride.  page_table[r * page_table_stride + lp]
   is the physical page of logical page lp of request row r (a logical page
   holds page_size consecutive positions / compressed rows). */
typedef struct dsv4_kv_pool {
    const void*    rows;               /* device, num_pages * page_size rows */
    int64_t        num_pages;
    int32_t        row_bytes;          /* 1024 (BF16) or 608 (FP8_PACKED) */
    int32_t        format;             /* DSV4_KV_BF16 or DSV4_KV_FP8_PACKED */
    const int32_t* page_table;         /* device int32 [page_table_rows, page_table_stride] */
    int32_t        page_table_rows;
    int32_t        page_table_stride;  /* logical pages per request row */
    int32_t        page_size;          /* must be 256 */
} dsv4_kv_pool;

/* SWA-only decode (compress ratio 0).  T = batch; token b sits at position
   seq_lens[b]-1 of request b. */
int dsv4_attn_swa(const void* q, int32_t batch, int32_t num_heads,
                  const int32_t* seq_lens, const int32_t* req_pool_indices,
                  const dsv4_kv_pool* swa, int32_t window,
                  const float* sink, float scale,
                  void* out, float* lse,
                  int32_t num_splits, void* workspace, size_t workspace_bytes,
                  int32_t* debug_rows, void* stream);

/* C4 decode: window plus the token's top-k compressed rows.  topk_idx is
   int32 [batch, topk]: logical compressed-row numbers of the token's request
   (< n_c(p)); negative entries are absent slots.  Both pools use the same
   req_pool_indices row. */
int dsv4_attn_c4_sparse(const void* q, int32_t batch, int32_t num_heads,
                        const int32_t* seq_lens, const int32_t* req_pool_indices,
                        const dsv4_kv_pool* swa, int32_t window,
                        const dsv4_kv_pool* extra,
                        const int32_t* topk_idx, int32_t topk,
                        const float* sink, float scale,
                        void* out, float* lse,
                        int32_t num_splits, void* workspace, size_t workspace_bytes,
                        int32_t* debug_rows, void* stream);

/* C128 decode: window plus every visible compressed row (n_c(p) of them).
   max_seq_len bounds seq_lens (it sizes the split plan). */
int dsv4_attn_c128_dense(const void* q, int32_t batch, int32_t num_heads,
                         const int32_t* seq_lens, const int32_t* req_pool_indices,
                         const dsv4_kv_pool* swa, int32_t window,
                         const dsv4_kv_pool* extra, int32_t max_seq_len,
                         const float* sink, float scale,
                         void* out, float* lse,
                         int32_t num_splits, void* workspace, size_t workspace_bytes,
                         int32_t* debug_rows, void* stream);

/* Target-verify / draft-extend: request b owns query rows
   cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 (int32 [batch+1], cu_seqlens_q[0]
   = 0, T = cu_seqlens_q[batch] = num_tokens); they are its last qlen_b
   positions, so row i sits at seq_lens[b] - qlen_b + (i - cu_seqlens_q[b])
   and sees only keys up to its own position.  compress_ratio 0, 4 or 128
   selects the extra set as above (extra may be NULL for 0; topk_idx is
   int32 [num_tokens, topk] for 4; max_seq_len is needed for 128). */
int dsv4_attn_verify(const void* q, int32_t num_tokens, int32_t batch, int32_t num_heads,
                     const int32_t* seq_lens, const int32_t* cu_seqlens_q,
                     const int32_t* req_pool_indices,
                     const dsv4_kv_pool* swa, int32_t window,
                     int32_t compress_ratio, const dsv4_kv_pool* extra,
                     const int32_t* topk_idx, int32_t topk, int32_t max_seq_len,
                     const float* sink, float scale,
                     void* out, float* lse,
                     int32_t num_splits, void* workspace, size_t workspace_bytes,
                     int32_t* debug_rows, void* stream);

/* Same computation, arguments and results as dsv4_attn_c4_sparse, for callers
   that cannot allocate device memory themselves: code running where no
   allocator may be called (inside another library's hot loop, in a process
   whose memory is fully reserved up front, or from a runtime that only hands
   out pointers it owns).  There is no workspace argument: the scratch a
   split plan needs (the bf16 partial rows the slices of a cluster exchange,
   and with grid_splits > 1 the fp32 partial results the combine kernel
   merges) comes from a buffer inside this library, a static device array of
   DSV4_NOALLOC_SCRATCH_BYTES that every GPU which loads the library holds
   until the process exits.  This entry point has no counterpart on the
   source pages; it only changes where the scratch lives.
   - The first call on a device looks up the buffer's device address (one
     runtime query, no allocation); make that first call before any stream
     capture on that device.
   - Every call uses the same buffer: calls that can overlap on the GPU (on
     different streams without ordering between them) race and corrupt each
     other's results.  Nothing in the buffer needs to start at zero; each call
     writes every scratch byte it later reads.
   - A call whose split plan needs more than DSV4_NOALLOC_SCRATCH_BYTES returns
     DSV4_ERR_SCRATCH_LIMIT and launches nothing (dsv4_attn_workspace_size with
     the same shapes gives the amount a call needs); a failing plan query
     returns its own status.
   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
#define DSV4_NOALLOC_SCRATCH_BYTES (16u << 20)
int dsv4_attn_c4_sparse_noalloc(const void* q, int32_t batch, int32_t num_heads,
                                const int32_t* seq_lens, const int32_t* req_pool_indices,
                                const dsv4_kv_pool* swa, int32_t window,
                                const dsv4_kv_pool* extra,
                                const int32_t* topk_idx, int32_t topk,
                                const float* sink, float scale,
                                void* out, float* lse,
                                int32_t num_splits, int32_t* debug_rows, void* stream);

/* The split plan the library uses for these shapes on the current device
   (num_splits as passed to an entry point; 0 = automatic).  Writes the
   number of key-list pieces merged inside the attention launch by one
   thread-block cluster per token and 64-head group (1..8) and the number of
   such cluster results merged through the workspace by the combine kernel.
   Returns DSV4_OK or an error. */
int dsv4_attn_plan(int32_t num_tokens, int32_t num_heads, int32_t compress_ratio,
                   int32_t window, int32_t topk, int32_t max_seq_len, int32_t num_splits,
                   int32_t* cluster_splits, int32_t* grid_splits);

/* Bytes of workspace a call with these shapes needs (0 when the plan keeps
   every merge on chip).  Same arguments as dsv4_attn_plan. */
size_t dsv4_attn_workspace_size(int32_t num_tokens, int32_t num_heads, int32_t compress_ratio,
                                int32_t window, int32_t topk, int32_t max_seq_len,
                                int32_t num_splits);

/* Waits for `stream`, copies the current device's error word into *flags
   (DSV4_DEV_ERR_* bits accumulated since the last read) and clears it. */
int dsv4_attn_get_device_error(uint32_t* flags, void* stream);

/* Human-readable text for a status code. */
const char* dsv4_attn_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* DSV4ATTN_H */
