/*
 * kvc.h -- C ABI of the GB300 persistent KV-cache library (libkvc.so).
 *
 * One step of the hot path appends new key/value rows to a persistent cache
 * and runs grouped-query attention (GQA) over it:
 *
 *     kvc_seq_lengths      lengths derived on the device from seqlens_k
 *     kvc_window_append    append (contiguous cache), in-place compaction +
 *                          append (windowed cache, one token), or C + S
 *                          staging seed / copy-back (windowed, several tokens)
 *     kvc_gqa_decode       one-token GQA attention over the cache
 *     kvc_gqa_decode_ring  the same over a ring of C slots (circular addressing)
 *     kvc_window_append_inplace  the staging step with the stage in the cache's rows
 *     kvc_paged_append, kvc_gqa_decode_paged  append and decode on a paged cache
 *     kvc_quantize_pages, kvc_gqa_decode_paged_q  int8 pages and decode over
 *                          a cache of 16-bit and int8 pages
 *     kvc_decode_step      lengths + append + decode in one launch (contiguous
 *                          cache or ring)
 *     kvc_window_decode_step  the same for a windowed cache
 *     kvc_gqa_prefill_chunk  multi-token GQA attention over staged rows
 *     kvc_window_prefill_step  a windowed multi-token step that stages only
 *                          the rows whose eviction its chunk would see
 *     kvc_tensor_scatter   the ONNX TensorScatter cache update (linear/circular)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  * Ownership: the caller owns every buffer.  The library allocates nothing,
 *    keeps no state between calls (apart from cached device attributes and
 *    the scratch array of kvc_gqa_decode_noalloc) and never reads device
 *    memory on the host, so the calls listed above can be captured in a CUDA
 *    graph.  Pointers marked "device" must be device (or managed)
 *    memory of the current device; pointers marked "host" are read during
 *    the call only.
 *  * Streams: `stream` is a cudaStream_t (NULL = legacy default stream).  Work
 *    is enqueued, never waited for.
 *  * Layout: caches and staging buffers are BNSH: [batch, kv_heads, rows, D],
 *    row-major, rows of D contiguous elements.  Queries and outputs are
 *    [batch, q_heads, new_tokens, D].  Query head h reads KV head
 *    h / (q_heads / kv_heads).
 *  * Errors: arguments are validated on the host before any launch and a
 *    non-zero kvc_status is returned with nothing enqueued.  Errors that
 *    depend on device data (an index out of range, a bad seqlens_k, a RoPE
 *    position beyond the cos/sin cache) are OR-ed into the caller's device
 *    word `dev_status` (may be NULL) as KVC_DEV_* bits, and the offending
 *    batch row writes nothing.  A failed launch returns KVC_ERR_CUDA.
 *  * Element types: KVC_F32, KVC_BF16, KVC_F16.  Attention accumulates in
 *    fp32 and rounds the output to nearest-even in the input type.
 *
 * Sources (page title, section):
 *   "TensorScatter" operator page (ai.onnx, since version 24): spec,
 *     pseudocode, examples.
 *   "GQA support sliding_window_cache" (onnxruntime pull request 29904):
 *     section "Design" (windowed invariant, append formula, device-side
 *     lengths, C + S staging) and the follow-up commits (int64 widening,
 *     RoPE bounded by the cos/sin cache length, not by the capacity).
 *   "Persistent KV Cache and Decode Performance Roadmap", section "Phase 1"
 *     (streaming decode with online softmax, GQA heads sharing a KV block,
 *     split of one query row across workers with an (m, l, o) merge).
 *   "Stateful decode & KV cache", section "Sliding-window ring buffer"
 *     (RoPE baked into K at write time; the mask depends on positions only).
 *   "Persistent KV Cache and Decode Performance Roadmap", "Phase 2" and the
 *     CPU backend's "fixed-size paged blocks and a page-table iterator
 *     consumed directly by Attention" (the paged calls).
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVC_ABI_VERSION 7

typedef enum {
    KVC_OK = 0,
    KVC_ERR_NULL = 1,        /* a required pointer is NULL                       */
    KVC_ERR_SHAPE = 2,       /* a size is out of range or buffers overlap badly  */
    KVC_ERR_DTYPE = 3,       /* element type not supported by this entry point   */
    KVC_ERR_ALIGN = 4,       /* a buffer is not 16-byte aligned where required   */
    KVC_ERR_UNSUPPORTED = 5, /* a valid combination the library does not cover   */
    KVC_ERR_CAPACITY = 6,    /* capacity < 1 or too small for the request        */
    KVC_ERR_WINDOW = 7,      /* windowed cache needs 0 < local_window_size <= C  */
    KVC_ERR_WORKSPACE = 8,   /* workspace NULL or smaller than required          */
    KVC_ERR_CUDA = 9         /* a CUDA call failed (launch or driver)            */
} kvc_status;

typedef enum { KVC_F32 = 0, KVC_BF16 = 1, KVC_F16 = 2 } kvc_dtype;
typedef enum { KVC_LINEAR = 0, KVC_CIRCULAR = 1 } kvc_mode;
typedef enum { KVC_APPEND = 0, KVC_COPY_BACK = 1 } kvc_phase;
/* How the resident rows of a cache follow the absolute length T (the
 * `windowed` argument of the calls below). */
typedef enum {
    KVC_CONTIGUOUS = 0, /* every token stays: rows [0, T), T <= C               */
    KVC_WINDOWED = 1,   /* the last min(T, C) tokens; compaction on every step
                           once the cache is full                              */
    KVC_DRIFTING = 2,   /* the last end(T) tokens, W <= end(T) <= C: compaction
                           reclaims C - W + 1 rows at once, every C - W + 1
                           one-token steps                                     */
    KVC_RING = 3        /* a ring of C slots: token p lives in slot p mod C and
                           nothing ever moves ("Stateful decode & KV cache",
                           "Sliding-window ring buffer")                       */
} kvc_cache_policy;

/* device status bits (OR-ed into *dev_status) */
#define KVC_DEV_INDEX_OOB 1u    /* TensorScatter linear: wi < 0 or wi + S > max_seq    */
#define KVC_DEV_SEQLEN_RANGE 2u /* seqlens_k + 1 < new_tokens, or >= 2^31             */
#define KVC_DEV_CAPACITY 4u     /* contiguous cache: seqlens_k + 1 > capacity          */
#define KVC_DEV_ROPE_RANGE 8u   /* an absolute position >= rope_max_pos                */
#define KVC_DEV_TIMEOUT 16u     /* a bounded wait inside a kernel gave up              */

/*
 * Per-batch lengths, five device int32 arrays of [batch] each, written by
 * kvc_seq_lengths and read by the other calls ("GQA support
 * sliding_window_cache", "Design": absolute lengths for RoPE, cache-relative
 * lengths for addressing, and the evict count).  A rejected row holds -1 in
 * all five.
 *   past_abs    P  = T - S        absolute tokens before this step
 *   total_abs   T  = seqlens_k+1  absolute tokens after this step
 *   cache_past  Lp                rows resident before the step
 *   cache_total L                 rows resident after the step
 *   evict       E                 rows evicted by the step
 */
typedef struct {
    int32_t *past_abs;
    int32_t *total_abs;
    int32_t *cache_past;
    int32_t *cache_total;
    int32_t *evict;
} kvc_lengths;

/*
 * kvc_tensor_scatter -- ONNX TensorScatter ("TensorScatter" operator page,
 * opset 24: spec and pseudocode).
 *
 * present_cache  device, shape cache_shape, elem_bytes per element.
 * past_cache     device, same shape.  present_cache == past_cache runs in
 *                place (only the updated rows move); distinct buffers run the
 *                functional form (every row of present is written once, from
 *                update or from past).  Partially overlapping buffers ->
 *                KVC_ERR_SHAPE.
 * update         device, cache_shape with dimension `axis` = update_seq_len.
 * write_indices  device int64 [cache_shape[0]], or NULL (all zeros).
 * rank           2..8; cache_shape is a HOST array of `rank` sizes.
 * axis           sequence axis, != 0 (negative counts from the end; the
 *                operator's default is -2).
 * mode           KVC_LINEAR: row b writes [wi, wi + S); wi < 0 or
 *                wi + S > max_seq sets KVC_DEV_INDEX_OOB and leaves row b of
 *                present equal to past.  KVC_CIRCULAR: index mod max_seq
 *                (floor modulo, so negative wi wraps).
 * update_seq_len 0..max_seq (a longer update is a shape error).
 * elem_bytes     1, 2, 4 or 8: rows are copied as bytes, any element type.
 */
kvc_status kvc_tensor_scatter(void *present_cache, const void *past_cache, const void *update,
                              const int64_t *write_indices, int rank, const int64_t *cache_shape,
                              int64_t update_seq_len, int axis, int mode, int elem_bytes,
                              int32_t *dev_status, void *stream);

/*
 * kvc_seq_lengths -- derive the five length arrays on the device ("GQA
 * support sliding_window_cache", "Design"; int64 arithmetic per the PR's
 * widening commit).  T = seqlens_k[b] + 1 computed in 64 bits, P = T - S.
 *   KVC_WINDOWED, KVC_RING:
 *                   Lp = min(P, C), E = max(0, Lp + S - C), L = Lp - E + S
 *                   (for a ring: slots holding a token before / after the
 *                   step, and old tokens the step overwrites)
 *   KVC_DRIFTING:   Lp = end(P), L = end(T), E = Lp + S - L, where (the PR's
 *                   CPU commit, "drifting layout") gap = C - W + 1 and
 *                   end(T) = T for T <= C, else T - gap * ceil((T - C) / gap)
 *   KVC_CONTIGUOUS: Lp = P, E = 0, L = T; T > C sets KVC_DEV_CAPACITY.
 * T < S or T >= 2^31 sets KVC_DEV_SEQLEN_RANGE.  A rejected row gets -1 in
 * every array.
 * seqlens_k        device int32 [batch].
 * new_tokens       S >= 1.
 * capacity         C >= 1 rows per head.
 * windowed         a kvc_cache_policy (other values: KVC_ERR_UNSUPPORTED).
 * local_window_size  windowed, drifting or ring cache: must satisfy 0 < W <= C
 *                  (KVC_ERR_WINDOW otherwise); ignored for a contiguous cache.
 */
kvc_status kvc_seq_lengths(const int32_t *seqlens_k, int batch, int new_tokens, int64_t capacity,
                           int windowed, int local_window_size, kvc_lengths out,
                           int32_t *dev_status, void *stream);

/*
 * kvc_window_append -- write S new K/V rows per (batch, kv head) ("GQA
 * support sliding_window_cache", "Design").  K rows are rotated (RoPE,
 * rotate-half pairs (i, i + D/2), float32 with every product and sum
 * rounded separately) at their ABSOLUTE position P + i before they are
 * stored; V rows are stored as given.
 *
 * k_cache, v_cache  device [batch, kv_heads, capacity, head_dim].
 * new_k, new_v      device [batch, kv_heads, new_tokens, head_dim].
 * k_stage, v_stage  device [batch, kv_heads, capacity + new_tokens, head_dim]
 *                   for a windowed cache with S > 1, else ignored (may be NULL).
 * len               outputs of kvc_seq_lengths for the same S and C.
 * windowed          a kvc_cache_policy; KVC_WINDOWED and KVC_DRIFTING append
 *                   alike (what differs is in `len`) and are called
 *                   "windowed" below.  KVC_RING: row i goes to slot
 *                   (P + i) mod C for any S, nothing moves and no stage is
 *                   used (when S > C only the last C rows are written, the
 *                   ones that would survive); phase must be KVC_APPEND.
 * phase = KVC_APPEND:
 *   contiguous cache:      rows [P, P + S) of the cache.
 *   windowed, S == 1:      in place: rows [E, Lp) move to [0, Lp - E)
 *                          (E <= 1 for KVC_WINDOWED, 0 or C - W + 1 for
 *                          KVC_DRIFTING), then the new row goes to Lp - E.
 *   windowed, S > 1:       seeds the stage: stage[0, Lp) = cache[0, Lp),
 *                          stage[Lp + i] = new row i.  Attention then runs on
 *                          the stage (kvc_gqa_prefill_chunk).
 * phase = KVC_COPY_BACK (windowed, S > 1 only):
 *                          cache[0, L) = stage[E, Lp + S).
 * rope_cos, rope_sin  device float32 [rope_max_pos, head_dim / 2] indexed by
 *                   absolute position, or both NULL for no rotation.  A row
 *                   with P + S > rope_max_pos sets KVC_DEV_ROPE_RANGE and is
 *                   not written.
 * head_dim          even, 2..1024; dtype KVC_F32/KVC_BF16/KVC_F16.
 */
kvc_status kvc_window_append(void *k_cache, void *v_cache, const void *new_k, const void *new_v,
                             void *k_stage, void *v_stage, kvc_lengths len, int batch,
                             int kv_heads, int new_tokens, int64_t capacity, int head_dim,
                             int dtype, int windowed, int phase, const float *rope_cos,
                             const float *rope_sin, int64_t rope_max_pos, int32_t *dev_status,
                             void *stream);

/*
 * kvc_window_append_inplace -- the C + S staging step of a windowed cache
 * with the stage held in the cache's own rows ("GQA support
 * sliding_window_cache", "Design": a step with S new tokens attends over the
 * cached rows and the new ones, then keeps the last positions; here the stage
 * is not a second buffer).  The cache lives in rows [0, Lp) of a buffer with
 * rows_per_head >= capacity + new_tokens rows per head, so the rows a stage
 * would hold are already in place and no seed copy is made.
 *
 * k_rows, v_rows  device [batch, kv_heads, rows_per_head, head_dim]; rows
 *                 [0, Lp) hold the cache (Lp = len.cache_past).  Other calls
 *                 that read this cache take rows_per_head as their row pitch
 *                 (their `capacity` argument), while kvc_seq_lengths takes the
 *                 cache's capacity C.
 * new_k, new_v    device [batch, kv_heads, new_tokens, head_dim].
 * len             outputs of kvc_seq_lengths for the same S and C.
 * windowed        KVC_WINDOWED or KVC_DRIFTING.
 * phase = KVC_APPEND:     rows [Lp, Lp + S) <- the new rows (K rotated at
 *                         P + i, as kvc_window_append).  Attention then runs
 *                         on these rows (kvc_gqa_prefill_chunk with this
 *                         rows_per_head).
 * phase = KVC_COPY_BACK:  rows [0, L) <- rows [E, Lp + S), moved in place
 *                         (one CTA per (batch, kv head, K/V) walks the range
 *                         in ascending chunks, so every row is read before it
 *                         is overwritten).  Rows [0, L) are then byte for byte
 *                         what kvc_window_append's staged pair leaves in a
 *                         cache of `capacity` rows; rows past L are scratch.
 * A row rejected by kvc_seq_lengths (lengths -1) or for its RoPE range is left
 * untouched by both phases (KVC_DEV_ROPE_RANGE as kvc_window_append).
 * head_dim * element size a multiple of 16 bytes (KVC_ERR_UNSUPPORTED);
 * buffers 16-byte aligned; rows_per_head < capacity + new_tokens ->
 * KVC_ERR_CAPACITY.
 */
kvc_status kvc_window_append_inplace(void *k_rows, void *v_rows, const void *new_k,
                                     const void *new_v, kvc_lengths len, int batch, int kv_heads,
                                     int new_tokens, int64_t capacity, int64_t rows_per_head,
                                     int head_dim, int dtype, int windowed, int phase,
                                     const float *rope_cos, const float *rope_sin,
                                     int64_t rope_max_pos, int32_t *dev_status, void *stream);

/*
 * kvc_gqa_decode -- one-token grouped-query attention over the cache after
 * the append ("Persistent KV Cache and Decode Performance Roadmap", Phase 1:
 * streaming online softmax, a KV block read once per query-head group, a
 * split of long rows across CTAs merged by (m, l, o); masks from "GQA support
 * sliding_window_cache").
 *
 * For batch row b: rows [0, L) of each head (L = len.cache_total[b]) hold
 * absolute positions T - L + r (T = len.total_abs[b]); the query is at
 * T - 1 and is rotated there when rope tables are given.  Row r is visible
 * iff local_window_size <= 0 or (T - 1) - pos(r) < local_window_size.
 *
 * out, q        device [batch, q_heads, 1, head_dim], same dtype as the cache.
 * k_cache/v_cache device [batch, kv_heads, capacity, head_dim].
 * scale         0 -> 1/sqrt(head_dim).
 * workspace     device scratch of kvc_gqa_decode_workspace_size(...) bytes
 *               (holds per-split partial (m, l, o)); 256-byte aligned.
 * Supported: KVC_BF16/KVC_F16 with head_dim in {64, 128, 256} and
 * q_heads / kv_heads <= 16 (tensor-core path); KVC_F32 with head_dim <= 256.
 * All buffers 16-byte aligned (KVC_ERR_ALIGN).
 */
kvc_status kvc_gqa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                          kvc_lengths len, int batch, int q_heads, int kv_heads, int64_t capacity,
                          int head_dim, int dtype, int local_window_size, float scale,
                          const float *rope_cos, const float *rope_sin, int64_t rope_max_pos,
                          void *workspace, size_t workspace_bytes, int32_t *dev_status,
                          void *stream);

/* Bytes of workspace kvc_gqa_decode needs for these sizes (0 on bad sizes). */
size_t kvc_gqa_decode_workspace_size(int batch, int q_heads, int kv_heads, int64_t capacity,
                                     int head_dim, int dtype);

/* Size of the library's own decode scratch array (see kvc_gqa_decode_noalloc). */
#define KVC_DECODE_STATIC_SCRATCH_BYTES (16u << 20)

/*
 * kvc_gqa_decode_noalloc -- kvc_gqa_decode for callers that cannot allocate
 * device memory.  The source pages have no counterpart of this call; it is a
 * convenience of this library.
 *
 * Who needs it: code that runs where it has no device allocator to call, or
 * is not allowed to use one -- for example a plugin or operator inside a host
 * framework that owns all device memory through its own pool and gives its
 * kernels no way to request scratch, or a caller that has sized its memory
 * up front and must not grow it while serving.  Such a caller still owns and
 * passes every input and output; only the decode's split partials (the
 * workspace of kvc_gqa_decode) move into memory the library provides.
 *
 * The scratch is one file-scope device array of
 * KVC_DECODE_STATIC_SCRATCH_BYTES (16 MiB) that every device loading the
 * library keeps until the process exits.  Sizes whose workspace
 * (kvc_gqa_decode_workspace_size) exceeds it are rejected with
 * KVC_ERR_WORKSPACE before anything is enqueued.  The call itself allocates
 * nothing: no cudaMalloc, cudaFree or allocating library routine.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  All calls share the one array and it keeps the
 * previous call's contents: nothing in it needs to start at zero (every
 * partial is written before it is read within a call), but two calls whose
 * kernels overlap on the GPU -- on different streams, or different threads
 * -- race on it and may return wrong results.  Serialise them (one stream,
 * or events).
 *
 * Arguments, layouts, supported sizes and errors are those of
 * kvc_gqa_decode without the workspace pair.
 */
kvc_status kvc_gqa_decode_noalloc(void *out, const void *q, const void *k_cache,
                                  const void *v_cache, kvc_lengths len, int batch, int q_heads,
                                  int kv_heads, int64_t capacity, int head_dim, int dtype,
                                  int local_window_size, float scale, const float *rope_cos,
                                  const float *rope_sin, int64_t rope_max_pos,
                                  int32_t *dev_status, void *stream);

/*
 * kvc_gqa_decode_ring -- kvc_gqa_decode over a ring of C slots ("Stateful
 * decode & KV cache", "Sliding-window ring buffer"; the ring written by
 * kvc_window_append(KVC_RING) or by kvc_tensor_scatter in KVC_CIRCULAR mode
 * at write index P): slot r holds position T - 1 - ((T - 1 - r) mod C).  The
 * query at T - 1 sees the newest n = min(L, W) positions (n = L when
 * local_window_size <= 0), where L = len.cache_total[b] (min(T, C) from
 * kvc_seq_lengths) and T = len.total_abs[b]; they occupy slots
 * (T - n) mod C onwards, wrapping at C.  Equal to kvc_gqa_decode over the
 * full history whenever W <= C.  Arguments, layouts, supported sizes,
 * workspace and errors are those of kvc_gqa_decode.
 */
kvc_status kvc_gqa_decode_ring(void *out, const void *q, const void *k_cache, const void *v_cache,
                               kvc_lengths len, int batch, int q_heads, int kv_heads,
                               int64_t capacity, int head_dim, int dtype, int local_window_size,
                               float scale, const float *rope_cos, const float *rope_sin,
                               int64_t rope_max_pos, void *workspace, size_t workspace_bytes,
                               int32_t *dev_status, void *stream);

/*
 * Paged cache ("Persistent KV Cache and Decode Performance Roadmap", Phase 2:
 * fixed-size pages read through a page table, never gathered into one
 * contiguous cache).  K and V live in page pools [n_pool_pages, kv_heads,
 * page_size, head_dim] (one page holds page_size consecutive tokens of every
 * KV head).  block_table is device int32 [batch, max_pages]: logical row r of
 * batch row b is slot r % page_size of page block_table[b * max_pages +
 * r / page_size].  The caller allocates the pages (the table entries a step
 * touches must name pages of the pool); the lengths are those of a
 * contiguous cache of capacity max_pages * page_size (kvc_seq_lengths with
 * KVC_CONTIGUOUS).
 *
 * kvc_paged_append -- write the S new rows (K rotated at P + i as in
 * kvc_window_append) at logical rows [P, P + S).  A row whose new tokens
 * would land in a page id outside [0, n_pool_pages) sets KVC_DEV_INDEX_OOB
 * and writes nothing.  Any even head_dim <= 1024; all dtypes.
 */
kvc_status kvc_paged_append(void *k_pool, void *v_pool, const void *new_k, const void *new_v,
                            const int32_t *block_table, int max_pages, int64_t n_pool_pages,
                            int page_size, kvc_lengths len, int batch, int kv_heads,
                            int new_tokens, int head_dim, int dtype, const float *rope_cos,
                            const float *rope_sin, int64_t rope_max_pos, int32_t *dev_status,
                            void *stream);

/*
 * kvc_gqa_decode_paged -- kvc_gqa_decode over a paged cache: the split
 * kernel streams 64-row tiles straight from the pages (page_size must be a
 * positive multiple of 64, so that no tile straddles two pages).  A page id
 * outside the pool sets KVC_DEV_INDEX_OOB; that row's output is then
 * undefined.  Workspace: kvc_gqa_decode_workspace_size(batch, q_heads,
 * kv_heads, max_pages * page_size, head_dim, dtype).  Supported:
 * KVC_BF16/KVC_F16, head_dim in {64, 128, 256}, q_heads / kv_heads <= 16.
 */
kvc_status kvc_gqa_decode_paged(void *out, const void *q, const void *k_pool,
                                const void *v_pool, const int32_t *block_table, int max_pages,
                                int64_t n_pool_pages, int page_size, kvc_lengths len, int batch,
                                int q_heads, int kv_heads, int head_dim, int dtype,
                                int local_window_size, float scale, const float *rope_cos,
                                const float *rope_sin, int64_t rope_max_pos, void *workspace,
                                size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * Quantized pages ("Persistent input/output feedback", "Optional
 * heterogeneous paged KV": selected-block affine quantization; "Persistent
 * KV Cache and Decode Performance Roadmap", "Phase 3": cold pages to INT8,
 * recent tokens kept in the native type).  Int8 pages live in pools
 * qk_pool, qv_pool [n_qpool_pages, kv_heads, page_size, head_dim] of bytes; a
 * block-table entry with KVC_PAGE_QUANT set names page
 * (entry & ~KVC_PAGE_QUANT) of these pools.  qparams is device float
 * [n_qpool_pages][4] = (k_scale, k_zp, v_scale, v_zp) per int8 page, so that
 * a stored byte u (unsigned) reconstructs as (u - zp) * scale.
 *
 * Payload order (the MMA fragment order of the decode): the page_size rows of
 * a (page, kv head) are cut into groups of 16; group G is 16 * head_dim
 * bytes at G * 16 * head_dim.  Within a group, with D = head_dim:
 *   K element (row j, column d):  nb = j / 8, g = j % 8, kk = d / 16,
 *     dd = d % 16, lane = 4 g + (dd % 8) / 2,
 *     f = (2 kk + dd / 8) * 4 + 2 nb + dd % 2
 *   V element (row j, column c):  mb = c / 16, cc = c % 16,
 *     lane = 4 (cc % 8) + (j % 8) / 2, f = (2 mb + j / 8) * 4 + 2 (cc / 8) + j % 2
 *   byte = (f / 16) * 512 + lane * 16 + f % 16
 * (lane l's D / 2 bytes are the A fragments of its mma.m16n8k16 steps --
 * the 16 rows are the MMA's M dimension, K as it is and V transposed --
 * stored as 16-byte pieces interleaved across the 32 lanes).
 */
#define KVC_PAGE_QUANT 0x40000000

/*
 * kvc_quantize_pages -- page src_pages[i] of the 16-bit pools (every row and
 * KV head) becomes int8 page dst_pages[i], for i < n_pages:
 *     code = saturate(round_half_even(x / scale) + zero_point)
 * with x / scale in float32, saturated to [-128, 127] (INT8) or [0, 255]
 * (UINT8: *_unsigned != 0); the stored byte is the unsigned code + 128 - bias
 * (bias 0 for INT8, 128 for UINT8: an INT8 code c is stored as c + 128, a
 * UINT8 code as itself) and qparams[dst] = (k_scale, k_zero_point + 128 -
 * k_bias, v_scale, v_zero_point + 128 - v_bias).  K and V may use different
 * formats.
 * k_pool, v_pool     device [n_pool_pages, kv_heads, page_size, head_dim],
 *                    KVC_BF16 or KVC_F16.
 * src_pages, dst_pages  device int32 [n_pages]; a pair with an id outside its
 *                    pool sets KVC_DEV_INDEX_OOB and is skipped.  Destinations
 *                    must be distinct.  The block table is not touched: the
 *                    caller points its entries at (dst | KVC_PAGE_QUANT).
 * Scales positive and finite, zero points inside the code range
 * (KVC_ERR_SHAPE otherwise); page_size a multiple of 16; head_dim a multiple
 * of 32.
 */
kvc_status kvc_quantize_pages(const void *k_pool, const void *v_pool, void *qk_pool,
                              void *qv_pool, const int32_t *src_pages, const int32_t *dst_pages,
                              int n_pages, int64_t n_pool_pages, int64_t n_qpool_pages,
                              int page_size, int kv_heads, int head_dim, int dtype, float k_scale,
                              int k_zero_point, int k_unsigned, float v_scale, int v_zero_point,
                              int v_unsigned, float *qparams, int32_t *dev_status, void *stream);

/*
 * kvc_gqa_decode_paged_q -- kvc_gqa_decode_paged over a cache whose pages are
 * 16-bit (entries naming the k_pool / v_pool pages) or int8 (entries with
 * KVC_PAGE_QUANT).  An int8 tile is read at half the bytes and its
 * reconstruction (u - zp) * scale enters the attention with the page's
 * scale applied in float32 after the products: scores = k_scale * q . (u - zp),
 * values = v_scale * sum p (u - zp).  An entry outside its pool sets
 * KVC_DEV_INDEX_OOB (that row's output is undefined).  Same arguments and
 * limits as kvc_gqa_decode_paged plus the int8 pools, qparams (16-byte
 * aligned) and n_qpool_pages.
 */
kvc_status kvc_gqa_decode_paged_q(void *out, const void *q, const void *k_pool,
                                  const void *v_pool, const void *qk_pool, const void *qv_pool,
                                  const float *qparams, int64_t n_qpool_pages,
                                  const int32_t *block_table, int max_pages, int64_t n_pool_pages,
                                  int page_size, kvc_lengths len, int batch, int q_heads,
                                  int kv_heads, int head_dim, int dtype, int local_window_size,
                                  float scale, const float *rope_cos, const float *rope_sin,
                                  int64_t rope_max_pos, void *workspace, size_t workspace_bytes,
                                  int32_t *dev_status, void *stream);

/*
 * kvc_decode_step -- one fused one-token step on a contiguous cache or a
 * ring: kvc_seq_lengths + kvc_window_append (S = 1) + kvc_gqa_decode (or
 * kvc_gqa_decode_ring) with the same results, the lengths, the append and
 * the attention in one launch ("Persistent KV Cache and Decode Performance
 * Roadmap", Phase 1; "GQA support sliding_window_cache", "Design";
 * "Stateful decode & KV cache", "Sliding-window ring buffer").  The CTA that
 * holds the newest position rotates the new K row at T - 1 and stores it and
 * the V row to the cache (row T - 1, or slot (T - 1) mod C) while its first
 * tiles are in flight, then places both in its last tile on chip.  Rows long
 * enough for several splits are merged by a second launch, as in
 * kvc_gqa_decode.
 *
 * out, q          device [batch, q_heads, 1, head_dim].
 * k_cache/v_cache device [batch, kv_heads, capacity, head_dim], updated in place.
 * new_k, new_v    device [batch, kv_heads, 1, head_dim].
 * seqlens_k       device int32 [batch] (total after this token, minus one).
 * len             the five length arrays to fill (as kvc_seq_lengths would,
 *                 same policy, S = 1), or all five NULL.
 * windowed        KVC_CONTIGUOUS (T > C sets KVC_DEV_CAPACITY) or KVC_RING;
 *                 else KVC_ERR_UNSUPPORTED.
 * local_window_size, scale, rope_*: as kvc_gqa_decode.
 * workspace       device, kvc_decode_step_workspace_size(...) bytes (the same
 *                 as kvc_gqa_decode_workspace_size), 256-byte aligned.
 * Supported: KVC_BF16/KVC_F16, head_dim in {64, 128, 256}, q_heads / kv_heads
 * <= 16 (KVC_ERR_UNSUPPORTED otherwise).
 * Device errors as kvc_seq_lengths / kvc_window_append / kvc_gqa_decode.
 */
kvc_status kvc_decode_step(void *out, const void *q, void *k_cache, void *v_cache,
                           const void *new_k, const void *new_v, const int32_t *seqlens_k,
                           kvc_lengths len, int batch, int q_heads, int kv_heads, int64_t capacity,
                           int head_dim, int dtype, int windowed, int local_window_size,
                           float scale, const float *rope_cos, const float *rope_sin,
                           int64_t rope_max_pos, void *workspace, size_t workspace_bytes,
                           int32_t *dev_status, void *stream);

/* Bytes of workspace kvc_decode_step needs for these sizes (0 on bad sizes). */
size_t kvc_decode_step_workspace_size(int batch, int q_heads, int kv_heads, int64_t capacity,
                                      int head_dim, int dtype);

/*
 * kvc_window_decode_step -- one one-token step on a windowed cache:
 * kvc_seq_lengths + kvc_window_append (S = 1) + kvc_gqa_decode with the same
 * results ("GQA support sliding_window_cache", "Design": rows [E, Lp) move
 * to [0, Lp - E), the new row goes to Lp - E; attention over the window that
 * results).
 *   Small windows, capacity * head_dim <= 32768 (C <= 512 at D = 64, 256 at
 *   D = 128, 128 at D = 256): a single launch.  One CTA owns a (batch row, kv
 *   head) slice and reads it once: the resident rows are loaded into shared
 *   memory (when nothing is evicted, only those the window can see), written
 *   back E rows lower when rows were evicted (else only the new row is
 *   stored), and attended over from there.  No workspace is used.
 *   Larger windows: a ring runs as kvc_decode_step(KVC_RING); a windowed or
 *   drifting cache runs as kvc_seq_lengths, kvc_window_append (the in-place
 *   compaction of large slices runs as a cluster of CTAs per slice) and
 *   kvc_gqa_decode.  The workspace holds the split partials, and the lengths
 *   when `len` is all NULL.
 *
 * out, q          device [batch, q_heads, 1, head_dim].
 * k_cache/v_cache device [batch, kv_heads, capacity, head_dim], updated in place.
 * new_k, new_v    device [batch, kv_heads, 1, head_dim].
 * seqlens_k       device int32 [batch] (total after this token, minus one).
 * len             the five length arrays to fill (as kvc_seq_lengths would,
 *                 same policy, S = 1), or all five NULL.
 * windowed        KVC_WINDOWED, KVC_DRIFTING or KVC_RING (else
 *                 KVC_ERR_UNSUPPORTED).  For a ring the new row goes to slot
 *                 (T - 1) mod C, nothing else is written, and attention
 *                 reads the slots as kvc_gqa_decode_ring does.
 * workspace       device, kvc_window_decode_step_workspace_size(...) bytes,
 *                 256-byte aligned (0 bytes, NULL allowed, for small windows).
 * Requires 0 < local_window_size <= capacity (KVC_ERR_WINDOW).  Supported:
 * KVC_BF16/KVC_F16, head_dim in {64, 128, 256}, q_heads / kv_heads <= 16.
 * Device errors as kvc_seq_lengths / kvc_window_append / kvc_gqa_decode.
 */
kvc_status kvc_window_decode_step(void *out, const void *q, void *k_cache, void *v_cache,
                                  const void *new_k, const void *new_v, const int32_t *seqlens_k,
                                  kvc_lengths len, int batch, int q_heads, int kv_heads,
                                  int64_t capacity, int head_dim, int dtype, int windowed,
                                  int local_window_size, float scale, const float *rope_cos,
                                  const float *rope_sin, int64_t rope_max_pos, void *workspace,
                                  size_t workspace_bytes, int32_t *dev_status, void *stream);

/* Bytes of workspace kvc_window_decode_step needs for these sizes (0 for a
 * window held on chip, or on bad sizes). */
size_t kvc_window_decode_step_workspace_size(int batch, int q_heads, int kv_heads,
                                             int64_t capacity, int head_dim, int dtype);

/*
 * kvc_gqa_prefill_chunk -- attention of an S-token chunk over staged rows
 * ("GQA support sliding_window_cache", "Design": multi-token steps run
 * against the C + S staging cache; causal plus local-window mask).
 *
 * For batch row b with Lp = len.cache_past[b], P = len.past_abs[b]: rows
 * [0, Lp + S) of each head of k_rows/v_rows hold positions P - Lp + r (the
 * stage after kvc_window_append(KVC_APPEND), or a contiguous cache after its
 * append, where Lp = P).  Query i is at P + i and sees row r iff
 * pos(r) <= P + i and (local_window_size <= 0 or P + i - pos(r) <
 * local_window_size).  Queries are rotated at P + i when rope tables are
 * given.
 *
 * out, q          device [batch, q_heads, new_tokens, head_dim].
 * k_rows, v_rows  device [batch, kv_heads, rows_per_head, head_dim],
 *                 rows_per_head >= Lp + S for every row (C + S for a stage).
 * workspace       device scratch of kvc_gqa_prefill_workspace_size(...) bytes,
 *                 256-byte aligned, or NULL.  When the launch would not fill
 *                 the GPU (few query blocks), each block's key range is split
 *                 over several CTAs whose (o, m, l) partials go to the
 *                 workspace and are merged by a second launch; with NULL (or
 *                 too small a workspace) the call runs unsplit, with the same
 *                 results up to floating-point rounding order.
 * Supported: KVC_BF16/KVC_F16 with head_dim in {64, 128, 256} and
 * q_heads / kv_heads in {1, 2, 4, 8, 16} (tcgen05 tensor-core path);
 * KVC_F32 with head_dim <= 256 (no workspace used).  Buffers, the rope
 * tables included, 16-byte aligned (KVC_ERR_ALIGN).
 */
kvc_status kvc_gqa_prefill_chunk(void *out, const void *q, const void *k_rows, const void *v_rows,
                                 int64_t rows_per_head, kvc_lengths len, int batch, int q_heads,
                                 int kv_heads, int new_tokens, int head_dim, int dtype,
                                 int local_window_size, float scale, const float *rope_cos,
                                 const float *rope_sin, int64_t rope_max_pos, void *workspace,
                                 size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * kvc_window_prefill_step -- one whole step of S new tokens on a windowed or
 * drifting cache of C rows: append, chunk attention and row movement, with
 * the C + S stage used only for the rows that need it ("GQA support
 * sliding_window_cache", CPU commit: "Staging for hazardous steps"; the
 * decision is taken per batch row on the device, from the lengths).
 *
 * Batch row b with Lp = len.cache_past[b], E = len.evict[b] is hazardous
 * when E > 0 and E > Lp - W + 1: the rows [0, E) that the step evicts
 * include one that its first query (at stage row Lp) still sees.
 *   hazardous rows:  the new rows go to stage[Lp, Lp + S) and the 127 old
 *                    rows below them to stage[Lp - 127, Lp) (fewer when Lp <
 *                    127); the attention reads its 128-key tiles that lie
 *                    below Lp from the cache and the others from the stage;
 *                    then cache rows [E, Lp) move to [0, Lp - E) in place
 *                    and stage rows [max(E, Lp), Lp + S) follow them -- the
 *                    rows and results of kvc_window_append's staged pair at
 *                    about half its row traffic (the seed and copy-back of
 *                    the whole window become one move of it);
 *   the other rows:  cache rows [E, Lp) move to [0, Lp - E) in place, the new
 *                    rows go to [Lp - E, L), and the attention reads the
 *                    cache; no stage traffic (E = 0: only the new rows).
 * Either way the cache ends byte for byte as kvc_window_append leaves it and
 * the output is the attention of kvc_gqa_prefill_chunk over the stage (up to
 * floating-point summation order).  A row rejected by kvc_seq_lengths
 * (lengths -1) or for its RoPE range is left as kvc_window_append leaves it.
 *
 * out, q          device [batch, q_heads, new_tokens, head_dim].
 * k_cache, v_cache  device [batch, kv_heads, capacity, head_dim].
 * new_k, new_v    device [batch, kv_heads, new_tokens, head_dim].
 * k_stage, v_stage  device [batch, kv_heads, capacity + new_tokens, head_dim]
 *                 for S > 1, rows indexed as the cache's (only hazardous rows
 *                 write or read them, at most 127 + S rows each); may be NULL
 *                 for S = 1, which never stages.
 * len             kvc_seq_lengths outputs for this S, C, policy and window.
 * windowed        KVC_WINDOWED or KVC_DRIFTING; 0 < local_window_size <= C
 *                 (KVC_ERR_WINDOW).
 * workspace       kvc_gqa_prefill_workspace_size(batch, q_heads, kv_heads,
 *                 new_tokens, capacity, head_dim, dtype, local_window_size)
 *                 bytes, or NULL (as kvc_gqa_prefill_chunk).
 * Supported: KVC_BF16/KVC_F16 with head_dim in {64, 128, 256} and
 * q_heads / kv_heads in {1, 2, 4, 8, 16}; KVC_F32 with head_dim <= 256
 * (there every row of an S > 1 step is staged).  head_dim * element size a
 * multiple of 16 bytes (KVC_ERR_UNSUPPORTED); buffers 16-byte aligned.
 * Launches: the row movement before the attention (stage seed, in-place
 * move, new rows), the attention (+ its merge), and the copy-back.
 */
kvc_status kvc_window_prefill_step(void *out, const void *q, void *k_cache, void *v_cache,
                                   const void *new_k, const void *new_v, void *k_stage,
                                   void *v_stage, kvc_lengths len, int batch, int q_heads,
                                   int kv_heads, int new_tokens, int64_t capacity, int head_dim,
                                   int dtype, int windowed, int local_window_size, float scale,
                                   const float *rope_cos, const float *rope_sin,
                                   int64_t rope_max_pos, void *workspace, size_t workspace_bytes,
                                   int32_t *dev_status, void *stream);

/* Bytes of workspace kvc_gqa_prefill_chunk uses for these sizes on the
 * current device (0: it would not split). */
size_t kvc_gqa_prefill_workspace_size(int batch, int q_heads, int kv_heads, int new_tokens,
                                      int64_t rows_per_head, int head_dim, int dtype,
                                      int local_window_size);

/* Human-readable name of a status code (static storage). */
const char *kvc_status_string(kvc_status status);

/* KVC_ABI_VERSION of the loaded library. */
int kvc_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
