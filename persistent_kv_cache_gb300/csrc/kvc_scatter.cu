// kvc_scatter.cu -- ONNX TensorScatter ("TensorScatter" operator page,
// ai.onnx opset 24: spec and pseudocode), plus the library's shared host
// helpers (status strings, SM count, tensor-map encoding).
//
// In place (present == past) only the S updated rows of every prefix move:
// one thread copies one vector (the widest the alignment allows) of one
// trailing slice ("row"), its update load issued before the index load so
// that the two latencies overlap.  The functional form writes every vector of
// present once in a single bandwidth-bound pass, each from the update or from
// past; with no update rows it is a plain vector copy.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "kvc_common.cuh"

namespace {

template <typename V>
__global__ void __launch_bounds__(256)
scatter_rows_kernel(char *__restrict__ present, const char *__restrict__ update,
                    const int64_t *__restrict__ write_indices, int64_t n_prefix,
                    int64_t prefixes_per_batch, int64_t max_seq, int64_t seq_len,
                    int64_t row_vecs, int circular, int32_t *status)
{
    const int64_t n_vec = n_prefix * seq_len * row_vecs;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec; i += stride) {
        const V v = reinterpret_cast<const V *>(update)[i];
        const int64_t row = i / row_vecs, c = i - row * row_vecs;
        const int64_t p = row / seq_len;
        const int64_t s = row - p * seq_len;
        const int64_t b = p / prefixes_per_batch;
        const int64_t wi = write_indices ? write_indices[b] : 0;
        int64_t idx = wi + s;
        if (circular) {
            idx %= max_seq;
            if (idx < 0)
                idx += max_seq;
        } else if (wi < 0 || wi + seq_len > max_seq) {
            if (s == 0 && c == 0 && p == b * prefixes_per_batch)
                kvc::raise_status(status, KVC_DEV_INDEX_OOB);
            continue;
        }
        reinterpret_cast<V *>(present)[(p * max_seq + idx) * row_vecs + c] = v;
    }
}

// the source of present's vector k in a prefix: the update when k lies in the
// written range (offset from base, modulo span, below n_upd), else past
template <typename V>
__device__ __forceinline__ const V *pick_source(const V *src, const V *upd, int64_t k,
                                                int64_t base, int64_t span, int64_t n_upd)
{
    int64_t off = k - base;
    if (off < 0)
        off += span;
    return off < n_upd ? upd + off : src + k;
}

// Functional TensorScatter in one pass: every vector of present is written
// once, from the update when its row is one of the S rows written into its
// prefix, else from past.  A prefix holds span = max_seq * row_vecs vectors;
// its written rows start at vector base = (first written row) * row_vecs and
// run on, modulo span in circular mode, so a vector's distance from base
// (taken modulo span) is at once the test (< S * row_vecs) and its offset in
// the prefix's block of the update: no division per vector.  Linear mode with
// an index out of range leaves that batch row equal to past and raises
// KVC_DEV_INDEX_OOB, as the in-place form does.  A block covers one tile of
// kCopyTile vectors of one prefix, so the host sends prefixes shorter than a
// tile to the copy + in-place scatter pair instead.
constexpr int64_t kCopyTile = 1024;

template <typename V>
__global__ void __launch_bounds__(256, 6)
scatter_copy_kernel(V *__restrict__ present, const V *__restrict__ past,
                    const V *__restrict__ update, const int64_t *__restrict__ write_indices,
                    int64_t n_prefix, int64_t prefixes_per_batch, int64_t max_seq,
                    int64_t seq_len, int64_t row_vecs, int circular, int32_t *status)
{
    // one contiguous tile of 4 x 256 vectors of one prefix per block: each
    // warp reads and writes 32 consecutive vectors per access, four in flight
    const int64_t span = max_seq * row_vecs, upd_vecs = seq_len * row_vecs;
    const int64_t k0 = (int64_t)blockIdx.x * kCopyTile + threadIdx.x;
    for (int64_t p = blockIdx.y; p < n_prefix; p += gridDim.y) {
        const int64_t b = p / prefixes_per_batch;
        const int64_t wi = write_indices ? write_indices[b] : 0;
        int64_t base = 0, n_upd = upd_vecs;
        if (circular) {
            int64_t lo = wi % max_seq;
            if (lo < 0)
                lo += max_seq;
            base = lo * row_vecs;
        } else if (wi < 0 || wi + seq_len > max_seq) {
            n_upd = 0;
            if (blockIdx.x == 0 && threadIdx.x == 0 && p == b * prefixes_per_batch)
                kvc::raise_status(status, KVC_DEV_INDEX_OOB);
        } else {
            base = wi * row_vecs;
        }
        const V *src = past + p * span;
        const V *upd = update + p * upd_vecs;
        V *dst = present + p * span;
        V v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t k = k0 + j * 256;
            if (k < span)
                v[j] = *pick_source(src, upd, k, base, span, n_upd);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t k = k0 + j * 256;
            if (k < span)
                dst[k] = v[j];
        }
    }
}

template <typename V>
void launch_scatter_copy(char *present, const char *past, const char *update, const int64_t *wi,
                         int64_t n_prefix, int64_t ppb, int64_t max_seq, int64_t S,
                         int64_t slice_bytes, int circular, int32_t *status, cudaStream_t stream)
{
    // x: the 1024-vector tiles of one prefix; y: prefixes (looped past 65535)
    const int64_t row_vecs = slice_bytes / (int64_t)sizeof(V);
    const int64_t gx = (max_seq * row_vecs + kCopyTile - 1) / kCopyTile;
    const int64_t gy = n_prefix < 65535 ? n_prefix : 65535;
    scatter_copy_kernel<V><<<dim3((unsigned)gx, (unsigned)gy), 256, 0, stream>>>(
        reinterpret_cast<V *>(present), reinterpret_cast<const V *>(past),
        reinterpret_cast<const V *>(update), wi, n_prefix, ppb, max_seq, S, row_vecs, circular,
        status);
}

// dst[i] = src[i] for i < n (16-byte vectors, four in flight per thread)
__global__ void __launch_bounds__(256)
copy_vec16_kernel(uint4 *__restrict__ dst, const uint4 *__restrict__ src, int64_t n)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n; i += 4 * stride) {
        uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
        dst[i] = a;
        dst[i + stride] = b;
        dst[i + 2 * stride] = c;
        dst[i + 3 * stride] = d;
    }
    for (; i < n; i += stride)
        dst[i] = src[i];
}

__global__ void copy_bytes_kernel(char *__restrict__ dst, const char *__restrict__ src, int64_t n)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        dst[i] = src[i];
}

template <typename V>
void launch_scatter(char *present, const char *update, const int64_t *wi, int64_t n_prefix,
                    int64_t ppb, int64_t max_seq, int64_t S, int64_t slice_bytes, int circular,
                    int32_t *status, cudaStream_t stream)
{
    const int64_t rows = n_prefix * S;
    int64_t blocks = (rows * (slice_bytes / (int64_t)sizeof(V)) + 255) / 256;
    const int64_t cap = (int64_t)kvc_host::sm_count() * 16;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    scatter_rows_kernel<V><<<(unsigned)blocks, 256, 0, stream>>>(
        present, update, wi, n_prefix, ppb, max_seq, S, slice_bytes / (int64_t)sizeof(V),
        circular, status);
}

} // namespace

namespace kvc_host {

// SM count of the current device, looked up once per device; host threads
// may call the library concurrently, so the cache is atomic
int sm_count()
{
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 152;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            n <= 0)
            n = 152;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool encode_3d_sw128(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows, uint32_t box_blocks, CUtensorMapDataType type)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn || cols % 64 != 0)
        return false;
    cuuint64_t dims[3] = {64, rows, cols / 64};
    cuuint64_t strides[2] = {cols * 2, 128};
    cuuint32_t box[3] = {64, box_rows, box_blocks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, type, 3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_2d_bf16_sw128(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                          uint32_t box_rows, CUtensorMapDataType type)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, type, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_4d_heads_sw128(CUtensorMap *map, const void *base, uint64_t heads, uint64_t rows,
                           uint64_t cols, uint32_t elem_bytes, uint32_t box_rows,
                           uint32_t box_heads, CUtensorMapDataType type)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn || elem_bytes == 0 || 128 % elem_bytes != 0)
        return false;
    const uint64_t span = 128 / elem_bytes;
    if (cols % span != 0)
        return false;
    cuuint64_t dims[4] = {span, rows, cols / span, heads};
    cuuint64_t strides[3] = {cols * elem_bytes, 128, rows * cols * elem_bytes};
    cuuint32_t box[4] = {(cuuint32_t)span, box_rows, (cuuint32_t)(cols / span), box_heads};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, type, 4, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_4d_blocks_sw128(CUtensorMap *map, const void *base, uint64_t heads, uint64_t rows,
                            uint64_t cols, uint32_t elem_bytes, uint32_t box_rows,
                            uint32_t box_heads, CUtensorMapDataType type)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn || elem_bytes == 0 || 128 % elem_bytes != 0)
        return false;
    const uint64_t span = 128 / elem_bytes;
    if (cols % span != 0)
        return false;
    cuuint64_t dims[4] = {span, rows, heads, cols / span};
    cuuint64_t strides[3] = {cols * elem_bytes, rows * cols * elem_bytes, 128};
    cuuint32_t box[4] = {(cuuint32_t)span, box_rows, box_heads, (cuuint32_t)(cols / span)};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, type, 4, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

} // namespace kvc_host

KVC_API kvc_status kvc_tensor_scatter(void *present_cache, const void *past_cache,
                                      const void *update, const int64_t *write_indices, int rank,
                                      const int64_t *cache_shape, int64_t update_seq_len,
                                      int axis, int mode, int elem_bytes, int32_t *dev_status,
                                      void *stream_)
{
    if (!present_cache || !past_cache || !cache_shape)
        return KVC_ERR_NULL;
    if (rank < 2 || rank > 8)
        return KVC_ERR_SHAPE;
    if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)
        return KVC_ERR_DTYPE;
    if (mode != KVC_LINEAR && mode != KVC_CIRCULAR)
        return KVC_ERR_UNSUPPORTED;
    if (axis < 0)
        axis += rank;
    if (axis <= 0 || axis >= rank)
        return KVC_ERR_SHAPE;
    int64_t n_elems = 1, n_prefix = 1, slice = elem_bytes;
    for (int d = 0; d < rank; ++d) {
        if (cache_shape[d] < 0)
            return KVC_ERR_SHAPE;
        n_elems *= cache_shape[d];
        if (d < axis)
            n_prefix *= cache_shape[d];
        if (d > axis)
            slice *= cache_shape[d];
    }
    const int64_t max_seq = cache_shape[axis];
    if (update_seq_len < 0 || update_seq_len > max_seq)
        return KVC_ERR_SHAPE;
    if (update_seq_len > 0 && !update)
        return KVC_ERR_NULL;
    const size_t total = (size_t)n_elems * (size_t)elem_bytes;
    const bool in_place = present_cache == past_cache;
    if (!in_place && kvc_host::overlaps(present_cache, total, past_cache, total))
        return KVC_ERR_SHAPE;
    if (update_seq_len > 0 &&
        kvc_host::overlaps(present_cache, total, update,
                           (size_t)(n_prefix * update_seq_len * slice)))
        return KVC_ERR_SHAPE;
    if (n_elems == 0)
        return KVC_OK;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    const int64_t ppb = n_prefix / cache_shape[0];
    const int circ = mode == KVC_CIRCULAR;

    const char *upd_c = static_cast<const char *>(update);
    const uintptr_t a_all = reinterpret_cast<uintptr_t>(present_cache) |
                            reinterpret_cast<uintptr_t>(past_cache) |
                            reinterpret_cast<uintptr_t>(upd_c);
    // vector width of the one-pass form (the widest every pointer allows)
    const int64_t vw = (slice % 16 == 0 && (a_all & 15u) == 0)  ? 16
                       : (slice % 8 == 0 && (a_all & 7u) == 0) ? 8
                       : (slice % 4 == 0 && (a_all & 3u) == 0) ? 4
                       : (slice % 2 == 0 && (a_all & 1u) == 0) ? 2
                                                                : 1;
    if (!in_place && update_seq_len > 0 && max_seq * slice >= kCopyTile * vw) {
        // copy and scatter in one pass: each prefix fills at least one tile
        char *dst = static_cast<char *>(present_cache);
        const char *src = static_cast<const char *>(past_cache);
        const char *upd = upd_c;
        const uintptr_t a = a_all;
        if (slice % 16 == 0 && (a & 15u) == 0)
            launch_scatter_copy<uint4>(dst, src, upd, write_indices, n_prefix, ppb, max_seq,
                                       update_seq_len, slice, circ, dev_status, stream);
        else if (slice % 8 == 0 && (a & 7u) == 0)
            launch_scatter_copy<uint2>(dst, src, upd, write_indices, n_prefix, ppb, max_seq,
                                       update_seq_len, slice, circ, dev_status, stream);
        else if (slice % 4 == 0 && (a & 3u) == 0)
            launch_scatter_copy<uint32_t>(dst, src, upd, write_indices, n_prefix, ppb, max_seq,
                                          update_seq_len, slice, circ, dev_status, stream);
        else if (slice % 2 == 0 && (a & 1u) == 0)
            launch_scatter_copy<uint16_t>(dst, src, upd, write_indices, n_prefix, ppb, max_seq,
                                          update_seq_len, slice, circ, dev_status, stream);
        else
            launch_scatter_copy<uint8_t>(dst, src, upd, write_indices, n_prefix, ppb, max_seq,
                                         update_seq_len, slice, circ, dev_status, stream);
        return kvc_host::launch_status();
    }

    if (!in_place) {
        char *dst = static_cast<char *>(present_cache);
        const char *src = static_cast<const char *>(past_cache);
        const int blocks = kvc_host::sm_count() * 8;
        if (kvc_host::aligned16(dst) && kvc_host::aligned16(src)) {
            const int64_t nv = (int64_t)(total / 16);
            if (nv > 0)
                copy_vec16_kernel<<<blocks, 256, 0, stream>>>(
                    reinterpret_cast<uint4 *>(dst), reinterpret_cast<const uint4 *>(src), nv);
            const int64_t tail = (int64_t)(total - (size_t)nv * 16);
            if (tail > 0)
                copy_bytes_kernel<<<1, 256, 0, stream>>>(dst + nv * 16, src + nv * 16, tail);
        } else {
            copy_bytes_kernel<<<blocks, 256, 0, stream>>>(dst, src, (int64_t)total);
        }
    }
    if (update_seq_len == 0)
        return kvc_host::launch_status();

    char *present = static_cast<char *>(present_cache);
    const char *upd = static_cast<const char *>(update);
    const uintptr_t a = reinterpret_cast<uintptr_t>(present) | reinterpret_cast<uintptr_t>(upd);
    if (slice % 16 == 0 && (a & 15u) == 0)
        launch_scatter<uint4>(present, upd, write_indices, n_prefix, ppb, max_seq,
                              update_seq_len, slice, circ, dev_status, stream);
    else if (slice % 8 == 0 && (a & 7u) == 0)
        launch_scatter<uint2>(present, upd, write_indices, n_prefix, ppb, max_seq,
                              update_seq_len, slice, circ, dev_status, stream);
    else if (slice % 4 == 0 && (a & 3u) == 0)
        launch_scatter<uint32_t>(present, upd, write_indices, n_prefix, ppb, max_seq,
                                 update_seq_len, slice, circ, dev_status, stream);
    else if (slice % 2 == 0 && (a & 1u) == 0)
        launch_scatter<uint16_t>(present, upd, write_indices, n_prefix, ppb, max_seq,
                                 update_seq_len, slice, circ, dev_status, stream);
    else
        launch_scatter<uint8_t>(present, upd, write_indices, n_prefix, ppb, max_seq,
                                update_seq_len, slice, circ, dev_status, stream);
    return kvc_host::launch_status();
}

KVC_API const char *kvc_status_string(kvc_status s)
{
    switch (s) {
    case KVC_OK: return "ok";
    case KVC_ERR_NULL: return "a required pointer is NULL";
    case KVC_ERR_SHAPE: return "size out of range or overlapping buffers";
    case KVC_ERR_DTYPE: return "element type not supported";
    case KVC_ERR_ALIGN: return "buffer not 16-byte aligned";
    case KVC_ERR_UNSUPPORTED: return "combination not supported by the library";
    case KVC_ERR_CAPACITY: return "capacity out of range";
    case KVC_ERR_WINDOW: return "windowed cache needs 0 < local_window_size <= capacity";
    case KVC_ERR_WORKSPACE: return "workspace missing or too small";
    case KVC_ERR_CUDA: return "CUDA launch or driver call failed";
    }
    return "unknown status";
}

KVC_API int kvc_abi_version(void) { return KVC_ABI_VERSION; }
