// kvc_cache.cu -- device-side sequence lengths and the persistent-cache
// append ("GQA support sliding_window_cache", onnxruntime PR 29904, section
// "Design"):
//
//   windowed cache of capacity C, S new tokens on past length P:
//     Lp = min(P, C), E = max(0, Lp + S - C)
//     shift cache[E .. Lp) -> cache[0 .. Lp - E), new rows -> [Lp - E, Lp - E + S)
//   drifting layout (the PR's CPU commit): Lp = end(P), L = end(T),
//     E = Lp + S - L, the same shift and append with E = 0 on most steps
//   S == 1 runs in place; S > 1 runs through a C + S staging cache that is
//   seeded, attended over, and copied back.
//   ring of C slots ("Stateful decode & KV cache", "Sliding-window ring
//   buffer"): new row i goes to slot (P + i) mod C, nothing moves.
//
// K rows are rotated at their absolute position while they are written (RoPE
// baked into K: "Stateful decode & KV cache", "Sliding-window ring buffer").
//
// Kernels (all K and V in one launch; blockIdx.z selects K or V):
//   seq_lengths_kernel   one thread per batch row, int64 arithmetic
//   new_rows_kernel      writes the S new rows (RoPE on K) at a per-row offset
//   copy_range_kernel    per-(b, head) contiguous row range copy (stage seed,
//                        copy-back), 16-byte vectors
//   compact_kernel       windowed S == 1: in-place E-row left shift of the
//                        resident rows in ascending tiles, then the new row
//   quantize_pages_kernel  affine int8 quantization of selected cache pages
//                        ("Persistent input/output feedback", "Optional
//                        heterogeneous paged KV": selected-block quantization)
//   shift_rows_kernel    the copy-back of a stage held in the cache's own rows
//                        (kvc_window_append_inplace): an in-place E-row left
//                        shift of a whole slice through bulk copies
#include <cmath>

#include "kvc_common.cuh"

namespace {

__global__ void seq_lengths_kernel(const int32_t *__restrict__ seqlens_k, int batch, int S,
                                   int64_t C, int policy, int64_t W, kvc_lengths out,
                                   int32_t *status)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= batch)
        return;
    const int64_t T = (int64_t)seqlens_k[b] + 1;
    uint32_t bad = 0;
    if (T < S || T > (int64_t)INT32_MAX)
        bad = KVC_DEV_SEQLEN_RANGE;
    else if (policy == KVC_CONTIGUOUS && T > C)
        bad = KVC_DEV_CAPACITY;
    if (bad) {
        kvc::raise_status(status, bad);
        out.past_abs[b] = out.total_abs[b] = out.cache_past[b] = out.cache_total[b] =
            out.evict[b] = -1;
        return;
    }
    int64_t Lp, E, L;
    kvc::cache_lengths(policy, T, S, C, W, Lp, E, L);
    out.past_abs[b] = (int32_t)(T - S);
    out.total_abs[b] = (int32_t)T;
    out.cache_past[b] = (int32_t)Lp;
    out.cache_total[b] = (int32_t)L;
    out.evict[b] = (int32_t)E;
}

// one thread per (row, pair-vector): loads VEC elements of the low half and
// the matching VEC of the high half of a new row, rotates K, stores both
template <typename T, int VEC>
struct alignas(sizeof(T) * VEC) Vec {
    T v[VEC];
};

template <typename T, int VEC>
__device__ __forceinline__ void write_new_pair(T *__restrict__ dst_row,
                                               const T *__restrict__ src_row, int D, int j,
                                               bool rotate, const float *__restrict__ cs,
                                               const float *__restrict__ sn)
{
    const int half = D / 2;
    Vec<T, VEC> lo = *reinterpret_cast<const Vec<T, VEC> *>(src_row + j * VEC);
    Vec<T, VEC> hi = *reinterpret_cast<const Vec<T, VEC> *>(src_row + half + j * VEC);
    if (rotate) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            float a = kvc::Elem<T>::to_f32(lo.v[e]);
            float b = kvc::Elem<T>::to_f32(hi.v[e]);
            kvc::rope_pair(a, b, cs[j * VEC + e], sn[j * VEC + e]);
            lo.v[e] = kvc::Elem<T>::from_f32(a);
            hi.v[e] = kvc::Elem<T>::from_f32(b);
        }
    }
    *reinterpret_cast<Vec<T, VEC> *>(dst_row + j * VEC) = lo;
    *reinterpret_cast<Vec<T, VEC> *>(dst_row + half + j * VEC) = hi;
}

// page table of a paged cache: logical row r of batch row b is slot
// r % page_size of page table[b * max_pages + r / page_size] of a pool
// [n_pages, kv_heads, page_size, D]
struct PageTable {
    const int32_t *table;
    int max_pages, page_size;
    int64_t n_pages;
};

// the second destination of new_rows_kernel's hazard-step mode: rows that
// step_staged() marks go to a stage of `rows` rows a head at cache_past + i
struct AltRows {
    void *k, *v;
    int64_t rows;
    int window;
};

// grid: x over (i, pair-vector) of one (b, head) slice, y = b * Hkv + h, z = K/V
// dst row of token i, in a buffer with dst_rows rows/head: P + i (base_mode
// 0), cache_past + i (1), (P + i) mod dst_rows for a ring (2, where only the
// last dst_rows tokens are written), row P + i of a paged cache (3), or
// (4, kvc_window_prefill_step) cache_past - evict + i of the cache, or
// cache_past + i of the stage `alt` for a row that step_staged() marks
template <typename T, int VEC>
__global__ void __launch_bounds__(128)
new_rows_kernel(T *__restrict__ k_dst, T *__restrict__ v_dst, const T *__restrict__ new_k,
                const T *__restrict__ new_v, kvc_lengths len, int kv_heads, int S, int D,
                int64_t dst_rows, int base_mode, const float *__restrict__ cos_t,
                const float *__restrict__ sin_t, int64_t rope_max_pos, int32_t *status,
                PageTable pt, AltRows alt)
{
    const int slice = blockIdx.y;
    const int b = slice / kv_heads;
    const bool is_k = blockIdx.z == 0;
    const int L = len.cache_total[b];
    if (L < 0)
        return;
    const int P = len.past_abs[b];
    const bool rotate = is_k && cos_t != nullptr;
    if (cos_t != nullptr && (int64_t)P + S > rope_max_pos) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.z == 0 && slice % kv_heads == 0)
            kvc::raise_status(status, KVC_DEV_ROPE_RANGE);
        return;
    }
    const bool ring = base_mode == 2, paged = base_mode == 3;
    const bool lead = threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.z == 0 &&
                      slice % kv_heads == 0;
    int base = base_mode == 1 ? len.cache_past[b] : P;
    if (base_mode == 4) {
        base = len.cache_past[b];
        if (kvc::step_staged(base, len.evict[b], alt.window)) {
            k_dst = static_cast<T *>(alt.k);
            v_dst = static_cast<T *>(alt.v);
            dst_rows = alt.rows;
        } else {
            base -= len.evict[b];
        }
    }
    if (base < 0 || (!ring && (int64_t)base + S > dst_rows)) {
        // lengths computed for another capacity: refuse rather than overrun
        if (lead)
            kvc::raise_status(status, KVC_DEV_CAPACITY);
        return;
    }
    if (paged) {
        // every page the row's new tokens land in must exist, else the row
        // writes nothing
        const int p0 = P / pt.page_size, p1 = (P + S - 1) / pt.page_size;
        for (int p = p0; p <= p1; ++p) {
            const int id = pt.table[(int64_t)b * pt.max_pages + p];
            if (id < 0 || (int64_t)id >= pt.n_pages) {
                if (lead)
                    kvc::raise_status(status, KVC_DEV_INDEX_OOB);
                return;
            }
        }
    }
    const int pairs = D / (2 * VEC);
    // a ring keeps only the last dst_rows tokens of the step
    const int i0 = ring && (int64_t)S > dst_rows ? (int)(S - dst_rows) : 0;
    const int64_t work = (int64_t)(S - i0) * pairs;
    T *dst = (is_k ? k_dst : v_dst) + (int64_t)slice * dst_rows * D;
    const T *src = (is_k ? new_k : new_v) + (int64_t)slice * S * D;
    for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < work;
         w += (int64_t)gridDim.x * blockDim.x) {
        const int i = i0 + (int)(w / pairs);
        const int j = (int)(w % pairs);
        const int64_t pos = (int64_t)P + i;
        const float *cs = rotate ? cos_t + pos * (D / 2) : nullptr;
        const float *sn = rotate ? sin_t + pos * (D / 2) : nullptr;
        T *drow;
        if (paged) {
            const int64_t page = pt.table[(int64_t)b * pt.max_pages + pos / pt.page_size];
            drow = (is_k ? k_dst : v_dst) +
                   ((page * kv_heads + slice % kv_heads) * pt.page_size + pos % pt.page_size) * D;
        } else {
            drow = dst + (ring ? pos % dst_rows : (int64_t)base + i) * D;
        }
        write_new_pair<T, VEC>(drow, src + (int64_t)i * D, D, j, rotate, cs, sn);
    }
}

// Copies, for every (b, head), rows [src0, src0 + n) of src to rows [0, n) of
// dst.  copy_back = 0: stage seed, src0 = 0, n = Lp.  copy_back = 1: src0 = E,
// n = L.  Row counts come from the device lengths; the grid covers the
// largest possible range.
// hazard_w > 0 (kvc_window_prefill_step): only the rows step_staged() marks
// for that window, and only what they need: the seed copies rows
// [Lp - kStageSeedRows, Lp) to the same rows of the stage, the copy-back
// stage rows [max(E, Lp), Lp + S) to cache rows from max(E, Lp) - E on.
template <typename V>
__global__ void __launch_bounds__(256)
copy_range_kernel(char *__restrict__ k_dst, char *__restrict__ v_dst,
                  const char *__restrict__ k_src, const char *__restrict__ v_src,
                  kvc_lengths len, int kv_heads, int64_t row_bytes, int64_t dst_rows,
                  int64_t src_rows, int copy_back, int64_t rope_limit_rows, int S,
                  int32_t *status, int hazard_w)
{
    const int slice = blockIdx.y;
    const int b = slice / kv_heads;
    const bool is_k = blockIdx.z == 0;
    const int L = len.cache_total[b];
    if (L < 0)
        return;
    if (hazard_w > 0 && !kvc::step_staged(len.cache_past[b], len.evict[b], hazard_w))
        return;
    // a row rejected for its RoPE range is rejected as a whole
    if (rope_limit_rows >= 0 && (int64_t)len.past_abs[b] + S > rope_limit_rows)
        return;
    int64_t src0 = copy_back ? len.evict[b] : 0, dst0 = 0;
    int64_t n = copy_back ? L : len.cache_past[b];
    if (hazard_w > 0) {
        const int64_t Lp = len.cache_past[b], E = len.evict[b];
        if (copy_back) {
            const int64_t first = E > Lp ? E : Lp;  // the kept rows that come from the stage
            src0 = first;
            dst0 = first - E;
            n = Lp + S - first;
        } else {
            src0 = dst0 = Lp > kvc::kStageSeedRows ? Lp - kvc::kStageSeedRows : 0;
            n = Lp - src0;
        }
    }
    if (src0 < 0 || dst0 < 0 || n < 0 || dst0 + n > dst_rows || src0 + n > src_rows) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.z == 0 && slice % kv_heads == 0)
            kvc::raise_status(status, KVC_DEV_CAPACITY);
        return;
    }
    const int64_t nv = n * row_bytes / (int64_t)sizeof(V);
    const V *src = reinterpret_cast<const V *>((is_k ? k_src : v_src) +
                                               ((int64_t)slice * src_rows + src0) * row_bytes);
    V *dst = reinterpret_cast<V *>((is_k ? k_dst : v_dst) +
                                   ((int64_t)slice * dst_rows + dst0) * row_bytes);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + stride < nv; i += 2 * stride) {
        V a = src[i], c = src[i + stride];
        dst[i] = a;
        dst[i + stride] = c;
    }
    if (i < nv)
        dst[i] = src[i];
}

// Windowed S == 1, in place.  One CTA per (b, head, K/V).  When E > 0 the
// rows [E, Lp) move down by E rows: the slice is walked in ascending tiles,
// each tile loaded into registers, then (after a barrier) stored E rows
// lower.  A tile's stores land below everything that it or any later tile
// still has to load, so the move needs no scratch buffer.  The new row is
// written after the last tile.
template <typename T, int VEC>
__global__ void __launch_bounds__(256)
compact_kernel(T *__restrict__ k_cache, T *__restrict__ v_cache, const T *__restrict__ new_k,
               const T *__restrict__ new_v, kvc_lengths len, int kv_heads, int D, int64_t C,
               const float *__restrict__ cos_t, const float *__restrict__ sin_t,
               int64_t rope_max_pos, int32_t *status)
{
    constexpr int U = 4;
    const int slice = blockIdx.x;
    const int b = slice / kv_heads;
    const bool is_k = blockIdx.y == 0;
    const int L = len.cache_total[b];
    if (L < 0)
        return;
    const int P = len.past_abs[b];
    if (cos_t != nullptr && (int64_t)P + 1 > rope_max_pos) {
        if (threadIdx.x == 0 && is_k && slice % kv_heads == 0)
            kvc::raise_status(status, KVC_DEV_ROPE_RANGE);
        return;
    }
    const int Lp = len.cache_past[b];
    const int E = len.evict[b];
    if (Lp < 0 || Lp > C || E < 0 || E > Lp || Lp - E + 1 > C) {
        if (threadIdx.x == 0 && is_k && slice % kv_heads == 0)
            kvc::raise_status(status, KVC_DEV_CAPACITY);
        return;
    }
    T *cache = (is_k ? k_cache : v_cache) + (int64_t)slice * C * D;
    if (E > 0) {
        // move (Lp - E) rows down by E: flat copy of 16-byte vectors
        uint4 *base = reinterpret_cast<uint4 *>(cache);
        const int64_t shift_v = (int64_t)E * D * sizeof(T) / 16;
        const int64_t n = (int64_t)(Lp - E) * D * sizeof(T) / 16;
        const int64_t tile = (int64_t)blockDim.x * U;
        for (int64_t t0 = 0; t0 < n; t0 += tile) {
            uint4 r[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = t0 + (int64_t)u * blockDim.x + threadIdx.x;
                if (i < n)
                    r[u] = base[i + shift_v];
            }
            __syncthreads();
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t i = t0 + (int64_t)u * blockDim.x + threadIdx.x;
                if (i < n)
                    base[i] = r[u];
            }
            __syncthreads();
        }
    }
    const int dst_row = Lp - E;
    const bool rotate = is_k && cos_t != nullptr;
    const int pairs = D / (2 * VEC);
    const T *src = (is_k ? new_k : new_v) + (int64_t)slice * D;
    for (int j = threadIdx.x; j < pairs; j += blockDim.x) {
        const float *cs = rotate ? cos_t + (int64_t)P * (D / 2) : nullptr;
        const float *sn = rotate ? sin_t + (int64_t)P * (D / 2) : nullptr;
        write_new_pair<T, VEC>(cache + (int64_t)dst_row * D, src, D, j, rotate, cs, sn);
    }
}

// Windowed S == 1 for large slices, in place, by a thread-block cluster of CL
// CTAs per (b, head, K/V).  The move is one downward memmove of
// N = (Lp - E) * row_bytes bytes by S = E * row_bytes.  CTA c owns destination
// bytes [lo, hi) (a 16-byte multiple Q = ceil(N / CL) each) and reads sources
// [lo + S, hi + S).  Sources at or above hi are destinations of later CTAs:
// each CTA copies that part of its sources (min(S, hi - lo) bytes) into
// shared memory first, then the cluster meets at its hardware barrier; after
// it no CTA can overwrite bytes another has yet to read, and each CTA streams
// its own range downwards in ascending pieces (one thread, 1-D bulk copies
// through a ring of shared-memory slots: a piece's store overwrites only
// bytes that it or earlier pieces read, and is issued after their loads
// landed), the saved bytes going out last.  A shift longer than the save
// buffer (a drifting cache with a large gap) is moved by the cluster's first
// CTA alone, which is safe by the same ascending order.  The last CTA writes
// the new row (K rotated at P) at row Lp - E after the barrier, once the
// bytes it replaces have been saved.
constexpr int kCompactSlots = 4;
constexpr int kCompactPiece = 16384;
constexpr int kCompactSave = 16384;
constexpr int kCompactSmem = kCompactSlots * kCompactPiece + kCompactSave + 8 * (kCompactSlots + 1) + 128;
// slices of at least this many bytes take the cluster kernel, one CTA per
// kCompactClusterBytes of slice (at most 8, the portable cluster size)
constexpr int64_t kCompactClusterMin = 65536;
constexpr int64_t kCompactClusterBytes = 262144;

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <typename T>
__global__ void __launch_bounds__(32)
compact_cluster_kernel(T *__restrict__ k_cache, T *__restrict__ v_cache,
                       const T *__restrict__ new_k, const T *__restrict__ new_v,
                       kvc_lengths len, int kv_heads, int D, int64_t C,
                       const float *__restrict__ cos_t, const float *__restrict__ sin_t,
                       int64_t rope_max_pos, int32_t *status)
{
    extern __shared__ uint8_t compact_smem_raw[];
    const int CL = (int)gridDim.x;  // the cluster spans blockIdx.x
    const int c = (int)blockIdx.x;
    const int slice = blockIdx.y;
    const int b = slice / kv_heads;
    const bool is_k = blockIdx.z == 0;
    const bool lead = c == 0 && is_k && slice % kv_heads == 0 && threadIdx.x == 0;
    // every CTA of the cluster takes the same early exits (they depend on the
    // batch row only), so none is left waiting at the barrier below
    const int L = len.cache_total[b];
    if (L < 0)
        return;
    const int P = len.past_abs[b];
    if (cos_t != nullptr && (int64_t)P + 1 > rope_max_pos) {
        if (lead)
            kvc::raise_status(status, KVC_DEV_ROPE_RANGE);
        return;
    }
    const int Lp = len.cache_past[b];
    const int E = len.evict[b];
    if (Lp < 0 || Lp > C || E < 0 || E > Lp || Lp - E + 1 > C) {
        if (lead)
            kvc::raise_status(status, KVC_DEV_CAPACITY);
        return;
    }
    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(compact_smem_raw) + 127) & ~uintptr_t(127));
    uint8_t *save = ring + kCompactSlots * kCompactPiece;
    uint64_t *full = reinterpret_cast<uint64_t *>(save + kCompactSave);  // [slots + 1]
    const int64_t rb = (int64_t)D * sizeof(T);
    char *base = reinterpret_cast<char *>((is_k ? k_cache : v_cache) + (int64_t)slice * C * D);
    const int64_t N = (int64_t)(Lp - E) * rb, S = (int64_t)E * rb;
    // this CTA's destination range; the whole range for the first CTA when
    // the shift is longer than the save buffer
    const bool solo = S > kCompactSave;
    const int64_t Q = ((N + CL - 1) / CL + 15) / 16 * 16;
    int64_t lo = solo ? (c == 0 ? 0 : N) : (int64_t)c * Q;
    int64_t hi = solo ? N : lo + Q;
    lo = lo < N ? lo : N;
    hi = hi < N ? hi : N;
    const int64_t keep = solo ? 0 : (S < hi - lo ? S : hi - lo);  // saved source bytes
    const int64_t n_ring = hi - lo - keep;  // bytes streamed through the ring
    const int64_t npieces = E > 0 ? (n_ring + kCompactPiece - 1) / kCompactPiece : 0;
    auto piece_bytes = [&](int64_t p) -> uint32_t {
        const int64_t rest = n_ring - p * kCompactPiece;
        return (uint32_t)(rest < kCompactPiece ? rest : kCompactPiece);
    };
    auto load = [&](int64_t p) {
        const int slot = (int)(p % kCompactSlots);
        kvc::mbar_arrive_expect_tx(&full[slot], piece_bytes(p));
        kvc::bulk_load(ring + slot * kCompactPiece, base + lo + S + p * kCompactPiece,
                       piece_bytes(p), &full[slot]);
    };
    bool ok = true;
    int64_t issued = 0;
    if (threadIdx.x == 0) {
        for (int i = 0; i <= kCompactSlots; ++i)
            kvc::mbar_init(&full[i], 1);
        kvc::fence_mbar_init();
        if (E > 0 && keep > 0) {
            kvc::mbar_arrive_expect_tx(&full[kCompactSlots], (uint32_t)keep);
            kvc::bulk_load(save, base + hi + S - keep, (uint32_t)keep, &full[kCompactSlots]);
        }
        // the ring's first loads read this CTA's own range: nothing writes
        // there before the barrier, so they may start now
        for (; issued < npieces && issued < kCompactSlots; ++issued)
            load(issued);
        if (E > 0 && keep > 0 && !kvc::mbar_wait(&full[kCompactSlots], 0))
            ok = false;
    }
    __syncwarp();
    cluster_sync_all();
    if (threadIdx.x == 0) {
        for (int64_t p = 0; p < npieces; ++p) {
            const int slot = (int)(p % kCompactSlots);
            if (!ok || !kvc::mbar_wait(&full[slot], (uint32_t)(p / kCompactSlots) & 1u)) {
                ok = false;
                break;
            }
            kvc::bulk_store(base + lo + p * kCompactPiece, ring + slot * kCompactPiece,
                            piece_bytes(p));
            kvc::tma_store_commit();
            if (issued < npieces) {
                kvc::tma_store_wait_read();  // the slot's bytes have left shared memory
                load(issued++);
            }
        }
        if (ok && keep > 0) {
            kvc::bulk_store(base + hi - keep, save, (uint32_t)keep);
            kvc::tma_store_commit();
        }
        if (!ok) {
            // a load that never landed: report it and let the others land
            kvc::raise_status(status, KVC_DEV_TIMEOUT);
            for (int64_t p = 0; p < issued; ++p)
                kvc::mbar_wait(&full[p % kCompactSlots], (uint32_t)(p / kCompactSlots) & 1u);
        }
        kvc::tma_store_wait_all();
    }
    __syncwarp();
    ok = __shfl_sync(0xffffffffu, ok, 0);
    // the new row, by the last CTA: its old bytes were saved (or, when the
    // first CTA moved everything alone, read by it) before they are replaced
    const int writer = solo ? 0 : CL - 1;
    if (c != writer || !ok)
        return;
    const bool rotate = is_k && cos_t != nullptr;
    T *dst = reinterpret_cast<T *>(base) + (int64_t)(Lp - E) * D;
    const T *src = (is_k ? new_k : new_v) + (int64_t)slice * D;
    for (int j = threadIdx.x; j < D / 2; j += 32) {
        float lo_v = kvc::Elem<T>::to_f32(src[j]), hi_v = kvc::Elem<T>::to_f32(src[j + D / 2]);
        if (rotate)
            kvc::rope_pair(lo_v, hi_v, cos_t[(int64_t)P * (D / 2) + j],
                           sin_t[(int64_t)P * (D / 2) + j]);
        dst[j] = kvc::Elem<T>::from_f32(lo_v);
        dst[j + D / 2] = kvc::Elem<T>::from_f32(hi_v);
    }
}

// In-place move of rows [E, E + L) of a (b, head) slice to rows [0, L): the
// copy-back of kvc_window_append_inplace.  One CTA per (b, head, K/V); its
// first thread streams the slice's contiguous byte range through a ring of
// shared-memory chunks with 1-D bulk copies: chunk c comes from source bytes
// E * row_bytes + [c CH, (c + 1) CH) and goes to [c CH, (c + 1) CH).  The move
// is downwards, so chunk c's store overwrites only bytes that chunks <= c
// read, and it is issued after those loads have landed; every later load
// reads above every byte stored so far.  No second buffer is needed.
constexpr int kShiftSlots = 6;
constexpr int kShiftChunk = 32768;
constexpr int kShiftSmem = kShiftSlots * kShiftChunk + kShiftSlots * 8 + 128;

// hazard_w > 0 (kvc_window_prefill_step): rows [E, Lp) of a cache of
// rows_per_head = C rows a head move to [0, Lp - E) -- before the attention
// (staged_rows 0) for the rows step_staged() leaves to the cache, after it
// (staged_rows 1) for the rows it marks; the other rows stay.
__global__ void __launch_bounds__(32)
shift_rows_kernel(char *__restrict__ k_rows, char *__restrict__ v_rows, kvc_lengths len,
                  int kv_heads, int64_t row_bytes, int64_t rows_per_head, int S,
                  int64_t rope_limit_rows, int32_t *status, int hazard_w, int staged_rows)
{
    extern __shared__ uint8_t shift_smem_raw[];
    if (threadIdx.x != 0)
        return;
    const int slice = blockIdx.x;
    const int b = slice / kv_heads;
    const bool is_k = blockIdx.y == 0;
    const int L = len.cache_total[b];
    if (L < 0)
        return;
    // a row rejected for its RoPE range had nothing appended: nothing moves
    if (rope_limit_rows >= 0 && (int64_t)len.past_abs[b] + S > rope_limit_rows)
        return;
    const int64_t E = len.evict[b];
    const int64_t Lp = len.cache_past[b];
    if (E < 0 || Lp < 0 || E + L != Lp + S ||
        (hazard_w > 0 ? L > rows_per_head : Lp + S > rows_per_head)) {
        if (is_k && slice % kv_heads == 0)
            kvc::raise_status(status, KVC_DEV_CAPACITY);
        return;
    }
    if (hazard_w > 0 && kvc::step_staged(Lp, E, hazard_w) != (staged_rows != 0))
        return;  // the other kind of row
    // rows that move: the L rows of the stage held in place, or the Lp - E
    // old rows that stay in the cache (none when the step evicts them all)
    const int64_t nrows = hazard_w > 0 ? (Lp > E ? Lp - E : 0) : L;
    if (E == 0 || nrows == 0)
        return;  // the rows are already in place
    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(shift_smem_raw) + 127) & ~uintptr_t(127));
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + kShiftSlots * kShiftChunk);
    for (int i = 0; i < kShiftSlots; ++i)
        kvc::mbar_init(&full[i], 1);
    kvc::fence_mbar_init();
    char *dst = (is_k ? k_rows : v_rows) + (int64_t)slice * rows_per_head * row_bytes;
    const char *src = dst + E * row_bytes;
    const int64_t n = nrows * row_bytes;
    const int64_t nchunks = (n + kShiftChunk - 1) / kShiftChunk;
    auto chunk_bytes = [&](int64_t c) -> uint32_t {
        const int64_t rest = n - c * kShiftChunk;
        return (uint32_t)(rest < kShiftChunk ? rest : kShiftChunk);
    };
    auto load = [&](int64_t c) {
        const int slot = (int)(c % kShiftSlots);
        kvc::mbar_arrive_expect_tx(&full[slot], chunk_bytes(c));
        kvc::bulk_load(ring + slot * kShiftChunk, src + c * kShiftChunk, chunk_bytes(c),
                       &full[slot]);
    };
    const int64_t lead = nchunks < kShiftSlots ? nchunks : kShiftSlots;
    for (int64_t c = 0; c < lead; ++c)
        load(c);
    int64_t issued = lead;
    for (int64_t c = 0; c < nchunks; ++c) {
        const int slot = (int)(c % kShiftSlots);
        if (!kvc::mbar_wait(&full[slot], (uint32_t)(c / kShiftSlots) & 1u)) {
            // a load that never lands: record it, let the other loads in
            // flight land, and leave the slice as it is from chunk c on
            kvc::raise_status(status, KVC_DEV_TIMEOUT);
            for (int64_t d = c + 1; d < issued; ++d)
                kvc::mbar_wait(&full[d % kShiftSlots], (uint32_t)(d / kShiftSlots) & 1u);
            break;
        }
        kvc::bulk_store(dst + c * kShiftChunk, ring + slot * kShiftChunk, chunk_bytes(c));
        kvc::tma_store_commit();
        if (issued < nchunks) {
            kvc::tma_store_wait_read();  // the slot's bytes have left shared memory
            load(issued++);
        }
    }
    kvc::tma_store_wait_all();
}

// Page src[i] of a 16-bit pool -> int8 page dst[i], one CTA per (i, kv head,
// K/V): code = saturate(rint(x / scale) + zp) with x / scale rounded once in
// float32 and rint rounding ties to even, stored as the unsigned byte
// code + 128 - bias (bias 128 for UINT8, 0 for INT8: one payload serves both
// code types, and the decode places the byte as it is), in the fragment
// order of include/kvc.h (q8_k_pos / q8_v_pos below): the decode's lanes then
// load their MMA operand bytes with 16-byte loads and no shuffling.

// byte of element (row j, column d) within a 16-row group of a K payload:
// the A fragment of the scores' MMA over columns [16 kk, 16 kk + 16)
// (rows = keys), word 2 kk + (dd / 8) of the lane, two keys of a column pair
__device__ __forceinline__ int q8_k_pos(int j, int d)
{
    const int nb = j >> 3, g = j & 7, kk = d >> 4, dd = d & 15;
    const int lane = 4 * g + ((dd & 7) >> 1);
    const int fb = (2 * kk + (dd >> 3)) * 4 + 2 * nb + (dd & 1);
    return (fb >> 4) * 512 + lane * 16 + (fb & 15);
}

// byte of element (row j, column c) within a 16-row group of a V payload:
// the A fragment (V transposed, rows = columns of V) of the output's MMA
// over columns [16 mb, 16 mb + 16), word 2 mb + (j / 8) of the lane
__device__ __forceinline__ int q8_v_pos(int j, int c)
{
    const int mb = c >> 4, cc = c & 15;
    const int lane = 4 * (cc & 7) + ((j & 7) >> 1);
    const int fb = (2 * mb + (j >> 3)) * 4 + 2 * (cc >> 3) + (j & 1);
    return (fb >> 4) * 512 + lane * 16 + (fb & 15);
}
struct QuantSpec {
    float scale;
    int zp, lo, hi, bias;
};

template <typename T>
__global__ void __launch_bounds__(256)
quantize_pages_kernel(const T *__restrict__ k_pool, const T *__restrict__ v_pool,
                      uint8_t *__restrict__ qk_pool, uint8_t *__restrict__ qv_pool,
                      const int32_t *__restrict__ src_pages, const int32_t *__restrict__ dst_pages,
                      int64_t n_pool_pages, int64_t n_q_pages, int kv_heads, int D, int64_t slab,
                      QuantSpec kq, QuantSpec vq, float *__restrict__ qparams, int32_t *status)
{
    const int i = blockIdx.x, h = blockIdx.y;
    const bool is_k = blockIdx.z == 0;
    const int src = src_pages[i], dst = dst_pages[i];
    if (src < 0 || (int64_t)src >= n_pool_pages || dst < 0 || (int64_t)dst >= n_q_pages) {
        if (threadIdx.x == 0 && h == 0 && is_k)
            kvc::raise_status(status, KVC_DEV_INDEX_OOB);
        return;
    }
    const QuantSpec q = is_k ? kq : vq;
    if (threadIdx.x == 0 && h == 0) {
        qparams[(int64_t)dst * 4 + (is_k ? 0 : 2)] = q.scale;
        qparams[(int64_t)dst * 4 + (is_k ? 1 : 3)] = (float)(q.zp + 128 - q.bias);
    }
    // slab = page_size * head_dim elements of one (page, head), a multiple of 8
    const int64_t so = ((int64_t)src * kv_heads + h) * slab;
    const int64_t dof = ((int64_t)dst * kv_heads + h) * slab;
    const uint4 *in = reinterpret_cast<const uint4 *>((is_k ? k_pool : v_pool) + so);
    uint8_t *out = (is_k ? qk_pool : qv_pool) + dof;
    const float lo = (float)q.lo, hi = (float)q.hi, zp = (float)q.zp;
    const int cpr = D / 8;  // 8-element chunks per row
    for (int64_t c = threadIdx.x; c < slab / 8; c += blockDim.x) {
        const uint4 x = in[c];
        const T *e = reinterpret_cast<const T *>(&x);
        const int row = (int)(c / cpr), d0 = (int)(c % cpr) * 8;
        uint8_t *grp = out + (int64_t)(row >> 4) * 16 * D;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float t = __fdiv_rn(kvc::Elem<T>::to_f32(e[k]), q.scale);
            const float code = fminf(fmaxf(rintf(t) + zp, lo), hi);
            grp[is_k ? q8_k_pos(row & 15, d0 + k) : q8_v_pos(row & 15, d0 + k)] =
                (uint8_t)((int)code + 128 - q.bias);
        }
    }
}

// hazard_w > 0: the rows of kvc_window_prefill_step with that window (a
// windowed cache and S > 1; see kvc_host::hazard_rows)
template <typename T>
kvc_status append_typed(void *k_cache, void *v_cache, const void *new_k, const void *new_v,
                        void *k_stage, void *v_stage, const kvc_lengths &len, int batch,
                        int kv_heads, int S, int64_t C, int D, int windowed, int phase,
                        const float *cos_t, const float *sin_t, int64_t rope_max_pos,
                        int32_t *status, cudaStream_t stream, int hazard_w = 0)
{
    constexpr int VEC = 16 / sizeof(T);
    const int slices = batch * kv_heads;
    const bool vec_ok = (D / 2) % VEC == 0;
    T *kc = static_cast<T *>(k_cache);
    T *vc = static_cast<T *>(v_cache);
    const T *nk = static_cast<const T *>(new_k);
    const T *nv = static_cast<const T *>(new_v);
    auto launch_new_rows = [&](T *kd, T *vd, int64_t dst_rows, int base_mode,
                               PageTable pt = PageTable{nullptr, 0, 0, 0},
                               AltRows alt = AltRows{nullptr, nullptr, 0, 0}) {
        const int pairs = vec_ok ? D / (2 * VEC) : D / 2;
        const int64_t work = (int64_t)S * pairs;
        int gx = (int)((work + 127) / 128);
        gx = gx < 1 ? 1 : (gx > 64 ? 64 : gx);
        dim3 grid(gx, slices, 2);
        if (vec_ok)
            new_rows_kernel<T, VEC><<<grid, 128, 0, stream>>>(kd, vd, nk, nv, len, kv_heads, S, D,
                                                              dst_rows, base_mode, cos_t,
                                                              sin_t, rope_max_pos, status, pt,
                                                              alt);
        else
            new_rows_kernel<T, 1><<<grid, 128, 0, stream>>>(kd, vd, nk, nv, len, kv_heads, S, D,
                                                            dst_rows, base_mode, cos_t,
                                                            sin_t, rope_max_pos, status, pt,
                                                            alt);
    };
    auto launch_copy = [&](char *kd, char *vd, const char *ks, const char *vs, int64_t dst_rows,
                           int64_t src_rows, int copy_back, int64_t max_rows, int hazard_w = 0) {
        const int64_t row_bytes = (int64_t)D * sizeof(T);
        const int64_t max_v = max_rows * row_bytes / 16;
        int gx = (int)((max_v + 511) / 512);
        const int cap = kvc_host::sm_count() * 8 / (slices * 2 > 0 ? slices * 2 : 1) + 1;
        gx = gx < 1 ? 1 : (gx > cap ? cap : gx);
        dim3 grid(gx, slices, 2);
        const int64_t rope_rows = cos_t ? rope_max_pos : -1;
        if (row_bytes % 16 == 0)
            copy_range_kernel<uint4><<<grid, 256, 0, stream>>>(kd, vd, ks, vs, len, kv_heads,
                                                               row_bytes, dst_rows, src_rows,
                                                               copy_back, rope_rows, S, status,
                                                               hazard_w);
        else
            copy_range_kernel<uint32_t><<<grid, 256, 0, stream>>>(kd, vd, ks, vs, len, kv_heads,
                                                                  row_bytes, dst_rows, src_rows,
                                                                  copy_back, rope_rows, S,
                                                                  status, hazard_w);
    };

    if (windowed == KVC_CONTIGUOUS || windowed == KVC_RING) {
        if (phase != KVC_APPEND)
            return KVC_ERR_UNSUPPORTED;
        launch_new_rows(kc, vc, C, windowed == KVC_RING ? 2 : 0);
    } else if (S == 1) {
        if (phase != KVC_APPEND)
            return KVC_ERR_UNSUPPORTED;
        if (!vec_ok || (D * sizeof(T)) % 16 != 0)
            return KVC_ERR_UNSUPPORTED;
        const int64_t slice_bytes = C * D * (int64_t)sizeof(T);
        if (slice_bytes < kCompactClusterMin) {
            // small slices: one CTA per (b, head, K/V), register tiles
            compact_kernel<T, VEC><<<dim3(slices, 2), 256, 0, stream>>>(
                kc, vc, nk, nv, len, kv_heads, D, C, cos_t, sin_t, rope_max_pos, status);
        } else {
            // large slices: a cluster of up to 8 CTAs per (b, head, K/V)
            int cl = (int)((slice_bytes + kCompactClusterBytes - 1) / kCompactClusterBytes);
            cl = cl < 1 ? 1 : (cl > 8 ? 8 : cl);
            auto kern = compact_cluster_kernel<T>;
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kCompactSmem) != cudaSuccess)
                return KVC_ERR_CUDA;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(cl, slices, 2);
            cfg.blockDim = dim3(32);
            cfg.dynamicSmemBytes = kCompactSmem;
            cfg.stream = stream;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = cl;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaLaunchKernelEx(&cfg, kern, kc, vc, nk, nv, len, kv_heads, D, C, cos_t, sin_t,
                                   rope_max_pos, status) != cudaSuccess)
                return KVC_ERR_CUDA;
        }
    } else if (hazard_w > 0 && phase == KVC_APPEND) {
        // kvc_window_prefill_step: staged rows seed the stage; the others
        // move their old rows down in the cache; then every row's new rows
        // go where its attention will read them
        launch_copy(static_cast<char *>(k_stage), static_cast<char *>(v_stage),
                    reinterpret_cast<const char *>(kc), reinterpret_cast<const char *>(vc), C + S,
                    C, 0, kvc::kStageSeedRows, hazard_w);
        if (cudaFuncSetAttribute(shift_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kShiftSmem) != cudaSuccess)
            return KVC_ERR_CUDA;
        shift_rows_kernel<<<dim3(slices, 2), 32, kShiftSmem, stream>>>(
            reinterpret_cast<char *>(kc), reinterpret_cast<char *>(vc), len, kv_heads,
            (int64_t)D * sizeof(T), C, S, cos_t ? rope_max_pos : -1, status, hazard_w, 0);
        launch_new_rows(kc, vc, C, 4, PageTable{nullptr, 0, 0, 0},
                        AltRows{k_stage, v_stage, C + S, hazard_w});
    } else if (hazard_w > 0) {
        // kvc_window_prefill_step's copy-back: the staged rows' old rows
        // move down in the cache, then their new rows follow from the stage
        if (cudaFuncSetAttribute(shift_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kShiftSmem) != cudaSuccess)
            return KVC_ERR_CUDA;
        shift_rows_kernel<<<dim3(slices, 2), 32, kShiftSmem, stream>>>(
            reinterpret_cast<char *>(kc), reinterpret_cast<char *>(vc), len, kv_heads,
            (int64_t)D * sizeof(T), C, S, cos_t ? rope_max_pos : -1, status, hazard_w, 1);
        launch_copy(reinterpret_cast<char *>(kc), reinterpret_cast<char *>(vc),
                    static_cast<const char *>(k_stage), static_cast<const char *>(v_stage), C,
                    C + S, 1, S, hazard_w);
    } else if (phase == KVC_APPEND) {
        launch_copy(static_cast<char *>(k_stage), static_cast<char *>(v_stage),
                    reinterpret_cast<const char *>(kc), reinterpret_cast<const char *>(vc), C + S,
                    C, 0, C);
        launch_new_rows(static_cast<T *>(k_stage), static_cast<T *>(v_stage), C + S, 1);
    } else {
        launch_copy(reinterpret_cast<char *>(kc), reinterpret_cast<char *>(vc),
                    static_cast<const char *>(k_stage), static_cast<const char *>(v_stage), C,
                    C + S, 1, C);
    }
    return kvc_host::launch_status();
}

// new rows at [Lp, Lp + S) of a buffer with rows_per_head rows per head
template <typename T>
kvc_status append_stage_rows(void *k_rows, void *v_rows, const void *new_k, const void *new_v,
                             const kvc_lengths &len, int batch, int kv_heads, int S,
                             int64_t rows_per_head, int D, const float *cos_t, const float *sin_t,
                             int64_t rope_max_pos, int32_t *status, cudaStream_t stream)
{
    constexpr int VEC = 16 / sizeof(T);
    const bool vec_ok = (D / 2) % VEC == 0;
    const int pairs = vec_ok ? D / (2 * VEC) : D / 2;
    const int64_t work = (int64_t)S * pairs;
    int gx = (int)((work + 127) / 128);
    gx = gx < 1 ? 1 : (gx > 64 ? 64 : gx);
    dim3 grid(gx, batch * kv_heads, 2);
    T *kd = static_cast<T *>(k_rows);
    T *vd = static_cast<T *>(v_rows);
    const T *nk = static_cast<const T *>(new_k);
    const T *nv = static_cast<const T *>(new_v);
    const PageTable none{nullptr, 0, 0, 0};
    if (vec_ok)
        new_rows_kernel<T, VEC><<<grid, 128, 0, stream>>>(kd, vd, nk, nv, len, kv_heads, S, D,
                                                          rows_per_head, 1, cos_t, sin_t,
                                                          rope_max_pos, status, none, AltRows{});
    else
        new_rows_kernel<T, 1><<<grid, 128, 0, stream>>>(kd, vd, nk, nv, len, kv_heads, S, D,
                                                        rows_per_head, 1, cos_t, sin_t,
                                                        rope_max_pos, status, none, AltRows{});
    return kvc_host::launch_status();
}

template <typename T>
kvc_status paged_append_typed(void *k_pool, void *v_pool, const void *new_k, const void *new_v,
                              const kvc_lengths &len, int batch, int kv_heads, int S, int D,
                              const PageTable &pt, const float *cos_t, const float *sin_t,
                              int64_t rope_max_pos, int32_t *status, cudaStream_t stream)
{
    constexpr int VEC = 16 / sizeof(T);
    const bool vec_ok = (D / 2) % VEC == 0;
    const int pairs = vec_ok ? D / (2 * VEC) : D / 2;
    const int64_t work = (int64_t)S * pairs;
    int gx = (int)((work + 127) / 128);
    gx = gx < 1 ? 1 : (gx > 64 ? 64 : gx);
    dim3 grid(gx, batch * kv_heads, 2);
    const int64_t capacity = (int64_t)pt.max_pages * pt.page_size;
    T *kp = static_cast<T *>(k_pool);
    T *vp = static_cast<T *>(v_pool);
    const T *nk = static_cast<const T *>(new_k);
    const T *nv = static_cast<const T *>(new_v);
    if (vec_ok)
        new_rows_kernel<T, VEC><<<grid, 128, 0, stream>>>(kp, vp, nk, nv, len, kv_heads, S, D,
                                                          capacity, 3, cos_t, sin_t,
                                                          rope_max_pos, status, pt, AltRows{});
    else
        new_rows_kernel<T, 1><<<grid, 128, 0, stream>>>(kp, vp, nk, nv, len, kv_heads, S, D,
                                                        capacity, 3, cos_t, sin_t, rope_max_pos,
                                                        status, pt, AltRows{});
    return kvc_host::launch_status();
}

} // namespace

KVC_API kvc_status kvc_quantize_pages(const void *k_pool, const void *v_pool, void *qk_pool,
                                      void *qv_pool, const int32_t *src_pages,
                                      const int32_t *dst_pages, int n_pages,
                                      int64_t n_pool_pages, int64_t n_qpool_pages, int page_size,
                                      int kv_heads, int head_dim, int dtype, float k_scale,
                                      int k_zero_point, int k_unsigned, float v_scale,
                                      int v_zero_point, int v_unsigned, float *qparams,
                                      int32_t *dev_status, void *stream_)
{
    if (dtype != KVC_BF16 && dtype != KVC_F16)
        return kvc_host::elem_bytes_of(dtype) ? KVC_ERR_UNSUPPORTED : KVC_ERR_DTYPE;
    // the payload's fragment order works in 16-row groups and 32-column blocks
    if (n_pages < 0 || kv_heads < 1 || page_size < 16 || page_size % 16 != 0 || head_dim < 32 ||
        head_dim % 32 != 0 || n_pool_pages < 1 || n_qpool_pages < 1)
        return KVC_ERR_SHAPE;
    if (n_pages > 65535 || kv_heads > 65535)
        return KVC_ERR_SHAPE;
    auto spec = [](float scale, int zp, int uns, QuantSpec &q) {
        if (!(scale > 0.f) || !std::isfinite(scale))
            return false;
        q.scale = scale;
        q.zp = zp;
        q.lo = uns ? 0 : -128;
        q.hi = uns ? 255 : 127;
        q.bias = uns ? 128 : 0;
        return zp >= q.lo && zp <= q.hi;
    };
    QuantSpec kq, vq;
    if (!spec(k_scale, k_zero_point, k_unsigned, kq) || !spec(v_scale, v_zero_point, v_unsigned, vq))
        return KVC_ERR_SHAPE;
    if (n_pages == 0)
        return KVC_OK;
    if (!k_pool || !v_pool || !qk_pool || !qv_pool || !src_pages || !dst_pages || !qparams)
        return KVC_ERR_NULL;
    for (const void *p : {k_pool, v_pool, (const void *)qk_pool, (const void *)qv_pool,
                          (const void *)qparams})
        if (!kvc_host::aligned16(p))
            return KVC_ERR_ALIGN;
    const int64_t slab = (int64_t)page_size * head_dim;
    const size_t qb = (size_t)n_qpool_pages * kv_heads * slab;
    if (kvc_host::overlaps(qk_pool, qb, qv_pool, qb))
        return KVC_ERR_SHAPE;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    const dim3 grid(n_pages, kv_heads, 2);
    if (dtype == KVC_BF16)
        quantize_pages_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(k_pool), static_cast<const __nv_bfloat16 *>(v_pool),
            static_cast<uint8_t *>(qk_pool), static_cast<uint8_t *>(qv_pool), src_pages, dst_pages,
            n_pool_pages, n_qpool_pages, kv_heads, head_dim, slab, kq, vq, qparams, dev_status);
    else
        quantize_pages_kernel<__half><<<grid, 256, 0, stream>>>(
            static_cast<const __half *>(k_pool), static_cast<const __half *>(v_pool),
            static_cast<uint8_t *>(qk_pool), static_cast<uint8_t *>(qv_pool), src_pages, dst_pages,
            n_pool_pages, n_qpool_pages, kv_heads, head_dim, slab, kq, vq, qparams, dev_status);
    return kvc_host::launch_status();
}

KVC_API kvc_status kvc_window_append_inplace(void *k_rows, void *v_rows, const void *new_k,
                                             const void *new_v, kvc_lengths len, int batch,
                                             int kv_heads, int new_tokens, int64_t capacity,
                                             int64_t rows_per_head, int head_dim, int dtype,
                                             int windowed, int phase, const float *rope_cos,
                                             const float *rope_sin, int64_t rope_max_pos,
                                             int32_t *dev_status, void *stream_)
{
    const int eb = kvc_host::elem_bytes_of(dtype);
    if (eb == 0)
        return KVC_ERR_DTYPE;
    if (batch < 0 || kv_heads < 1 || new_tokens < 1 || head_dim < 2 || head_dim > 1024 ||
        (head_dim & 1))
        return KVC_ERR_SHAPE;
    if (capacity < 1 || capacity > (int64_t)INT32_MAX || rows_per_head < capacity + new_tokens ||
        rows_per_head > (int64_t)INT32_MAX)
        return KVC_ERR_CAPACITY;
    if (windowed != KVC_WINDOWED && windowed != KVC_DRIFTING)
        return KVC_ERR_UNSUPPORTED;
    if (phase != KVC_APPEND && phase != KVC_COPY_BACK)
        return KVC_ERR_UNSUPPORTED;
    if (((int64_t)head_dim * eb) % 16 != 0)
        return KVC_ERR_UNSUPPORTED;
    if ((rope_cos == nullptr) != (rope_sin == nullptr))
        return KVC_ERR_NULL;
    if (rope_cos && rope_max_pos < 1)
        return KVC_ERR_SHAPE;
    if (batch == 0)
        return KVC_OK;
    if (!k_rows || !v_rows || !kvc_host::lengths_ok(len))
        return KVC_ERR_NULL;
    if (phase == KVC_APPEND && (!new_k || !new_v))
        return KVC_ERR_NULL;
    const size_t rows_bytes = (size_t)batch * kv_heads * rows_per_head * head_dim * eb;
    if (kvc_host::overlaps(k_rows, rows_bytes, v_rows, rows_bytes))
        return KVC_ERR_SHAPE;
    for (const void *p : {(const void *)k_rows, (const void *)v_rows,
                          phase == KVC_APPEND ? new_k : nullptr,
                          phase == KVC_APPEND ? new_v : nullptr})
        if (p && !kvc_host::aligned16(p))
            return KVC_ERR_ALIGN;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    const int slices = batch * kv_heads;
    if (phase == KVC_APPEND) {
        // the stage append with the cache's own rows as the stage: rows
        // [Lp, Lp + S) of a buffer of rows_per_head rows
        switch (dtype) {
        case KVC_F32:
            return append_stage_rows<float>(k_rows, v_rows, new_k, new_v, len, batch, kv_heads,
                                            new_tokens, rows_per_head, head_dim, rope_cos,
                                            rope_sin, rope_max_pos, dev_status, stream);
        case KVC_BF16:
            return append_stage_rows<__nv_bfloat16>(k_rows, v_rows, new_k, new_v, len, batch,
                                                    kv_heads, new_tokens, rows_per_head,
                                                    head_dim, rope_cos, rope_sin, rope_max_pos,
                                                    dev_status, stream);
        default:
            return append_stage_rows<__half>(k_rows, v_rows, new_k, new_v, len, batch, kv_heads,
                                             new_tokens, rows_per_head, head_dim, rope_cos,
                                             rope_sin, rope_max_pos, dev_status, stream);
        }
    }
    if (cudaFuncSetAttribute(shift_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kShiftSmem) != cudaSuccess)
        return KVC_ERR_CUDA;
    shift_rows_kernel<<<dim3(slices, 2), 32, kShiftSmem, stream>>>(
        static_cast<char *>(k_rows), static_cast<char *>(v_rows), len, kv_heads,
        (int64_t)head_dim * eb, rows_per_head, new_tokens, rope_cos ? rope_max_pos : -1,
        dev_status, 0, 0);
    return kvc_host::launch_status();
}

KVC_API kvc_status kvc_seq_lengths(const int32_t *seqlens_k, int batch, int new_tokens,
                                   int64_t capacity, int windowed, int local_window_size,
                                   kvc_lengths out, int32_t *dev_status, void *stream)
{
    if (batch < 0 || new_tokens < 1)
        return KVC_ERR_SHAPE;
    if (capacity < 1 || capacity > (int64_t)INT32_MAX)
        return KVC_ERR_CAPACITY;
    if (windowed < KVC_CONTIGUOUS || windowed > KVC_RING)
        return KVC_ERR_UNSUPPORTED;
    if (windowed != KVC_CONTIGUOUS && (local_window_size <= 0 || local_window_size > capacity))
        return KVC_ERR_WINDOW;
    if (batch == 0)
        return KVC_OK;
    if (!seqlens_k || !kvc_host::lengths_ok(out))
        return KVC_ERR_NULL;
    seq_lengths_kernel<<<(batch + 127) / 128, 128, 0, static_cast<cudaStream_t>(stream)>>>(
        seqlens_k, batch, new_tokens, capacity, windowed, local_window_size, out, dev_status);
    return kvc_host::launch_status();
}

KVC_API kvc_status kvc_window_append(void *k_cache, void *v_cache, const void *new_k,
                                     const void *new_v, void *k_stage, void *v_stage,
                                     kvc_lengths len, int batch, int kv_heads, int new_tokens,
                                     int64_t capacity, int head_dim, int dtype, int windowed,
                                     int phase, const float *rope_cos, const float *rope_sin,
                                     int64_t rope_max_pos, int32_t *dev_status, void *stream_)
{
    const int eb = kvc_host::elem_bytes_of(dtype);
    if (eb == 0)
        return KVC_ERR_DTYPE;
    if (batch < 0 || kv_heads < 1 || new_tokens < 1 || head_dim < 2 || head_dim > 1024 ||
        (head_dim & 1))
        return KVC_ERR_SHAPE;
    if (capacity < 1 || capacity > (int64_t)INT32_MAX)
        return KVC_ERR_CAPACITY;
    if (phase != KVC_APPEND && phase != KVC_COPY_BACK)
        return KVC_ERR_UNSUPPORTED;
    if (windowed < KVC_CONTIGUOUS || windowed > KVC_RING)
        return KVC_ERR_UNSUPPORTED;
    if ((rope_cos == nullptr) != (rope_sin == nullptr))
        return KVC_ERR_NULL;
    if (rope_cos && rope_max_pos < 1)
        return KVC_ERR_SHAPE;
    if (batch == 0)
        return KVC_OK;
    if (!k_cache || !v_cache || !kvc_host::lengths_ok(len))
        return KVC_ERR_NULL;
    const bool staged =
        (windowed == KVC_WINDOWED || windowed == KVC_DRIFTING) && new_tokens > 1;
    if (phase == KVC_APPEND && (!new_k || !new_v))
        return KVC_ERR_NULL;
    if (staged && (!k_stage || !v_stage))
        return KVC_ERR_NULL;
    if (phase == KVC_COPY_BACK && !staged)
        return KVC_ERR_UNSUPPORTED;
    const size_t cache_bytes = (size_t)batch * kv_heads * capacity * head_dim * eb;
    if (kvc_host::overlaps(k_cache, cache_bytes, v_cache, cache_bytes))
        return KVC_ERR_SHAPE;
    if (staged) {
        const size_t st = (size_t)batch * kv_heads * (capacity + new_tokens) * head_dim * eb;
        if (kvc_host::overlaps(k_stage, st, v_stage, st) ||
            kvc_host::overlaps(k_stage, st, k_cache, cache_bytes) ||
            kvc_host::overlaps(v_stage, st, v_cache, cache_bytes) ||
            kvc_host::overlaps(k_stage, st, v_cache, cache_bytes) ||
            kvc_host::overlaps(v_stage, st, k_cache, cache_bytes))
            return KVC_ERR_SHAPE;
    }
    const void *ptrs[6] = {k_cache, v_cache, new_k, new_v, staged ? k_stage : nullptr,
                           staged ? v_stage : nullptr};
    for (const void *p : ptrs)
        if (p && !kvc_host::aligned16(p))
            return KVC_ERR_ALIGN;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    const int w = windowed;
    switch (dtype) {
    case KVC_F32:
        return append_typed<float>(k_cache, v_cache, new_k, new_v, k_stage, v_stage, len, batch,
                                   kv_heads, new_tokens, capacity, head_dim, w, phase, rope_cos,
                                   rope_sin, rope_max_pos, dev_status, stream);
    case KVC_BF16:
        return append_typed<__nv_bfloat16>(k_cache, v_cache, new_k, new_v, k_stage, v_stage, len,
                                           batch, kv_heads, new_tokens, capacity, head_dim, w,
                                           phase, rope_cos, rope_sin, rope_max_pos, dev_status,
                                           stream);
    default:
        return append_typed<__half>(k_cache, v_cache, new_k, new_v, k_stage, v_stage, len, batch,
                                    kv_heads, new_tokens, capacity, head_dim, w, phase, rope_cos,
                                    rope_sin, rope_max_pos, dev_status, stream);
    }
}

KVC_API kvc_status kvc_paged_append(void *k_pool, void *v_pool, const void *new_k,
                                    const void *new_v, const int32_t *block_table, int max_pages,
                                    int64_t n_pool_pages, int page_size, kvc_lengths len,
                                    int batch, int kv_heads, int new_tokens, int head_dim,
                                    int dtype, const float *rope_cos, const float *rope_sin,
                                    int64_t rope_max_pos, int32_t *dev_status, void *stream)
{
    const int eb = kvc_host::elem_bytes_of(dtype);
    if (eb == 0)
        return KVC_ERR_DTYPE;
    if (batch < 0 || kv_heads < 1 || new_tokens < 1 || head_dim < 2 || head_dim > 1024 ||
        (head_dim & 1))
        return KVC_ERR_SHAPE;
    if (page_size < 1 || max_pages < 1 || n_pool_pages < 1)
        return KVC_ERR_SHAPE;
    if ((int64_t)max_pages * page_size > (int64_t)INT32_MAX)
        return KVC_ERR_CAPACITY;
    if ((rope_cos == nullptr) != (rope_sin == nullptr))
        return KVC_ERR_NULL;
    if (rope_cos && rope_max_pos < 1)
        return KVC_ERR_SHAPE;
    if (batch == 0)
        return KVC_OK;
    if (!k_pool || !v_pool || !new_k || !new_v || !block_table || !kvc_host::lengths_ok(len))
        return KVC_ERR_NULL;
    const size_t pool_bytes = (size_t)n_pool_pages * kv_heads * page_size * head_dim * eb;
    if (kvc_host::overlaps(k_pool, pool_bytes, v_pool, pool_bytes))
        return KVC_ERR_SHAPE;
    for (const void *p : {(const void *)k_pool, (const void *)v_pool, new_k, new_v})
        if (!kvc_host::aligned16(p))
            return KVC_ERR_ALIGN;
    const PageTable pt{block_table, max_pages, page_size, n_pool_pages};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (dtype) {
    case KVC_F32:
        return paged_append_typed<float>(k_pool, v_pool, new_k, new_v, len, batch, kv_heads,
                                         new_tokens, head_dim, pt, rope_cos, rope_sin,
                                         rope_max_pos, dev_status, st);
    case KVC_BF16:
        return paged_append_typed<__nv_bfloat16>(k_pool, v_pool, new_k, new_v, len, batch,
                                                 kv_heads, new_tokens, head_dim, pt, rope_cos,
                                                 rope_sin, rope_max_pos, dev_status, st);
    default:
        return paged_append_typed<__half>(k_pool, v_pool, new_k, new_v, len, batch, kv_heads,
                                          new_tokens, head_dim, pt, rope_cos, rope_sin,
                                          rope_max_pos, dev_status, st);
    }
}

namespace kvc_host {

kvc_status hazard_rows(void *k_cache, void *v_cache, const void *new_k, const void *new_v,
                       void *k_stage, void *v_stage, const kvc_lengths &len, int batch,
                       int kv_heads, int S, int64_t C, int D, int dtype, int window, int phase,
                       const float *cos_t, const float *sin_t, int64_t rope_max_pos,
                       int32_t *status, cudaStream_t stream)
{
    switch (dtype) {
    case KVC_BF16:
        return append_typed<__nv_bfloat16>(k_cache, v_cache, new_k, new_v, k_stage, v_stage, len,
                                           batch, kv_heads, S, C, D, KVC_WINDOWED, phase, cos_t,
                                           sin_t, rope_max_pos, status, stream, window);
    case KVC_F16:
        return append_typed<__half>(k_cache, v_cache, new_k, new_v, k_stage, v_stage, len, batch,
                                    kv_heads, S, C, D, KVC_WINDOWED, phase, cos_t, sin_t,
                                    rope_max_pos, status, stream, window);
    default:
        return KVC_ERR_UNSUPPORTED;
    }
}

} // namespace kvc_host
