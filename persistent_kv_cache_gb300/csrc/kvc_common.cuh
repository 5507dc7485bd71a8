// kvc_common.cuh -- shared device/host helpers of the GB300 KV-cache library.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvc.h"

#define KVC_API extern "C" __attribute__((visibility("default")))

namespace kvc {

// --------------------------------------------------------------------------
// status reporting
// --------------------------------------------------------------------------

__device__ __forceinline__ void raise_status(int32_t *st, uint32_t bit)
{
    if (st)
        atomicOr(reinterpret_cast<int *>(st), (int)bit);
}

// a wait gives up after this many nanoseconds of %globaltimer
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// --------------------------------------------------------------------------
// cache-relative lengths of one batch row ("GQA support sliding_window_cache")
// --------------------------------------------------------------------------

// Rows resident after T absolute tokens under the drifting layout of the
// PR's CPU commit: the append point runs on to C, then a whole block of
// gap = C - W + 1 rows is reclaimed at once, so W <= end(T) <= C.
__host__ __device__ __forceinline__ int64_t drift_end(int64_t T, int64_t C, int64_t W)
{
    if (T <= C)
        return T;
    const int64_t gap = C - W + 1;
    return T - gap * ((T - C + gap - 1) / gap);
}

// Lp (resident before), E (evicted) and L (resident after) for a step of S
// tokens that ends at absolute length T.  policy KVC_CONTIGUOUS: the cache
// holds every token; KVC_WINDOWED and KVC_RING: the last min(T, C) tokens;
// KVC_DRIFTING: the last drift_end(T) tokens.  T >= S >= 1 and 1 <= W <= C are the
// caller's to check.
__host__ __device__ __forceinline__ void cache_lengths(int policy, int64_t T, int64_t S,
                                                       int64_t C, int64_t W, int64_t &Lp,
                                                       int64_t &E, int64_t &L)
{
    const int64_t P = T - S;
    if (policy == KVC_DRIFTING) {
        Lp = drift_end(P, C, W);
        L = drift_end(T, C, W);
        E = Lp + S - L;
    } else if (policy == KVC_WINDOWED || policy == KVC_RING) {
        Lp = P < C ? P : C;
        E = Lp + S - C > 0 ? Lp + S - C : 0;
        L = Lp - E + S;
    } else {
        Lp = P;
        E = 0;
        L = T;
    }
}

// Does a windowed step of S new tokens need the C + S stage ("GQA support
// sliding_window_cache", CPU commit: staging for hazardous steps)?  Its first
// query (row Lp of the stage) sees rows from Lp - W + 1 on; the step evicts
// rows [0, E).  When none of those is visible (E <= Lp - W + 1, E = 0
// included), the rows can move first and the chunk attend over the cache
// itself; otherwise the stage keeps the evicted rows for the attention.
__host__ __device__ __forceinline__ bool step_staged(int64_t Lp, int64_t E, int64_t W)
{
    return E > 0 && E > Lp - W + 1;
}

// A staged row of kvc_window_prefill_step keeps its old rows [0, Lp) in the
// cache while its chunk attends: the attention reads a 128-key tile from
// the cache when the tile lies below Lp and from the stage otherwise, so
// the stage needs the new rows and, below them, only the old rows a tile
// reaching Lp can start at: rows [Lp - kStageSeedRows, Lp).
constexpr int kStageSeedRows = 127;

// --------------------------------------------------------------------------
// element types
// --------------------------------------------------------------------------

template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float to_f32(float x) { return x; }
    static __device__ __forceinline__ float from_f32(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
};
template <> struct Elem<__half> {
    static __device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
    static __device__ __forceinline__ __half from_f32(float x) { return __float2half_rn(x); }
};

// rotate-half RoPE of one pair, every product and sum rounded separately
// (no fused multiply-add), so that the stored row is reproducible bit for bit
__device__ __forceinline__ void rope_pair(float &lo, float &hi, float c, float s)
{
    float lo_c = __fmul_rn(lo, c);
    float hi_s = __fmul_rn(hi, s);
    float hi_c = __fmul_rn(hi, c);
    float lo_s = __fmul_rn(lo, s);
    lo = __fsub_rn(lo_c, hi_s);
    hi = __fadd_rn(hi_c, lo_s);
}

// --------------------------------------------------------------------------
// shared-memory barriers and TMA (inline PTX)
// --------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// As mbar_try_wait, but the hardware may suspend the thread for up to
// `hint_ns` nanoseconds while the phase is incomplete instead of returning at
// once, so a waiting warp does not take issue slots from its neighbours.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity,
                                                    uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
                 : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity; returns false after about one
// second (the caller records KVC_DEV_TIMEOUT and winds down).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    uint64_t t0 = global_ns();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((i & 255u) == 255u && global_ns() - t0 > kWaitLimitNs)
            return false;
    }
}

// programmatic dependent launch: the next kernel of the stream, if launched
// with programmatic serialisation, may be scheduled once every CTA of this
// grid has signalled (or exited); a kernel so launched waits, before reading
// what the kernels before it wrote, until they have completed and their
// writes are visible (without the launch attribute both are no-ops)
__device__ __forceinline__ void grid_dep_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// asks L2 for `bytes` (a multiple of 16) at a 16-byte aligned global address;
// the copy lands nowhere else and nothing waits for it
__device__ __forceinline__ void prefetch_l2(const void *gsrc, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                     reinterpret_cast<uint64_t>(gsrc)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 1-D bulk copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global into this CTA's shared memory, completing on `bar`
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes,
                                          uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1], %2, [%3];" ::"r"(smem_u32(smem_dst)),
                 "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// 1-D bulk copy from shared to global memory (bulk-group completion: see
// tma_store_commit / tma_store_wait_*)
__device__ __forceinline__ void bulk_store(void *gdst, const void *smem_src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                     reinterpret_cast<uint64_t>(gdst)),
                 "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
// x (innermost, elements) must keep x * elem_size a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, int32_t x,
                                            int32_t y, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// 2-D tiled TMA store from shared memory (bulk-group completion); the
// coordinates must be inside the tensor (never negative)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int32_t x, int32_t y,
                                             const void *smem_src)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group"
                 " [%0, {%1, %2}], [%3];" ::"l"(reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(smem_u32(smem_src))
                 : "memory");
}
// 4-D tiled TMA store (see tma_store_2d)
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, int32_t x, int32_t y,
                                             int32_t z, int32_t w, const void *smem_src)
{
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group"
                 " [%0, {%1, %2, %3, %4}], [%5];" ::"l"(reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(smem_src))
                 : "memory");
}
__device__ __forceinline__ void tma_store_commit()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// waits until every committed TMA store has finished reading shared memory
__device__ __forceinline__ void tma_store_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// waits until every committed TMA store has completed
__device__ __forceinline__ void tma_store_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// 3-D tiled TMA load (see tma_load_2d; x is the innermost coordinate)
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, int32_t x,
                                            int32_t y, int32_t z, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// 4-D tiled TMA load (see tma_load_2d; x is the innermost coordinate)
__device__ __forceinline__ void tma_load_4d(void *smem_dst, const CUtensorMap *map, int32_t x,
                                            int32_t y, int32_t z, int32_t w, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
        : "memory");
}

// byte offset of 16-byte chunk `c` (0..7) of row `r` inside a box written by
// TMA with 128-byte swizzle (rows of 128 bytes, 1024-byte aligned box)
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t c)
{
    return r * 128u + ((c ^ (r & 7u)) << 4);
}

} // namespace kvc

// --------------------------------------------------------------------------
// host helpers
// --------------------------------------------------------------------------
namespace kvc_host {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [a, a + na) and [b, b + nb) share at least one byte
inline bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

inline int elem_bytes_of(int dtype)
{
    return dtype == KVC_F32 ? 4 : (dtype == KVC_BF16 || dtype == KVC_F16) ? 2 : 0;
}

inline kvc_status launch_status()
{
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

inline bool lengths_ok(const kvc_lengths &l)
{
    return l.past_abs && l.total_abs && l.cache_past && l.cache_total && l.evict;
}

// number of SMs of the current device (cached per device)
int sm_count();

// The row movement of kvc_window_prefill_step (kvc_cache.cu).  Before the
// chunk attention (phase KVC_APPEND): a row that step_staged() marks copies
// its old rows [Lp - kStageSeedRows, Lp) to the same rows of the stage and
// takes its new rows at stage rows [Lp, Lp + S); any other row moves rows
// [E, Lp) of the cache to [0, Lp - E) in place and takes the new rows at
// [Lp - E, L).  After it (KVC_COPY_BACK), a staged row moves its cache rows
// [E, Lp) to [0, Lp - E) and copies stage rows [max(E, Lp), Lp + S) after
// them.
kvc_status hazard_rows(void *k_cache, void *v_cache, const void *new_k, const void *new_v,
                       void *k_stage, void *v_stage, const kvc_lengths &len, int batch,
                       int kv_heads, int S, int64_t C, int D, int dtype, int window, int phase,
                       const float *cos_t, const float *sin_t, int64_t rope_max_pos,
                       int32_t *status, cudaStream_t stream);

// cuTensorMapEncodeTiled through the runtime's driver entry point
// (no link-time dependency on libcuda)
bool encode_2d_bf16_sw128(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                          uint32_t box_rows, CUtensorMapDataType type);

// 3-D view of a [rows, cols] 16-bit matrix as (64 columns, rows, cols / 64
// column blocks) with 128-byte swizzle; a box of (64, box_rows, box_blocks)
// lands in shared memory as box_blocks consecutive [box_rows][128 B] blocks
bool encode_3d_sw128(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows, uint32_t box_blocks, CUtensorMapDataType type);

// 4-D view of a [heads, rows, cols] tensor of elem_bytes-wide elements as
// (128-byte column span, rows, cols / span column blocks, heads) with
// 128-byte swizzle; a box of (span, box_rows, every block, box_heads) lands in
// shared memory as [box_heads][blocks][box_rows][128 B]
bool encode_4d_heads_sw128(CUtensorMap *map, const void *base, uint64_t heads, uint64_t rows,
                           uint64_t cols, uint32_t elem_bytes, uint32_t box_rows,
                           uint32_t box_heads, CUtensorMapDataType type);

// the same tensor as (span, rows, heads, column blocks): a box of (span,
// box_rows, box_heads, every block) lands as [blocks][box_heads][box_rows]
// [128 B], i.e. column block by column block, the heads' rows stacked
bool encode_4d_blocks_sw128(CUtensorMap *map, const void *base, uint64_t heads, uint64_t rows,
                            uint64_t cols, uint32_t elem_bytes, uint32_t box_rows,
                            uint32_t box_heads, CUtensorMapDataType type);

} // namespace kvc_host

// fp32 attention on CUDA cores (kvc_decode.cu); n_rows_mode 0 attends over
// rows [0, cache_total) with S = 1, mode 1 over rows [0, cache_past + S)
namespace kvc_f32 {
kvc_status launch(void *out, const void *q, const void *k_rows, const void *v_rows,
                  int64_t rows_per_head, const kvc_lengths &len, int batch, int q_heads,
                  int kv_heads, int S, int D, int window, float scale, const float *cos_t,
                  const float *sin_t, int64_t rope_max_pos, int n_rows_mode, int32_t *status,
                  cudaStream_t stream);
}
