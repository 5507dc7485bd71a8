// kvc_prefill.cu -- attention of a multi-token chunk over staged rows
// ("GQA support sliding_window_cache", section "Design": a step with S > 1
// runs against the C + S staging cache; causal plus local-window mask on
// absolute positions, cache-relative row addressing).
//
// 16-bit path: one CTA per (query block, kv head, batch row) on the 5th-gen
// tensor cores.  The M = 128 tile packs the GQA group: row m holds query head
// m / QB of the group and query qb * QB + m % QB (QB = 128 / group), so every
// K/V tile is read once for all heads of the group.  Key tiles are 128 rows.
//
//   TMEM columns  O [0, D) fp32 | S/P double buffer [D, D + 256)
//   shared mem    Q tile (128 x D, 128-byte swizzled) | ring of K/V slabs;
//                 the output tile is staged over both at the end
//   entry         one thread loads the raw query tile with a single 4-D TMA
//                 load straight into the MMA's layout (column block by
//                 column block, the group's heads' rows stacked)
//   warp 0        allocates tensor memory and issues tcgen05.mma in the order
//                 S_0, S_1, PV_0, S_2, PV_1, ...:
//                   S_j = Q K_j^T   A = Q (shared), B = K slabs (K-major)
//                   O  += P_j V_j   A = P_j in TMEM, B = V slabs (MN-major)
//                 so the next scores are always queued behind the current PV
//   warps 1-8     two threads per row (= TMEM lane), each owning half of the
//                 score columns and half of O: rotate the query rows in
//                 place in the Q tile, then per tile read its S_j half, mask only tiles the
//                 window or diagonal cuts, exchange the row max with the
//                 partner thread, online softmax in the log2 domain (the
//                 running max is only raised when it grows by more than 2^8,
//                 exact after the final division), write P_j as 16-bit pairs
//                 over S_j, rescale its half of O when the max moved, and at
//                 the end divide by l and stage its half of the output row
//                 in shared memory; one TMA store writes the block's tile.
//   warp 9        TMA producer: streams the K and V slabs into the ring in
//                 the order the tensor pipe consumes them (K_0, K_1, V_0,
//                 K_2, V_1, ...), one 3-D box of up to 32 KB per slot (the
//                 cost of a TMA operation hardly grows from 16 KB to 32 KB,
//                 so large boxes double the bytes a single stream delivers).
// Every mbarrier wait is bounded; a timeout sets KVC_DEV_TIMEOUT, every role
// winds down, outstanding tensor-core work is drained and TMEM is freed.
//
// fp32 path: the CUDA-core attn_f32_kernel (kvc_decode.cu).
#include <algorithm>
#include <type_traits>

#include "kvc_common.cuh"

namespace {

constexpr int kBM = 128;       // rows of the M tile (query heads x queries)
constexpr int kBN = 128;       // KV rows per tile
constexpr int kSoftmaxWarps = 8;
constexpr int kThreads = 32 * (1 + kSoftmaxWarps + 1);  // MMA, softmax x 8, TMA
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint32_t kEpilogueBar = 5;       // named barrier of the softmax warps (1-4: pairs)

// ---------------- tcgen05 helpers (inline PTX) ----------------

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     kvc::smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            kvc::smem_u32(bar))
        : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16, one CTA
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16: A's rows are TMEM lanes and
// its 16-bit elements are packed two per 32-bit column
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// 32-bit words to consecutive columns of this thread's TMEM lane

// 32 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                   "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
                 "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
                 "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
                 "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])),
                 "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                 "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
                 "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
                 "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
                 "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
                 "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])),
                 "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
                 "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
                 "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])),
                 "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
                 "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
                 : "memory");
}

// 64 consecutive fp32 columns of this thread's TMEM lane in one load
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64])
{
    uint32_t r[64];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {"
                 "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
                 "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
                 "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63"
                 "}, [%64];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                   "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]),
                   "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]),
                   "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
                   "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]),
                   "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]),
                   "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i)
        v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st_words(uint32_t taddr, const uint32_t (&w)[32])
{
    float f[32];
#pragma unroll
    for (int i = 0; i < 32; ++i)
        f[i] = __uint_as_float(w[i]);
    tmem_st32(taddr, f);
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2^x on the special-function unit (ex2.approx, flush-to-zero; 2^-inf = 0)
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <typename T> __device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    if constexpr (std::is_same<T, __half>::value) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
}


// Shared-memory matrix descriptor for a 128-byte-swizzled operand: rows of
// 128 bytes, 8-row groups 1024 bytes apart (stride byte offset), `lbo` bytes
// between 64-element column blocks for operands whose other dimension is the
// contiguous one; version 1 (bit 46), swizzle mode 2 = 128B (bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr, uint32_t lbo_bytes)
{
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate, A/B type (0 f16, 1 bf16),
// A K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1), N >> 3, M >> 4.
__host__ __device__ constexpr uint32_t f16_idesc(uint32_t ab_type, uint32_t b_mn, uint32_t M,
                                                 uint32_t N)
{
    return (1u << 4) | (ab_type << 7) | (ab_type << 10) | (b_mn << 16) | ((N >> 3) << 17) |
           ((M >> 4) << 24);
}

// One lane's share of a query row when a warp's 32 lanes cover the D/2
// rotation pairs: N 16-bit values (q) and N floats (f) per half row.
template <int N> struct QuarterRow;
template <> struct QuarterRow<4> { using q = uint2;          using f = float4; };
template <> struct QuarterRow<2> { using q = uint32_t;       using f = float2; };
template <> struct QuarterRow<1> { using q = unsigned short; using f = float; };

struct PrefillArgs {
    void *out;
    const void *q;
    kvc_lengths len;
    int batch, q_heads, kv_heads, group, qb_rows;  // qb_rows = 128 / group
    int S;
    int64_t rows_per_head;
    int window;
    float scale_log2;
    const float *cos_t, *sin_t;
    int64_t rope_max_pos;
    int32_t *status;
    // KV split (grids under one wave): blockIdx.x = q block * nsplit + split;
    // each split writes fp32 (o, m, l) partials of its rows, merged by
    // prefill_combine_kernel.  nsplit == 1: the output is written directly.
    int nsplit;
    float *ws_o, *ws_m, *ws_l;  // [nsplit][batch * q_heads * S] (x D for o)
    // kvc_window_prefill_step (hazard_w = the window, else 0): a row that
    // kvc::step_staged() marks keeps its old rows in the cache and its new
    // ones in the stage (tmap_k2 / tmap_v2, alt_rows rows a head, the chunk
    // at rows [Lp, Lp + S), the old rows [Lp - kStageSeedRows, Lp) copied
    // there too): a 128-key tile below Lp is read from the cache, any other
    // from the stage; any other row was moved and appended in the cache
    // itself (rows_per_head = C rows a head, its chunk at rows [Lp - E, L))
    int hazard_w;
    int64_t alt_rows;
};
static_assert(kvc::kStageSeedRows == kBN - 1,
              "a key tile that reaches the new rows starts at most kBN - 1 rows below them");

// The rows the chunk of batch row b attends: the row of its first query (a
// position P at row Lp, so key row r holds position P - Lp + r), the row
// pitch of the buffer holding its new rows and whether that buffer is the
// stage.  False when the lengths do not fit that buffer.
__device__ __forceinline__ bool chunk_rows(const PrefillArgs &a, int b, int &Lp, int64_t &pitch,
                                           bool &alt)
{
    Lp = a.len.cache_past[b];
    pitch = a.rows_per_head;
    alt = false;
    if (a.hazard_w > 0) {
        const int E = a.len.evict[b];
        if (kvc::step_staged(Lp, E, a.hazard_w)) {
            alt = true;
            pitch = a.alt_rows;
        } else {
            Lp -= E;
        }
    }
    return Lp >= 0 && (int64_t)Lp + a.S <= pitch;
}

template <int D> struct PrefillSmem {
    // A TMA operation costs about the same for 16 KB as for 32 KB, so each
    // ring slot is filled by one 3-D box of up to 32 KB.
    static constexpr int TILE = kBN * D * 2;             // one K (or V) tile
    static constexpr int SLAB = TILE < 32768 ? TILE : 32768;
    static constexpr int NSLAB_T = TILE / SLAB;          // slabs per K (or V) tile
    static constexpr int DB = SLAB / (kBN * 128);        // 64-column blocks per K slab
    static constexpr int KPS = SLAB / (D * 2);           // keys per V slab
    static constexpr int Q_BYTES = kBM * D * 2;          // D/64 boxes of 128 x 64
    // Ring depth: every slot the opt-in shared memory of a CTA (227 KB)
    // leaves beside the Q tile and the barriers / exchange area (at most
    // 2.3 KB).
    static constexpr int SMEM_BUDGET = 227 * 1024;
    static constexpr int MISC_MAX = (2 * 12 + 9) * 8 + 16 + 4 * kBM * 4;
    static constexpr int NSLAB_MAX = (SMEM_BUDGET - Q_BYTES - MISC_MAX) / SLAB;
    static constexpr int NSLAB = NSLAB_MAX < 12 ? NSLAB_MAX : 12;
    static constexpr int Q_OFF = 0;
    static constexpr int RING_OFF = Q_OFF + Q_BYTES;
    static constexpr int BAR_OFF = RING_OFF + NSLAB * SLAB;
    // barriers: full[NSLAB], empty[NSLAB], s_full[2], p_full[2], o_done[2],
    //           q_full, drain, q_tma
    static constexpr int NBAR = 2 * NSLAB + 9;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;  // tmem addr, abort flag
    static constexpr int RED_OFF = MISC_OFF + 16;        // row max / sum exchange, 4 x 128 floats
    static constexpr int TOTAL = RED_OFF + 4 * kBM * 4;
    // the epilogue stages the output tile (16-bit, or the fp32 partial of a
    // KV split) over the Q tile and the ring, which are free by then
    static constexpr int O_OFF = Q_OFF;
    static_assert(kBM * D * 4 <= RING_OFF + NSLAB * SLAB, "fp32 output tile must fit");
    static_assert(TOTAL <= SMEM_BUDGET, "layout exceeds the opt-in shared memory");
    // TMEM columns: O [0, D) fp32 | S/P double buffer [D, D + 256)
    static constexpr uint32_t COL_O = 0, COL_S = D;
    static constexpr uint32_t TMEM_COLS = 512;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              int32_t *status)
{
    if (kvc::mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = kvc::global_ns();
    for (uint32_t i = 0;; ++i) {
        if (kvc::mbar_try_wait_sleep(bar, parity, 20000))
            return true;
        if ((i & 7u) == 7u) {
            if (*abort_flag)
                return false;
            if (kvc::global_ns() - t0 > kvc::kWaitLimitNs) {
                kvc::raise_status(status, KVC_DEV_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// The K and V slabs stream through one ring in the order the tensor pipe
// consumes them: K_0, K_1, then V_j followed by K_{j+2} while that tile
// exists, so the tail is ..., V_{n-2}, V_{n-1}.  Group g of that order is
// one (operand, tile); each group is D/64 slabs.
__device__ __forceinline__ void slab_group(int g, int ntiles, bool &is_v, int &tile)
{
    const int lead = ntiles < 2 ? ntiles : 2;
    if (g < lead) {
        is_v = false;
        tile = g;
        return;
    }
    const int r = g - lead;
    const int paired = ntiles > 2 ? ntiles - 2 : 0;  // tiles j with a K_{j+2} after V_j
    if (r < 2 * paired) {
        is_v = (r & 1) == 0;
        tile = is_v ? (r >> 1) : (r >> 1) + 2;
    } else {
        is_v = true;
        tile = paired + (r - 2 * paired);
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v,
                  const __grid_constant__ CUtensorMap tmap_k2,
                  const __grid_constant__ CUtensorMap tmap_v2,
                  const __grid_constant__ CUtensorMap tmap_o, const PrefillArgs a)
{
    using SM = PrefillSmem<D>;
    constexpr int BOXES = D / 64;
    constexpr int NSLAB = SM::NSLAB, NST = SM::NSLAB_T, KPS = SM::KPS, DB = SM::DB;
    constexpr uint32_t AB = std::is_same<T, __half>::value ? 0u : 1u;
    constexpr uint32_t IDESC_S = f16_idesc(AB, 0, kBM, kBN);
    constexpr uint32_t IDESC_O = f16_idesc(AB, 1, kBM, D);
    constexpr uint32_t COL_O = SM::COL_O, COL_S = SM::COL_S;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    {
        // the swizzled tiles need a 1024-byte aligned base; check the layout
        // fits the dynamic allocation the launch obtained
        uint32_t dyn;
        asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
        if ((uint32_t)(smem - smem_raw) + SM::TOTAL > dyn) {
            if (threadIdx.x == 0)
                kvc::raise_status(a.status, KVC_DEV_CAPACITY);
            return;
        }
    }
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SM::BAR_OFF);
    uint64_t *full = bars, *empty = bars + NSLAB, *s_full = bars + 2 * NSLAB,
             *p_full = s_full + 2, *o_done = s_full + 4, *q_full = s_full + 6,
             *drain = s_full + 7, *q_tma = s_full + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + SM::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SM::MISC_OFF + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qblk = blockIdx.x / a.nsplit, split = blockIdx.x % a.nsplit;
    const int kvh = blockIdx.y, b = blockIdx.z;
    const int g = a.group, QB = a.qb_rows, S = a.S;
    const int q0 = qblk * QB;
    if (q0 >= S)
        return;

    // The raw query tile needs no lengths: one TMA load issued at entry
    // brings it in the MMA's layout (block of 64 columns by block, row
    // m = head * QB + query; rows past S are zero-filled) while the lengths
    // arrive; a CTA that leaves before its pipeline starts lets it land.
    if (threadIdx.x == 0) {
        kvc::mbar_init(q_tma, 1);
        kvc::fence_mbar_init();
        kvc::tma_prefetch_desc(&tmap_q);
        kvc::mbar_arrive_expect_tx(q_tma, SM::Q_BYTES);
        kvc::tma_load_4d(smem + SM::Q_OFF, &tmap_q, 0, q0, b * a.q_heads + kvh * g, 0, q_tma);
    }
    auto leave = [&]() {
        if (threadIdx.x == 0)
            kvc::mbar_wait(q_tma, 0);
    };

    // ---- per batch row geometry (uniform over the CTA) ----
    const int L = a.len.cache_total[b];
    if (L < 0) {
        leave();
        return;
    }
    int Lp;
    int64_t pitch;
    bool alt;
    const int P = a.len.past_abs[b];
    if (!chunk_rows(a, b, Lp, pitch, alt)) {
        if (threadIdx.x == 0 && qblk == 0 && kvh == 0)
            kvc::raise_status(a.status, KVC_DEV_CAPACITY);
        leave();
        return;
    }
    // a staged row reads its tiles below Lp from the cache (C rows a head)
    // and the rest from the stage
    const int64_t cache_base = ((int64_t)b * a.kv_heads + kvh) * a.rows_per_head;
    if (a.cos_t && (int64_t)P + S > a.rope_max_pos) {
        if (threadIdx.x == 0 && qblk == 0 && kvh == 0)
            kvc::raise_status(a.status, KVC_DEV_ROPE_RANGE);
        leave();
        return;
    }
    // the rotation rows of the block's queries are asked of L2 at once: the
    // softmax warps read them right after, behind the start of the K/V stream
    if (threadIdx.x == 0 && a.cos_t) {
        const int64_t o = (int64_t)(P + q0) * (D / 2);
        const uint32_t nb = (uint32_t)(min(QB, S - q0) * (D / 2) * sizeof(float));
        kvc::prefetch_l2(a.cos_t + o, nb);
        kvc::prefetch_l2(a.sin_t + o, nb);
    }
    const int q_last = min(S - 1, q0 + QB - 1);
    const int hi = Lp + q_last;  // last visible row of the block
    int lo = 0;
    if (a.window > 0)
        lo = max(0, Lp + q0 - a.window + 1);
    // this split's share [t0, t1) of the block's key tiles
    const int ntiles_all = (hi - lo + kBN) / kBN;
    const int t0 = (int)((int64_t)split * ntiles_all / a.nsplit);
    const int t1 = (int)((int64_t)(split + 1) * ntiles_all / a.nsplit);
    const int64_t rows_total = (int64_t)a.batch * a.q_heads * S;
    if (t1 == t0) {
        // nothing to attend: a partial that the merge skips
        for (int m = threadIdx.x; m < kBM; m += kThreads) {
            const int hh = m / QB, ii = q0 + (m - (m / QB) * QB);
            if (ii < S && hh < g) {
                const int64_t qrow = ((int64_t)b * a.q_heads + kvh * g + hh) * S + ii;
                a.ws_m[split * rows_total + qrow] = -INFINITY;
                a.ws_l[split * rows_total + qrow] = 0.f;
            }
        }
        leave();
        return;
    }
    lo += t0 * kBN;
    const int ntiles = t1 - t0;
    const int nslabs = 2 * ntiles * NST;
    const int64_t row_base = ((int64_t)b * a.kv_heads + kvh) * pitch;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSLAB; ++i) {
            kvc::mbar_init(&full[i], 1);
            kvc::mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            kvc::mbar_init(&s_full[i], 1);
            kvc::mbar_init(&p_full[i], 8);
            kvc::mbar_init(&o_done[i], 1);
        }
        kvc::mbar_init(q_full, 8);
        kvc::mbar_init(drain, 1);
        *abort_flag = 0;
        kvc::fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, SM::TMEM_COLS);
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t smem_base = kvc::smem_u32(smem);

    if (warp == 1 + kSoftmaxWarps) {
        // ======================= TMA producer =======================
        // one 3-D box per ring slot: a K slab is DB column blocks of 128 rows,
        // a V slab is KPS rows of every column block (128-byte swizzled rows)
        if (lane == 0) {
            kvc::tma_prefetch_desc(&tmap_k);
            kvc::tma_prefetch_desc(&tmap_v);
            if (alt) {
                kvc::tma_prefetch_desc(&tmap_k2);
                kvc::tma_prefetch_desc(&tmap_v2);
            }
            int issued = 0;
            for (int q = 0; q < nslabs; ++q) {
                const int slot = q % NSLAB;
                if (q >= NSLAB &&
                    !wait_or_abort(&empty[slot], ((q / NSLAB) - 1) & 1, abort_flag, a.status))
                    break;
                bool is_v;
                int tile;
                slab_group(q / NST, ntiles, is_v, tile);
                const int sl = q % NST;
                uint8_t *dst = smem + SM::RING_OFF + slot * SM::SLAB;
                const int r0 = lo + tile * kBN;  // the tile's first key row
                const bool stage = alt && r0 + kBN > Lp;
                const int32_t y0 = (int32_t)((stage ? row_base : cache_base) + r0);
                kvc::mbar_arrive_expect_tx(&full[slot], SM::SLAB);
                if (!is_v)
                    kvc::tma_load_3d(dst, stage ? &tmap_k2 : &tmap_k, 0, y0, sl * DB, &full[slot]);
                else
                    kvc::tma_load_3d(dst, stage ? &tmap_v2 : &tmap_v, 0, y0 + sl * KPS, 0,
                                     &full[slot]);
                issued = q + 1;
            }
            if (*abort_flag) {
                // wind-down: let the loads already in flight land before the CTA exits
                for (int q = max(0, issued - NSLAB); q < issued; ++q)
                    kvc::mbar_wait(&full[q % NSLAB], (q / NSLAB) & 1);
            }
        }
    } else if (warp == 0) {
        // ======================= MMA issuer =======================
        // tensor-pipe order: S_0, S_1, PV_0, S_2, PV_1, ...  S_{j+2} reuses the
        // TMEM buffer that holds P_j, after PV_j in issue order.
        // A single thread issues every MMA, so its issue cost is per MMA: the
        // shared-memory descriptors are built once and stepped by constant
        // offsets (the start-address field counts 16-byte units and shared
        // addresses stay below 256 KB, so adding to it never carries out).
        if (lane == 0) {
            bool ok = wait_or_abort(q_full, 0, abort_flag, a.status);
            int q = 0;  // next slab of the ring, in consumption order
            const uint64_t q_desc = sw128_desc(smem_base + SM::Q_OFF, 16);
            const uint64_t k_ring = sw128_desc(smem_base + SM::RING_OFF, 16);
            const uint64_t v_ring = sw128_desc(smem_base + SM::RING_OFF, KPS * 128);
            auto issue_s = [&](int j) -> bool {
                const uint32_t d_s = tmem + COL_S + (j & 1) * kBN;
                for (int sl = 0; sl < NST; ++sl, ++q) {
                    const int slot = q % NSLAB;
                    if (!wait_or_abort(&full[slot], (q / NSLAB) & 1, abort_flag, a.status))
                        return false;
                    tc_fence_after();
                    const uint64_t qd = q_desc + (uint64_t)(sl * DB * (kBM * 128 / 16));
                    const uint64_t kd = k_ring + (uint64_t)(slot * (SM::SLAB / 16));
#pragma unroll
                    for (int blk = 0; blk < DB; ++blk) {
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4) {
                            const uint64_t ad = qd + (uint64_t)((blk * (kBM * 128) + k4 * 32) / 16);
                            const uint64_t bd = kd + (uint64_t)((blk * (kBN * 128) + k4 * 32) / 16);
                            tc_mma_ss(d_s, ad, bd, IDESC_S, (sl | blk | k4) != 0);
                        }
                    }
                    tc_commit(&empty[slot]);
                }
                tc_commit(&s_full[j & 1]);
                return true;
            };
            for (int j = 0; ok && j < 2 && j < ntiles; ++j)
                ok = issue_s(j);
            for (int j = 0; ok && j < ntiles; ++j) {
                const int s = j & 1;
                if (!wait_or_abort(&p_full[s], (j >> 1) & 1, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int sl = 0; sl < NST && ok; ++sl, ++q) {
                    const int slot = q % NSLAB;
                    if (!wait_or_abort(&full[slot], (q / NSLAB) & 1, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t vd = v_ring + (uint64_t)(slot * (SM::SLAB / 16));
                    const uint32_t pa = tmem + COL_S + s * kBN + sl * (KPS / 16) * 8;
#pragma unroll
                    for (int k2 = 0; k2 < KPS / 16; ++k2) {
                        // 16-key step k2 of this slab: P columns (16-bit pairs) and V rows
                        tc_mma_ts(tmem + COL_O, pa + k2 * 8, vd + (uint64_t)(k2 * (2048 / 16)),
                                  IDESC_O, (j > 0 || sl > 0 || k2 > 0) ? 1u : 0u);
                    }
                    tc_commit(&empty[slot]);
                }
                if (!ok)
                    break;
                tc_commit(&o_done[s]);
                if (j + 2 < ntiles)
                    ok = issue_s(j + 2);
            }
            // drain: everything issued above has completed once this arrives
            // (a plain bounded wait, also on the abort path)
            tc_commit(drain);
            kvc::mbar_wait(drain, 0);
        }
    } else {
        // ======================= softmax / epilogue =======================
        // two warps per TMEM lane quadrant: `half` 0 owns score columns
        // [0, 64) of every tile and O columns [0, D/2), `half` 1 the rest
        const int sw = warp - 1;                   // 0..7
        const int quad = warp & 3;                 // TMEM lane quadrant of this warp
        const int half = sw >> 2;
        const int m = quad * 32 + lane;            // tile row == TMEM lane
        const int hh = m / QB;                     // head within the group
        const int ii = q0 + (m - hh * QB);         // query index in the chunk
        const bool row_valid = ii < S && hh < g;
        const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
        const int64_t qrow = ((int64_t)b * a.q_heads + kvh * g + hh) * S + ii;
        float *red = reinterpret_cast<float *>(smem + SM::RED_OFF);  // [2 tiles][2 halves][128]
        const uint32_t pair_bar = 1 + quad;       // named barrier of the two warps of a quadrant

        // query tile: the raw rows landed by TMA; each warp rotates its 16
        // rows in place at absolute position P + (the row's query), its lanes
        // spread along D (lane l owns the rotation pairs (c, c + D/2) for c
        // in [PPL*l, PPL*l + PPL)), the cos/sin loads of all 16 rows issued
        // together.  Rows past S stay zero.  The tensor pipe waits on this.
        {
            const bool q_ok = wait_or_abort(q_tma, 0, abort_flag, a.status);
            if (q_ok && a.cos_t) {
                using QVec = typename QuarterRow<D / 64>::q;
                using FVec = typename QuarterRow<D / 64>::f;
                constexpr int PPL = D / 64;
                constexpr int ROWS = kBM / kSoftmaxWarps;
                uint8_t *qt = smem + SM::Q_OFF;
                const int c0 = PPL * lane;
                const uint32_t off_lo = (uint32_t)(c0 >> 6) * (kBM * 128), sub = (uint32_t)(c0 & 7) * 2;
                const uint32_t off_hi = (uint32_t)((D / 2 + c0) >> 6) * (kBM * 128);
                const uint32_t ch_lo = (uint32_t)(c0 & 63) >> 3, ch_hi = (uint32_t)((D / 2 + c0) & 63) >> 3;
                FVec cv[ROWS], sv[ROWS];
#pragma unroll
                for (int u = 0; u < ROWS; ++u) {
                    const int mr = sw * ROWS + u;
                    const int ir = q0 + (mr - (mr / QB) * QB);
                    if (ir < S) {
                        const int64_t o = (int64_t)(P + ir) * (D / 2) + c0;
                        cv[u] = *reinterpret_cast<const FVec *>(a.cos_t + o);
                        sv[u] = *reinterpret_cast<const FVec *>(a.sin_t + o);
                    }
                }
#pragma unroll
                for (int u = 0; u < ROWS; ++u) {
                    const int mr = sw * ROWS + u;
                    const int ir = q0 + (mr - (mr / QB) * QB);
                    if (ir < S) {
                        QVec *plo = reinterpret_cast<QVec *>(qt + off_lo + kvc::sw128(mr, ch_lo) + sub);
                        QVec *phi = reinterpret_cast<QVec *>(qt + off_hi + kvc::sw128(mr, ch_hi) + sub);
                        QVec lo = *plo, hi = *phi;
                        T *lv = reinterpret_cast<T *>(&lo);
                        T *hv = reinterpret_cast<T *>(&hi);
                        const float *cf = reinterpret_cast<const float *>(&cv[u]);
                        const float *sf = reinterpret_cast<const float *>(&sv[u]);
#pragma unroll
                        for (int e = 0; e < PPL; ++e) {
                            float x = kvc::Elem<T>::to_f32(lv[e]), y = kvc::Elem<T>::to_f32(hv[e]);
                            kvc::rope_pair(x, y, cf[e], sf[e]);
                            lv[e] = kvc::Elem<T>::from_f32(x);
                            hv[e] = kvc::Elem<T>::from_f32(y);
                        }
                        *plo = lo;
                        *phi = hi;
                    }
                }
            }
            kvc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                kvc::mbar_arrive(q_full);
        }

        // visible rows of this query: [r_lo, r_hi]
        const int r_hi = Lp + ii;
        const int r_lo = a.window > 0 ? max(0, r_hi - a.window + 1) : 0;
        const float c_log2 = a.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const int s = j & 1;
            const int t_lo = lo + j * kBN;
            const int c0 = t_lo + 64 * half;  // key row of my first column
            if (!wait_or_abort(&s_full[s], (j >> 1) & 1, abort_flag, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float v[64];
            tmem_ld64(lane_addr + COL_S + s * kBN + 64 * half, v);

            // mask only where the window or the diagonal cuts these columns
            const bool all_in = row_valid && c0 >= r_lo && c0 + 63 <= r_hi;
            if (!all_in) {
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const int r = c0 + c;
                    v[c] = (row_valid && r >= r_lo && r <= r_hi) ? v[c] : -INFINITY;
                }
            }
            float mx0 = fmaxf(v[0], v[1]), mx1 = fmaxf(v[2], v[3]);
#pragma unroll
            for (int c = 4; c < 64; c += 4) {
                mx0 = fmaxf(mx0, fmaxf(v[c], v[c + 1]));
                mx1 = fmaxf(mx1, fmaxf(v[c + 2], v[c + 3]));
            }
            float mx = fmaxf(mx0, mx1);
            // the exchange barrier also orders both halves' S reads before
            // either half overwrites the buffer with P
            red[((j & 1) * 2 + half) * kBM + m] = mx;
            named_bar_sync(pair_bar, 64);
            mx = fmaxf(mx, red[((j & 1) * 2 + (half ^ 1)) * kBM + m]);
            const float mt = mx * c_log2;  // tile max in log2 units (c_log2 > 0)

            float alpha = 1.f;
            bool rescale = false;
            if (mt > m_run + kRescaleThreshold || (m_run == -INFINITY && mt > -INFINITY)) {
                if (j > 0 && m_run > -INFINITY) {
                    alpha = fast_exp2(m_run - mt);
                    rescale = true;
                }
                m_run = mt;
            }
            const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
            float ps0 = 0.f, ps1 = 0.f;
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
                const float p0 = fast_exp2(fmaf(v[c], c_log2, neg_m));
                const float p1 = fast_exp2(fmaf(v[c + 1], c_log2, neg_m));
                ps0 += p0;
                ps1 += p1;
                pk[c / 2] = pack2<T>(p0, p1);
            }
            l_run = l_run * alpha + (ps0 + ps1);
            // P_j (16-bit pairs) over the S_j columns of this row
            tmem_st_words(lane_addr + COL_S + s * kBN + 32 * half, pk);

            // rows past the last visible row of the block (last tile only):
            // zero them in the V slabs so that 0 * (stale or uninitialised
            // bytes) stays 0 in O += P V
            if (t_lo + kBN - 1 > hi) {
                const int first_bad = hi + 1 - t_lo;  // rows [first_bad, 128) of the tile
                const int q_first = (2 * ntiles - 1) * NST;  // V_{n-1} is the last group
                for (int sl = first_bad / KPS; sl < NST; ++sl) {
                    const int q = q_first + sl;
                    if (!wait_or_abort(&full[q % NSLAB], (q / NSLAB) & 1, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    uint8_t *vt = smem + SM::RING_OFF + (q % NSLAB) * SM::SLAB;
                    const int r0 = max(0, first_bad - sl * KPS);  // first bad row in this slab
                    const int nbad = KPS - r0;
                    for (int idx = threadIdx.x - 32; idx < nbad * BOXES * 8; idx += 256) {
                        const int rr = r0 + idx / (BOXES * 8);
                        const int bx = (idx / 8) % BOXES, cc = idx % 8;
                        *reinterpret_cast<uint4 *>(vt + bx * (KPS * 128) + rr * 128 + cc * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                }
                if (!ok)
                    break;
                kvc::fence_proxy_async_smem();
            }

            // the running max moved: rescale my half of this O row (PV_{j-1} done)
            if (__any_sync(0xffffffffu, rescale)) {
                if (!wait_or_abort(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag,
                                   a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int cc = half * (D / 2); cc < (half + 1) * (D / 2); cc += 32) {
                    float o[32];
                    tmem_ld32(lane_addr + COL_O + cc, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        o[i] *= alpha;
                    tmem_st32(lane_addr + COL_O + cc, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                kvc::mbar_arrive(&p_full[s]);
        }

        // epilogue: combine the two halves' sums, wait for the last PV, then
        // stage my half of the row in shared memory, where the Q tile and
        // the ring were (every MMA that read them has completed once the
        // last PV has), in the output box's order [head][column block]
        // [query][128 B] (128-byte swizzled), and one thread stores the tile
        // with a single TMA store that clips the queries past S.
        // (the buffer of parity ntiles & 1 was last read before the final tile's barrier)
        red[((ntiles & 1) * 2 + half) * kBM + m] = l_run;
        named_bar_sync(pair_bar, 64);
        const float l_tot = l_run + red[((ntiles & 1) * 2 + (half ^ 1)) * kBM + m];
        const bool have_o = ok && wait_or_abort(&o_done[(ntiles - 1) & 1],
                                                ((ntiles - 1) >> 1) & 1, abort_flag, a.status);
        const int r_in = m - hh * QB;  // query of this row within the block
        if (have_o) {
            tc_fence_after();
            if (a.nsplit == 1) {
                // 16-bit output: a 128-byte row holds 64 columns
                const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
#pragma unroll 1
                for (int cc = half * (D / 2); cc < (half + 1) * (D / 2); cc += 32) {
                    float o[32];
                    tmem_ld32(lane_addr + COL_O + cc, o);
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        uint4 pkt;
                        T *e = reinterpret_cast<T *>(&pkt);
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            e[u] = kvc::Elem<T>::from_f32(o[c + u] * inv);
                        const int col = cc + c;
                        const uint32_t row = (uint32_t)((hh * (D / 64) + (col >> 6)) * QB + r_in);
                        *reinterpret_cast<uint4 *>(smem + SM::O_OFF + kvc::sw128(row, (col & 63) >> 3)) = pkt;
                    }
                }
            } else {
                // this split's partial, fp32: o unnormalised (a 128-byte row
                // holds 32 columns), l, and the reference max m (log2 units)
                // that o and l are relative to
#pragma unroll 1
                for (int cc = half * (D / 2); cc < (half + 1) * (D / 2); cc += 32) {
                    float o[32];
                    tmem_ld32(lane_addr + COL_O + cc, o);
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        const int col = cc + c;
                        const uint32_t row = (uint32_t)((hh * (D / 32) + (col >> 5)) * QB + r_in);
                        *reinterpret_cast<float4 *>(smem + SM::O_OFF + kvc::sw128(row, (col & 31) >> 2)) =
                            make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
                    }
                }
                if (row_valid && half == 0) {
                    const int64_t pr = split * rows_total + qrow;
                    a.ws_m[pr] = m_run;
                    a.ws_l[pr] = l_tot;
                }
            }
        }
        tc_fence_before();
        kvc::fence_proxy_async_smem();
        named_bar_sync(kEpilogueBar, 32 * kSoftmaxWarps);
        if (sw == 0 && lane == 0 && !*abort_flag) {
            // a failed wait anywhere raised the abort flag: then nothing is stored
            const int head0 = b * a.q_heads + kvh * g;
            const int h = a.nsplit == 1 ? head0 : split * a.batch * a.q_heads + head0;
            kvc::tma_store_4d(&tmap_o, 0, q0, 0, h, smem + SM::O_OFF);
            kvc::tma_store_commit();
            kvc::tma_store_wait_read();  // the CTA may leave once the tile has been read
        }
    }

    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, SM::TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag)
        kvc::mbar_wait(q_tma, 0);  // a query tile still in flight lands before the CTA leaves
}

// Merges the KV splits' partials of every query row (one warp per row): the
// weights 2^(m_j - max m) over the splits that saw a visible key, then
// out = sum w_j o_j / sum w_j l_j, rounded to the output type.
template <typename T, int D>
__global__ void __launch_bounds__(128)
prefill_combine_kernel(const PrefillArgs a)
{
    constexpr int PER = D / 32;  // columns per lane
    const int lane = threadIdx.x & 31;
    const int64_t rows_total = (int64_t)a.batch * a.q_heads * a.S;
    const int64_t qrow = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (qrow >= rows_total)
        return;
    const int b = (int)(qrow / ((int64_t)a.q_heads * a.S));
    // the rows the attention kernel refused (status already raised there)
    const int L = a.len.cache_total[b];
    if (L < 0)
        return;
    int Lp;
    int64_t pitch;
    bool alt;
    const int P = a.len.past_abs[b];
    if (!chunk_rows(a, b, Lp, pitch, alt))
        return;
    if (a.cos_t && (int64_t)P + a.S > a.rope_max_pos)
        return;
    float mstar = -INFINITY;
    for (int j = 0; j < a.nsplit; ++j)
        mstar = fmaxf(mstar, a.ws_m[j * rows_total + qrow]);
    float acc[PER];
#pragma unroll
    for (int c = 0; c < PER; ++c)
        acc[c] = 0.f;
    float l = 0.f;
    for (int j = 0; j < a.nsplit; ++j) {
        const float mj = a.ws_m[j * rows_total + qrow];
        if (mj == -INFINITY)
            continue;
        const float w = exp2f(mj - mstar);
        l += w * a.ws_l[j * rows_total + qrow];
        const float *o = a.ws_o + (j * rows_total + qrow) * D;
#pragma unroll
        for (int c = 0; c < PER; ++c)
            acc[c] += w * o[lane + 32 * c];
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    T *dst = static_cast<T *>(a.out) + qrow * D;
#pragma unroll
    for (int c = 0; c < PER; ++c)
        dst[lane + 32 * c] = kvc::Elem<T>::from_f32(acc[c] * inv);
}

// KV splits for grids under one wave (one CTA per SM): as many as fill the
// SMs without a second wave, each with at least two key tiles
int prefill_splits(int batch, int q_heads, int kv_heads, int S, int64_t rows_per_head, int window)
{
    const int g = q_heads / kv_heads;
    const int qb = kBM / g;
    const int64_t ctas = (int64_t)((S + qb - 1) / qb) * kv_heads * batch;
    const int sms = kvc_host::sm_count();
    if (ctas <= 0 || ctas * 2 > sms)
        return 1;
    const int64_t keys = window > 0 ? std::min<int64_t>(rows_per_head, (int64_t)window + qb)
                                    : rows_per_head;
    const int64_t tiles = (keys + kBN - 1) / kBN;
    int64_t n = sms / ctas;
    n = std::min<int64_t>(n, std::max<int64_t>(1, tiles / 2));
    return (int)std::min<int64_t>(n, 16);
}

size_t prefill_ws_bytes(int nsplit, int batch, int q_heads, int S, int head_dim)
{
    if (nsplit <= 1)
        return 0;
    return (size_t)nsplit * batch * q_heads * S * (head_dim + 2) * sizeof(float);
}

// the second K/V source of kvc_window_prefill_step (hazard_w = the window;
// 0 or NULL pointers: none)
struct AltSource {
    const void *k, *v;
    int64_t rows;
    int hazard_w;
};

template <typename T, int D>
kvc_status launch_prefill_tc(void *out, const void *q, const void *k_rows, const void *v_rows,
                             int64_t R, const kvc_lengths &len, int batch, int q_heads,
                             int kv_heads, int S, int window, float scale, const float *cos_t,
                             const float *sin_t, int64_t rope_max_pos, void *workspace,
                             size_t workspace_bytes, int32_t *status, cudaStream_t stream,
                             const AltSource &alt)
{
    using SM = PrefillSmem<D>;
    const uint64_t rows = (uint64_t)batch * kv_heads * R;
    if (rows > (uint64_t)INT32_MAX)
        return KVC_ERR_SHAPE;
    const CUtensorMapDataType tt = std::is_same<T, __half>::value
                                       ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap tq, tk, tv, tk2, tv2, to;
    // the stage, when the step has one (no stage: S = 1, no row is staged)
    const bool has_alt = alt.hazard_w > 0 && alt.k && alt.v;
    const int64_t R2 = has_alt ? alt.rows : R;
    const uint64_t rows2 = (uint64_t)batch * kv_heads * R2;
    if (rows2 > (uint64_t)INT32_MAX)
        return KVC_ERR_SHAPE;
    if (!kvc_host::encode_3d_sw128(&tk, k_rows, rows, D, kBN, SM::DB, tt) ||
        !kvc_host::encode_3d_sw128(&tv, v_rows, rows, D, SM::KPS, D / 64, tt) ||
        !kvc_host::encode_3d_sw128(&tk2, has_alt ? alt.k : k_rows, rows2, D, kBN, SM::DB, tt) ||
        !kvc_host::encode_3d_sw128(&tv2, has_alt ? alt.v : v_rows, rows2, D, SM::KPS, D / 64,
                                   tt) ||
        !kvc_host::encode_4d_blocks_sw128(&tq, q, (uint64_t)batch * q_heads, (uint64_t)S, D,
                                          sizeof(T), (uint32_t)(kBM / (q_heads / kv_heads)),
                                          (uint32_t)(q_heads / kv_heads), tt))
        return KVC_ERR_CUDA;
    PrefillArgs a;
    a.out = out;
    a.q = q;
    a.len = len;
    a.batch = batch;
    a.q_heads = q_heads;
    a.kv_heads = kv_heads;
    a.group = q_heads / kv_heads;
    a.qb_rows = kBM / a.group;
    // a KV split when the grid is under one wave and the caller gave room
    // for the partials; otherwise one CTA per query block
    a.nsplit = prefill_splits(batch, q_heads, kv_heads, S, R, window);
    if (!workspace || workspace_bytes < prefill_ws_bytes(a.nsplit, batch, q_heads, S, D))
        a.nsplit = 1;
    const int64_t rows_total = (int64_t)batch * q_heads * S;
    a.ws_o = static_cast<float *>(workspace);
    a.ws_m = a.ws_o ? a.ws_o + (int64_t)a.nsplit * rows_total * D : nullptr;
    a.ws_l = a.ws_m ? a.ws_m + (int64_t)a.nsplit * rows_total : nullptr;
    a.S = S;
    a.rows_per_head = R;
    a.hazard_w = alt.hazard_w > 0 ? alt.hazard_w : 0;
    a.alt_rows = R2;
    a.window = window;
    a.scale_log2 = scale * kLog2e;
    a.cos_t = cos_t;
    a.sin_t = sin_t;
    a.rope_max_pos = rope_max_pos;
    a.status = status;
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    // the dynamic window starts 1024-byte aligned after the reserved area;
    // the kernel checks its layout fits what it was given (KVC_DEV_CAPACITY)
    const size_t smem = std::min<size_t>((size_t)SM::TOTAL + 1024, (size_t)optin);
    if (smem < (size_t)SM::TOTAL)
        return KVC_ERR_UNSUPPORTED;
    auto kern = prefill_tc_kernel<T, D>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return KVC_ERR_CUDA;
    // the output tile store: [batch * q_heads, S, D] 16-bit, or the fp32
    // partials [nsplit * batch * q_heads, S, D]; a box is one query block of
    // every head of a group
    const bool part = a.nsplit > 1;
    if (!kvc_host::encode_4d_heads_sw128(
            &to, part ? static_cast<void *>(a.ws_o) : out,
            (uint64_t)(part ? a.nsplit : 1) * batch * q_heads, (uint64_t)S, D, part ? 4 : 2,
            (uint32_t)a.qb_rows, (uint32_t)a.group,
            part ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : tt))
        return KVC_ERR_CUDA;
    const int qblocks = (S + a.qb_rows - 1) / a.qb_rows;
    dim3 grid(qblocks * a.nsplit, kv_heads, batch);
    kern<<<grid, kThreads, smem, stream>>>(tq, tk, tv, tk2, tv2, to, a);
    if (a.nsplit > 1)
        prefill_combine_kernel<T, D><<<(unsigned)((rows_total + 3) / 4), 128, 0, stream>>>(a);
    return kvc_host::launch_status();
}

template <typename T>
kvc_status dispatch_prefill16(int D, void *out, const void *q, const void *k, const void *v,
                              int64_t R, const kvc_lengths &len, int B, int Hq, int Hkv, int S,
                              int W, float scale, const float *cs, const float *sn, int64_t rmax,
                              void *ws, size_t ws_bytes, int32_t *st, cudaStream_t stream,
                              const AltSource &alt = AltSource{nullptr, nullptr, 0, 0})
{
    switch (D) {
    case 64:
        return launch_prefill_tc<T, 64>(out, q, k, v, R, len, B, Hq, Hkv, S, W, scale, cs, sn,
                                        rmax, ws, ws_bytes, st, stream, alt);
    case 128:
        return launch_prefill_tc<T, 128>(out, q, k, v, R, len, B, Hq, Hkv, S, W, scale, cs, sn,
                                         rmax, ws, ws_bytes, st, stream, alt);
    case 256:
        return launch_prefill_tc<T, 256>(out, q, k, v, R, len, B, Hq, Hkv, S, W, scale, cs, sn,
                                         rmax, ws, ws_bytes, st, stream, alt);
    default:
        return KVC_ERR_UNSUPPORTED;
    }
}

} // namespace

KVC_API size_t kvc_gqa_prefill_workspace_size(int batch, int q_heads, int kv_heads,
                                              int new_tokens, int64_t rows_per_head,
                                              int head_dim, int dtype, int local_window_size)
{
    if (batch < 1 || q_heads < 1 || kv_heads < 1 || q_heads % kv_heads != 0 || new_tokens < 1 ||
        head_dim < 1 || dtype == KVC_F32 || kvc_host::elem_bytes_of(dtype) == 0)
        return 0;
    const int g = q_heads / kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16)
        return 0;
    return prefill_ws_bytes(prefill_splits(batch, q_heads, kv_heads, new_tokens, rows_per_head,
                                           local_window_size),
                            batch, q_heads, new_tokens, head_dim);
}

KVC_API kvc_status kvc_gqa_prefill_chunk(void *out, const void *q, const void *k_rows,
                                         const void *v_rows, int64_t rows_per_head,
                                         kvc_lengths len, int batch, int q_heads, int kv_heads,
                                         int new_tokens, int head_dim, int dtype,
                                         int local_window_size, float scale,
                                         const float *rope_cos, const float *rope_sin,
                                         int64_t rope_max_pos, void *workspace,
                                         size_t workspace_bytes, int32_t *dev_status,
                                         void *stream_)
{
    const int eb = kvc_host::elem_bytes_of(dtype);
    if (eb == 0)
        return KVC_ERR_DTYPE;
    if (batch < 0 || q_heads < 1 || kv_heads < 1 || q_heads % kv_heads != 0 || new_tokens < 1 ||
        head_dim < 2 || (head_dim & 1))
        return KVC_ERR_SHAPE;
    if (rows_per_head < new_tokens || rows_per_head > (int64_t)INT32_MAX)
        return KVC_ERR_CAPACITY;
    if ((rope_cos == nullptr) != (rope_sin == nullptr))
        return KVC_ERR_NULL;
    if (rope_cos && rope_max_pos < 1)
        return KVC_ERR_SHAPE;
    const int g = q_heads / kv_heads;
    if (dtype == KVC_F32) {
        if (head_dim > 256)
            return KVC_ERR_UNSUPPORTED;
    } else if ((head_dim != 64 && head_dim != 128 && head_dim != 256) ||
               (g != 1 && g != 2 && g != 4 && g != 8 && g != 16)) {
        return KVC_ERR_UNSUPPORTED;
    }
    if (batch == 0)
        return KVC_OK;
    if (!out || !q || !k_rows || !v_rows || !kvc_host::lengths_ok(len))
        return KVC_ERR_NULL;
    for (const void *p : {(const void *)out, q, k_rows, v_rows})
        if (!kvc_host::aligned16(p))
            return KVC_ERR_ALIGN;
    if (rope_cos && (!kvc_host::aligned16(rope_cos) || !kvc_host::aligned16(rope_sin)))
        return KVC_ERR_ALIGN;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return KVC_ERR_ALIGN;
    if (scale == 0.f)
        scale = 1.0f / sqrtf((float)head_dim);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (dtype == KVC_F32)
        return kvc_f32::launch(out, q, k_rows, v_rows, rows_per_head, len, batch, q_heads,
                               kv_heads, new_tokens, head_dim, local_window_size, scale, rope_cos,
                               rope_sin, rope_max_pos, 1, dev_status, stream);
    if (dtype == KVC_BF16)
        return dispatch_prefill16<__nv_bfloat16>(head_dim, out, q, k_rows, v_rows, rows_per_head,
                                                 len, batch, q_heads, kv_heads, new_tokens,
                                                 local_window_size, scale, rope_cos, rope_sin,
                                                 rope_max_pos, workspace, workspace_bytes,
                                                 dev_status, stream);
    return dispatch_prefill16<__half>(head_dim, out, q, k_rows, v_rows, rows_per_head, len, batch,
                                      q_heads, kv_heads, new_tokens, local_window_size, scale,
                                      rope_cos, rope_sin, rope_max_pos, workspace,
                                      workspace_bytes, dev_status, stream);
}

KVC_API kvc_status kvc_window_prefill_step(void *out, const void *q, void *k_cache, void *v_cache,
                                           const void *new_k, const void *new_v, void *k_stage,
                                           void *v_stage, kvc_lengths len, int batch,
                                           int q_heads, int kv_heads, int new_tokens,
                                           int64_t capacity, int head_dim, int dtype,
                                           int windowed, int local_window_size, float scale,
                                           const float *rope_cos, const float *rope_sin,
                                           int64_t rope_max_pos, void *workspace,
                                           size_t workspace_bytes, int32_t *dev_status,
                                           void *stream_)
{
    const int eb = kvc_host::elem_bytes_of(dtype);
    if (eb == 0)
        return KVC_ERR_DTYPE;
    if (batch < 0 || q_heads < 1 || kv_heads < 1 || q_heads % kv_heads != 0 || new_tokens < 1 ||
        head_dim < 2 || (head_dim & 1))
        return KVC_ERR_SHAPE;
    if (windowed != KVC_WINDOWED && windowed != KVC_DRIFTING)
        return KVC_ERR_UNSUPPORTED;
    if (capacity < 1 || capacity + new_tokens > (int64_t)INT32_MAX)
        return KVC_ERR_CAPACITY;
    if (local_window_size < 1 || local_window_size > capacity)
        return KVC_ERR_WINDOW;
    if ((rope_cos == nullptr) != (rope_sin == nullptr))
        return KVC_ERR_NULL;
    if (rope_cos && rope_max_pos < 1)
        return KVC_ERR_SHAPE;
    const int g = q_heads / kv_heads;
    if (dtype == KVC_F32) {
        if (head_dim > 256)
            return KVC_ERR_UNSUPPORTED;
    } else if ((head_dim != 64 && head_dim != 128 && head_dim != 256) ||
               (g != 1 && g != 2 && g != 4 && g != 8 && g != 16)) {
        return KVC_ERR_UNSUPPORTED;
    }
    if (((int64_t)head_dim * eb) % 16 != 0)
        return KVC_ERR_UNSUPPORTED;
    if (batch == 0)
        return KVC_OK;
    const bool staged = new_tokens > 1;
    if (!out || !q || !k_cache || !v_cache || !new_k || !new_v || !kvc_host::lengths_ok(len) ||
        (staged && (!k_stage || !v_stage)))
        return KVC_ERR_NULL;
    for (const void *p : {(const void *)out, q, (const void *)k_cache, (const void *)v_cache,
                          new_k, new_v, (const void *)(staged ? k_stage : nullptr),
                          (const void *)(staged ? v_stage : nullptr)})
        if (p && !kvc_host::aligned16(p))
            return KVC_ERR_ALIGN;
    if (rope_cos && (!kvc_host::aligned16(rope_cos) || !kvc_host::aligned16(rope_sin)))
        return KVC_ERR_ALIGN;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return KVC_ERR_ALIGN;
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
    if (scale == 0.f)
        scale = 1.0f / sqrtf((float)head_dim);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    const int S = new_tokens, W = local_window_size;
    kvc_status st;
    if (dtype == KVC_F32) {
        // the CUDA-core path: every row through the stage (S = 1: the
        // in-place compaction and one query over the cache)
        st = kvc_window_append(k_cache, v_cache, new_k, new_v, k_stage, v_stage, len, batch,
                               kv_heads, S, capacity, head_dim, dtype, windowed, KVC_APPEND,
                               rope_cos, rope_sin, rope_max_pos, dev_status, stream);
        if (st != KVC_OK)
            return st;
        st = staged ? kvc_f32::launch(out, q, k_stage, v_stage, capacity + S, len, batch, q_heads,
                                      kv_heads, S, head_dim, W, scale, rope_cos, rope_sin,
                                      rope_max_pos, 1, dev_status, stream)
                    : kvc_f32::launch(out, q, k_cache, v_cache, capacity, len, batch, q_heads,
                                      kv_heads, 1, head_dim, W, scale, rope_cos, rope_sin,
                                      rope_max_pos, 0, dev_status, stream);
        if (st != KVC_OK || !staged)
            return st;
        return kvc_window_append(k_cache, v_cache, nullptr, nullptr, k_stage, v_stage, len, batch,
                                 kv_heads, S, capacity, head_dim, dtype, windowed, KVC_COPY_BACK,
                                 rope_cos, rope_sin, rope_max_pos, dev_status, stream);
    }
    st = kvc_host::hazard_rows(k_cache, v_cache, new_k, new_v, k_stage, v_stage, len, batch,
                               kv_heads, S, capacity, head_dim, dtype, W, KVC_APPEND, rope_cos,
                               rope_sin, rope_max_pos, dev_status, stream);
    if (st != KVC_OK)
        return st;
    const AltSource alt{staged ? k_stage : nullptr, staged ? v_stage : nullptr, capacity + S, W};
    st = dtype == KVC_BF16
             ? dispatch_prefill16<__nv_bfloat16>(head_dim, out, q, k_cache, v_cache, capacity,
                                                 len, batch, q_heads, kv_heads, S, W, scale,
                                                 rope_cos, rope_sin, rope_max_pos, workspace,
                                                 workspace_bytes, dev_status, stream, alt)
             : dispatch_prefill16<__half>(head_dim, out, q, k_cache, v_cache, capacity, len,
                                          batch, q_heads, kv_heads, S, W, scale, rope_cos,
                                          rope_sin, rope_max_pos, workspace, workspace_bytes,
                                          dev_status, stream, alt);
    if (st != KVC_OK || !staged)
        return st;
    return kvc_host::hazard_rows(k_cache, v_cache, nullptr, nullptr, k_stage, v_stage, len, batch,
                                 kv_heads, S, capacity, head_dim, dtype, W, KVC_COPY_BACK, rope_cos,
                                 rope_sin, rope_max_pos, dev_status, stream);
}
