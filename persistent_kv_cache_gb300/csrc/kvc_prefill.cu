// kvc_prefill.cu -- attention of a multi-token chunk over staged rows
// ("GQA support sliding_window_cache", section "Design": a step with S > 1
// runs against the C + S staging cache; causal plus local-window mask on
// absolute positions, cache-relative row addressing).
//
// 16-bit path: one CTA per (query block, kv head, batch row) on the 5th-gen
// tensor cores.  The M = 128 tile packs the GQA group: row m holds query head
// m / QB of the group and query qb * QB + m % QB (QB = 128 / group), so every
// K/V tile is read once for all heads of the group.  Q, S, P and O all live
// in tensor memory, which leaves shared memory to the K and V rings:
//
//   TMEM columns  O [0, D) fp32 | S/P double buffer [D, D + 128) | Q [.., + D/2)
//   warp 0        TMA producer of 64-row K tiles (128-byte swizzled boxes of
//                 64 columns) into an NK-stage ring; a stage is refilled as
//                 soon as the S MMA that read it has completed
//   warp 2        the same for V (NV stages), refilled after the PV MMA
//   warp 1        allocates tensor memory and issues tcgen05.mma in the order
//                 S_0, S_1, PV_0, S_2, PV_1, ...:
//                   S_j = Q K_j^T   A = Q in TMEM, B = K tile (K-major)
//                   O  += P_j V_j   A = P_j in TMEM, B = V tile (MN-major)
//                 so the next scores are always queued behind the current PV
//   warps 3-10    two threads per row (= TMEM lane), each owning half of the
//                 score columns and half of O: rotate the query row into
//                 TMEM, then per tile read its S_j half, mask only tiles the
//                 window or diagonal cuts, exchange the row max with the
//                 partner thread, online softmax in the log2 domain (the
//                 running max is only raised when it grows by more than 2^8,
//                 exact after the final division), write P_j as 16-bit pairs
//                 over S_j, rescale its half of O when the max moved, and at
//                 the end divide by l and store its half of the output row.
// Every mbarrier wait is bounded; a timeout sets KVC_DEV_TIMEOUT, every role
// winds down, outstanding tensor-core work is drained and TMEM is freed.
//
// fp32 path: the CUDA-core attn_f32_kernel (kvc_decode.cu).
#include <algorithm>
#include <type_traits>

#include "kvc_common.cuh"

namespace {

constexpr int kBM = 128;       // rows of the M tile (query heads x queries)
constexpr int kBN = 64;        // KV rows per tile
constexpr int kThreads = 352;  // 11 warps
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

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
__device__ __forceinline__ void tmem_st_words(uint32_t taddr, const uint32_t (&w)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                     taddr),
                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
                 "r"(w[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_st_words(uint32_t taddr, const uint32_t (&w)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
                 "r"(w[7]), "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]),
                 "r"(w[13]), "r"(w[14]), "r"(w[15])
                 : "memory");
}

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

__device__ __forceinline__ int t_lo_of(int lo, int j) { return lo + j * 64; }

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

struct PrefillArgs {
    void *out;
    const void *q;
    kvc_lengths len;
    int q_heads, kv_heads, group, qb_rows;  // qb_rows = 128 / group
    int S;
    int64_t rows_per_head;
    int window;
    float scale_log2;
    const float *cos_t, *sin_t;
    int64_t rope_max_pos;
    int32_t *status;
};

template <int D> struct PrefillSmem {
    static constexpr int KV_TILE = kBN * D * 2;          // D/64 boxes of 64 x 64
    static constexpr int NK = D >= 256 ? 3 : 4;          // K ring depth
    static constexpr int NV = D >= 256 ? 3 : 4;          // V ring depth
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + NK * KV_TILE;
    static constexpr int BAR_OFF = V_OFF + NV * KV_TILE;
    // barriers: k_full[4], k_empty[4], v_full[4], v_empty[4], s_full[2],
    //           p_full[2], o_done[2], q_full, drain -> 24 x 8 bytes
    static constexpr int MISC_OFF = BAR_OFF + 24 * 8;  // tmem addr, abort flag
    static constexpr int RED_OFF = MISC_OFF + 16;      // row max / sum exchange, 4 x 128 floats
    static constexpr int TOTAL = RED_OFF + 4 * kBM * 4;
    // TMEM columns: O [0, D), S double buffer [D, D + 128), Q [D + 128, D + 128 + D/2)
    static constexpr uint32_t COL_O = 0, COL_S = D, COL_Q = D + 2 * kBN;
    static constexpr uint32_t TMEM_NEED = D + 2 * kBN + D / 2;
    static constexpr uint32_t TMEM_COLS = TMEM_NEED <= 256 ? 256 : 512;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              int32_t *status)
{
    if (kvc::mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = kvc::global_ns();
    for (uint32_t i = 0;; ++i) {
        if (kvc::mbar_try_wait(bar, parity))
            return true;
        if ((i & 63u) == 63u) {
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

// Stream one operand's 64-row tiles through a ring of NST shared-memory
// stages: stage j % NST is reloaded once the MMA that read its previous
// tile has completed (`empty`, signalled by tcgen05.commit).
template <int NST, int BOXES, int KV_TILE>
__device__ __forceinline__ void produce_tiles(const CUtensorMap *map, uint8_t *ring,
                                              uint64_t *full, uint64_t *empty, int64_t row0,
                                              int ntiles, volatile int *abort_flag,
                                              int32_t *status)
{
    kvc::tma_prefetch_desc(map);
    int issued = 0;
    for (int j = 0; j < ntiles; ++j) {
        const int st = j % NST;
        if (j >= NST && !wait_or_abort(&empty[st], ((j / NST) - 1) & 1, abort_flag, status))
            break;
        uint8_t *dst = ring + st * KV_TILE;
        kvc::mbar_arrive_expect_tx(&full[st], KV_TILE);
        const int32_t y = (int32_t)(row0 + j * kBN);
#pragma unroll
        for (int bx = 0; bx < BOXES; ++bx)
            kvc::tma_load_2d(dst + bx * (kBN * 128), map, bx * 64, y, &full[st]);
        issued = j + 1;
    }
    if (*abort_flag) {
        // wind-down: let the loads already in flight land before the CTA exits
        for (int j = max(0, issued - NST); j < issued; ++j)
            kvc::mbar_wait(&full[j % NST], (j / NST) & 1);
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, const PrefillArgs a)
{
    using SM = PrefillSmem<D>;
    constexpr int BOXES = D / 64;
    constexpr int NK = SM::NK, NV = SM::NV;
    constexpr uint32_t AB = std::is_same<T, __half>::value ? 0u : 1u;
    constexpr uint32_t IDESC_S = f16_idesc(AB, 0, kBM, kBN);
    constexpr uint32_t IDESC_O = f16_idesc(AB, 1, kBM, D);
    constexpr uint32_t COL_O = SM::COL_O, COL_S = SM::COL_S, COL_Q = SM::COL_Q;

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
    uint64_t *k_full = bars + 0, *k_empty = bars + 4, *v_full = bars + 8, *v_empty = bars + 12,
             *s_full = bars + 16, *p_full = bars + 18, *o_done = bars + 20, *q_full = bars + 22,
             *drain = bars + 23;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + SM::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SM::MISC_OFF + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qblk = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int g = a.group, QB = a.qb_rows, S = a.S;

    // ---- per batch row geometry (uniform over the CTA) ----
    const int L = a.len.cache_total[b];
    if (L < 0)
        return;
    const int Lp = a.len.cache_past[b];
    const int P = a.len.past_abs[b];
    if (Lp < 0 || (int64_t)Lp + S > a.rows_per_head) {
        if (threadIdx.x == 0 && qblk == 0 && kvh == 0)
            kvc::raise_status(a.status, KVC_DEV_CAPACITY);
        return;
    }
    if (a.cos_t && (int64_t)P + S > a.rope_max_pos) {
        if (threadIdx.x == 0 && qblk == 0 && kvh == 0)
            kvc::raise_status(a.status, KVC_DEV_ROPE_RANGE);
        return;
    }
    const int q0 = qblk * QB;
    if (q0 >= S)
        return;
    const int q_last = min(S - 1, q0 + QB - 1);
    const int hi = Lp + q_last;  // last visible row of the block
    int lo = 0;
    if (a.window > 0)
        lo = max(0, Lp + q0 - a.window + 1);
    const int ntiles = (hi - lo + kBN) / kBN;
    const int64_t row_base = ((int64_t)b * a.kv_heads + kvh) * a.rows_per_head;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 4; ++i) {
            kvc::mbar_init(&k_full[i], 1);
            kvc::mbar_init(&k_empty[i], 1);
            kvc::mbar_init(&v_full[i], 1);
            kvc::mbar_init(&v_empty[i], 1);
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
    if (warp == 1) {
        tmem_alloc(tmem_slot, SM::TMEM_COLS);
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t smem_base = kvc::smem_u32(smem);

    if (warp == 0) {
        // ======================= K producer =======================
        if (lane == 0)
            produce_tiles<NK, BOXES, SM::KV_TILE>(&tmap_k, smem + SM::K_OFF, k_full, k_empty,
                                                  row_base + lo, ntiles, abort_flag, a.status);
    } else if (warp == 2) {
        // ======================= V producer =======================
        if (lane == 0)
            produce_tiles<NV, BOXES, SM::KV_TILE>(&tmap_v, smem + SM::V_OFF, v_full, v_empty,
                                                  row_base + lo, ntiles, abort_flag, a.status);
    } else if (warp == 1) {
        // ======================= MMA issuer =======================
        // tensor-pipe order: S_0, S_1, PV_0, S_2, PV_1, S_3, ...  S_{j+2}
        // reuses the TMEM buffer that holds P_j, after PV_j in issue order
        if (lane == 0) {
            bool ok = wait_or_abort(q_full, 0, abort_flag, a.status);
            auto issue_s = [&](int j) -> bool {
                const int ks = j % NK;
                if (!wait_or_abort(&k_full[ks], (j / NK) & 1, abort_flag, a.status))
                    return false;
                tc_fence_after();
                const uint32_t kb = smem_base + SM::K_OFF + ks * SM::KV_TILE;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t box = kk >> 2, within = (kk & 3) * 32;
                    const uint64_t bd = sw128_desc(kb + box * (kBN * 128) + within, 16);
                    tc_mma_ts(tmem + COL_S + (j & 1) * kBN, tmem + COL_Q + kk * 8, bd, IDESC_S,
                              kk > 0);
                }
                tc_commit(&s_full[j & 1]);
                tc_commit(&k_empty[ks]);
                return true;
            };
            for (int j = 0; ok && j < 2 && j < ntiles; ++j)
                ok = issue_s(j);
            for (int j = 0; ok && j < ntiles; ++j) {
                const int s = j & 1, vs = j % NV;
                ok = wait_or_abort(&p_full[s], (j >> 1) & 1, abort_flag, a.status) &&
                     wait_or_abort(&v_full[vs], (j / NV) & 1, abort_flag, a.status);
                if (!ok)
                    break;
                tc_fence_after();
                const uint32_t vb = smem_base + SM::V_OFF + vs * SM::KV_TILE;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint64_t bd = sw128_desc(vb + kk * 2048, kBN * 128);
                    tc_mma_ts(tmem + COL_O, tmem + COL_S + s * kBN + kk * 8, bd, IDESC_O,
                              (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&o_done[s]);
                tc_commit(&v_empty[vs]);
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
        // [0, 32) of every tile and O columns [0, D/2), `half` 1 the rest
        const int sw = warp - 3;                   // 0..7
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

        // query row: rotate at absolute position P + ii and store it as packed
        // 16-bit pairs in TMEM (row m = lane m; element e in column COL_Q + e/2).
        // Each half takes half of the rotation pairs (i, i + D/2).
        {
            constexpr int NW = D / 8;  // words of each half's lo (and hi) part
            uint32_t wlo[NW], whi[NW];
            const T *qsrc = static_cast<const T *>(a.q) + qrow * D;
            const float *cs = (a.cos_t && row_valid) ? a.cos_t + (int64_t)(P + ii) * (D / 2) : nullptr;
            const float *sn = (a.cos_t && row_valid) ? a.sin_t + (int64_t)(P + ii) * (D / 2) : nullptr;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                const int c = half * (D / 32) + cc;  // chunk of 8 elements in the low half
                uint4 lo4 = make_uint4(0, 0, 0, 0), hi4 = make_uint4(0, 0, 0, 0);
                if (row_valid) {
                    lo4 = *reinterpret_cast<const uint4 *>(qsrc + c * 8);
                    hi4 = *reinterpret_cast<const uint4 *>(qsrc + D / 2 + c * 8);
                }
                if (cs) {
                    T *lv = reinterpret_cast<T *>(&lo4);
                    T *hv = reinterpret_cast<T *>(&hi4);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        float x = kvc::Elem<T>::to_f32(lv[e]), y = kvc::Elem<T>::to_f32(hv[e]);
                        kvc::rope_pair(x, y, cs[c * 8 + e], sn[c * 8 + e]);
                        lv[e] = kvc::Elem<T>::from_f32(x);
                        hv[e] = kvc::Elem<T>::from_f32(y);
                    }
                }
                wlo[cc * 4 + 0] = lo4.x; wlo[cc * 4 + 1] = lo4.y;
                wlo[cc * 4 + 2] = lo4.z; wlo[cc * 4 + 3] = lo4.w;
                whi[cc * 4 + 0] = hi4.x; whi[cc * 4 + 1] = hi4.y;
                whi[cc * 4 + 2] = hi4.z; whi[cc * 4 + 3] = hi4.w;
            }
            tmem_st_words(lane_addr + COL_Q + half * NW, wlo);
            tmem_st_words(lane_addr + COL_Q + D / 4 + half * NW, whi);
            tmem_wait_st();
            tc_fence_before();
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
            const int t_lo = t_lo_of(lo, j);
            const int c0 = t_lo + 32 * half;  // key row of my first column
            if (!wait_or_abort(&s_full[s], (j >> 1) & 1, abort_flag, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float v[32];
            tmem_ld32(lane_addr + COL_S + s * kBN + 32 * half, v);

            // mask only where the window or the diagonal cuts these columns
            const bool all_in = row_valid && c0 >= r_lo && c0 + 31 <= r_hi;
            if (!all_in) {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int r = c0 + c;
                    v[c] = (row_valid && r >= r_lo && r <= r_hi) ? v[c] : -INFINITY;
                }
            }
            float mx0 = fmaxf(v[0], v[1]), mx1 = fmaxf(v[2], v[3]);
#pragma unroll
            for (int c = 4; c < 32; c += 4) {
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
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
                const float p0 = fast_exp2(fmaf(v[c], c_log2, neg_m));
                const float p1 = fast_exp2(fmaf(v[c + 1], c_log2, neg_m));
                ps0 += p0;
                ps1 += p1;
                pk[c / 2] = pack2<T>(p0, p1);
            }
            l_run = l_run * alpha + (ps0 + ps1);
            // P_j (16-bit pairs) over the S_j columns of this row
            tmem_st_words(lane_addr + COL_S + s * kBN + 16 * half, pk);

            // rows past the last visible row of the block: zero V so that
            // 0 * (stale or uninitialised bytes) stays 0 in O += P V
            if (t_lo + kBN - 1 > hi) {
                const int vs = j % NV;
                if (!wait_or_abort(&v_full[vs], (j / NV) & 1, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                const int first_bad = hi + 1 - t_lo;  // rows [first_bad, 64) of the tile
                uint8_t *vt = smem + SM::V_OFF + vs * SM::KV_TILE;
                const int nbad = kBN - first_bad;
                for (int idx = threadIdx.x - 96; idx < nbad * BOXES * 8; idx += 256) {
                    const int rr = first_bad + idx / (BOXES * 8);
                    const int bx = (idx / 8) % BOXES, cc = idx % 8;
                    *reinterpret_cast<uint4 *>(vt + bx * (kBN * 128) + rr * 128 + cc * 16) =
                        make_uint4(0, 0, 0, 0);
                }
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

        // epilogue: combine the two halves' sums, wait for the last PV,
        // divide by l and store my half of the output row
        // (the buffer of parity ntiles & 1 was last read before the final tile's barrier)
        red[((ntiles & 1) * 2 + half) * kBM + m] = l_run;
        named_bar_sync(pair_bar, 64);
        const float l_tot = l_run + red[((ntiles & 1) * 2 + (half ^ 1)) * kBM + m];
        if (ok && ntiles > 0 &&
            wait_or_abort(&o_done[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, abort_flag,
                          a.status)) {
            tc_fence_after();
            const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
            T *dst = static_cast<T *>(a.out) + qrow * D;
#pragma unroll 1
            for (int cc = half * (D / 2); cc < (half + 1) * (D / 2); cc += 32) {
                float o[32];
                tmem_ld32(lane_addr + COL_O + cc, o);
                if (row_valid) {
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        uint4 pkt;
                        T *e = reinterpret_cast<T *>(&pkt);
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            e[u] = kvc::Elem<T>::from_f32(o[c + u] * inv);
                        *reinterpret_cast<uint4 *>(dst + cc + c) = pkt;
                    }
                }
            }
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, SM::TMEM_COLS);
    }
}

template <typename T, int D>
kvc_status launch_prefill_tc(void *out, const void *q, const void *k_rows, const void *v_rows,
                             int64_t R, const kvc_lengths &len, int batch, int q_heads,
                             int kv_heads, int S, int window, float scale, const float *cos_t,
                             const float *sin_t, int64_t rope_max_pos, int32_t *status,
                             cudaStream_t stream)
{
    using SM = PrefillSmem<D>;
    const CUtensorMapDataType tt = std::is_same<T, __half>::value
                                       ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t rows = (uint64_t)batch * kv_heads * R;
    if (rows > (uint64_t)INT32_MAX)
        return KVC_ERR_SHAPE;
    CUtensorMap tk, tv;
    if (!kvc_host::encode_2d_bf16_sw128(&tk, k_rows, rows, D, kBN, tt) ||
        !kvc_host::encode_2d_bf16_sw128(&tv, v_rows, rows, D, kBN, tt))
        return KVC_ERR_CUDA;
    PrefillArgs a;
    a.out = out;
    a.q = q;
    a.len = len;
    a.q_heads = q_heads;
    a.kv_heads = kv_heads;
    a.group = q_heads / kv_heads;
    a.qb_rows = kBM / a.group;
    a.S = S;
    a.rows_per_head = R;
    a.window = window;
    a.scale_log2 = scale * kLog2e;
    a.cos_t = cos_t;
    a.sin_t = sin_t;
    a.rope_max_pos = rope_max_pos;
    a.status = status;
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    const size_t smem = std::min<size_t>((size_t)SM::TOTAL + 1024, (size_t)optin);
    if (smem < (size_t)SM::TOTAL)
        return KVC_ERR_UNSUPPORTED;
    auto kern = prefill_tc_kernel<T, D>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return KVC_ERR_CUDA;
    const int qblocks = (S + a.qb_rows - 1) / a.qb_rows;
    dim3 grid(qblocks, kv_heads, batch);
    kern<<<grid, kThreads, smem, stream>>>(tk, tv, a);
    return kvc_host::launch_status();
}

template <typename T>
kvc_status dispatch_prefill16(int D, void *out, const void *q, const void *k, const void *v,
                              int64_t R, const kvc_lengths &len, int B, int Hq, int Hkv, int S,
                              int W, float scale, const float *cs, const float *sn, int64_t rmax,
                              int32_t *st, cudaStream_t stream)
{
    switch (D) {
    case 64:
        return launch_prefill_tc<T, 64>(out, q, k, v, R, len, B, Hq, Hkv, S, W, scale, cs, sn,
                                        rmax, st, stream);
    case 128:
        return launch_prefill_tc<T, 128>(out, q, k, v, R, len, B, Hq, Hkv, S, W, scale, cs, sn,
                                         rmax, st, stream);
    case 256:
        return launch_prefill_tc<T, 256>(out, q, k, v, R, len, B, Hq, Hkv, S, W, scale, cs, sn,
                                         rmax, st, stream);
    default:
        return KVC_ERR_UNSUPPORTED;
    }
}

} // namespace

KVC_API kvc_status kvc_gqa_prefill_chunk(void *out, const void *q, const void *k_rows,
                                         const void *v_rows, int64_t rows_per_head,
                                         kvc_lengths len, int batch, int q_heads, int kv_heads,
                                         int new_tokens, int head_dim, int dtype,
                                         int local_window_size, float scale,
                                         const float *rope_cos, const float *rope_sin,
                                         int64_t rope_max_pos, int32_t *dev_status, void *stream_)
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
                                                 rope_max_pos, dev_status, stream);
    return dispatch_prefill16<__half>(head_dim, out, q, k_rows, v_rows, rows_per_head, len, batch,
                                      q_heads, kv_heads, new_tokens, local_window_size, scale,
                                      rope_cos, rope_sin, rope_max_pos, dev_status, stream);
}
