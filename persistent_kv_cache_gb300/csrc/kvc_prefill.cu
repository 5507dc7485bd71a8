// kvc_prefill.cu -- attention of a multi-token chunk over staged rows
// ("GQA support sliding_window_cache", section "Design": a step with S > 1
// runs against the C + S staging cache; causal plus local-window mask on
// absolute positions, cache-relative row addressing).
//
// 16-bit path: one CTA per (query block, kv head, batch row) on the 5th-gen
// tensor cores.  The M = 128 tile packs the GQA group: row m holds query head
// m / QB of the group and query qb * QB + m % QB (QB = 128 / group), so every
// K/V tile is read once for all heads of the group.
//
//   warp 0      TMA producer: 64-row K and V tiles (128-byte swizzled boxes
//               of 64 columns) into a 2-stage ring (full/empty mbarriers)
//   warp 1      allocates tensor memory and issues tcgen05.mma:
//                 S_j = Q K_j^T   (M 128, N 64,  K = D)  -> TMEM, 2 buffers
//                 O  += P_j V_j   (M 128, N = D, K = 64)  -> TMEM
//               S_{j+1} is issued before waiting for P_j, so the tensor
//               cores compute the next scores while the softmax runs
//   warps 2-5   one thread per row (= TMEM lane): rotate and stage the query
//               row, then per tile read S_j from TMEM, mask, online softmax
//               (log2 domain, the running max is only raised when it grows
//               by more than 2^8, which keeps the result exact after the
//               final division), write P_j as bf16 into a swizzled shared
//               tile, rescale the O row in TMEM when the max moved, and at
//               the end divide by l and store the output row.
// Every mbarrier wait is bounded; a timeout sets KVC_DEV_TIMEOUT, every role
// winds down, outstanding tensor-core work is drained and TMEM is freed.
//
// fp32 path: the CUDA-core attn_f32_kernel (kvc_decode.cu).
#include <type_traits>

#include "kvc_common.cuh"

namespace {

constexpr int kBM = 128;       // rows of the M tile (query heads x queries)
constexpr int kBN = 64;        // KV rows per tile
constexpr int kStages = 2;     // K/V ring depth
constexpr int kThreads = 192;  // 6 warps
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

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16, one CTA
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
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

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

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
    static constexpr int Q_BYTES = kBM * D * 2;        // D/64 boxes of 128 x 64
    static constexpr int KV_TILE = kBN * D * 2;        // D/64 boxes of 64 x 64
    static constexpr int P_BYTES = kBM * kBN * 2;      // one 128 x 64 box
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + Q_BYTES;
    static constexpr int V_OFF = K_OFF + kStages * KV_TILE;
    static constexpr int P_OFF = V_OFF + kStages * KV_TILE;
    static constexpr int BAR_OFF = P_OFF + 2 * P_BYTES;
    // barriers: k_full[2], v_full[2], kv_empty[2], s_full[2], s_empty[2],
    //           p_full[2], o_done[2], q_full, drain  -> 16 x 8 bytes
    static constexpr int MISC_OFF = BAR_OFF + 16 * 8;  // tmem addr, abort flag
    static constexpr int TOTAL = MISC_OFF + 16;
    static constexpr uint32_t TMEM_COLS = (D + 2 * kBN) <= 256 ? 256 : 512;
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

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, const PrefillArgs a)
{
    using SM = PrefillSmem<D>;
    constexpr int BOXES = D / 64;
    constexpr uint32_t AB = std::is_same<T, __half>::value ? 0u : 1u;
    constexpr uint32_t IDESC_S = f16_idesc(AB, 0, kBM, kBN);
    constexpr uint32_t IDESC_O = f16_idesc(AB, 1, kBM, D);
    constexpr uint32_t COL_O = 0, COL_S = D;  // TMEM columns: O [0, D), S buffers after

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SM::BAR_OFF);
    uint64_t *k_full = bars + 0, *v_full = bars + 2, *kv_empty = bars + 4, *s_full = bars + 6,
             *s_empty = bars + 8, *p_full = bars + 10, *o_done = bars + 12, *q_full = bars + 14,
             *drain = bars + 15;
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
        for (int i = 0; i < 2; ++i) {
            kvc::mbar_init(&k_full[i], 1);
            kvc::mbar_init(&v_full[i], 1);
            kvc::mbar_init(&kv_empty[i], 1);
            kvc::mbar_init(&s_full[i], 1);
            kvc::mbar_init(&s_empty[i], 4);
            kvc::mbar_init(&p_full[i], 4);
            kvc::mbar_init(&o_done[i], 1);
        }
        kvc::mbar_init(q_full, 4);
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
        // ======================= TMA producer =======================
        if (lane == 0) {
            kvc::tma_prefetch_desc(&tmap_k);
            kvc::tma_prefetch_desc(&tmap_v);
            int issued = 0;
            for (int j = 0; j < ntiles; ++j) {
                const int s = j & 1;
                if (j >= kStages &&
                    !wait_or_abort(&kv_empty[s], ((j >> 1) - 1) & 1, abort_flag, a.status))
                    break;
                const int32_t y = (int32_t)(row_base + lo + j * kBN);
                uint8_t *kd = smem + SM::K_OFF + s * SM::KV_TILE;
                uint8_t *vd = smem + SM::V_OFF + s * SM::KV_TILE;
                kvc::mbar_arrive_expect_tx(&k_full[s], SM::KV_TILE);
#pragma unroll
                for (int bx = 0; bx < BOXES; ++bx)
                    kvc::tma_load_2d(kd + bx * (kBN * 128), &tmap_k, bx * 64, y, &k_full[s]);
                kvc::mbar_arrive_expect_tx(&v_full[s], SM::KV_TILE);
#pragma unroll
                for (int bx = 0; bx < BOXES; ++bx)
                    kvc::tma_load_2d(vd + bx * (kBN * 128), &tmap_v, bx * 64, y, &v_full[s]);
                issued = j + 1;
            }
            if (*abort_flag) {
                // wind-down: let the last loads land before the CTA exits
                for (int j = max(0, issued - kStages); j < issued; ++j) {
                    kvc::mbar_wait(&k_full[j & 1], (j >> 1) & 1);
                    kvc::mbar_wait(&v_full[j & 1], (j >> 1) & 1);
                }
            }
        }
    } else if (warp == 1) {
        // ======================= MMA issuer =======================
        if (lane == 0) {
            bool ok = wait_or_abort(q_full, 0, abort_flag, a.status);
            auto issue_s = [&](int j) {
                const int s = j & 1;
                const uint32_t qa = smem_base + SM::Q_OFF;
                const uint32_t kb = smem_base + SM::K_OFF + s * SM::KV_TILE;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t box = kk >> 2, within = (kk & 3) * 32;
                    const uint64_t ad = sw128_desc(qa + box * (kBM * 128) + within, 16);
                    const uint64_t bd = sw128_desc(kb + box * (kBN * 128) + within, 16);
                    tc_mma(tmem + COL_S + s * kBN, ad, bd, IDESC_S, kk > 0);
                }
                tc_commit(&s_full[s]);
            };
            if (ok && ntiles > 0) {
                ok = wait_or_abort(&k_full[0], 0, abort_flag, a.status);
                if (ok) {
                    tc_fence_after();
                    issue_s(0);
                }
            }
            for (int j = 0; ok && j < ntiles; ++j) {
                const int s = j & 1;
                if (j + 1 < ntiles) {
                    const int n = j + 1, sn = n & 1;
                    if (n >= 2)
                        ok = wait_or_abort(&s_empty[sn], ((n >> 1) - 1) & 1, abort_flag, a.status);
                    if (ok)
                        ok = wait_or_abort(&k_full[sn], (n >> 1) & 1, abort_flag, a.status);
                    if (!ok)
                        break;
                    tc_fence_after();
                    issue_s(n);
                }
                ok = wait_or_abort(&p_full[s], (j >> 1) & 1, abort_flag, a.status) &&
                     wait_or_abort(&v_full[s], (j >> 1) & 1, abort_flag, a.status);
                if (!ok)
                    break;
                tc_fence_after();
                const uint32_t pa = smem_base + SM::P_OFF + s * SM::P_BYTES;
                const uint32_t vb = smem_base + SM::V_OFF + s * SM::KV_TILE;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint64_t ad = sw128_desc(pa + kk * 32, 16);
                    const uint64_t bd = sw128_desc(vb + kk * 2048, kBN * 128);
                    tc_mma(tmem + COL_O, ad, bd, IDESC_O, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&o_done[s]);
                tc_commit(&kv_empty[s]);
            }
            // drain: everything issued above has completed once this arrives
            // (a plain bounded wait, also on the abort path)
            tc_commit(drain);
            kvc::mbar_wait(drain, 0);
        }
    } else {
        // ======================= softmax / epilogue =======================
        const int quad = warp & 3;                 // TMEM lane quadrant of this warp
        const int m = quad * 32 + lane;            // tile row == TMEM lane
        const int hh = m / QB;                     // head within the group
        const int ii = q0 + (m - hh * QB);         // query index in the chunk
        const bool row_valid = ii < S && hh < g;
        const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
        const int64_t qrow = ((int64_t)b * a.q_heads + kvh * g + hh) * S + ii;

        // query row: rotate at absolute position P + ii, stage as bf16/f16 in
        // the swizzled Q tile (row m of each 64-column box)
        {
            const T *qsrc = static_cast<const T *>(a.q) + qrow * D;
            const float *cs = (a.cos_t && row_valid) ? a.cos_t + (int64_t)(P + ii) * (D / 2) : nullptr;
            const float *sn = (a.cos_t && row_valid) ? a.sin_t + (int64_t)(P + ii) * (D / 2) : nullptr;
            uint8_t *qt = smem + SM::Q_OFF;
#pragma unroll 1
            for (int c = 0; c < D / 16; ++c) {  // chunk of 8 elements in each half
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
                const int clo = c, chi = D / 16 + c;  // 16-byte chunk index along D
                *reinterpret_cast<uint4 *>(qt + (clo >> 3) * (kBM * 128) + kvc::sw128(m, clo & 7)) = lo4;
                *reinterpret_cast<uint4 *>(qt + (chi >> 3) * (kBM * 128) + kvc::sw128(m, chi & 7)) = hi4;
            }
            kvc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                kvc::mbar_arrive(q_full);
        }

        // visible rows of this query: [r_lo, r_hi]
        const int r_hi = Lp + ii;
        const int r_lo = a.window > 0 ? max(0, r_hi - a.window + 1) : 0;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const int s = j & 1;
            const int t_lo = lo + j * kBN;
            if (!wait_or_abort(&s_full[s], (j >> 1) & 1, abort_flag, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float sc[kBN];
            {
                float v[32];
                tmem_ld32(lane_addr + COL_S + s * kBN, v);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    sc[i] = v[i];
                tmem_ld32(lane_addr + COL_S + s * kBN + 32, v);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    sc[32 + i] = v[i];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                kvc::mbar_arrive(&s_empty[s]);

            float mt = -INFINITY;
#pragma unroll
            for (int c = 0; c < kBN; ++c) {
                const int r = t_lo + c;
                const bool vis = row_valid && r >= r_lo && r <= r_hi;
                sc[c] = vis ? sc[c] * a.scale_log2 : -INFINITY;
                mt = fmaxf(mt, sc[c]);
            }
            float alpha = 1.f;
            bool rescale = false;
            if (mt > m_run + kRescaleThreshold || (m_run == -INFINITY && mt > -INFINITY)) {
                if (j > 0 && m_run > -INFINITY) {
                    alpha = exp2f(m_run - mt);
                    rescale = true;
                }
                m_run = mt;
            }
            const float m_use = m_run == -INFINITY ? 0.f : m_run;
            float psum = 0.f;
            uint32_t pk[kBN / 2];
#pragma unroll
            for (int c = 0; c < kBN; c += 2) {
                const float p0 = exp2f(sc[c] - m_use), p1 = exp2f(sc[c + 1] - m_use);
                psum += p0 + p1;
                if constexpr (std::is_same<T, __half>::value) {
                    __half2 h = __floats2half2_rn(p0, p1);
                    pk[c / 2] = *reinterpret_cast<uint32_t *>(&h);
                } else {
                    __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
                    pk[c / 2] = *reinterpret_cast<uint32_t *>(&h);
                }
            }
            l_run = l_run * alpha + psum;

            // P_j goes to buffer s, last read by PV_{j-2}
            if (j >= 2 && !wait_or_abort(&o_done[s], ((j >> 1) - 1) & 1, abort_flag, a.status)) {
                ok = false;
                break;
            }
            uint8_t *pt = smem + SM::P_OFF + s * SM::P_BYTES;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4 *>(pt + kvc::sw128(m, c)) =
                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);

            // rows past the last visible row of the block: zero V so that
            // 0 * (stale or uninitialised bytes) stays 0 in O += P V
            if (t_lo + kBN - 1 > hi) {
                if (!wait_or_abort(&v_full[s], (j >> 1) & 1, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                const int first_bad = hi + 1 - t_lo;  // rows [first_bad, 64) of the tile
                uint8_t *vt = smem + SM::V_OFF + s * SM::KV_TILE;
                const int nbad = kBN - first_bad;
                for (int idx = threadIdx.x - 64; idx < nbad * BOXES * 8; idx += 128) {
                    const int rr = first_bad + idx / (BOXES * 8);
                    const int bx = (idx / 8) % BOXES, c = idx % 8;
                    *reinterpret_cast<uint4 *>(vt + bx * (kBN * 128) + rr * 128 + c * 16) =
                        make_uint4(0, 0, 0, 0);
                }
            }

            // the running max moved: rescale this row of O (PV_{j-1} must be done)
            if (__any_sync(0xffffffffu, rescale)) {
                if (!wait_or_abort(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag,
                                   a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    float v[32];
                    tmem_ld32(lane_addr + COL_O + c0, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[i] *= alpha;
                    tmem_st32(lane_addr + COL_O + c0, v);
                }
                tmem_wait_st();
            }
            kvc::fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                kvc::mbar_arrive(&p_full[s]);
        }

        // epilogue: wait for the last PV, divide by l, store the row
        if (ok && ntiles > 0 &&
            wait_or_abort(&o_done[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, abort_flag,
                          a.status)) {
            tc_fence_after();
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            T *dst = static_cast<T *>(a.out) + qrow * D;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                float v[32];
                tmem_ld32(lane_addr + COL_O + c0, v);
                if (row_valid) {
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        uint4 pkt;
                        T *e = reinterpret_cast<T *>(&pkt);
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            e[u] = kvc::Elem<T>::from_f32(v[c + u] * inv);
                        *reinterpret_cast<uint4 *>(dst + c0 + c) = pkt;
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
    const size_t smem = SM::TOTAL + 1024;
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
