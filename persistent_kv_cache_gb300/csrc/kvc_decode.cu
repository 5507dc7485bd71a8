// kvc_decode.cu -- one-token grouped-query attention over the persistent cache
// ("Persistent KV Cache and Decode Performance Roadmap", section "Phase 1":
// stream KV blocks, update the online-softmax state, accumulate V, never store
// the score vector; heads that share a KV head read each block once; one
// query row may be split across workers when the outer dimensions cannot fill
// the machine, with an (m, l, o) merge.  Masks and cache-relative addressing
// from "GQA support sliding_window_cache", section "Design").
//
// 16-bit path (bf16 / fp16), one CTA per (split, kv head, batch row):
//   * warp 4 is the producer: one lane issues 2-D TMA loads of 64-row K and V
//     tiles (128-byte swizzled boxes of 64 columns) into an NS-stage ring of
//     shared-memory buffers guarded by full/empty mbarriers;
//   * warps 0-3 consume 16 rows of every tile each: S^T = K Q^T and
//     O^T += V^T P^T on the tensor cores (mma.sync m16n8k16, fp32 accumulate)
//     with the warp's 16 keys as the M dimension and the GQA group's query
//     heads as N, online softmax in registers with shuffles across the
//     warp's key lanes, then a 4-way (m, l, o) merge through shared memory;
//   * a split whose row holds more than one split writes (m, l, o) partials to
//     the workspace and decode_combine_kernel merges them; a single split
//     writes the output directly.
// The visible rows are the newest n positions.  In a cache they are rows
// [L - n, L); in a ring of C slots ("Stateful decode & KV cache",
// "Sliding-window ring buffer") they start at slot (T - n) mod C and wrap, so
// a split's rows are at most two contiguous runs of slots, each streamed as
// its own sequence of tiles (a tile never crosses the wrap).
// The fused step (kvc_decode_step) runs the same kernel with the lengths
// derived inline from seqlens_k, the new K/V row patched into the last tile
// in shared memory (and stored to the cache) by the split that owns the
// newest position; the split merge is a second launch.
// fp32 path: attn_f32_kernel, one warp per query row on CUDA cores (also used
// by the multi-token call for fp32).
#include <atomic>
#include <cfloat>
#include <mutex>
#include <type_traits>

#include "kvc_common.cuh"

namespace {

constexpr int kTile = 64;      // cache rows per TMA tile
constexpr int kConsumers = 4;  // consumer warps
constexpr float kLog2e = 1.4426950408889634f;

__host__ __device__ constexpr int decode_stages(int D) { return D >= 128 ? 3 : 4; }

// rows handled by one CTA (a multiple of the tile); shared by the kernel launch
// and the workspace size so both agree
constexpr int64_t kSplitRowsD256 = 1024;
inline int64_t decode_split_rows(int64_t C, int D)
{
    if (C >= 2048)
        return D >= 256 ? kSplitRowsD256 : 512;
    return (C + kTile - 1) / kTile * kTile;
}
inline int64_t decode_max_splits(int64_t C, int D)
{
    const int64_t sr = decode_split_rows(C, D);
    return (C + sr - 1) / sr;
}

template <typename T> struct Mma;
template <> struct Mma<__nv_bfloat16> {
    static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1)
    {
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                     "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                     : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi)
    {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    }
};
template <> struct Mma<__half> {
    static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1)
    {
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                     "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                     : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi)
    {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    }
};

// (lo, hi) rounded to bf16 and handed on as an fp16 pair: the same numbers
// whenever each rounded value is 0 or of magnitude in [2^-17, 65504] (its 8
// significant bits fit an fp16 normal or subnormal there)
__device__ __forceinline__ uint32_t pack_bf16_as_f16(float lo, float hi)
{
    const uint32_t b = Mma<__nv_bfloat16>::pack(lo, hi);
    return Mma<__half>::pack(__uint_as_float(b << 16), __uint_as_float(b & 0xffff0000u));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                          uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// consumer_sync() that also returns whether v holds in every consumer thread
__device__ __forceinline__ bool consumer_all(bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "setp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.and.pred q, 1, 128, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)v)
                 : "memory");
    return r != 0;
}

// 16 bytes from shared memory (a 32-bit shared-window address)
__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// 8x8 16-bit matrix held as a fragment (thread t: row t / 4, columns
// 2 (t % 4) and 2 (t % 4) + 1) -> the same fragment of its transpose
__device__ __forceinline__ uint32_t movm_trans(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// u - zp for the four unsigned bytes of w, exactly, as two 16-bit pairs
// (bytes 0, 1 -> lo; bytes 2, 3 -> hi): byte u goes into the low mantissa
// byte of 2^23 (0x4B000000), so the float is 2^23 + u, and one packed
// subtraction of off2 = (2^23 + zp) x 2 leaves u - zp for two bytes at once
// (|u - zp| <= 255: exact in fp32 and in bf16 / f16).
template <typename T>
__device__ __forceinline__ void u8x4_to_pairs(uint32_t w, uint64_t off2, uint32_t &lo, uint32_t &hi)
{
    const uint32_t b0 = __byte_perm(w, 0x4B000000u, 0x7540);
    const uint32_t b1 = __byte_perm(w, 0x4B000000u, 0x7541);
    const uint32_t b2 = __byte_perm(w, 0x4B000000u, 0x7542);
    const uint32_t b3 = __byte_perm(w, 0x4B000000u, 0x7543);
    uint64_t p01, p23;
    asm("mov.b64 %0, {%1, %2};" : "=l"(p01) : "r"(b0), "r"(b1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(p23) : "r"(b2), "r"(b3));
    asm("sub.rn.f32x2 %0, %0, %1;" : "+l"(p01) : "l"(off2));
    asm("sub.rn.f32x2 %0, %0, %1;" : "+l"(p23) : "l"(off2));
    float f0, f1, f2, f3;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f0), "=f"(f1) : "l"(p01));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f2), "=f"(f3) : "l"(p23));
    lo = Mma<T>::pack(f0, f1);
    hi = Mma<T>::pack(f2, f3);
}

// f16: byte u under the high byte 0x64 is the half 1024 + u (spacing 1 in
// [1024, 2048)), one byte permute for two codes, and one f16x2 subtraction
// of off2 = (1024 + zp) x 2 leaves u - zp exactly -- the same halves as the
// float route above, at a third of its ALU work
template <>
__device__ __forceinline__ void u8x4_to_pairs<__half>(uint32_t w, uint64_t off2, uint32_t &lo,
                                                      uint32_t &hi)
{
    const uint32_t l = __byte_perm(w, 0x64646464u, 0x4140);
    const uint32_t h = __byte_perm(w, 0x64646464u, 0x4342);
    const uint32_t o = (uint32_t)off2;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(l), "r"(o));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(h), "r"(o));
}

// the per-tile constant off2 of u8x4_to_pairs<T> for a zero point zp
// (an integer in [0, 255])
template <typename T> __device__ __forceinline__ uint64_t q8_offset(float zp)
{
    if constexpr (std::is_same<T, __half>::value) {
        const __half2 h = __float2half2_rn(1024.f + zp);
        return *reinterpret_cast<const uint32_t *>(&h);
    } else {
        const uint32_t f = __float_as_uint(8388608.f + zp);
        return ((uint64_t)f << 32) | f;
    }
}

// Attention state of one consumer warp over 64-row K/V tiles held in shared
// memory (128-byte swizzled boxes of 64 columns, 8 KB per box).  The warp
// owns rows [16 w, 16 w + 16) of every tile.  Those 16 keys are the M = 16
// rows of mma.sync m16n8k16 and the GQA group's query heads its N columns,
// in HB blocks of 8 heads:
//   scores   S^T[key][head]  = K[key][:] . Q[head][:]          (A = K, B = Q^T)
//   output   O^T[dim][head] += V^T[dim][key] . P^T[key][head]  (A = V^T, B = P^T)
// so a group of up to 8 heads costs one MMA per 16 keys x 16 columns for the
// scores and one per 16 columns for the output, and padding heads (zero
// queries, never published) take the N columns a group leaves free.
// Thread t (gid = t / 4, tig = t % 4) holds, per head block, the scores of
// keys gid and gid + 8 for heads 2 tig and 2 tig + 1, and the output of
// columns 16 mb + gid and 16 mb + gid + 8 for those two heads.  (m, l)
// follow the online softmax per head in the log2 domain; l sums this
// thread's keys only, until publish().
template <typename T, int D, int HB, bool QREG_ = true, bool SHORTCUTS = false>
struct GroupAttn {
    static constexpr int MB = D / 16;  // 16-column blocks of the head dim
    // the query's B fragments stay in registers, or (QREG false: head_dim
    // 256 with two head blocks, where the output alone takes 128 registers a
    // thread) are read from the staged rows, two 16-column blocks an ldmatrix
    static constexpr bool QREG = QREG_;
    uint32_t qb[QREG ? HB : 1][QREG ? MB : 1][2];
    uint32_t q_addr, q_hstride;  // !QREG: this lane's ldmatrix row address; bytes per 8 heads
    // int8 tiles of a bf16 cache: this lane's ldmatrix row address in the
    // fp16 copy of the query rows (load_q16)
    uint32_t q16_addr;
    float o[HB][MB][4];
    float m[HB][2], l[HB][2];

    __device__ __forceinline__ void init()
    {
#pragma unroll
        for (int hb = 0; hb < HB; ++hb) {
#pragma unroll
            for (int mb = 0; mb < MB; ++mb)
                o[hb][mb][0] = o[hb][mb][1] = o[hb][mb][2] = o[hb][mb][3] = 0.f;
            m[hb][0] = m[hb][1] = -INFINITY;
            l[hb][0] = l[hb][1] = 0.f;
        }
    }

    // B fragments of query columns [16 kk, 16 kk + 32) of head block hb:
    // f[0], f[1] for block kk, f[2], f[3] for block kk + 1 (kk even)
    __device__ __forceinline__ void q_frag2(int hb, int kk, uint32_t (&f)[4]) const
    {
        if constexpr (QREG) {
            f[0] = qb[hb][kk][0];
            f[1] = qb[hb][kk][1];
            f[2] = qb[hb][kk + 1][0];
            f[3] = qb[hb][kk + 1][1];
        } else {
            ldsm_x4(q_addr + hb * q_hstride + kk * 32, f[0], f[1], f[2], f[3]);
        }
    }

    // fp16 B fragments of query columns [16 kk, 16 kk + 32) of head block hb
    // from the fp16 copy of the rows
    __device__ __forceinline__ void q16_frag2(int hb, int kk, uint32_t (&f)[4]) const
    {
        ldsm_x4(q16_addr + hb * 8 * (D + 8) * 2 + kk * 32, f[0], f[1], f[2], f[3]);
    }
    // the fp16 copy [16][D + 8] of the query rows, for the int8 tiles of a
    // bf16 cache (used only when every element is 0 or of magnitude in
    // [2^-17, 65504], where a bf16 value is exact in fp16)
    __device__ __forceinline__ void load_q16(const __half *qs16, int lane)
    {
        q16_addr = kvc::smem_u32(qs16 + (lane & 7) * (D + 8) + (lane >> 3) * 8);
    }

    // the rotated query rows staged as qs[16][QS] (heads >= g zero; at
    // QREG false the rows must stay in place while the tiles are attended)
    __device__ __forceinline__ void load_q(const T *qs, int QS, int lane)
    {
        if constexpr (!QREG) {
            // ldmatrix x4: lanes 8 m .. 8 m + 7 address head rows 0-7 at
            // columns 8 m .. 8 m + 7 of a 32-column span
            q_addr = kvc::smem_u32(qs + (lane & 7) * QS + (lane >> 3) * 8);
            q_hstride = 8 * QS * 2;
            return;
        }
        const int gid = lane >> 2, c = (lane & 3) * 2;
#pragma unroll
        for (int hb = 0; hb < HB; ++hb)
#pragma unroll
            for (int kk = 0; kk < MB; ++kk) {
                const T *r = qs + (8 * hb + gid) * QS + 16 * kk + c;
                qb[hb][kk][0] = *reinterpret_cast<const uint32_t *>(r);
                qb[hb][kk][1] = *reinterpret_cast<const uint32_t *>(r + 8);
            }
    }

    // Online-softmax update with the raw scores sc of this warp's 16 keys:
    // mask keys outside [lo, hi), move the reference max, rescale l and o,
    // and pack P (times vscale; VS false: times 1) as the B fragments of
    // the output MMAs, in T or, F16P, rounded to bf16 and handed on as fp16
    // (pack_bf16_as_f16).  The reference max of a head moves only when the
    // tile's max exceeds it by more than 8 (log2 units), so P stays at or
    // below 2^8 and o and l are rescaled on few tiles after the first (O / l
    // is the same for any reference).  SHORTCUTS (the split kernel): the
    // key mask is skipped on tiles whose 16 keys are all visible.
    template <bool VS, bool F16P = false>
    __device__ __forceinline__ void softmax_step(float (&sc)[HB][4], int lane, int lo, int hi,
                                                 float scale_log2, float vscale,
                                                 uint32_t (&pb)[HB][2])
    {
        const int k0 = lane >> 2, k1 = k0 + 8;  // this thread's keys
        const bool whole = SHORTCUTS && lo == 0 && hi == 16;  // every key visible
        const bool in0 = whole || (k0 >= lo && k0 < hi);
        const bool in1 = whole || (k1 >= lo && k1 < hi);
        float mx[HB][2];
        bool up = false;
#pragma unroll
        for (int hb = 0; hb < HB; ++hb)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float v0 = sc[hb][j] * scale_log2, v1 = sc[hb][2 + j] * scale_log2;
                if (!whole) {
                    v0 = in0 ? v0 : -INFINITY;
                    v1 = in1 ? v1 : -INFINITY;
                }
                sc[hb][j] = v0;
                sc[hb][2 + j] = v1;
                float x = fmaxf(v0, v1);
                x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
                x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 8));
                x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 16));
                mx[hb][j] = x;
                // (false for a fully masked tile; true for the first visible
                // keys of a head, whose m is still -inf)
                up |= x > m[hb][j] + 8.f;
            }
        if (__any_sync(0xffffffffu, up)) {
#pragma unroll
            for (int hb = 0; hb < HB; ++hb) {
                float al[2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const bool u = mx[hb][j] > m[hb][j] + 8.f;
                    const float mn = u ? mx[hb][j] : m[hb][j];
                    al[j] = u ? exp2f(m[hb][j] - mn) : 1.f;
                    m[hb][j] = mn;
                    l[hb][j] *= al[j];
                }
#pragma unroll
                for (int mb = 0; mb < MB; ++mb) {
                    o[hb][mb][0] *= al[0];
                    o[hb][mb][1] *= al[1];
                    o[hb][mb][2] *= al[0];
                    o[hb][mb][3] *= al[1];
                }
            }
        }
#pragma unroll
        for (int hb = 0; hb < HB; ++hb) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                // a head with nothing visible yet keeps m = -inf and contributes 0
                const float ref = m[hb][j] == -INFINITY ? 0.f : m[hb][j];
                const float p0 = exp2f(sc[hb][j] - ref), p1 = exp2f(sc[hb][2 + j] - ref);
                l[hb][j] += p0 + p1;
                sc[hb][j] = p0;
                sc[hb][2 + j] = p1;
            }
            const float f = VS ? vscale : 1.f;
            uint32_t x0, x1;
            if constexpr (F16P) {
                x0 = pack_bf16_as_f16(sc[hb][0] * f, sc[hb][1] * f);
                x1 = pack_bf16_as_f16(sc[hb][2] * f, sc[hb][3] * f);
            } else {
                x0 = Mma<T>::pack(sc[hb][0] * f, sc[hb][1] * f);
                x1 = Mma<T>::pack(sc[hb][2] * f, sc[hb][3] * f);
            }
            pb[hb][0] = movm_trans(x0);  // P^T keys 2 tig, 2 tig + 1; head gid
            pb[hb][1] = movm_trans(x1);  // keys 2 tig + 8, 2 tig + 9
        }
    }

    // One tile: keys [lo, hi) of this warp's 16 rows are visible (the caller
    // guarantees that V rows at and past `hi` hold finite values); VS: P is
    // multiplied by vscale (a power of two) before it is packed.
    template <bool VS = false>
    __device__ __forceinline__ void tile(uint32_t kb, uint32_t vb, int warp, int lane, int lo,
                                         int hi, float scale_log2, float vscale = 1.f)
    {
        float sc[HB][4];
#pragma unroll
        for (int hb = 0; hb < HB; ++hb)
            sc[hb][0] = sc[hb][1] = sc[hb][2] = sc[hb][3] = 0.f;
        // ldmatrix x4 of an A fragment: matrix m = lane / 8 holds keys
        // 8 (m % 2) .. + 7 at columns 8 (m / 2) .. + 7 of the 16-column block
        const int mat = lane >> 3;
        const int krow = 16 * warp + ((mat & 1) << 3) + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < MB; kk += 2) {
            uint32_t qf[HB][4];
#pragma unroll
            for (int hb = 0; hb < HB; ++hb)
                q_frag2(hb, kk, qf[hb]);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int cidx = 2 * (kk + u) + (mat >> 1);
                uint32_t a[4];
                ldsm_x4(kb + (cidx >> 3) * 8192 + kvc::sw128(krow, cidx & 7), a[0], a[1], a[2],
                        a[3]);
#pragma unroll
                for (int hb = 0; hb < HB; ++hb)
                    Mma<T>::run(sc[hb], a, qf[hb][2 * u], qf[hb][2 * u + 1]);
            }
        }
        uint32_t pb[HB][2];
        softmax_step<VS>(sc, lane, lo, hi, scale_log2, vscale, pb);
        // A = V^T by transposing loads: matrix m holds keys 8 (m / 2) .. + 7
        // at columns 8 (m % 2) .. + 7 of the 16-column block
        const int vrow = 16 * warp + ((mat >> 1) << 3) + (lane & 7);
#pragma unroll
        for (int mb = 0; mb < MB; ++mb) {
            const int cidx = 2 * mb + (mat & 1);
            uint32_t a[4];
            ldsm_x4_t(vb + (cidx >> 3) * 8192 + kvc::sw128(vrow, cidx & 7), a[0], a[1], a[2],
                      a[3]);
#pragma unroll
            for (int hb = 0; hb < HB; ++hb)
                Mma<T>::run(o[hb][mb], a, pb[hb][0], pb[hb][1]);
        }
    }

    // One tile of an int8 page: kq / vq = shared-memory addresses of this
    // warp's 16-row group of the K and V payloads in fragment order
    // (kvc_quantize_pages): the lane's
    // D / 2 bytes of each are the exact A fragments of its MMAs, as 16-byte
    // pieces interleaved across the warp (piece i of lane l at i * 512 +
    // l * 16), piece i holding 16-column blocks 2 i and 2 i + 1.  They become
    // the integers u - zp in registers, as fp16 halves for f16 MMAs (a third
    // of the conversion work of the bf16 route).  The K codes meet the query
    // when F16S (koff2 = q8_offset<__half>(zp); for a bf16 cache the query's
    // fp16 copy, load_q16, holding the same values, so the products are the
    // same exact numbers as with bf16 operands), else they take T's route
    // (q8_offset<T>).  The V codes (voff2 = q8_offset<__half>(zp)) meet the
    // probabilities times vscale -- the page's V scale, for a bf16 cache
    // times the CTA's power of two -- rounded as T and, for a bf16 cache,
    // handed on as fp16 (pack_bf16_as_f16).  The page's K scale is folded
    // into scale_log2.  Every converted value is finite, and P is 0 past
    // `hi`, so the rows past the split end need no zeroing.
    template <bool F16S>
    __device__ __forceinline__ void tile_q8(uint32_t kq, uint32_t vq, int lane, int lo,
                                            int hi, float scale_log2, float vscale, uint64_t koff2,
                                            uint64_t voff2)
    {
        using KT = typename std::conditional<F16S, __half, T>::type;
        constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
        constexpr int NP = D / 32;  // 16-byte pieces of a lane's fragment bytes
        float sc[HB][4];
#pragma unroll
        for (int hb = 0; hb < HB; ++hb)
            sc[hb][0] = sc[hb][1] = sc[hb][2] = sc[hb][3] = 0.f;
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            // words: (block 2p, keys 0-7 | 8-15 at columns +0 / +8), (block 2p + 1, ...)
            const uint4 w = lds128(kq + p * 512 + lane * 16);
            uint32_t qf[HB][4];
#pragma unroll
            for (int hb = 0; hb < HB; ++hb) {
                if constexpr (F16S && kBf16)
                    q16_frag2(hb, 2 * p, qf[hb]);
                else
                    q_frag2(hb, 2 * p, qf[hb]);
            }
            uint32_t a[4];
            u8x4_to_pairs<KT>(w.x, koff2, a[0], a[1]);
            u8x4_to_pairs<KT>(w.y, koff2, a[2], a[3]);
#pragma unroll
            for (int hb = 0; hb < HB; ++hb)
                Mma<KT>::run(sc[hb], a, qf[hb][0], qf[hb][1]);
            u8x4_to_pairs<KT>(w.z, koff2, a[0], a[1]);
            u8x4_to_pairs<KT>(w.w, koff2, a[2], a[3]);
#pragma unroll
            for (int hb = 0; hb < HB; ++hb)
                Mma<KT>::run(sc[hb], a, qf[hb][2], qf[hb][3]);
        }
        uint32_t pb[HB][2];
        softmax_step<true, kBf16>(sc, lane, lo, hi, scale_log2, vscale, pb);
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            // words: (columns of block 2p, keys 0-7), (block 2p, keys 8-15), (block 2p + 1, ...)
            const uint4 w = lds128(vq + p * 512 + lane * 16);
            uint32_t a[4];
            u8x4_to_pairs<__half>(w.x, voff2, a[0], a[1]);
            u8x4_to_pairs<__half>(w.y, voff2, a[2], a[3]);
#pragma unroll
            for (int hb = 0; hb < HB; ++hb)
                Mma<__half>::run(o[hb][2 * p], a, pb[hb][0], pb[hb][1]);
            u8x4_to_pairs<__half>(w.z, voff2, a[0], a[1]);
            u8x4_to_pairs<__half>(w.w, voff2, a[2], a[3]);
#pragma unroll
            for (int hb = 0; hb < HB; ++hb)
                Mma<__half>::run(o[hb][2 * p + 1], a, pb[hb][0], pb[hb][1]);
        }
    }

    // finish l across the warp's keys and publish (m, l, o * oscale) of
    // heads < g for the 4-warp merge: cm/cl [4][16], co [4][rows][pitch]
    // (rows >= g; a pitch of D + 4 floats keeps the stores of the four head
    // pairs apart in the banks)
    __device__ __forceinline__ void publish(float *cm, float *cl, float *co, int warp, int lane,
                                            int g, int rows, int pitch, float oscale = 1.f)
    {
        const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int hb = 0; hb < HB; ++hb)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float s = l[hb][j];
                s += __shfl_xor_sync(0xffffffffu, s, 4);
                s += __shfl_xor_sync(0xffffffffu, s, 8);
                s += __shfl_xor_sync(0xffffffffu, s, 16);
                const int h = 8 * hb + 2 * tig + j;
                if (gid == 0) {
                    cm[warp * 16 + h] = m[hb][j];
                    cl[warp * 16 + h] = s;
                }
                if (h < g) {
                    float *dst = co + (warp * rows + h) * pitch + gid;
#pragma unroll
                    for (int mb = 0; mb < MB; ++mb) {
                        dst[16 * mb] = o[hb][mb][j] * oscale;
                        dst[16 * mb + 8] = o[hb][mb][2 + j] * oscale;
                    }
                }
            }
    }
};
// merged (unnormalised o, l, reference max) of head h, columns [d, d + 4)
// over the four warps' published partials (cm/cl [4][16], co
// [4][rows][pitch]; d a multiple of 4): one round of shared-memory loads,
// the partials of the four columns read as one float4 per warp
struct Merged4 {
    float mstar, lsum, o[4];
};
__device__ __forceinline__ Merged4 merge4(const float *cm, const float *cl, const float *co,
                                          int pitch, int rows, int h, int d)
{
    Merged4 r;
    float mw[kConsumers];
    r.mstar = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumers; ++w) {
        mw[w] = cm[w * 16 + h];
        r.mstar = fmaxf(r.mstar, mw[w]);
    }
    const float ref = r.mstar == -INFINITY ? 0.f : r.mstar;
    r.lsum = 0.f;
    r.o[0] = r.o[1] = r.o[2] = r.o[3] = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumers; ++w) {
        const float f = exp2f(mw[w] - ref);
        r.lsum += cl[w * 16 + h] * f;
        const float4 v = *reinterpret_cast<const float4 *>(co + (w * rows + h) * pitch + d);
        r.o[0] += v.x * f;
        r.o[1] += v.y * f;
        r.o[2] += v.z * f;
        r.o[3] += v.w * f;
    }
    return r;
}

// out[0, 4) = o[0, 4) / l, rounded to T, as one 8-byte store
template <typename T>
__device__ __forceinline__ void store_out4(T *out, const Merged4 &r)
{
    uint2 v;
    v.x = Mma<T>::pack(r.o[0] / r.lsum, r.o[1] / r.lsum);
    v.y = Mma<T>::pack(r.o[2] / r.lsum, r.o[3] / r.lsum);
    *reinterpret_cast<uint2 *>(out) = v;
}

struct DecodeArgs {
    void *out;
    const void *q;
    kvc_lengths len;
    int batch, q_heads, kv_heads, group;
    int64_t capacity;
    int ring;    // slots addressed as a ring of `capacity` (kvc_gqa_decode_ring)
    int window;
    float scale_log2;
    const float *cos_t, *sin_t;
    int64_t rope_max_pos;
    float *ws_o, *ws_m, *ws_l;
    int64_t split_rows;
    int max_splits;
    int32_t *status;
    // fused step only
    const int32_t *seqlens_k;
    const void *new_k, *new_v;
    void *k_cache, *v_cache;
    // paged cache only: logical row r of batch row b is slot r % page_size of
    // page block_table[b * max_pages + r / page_size] of the pool
    const int32_t *block_table;
    int max_pages, page_size;
    int64_t n_pool_pages;
    // int8 pages (kvc_gqa_decode_paged_q): a table entry with KVC_PAGE_QUANT
    // names page (entry & ~KVC_PAGE_QUANT) of these pools, read as
    // (stored - zp) * scale with qparams[page] = (k_scale, k_zp, v_scale, v_zp)
    const uint8_t *qk_pool, *qv_pool;
    const float *qparams;
    int64_t n_q_pages;
};

// what the split kernel reads: the lengths arrays over a cache or a ring
// (plain), seqlens_k with the append fused in (fused), or a paged cache
enum : int { kPlain = 0, kFused = 1, kPaged = 2, kPagedQ = 3 };

// First logical row a split count starts from: the window's first visible
// row, rounded down to a tile for a paged cache so that no tile straddles a
// page (the rows below the window are masked).
template <int MODE> __device__ __forceinline__ int split_origin(int vis0)
{
    return MODE >= kPaged ? vis0 & ~(kTile - 1) : vis0;
}

// (L, T) of batch row b: from the lengths arrays, or in the fused step from
// seqlens_k (kvc_seq_lengths for S = 1 on a contiguous cache or a ring).
// Returns the row's number of splits; 0 when it has nothing to attend
// (rejected row, lengths that do not fit this cache, RoPE out of range).
template <int MODE>
__device__ __forceinline__ int row_splits(const DecodeArgs &a, int b, int &L, int &tot)
{
    if constexpr (MODE == kFused) {
        const int64_t T64 = (int64_t)a.seqlens_k[b] + 1;
        if (T64 < 1 || T64 > (int64_t)INT32_MAX || (!a.ring && T64 > a.capacity))
            return 0;
        tot = (int)T64;
        L = (int)(a.ring && T64 > a.capacity ? a.capacity : T64);
    } else {
        L = a.len.cache_total[b];
        tot = a.len.total_abs[b];
        if (L <= 0 || (int64_t)L > a.capacity || (a.ring && tot < L))
            return 0;
    }
    if (a.cos_t && (int64_t)tot > a.rope_max_pos)
        return 0;
    const int vis0 = (a.window > 0 && L > a.window) ? L - a.window : 0;
    return (int)((L - split_origin<MODE>(vis0) + a.split_rows - 1) / a.split_rows);
}

// Errors of batch row b, raised once per row; the fused step also writes
// the row's lengths (as kvc_seq_lengths would).
template <int MODE>
__device__ __forceinline__ void row_check(const DecodeArgs &a, int b)
{
    if constexpr (MODE == kFused) {
        const int64_t T64 = (int64_t)a.seqlens_k[b] + 1;
        const bool write_len = a.len.cache_total != nullptr;
        uint32_t bad = 0;
        if (T64 < 1 || T64 > (int64_t)INT32_MAX)
            bad = KVC_DEV_SEQLEN_RANGE;
        else if (!a.ring && T64 > a.capacity)
            bad = KVC_DEV_CAPACITY;
        if (bad) {
            kvc::raise_status(a.status, bad);
            if (write_len)
                a.len.past_abs[b] = a.len.total_abs[b] = a.len.cache_past[b] =
                    a.len.cache_total[b] = a.len.evict[b] = -1;
            return;
        }
        int64_t Lp, E, L;
        kvc::cache_lengths(a.ring ? KVC_RING : KVC_CONTIGUOUS, T64, 1, a.capacity, 1, Lp, E, L);
        if (write_len) {
            a.len.past_abs[b] = (int32_t)(T64 - 1);
            a.len.total_abs[b] = (int32_t)T64;
            a.len.cache_past[b] = (int32_t)Lp;
            a.len.cache_total[b] = (int32_t)L;
            a.len.evict[b] = (int32_t)E;
        }
        if (a.cos_t && T64 > a.rope_max_pos)
            kvc::raise_status(a.status, KVC_DEV_ROPE_RANGE);
    } else {
        const int L = a.len.cache_total[b];
        const int tot = a.len.total_abs[b];
        if (L <= 0)
            return;  // rejected when the lengths were derived
        if ((int64_t)L > a.capacity || (a.ring && tot < L))
            kvc::raise_status(a.status, KVC_DEV_CAPACITY);  // lengths for another cache
        else if (a.cos_t && (int64_t)tot > a.rope_max_pos)
            kvc::raise_status(a.status, KVC_DEV_ROPE_RANGE);
    }
}

// does entry e of a kPagedQ table name a valid int8 page?
__device__ __forceinline__ bool int8_page(int e, const DecodeArgs &a)
{
    return e >= 0 && (e & KVC_PAGE_QUANT) && (int64_t)(e & ~KVC_PAGE_QUANT) < a.n_q_pages;
}

// Shared memory of the split kernel.  The tiles arrive in a ring: NS stages
// of one K and one V tile each (16-bit pages up to head_dim 128), or ring
// slots of one 64-row tile of K or of V each, a 16-bit tile taking two slots
// and an int8 tile (its K and V payloads, half the bytes) one.  Slots serve
// int8 pages, and head_dim 256, where a 64-row tile is 32 KB and three slots
// (96 KB) let two CTAs share an SM.
template <int D, int MODE> __host__ __device__ constexpr bool decode_uses_slots()
{
    return MODE == kPagedQ || D >= 256;
}
template <int D, int MODE> __host__ __device__ constexpr int decode_ring_slots()
{
    return D >= 256 ? 3 : MODE == kPagedQ ? (D == 128 ? 4 : 2 * decode_stages(D)) : decode_stages(D);
}
template <int D, int MODE> __host__ __device__ constexpr int decode_slot_bytes()
{
    return decode_uses_slots<D, MODE>() ? kTile * D * 2 : 2 * kTile * D * 2;
}
// At head_dim 256 the split kernel runs without a producer warp (four
// consumer warps, two CTAs an SM, up to 255 registers a thread: 64 of them
// the output accumulator of a head block, 128 of two), and the warp that
// releases a ring slot last issues that slot's next load -- measured faster
// than a fifth, producer warp, with or without spills.  (Over int8 pages,
// where the consumer warps' conversion work is the limit, the same scheme
// measured slower: the issuing lane stalls its warp.)
template <int D, int MODE> __host__ __device__ constexpr bool decode_no_producer()
{
    return D >= 256 && MODE != kPagedQ;
}
// the query's MMA fragments are held in registers, else read from shared
// memory at every tile: with two blocks of 8 heads at head_dim 256 (whose
// output accumulator alone takes 128 registers a thread) and over int8 pages
// (whose conversion work wants the registers for a third CTA an SM)
template <int D, int HB, int MODE = kPlain> __host__ __device__ constexpr bool decode_q_in_registers()
{
    return HB == 1 || (D <= 128 && MODE != kPagedQ);
}
template <int D, int MODE> __host__ __device__ constexpr int decode_threads()
{
    return decode_no_producer<D, MODE>() ? 128 : 160;
}
// bytes after the 1024-byte alignment pad: ring, staged query rows [16][D + 8],
// full/empty barriers, abort flag (+pad), the split's page ids [32], the
// fused step's new K and V row, and the slots' release counters
template <int D, int MODE> __host__ __device__ constexpr int decode_smem_bytes()
{
    return decode_ring_slots<D, MODE>() * decode_slot_bytes<D, MODE>() + 16 * (D + 8) * 2 +
           2 * decode_ring_slots<D, MODE>() * 8 + 16 + 32 * 4 + 2 * D * 2 +
           4 * decode_ring_slots<D, MODE>() + (MODE == kPagedQ ? 16 + 16 * (D + 8) * 2 : 0);
}

// One CTA per (split, kv head, batch row) for kvc_gqa_decode,
// kvc_gqa_decode_ring and the fused kvc_decode_step; the split partials go
// to decode_combine_kernel.  kFused: lengths from seqlens_k, and the CTA
// holding the newest position places the new K/V row in its tile on chip
// and stores it to the cache.  kPaged: tiles of 64 logical rows, each inside
// one page; the producer warp reads the split's page ids at once.  kPagedQ:
// the same over 16-bit and int8 pages (an int8 tile arrives by two 1-D bulk
// copies at half the bytes and is expanded on chip before its MMAs).
// (kPagedQ and head_dim 256: at most as many registers as the CTAs the
// shared memory lets share an SM can hold -- two at head_dim 256, three
// over int8 pages at head_dim 64 and 128)
template <typename T, int D, int MODE, int HB>
__global__ void __launch_bounds__(decode_threads<D, MODE>(),
                                  (MODE == kPagedQ || D >= 256) ? (D >= 256 ? 2 : 3) : 0)
decode_split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const DecodeArgs a)
{
    constexpr bool SLOTS = decode_uses_slots<D, MODE>();
    constexpr bool NOPROD = decode_no_producer<D, MODE>();
    constexpr int NBAR = decode_ring_slots<D, MODE>();
    constexpr int SLOT_BYTES = decode_slot_bytes<D, MODE>();
    constexpr int BOXES = D / 64;
    constexpr int KT_BYTES = kTile * D * 2;  // one K (or V) tile
    constexpr int QS = D + 8;                // padded Q row (elements)

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *stages = smem;
    T *qs = reinterpret_cast<T *>(smem + NBAR * SLOT_BYTES);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + NBAR * SLOT_BYTES + 16 * QS * 2);
    uint64_t *empty = full + NBAR;
    int *abort_flag = reinterpret_cast<int *>(empty + NBAR);
    int *page_ids = abort_flag + 4;  // [32] paged: the split's pages
    // kFused: the new row, K rotated at its position then V ([2][D])
    T *newrow = reinterpret_cast<T *>(page_ids + 32);
    // NOPROD: how many warps have released each slot in its current round
    int *released = reinterpret_cast<int *>(newrow + 2 * D);
    // kPagedQ: the query rows as fp16 [16][QS] for the int8 tiles' scores
    __half *qs16 = reinterpret_cast<__half *>(
        (reinterpret_cast<uintptr_t>(released + NBAR) + 15) & ~uintptr_t(15));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    if (threadIdx.x == 0 && split == 0 && kvh == 0)
        row_check<MODE>(a, b);
    int L, tot;
    const int nsplit = row_splits<MODE>(a, b, L, tot);
    if (split >= nsplit)
        return;
    const int vis0 = (a.window > 0 && L > a.window) ? L - a.window : 0;
    const int origin = split_origin<MODE>(vis0);
    const int vis = L - origin;
    // this split's rows [j0, j0 + cnt) from the origin, in position order, as
    // two runs of slots: [q0, q0 + cnt_a) and [0, cnt - cnt_a)
    const int C = (int)a.capacity;
    const int j0 = (int)(split * a.split_rows);
    const int cnt = (int)min((int64_t)vis - j0, a.split_rows);
    const int first = a.ring ? (int)(((int64_t)tot - vis) % C) : origin;
    int q0 = first + j0;
    if (q0 >= C)
        q0 -= C;
    const int cnt_a = min(cnt, C - q0);
    // rows of tile t below the window (a paged cache's first tile only)
    auto tile_lo = [&](int t) { return MODE >= kPaged ? max(0, vis0 - (q0 + t * kTile)) : 0; };
    const int nt_a = (cnt_a + kTile - 1) / kTile;
    const int ntiles = nt_a + (cnt - cnt_a + kTile - 1) / kTile;
    // first slot and number of valid rows of tile t
    auto tile_start = [&](int t) { return t < nt_a ? q0 + t * kTile : (t - nt_a) * kTile; };
    auto tile_rows = [&](int t) {
        return t < nt_a ? min(kTile, cnt_a - t * kTile)
                        : min(kTile, cnt - cnt_a - (t - nt_a) * kTile);
    };
    const int64_t row_base = ((int64_t)b * a.kv_heads + kvh) * a.capacity;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NBAR; ++s) {
            kvc::mbar_init(&full[s], 1);
            kvc::mbar_init(&empty[s], kConsumers);
            released[s] = 0;
        }
        *abort_flag = 0;
        kvc::fence_mbar_init();
    }
    if constexpr (MODE >= kPaged && NOPROD) {
        // the pages this split touches, one lane of the first warp each
        if (warp == 0) {
            const int page0 = q0 / a.page_size;
            const int npages = (q0 + cnt - 1) / a.page_size - page0 + 1;
            if (lane < npages) {
                int id = a.block_table[(int64_t)b * a.max_pages + page0 + lane];
                if (id < 0 || (int64_t)id >= a.n_pool_pages) {
                    kvc::raise_status(a.status, KVC_DEV_INDEX_OOB);
                    id = 0;  // read a page that exists; the row's result is void
                }
                page_ids[lane] = id;
            }
        }
    }
    __syncthreads();

    // NOPROD: load j of the split fills slot j % NBAR: K (j even) or V (j odd)
    // of tile j / 2; the first NBAR are issued here, each later one by the
    // warp that releases its slot last
    const int n_loads = 2 * ntiles;
    auto issue_load = [&](int j) {
        const int t = j >> 1;
        int32_t y;
        if constexpr (MODE >= kPaged) {
            const int r = q0 + t * kTile;  // logical row, a multiple of 64
            const int id = page_ids[r / a.page_size - q0 / a.page_size];
            y = (int32_t)(((int64_t)id * a.kv_heads + kvh) * a.page_size + r % a.page_size);
        } else {
            y = (int32_t)(row_base + tile_start(t));
        }
        const int sl = j % NBAR;
        uint8_t *dst = stages + sl * SLOT_BYTES;
        const CUtensorMap *map = (j & 1) ? &tmap_v : &tmap_k;
        kvc::mbar_arrive_expect_tx(&full[sl], KT_BYTES);
#pragma unroll
        for (int bx = 0; bx < BOXES; ++bx)
            kvc::tma_load_2d(dst + bx * 8192, map, bx * 64, y, &full[sl]);
    };
    if constexpr (NOPROD) {
        if (threadIdx.x == 0) {
            kvc::tma_prefetch_desc(&tmap_k);
            kvc::tma_prefetch_desc(&tmap_v);
            for (int j = 0; j < NBAR && j < n_loads; ++j)
                issue_load(j);
        }
    }
    // NOPROD: this warp is done with load j's slot; the last of the four to
    // say so issues load j + NBAR into it (the fences order every warp's use
    // of the slot, and any bytes it wrote there, before the copy overwrites it)
    auto release_slot = [&](int j) {
        if (lane == 0) {
            const int sl = j % NBAR;
            __threadfence_block();
            if (atomicAdd(&released[sl], 1) == kConsumers - 1) {
                released[sl] = 0;
                __threadfence_block();
                kvc::fence_proxy_async_smem();
                if (j + NBAR < n_loads && !*reinterpret_cast<volatile int *>(abort_flag))
                    issue_load(j + NBAR);
            }
        }
    };

    if (!NOPROD && warp == kConsumers) {
        // ---------------- producer ----------------
        int page0 = 0;
        if constexpr (MODE >= kPaged) {
            // the pages this split touches, one lane each (at most 32)
            page0 = q0 / a.page_size;
            const int npages = (q0 + cnt - 1) / a.page_size - page0 + 1;
            if (lane < npages) {
                int id = a.block_table[(int64_t)b * a.max_pages + page0 + lane];
                const bool q8 = MODE == kPagedQ && int8_page(id, a);
                if (!q8 && (id < 0 || (int64_t)id >= a.n_pool_pages)) {
                    kvc::raise_status(a.status, KVC_DEV_INDEX_OOB);
                    id = 0;  // read a page that exists; the row's result is void
                }
                page_ids[lane] = id;
            }
            __syncwarp();
        }
        if (lane == 0) {
            kvc::tma_prefetch_desc(&tmap_k);
            kvc::tma_prefetch_desc(&tmap_v);
            int pos = 0;  // slots: ring position of the next tile's first slot
            // paged: the tile's page among the split's and its first row in
            // that page, stepped per tile (q0 and the page size are
            // multiples of the tile)
            int ppi = 0, prow = MODE >= kPaged ? q0 % a.page_size : 0;
            for (int t = 0; t < ntiles; ++t) {
                // the tile's first row in the tensor maps, and whether it is int8
                int32_t y = 0;
                bool q8 = false;
                int64_t q8off = 0;
                if constexpr (MODE >= kPaged) {
                    const int id = page_ids[ppi];
                    if constexpr (MODE == kPagedQ)
                        q8 = int8_page(id, a);
                    if (q8)
                        q8off = (((int64_t)(id & ~KVC_PAGE_QUANT) * a.kv_heads + kvh) *
                                     a.page_size + prow) * D;
                    else
                        y = (int32_t)(((int64_t)id * a.kv_heads + kvh) * a.page_size + prow);
                    prow += kTile;
                    if (prow == a.page_size) {
                        prow = 0;
                        ++ppi;
                    }
                } else {
                    y = (int32_t)(row_base + tile_start(t));
                }
                if constexpr (SLOTS) {
                    const int need = q8 ? 1 : 2;
                    bool stop = false;
                    for (int u = 0; u < need && !stop; ++u) {
                        const int p = pos + u;
                        if (p >= NBAR &&
                            !kvc::mbar_wait(&empty[p % NBAR], ((p / NBAR) - 1) & 1)) {
                            kvc::raise_status(a.status, KVC_DEV_TIMEOUT);
                            stop = true;
                        }
                    }
                    if (stop || *reinterpret_cast<volatile int *>(abort_flag))
                        break;
                    const int s0 = pos % NBAR, s1 = (pos + 1) % NBAR;
                    uint8_t *b0 = stages + s0 * SLOT_BYTES;
                    if (q8) {
                        // the tile's 64 rows of K and of V payload, contiguous in the page
                        kvc::mbar_arrive_expect_tx(&full[s0], 2 * kTile * D);
                        kvc::bulk_load(b0, a.qk_pool + q8off, kTile * D, &full[s0]);
                        kvc::bulk_load(b0 + kTile * D, a.qv_pool + q8off, kTile * D, &full[s0]);
                    } else {
                        uint8_t *b1 = stages + s1 * SLOT_BYTES;
                        kvc::mbar_arrive_expect_tx(&full[s0], KT_BYTES);
#pragma unroll
                        for (int bx = 0; bx < BOXES; ++bx)
                            kvc::tma_load_2d(b0 + bx * 8192, &tmap_k, bx * 64, y, &full[s0]);
                        kvc::mbar_arrive_expect_tx(&full[s1], KT_BYTES);
#pragma unroll
                        for (int bx = 0; bx < BOXES; ++bx)
                            kvc::tma_load_2d(b1 + bx * 8192, &tmap_v, bx * 64, y, &full[s1]);
                    }
                    pos += need;
                } else {
                    const int s = t % NBAR, k = t / NBAR;
                    if (t >= NBAR && !kvc::mbar_wait(&empty[s], (k - 1) & 1)) {
                        kvc::raise_status(a.status, KVC_DEV_TIMEOUT);
                        break;
                    }
                    if (*reinterpret_cast<volatile int *>(abort_flag))
                        break;
                    uint8_t *kb = stages + s * SLOT_BYTES;
                    uint8_t *vb = kb + KT_BYTES;
                    kvc::mbar_arrive_expect_tx(&full[s], SLOT_BYTES);
#pragma unroll
                    for (int bx = 0; bx < BOXES; ++bx) {
                        kvc::tma_load_2d(kb + bx * 8192, &tmap_k, bx * 64, y, &full[s]);
                        kvc::tma_load_2d(vb + bx * 8192, &tmap_v, bx * 64, y, &full[s]);
                    }
                }
            }
        }
        return;
    }

    // ---------------- consumers ----------------
    const int g = a.group;
    bool q16_exact = true;  // kPagedQ: every query element is exact in fp16
    {
        // rotated query rows of the group (rows >= g stay zero)
        const T *qg = static_cast<const T *>(a.q) + ((int64_t)b * a.q_heads + kvh * g) * D;
        const float *cs = a.cos_t ? a.cos_t + (int64_t)(tot - 1) * (D / 2) : nullptr;
        const float *sn = a.cos_t ? a.sin_t + (int64_t)(tot - 1) * (D / 2) : nullptr;
        for (int idx = threadIdx.x; idx < 16 * (D / 2); idx += 128) {
            const int h = idx / (D / 2), i = idx % (D / 2);
            float lo = 0.f, hi = 0.f;
            if (h < g) {
                lo = kvc::Elem<T>::to_f32(qg[h * D + i]);
                hi = kvc::Elem<T>::to_f32(qg[h * D + i + D / 2]);
                if (cs)
                    kvc::rope_pair(lo, hi, cs[i], sn[i]);
            }
            const T tlo = kvc::Elem<T>::from_f32(lo), thi = kvc::Elem<T>::from_f32(hi);
            qs[h * QS + i] = tlo;
            qs[h * QS + i + D / 2] = thi;
            if constexpr (MODE == kPagedQ) {
                // the same (T-rounded) values in fp16: exact for 0 and for
                // magnitudes in [2^-17, 65504] (8 significant bits of a bf16
                // value fit an fp16 normal or subnormal there)
                const float flo = kvc::Elem<T>::to_f32(tlo), fhi = kvc::Elem<T>::to_f32(thi);
                qs16[h * QS + i] = __float2half_rn(flo);
                qs16[h * QS + i + D / 2] = __float2half_rn(fhi);
                q16_exact &= (flo == 0.f || (fabsf(flo) >= 0x1p-17f && fabsf(flo) <= 65504.f)) &&
                             (fhi == 0.f || (fabsf(fhi) >= 0x1p-17f && fabsf(fhi) <= 65504.f));
            }
        }
        if constexpr (MODE == kFused) {
            // the CTA whose split ends at the newest position (tot - 1) appends
            // it: while the first tiles are in flight, the new K row is rotated
            // there and both rows are stored to the cache and kept here for the
            // last tile, whose TMA copy of that row predates them
            if (split == nsplit - 1 && threadIdx.x < D / 2) {
                const int i = threadIdx.x;
                const int64_t slice = (int64_t)b * a.kv_heads + kvh;
                const int64_t dst_row = a.ring ? (int64_t)(tot - 1) % a.capacity : (int64_t)tot - 1;
                const T *nk = static_cast<const T *>(a.new_k) + slice * D;
                const T *nv = static_cast<const T *>(a.new_v) + slice * D;
                T *kc = static_cast<T *>(a.k_cache) + (slice * a.capacity + dst_row) * D;
                T *vc = static_cast<T *>(a.v_cache) + (slice * a.capacity + dst_row) * D;
                float lo = kvc::Elem<T>::to_f32(nk[i]), hi = kvc::Elem<T>::to_f32(nk[i + D / 2]);
                if (a.cos_t)
                    kvc::rope_pair(lo, hi, a.cos_t[(int64_t)(tot - 1) * (D / 2) + i],
                                   a.sin_t[(int64_t)(tot - 1) * (D / 2) + i]);
                const T klo = kvc::Elem<T>::from_f32(lo), khi = kvc::Elem<T>::from_f32(hi);
                const T vlo = nv[i], vhi = nv[i + D / 2];
                kc[i] = klo;
                kc[i + D / 2] = khi;
                vc[i] = vlo;
                vc[i + D / 2] = vhi;
                newrow[i] = klo;
                newrow[i + D / 2] = khi;
                newrow[D + i] = vlo;
                newrow[D + i + D / 2] = vhi;
            }
        }
    }
    // kPagedQ: the int8 tiles take fp16 scores when the whole query of the
    // group is exact in fp16 (always for an fp16 cache)
    const bool f16s = consumer_all(q16_exact);
    GroupAttn<T, D, HB, decode_q_in_registers<D, HB, MODE>(), true> ga;
    ga.init();
    ga.load_q(qs, QS, lane);
    if constexpr (MODE == kPagedQ)
        ga.load_q16(qs16, lane);
    bool timed_out = false;
    // kPagedQ: lane l holds the split's l-th table entry and, for an int8
    // page, its (k_scale, k_zp, v_scale, v_zp); a tile takes them by shuffle
    int my_e = 0;
    float my_p[4] = {1.f, 0.f, 1.f, 0.f};
    if constexpr (MODE == kPagedQ) {
        const int pg0 = q0 / a.page_size;
        if (lane < (q0 + cnt - 1) / a.page_size - pg0 + 1) {
            my_e = a.block_table[(int64_t)b * a.max_pages + pg0 + lane];
            if (int8_page(my_e, a)) {
                const float4 pr = *reinterpret_cast<const float4 *>(
                    a.qparams + 4 * (int64_t)(my_e & ~KVC_PAGE_QUANT));
                my_p[0] = pr.x;
                my_p[1] = pr.y;
                my_p[2] = pr.z;
                my_p[3] = pr.w;
            } else {
                my_e = 0;
            }
        }
    }
    // kPagedQ over a bf16 cache: the probabilities reach the int8 tiles' V
    // MMAs as fp16, multiplied by pscale = 2^k, which takes the largest V
    // scale of the split's int8 pages into [2^6, 2^7), so that P * scale *
    // 2^k stays at or below 2^15 (P <= 2^8) and small probabilities keep
    // their bits; the 16-bit tiles' P takes the same factor and o is scaled
    // back by 2^-k when it is published (both exact)
    float pscale = 1.f, oscale = 1.f;
    if constexpr (MODE == kPagedQ && std::is_same<T, __nv_bfloat16>::value) {
        float vmax = my_e != 0 ? my_p[2] : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
        if (vmax > 0.f && vmax <= FLT_MAX) {
            const int e = (int)((__float_as_uint(vmax) >> 23) & 0xffu) - 127;
            const int k = max(-64, min(64, 6 - e));
            pscale = __uint_as_float((uint32_t)(127 + k) << 23);
            oscale = __uint_as_float((uint32_t)(127 - k) << 23);
        }
    }

    int pos = 0;  // slots: ring position of the tile's first slot
    // kPagedQ: the tile's page among the split's (pi) and its place in that
    // page (tin, in 64-row tiles), stepped per tile without a division (q0
    // and the page size are multiples of the tile)
    const int tpp = MODE == kPagedQ ? a.page_size / kTile : 1;
    int pi = 0, tin = MODE == kPagedQ ? (q0 / kTile) % tpp : 0;
    for (int t = 0; t < ntiles; ++t) {
        bool q8 = false;
        if constexpr (MODE == kPagedQ)
            q8 = (__shfl_sync(0xffffffffu, my_e, pi) & KVC_PAGE_QUANT) != 0;
        // the tile's K and V (16-bit), or its int8 K and V payloads (kgen)
        uint8_t *kgen, *vgen;
        int s0, s1;
        if constexpr (SLOTS) {
            s0 = pos % NBAR;
            s1 = (pos + 1) % NBAR;
            kgen = stages + s0 * SLOT_BYTES;
            vgen = stages + s1 * SLOT_BYTES;
            if (!kvc::mbar_wait(&full[s0], (uint32_t)(pos / NBAR) & 1u) ||
                (!q8 && !kvc::mbar_wait(&full[s1], (uint32_t)((pos + 1) / NBAR) & 1u))) {
                timed_out = true;
                break;
            }
        } else {
            s0 = s1 = t % NBAR;
            kgen = stages + s0 * SLOT_BYTES;
            vgen = kgen + KT_BYTES;
            if (!kvc::mbar_wait(&full[s0], (uint32_t)(t / NBAR) & 1u)) {
                timed_out = true;
                break;
            }
        }
        const int rows_t = tile_rows(t);
        const int my_valid = min(16, max(0, rows_t - 16 * warp));
        const int my_lo = min(16, max(0, tile_lo(t) - 16 * warp));
        bool wrote = false;
        if (MODE == kFused && split == nsplit - 1 && t == ntiles - 1 && my_valid > 0 &&
            16 * warp + my_valid == rows_t) {
            // this warp owns the newest row (position tot - 1): place the new
            // K (rotated there) and V row, appended at the start, in the tile
            const int rr = rows_t - 1;
            for (int i = lane; i < D / 2; i += 32) {
                const T klo = newrow[i], khi = newrow[i + D / 2];
                const T vlo = newrow[D + i], vhi = newrow[D + i + D / 2];
                const int c0 = i, c1 = i + D / 2;
                const int o0 = (c0 >> 6) * 8192 + kvc::sw128(rr, (c0 & 63) >> 3) + (c0 & 7) * 2;
                const int o1 = (c1 >> 6) * 8192 + kvc::sw128(rr, (c1 & 63) >> 3) + (c1 & 7) * 2;
                *reinterpret_cast<T *>(kgen + o0) = klo;
                *reinterpret_cast<T *>(kgen + o1) = khi;
                *reinterpret_cast<T *>(vgen + o0) = vlo;
                *reinterpret_cast<T *>(vgen + o1) = vhi;
            }
            wrote = true;
            __syncwarp();
        }
        if (q8) {
            const float ks = __shfl_sync(0xffffffffu, my_p[0], pi);
            const float kz = __shfl_sync(0xffffffffu, my_p[1], pi);
            const float vs = __shfl_sync(0xffffffffu, my_p[2], pi);
            const float vz = __shfl_sync(0xffffffffu, my_p[3], pi);
            if (my_lo < my_valid) {
                const uint32_t kq = kvc::smem_u32(kgen) + warp * 16 * D;
                if (f16s)
                    ga.template tile_q8<true>(kq, kq + kTile * D, lane, my_lo, my_valid,
                                              a.scale_log2 * ks, vs * pscale,
                                              q8_offset<__half>(kz), q8_offset<__half>(vz));
                else
                    ga.template tile_q8<false>(kq, kq + kTile * D, lane, my_lo, my_valid,
                                               a.scale_log2 * ks, vs * pscale, q8_offset<T>(kz),
                                               q8_offset<__half>(vz));
            }
        } else if (my_valid > 0) {
            if (my_valid < 16) {
                // rows past the split end: zero V so that 0 * garbage stays 0
                for (int idx = lane; idx < (16 - my_valid) * BOXES * 8; idx += 32) {
                    const int rr = 16 * warp + my_valid + idx / (BOXES * 8);
                    const int bx = (idx / 8) % BOXES, c = idx % 8;
                    *reinterpret_cast<uint4 *>(vgen + bx * 8192 + rr * 128 + c * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
                wrote = true;
            }
            if (my_lo < my_valid) {
                if constexpr (MODE == kPagedQ && std::is_same<T, __nv_bfloat16>::value)
                    ga.template tile<true>(kvc::smem_u32(kgen), kvc::smem_u32(vgen), warp, lane,
                                           my_lo, my_valid, a.scale_log2, pscale);
                else
                    ga.tile(kvc::smem_u32(kgen), kvc::smem_u32(vgen), warp, lane, my_lo,
                            my_valid, a.scale_log2);
            }
        }
        if (wrote)
            kvc::fence_proxy_async_smem();
        __syncwarp();
        if constexpr (NOPROD) {
            release_slot(pos);
            release_slot(pos + 1);
        } else if (lane == 0) {
            kvc::mbar_arrive(&empty[s0]);
            if (SLOTS && !q8)
                kvc::mbar_arrive(&empty[s1]);
        }
        pos += q8 ? 1 : 2;
        if (MODE == kPagedQ && ++tin == tpp) {
            tin = 0;
            ++pi;
        }
    }
    if (timed_out) {
        if (lane == 0) {
            kvc::raise_status(a.status, KVC_DEV_TIMEOUT);
            atomicExch(abort_flag, 1);
        }
    }
    // ---- merge the four warps' (m, l, o) through shared memory ----
    consumer_sync();  // every warp is done with the stage buffers
    float *cm = reinterpret_cast<float *>(stages);        // [4][16]
    float *cl = cm + kConsumers * 16;                      // [4][16]
    float *co = cl + kConsumers * 16;                      // [4][16][D]
    ga.publish(cm, cl, co, warp, lane, g, 16, D + 4, oscale);
    consumer_sync();
    const int hq0 = kvh * g;
    for (int idx = threadIdx.x; idx < g * (D / 4); idx += 128) {
        const int h = idx / (D / 4), d = (idx % (D / 4)) * 4;
        const Merged4 r = merge4(cm, cl, co, D + 4, 16, h, d);
        const int64_t qrow = (int64_t)b * a.q_heads + hq0 + h;
        if (nsplit == 1) {
            store_out4(static_cast<T *>(a.out) + qrow * D + d, r);
        } else {
            const int64_t pr = qrow * a.max_splits + split;
            *reinterpret_cast<float4 *>(a.ws_o + pr * D + d) =
                make_float4(r.o[0], r.o[1], r.o[2], r.o[3]);
            if (d == 0) {
                a.ws_m[pr] = r.mstar;
                a.ws_l[pr] = r.lsum;
            }
        }
    }
}

// The same merge when a row has at most kFastSplits partials (capacity up
// to 8192 rows): the partials sit in L2 right after the split kernel, so the
// merge is a chain of round trips, not bytes.  Every thread loads all
// max_splits (m, l) pairs and its columns' partials at once, before the
// row's split count (which needs the lengths) is known; partials past that
// count are stale workspace and are dropped by selection, never multiplied
// in, so whatever they hold cannot reach the output.  D <= 128 * kFastCols.
constexpr int kFastSplits = 16, kFastCols = 2;
template <typename T, int MODE>
__global__ void __launch_bounds__(128)
decode_combine_fast_kernel(const DecodeArgs a, int D)
{
    const int h = blockIdx.x, b = blockIdx.y;
    const int MS = a.max_splits;
    const int64_t qrow = (int64_t)b * a.q_heads + h;
    const int64_t p0 = qrow * MS;
    float m[kFastSplits], l[kFastSplits], o[kFastSplits][kFastCols];
#pragma unroll
    for (int j = 0; j < kFastSplits; ++j) {
        m[j] = -INFINITY;
        l[j] = 0.f;
        if (j < MS) {
            m[j] = a.ws_m[p0 + j];
            l[j] = a.ws_l[p0 + j];
        }
#pragma unroll
        for (int c = 0; c < kFastCols; ++c) {
            const int d = threadIdx.x + 128 * c;
            o[j][c] = (j < MS && d < D) ? a.ws_o[(p0 + j) * D + d] : 0.f;
        }
    }
    int L, tot;
    const int nsplit = row_splits<MODE>(a, b, L, tot);
    if (nsplit <= 1)
        return;
    float mstar = -INFINITY;
#pragma unroll
    for (int j = 0; j < kFastSplits; ++j)
        mstar = j < nsplit ? fmaxf(mstar, m[j]) : mstar;
    float lsum = 0.f, acc[kFastCols];
#pragma unroll
    for (int c = 0; c < kFastCols; ++c)
        acc[c] = 0.f;
#pragma unroll
    for (int j = 0; j < kFastSplits; ++j) {
        if (j < nsplit) {
            const float w = exp2f(m[j] - mstar);
            lsum += l[j] * w;
#pragma unroll
            for (int c = 0; c < kFastCols; ++c)
                acc[c] += o[j][c] * w;
        }
    }
    const float inv_l = 1.f / lsum;
#pragma unroll
    for (int c = 0; c < kFastCols; ++c) {
        const int d = threadIdx.x + 128 * c;
        if (d < D)
            static_cast<T *>(a.out)[qrow * D + d] = kvc::Elem<T>::from_f32(acc[c] * inv_l);
    }
}

// merges the per-split partials of rows that used more than one split: the
// splits' m and l are read in parallel into shared memory, the weights
// 2^(m_j - max m) computed once, and each output column sums its partials
// with four loads in flight
template <typename T, int MODE>
__global__ void __launch_bounds__(128)
decode_combine_kernel(const DecodeArgs a, int D)
{
    extern __shared__ float wsh[];  // m [max_splits], then l * w [max_splits], w [max_splits]
    const int h = blockIdx.x, b = blockIdx.y;
    int L, tot;
    const int nsplit = row_splits<MODE>(a, b, L, tot);
    if (nsplit <= 1)
        return;
    const int MS = a.max_splits;
    float *sm = wsh, *slw = wsh + MS, *sw = wsh + 2 * MS;
    const int64_t qrow = (int64_t)b * a.q_heads + h;
    const int64_t p0 = qrow * MS;
    for (int j = threadIdx.x; j < nsplit; j += blockDim.x)
        sm[j] = a.ws_m[p0 + j];
    __syncthreads();
    float mstar = -INFINITY;
    for (int j = 0; j < nsplit; ++j)
        mstar = fmaxf(mstar, sm[j]);
    for (int j = threadIdx.x; j < nsplit; j += blockDim.x) {
        const float w = exp2f(sm[j] - mstar);
        sw[j] = w;
        slw[j] = a.ws_l[p0 + j] * w;
    }
    __syncthreads();
    float lsum = 0.f;
    for (int j = 0; j < nsplit; ++j)
        lsum += slw[j];
    const float inv_l = 1.f / lsum;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        const float *src = a.ws_o + p0 * D + d;
        float acc = 0.f;
        int j = 0;
        for (; j + 4 <= nsplit; j += 4) {
            const float v0 = src[(int64_t)j * D], v1 = src[(int64_t)(j + 1) * D];
            const float v2 = src[(int64_t)(j + 2) * D], v3 = src[(int64_t)(j + 3) * D];
            acc += v0 * sw[j] + v1 * sw[j + 1] + v2 * sw[j + 2] + v3 * sw[j + 3];
        }
        for (; j < nsplit; ++j)
            acc += src[(int64_t)j * D] * sw[j];
        static_cast<T *>(a.out)[qrow * D + d] = kvc::Elem<T>::from_f32(acc * inv_l);
    }
}


// --------------------------------------------------------------------------
// Fused one-token step on a windowed cache: lengths, compaction, RoPE append
// and GQA attention in one launch ("GQA support sliding_window_cache",
// "Design": rows [E, Lp) move to [0, Lp - E) and the new row goes to Lp - E;
// Lp, E, L from the windowed formula or from the drifting layout of the PR's
// CPU commit).  One CTA owns one (batch row, kv head) slice and keeps the new
// window in shared memory.  The step is bound by latency, not bandwidth, so
// the slice's rows are asked of L2 at entry, before seqlens_k has arrived;
// once it has, one thread brings the old rows in with 64-row TMA boxes
// (window row r from cache row r + E), one mbarrier per tile, while the
// others rotate the query and the new row.  The tiles are then taken in
// order as they land: the new row and the zeroed rows are placed in theirs,
// a tile goes back E rows lower by TMA store as soon as it is final (the
// stores of tile t only overwrite cache rows that tiles <= t were loaded
// from), and the warps run its attention.  A last partial tile goes back by
// thread stores; without an eviction only the visible rows are loaded (from
// the first visible row on, so a drifting cache with C > W reads W rows, not
// its whole resident length) and only the new row is stored.  A ring of
// C slots ("Stateful decode & KV cache", "Sliding-window ring buffer") never
// moves: its slots are loaded in slot order, the new row replaces slot
// (T - 1) mod C, and the attention masks the slots by position (the visible
// ones are at most two runs of slots).
// --------------------------------------------------------------------------
struct WindowStepArgs {
    void *out;
    const void *q;
    void *k_cache, *v_cache;
    const void *new_k, *new_v;
    const int32_t *seqlens_k;
    kvc_lengths len;  // all NULL: not written
    int q_heads, kv_heads, group;
    int64_t capacity;
    int policy;  // KVC_WINDOWED, KVC_DRIFTING or KVC_RING
    int window;
    float scale_log2;
    const float *cos_t, *sin_t;
    int64_t rope_max_pos;
    int32_t *status;
};

// largest capacity whose whole window (K and V) the fused step keeps in
// shared memory: capacity * head_dim at most kWindowStepMaxElems
constexpr int64_t kWindowStepMaxElems = 32768;
__host__ __device__ constexpr int64_t window_step_max_capacity(int D)
{
    return kWindowStepMaxElems / D;
}

template <typename T, int D, int HB>
__global__ void __launch_bounds__(128, D >= 256 ? 2 : 4)
window_step_kernel(const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const WindowStepArgs a)
{
    constexpr int BOXES = D / 64;
    constexpr int KT_BYTES = kTile * D * 2;  // one 64-row K (or V) tile
    constexpr int QS = D + 8;
    constexpr int CPR = D / 8;               // 16-byte chunks per row

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int64_t C = a.capacity;
    const int ntile_max = (int)((C + kTile - 1) / kTile);
    uint8_t *tiles = smem;  // tile t: K at t * 2 * KT_BYTES, V after it
    T *qs = reinterpret_cast<T *>(smem + (size_t)ntile_max * 2 * KT_BYTES);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + (size_t)ntile_max * 2 * KT_BYTES +
                                                 16 * QS * 2);  // [ntile_max]
    // byte offset of row r, 16-byte chunk c of the K (is_v = 0) or V tile
    auto at = [&](bool is_v, int r, int c) {
        return tiles + (size_t)(r / kTile) * 2 * KT_BYTES + (is_v ? KT_BYTES : 0) +
               (c >> 3) * 8192 + kvc::sw128(r % kTile, c & 7);
    };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x / a.kv_heads, kvh = blockIdx.x % a.kv_heads;
    const int g = a.group;
    const int64_t slice = (int64_t)b * a.kv_heads + kvh;

    // the whole slice is asked of L2 at once when every step reads nearly
    // all of it (C - W < 64: at most C - W of its rows go unread)
    if (threadIdx.x == 0) {
        if (C - a.window < kTile) {
            const uint32_t sb = (uint32_t)(C * D * sizeof(T));
            kvc::prefetch_l2(static_cast<const T *>(a.k_cache) + slice * C * D, sb);
            kvc::prefetch_l2(static_cast<const T *>(a.v_cache) + slice * C * D, sb);
        }
        for (int t = 0; t < ntile_max; ++t)
            kvc::mbar_init(&bar[t], 1);
        kvc::fence_mbar_init();
        kvc::tma_prefetch_desc(&tmap_k);
        kvc::tma_prefetch_desc(&tmap_v);
    }
    // the L2 requests above are hints and read nothing into the CTA; all
    // else waits for the kernels before this one (launched with
    // programmatic serialisation, the next step's kernel can meanwhile be
    // scheduled and ask L2 for its own rows)
    kvc::grid_dep_launch();
    kvc::grid_dep_wait();

    // 0. what does not depend on the lengths is loaded at once, beside
    //    seqlens_k: the group's query pairs (i, i + D/2) and the new row
    //    (thread i < D/2 holds a K pair, D/2 <= i < D a V pair)
    constexpr int QPT = 16 * (D / 2) / 128;  // query pairs per thread
    T q_lo[QPT], q_hi[QPT];
    {
        const T *qg = static_cast<const T *>(a.q) + ((int64_t)b * a.q_heads + kvh * g) * D;
#pragma unroll
        for (int j = 0; j < QPT; ++j) {
            const int idx = threadIdx.x + 128 * j;
            const int h = idx / (D / 2), i = idx % (D / 2);
            q_lo[j] = h < g ? qg[h * D + i] : T{};
            q_hi[j] = h < g ? qg[h * D + i + D / 2] : T{};
        }
    }
    // the new row's pairs: item x < D / 2 is K pair x, item D / 2 + i is V
    // pair i; thread t holds items t and t + 128 (the second only at D = 256)
    constexpr int RPT = D > 128 ? 2 : 1;
    bool row_thread[RPT], row_is_v[RPT];
    int row_i[RPT];
    T new_lo[RPT], new_hi[RPT];
#pragma unroll
    for (int u = 0; u < RPT; ++u) {
        const int x = threadIdx.x + 128 * u;
        row_thread[u] = x < D;
        row_is_v[u] = x >= D / 2;
        row_i[u] = row_is_v[u] ? x - D / 2 : x;
        new_lo[u] = new_hi[u] = T{};
        if (row_thread[u]) {
            const T *src = (row_is_v[u] ? static_cast<const T *>(a.new_v)
                                        : static_cast<const T *>(a.new_k)) + slice * D;
            new_lo[u] = src[row_i[u]];
            new_hi[u] = src[row_i[u] + D / 2];
        }
    }

    const int64_t T_ = (int64_t)a.seqlens_k[b] + 1;
    const bool write_len = kvh == 0 && threadIdx.x == 0 && a.len.cache_total != nullptr;
    if (T_ < 1 || T_ > (int64_t)INT32_MAX) {
        if (write_len) {
            a.len.past_abs[b] = a.len.total_abs[b] = a.len.cache_past[b] = a.len.cache_total[b] =
                a.len.evict[b] = -1;
        }
        if (kvh == 0 && threadIdx.x == 0)
            kvc::raise_status(a.status, KVC_DEV_SEQLEN_RANGE);
        return;
    }
    const int P = (int)(T_ - 1);
    int64_t Lp64, E64, L64;
    kvc::cache_lengths(a.policy, T_, 1, C, a.window, Lp64, E64, L64);
    const int Lp = (int)Lp64, E = (int)E64, L = (int)L64;
    if (write_len) {
        a.len.past_abs[b] = P;
        a.len.total_abs[b] = (int32_t)T_;
        a.len.cache_past[b] = Lp;
        a.len.cache_total[b] = L;
        a.len.evict[b] = E;
    }
    if (a.cos_t && T_ > a.rope_max_pos) {
        if (kvh == 0 && threadIdx.x == 0)
            kvc::raise_status(a.status, KVC_DEV_ROPE_RANGE);
        return;
    }
    const bool ring = a.policy == KVC_RING;
    const bool moves = !ring && E > 0;
    const int nvis = (a.window > 0 && L > a.window) ? a.window : L;  // visible positions
    const int vis0 = L - nvis;
    const int64_t row0 = slice * C;  // the slice's first row in the tensor maps
    T *kc = static_cast<T *>(a.k_cache) + row0 * D;
    T *vc = static_cast<T *>(a.v_cache) + row0 * D;

    // Shared-memory rows: the slot s (ring); the window row r when rows move
    // (loaded from cache row r + E); otherwise only the visible rows, shared
    // row r holding window (and cache) row win0 + r, win0 = vis0 -- at any
    // row, since a TMA box may start at any row.  new_r: the new row's
    // shared row; [t_lo, t_hi): tiles loaded from the cache (shared row r
    // from cache row r + src_off).
    int new_r, t_lo, t_hi, src_off, win0 = 0;
    if (ring) {
        new_r = (int)((T_ - 1) % C);
        const int held = (int)(T_ - 1 < C ? T_ - 1 : C);  // slots holding an old token
        t_lo = 0;
        t_hi = (held + kTile - 1) / kTile;
        src_off = 0;
    } else if (moves) {
        new_r = L - 1;
        t_lo = 0;
        t_hi = (L - 1 + kTile - 1) / kTile;  // rows [0, L - 1) hold old tokens
        src_off = E;
    } else {
        win0 = vis0;
        new_r = L - 1 - win0;
        t_lo = 0;
        t_hi = (L - 1 - win0 + kTile - 1) / kTile;
        src_off = win0;
    }
    const int ntiles = ring ? (int)((C + kTile - 1) / kTile) : (L - win0 + kTile - 1) / kTile;

    // 1. one thread starts the TMA loads of the old rows, one barrier a tile
    if (threadIdx.x == 0) {
        for (int t = t_lo; t < t_hi; ++t) {
            const int32_t y = (int32_t)(row0 + src_off + t * kTile);
            kvc::mbar_arrive_expect_tx(&bar[t], 2u * KT_BYTES);
#pragma unroll
            for (int bx = 0; bx < BOXES; ++bx) {
                kvc::tma_load_2d(tiles + (size_t)t * 2 * KT_BYTES + bx * 8192, &tmap_k, bx * 64,
                                 y, &bar[t]);
                kvc::tma_load_2d(tiles + (size_t)t * 2 * KT_BYTES + KT_BYTES + bx * 8192,
                                 &tmap_v, bx * 64, y, &bar[t]);
            }
        }
    }

    // 2. meanwhile: the query rows and the new K row rotated at P = T - 1
    //    (the cos/sin rows are the only loads that needed the lengths)
    const float *cs = a.cos_t ? a.cos_t + (int64_t)P * (D / 2) : nullptr;
    const float *sn = a.cos_t ? a.sin_t + (int64_t)P * (D / 2) : nullptr;
#pragma unroll
    for (int j = 0; j < QPT; ++j) {
        const int idx = threadIdx.x + 128 * j;
        const int h = idx / (D / 2), i = idx % (D / 2);
        float lo = kvc::Elem<T>::to_f32(q_lo[j]), hi = kvc::Elem<T>::to_f32(q_hi[j]);
        if (cs && h < g)
            kvc::rope_pair(lo, hi, cs[i], sn[i]);
        qs[h * QS + i] = kvc::Elem<T>::from_f32(lo);
        qs[h * QS + i + D / 2] = kvc::Elem<T>::from_f32(hi);
    }
#pragma unroll
    for (int u = 0; u < RPT; ++u) {
        if (row_thread[u] && !row_is_v[u] && cs) {
            float lo = kvc::Elem<T>::to_f32(new_lo[u]), hi = kvc::Elem<T>::to_f32(new_hi[u]);
            kvc::rope_pair(lo, hi, cs[row_i[u]], sn[row_i[u]]);
            new_lo[u] = kvc::Elem<T>::from_f32(lo);
            new_hi[u] = kvc::Elem<T>::from_f32(hi);
        }
    }

    // the new row goes to shared memory and, without an eviction, straight
    // to its cache row (a load of that row, if any, is overwritten below)
#pragma unroll
    for (int u = 0; u < RPT; ++u) {
        if (!moves && row_thread[u]) {
            T *dst = (row_is_v[u] ? vc : kc) + (int64_t)(new_r + win0) * D;
            dst[row_i[u]] = new_lo[u];
            dst[row_i[u] + D / 2] = new_hi[u];
        }
    }

    // rows whose V is zeroed: wherever attention might touch a row that
    // holds no token of the window (0 * stale bytes must stay 0) -- rows past
    // the window in its last tile; for a ring, the slots never written
    // (T <= C) and the slots past C
    const int z0 = ring ? (T_ < C ? (int)T_ : (int)C) : L - win0;
    const int z1 = ntiles * kTile;
    const int stored_tiles = moves ? L / kTile : 0;  // full tiles stored by TMA

    // visible rows: window rows [vis0, L) (shared rows from vis0 - win0), or
    // for a ring the nvis slots ending at new_r (one run, or [0, new_r] and
    // [C - rest, C))
    int lo1 = vis0 - win0, hi1 = L - win0, lo2 = 0, hi2 = 0;
    if (ring) {
        const int first = new_r - nvis + 1;
        if (first >= 0) {
            lo1 = first;
            hi1 = new_r + 1;
        } else {
            lo1 = 0;
            hi1 = new_r + 1;
            lo2 = (int)C + first;
            hi2 = (int)C;
        }
    }

    // 3-5. the tiles in order: wait for the tile, place what belongs in it,
    //      store it back when rows moved, run its attention
    __syncthreads();  // the barriers' initialisation is visible to all threads
    GroupAttn<T, D, HB, decode_q_in_registers<D, HB>()> ga;
    ga.init();
    ga.load_q(qs, QS, lane);
    // (a wait that runs out marks this thread; the loop goes on, skipping
    // the work, so that every thread meets the same barriers)
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
        if (t >= t_lo && t < t_hi && !kvc::mbar_wait(&bar[t], 0))
            ok = false;
        const int r_lo = t * kTile, r_hi = r_lo + kTile;
        const bool has_new = new_r >= r_lo && new_r < r_hi;
        const int zl = max(z0, r_lo), zh = min(z1, r_hi);
        if (has_new || zh > zl) {
#pragma unroll
            for (int u = 0; u < RPT; ++u) {
                if (has_new && row_thread[u]) {
                    const int ri = row_i[u];
                    const int c_lo = ri / 8, c_hi = (ri + D / 2) / 8;
                    *reinterpret_cast<T *>(at(row_is_v[u], new_r, c_lo) + (ri % 8) * 2) =
                        new_lo[u];
                    *reinterpret_cast<T *>(at(row_is_v[u], new_r, c_hi) +
                                           ((ri + D / 2) % 8) * 2) = new_hi[u];
                }
            }
            for (int idx = threadIdx.x; idx < (zh - zl) * CPR; idx += 128)
                *reinterpret_cast<uint4 *>(at(true, zl + idx / CPR, idx % CPR)) =
                    make_uint4(0, 0, 0, 0);
            kvc::fence_proxy_async_smem();
            __syncthreads();
        }
        if (t < stored_tiles) {
            if (threadIdx.x == 0 && ok) {
                const int32_t y = (int32_t)(row0 + r_lo);
#pragma unroll
                for (int bx = 0; bx < BOXES; ++bx) {
                    kvc::tma_store_2d(&tmap_k, bx * 64, y,
                                      tiles + (size_t)t * 2 * KT_BYTES + bx * 8192);
                    kvc::tma_store_2d(&tmap_v, bx * 64, y,
                                      tiles + (size_t)t * 2 * KT_BYTES + KT_BYTES + bx * 8192);
                }
                kvc::tma_store_commit();
            }
        } else if (moves && r_lo < L && ok) {
            // the last, partial tile: rows [r_lo, L) by the threads (its
            // final contents were made visible by the barrier above)
            const int n = (L - r_lo) * CPR;
            for (int idx = threadIdx.x; idx < 2 * n; idx += 128) {
                const bool is_v = idx >= n;
                const int w = is_v ? idx - n : idx;
                const int r = r_lo + w / CPR, c = w % CPR;
                *reinterpret_cast<uint4 *>((is_v ? vc : kc) + (int64_t)r * D + c * 8) =
                    *reinterpret_cast<const uint4 *>(at(is_v, r, c));
            }
        }
        const int r0 = r_lo + 16 * warp;  // this warp's 16 rows of the tile
        const uint32_t kb = kvc::smem_u32(tiles + (size_t)t * 2 * KT_BYTES);
        const int l1 = min(16, max(0, lo1 - r0)), h1 = min(16, max(0, hi1 - r0));
        const int l2 = min(16, max(0, lo2 - r0)), h2 = min(16, max(0, hi2 - r0));
        if (ok && h1 > l1)
            ga.tile(kb, kb + KT_BYTES, warp, lane, l1, h1, a.scale_log2);
        if (ok && h2 > l2)
            ga.tile(kb, kb + KT_BYTES, warp, lane, l2, h2, a.scale_log2);
    }
    if (threadIdx.x == 0 && stored_tiles > 0)
        kvc::tma_store_wait_read();  // the merge below reuses the tiles' memory
    if (!__syncthreads_and(ok)) {
        // a tile that never landed: report it, let every copy in flight land
        // (each wait bounded) and leave the output unwritten
        if (threadIdx.x == 0) {
            kvc::raise_status(a.status, KVC_DEV_TIMEOUT);
            for (int t = t_lo; t < t_hi; ++t)
                kvc::mbar_wait(&bar[t], 0);
        }
        return;
    }

    // 6. merge the four warps and write the group's output rows
    float *cm = reinterpret_cast<float *>(smem);
    float *cl = cm + kConsumers * 16;
    float *co = cl + kConsumers * 16;
    ga.publish(cm, cl, co, warp, lane, g, 16, D + 4);
    __syncthreads();
    for (int idx = threadIdx.x; idx < g * (D / 4); idx += 128) {
        const int h = idx / (D / 4), d = (idx % (D / 4)) * 4;
        const Merged4 r = merge4(cm, cl, co, D + 4, 16, h, d);
        const int64_t qrow = (int64_t)b * a.q_heads + kvh * g + h;
        store_out4(static_cast<T *>(a.out) + qrow * D + d, r);
    }
}

} // namespace

// --------------------------------------------------------------------------
// fp32 attention on CUDA cores (decode and multi-token), one warp per query
// --------------------------------------------------------------------------
namespace kvc_f32 {

// n_rows_mode 0: rows [0, cache_total) (decode); 1: rows [0, cache_past + S)
// (multi-token chunk over staged or contiguous rows); 2: the newest
// cache_total positions of a ring of rows_per_head slots (decode), position
// p in slot p mod rows_per_head
__global__ void __launch_bounds__(128)
attn_f32_kernel(float *__restrict__ out, const float *__restrict__ q,
                const float *__restrict__ k_rows, const float *__restrict__ v_rows,
                int64_t rows_per_head, kvc_lengths len, int batch, int q_heads, int kv_heads,
                int S, int D, int window, float scale, const float *__restrict__ cos_t,
                const float *__restrict__ sin_t, int64_t rope_max_pos, int n_rows_mode,
                int32_t *status)
{
    extern __shared__ float qsh[];  // [4][D]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t qrow = (int64_t)blockIdx.x * 4 + warp;  // over (b, h, i)
    if (qrow >= (int64_t)batch * q_heads * S)
        return;
    const int i = (int)(qrow % S);
    const int h = (int)((qrow / S) % q_heads);
    const int b = (int)(qrow / ((int64_t)S * q_heads));
    const int L = len.cache_total[b];
    if (L < 0)
        return;
    const int64_t T = len.total_abs[b];
    if (cos_t && T > rope_max_pos) {
        if (lane == 0 && h == 0 && i == 0)
            kvc::raise_status(status, KVC_DEV_ROPE_RANGE);
        return;
    }
    const int64_t n = n_rows_mode != 1 ? L : (int64_t)len.cache_past[b] + S;
    if (n > rows_per_head || n < S || (n_rows_mode == 2 && n > T)) {
        if (lane == 0 && h == 0 && i == 0)
            kvc::raise_status(status, KVC_DEV_CAPACITY);
        return;
    }
    const int64_t first_pos = T - n;
    const int64_t qpos = T - S + i;
    float *qv = qsh + warp * D;
    const float *qsrc = q + qrow * D;
    for (int d = lane; d < D / 2; d += 32) {
        float lo = qsrc[d], hi = qsrc[d + D / 2];
        if (cos_t)
            kvc::rope_pair(lo, hi, cos_t[qpos * (D / 2) + d], sin_t[qpos * (D / 2) + d]);
        qv[d] = lo;
        qv[d + D / 2] = hi;
    }
    __syncwarp();
    // visible rows: kpos in [qpos - window + 1, qpos], row r holds first_pos + r
    int64_t lo_r = 0, hi_r = qpos - first_pos;  // inclusive
    if (window > 0 && qpos - window + 1 - first_pos > lo_r)
        lo_r = qpos - window + 1 - first_pos;
    if (hi_r > n - 1)
        hi_r = n - 1;
    const int kvh = h / (q_heads / kv_heads);
    // logical row r (position first_pos + r) lives in row slot(r)
    const bool ring = n_rows_mode == 2;
    auto slot = [&](int64_t r) { return ring ? (first_pos + r) % rows_per_head : r; };
    const float *kb = k_rows + ((int64_t)b * kv_heads + kvh) * rows_per_head * D;
    const float *vb = v_rows + ((int64_t)b * kv_heads + kvh) * rows_per_head * D;
    float m = -INFINITY;
    for (int64_t r = lo_r + lane; r <= hi_r; r += 32) {
        float dot = 0.f;
        const float *kr = kb + slot(r) * D;
        for (int d = 0; d < D; ++d)
            dot += qv[d] * kr[d];
        m = fmaxf(m, dot * scale);
    }
    for (int off = 16; off > 0; off >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // d = lane + 32 j, D <= 256
    float l = 0.f;
    for (int64_t c0 = lo_r; c0 <= hi_r; c0 += 32) {
        const int64_t r = c0 + lane;
        float p = 0.f;
        if (r <= hi_r) {
            float dot = 0.f;
            const float *kr = kb + slot(r) * D;
            for (int d = 0; d < D; ++d)
                dot += qv[d] * kr[d];
            p = expf(dot * scale - m);
        }
        l += p;
        const int cnt = (int)min((int64_t)32, hi_r - c0 + 1);
        for (int j = 0; j < cnt; ++j) {
            const float pj = __shfl_sync(0xffffffffu, p, j);
            const float *vr = vb + slot(c0 + j) * D;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (lane + 32 * u < D)
                    acc[u] += pj * vr[lane + 32 * u];
        }
    }
    for (int off = 16; off > 0; off >>= 1)
        l += __shfl_xor_sync(0xffffffffu, l, off);
#pragma unroll
    for (int u = 0; u < 8; ++u)
        if (lane + 32 * u < D)
            out[qrow * D + lane + 32 * u] = acc[u] / l;
}

kvc_status launch(void *out, const void *q, const void *k_rows, const void *v_rows,
                  int64_t rows_per_head, const kvc_lengths &len, int batch, int q_heads,
                  int kv_heads, int S, int D, int window, float scale, const float *cos_t,
                  const float *sin_t, int64_t rope_max_pos, int n_rows_mode, int32_t *status,
                  cudaStream_t stream)
{
    const int64_t rows = (int64_t)batch * q_heads * S;
    const int64_t blocks = (rows + 3) / 4;
    if (blocks > INT32_MAX)
        return KVC_ERR_SHAPE;
    attn_f32_kernel<<<(unsigned)blocks, 128, 4 * D * sizeof(float), stream>>>(
        static_cast<float *>(out), static_cast<const float *>(q),
        static_cast<const float *>(k_rows), static_cast<const float *>(v_rows), rows_per_head, len,
        batch, q_heads, kv_heads, S, D, window, scale, cos_t, sin_t, rope_max_pos, n_rows_mode,
        status);
    return kvc_host::launch_status();
}

} // namespace kvc_f32

namespace {

// the page table of a paged cache (kvc_gqa_decode_paged)
struct PagedExtra {
    const int32_t *block_table;
    int max_pages, page_size;
    int64_t n_pool_pages;
    const uint8_t *qk_pool, *qv_pool;  // int8 pages (kvc_gqa_decode_paged_q), else NULL
    const float *qparams;
    int64_t n_q_pages;
};

// inputs of the fused step (kvc_decode_step) on top of the decode's own
struct StepExtra {
    const int32_t *seqlens_k;
    const void *new_k, *new_v;
    void *k_cache, *v_cache;
};

template <typename T, int D>
kvc_status launch_decode16(void *out, const void *q, const void *k_cache, const void *v_cache,
                           const kvc_lengths &len, int batch, int q_heads, int kv_heads,
                           int64_t C, int window, float scale, const float *cos_t,
                           const float *sin_t, int64_t rope_max_pos, void *workspace,
                           int ring, int32_t *status, cudaStream_t stream,
                           const StepExtra *fx = nullptr, const PagedExtra *px = nullptr)
{
    const CUtensorMapDataType tt = std::is_same<T, __half>::value
                                       ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap tk, tv;
    // a paged cache maps the whole page pool [pages, kv_heads, page_size, D]
    const uint64_t rows = px ? (uint64_t)px->n_pool_pages * kv_heads * px->page_size
                             : (uint64_t)batch * kv_heads * C;
    if (rows > (uint64_t)INT32_MAX)
        return KVC_ERR_SHAPE;
    if (!kvc_host::encode_2d_bf16_sw128(&tk, k_cache, rows, D, kTile, tt) ||
        !kvc_host::encode_2d_bf16_sw128(&tv, v_cache, rows, D, kTile, tt))
        return KVC_ERR_CUDA;
    DecodeArgs a{};
    a.out = out;
    a.q = q;
    a.len = len;
    a.batch = batch;
    a.q_heads = q_heads;
    a.kv_heads = kv_heads;
    a.group = q_heads / kv_heads;
    a.capacity = C;
    a.ring = ring;
    a.window = window;
    a.scale_log2 = scale * kLog2e;
    a.cos_t = cos_t;
    a.sin_t = sin_t;
    a.rope_max_pos = rope_max_pos;
    a.split_rows = decode_split_rows(C, D);
    // int8 pages: twice the rows per split (the same bytes per CTA as a
    // 16-bit split; fewer CTAs, so less of their fixed start and merge cost)
    if (px && px->qk_pool && C >= 4096)
        a.split_rows *= 2;
    a.max_splits = (int)((C + a.split_rows - 1) / a.split_rows);
    const int64_t np = (int64_t)batch * q_heads * a.max_splits;
    a.ws_o = static_cast<float *>(workspace);
    a.ws_m = a.ws_o + np * D;
    a.ws_l = a.ws_m + np;
    a.status = status;
    const int64_t n_items = (int64_t)a.max_splits * kv_heads * batch;
    if (n_items > (int64_t)INT32_MAX)
        return KVC_ERR_SHAPE;
    if (fx) {
        a.seqlens_k = fx->seqlens_k;
        a.new_k = fx->new_k;
        a.new_v = fx->new_v;
        a.k_cache = fx->k_cache;
        a.v_cache = fx->v_cache;
    }
    if (px) {
        a.block_table = px->block_table;
        a.max_pages = px->max_pages;
        a.page_size = px->page_size;
        a.n_pool_pages = px->n_pool_pages;
        a.qk_pool = px->qk_pool;
        a.qv_pool = px->qv_pool;
        a.qparams = px->qparams;
        a.n_q_pages = px->n_q_pages;
    }
    const bool q8 = px && px->qk_pool;
    const size_t smem = 1024 + (size_t)(q8 ? decode_smem_bytes<D, kPagedQ>()
                                           : decode_smem_bytes<D, kPlain>());
    const int threads = q8 ? decode_threads<D, kPagedQ>() : decode_threads<D, kPlain>();
    // one block of 8 query heads per KV head up to a group of 8, two up to 16
    const bool hb2 = a.group > 8;
    auto kern = fx ? (hb2 ? decode_split_kernel<T, D, kFused, 2> : decode_split_kernel<T, D, kFused, 1>)
                : q8 ? (hb2 ? decode_split_kernel<T, D, kPagedQ, 2>
                            : decode_split_kernel<T, D, kPagedQ, 1>)
                : px ? (hb2 ? decode_split_kernel<T, D, kPaged, 2> : decode_split_kernel<T, D, kPaged, 1>)
                     : (hb2 ? decode_split_kernel<T, D, kPlain, 2>
                            : decode_split_kernel<T, D, kPlain, 1>);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return KVC_ERR_CUDA;
    const dim3 grid(a.max_splits, kv_heads, batch);
    kern<<<grid, threads, smem, stream>>>(tk, tv, a);
    if (a.max_splits > 1) {
        dim3 g2(q_heads, batch);
        const size_t cs = 3 * a.max_splits * sizeof(float);
        const bool fast = a.max_splits <= kFastSplits && D <= 128 * kFastCols;
        if (fx && fast)
            decode_combine_fast_kernel<T, kFused><<<g2, 128, 0, stream>>>(a, D);
        else if (fx)
            decode_combine_kernel<T, kFused><<<g2, 128, cs, stream>>>(a, D);
        else if (px && fast)
            decode_combine_fast_kernel<T, kPaged><<<g2, 128, 0, stream>>>(a, D);
        else if (px)
            decode_combine_kernel<T, kPaged><<<g2, 128, cs, stream>>>(a, D);
        else if (fast)
            decode_combine_fast_kernel<T, kPlain><<<g2, 128, 0, stream>>>(a, D);
        else
            decode_combine_kernel<T, kPlain><<<g2, 128, cs, stream>>>(a, D);
    }
    return kvc_host::launch_status();
}

// the 16-bit tensor-core kernels: element type and head dimension as
// template arguments
template <typename T_, int D_> struct Dim16 {
    using T = T_;
    static constexpr int D = D_;
};
inline bool dim16_ok(int D) { return D == 64 || D == 128 || D == 256; }

template <typename F> kvc_status with_dim16(int dtype, int D, F &&f)
{
    if (dtype == KVC_BF16) {
        if (D == 64)
            return f(Dim16<__nv_bfloat16, 64>{});
        if (D == 128)
            return f(Dim16<__nv_bfloat16, 128>{});
        if (D == 256)
            return f(Dim16<__nv_bfloat16, 256>{});
    } else if (dtype == KVC_F16) {
        if (D == 64)
            return f(Dim16<__half, 64>{});
        if (D == 128)
            return f(Dim16<__half, 128>{});
        if (D == 256)
            return f(Dim16<__half, 256>{});
    }
    return KVC_ERR_UNSUPPORTED;
}

} // namespace

KVC_API size_t kvc_gqa_decode_workspace_size(int batch, int q_heads, int kv_heads,
                                             int64_t capacity, int head_dim, int dtype)
{
    if (batch < 0 || q_heads < 1 || kv_heads < 1 || capacity < 1 || head_dim < 1)
        return 0;
    if (dtype == KVC_F32)
        return 256;  // the CUDA-core path keeps everything on chip
    const int64_t ns = decode_max_splits(capacity, head_dim);
    if (ns <= 1)
        return 256;
    const int64_t np = (int64_t)batch * q_heads * ns;
    return (size_t)(np * (head_dim + 2) * sizeof(float));
}

namespace {

kvc_status decode_entry(void *out, const void *q, const void *k_cache, const void *v_cache,
                        kvc_lengths len, int batch, int q_heads, int kv_heads, int64_t capacity,
                        int head_dim, int dtype, int local_window_size, float scale,
                        const float *rope_cos, const float *rope_sin, int64_t rope_max_pos,
                        void *workspace, size_t workspace_bytes, int ring, int32_t *dev_status,
                        void *stream_)
{
    const int eb = kvc_host::elem_bytes_of(dtype);
    if (eb == 0)
        return KVC_ERR_DTYPE;
    if (batch < 0 || q_heads < 1 || kv_heads < 1 || q_heads % kv_heads != 0 || head_dim < 2 ||
        (head_dim & 1))
        return KVC_ERR_SHAPE;
    if (capacity < 1 || capacity > (int64_t)INT32_MAX)
        return KVC_ERR_CAPACITY;
    if ((rope_cos == nullptr) != (rope_sin == nullptr))
        return KVC_ERR_NULL;
    if (rope_cos && rope_max_pos < 1)
        return KVC_ERR_SHAPE;
    const int g = q_heads / kv_heads;
    if (dtype == KVC_F32 ? head_dim > 256 : (!dim16_ok(head_dim) || g > 16))
        return KVC_ERR_UNSUPPORTED;
    if (batch == 0)
        return KVC_OK;
    if (!out || !q || !k_cache || !v_cache || !kvc_host::lengths_ok(len))
        return KVC_ERR_NULL;
    for (const void *p : {(const void *)out, q, k_cache, v_cache})
        if (!kvc_host::aligned16(p))
            return KVC_ERR_ALIGN;
    const size_t need =
        kvc_gqa_decode_workspace_size(batch, q_heads, kv_heads, capacity, head_dim, dtype);
    if (need > 256 && (!workspace || workspace_bytes < need))
        return KVC_ERR_WORKSPACE;
    if (need > 256 && (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return KVC_ERR_ALIGN;
    if (scale == 0.f)
        scale = 1.0f / sqrtf((float)head_dim);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (dtype == KVC_F32)
        return kvc_f32::launch(out, q, k_cache, v_cache, capacity, len, batch, q_heads, kv_heads,
                               1, head_dim, local_window_size, scale, rope_cos, rope_sin,
                               rope_max_pos, ring ? 2 : 0, dev_status, stream);
    return with_dim16(dtype, head_dim, [&](auto td) {
        using TD = decltype(td);
        return launch_decode16<typename TD::T, TD::D>(
            out, q, k_cache, v_cache, len, batch, q_heads, kv_heads, capacity, local_window_size,
            scale, rope_cos, rope_sin, rope_max_pos, workspace, ring, dev_status, stream);
    });
}

} // namespace

KVC_API kvc_status kvc_gqa_decode(void *out, const void *q, const void *k_cache,
                                  const void *v_cache, kvc_lengths len, int batch, int q_heads,
                                  int kv_heads, int64_t capacity, int head_dim, int dtype,
                                  int local_window_size, float scale, const float *rope_cos,
                                  const float *rope_sin, int64_t rope_max_pos, void *workspace,
                                  size_t workspace_bytes, int32_t *dev_status, void *stream)
{
    return decode_entry(out, q, k_cache, v_cache, len, batch, q_heads, kv_heads, capacity,
                        head_dim, dtype, local_window_size, scale, rope_cos, rope_sin,
                        rope_max_pos, workspace, workspace_bytes, 0, dev_status, stream);
}

KVC_API kvc_status kvc_gqa_decode_ring(void *out, const void *q, const void *k_cache,
                                       const void *v_cache, kvc_lengths len, int batch,
                                       int q_heads, int kv_heads, int64_t capacity, int head_dim,
                                       int dtype, int local_window_size, float scale,
                                       const float *rope_cos, const float *rope_sin,
                                       int64_t rope_max_pos, void *workspace,
                                       size_t workspace_bytes, int32_t *dev_status, void *stream)
{
    return decode_entry(out, q, k_cache, v_cache, len, batch, q_heads, kv_heads, capacity,
                        head_dim, dtype, local_window_size, scale, rope_cos, rope_sin,
                        rope_max_pos, workspace, workspace_bytes, 1, dev_status, stream);
}

namespace {

kvc_status paged_decode_entry(void *out, const void *q, const void *k_pool, const void *v_pool,
                              const uint8_t *qk_pool, const uint8_t *qv_pool, const float *qparams,
                              int64_t n_q_pages, const int32_t *block_table, int max_pages,
                              int64_t n_pool_pages, int page_size, kvc_lengths len, int batch,
                              int q_heads, int kv_heads, int head_dim, int dtype,
                              int local_window_size, float scale, const float *rope_cos,
                              const float *rope_sin, int64_t rope_max_pos, void *workspace,
                              size_t workspace_bytes, int32_t *dev_status, void *stream)
{
    if (dtype != KVC_BF16 && dtype != KVC_F16)
        return dtype == KVC_F32 ? KVC_ERR_UNSUPPORTED : KVC_ERR_DTYPE;
    if (batch < 0 || q_heads < 1 || kv_heads < 1 || q_heads % kv_heads != 0)
        return KVC_ERR_SHAPE;
    if (!dim16_ok(head_dim) || q_heads / kv_heads > 16)
        return KVC_ERR_UNSUPPORTED;
    // pages hold whole 64-row tiles
    if (page_size < kTile || page_size % kTile != 0 || max_pages < 1 || n_pool_pages < 1)
        return KVC_ERR_SHAPE;
    const int64_t capacity = (int64_t)max_pages * page_size;
    if (capacity > (int64_t)INT32_MAX ||
        n_pool_pages * kv_heads * (int64_t)page_size > (int64_t)INT32_MAX)
        return KVC_ERR_CAPACITY;
    if ((rope_cos == nullptr) != (rope_sin == nullptr))
        return KVC_ERR_NULL;
    if (rope_cos && rope_max_pos < 1)
        return KVC_ERR_SHAPE;
    if (batch == 0)
        return KVC_OK;
    if (!out || !q || !k_pool || !v_pool || !block_table || !kvc_host::lengths_ok(len))
        return KVC_ERR_NULL;
    for (const void *p : {(const void *)out, q, k_pool, v_pool})
        if (!kvc_host::aligned16(p))
            return KVC_ERR_ALIGN;
    const size_t pool_bytes = (size_t)n_pool_pages * kv_heads * page_size * head_dim * 2;
    if (kvc_host::overlaps(k_pool, pool_bytes, v_pool, pool_bytes))
        return KVC_ERR_SHAPE;
    const size_t need =
        kvc_gqa_decode_workspace_size(batch, q_heads, kv_heads, capacity, head_dim, dtype);
    if (need > 256 && (!workspace || workspace_bytes < need))
        return KVC_ERR_WORKSPACE;
    if (need > 256 && (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return KVC_ERR_ALIGN;
    if (scale == 0.f)
        scale = 1.0f / sqrtf((float)head_dim);
    const PagedExtra px{block_table, max_pages, page_size, n_pool_pages, qk_pool, qv_pool, qparams,
                        n_q_pages};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return with_dim16(dtype, head_dim, [&](auto td) {
        using TD = decltype(td);
        return launch_decode16<typename TD::T, TD::D>(
            out, q, k_pool, v_pool, len, batch, q_heads, kv_heads, capacity, local_window_size,
            scale, rope_cos, rope_sin, rope_max_pos, workspace, 0, dev_status, st, nullptr, &px);
    });
}

} // namespace

KVC_API kvc_status kvc_gqa_decode_paged(void *out, const void *q, const void *k_pool,
                                        const void *v_pool, const int32_t *block_table,
                                        int max_pages, int64_t n_pool_pages, int page_size,
                                        kvc_lengths len, int batch, int q_heads, int kv_heads,
                                        int head_dim, int dtype, int local_window_size,
                                        float scale, const float *rope_cos,
                                        const float *rope_sin, int64_t rope_max_pos,
                                        void *workspace, size_t workspace_bytes,
                                        int32_t *dev_status, void *stream)
{
    return paged_decode_entry(out, q, k_pool, v_pool, nullptr, nullptr, nullptr, 0, block_table,
                              max_pages, n_pool_pages, page_size, len, batch, q_heads, kv_heads,
                              head_dim, dtype, local_window_size, scale, rope_cos, rope_sin,
                              rope_max_pos, workspace, workspace_bytes, dev_status, stream);
}

KVC_API kvc_status kvc_gqa_decode_paged_q(void *out, const void *q, const void *k_pool,
                                          const void *v_pool, const void *qk_pool,
                                          const void *qv_pool, const float *qparams,
                                          int64_t n_qpool_pages, const int32_t *block_table,
                                          int max_pages, int64_t n_pool_pages, int page_size,
                                          kvc_lengths len, int batch, int q_heads, int kv_heads,
                                          int head_dim, int dtype, int local_window_size,
                                          float scale, const float *rope_cos,
                                          const float *rope_sin, int64_t rope_max_pos,
                                          void *workspace, size_t workspace_bytes,
                                          int32_t *dev_status, void *stream)
{
    if (n_qpool_pages < 1 || n_qpool_pages * kv_heads * (int64_t)page_size * head_dim >
                                 ((int64_t)1 << 40))
        return KVC_ERR_SHAPE;
    if (batch > 0) {
        if (!qk_pool || !qv_pool || !qparams)
            return KVC_ERR_NULL;
        for (const void *p : {qk_pool, qv_pool, (const void *)qparams})
            if (!kvc_host::aligned16(p))
                return KVC_ERR_ALIGN;
        const size_t qb = (size_t)n_qpool_pages * kv_heads * page_size * head_dim;
        if (kvc_host::overlaps(qk_pool, qb, qv_pool, qb))
            return KVC_ERR_SHAPE;
    }
    return paged_decode_entry(out, q, k_pool, v_pool, static_cast<const uint8_t *>(qk_pool),
                              static_cast<const uint8_t *>(qv_pool), qparams, n_qpool_pages,
                              block_table, max_pages, n_pool_pages, page_size, len, batch,
                              q_heads, kv_heads, head_dim, dtype, local_window_size, scale,
                              rope_cos, rope_sin, rope_max_pos, workspace, workspace_bytes,
                              dev_status, stream);
}

// --------------------------------------------------------------------------
// kvc_decode_step: lengths + one-token append + split decode of a contiguous
// cache or a ring in one launch (plus the split merge for long rows)
// --------------------------------------------------------------------------

// the step's workspace holds the same split partials as the decode's
KVC_API size_t kvc_decode_step_workspace_size(int batch, int q_heads, int kv_heads,
                                              int64_t capacity, int head_dim, int dtype)
{
    if (dtype == KVC_F32)
        return 0;
    return kvc_gqa_decode_workspace_size(batch, q_heads, kv_heads, capacity, head_dim, dtype);
}

KVC_API kvc_status kvc_decode_step(void *out, const void *q, void *k_cache, void *v_cache,
                                   const void *new_k, const void *new_v, const int32_t *seqlens_k,
                                   kvc_lengths len, int batch, int q_heads, int kv_heads,
                                   int64_t capacity, int head_dim, int dtype, int windowed,
                                   int local_window_size, float scale, const float *rope_cos,
                                   const float *rope_sin, int64_t rope_max_pos, void *workspace,
                                   size_t workspace_bytes, int32_t *dev_status, void *stream)
{
    if (kvc_host::elem_bytes_of(dtype) == 0)
        return KVC_ERR_DTYPE;
    if (batch < 0 || q_heads < 1 || kv_heads < 1 || q_heads % kv_heads != 0)
        return KVC_ERR_SHAPE;
    if (capacity < 1 || capacity > (int64_t)INT32_MAX)
        return KVC_ERR_CAPACITY;
    if (windowed != KVC_CONTIGUOUS && windowed != KVC_RING)
        return KVC_ERR_UNSUPPORTED;
    if ((rope_cos == nullptr) != (rope_sin == nullptr))
        return KVC_ERR_NULL;
    if (rope_cos && rope_max_pos < 1)
        return KVC_ERR_SHAPE;
    const int g = q_heads / kv_heads;
    // the merge keeps 3 x 16 x splits floats next to the 4-warp partials in
    // the stage buffers: at most 128 splits (capacity 65536)
    if (dtype == KVC_F32 || !dim16_ok(head_dim) || g > 16 ||
        decode_max_splits(capacity, head_dim) > 128)
        return KVC_ERR_UNSUPPORTED;
    const bool some_len = len.past_abs || len.total_abs || len.cache_past || len.cache_total ||
                          len.evict;
    if (some_len && !kvc_host::lengths_ok(len))
        return KVC_ERR_NULL;
    if (batch == 0)
        return KVC_OK;
    if (!out || !q || !k_cache || !v_cache || !new_k || !new_v || !seqlens_k)
        return KVC_ERR_NULL;
    for (const void *p : {(const void *)out, q, (const void *)k_cache, (const void *)v_cache, new_k,
                          new_v})
        if (!kvc_host::aligned16(p))
            return KVC_ERR_ALIGN;
    const size_t cache_bytes = (size_t)batch * kv_heads * capacity * head_dim * 2;
    if (kvc_host::overlaps(k_cache, cache_bytes, v_cache, cache_bytes))
        return KVC_ERR_SHAPE;
    const size_t need =
        kvc_decode_step_workspace_size(batch, q_heads, kv_heads, capacity, head_dim, dtype);
    if (need > 256 && (!workspace || workspace_bytes < need))
        return KVC_ERR_WORKSPACE;
    if (need > 256 && (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return KVC_ERR_ALIGN;
    if (scale == 0.f)
        scale = 1.0f / sqrtf((float)head_dim);
    StepExtra fx;
    fx.seqlens_k = seqlens_k;
    fx.new_k = new_k;
    fx.new_v = new_v;
    fx.k_cache = k_cache;
    fx.v_cache = v_cache;
    const kvc_lengths l = some_len ? len : kvc_lengths{nullptr, nullptr, nullptr, nullptr, nullptr};
    const int ring = windowed == KVC_RING;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return with_dim16(dtype, head_dim, [&](auto td) {
        using TD = decltype(td);
        return launch_decode16<typename TD::T, TD::D>(
            out, q, k_cache, v_cache, l, batch, q_heads, kv_heads, capacity, local_window_size,
            scale, rope_cos, rope_sin, rope_max_pos, workspace, ring, dev_status, st, &fx);
    });
}

namespace {

// shared memory of one SM (cached per device)
size_t smem_per_sm()
{
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 233472;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
                cudaSuccess ||
            n <= 0)
            n = 233472;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return (size_t)n;
}

template <typename T, int D>
kvc_status launch_window_step(const WindowStepArgs &a, int batch, cudaStream_t stream)
{
    const int64_t ntile_max = (a.capacity + kTile - 1) / kTile;
    // tiles, query rows and barriers; the merge's (m, l, o) reuses the tiles
    // and, for a window of one tile, part of the query rows after them (both
    // done with by then; it never reaches the barriers)
    const size_t tiles = (size_t)ntile_max * 2 * kTile * D * 2;
    const size_t merge = (2 * kConsumers * 16 + (size_t)kConsumers * 16 * (D + 4)) * sizeof(float);
    size_t smem = 1024 + (tiles > merge ? tiles : merge) + 16 * (D + 8) * 2 + 8 * ntile_max;
    // a window that compacts on every step writes its rows back each step:
    // at most four CTAs an SM, so that the next step's early CTAs (launched
    // as this one's signal at entry allows) do not crowd this step's loads
    // and stores in DRAM (five an SM measured 0.8 us slower a step on the
    // 128-row window; without the write-back, five are slightly faster)
    if (a.policy == KVC_WINDOWED) {
        const size_t four_an_sm = smem_per_sm() / 5 + 1;  // a fifth CTA no longer fits
        if (smem < four_an_sm)
            smem = four_an_sm;
    }
    const CUtensorMapDataType tt = std::is_same<T, __half>::value
                                       ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t rows = (uint64_t)batch * a.kv_heads * a.capacity;
    if (rows > (uint64_t)INT32_MAX)
        return KVC_ERR_SHAPE;
    CUtensorMap tk, tv;
    if (!kvc_host::encode_2d_bf16_sw128(&tk, a.k_cache, rows, D, kTile, tt) ||
        !kvc_host::encode_2d_bf16_sw128(&tv, a.v_cache, rows, D, kTile, tt))
        return KVC_ERR_CUDA;
    auto kern = a.group > 8 ? window_step_kernel<T, D, 2> : window_step_kernel<T, D, 1>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return KVC_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(batch * a.kv_heads));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tk, tv, a) != cudaSuccess)
        return KVC_ERR_CUDA;
    return kvc_host::launch_status();
}

} // namespace

namespace {

// the large-window step's workspace: the five length arrays (when the caller
// passes none), then the decode's split partials, each 256-byte aligned
inline size_t window_step_len_bytes(int batch) { return ((size_t)5 * batch * 4 + 255) / 256 * 256; }

} // namespace

KVC_API size_t kvc_window_decode_step_workspace_size(int batch, int q_heads, int kv_heads,
                                                     int64_t capacity, int head_dim, int dtype)
{
    if (batch < 0 || q_heads < 1 || kv_heads < 1 || capacity < 1 || head_dim < 1)
        return 0;
    if (capacity * head_dim <= kWindowStepMaxElems)
        return 0;  // the one-launch step keeps everything on chip
    return window_step_len_bytes(batch) +
           kvc_gqa_decode_workspace_size(batch, q_heads, kv_heads, capacity, head_dim, dtype);
}

KVC_API kvc_status kvc_window_decode_step(void *out, const void *q, void *k_cache, void *v_cache,
                                          const void *new_k, const void *new_v,
                                          const int32_t *seqlens_k, kvc_lengths len, int batch,
                                          int q_heads, int kv_heads, int64_t capacity,
                                          int head_dim, int dtype, int windowed,
                                          int local_window_size, float scale,
                                          const float *rope_cos, const float *rope_sin,
                                          int64_t rope_max_pos, void *workspace,
                                          size_t workspace_bytes, int32_t *dev_status,
                                          void *stream)
{
    if (kvc_host::elem_bytes_of(dtype) == 0)
        return KVC_ERR_DTYPE;
    if (windowed != KVC_WINDOWED && windowed != KVC_DRIFTING && windowed != KVC_RING)
        return KVC_ERR_UNSUPPORTED;
    if (batch < 0 || q_heads < 1 || kv_heads < 1 || q_heads % kv_heads != 0)
        return KVC_ERR_SHAPE;
    if (capacity < 1 || capacity > (int64_t)INT32_MAX)
        return KVC_ERR_CAPACITY;
    if (local_window_size <= 0 || local_window_size > capacity)
        return KVC_ERR_WINDOW;
    if ((rope_cos == nullptr) != (rope_sin == nullptr))
        return KVC_ERR_NULL;
    if (rope_cos && rope_max_pos < 1)
        return KVC_ERR_SHAPE;
    const int g = q_heads / kv_heads;
    if (dtype == KVC_F32 || !dim16_ok(head_dim) || g > 16)
        return KVC_ERR_UNSUPPORTED;
    const bool some_len = len.past_abs || len.total_abs || len.cache_past || len.cache_total ||
                          len.evict;
    if (some_len && !kvc_host::lengths_ok(len))
        return KVC_ERR_NULL;
    const bool large = capacity > window_step_max_capacity(head_dim);
    if (large && windowed == KVC_RING && decode_max_splits(capacity, head_dim) > 128)
        return KVC_ERR_UNSUPPORTED;
    if (batch == 0)
        return KVC_OK;
    if (large) {
        // A window too large to hold on chip: the ring runs as the fused
        // split step (nothing moves); a windowed or drifting cache runs
        // lengths, the in-place compaction + append, and the split decode.
        const size_t need = kvc_window_decode_step_workspace_size(batch, q_heads, kv_heads,
                                                                  capacity, head_dim, dtype);
        if (!workspace || workspace_bytes < need)
            return KVC_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 255u)
            return KVC_ERR_ALIGN;
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        const size_t lb = window_step_len_bytes(batch);
        if (windowed == KVC_RING)
            return kvc_decode_step(out, q, k_cache, v_cache, new_k, new_v, seqlens_k, len, batch,
                                   q_heads, kv_heads, capacity, head_dim, dtype, KVC_RING,
                                   local_window_size, scale, rope_cos, rope_sin, rope_max_pos,
                                   ws + lb, workspace_bytes - lb, dev_status, stream);
        kvc_lengths l = len;
        if (!some_len) {
            int32_t *w32 = reinterpret_cast<int32_t *>(ws);
            l = kvc_lengths{w32, w32 + batch, w32 + 2 * batch, w32 + 3 * batch, w32 + 4 * batch};
        }
        kvc_status st = kvc_seq_lengths(seqlens_k, batch, 1, capacity, windowed,
                                        local_window_size, l, dev_status, stream);
        if (st == KVC_OK)
            st = kvc_window_append(k_cache, v_cache, new_k, new_v, nullptr, nullptr, l, batch,
                                   kv_heads, 1, capacity, head_dim, dtype, windowed, KVC_APPEND,
                                   rope_cos, rope_sin, rope_max_pos, dev_status, stream);
        if (st == KVC_OK)
            st = kvc_gqa_decode(out, q, k_cache, v_cache, l, batch, q_heads, kv_heads, capacity,
                                head_dim, dtype, local_window_size, scale, rope_cos, rope_sin,
                                rope_max_pos, ws + lb, workspace_bytes - lb, dev_status, stream);
        return st;
    }
    if (!out || !q || !k_cache || !v_cache || !new_k || !new_v || !seqlens_k)
        return KVC_ERR_NULL;
    for (const void *p : {(const void *)out, q, (const void *)k_cache, (const void *)v_cache, new_k,
                          new_v})
        if (!kvc_host::aligned16(p))
            return KVC_ERR_ALIGN;
    const size_t cache_bytes = (size_t)batch * kv_heads * capacity * head_dim * 2;
    if (kvc_host::overlaps(k_cache, cache_bytes, v_cache, cache_bytes))
        return KVC_ERR_SHAPE;
    if (scale == 0.f)
        scale = 1.0f / sqrtf((float)head_dim);
    WindowStepArgs a;
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.new_k = new_k;
    a.new_v = new_v;
    a.seqlens_k = seqlens_k;
    a.len = some_len ? len : kvc_lengths{nullptr, nullptr, nullptr, nullptr, nullptr};
    a.q_heads = q_heads;
    a.kv_heads = kv_heads;
    a.group = g;
    a.capacity = capacity;
    a.policy = windowed;
    a.window = local_window_size;
    a.scale_log2 = scale * kLog2e;
    a.cos_t = rope_cos;
    a.sin_t = rope_sin;
    a.rope_max_pos = rope_max_pos;
    a.status = dev_status;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return with_dim16(dtype, head_dim, [&](auto td) {
        using TD = decltype(td);
        return launch_window_step<typename TD::T, TD::D>(a, batch, st);
    });
}

// --------------------------------------------------------------------------
// kvc_gqa_decode_noalloc: the same decode for callers that cannot allocate
// device memory themselves.  Its split partials live in one file-scope device
// array of KVC_DECODE_STATIC_SCRATCH_BYTES; the module holds that array on
// every device that loads the library until the process exits.
// --------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[KVC_DECODE_STATIC_SCRATCH_BYTES];

std::mutex g_scratch_mutex;
void *g_scratch_addr[256] = {};  // device address of g_decode_scratch, per device ordinal

// Host code may not pass g_decode_scratch itself to a kernel (on the host it
// names a stand-in, not device memory); the device address is looked up once
// per device, with that device current.
kvc_status scratch_address(void **addr)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256)
        return KVC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
            return KVC_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return KVC_OK;
}

} // namespace

KVC_API kvc_status kvc_gqa_decode_noalloc(void *out, const void *q, const void *k_cache,
                                          const void *v_cache, kvc_lengths len, int batch,
                                          int q_heads, int kv_heads, int64_t capacity,
                                          int head_dim, int dtype, int local_window_size,
                                          float scale, const float *rope_cos,
                                          const float *rope_sin, int64_t rope_max_pos,
                                          int32_t *dev_status, void *stream)
{
    const size_t need =
        kvc_gqa_decode_workspace_size(batch, q_heads, kv_heads, capacity, head_dim, dtype);
    if (need > KVC_DECODE_STATIC_SCRATCH_BYTES)
        return KVC_ERR_WORKSPACE;
    void *scratch = nullptr;
    const kvc_status st = scratch_address(&scratch);
    if (st != KVC_OK)
        return st;
    return kvc_gqa_decode(out, q, k_cache, v_cache, len, batch, q_heads, kv_heads, capacity,
                          head_dim, dtype, local_window_size, scale, rope_cos, rope_sin,
                          rope_max_pos, scratch, KVC_DECODE_STATIC_SCRATCH_BYTES, dev_status,
                          stream);
}
