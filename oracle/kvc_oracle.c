/*
 * kvc_oracle.c -- plain, slow CPU oracle for the persistent KV-cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the test suite, the package smoke check and the
 * benchmark's CPU-baseline / reference arm do.  It shares no code, header,
 * table or constant with the CUDA library: every rule below is restated from
 * the source pages in the simplest form that can be checked by eye.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared -o liboracle.so kvc_oracle.c -lm
 * (-ffp-contract=off keeps every float multiply and add separately rounded,
 * which the bit-exact RoPE rows rely on.)
 *
 * Sources (page title, section):
 *   [TS]  "TensorScatter" operator page (ai.onnx, since version 24): the spec
 *         text, its pseudocode and its three worked examples.
 *   [GQA] "GQA support sliding_window_cache" (onnxruntime pull request 29904):
 *         section "Design" (windowed-cache invariant and append formula,
 *         staging cache for S > 1, device-side lengths from seqlens_k) and the
 *         follow-up commits (int64 widening of seqlens_k + 1, absolute-position
 *         RoPE bounded by the cos/sin cache length).
 *   [RM]  "Persistent KV Cache and Decode Performance Roadmap", section
 *         "Phase 1: decode with contiguous KV cache" (what decode attention
 *         computes; GQA heads share one KV head).
 *   [SW]  "Stateful decode & KV cache", section "Sliding-window ring buffer"
 *         (RoPE baked into K at write time; mask from positions only).
 *
 * Parity pins for each function live in tests/test_oracle_*.py.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>
#include <stdlib.h>

/* element types, numbered for this file only */
#define ORC_F32 0
#define ORC_BF16 1
#define ORC_F16 2

/* per-batch-row flags written by the oracle (its own numbering) */
#define ORC_BAD_INDEX 1   /* TensorScatter linear: write_indices out of range   */
#define ORC_BAD_SEQLEN 2  /* seqlens_k + 1 < S, or does not fit in int32        */
#define ORC_BAD_CAPACITY 4 /* contiguous cache: total length > capacity         */
#define ORC_BAD_ROPE 8    /* a RoPE position is outside the cos/sin cache       */

/* ------------------------------------------------------------------ */
/* element conversions                                                  */
/* ------------------------------------------------------------------ */

/* bfloat16 is the upper half of an IEEE binary32. */
static float bf16_bits_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* binary32 -> bfloat16, round to nearest, ties to even (NaN stays NaN). */
static uint16_t float_to_bf16_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16;
    uint32_t rest = u & 0xffffu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))
        keep += 1u;
    return (uint16_t)keep;
}

static double load_elem(const void *base, int64_t i, int dtype)
{
    if (dtype == ORC_F32)
        return (double)((const float *)base)[i];
    if (dtype == ORC_BF16)
        return (double)bf16_bits_to_float(((const uint16_t *)base)[i]);
    return (double)((const _Float16 *)base)[i];
}

static float load_elem_f32(const void *base, int64_t i, int dtype)
{
    if (dtype == ORC_F32)
        return ((const float *)base)[i];
    if (dtype == ORC_BF16)
        return bf16_bits_to_float(((const uint16_t *)base)[i]);
    return (float)((const _Float16 *)base)[i];
}

/* store a float32 value, rounding to nearest-even into the element type */
static void store_elem_f32(void *base, int64_t i, int dtype, float v)
{
    if (dtype == ORC_F32)
        ((float *)base)[i] = v;
    else if (dtype == ORC_BF16)
        ((uint16_t *)base)[i] = float_to_bf16_bits(v);
    else
        ((_Float16 *)base)[i] = (_Float16)v;
}

/* store a double rounded to the element type; bfloat16 goes through binary32
 * (a double rounding that can move a tie by one bfloat16 ulp, far inside the
 * attention tolerance) */
static void store_elem_f64(void *base, int64_t i, int dtype, double v)
{
    if (dtype == ORC_F32)
        ((float *)base)[i] = (float)v;
    else if (dtype == ORC_BF16)
        ((uint16_t *)base)[i] = float_to_bf16_bits((float)v);
    else
        ((_Float16 *)base)[i] = (_Float16)v;
}

static int elem_size(int dtype) { return dtype == ORC_F32 ? 4 : 2; }

/* ------------------------------------------------------------------ */
/* [TS] TensorScatter                                                   */
/* ------------------------------------------------------------------ */

static int64_t floor_mod(int64_t a, int64_t m)
{
    int64_t r = a % m;
    return r < 0 ? r + m : r;
}

/*
 * present = past, then for every prefix index (the dimensions before `axis`,
 * enumerated in row-major order, whose first component is the batch index b)
 * and every s in [0, seq_len): the trailing slice of `update` at
 * (prefix, s) is written to the trailing slice of `present` at
 * (prefix, write_indices[b] + s).  In circular mode the sequence index is
 * taken modulo max_sequence_length (shape[axis]); only the sequence component
 * is reduced.  Linear mode requires 0 <= wi and wi + seq_len <= max_seq; a
 * batch row that breaks this is left equal to `past` and flagged.
 * The update's sequence length may not exceed max_sequence_length (a shape
 * rule of the operator).
 * Returns 0, or -1 for an argument the operator does not define.
 */
int orc_tensor_scatter(void *present, const void *past, const void *update,
                       const int64_t *write_indices, int rank, const int64_t *shape,
                       int64_t seq_len, int axis, int mode, int elem_bytes,
                       int32_t *batch_flags)
{
    if (rank < 2 || elem_bytes <= 0 || seq_len < 0)
        return -1;
    if (axis < 0)
        axis += rank;
    if (axis <= 0 || axis >= rank)
        return -1;
    if (seq_len > shape[axis])
        return -1;

    int64_t n_elems = 1;
    for (int d = 0; d < rank; ++d)
        n_elems *= shape[d];
    int64_t max_seq = shape[axis];
    int64_t slice_bytes = elem_bytes;
    for (int d = axis + 1; d < rank; ++d)
        slice_bytes *= shape[d];
    int64_t n_prefix = 1;
    for (int d = 0; d < axis; ++d)
        n_prefix *= shape[d];
    int64_t batch = shape[0];
    int64_t prefixes_per_batch = batch > 0 ? n_prefix / batch : 0;

    if (present != past)
        memcpy(present, past, (size_t)(n_elems * elem_bytes));

    for (int64_t b = 0; b < batch; ++b) {
        int64_t wi = write_indices ? write_indices[b] : 0;
        batch_flags[b] = 0;
        if (mode == 0 && (wi < 0 || wi + seq_len > max_seq))
            batch_flags[b] = ORC_BAD_INDEX;
    }
    if (max_seq == 0)
        return 0;

    for (int64_t p = 0; p < n_prefix; ++p) {
        int64_t b = p / prefixes_per_batch;
        if (batch_flags[b])
            continue;
        int64_t wi = write_indices ? write_indices[b] : 0;
        for (int64_t s = 0; s < seq_len; ++s) {
            int64_t idx = wi + s;
            if (mode == 1)
                idx = floor_mod(idx, max_seq);
            char *dst = (char *)present + (p * max_seq + idx) * slice_bytes;
            const char *src = (const char *)update + (p * seq_len + s) * slice_bytes;
            memcpy(dst, src, (size_t)slice_bytes);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* [GQA] sequence lengths derived from seqlens_k                        */
/* ------------------------------------------------------------------ */

/*
 * [GQA] CPU commit "drifting layout": with gap = C - W + 1 the resident rows
 * of a windowed cache are [0, end(T)) where
 *     end(T) = T                              while T <= C
 *            = T - gap * ceil((T - C) / gap)  afterwards  (so W <= end <= C)
 * a pure function of the absolute length, so compaction happens once every
 * gap steps instead of every step.
 */
static int64_t drift_end(int64_t T, int64_t C, int64_t W)
{
    if (T <= C)
        return T;
    int64_t gap = C - W + 1;
    int64_t k = (T - C + gap - 1) / gap;
    return T - gap * k;
}

/*
 * seqlens_k[b] holds the running total after this step minus one, so the
 * absolute total is T = seqlens_k[b] + 1 (computed in 64-bit) and the absolute
 * past length is P = T - S.  Windowed cache of capacity C (policy 1):
 *     Lp = min(P, C)          resident tokens before the step
 *     E  = max(0, Lp + S - C) tokens evicted by the step
 *     L  = Lp - E + S         resident tokens after the step
 * Drifting windowed cache (policy 2, window W): Lp = end(P), L = end(T),
 * E = Lp + S - L.
 * Contiguous cache (policy 0): Lp = P, E = 0, L = T, and T must not exceed C.
 * A row is rejected (all five outputs -1, flag set) when T < S, when T does
 * not fit in int32, (contiguous) when T > C, or (drifting) when W is outside
 * [1, C].
 */
void orc_seq_lengths(const int32_t *seqlens_k, int batch, int new_tokens,
                     int64_t capacity, int windowed, int window, int32_t *past_abs,
                     int32_t *total_abs, int32_t *cache_past, int32_t *cache_total,
                     int32_t *evict, int32_t *batch_flags)
{
    for (int b = 0; b < batch; ++b) {
        int64_t T = (int64_t)seqlens_k[b] + 1;
        int64_t S = new_tokens;
        int flag = 0;
        if (T < S || T > INT32_MAX)
            flag |= ORC_BAD_SEQLEN;
        else if (!windowed && T > capacity)
            flag |= ORC_BAD_CAPACITY;
        else if (windowed == 2 && (window < 1 || window > capacity))
            flag |= ORC_BAD_CAPACITY;   /* the layout needs W <= C */
        batch_flags[b] = flag;
        if (flag) {
            past_abs[b] = total_abs[b] = cache_past[b] = cache_total[b] = evict[b] = -1;
            continue;
        }
        int64_t P = T - S;
        int64_t Lp, E, L;
        if (windowed == 2) {
            Lp = drift_end(P, capacity, window);
            L = drift_end(T, capacity, window);
            E = Lp + S - L;
        } else if (windowed) {
            Lp = P < capacity ? P : capacity;
            E = Lp + S - capacity;
            if (E < 0)
                E = 0;
            L = Lp - E + S;
        } else {
            Lp = P;
            E = 0;
            L = T;
        }
        past_abs[b] = (int32_t)P;
        total_abs[b] = (int32_t)T;
        cache_past[b] = (int32_t)Lp;
        cache_total[b] = (int32_t)L;
        evict[b] = (int32_t)E;
    }
}

/* ------------------------------------------------------------------ */
/* RoPE (rotate-half pairs (i, i + D/2)), float32, no contraction       */
/* ------------------------------------------------------------------ */

/*
 * Rotates one row x[0..D) in place for the angle whose cosine/sine row is
 * given (the cos/sin caches are inputs of the operator, indexed by the
 * ABSOLUTE position).  Each product and each sum is rounded to binary32:
 *     lo' = (lo*c) - (hi*s),   hi' = (hi*c) + (lo*s).
 */
static void rope_rotate_f32(float *x, int D, const float *c_row, const float *s_row)
{
    int half = D / 2;
    for (int i = 0; i < half; ++i) {
        float lo = x[i];
        float hi = x[i + half];
        float c = c_row[i];
        float s = s_row[i];
        float lo_c = lo * c;
        float hi_s = hi * s;
        float hi_c = hi * c;
        float lo_s = lo * s;
        x[i] = lo_c - hi_s;
        x[i + half] = hi_c + lo_s;
    }
}

/* Exposed for the RoPE pins: rotate `n_rows` rows of width D, row r at
 * position pos[r]; input and output in `dtype`. Returns -1 if a position is
 * outside [0, rope_max_pos). */
int orc_rope_rows(void *out, const void *in, const int64_t *pos, int64_t n_rows, int D,
                  int dtype, const float *cos_cache, const float *sin_cache,
                  int64_t rope_max_pos)
{
    float *row = (float *)malloc(sizeof(float) * (size_t)D);
    int rc = 0;
    for (int64_t r = 0; r < n_rows; ++r) {
        if (pos[r] < 0 || pos[r] >= rope_max_pos) {
            rc = -1;
            continue;
        }
        for (int d = 0; d < D; ++d)
            row[d] = load_elem_f32(in, r * D + d, dtype);
        rope_rotate_f32(row, D, cos_cache + pos[r] * (D / 2), sin_cache + pos[r] * (D / 2));
        for (int d = 0; d < D; ++d)
            store_elem_f32(out, r * D + d, dtype, row[d]);
    }
    free(row);
    return rc;
}

/* ------------------------------------------------------------------ */
/* [GQA] cache append: contiguous, windowed S == 1, windowed staging    */
/* ------------------------------------------------------------------ */

static void copy_row(void *dst, int64_t dst_row, const void *src, int64_t src_row,
                     int64_t row_bytes)
{
    memmove((char *)dst + dst_row * row_bytes, (const char *)src + src_row * row_bytes,
            (size_t)row_bytes);
}

/* the new K row i of (b, h), rotated at absolute position pos when tables
 * are given, written to dst row `dst_row` */
static void write_new_k(void *dst, int64_t dst_row, const void *new_k, int64_t src_row,
                        int D, int dtype, const float *cos_cache, const float *sin_cache,
                        int64_t pos, float *tmp)
{
    for (int d = 0; d < D; ++d)
        tmp[d] = load_elem_f32(new_k, src_row * D + d, dtype);
    if (cos_cache)
        rope_rotate_f32(tmp, D, cos_cache + pos * (D / 2), sin_cache + pos * (D / 2));
    for (int d = 0; d < D; ++d)
        store_elem_f32(dst, dst_row * D + d, dtype, tmp[d]);
}

/*
 * Appends S new tokens per (b, kv head).  Layouts: caches [B, Hkv, C, D],
 * new_k/new_v [B, Hkv, S, D], stages [B, Hkv, C + S, D].  The lengths are the
 * outputs of orc_seq_lengths (a row with cache_total < 0 is skipped).
 *
 * Contiguous cache: new token i goes to row P + i.
 * Windowed, S == 1 (in place): cache[E..Lp) -> cache[0..Lp-E), then the new
 *   token goes to row Lp - E.
 * Windowed, S > 1 (staging): stage[0..Lp) = cache[0..Lp),
 *   stage[Lp + i] = new token i, then cache[0..L) = stage[E..Lp+S).  The stage
 *   is left holding the seeded rows, which is what the chunk's attention reads.
 * K rows are rotated at absolute position P + i; V rows are copied as is.
 * A row whose last position P + S - 1 is not below rope_max_pos is flagged and
 * left unchanged.
 */
int orc_window_append(void *k_cache, void *v_cache, const void *new_k, const void *new_v,
                      void *k_stage, void *v_stage, const int32_t *past_abs,
                      const int32_t *cache_past, const int32_t *cache_total,
                      const int32_t *evict, int batch, int kv_heads, int new_tokens,
                      int64_t capacity, int head_dim, int dtype, int windowed,
                      const float *cos_cache, const float *sin_cache, int64_t rope_max_pos,
                      int32_t *batch_flags)
{
    int D = head_dim;
    int64_t S = new_tokens;
    int64_t C = capacity;
    int64_t row_bytes = (int64_t)D * elem_size(dtype);
    if (windowed && S > 1 && (!k_stage || !v_stage))
        return -1;
    float *tmp = (float *)malloc(sizeof(float) * (size_t)D);

    for (int b = 0; b < batch; ++b) {
        batch_flags[b] = 0;
        if (cache_total[b] < 0)
            continue;
        int64_t P = past_abs[b], Lp = cache_past[b], E = evict[b], L = cache_total[b];
        if (cos_cache && P + S > rope_max_pos) {
            batch_flags[b] = ORC_BAD_ROPE;
            continue;
        }
        for (int h = 0; h < kv_heads; ++h) {
            int64_t slice = (int64_t)b * kv_heads + h;
            int64_t cbase = slice * C;          /* first cache row of (b, h) */
            int64_t nbase = slice * S;          /* first new row of (b, h)   */
            if (!windowed) {
                for (int64_t i = 0; i < S; ++i) {
                    write_new_k(k_cache, cbase + P + i, new_k, nbase + i, D, dtype,
                                cos_cache, sin_cache, P + i, tmp);
                    copy_row(v_cache, cbase + P + i, new_v, nbase + i, row_bytes);
                }
            } else if (S == 1) {
                for (int64_t r = E; r < Lp; ++r) {
                    copy_row(k_cache, cbase + r - E, k_cache, cbase + r, row_bytes);
                    copy_row(v_cache, cbase + r - E, v_cache, cbase + r, row_bytes);
                }
                write_new_k(k_cache, cbase + Lp - E, new_k, nbase, D, dtype, cos_cache,
                            sin_cache, P, tmp);
                copy_row(v_cache, cbase + Lp - E, new_v, nbase, row_bytes);
            } else {
                int64_t sbase = slice * (C + S); /* first stage row of (b, h) */
                for (int64_t r = 0; r < Lp; ++r) {
                    copy_row(k_stage, sbase + r, k_cache, cbase + r, row_bytes);
                    copy_row(v_stage, sbase + r, v_cache, cbase + r, row_bytes);
                }
                for (int64_t i = 0; i < S; ++i) {
                    write_new_k(k_stage, sbase + Lp + i, new_k, nbase + i, D, dtype,
                                cos_cache, sin_cache, P + i, tmp);
                    copy_row(v_stage, sbase + Lp + i, new_v, nbase + i, row_bytes);
                }
                for (int64_t r = 0; r < L; ++r) {
                    copy_row(k_cache, cbase + r, k_stage, sbase + E + r, row_bytes);
                    copy_row(v_cache, cbase + r, v_stage, sbase + E + r, row_bytes);
                }
            }
        }
    }
    free(tmp);
    return 0;
}

/* ------------------------------------------------------------------ */
/* [RM][GQA][SW] grouped-query attention over cached rows               */
/* ------------------------------------------------------------------ */

/*
 * q, out: [B, Hq, S, D].  k_rows, v_rows: [B, Hkv, rows_per_head, D].  For
 * batch b the first n_rows[b] rows of each head hold the most recent tokens,
 * contiguously, ending at absolute position T - 1 (T = total_abs[b]): row r
 * holds position T - n_rows[b] + r.  Query i holds position T - S + i.
 * Query head h reads KV head h / (Hq / Hkv).
 * Key at kpos is visible to the query at qpos iff kpos <= qpos and, when
 * window > 0, qpos - kpos < window.
 * The query row is rotated at its absolute position (double precision) when
 * cos/sin caches are given; K rows are used as stored.
 * Everything after loading is double precision: s_j = scale * sum_d q_d k_jd
 * over the visible rows in ascending position, m = max s, p_j = exp(s_j - m),
 * out = (sum_j p_j v_j) / (sum_j p_j), rounded to the output type (the
 * 16-bit types go through binary32 on the way).
 * A batch row with n_rows[b] < 0 is skipped (its output is not written).
 * Returns -1 on a shape it cannot describe.
 */
int orc_gqa_attention(void *out, const void *q, const void *k_rows, const void *v_rows,
                      int64_t rows_per_head, const int32_t *n_rows, const int32_t *total_abs,
                      int batch, int q_heads, int kv_heads, int new_tokens, int head_dim,
                      int dtype, int window, double scale, const float *cos_cache,
                      const float *sin_cache, int64_t rope_max_pos, int32_t *batch_flags)
{
    if (kv_heads <= 0 || q_heads % kv_heads != 0 || head_dim <= 0)
        return -1;
    int D = head_dim;
    int64_t S = new_tokens;
    int group = q_heads / kv_heads;
    double *qv = (double *)malloc(sizeof(double) * (size_t)D);
    double *acc = (double *)malloc(sizeof(double) * (size_t)D);
    double *sc = (double *)malloc(sizeof(double) * (size_t)(rows_per_head > 0 ? rows_per_head : 1));

    for (int b = 0; b < batch; ++b) {
        batch_flags[b] = 0;
        int64_t n = n_rows[b];
        if (n < 0)
            continue;
        int64_t T = total_abs[b];
        if (cos_cache && T > rope_max_pos) {
            batch_flags[b] = ORC_BAD_ROPE;
            continue;
        }
        int64_t first_pos = T - n;
        for (int h = 0; h < q_heads; ++h) {
            int kvh = h / group;
            int64_t kbase = ((int64_t)b * kv_heads + kvh) * rows_per_head;
            for (int64_t i = 0; i < S; ++i) {
                int64_t qrow = ((int64_t)b * q_heads + h) * S + i;
                int64_t qpos = T - S + i;
                for (int d = 0; d < D; ++d)
                    qv[d] = load_elem(q, qrow * D + d, dtype);
                if (cos_cache) {
                    int half = D / 2;
                    const float *cr = cos_cache + qpos * half;
                    const float *sr = sin_cache + qpos * half;
                    for (int d = 0; d < half; ++d) {
                        double lo = qv[d], hi = qv[d + half];
                        qv[d] = lo * (double)cr[d] - hi * (double)sr[d];
                        qv[d + half] = hi * (double)cr[d] + lo * (double)sr[d];
                    }
                }
                /* pass 1: scores of the visible rows, and their maximum */
                double m = -INFINITY;
                for (int64_t r = 0; r < n; ++r) {
                    int64_t kpos = first_pos + r;
                    int visible = kpos <= qpos && (window <= 0 || qpos - kpos < window);
                    if (!visible)
                        continue;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += qv[d] * load_elem(k_rows, (kbase + r) * D + d, dtype);
                    sc[r] = dot * scale;
                    if (sc[r] > m)
                        m = sc[r];
                }
                /* pass 2: normalised weighted sum of V */
                double l = 0.0;
                for (int d = 0; d < D; ++d)
                    acc[d] = 0.0;
                for (int64_t r = 0; r < n; ++r) {
                    int64_t kpos = first_pos + r;
                    int visible = kpos <= qpos && (window <= 0 || qpos - kpos < window);
                    if (!visible)
                        continue;
                    double p = exp(sc[r] - m);
                    l += p;
                    for (int d = 0; d < D; ++d)
                        acc[d] += p * load_elem(v_rows, (kbase + r) * D + d, dtype);
                }
                for (int d = 0; d < D; ++d)
                    store_elem_f64(out, qrow * D + d, dtype, l > 0.0 ? acc[d] / l : 0.0);
            }
        }
    }
    free(qv);
    free(acc);
    free(sc);
    return 0;
}
