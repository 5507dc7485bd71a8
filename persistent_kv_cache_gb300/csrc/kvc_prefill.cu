// kvc_prefill.cu -- attention of a multi-token chunk over staged rows
// ("GQA support sliding_window_cache", section "Design": a step with S > 1
// runs against the C + S staging cache; causal plus local-window mask on
// absolute positions, cache-relative row addressing).
#include "kvc_common.cuh"

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
    if (dtype != KVC_F32 || head_dim > 256)
        return KVC_ERR_UNSUPPORTED;
    if (batch == 0)
        return KVC_OK;
    if (!out || !q || !k_rows || !v_rows || !kvc_host::lengths_ok(len))
        return KVC_ERR_NULL;
    for (const void *p : {(const void *)out, q, k_rows, v_rows})
        if (!kvc_host::aligned16(p))
            return KVC_ERR_ALIGN;
    if (scale == 0.f)
        scale = 1.0f / sqrtf((float)head_dim);
    return kvc_f32::launch(out, q, k_rows, v_rows, rows_per_head, len, batch, q_heads, kv_heads,
                           new_tokens, head_dim, local_window_size, scale, rope_cos, rope_sin,
                           rope_max_pos, 1, dev_status, static_cast<cudaStream_t>(stream_));
}
