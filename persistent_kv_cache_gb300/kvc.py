"""Python binding of the C ABI in include/kvc.h (argument marshalling only).

Every function has the C entry point's name and forwards torch tensors as raw
pointers plus the current CUDA stream; all the work happens in libkvc.so's
kernels.  There is no CPU path: a missing library raises ``KvcLibraryMissing``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvc.so")

KVC_F32, KVC_BF16, KVC_F16 = 0, 1, 2
KVC_LINEAR, KVC_CIRCULAR = 0, 1
KVC_APPEND, KVC_COPY_BACK = 0, 1

KVC_OK = 0
STATUS_NAMES = {
    0: "KVC_OK", 1: "KVC_ERR_NULL", 2: "KVC_ERR_SHAPE", 3: "KVC_ERR_DTYPE", 4: "KVC_ERR_ALIGN",
    5: "KVC_ERR_UNSUPPORTED", 6: "KVC_ERR_CAPACITY", 7: "KVC_ERR_WINDOW",
    8: "KVC_ERR_WORKSPACE", 9: "KVC_ERR_CUDA",
}
# cache policies (the `windowed` argument)
KVC_CONTIGUOUS, KVC_WINDOWED, KVC_DRIFTING, KVC_RING = 0, 1, 2, 3
KVC_DEV_INDEX_OOB = 1
KVC_DEV_SEQLEN_RANGE = 2
KVC_DEV_CAPACITY = 4
KVC_DEV_ROPE_RANGE = 8
KVC_DEV_TIMEOUT = 16

EXPORTS = ("kvc_tensor_scatter", "kvc_seq_lengths", "kvc_window_append", "kvc_gqa_decode",
           "kvc_gqa_decode_workspace_size", "kvc_gqa_decode_noalloc", "kvc_gqa_decode_ring",
           "kvc_decode_step", "kvc_decode_step_workspace_size", "kvc_window_decode_step",
           "kvc_window_decode_step_workspace_size",
           "kvc_paged_append", "kvc_gqa_decode_paged", "kvc_window_append_inplace",
           "kvc_quantize_pages", "kvc_gqa_decode_paged_q",
           "kvc_gqa_prefill_chunk", "kvc_gqa_prefill_workspace_size", "kvc_window_prefill_step",
           "kvc_status_string", "kvc_abi_version")
KVC_DECODE_STATIC_SCRATCH_BYTES = 16 << 20
KVC_PAGE_QUANT = 0x40000000  # block-table flag: the entry names an int8 page


class KvcLibraryMissing(RuntimeError):
    pass


class KvcError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}")


class KvcLengths(ctypes.Structure):
    _fields_ = [("past_abs", ctypes.c_void_p), ("total_abs", ctypes.c_void_p),
                ("cache_past", ctypes.c_void_p), ("cache_total", ctypes.c_void_p),
                ("evict", ctypes.c_void_p)]


class Lengths:
    """Five int32 device tensors of [batch] (past_abs, total_abs, cache_past,
    cache_total, evict) written by kvc_seq_lengths."""

    FIELDS = ("past_abs", "total_abs", "cache_past", "cache_total", "evict")

    def __init__(self, batch: int, device):
        self.buf = torch.empty((5, batch), dtype=torch.int32, device=device)
        self._c = KvcLengths(*[self.buf[i].data_ptr() for i in range(5)])

    def __getattr__(self, name):
        if name in Lengths.FIELDS:
            return self.buf[Lengths.FIELDS.index(name)]
        raise AttributeError(name)

    def c(self) -> KvcLengths:
        return self._c


_lib = None


def library() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise KvcLibraryMissing(
                f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, I64, F, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                            ctypes.c_size_t)
        L = KvcLengths
        sig = {
            "kvc_tensor_scatter": [P, P, P, P, I, P, I64, I, I, I, P, P],
            "kvc_seq_lengths": [P, I, I, I64, I, I, L, P, P],
            "kvc_window_append": [P, P, P, P, P, P, L, I, I, I, I64, I, I, I, I, P, P, I64, P, P],
            "kvc_window_append_inplace": [P, P, P, P, L, I, I, I, I64, I64, I, I, I, I, P, P, I64,
                                          P, P],
            "kvc_gqa_decode": [P, P, P, P, L, I, I, I, I64, I, I, I, F, P, P, I64, P, SZ, P, P],
            "kvc_gqa_decode_ring": [P, P, P, P, L, I, I, I, I64, I, I, I, F, P, P, I64, P, SZ, P,
                                    P],
            "kvc_gqa_decode_workspace_size": [I, I, I, I64, I, I],
            "kvc_paged_append": [P, P, P, P, P, I, I64, I, L, I, I, I, I, I, P, P, I64, P, P],
            "kvc_gqa_decode_paged": [P, P, P, P, P, I, I64, I, L, I, I, I, I, I, I, F, P, P, I64,
                                     P, SZ, P, P],
            "kvc_quantize_pages": [P, P, P, P, P, P, I, I64, I64, I, I, I, I, F, I, I, F, I, I, P,
                                   P, P],
            "kvc_gqa_decode_paged_q": [P, P, P, P, P, P, P, I64, P, I, I64, I, L, I, I, I, I, I, I,
                                       F, P, P, I64, P, SZ, P, P],
            "kvc_decode_step": [P, P, P, P, P, P, P, L, I, I, I, I64, I, I, I, I, F, P, P, I64, P,
                                SZ, P, P],
            "kvc_decode_step_workspace_size": [I, I, I, I64, I, I],
            "kvc_gqa_decode_noalloc": [P, P, P, P, L, I, I, I, I64, I, I, I, F, P, P, I64, P, P],
            "kvc_window_decode_step": [P, P, P, P, P, P, P, L, I, I, I, I64, I, I, I, I, F, P, P,
                                       I64, P, SZ, P, P],
            "kvc_window_decode_step_workspace_size": [I, I, I, I64, I, I],
            "kvc_gqa_prefill_chunk": [P, P, P, P, I64, L, I, I, I, I, I, I, I, F, P, P, I64, P, SZ,
                                      P, P],
            "kvc_gqa_prefill_workspace_size": [I, I, I, I, I64, I, I, I],
            "kvc_window_prefill_step": [P, P, P, P, P, P, P, P, L, I, I, I, I, I64, I, I, I, I,
                                        F, P, P, I64, P, SZ, P, P],
            "kvc_status_string": [I],
            "kvc_abi_version": [],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = I
        lib.kvc_gqa_decode_workspace_size.restype = SZ
        lib.kvc_decode_step_workspace_size.restype = SZ
        lib.kvc_window_decode_step_workspace_size.restype = SZ
        lib.kvc_gqa_prefill_workspace_size.restype = SZ
        lib.kvc_status_string.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def _ptr(t):
    """Device address of a tensor the library reads or writes as a dense
    array: it must live on a CUDA device and be contiguous (a strided view
    would be read in the wrong order, or past its storage)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got one on {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"expected a contiguous tensor, got shape {tuple(t.shape)} "
                         f"with strides {t.stride()}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _dtype_code(t: torch.Tensor) -> int:
    return {torch.float32: KVC_F32, torch.bfloat16: KVC_BF16, torch.float16: KVC_F16}[t.dtype]


def _check(fn: str, status: int):
    if status != KVC_OK:
        raise KvcError(fn, status)


def _rope(rope):
    if rope is None:
        return None, None, 0
    cos, sin = rope
    if cos.dtype != torch.float32 or sin.dtype != torch.float32 or cos.shape != sin.shape:
        raise ValueError("rope: cos and sin are float32 tables of the same shape [max_pos, D/2]")
    return _ptr(cos), _ptr(sin), cos.shape[0]


def kvc_tensor_scatter(present, past, update, write_indices=None, axis=-2, mode=KVC_LINEAR,
                       status=None, stream=None):
    shape = (ctypes.c_int64 * past.dim())(*past.shape)
    seq_axis = axis if axis >= 0 else axis + past.dim()
    _check("kvc_tensor_scatter", library().kvc_tensor_scatter(
        _ptr(present), _ptr(past), _ptr(update), _ptr(write_indices), past.dim(), shape,
        update.shape[seq_axis], axis, mode, past.element_size(), _ptr(status), _stream(stream)))
    return present


def kvc_seq_lengths(seqlens_k, new_tokens, capacity, windowed, local_window_size=0, out=None,
                    status=None, stream=None):
    out = Lengths(seqlens_k.shape[0], seqlens_k.device) if out is None else out
    _check("kvc_seq_lengths", library().kvc_seq_lengths(
        _ptr(seqlens_k), seqlens_k.shape[0], new_tokens, capacity, int(windowed),
        local_window_size, out.c(), _ptr(status), _stream(stream)))
    return out


def kvc_window_append(k_cache, v_cache, new_k, new_v, lengths, windowed, phase=KVC_APPEND,
                      k_stage=None, v_stage=None, rope=None, status=None, stream=None):
    B, Hkv, C, D = k_cache.shape
    S = new_k.shape[2] if new_k is not None else (k_stage.shape[2] - C)
    cs, sn, rmax = _rope(rope)
    _check("kvc_window_append", library().kvc_window_append(
        _ptr(k_cache), _ptr(v_cache), _ptr(new_k), _ptr(new_v), _ptr(k_stage), _ptr(v_stage),
        lengths.c(), B, Hkv, S, C, D, _dtype_code(k_cache), int(windowed), phase, cs, sn, rmax,
        _ptr(status), _stream(stream)))


def kvc_window_append_inplace(k_rows, v_rows, new_k, new_v, lengths, capacity, windowed,
                              phase=KVC_APPEND, new_tokens=None, rope=None, status=None,
                              stream=None):
    """k_rows/v_rows: [B, Hkv, rows_per_head, D] with rows_per_head >= capacity + S; the
    cache lives in rows [0, Lp).  new_tokens is needed when new_k is None (KVC_COPY_BACK)."""
    B, Hkv, R, D = k_rows.shape
    S = new_k.shape[2] if new_k is not None else int(new_tokens)
    cs, sn, rmax = _rope(rope)
    _check("kvc_window_append_inplace", library().kvc_window_append_inplace(
        _ptr(k_rows), _ptr(v_rows), _ptr(new_k), _ptr(new_v), lengths.c(), B, Hkv, S, capacity, R,
        D, _dtype_code(k_rows), int(windowed), phase, cs, sn, rmax, _ptr(status),
        _stream(stream)))


def kvc_gqa_decode_workspace_size(batch, q_heads, kv_heads, capacity, head_dim, dtype):
    return library().kvc_gqa_decode_workspace_size(batch, q_heads, kv_heads, capacity, head_dim,
                                                   dtype)


def decode_workspace(q, k_cache):
    B, Hq, _, D = q.shape
    n = kvc_gqa_decode_workspace_size(B, Hq, k_cache.shape[1], k_cache.shape[2], D,
                                      _dtype_code(q))
    return torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)


def kvc_gqa_decode(out, q, k_cache, v_cache, lengths, local_window_size=0, scale=0.0, rope=None,
                   workspace=None, status=None, stream=None):
    B, Hq, _, D = q.shape
    _, Hkv, C, _ = k_cache.shape
    ws = decode_workspace(q, k_cache) if workspace is None else workspace
    cs, sn, rmax = _rope(rope)
    _check("kvc_gqa_decode", library().kvc_gqa_decode(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), lengths.c(), B, Hq, Hkv, C, D,
        _dtype_code(q), local_window_size, scale, cs, sn, rmax, _ptr(ws), ws.numel(),
        _ptr(status), _stream(stream)))
    return out


def kvc_gqa_decode_ring(out, q, k_cache, v_cache, lengths, local_window_size=0, scale=0.0,
                        rope=None, workspace=None, status=None, stream=None):
    """kvc_gqa_decode over a ring of C slots (include/kvc.h)."""
    B, Hq, _, D = q.shape
    _, Hkv, C, _ = k_cache.shape
    ws = decode_workspace(q, k_cache) if workspace is None else workspace
    cs, sn, rmax = _rope(rope)
    _check("kvc_gqa_decode_ring", library().kvc_gqa_decode_ring(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), lengths.c(), B, Hq, Hkv, C, D,
        _dtype_code(q), local_window_size, scale, cs, sn, rmax, _ptr(ws), ws.numel(),
        _ptr(status), _stream(stream)))
    return out


def kvc_paged_append(k_pool, v_pool, new_k, new_v, block_table, lengths, rope=None, status=None,
                     stream=None):
    """Append on a paged cache: pools [pages, Hkv, page_size, D], block_table
    int32 [B, max_pages] (include/kvc.h)."""
    n_pages, Hkv, ps, D = k_pool.shape
    B, _, S, _ = new_k.shape
    cs, sn, rmax = _rope(rope)
    _check("kvc_paged_append", library().kvc_paged_append(
        _ptr(k_pool), _ptr(v_pool), _ptr(new_k), _ptr(new_v), _ptr(block_table),
        block_table.shape[1], n_pages, ps, lengths.c(), B, Hkv, S, D, _dtype_code(k_pool), cs,
        sn, rmax, _ptr(status), _stream(stream)))


def kvc_quantize_pages(k_pool, v_pool, qk_pool, qv_pool, src_pages, dst_pages, qparams, k_scale,
                       k_zero_point=0, k_unsigned=False, v_scale=None, v_zero_point=None,
                       v_unsigned=None, status=None, stream=None):
    """Int8 pages dst_pages[i] <- 16-bit pages src_pages[i] (include/kvc.h); V takes K's
    format unless given its own."""
    n_pool, Hkv, ps, D = k_pool.shape
    v_scale = k_scale if v_scale is None else v_scale
    v_zero_point = k_zero_point if v_zero_point is None else v_zero_point
    v_unsigned = k_unsigned if v_unsigned is None else v_unsigned
    _check("kvc_quantize_pages", library().kvc_quantize_pages(
        _ptr(k_pool), _ptr(v_pool), _ptr(qk_pool), _ptr(qv_pool), _ptr(src_pages),
        _ptr(dst_pages), src_pages.numel(), n_pool, qk_pool.shape[0], ps, Hkv, D,
        _dtype_code(k_pool), float(k_scale), int(k_zero_point), int(bool(k_unsigned)),
        float(v_scale), int(v_zero_point), int(bool(v_unsigned)), _ptr(qparams), _ptr(status),
        _stream(stream)))


def kvc_gqa_decode_paged_q(out, q, k_pool, v_pool, qk_pool, qv_pool, qparams, block_table,
                           lengths, local_window_size=0, scale=0.0, rope=None, workspace=None,
                           status=None, stream=None):
    """kvc_gqa_decode_paged over 16-bit and int8 pages (include/kvc.h)."""
    B, Hq, _, D = q.shape
    n_pages, Hkv, ps, _ = k_pool.shape
    max_pages = block_table.shape[1]
    if workspace is None:
        n = kvc_gqa_decode_workspace_size(B, Hq, Hkv, max_pages * ps, D, _dtype_code(q))
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    cs, sn, rmax = _rope(rope)
    _check("kvc_gqa_decode_paged_q", library().kvc_gqa_decode_paged_q(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(qk_pool), _ptr(qv_pool),
        _ptr(qparams), qk_pool.shape[0], _ptr(block_table), max_pages, n_pages, ps, lengths.c(),
        B, Hq, Hkv, D, _dtype_code(q), local_window_size, scale, cs, sn, rmax, _ptr(workspace),
        workspace.numel(), _ptr(status), _stream(stream)))
    return out


def kvc_gqa_decode_paged(out, q, k_pool, v_pool, block_table, lengths, local_window_size=0,
                         scale=0.0, rope=None, workspace=None, status=None, stream=None):
    """kvc_gqa_decode over a paged cache (include/kvc.h)."""
    B, Hq, _, D = q.shape
    n_pages, Hkv, ps, _ = k_pool.shape
    max_pages = block_table.shape[1]
    if workspace is None:
        n = kvc_gqa_decode_workspace_size(B, Hq, Hkv, max_pages * ps, D, _dtype_code(q))
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    cs, sn, rmax = _rope(rope)
    _check("kvc_gqa_decode_paged", library().kvc_gqa_decode_paged(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table), max_pages, n_pages,
        ps, lengths.c(), B, Hq, Hkv, D, _dtype_code(q), local_window_size, scale, cs, sn, rmax,
        _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream)))
    return out


def kvc_gqa_decode_noalloc(out, q, k_cache, v_cache, lengths, local_window_size=0, scale=0.0,
                           rope=None, status=None, stream=None):
    """kvc_gqa_decode with the library's own scratch (see include/kvc.h)."""
    B, Hq, _, D = q.shape
    _, Hkv, C, _ = k_cache.shape
    cs, sn, rmax = _rope(rope)
    _check("kvc_gqa_decode_noalloc", library().kvc_gqa_decode_noalloc(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), lengths.c(), B, Hq, Hkv, C, D,
        _dtype_code(q), local_window_size, scale, cs, sn, rmax, _ptr(status), _stream(stream)))
    return out


def decode_step_workspace(q, k_cache):
    """Workspace for kvc_decode_step (the split partials)."""
    B, Hq, _, D = q.shape
    n = library().kvc_decode_step_workspace_size(B, Hq, k_cache.shape[1], k_cache.shape[2], D,
                                                 _dtype_code(q))
    return torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)


def kvc_decode_step(out, q, k_cache, v_cache, new_k, new_v, seqlens_k, local_window_size=0,
                    lengths=None, scale=0.0, rope=None, workspace=None, status=None, stream=None,
                    windowed=None):
    """Fused lengths + one-token append + split decode on a contiguous cache
    (default) or a ring (windowed=KVC_RING); include/kvc.h."""
    windowed = KVC_CONTIGUOUS if windowed is None else int(windowed)
    B, Hq, _, D = q.shape
    _, Hkv, C, _ = k_cache.shape
    ws = decode_step_workspace(q, k_cache) if workspace is None else workspace
    cs, sn, rmax = _rope(rope)
    lc = lengths.c() if lengths is not None else KvcLengths(None, None, None, None, None)
    _check("kvc_decode_step", library().kvc_decode_step(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(new_k), _ptr(new_v),
        _ptr(seqlens_k), lc, B, Hq, Hkv, C, D, _dtype_code(q), windowed, local_window_size,
        scale, cs, sn, rmax, _ptr(ws), ws.numel(), _ptr(status), _stream(stream)))
    return out


def window_step_workspace(q, k_cache):
    """Workspace for kvc_window_decode_step (None for a window held on chip)."""
    B, Hq, _, D = q.shape
    n = library().kvc_window_decode_step_workspace_size(B, Hq, k_cache.shape[1],
                                                        k_cache.shape[2], D, _dtype_code(q))
    return torch.empty(n, dtype=torch.uint8, device=q.device) if n else None


def kvc_window_decode_step(out, q, k_cache, v_cache, new_k, new_v, seqlens_k, local_window_size,
                           lengths=None, scale=0.0, rope=None, status=None, stream=None,
                           windowed=None, workspace="auto"):
    """Lengths + windowed one-token append + GQA decode (include/kvc.h).
    ``windowed``: KVC_WINDOWED (default), KVC_DRIFTING or KVC_RING;
    ``workspace``: "auto" allocates what the call needs (large windows only)."""
    windowed = KVC_WINDOWED if windowed is None else int(windowed)
    B, Hq, _, D = q.shape
    _, Hkv, C, _ = k_cache.shape
    if isinstance(workspace, str):
        workspace = window_step_workspace(q, k_cache)
    cs, sn, rmax = _rope(rope)
    lc = lengths.c() if lengths is not None else KvcLengths(None, None, None, None, None)
    _check("kvc_window_decode_step", library().kvc_window_decode_step(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(new_k), _ptr(new_v),
        _ptr(seqlens_k), lc, B, Hq, Hkv, C, D, _dtype_code(q), windowed, local_window_size,
        scale, cs, sn, rmax, _ptr(workspace), 0 if workspace is None else workspace.numel(),
        _ptr(status), _stream(stream)))
    return out


def prefill_workspace(q, k_rows, local_window_size=0):
    """Workspace for kvc_gqa_prefill_chunk's KV split (None when it would
    not split)."""
    B, Hq, S, D = q.shape
    _, Hkv, R, _ = k_rows.shape
    n = library().kvc_gqa_prefill_workspace_size(B, Hq, Hkv, S, R, D, _dtype_code(q),
                                                 local_window_size)
    return torch.empty(n, dtype=torch.uint8, device=q.device) if n else None


def kvc_gqa_prefill_chunk(out, q, k_rows, v_rows, lengths, local_window_size=0, scale=0.0,
                          rope=None, status=None, stream=None, workspace="auto"):
    """workspace: "auto" allocates what the call can use, None runs unsplit."""
    B, Hq, S, D = q.shape
    _, Hkv, R, _ = k_rows.shape
    if isinstance(workspace, str):
        workspace = prefill_workspace(q, k_rows, local_window_size)
    cs, sn, rmax = _rope(rope)
    _check("kvc_gqa_prefill_chunk", library().kvc_gqa_prefill_chunk(
        _ptr(out), _ptr(q), _ptr(k_rows), _ptr(v_rows), R, lengths.c(), B, Hq, Hkv, S, D,
        _dtype_code(q), local_window_size, scale, cs, sn, rmax, _ptr(workspace),
        0 if workspace is None else workspace.numel(), _ptr(status), _stream(stream)))
    return out


def kvc_status_string(code: int) -> str:
    return library().kvc_status_string(code).decode()


def kvc_abi_version() -> int:
    return library().kvc_abi_version()


def kvc_window_prefill_step(out, q, k_cache, v_cache, new_k, new_v, lengths, windowed,
                            local_window_size, k_stage=None, v_stage=None, scale=0.0, rope=None,
                            status=None, stream=None, workspace="auto"):
    """One windowed S-token step that stages only the rows whose eviction its
    chunk would see (include/kvc.h).  k_stage/v_stage: [B, Hkv, C + S, D]
    (needed for S > 1).  workspace: "auto" allocates what the attention can
    use, None runs it unsplit."""
    B, Hq, S, D = q.shape
    _, Hkv, C, _ = k_cache.shape
    if isinstance(workspace, str):
        n = library().kvc_gqa_prefill_workspace_size(B, Hq, Hkv, S, C, D, _dtype_code(q),
                                                     local_window_size)
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device) if n else None
    cs, sn, rmax = _rope(rope)
    _check("kvc_window_prefill_step", library().kvc_window_prefill_step(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(new_k), _ptr(new_v),
        _ptr(k_stage), _ptr(v_stage), lengths.c(), B, Hq, Hkv, S, C, D, _dtype_code(q),
        int(windowed), local_window_size, scale, cs, sn, rmax, _ptr(workspace),
        0 if workspace is None else workspace.numel(), _ptr(status), _stream(stream)))
    return out
