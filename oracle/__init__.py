"""CPU oracle for the persistent KV-cache hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import this package.  The product library never loads it
and shares no code with it (``kvc_oracle.c`` is compiled on its own with gcc).

Every function takes numpy arrays (16-bit floats travel as ``uint16`` bit
patterns) and returns numpy arrays; each one cites the page it restates:

* ``tensor_scatter``  -- "TensorScatter" operator page (opset 24), spec and
  pseudocode.
* ``seq_lengths``     -- "GQA support sliding_window_cache" (onnxruntime PR
  29904), section "Design" (lengths derived on device from ``seqlens_k``).
* ``window_append``   -- same PR, "Design": windowed invariant, append formula,
  in-place S == 1 compaction and C + S staging for S > 1.
* ``rope_rows``       -- same PR (absolute-position RoPE bounded by the cos/sin
  cache) and "Stateful decode & KV cache", "Sliding-window ring buffer" (RoPE
  baked into K at write time).
* ``gqa_attention``   -- "Persistent KV Cache and Decode Performance Roadmap",
  "Phase 1" (what decode attention computes, GQA sharing) with the causal and
  local-window mask of the PR.
* ``paged_rows``, ``paged_append``, ``paged_attention`` -- "Persistent KV
  Cache and Decode Performance Roadmap", "Phase 2" and the CPU backend's
  "fixed-size paged blocks and a page-table iterator": logical row r of batch
  row b lives in page block_table[b][r // P] at slot r % P of a shared page
  pool; attention over the logical rows is the plain attention above.
* ``ring_slot_positions``, ``ring_append``, ``ring_attention`` -- "Stateful
  decode & KV cache", "Sliding-window ring buffer": token p lives in slot
  p mod C (TensorScatter circular with write index P, K rotated at write
  time); attention lists the ring's slots in position order and is then the
  plain attention above.

* ``quantize_affine``, ``dequantize_affine``, ``quantize_page``,
  ``paged_attention_q`` -- "Persistent input/output feedback", "Optional
  heterogeneous paged KV" (selected-block quantization: affine codes with a
  scale and zero point per K or V block, ties to even, saturation to the
  code range, reconstruction (code - zero point) * scale) and the roadmap's
  "Phase 3: cache quantization and fusion" (cold pages quantized to INT8):
  attention over a paged cache whose pages are 16-bit or INT8 is the plain
  attention above over the reconstructed rows.

Pins: every function is checked in ``tests/test_oracle_*.py`` against the
pages' worked examples, closed forms, brute-force simulations and library
routines (see the docstrings there).  No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvc_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16, F16 = 0, 1, 2
LINEAR, CIRCULAR = 0, 1

# per-row flags (the oracle's own numbering, mirrored from kvc_oracle.c)
BAD_INDEX, BAD_SEQLEN, BAD_CAPACITY, BAD_ROPE = 1, 2, 4, 8


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with gcc (no contraction of float ops)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I32, I64, DBL = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.orc_tensor_scatter.argtypes = [P, P, P, P, I32, P, I64, I32, I32, I32, P]
        lib.orc_tensor_scatter.restype = I32
        lib.orc_seq_lengths.argtypes = [P, I32, I32, I64, I32, I32, P, P, P, P, P, P]
        lib.orc_seq_lengths.restype = None
        lib.orc_rope_rows.argtypes = [P, P, P, I64, I32, I32, P, P, I64]
        lib.orc_rope_rows.restype = I32
        lib.orc_window_append.argtypes = [P, P, P, P, P, P, P, P, P, P, I32, I32, I32, I64,
                                          I32, I32, I32, P, P, I64, P]
        lib.orc_window_append.restype = I32
        lib.orc_gqa_attention.argtypes = [P, P, P, P, I64, P, P, I32, I32, I32, I32, I32,
                                          I32, I32, DBL, P, P, I64, P]
        lib.orc_gqa_attention.restype = I32
        _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float16:
        return F16
    raise TypeError(f"unsupported element type {a.dtype}")


def tensor_scatter(past, update, write_indices, axis=-2, mode=LINEAR, out=None):
    """TensorScatter: returns (present, per-batch flags).  ``out is past`` runs
    in place.  Any element type: rows are copied as bytes."""
    past = np.ascontiguousarray(past)
    update = np.ascontiguousarray(update)
    present = np.empty_like(past) if out is None else out
    shape = np.asarray(past.shape, dtype=np.int64)
    wi = None if write_indices is None else np.ascontiguousarray(write_indices, dtype=np.int64)
    flags = np.zeros(past.shape[0], dtype=np.int32)
    seq_axis = axis if axis >= 0 else axis + past.ndim
    rc = _load().orc_tensor_scatter(_ptr(present), _ptr(past), _ptr(update), _ptr(wi),
                                    past.ndim, _ptr(shape), update.shape[seq_axis], axis,
                                    mode, past.itemsize, _ptr(flags))
    if rc != 0:
        raise ValueError("tensor_scatter: arguments outside the operator's definition")
    return present, flags


CONTIGUOUS, WINDOWED, DRIFTING, RING = 0, 1, 2, 3


def seq_lengths(seqlens_k, new_tokens, capacity, windowed, window=0):
    """Returns dict(past_abs, total_abs, cache_past, cache_total, evict, flags).
    windowed: 0 contiguous, 1 windowed (compact every step), 2 drifting
    (needs the window), 3 ring (a ring of C slots holds the last min(T, C)
    tokens, so its counts are the windowed ones)."""
    if int(windowed) == RING:
        windowed = WINDOWED
    sk = np.ascontiguousarray(seqlens_k, dtype=np.int32)
    B = sk.shape[0]
    outs = {k: np.zeros(B, dtype=np.int32) for k in
            ("past_abs", "total_abs", "cache_past", "cache_total", "evict", "flags")}
    _load().orc_seq_lengths(_ptr(sk), B, new_tokens, capacity, int(windowed), int(window),
                            _ptr(outs["past_abs"]), _ptr(outs["total_abs"]),
                            _ptr(outs["cache_past"]), _ptr(outs["cache_total"]),
                            _ptr(outs["evict"]), _ptr(outs["flags"]))
    return outs


def rope_rows(x, pos, cos_cache, sin_cache):
    """Rotate rows x[..., D] at the absolute positions ``pos`` (one per row)."""
    x = np.ascontiguousarray(x)
    D = x.shape[-1]
    n = x.size // D
    pos = np.ascontiguousarray(pos, dtype=np.int64).reshape(-1)
    assert pos.shape[0] == n
    out = np.empty_like(x)
    rc = _load().orc_rope_rows(_ptr(out), _ptr(x), _ptr(pos), n, D, _dtype_code(x),
                               _ptr(np.ascontiguousarray(cos_cache, dtype=np.float32)),
                               _ptr(np.ascontiguousarray(sin_cache, dtype=np.float32)),
                               cos_cache.shape[0])
    if rc != 0:
        raise ValueError("rope_rows: position outside the cos/sin cache")
    return out


def window_append(k_cache, v_cache, new_k, new_v, lengths, windowed, cos_cache=None,
                  sin_cache=None, k_stage=None, v_stage=None):
    """Append in place into ``k_cache``/``v_cache`` ([B, Hkv, C, D]); returns the
    per-row flags.  For windowed S > 1 the stages ([B, Hkv, C + S, D]) are
    filled with the seeded rows."""
    B, Hkv, C, D = k_cache.shape
    S = new_k.shape[2]
    flags = np.zeros(B, dtype=np.int32)
    cc = None if cos_cache is None else np.ascontiguousarray(cos_cache, dtype=np.float32)
    ss = None if sin_cache is None else np.ascontiguousarray(sin_cache, dtype=np.float32)
    rmax = 0 if cc is None else cc.shape[0]
    rc = _load().orc_window_append(
        _ptr(k_cache), _ptr(v_cache), _ptr(np.ascontiguousarray(new_k)),
        _ptr(np.ascontiguousarray(new_v)), _ptr(k_stage), _ptr(v_stage),
        _ptr(lengths["past_abs"]), _ptr(lengths["cache_past"]), _ptr(lengths["cache_total"]),
        _ptr(lengths["evict"]), B, Hkv, S, C, D, _dtype_code(k_cache), int(windowed),
        _ptr(cc), _ptr(ss), rmax, _ptr(flags))
    if rc != 0:
        raise ValueError("window_append: staging buffers required for windowed S > 1")
    return flags


def gqa_attention(q, k_rows, v_rows, n_rows, total_abs, window=0, scale=None,
                  cos_cache=None, sin_cache=None):
    """Attention of q [B, Hq, S, D] over k/v rows [B, Hkv, R, D]; returns
    (out [B, Hq, S, D] in q's type, per-row flags)."""
    q = np.ascontiguousarray(q)
    B, Hq, S, D = q.shape
    _, Hkv, R, _ = k_rows.shape
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.zeros_like(q)
    flags = np.zeros(B, dtype=np.int32)
    cc = None if cos_cache is None else np.ascontiguousarray(cos_cache, dtype=np.float32)
    ss = None if sin_cache is None else np.ascontiguousarray(sin_cache, dtype=np.float32)
    rmax = 0 if cc is None else cc.shape[0]
    rc = _load().orc_gqa_attention(
        _ptr(out), _ptr(q), _ptr(np.ascontiguousarray(k_rows)), _ptr(np.ascontiguousarray(v_rows)),
        R, _ptr(np.ascontiguousarray(n_rows, dtype=np.int32)),
        _ptr(np.ascontiguousarray(total_abs, dtype=np.int32)), B, Hq, Hkv, S, D,
        _dtype_code(q), int(window), float(scale), _ptr(cc), _ptr(ss), rmax, _ptr(flags))
    if rc != 0:
        raise ValueError("gqa_attention: q_heads must be a multiple of kv_heads")
    return out, flags


# --------------------------------------------------------------------------
# ring buffer ("Stateful decode & KV cache", "Sliding-window ring buffer")
# --------------------------------------------------------------------------

def ring_slot_positions(T, C):
    """Absolute position held by each of the C slots after T tokens were
    written one by one at slot (position mod C); -1 for a slot never written.
    Slot r holds the newest p < T with p = r (mod C)."""
    pos = np.full(C, -1, dtype=np.int64)
    for r in range(C):
        p = (T - 1) - ((T - 1 - r) % C)
        pos[r] = p if p >= 0 else -1
    return pos


def ring_append(k_ring, v_ring, new_k, new_v, past_abs, cos_cache=None, sin_cache=None):
    """Write S new rows per (b, kv head) into rings [B, Hkv, C, D] in place:
    row i of batch row b (absolute position P_b + i) goes to slot
    (P_b + i) mod C, K rotated there first when the cos/sin tables are given.
    This is TensorScatter circular with write index P_b on the rotated rows
    (when S > C the later rows overwrite the earlier ones)."""
    B, Hkv, S, D = new_k.shape
    P = np.asarray(past_abs, dtype=np.int64)
    nk = np.ascontiguousarray(new_k)
    if cos_cache is not None:
        pos = np.broadcast_to((P[:, None, None] + np.arange(S)[None, None, :]), (B, Hkv, S))
        nk = rope_rows(nk, np.ascontiguousarray(pos).reshape(-1), cos_cache, sin_cache)
    nv = np.ascontiguousarray(new_v)
    C = k_ring.shape[2]
    if S > C:
        # TensorScatter takes at most max_seq rows; the earlier ones would be
        # overwritten by the later ones anyway
        nk = np.ascontiguousarray(nk[:, :, S - C:])
        nv = np.ascontiguousarray(nv[:, :, S - C:])
        P = P + (S - C)
    _, fk = tensor_scatter(k_ring, nk, P, mode=CIRCULAR, out=k_ring)
    _, fv = tensor_scatter(v_ring, nv, P, mode=CIRCULAR, out=v_ring)
    return fk | fv


def ring_attention(q, k_ring, v_ring, total_abs, window=0, scale=None, cos_cache=None,
                   sin_cache=None):
    """Attention of q [B, Hq, S, D] (query i at position T - S + i) over a
    ring [B, Hkv, C, D] after T tokens: the ring's newest n = min(T, C, W)
    positions (W <= 0: no window) are read from their slots in position
    order, then the causal and window mask apply as in gqa_attention.  Exact
    for the last query; earlier queries of a chunk that wrapped the ring miss
    the keys it overwrote.  Returns (out, flags) like gqa_attention."""
    B, Hkv, C, D = k_ring.shape
    T = np.asarray(total_abs, dtype=np.int64)
    k = np.zeros_like(k_ring)
    v = np.zeros_like(v_ring)
    n = np.zeros(B, dtype=np.int32)
    for b in range(B):
        nb = min(int(T[b]), C) if window <= 0 else min(int(T[b]), C, window)
        held = ring_slot_positions(int(T[b]), C)
        order = [int(np.nonzero(held == p)[0][0]) for p in range(int(T[b]) - nb, int(T[b]))]
        k[b, :, :nb] = k_ring[b][:, order]
        v[b, :, :nb] = v_ring[b][:, order]
        n[b] = nb
    return gqa_attention(q, k, v, n, T.astype(np.int32), window=window, scale=scale,
                         cos_cache=cos_cache, sin_cache=sin_cache)


# --------------------------------------------------------------------------
# paged cache ("Persistent KV Cache and Decode Performance Roadmap", Phase 2:
# fixed-size pages and a page table consumed directly by attention)
# --------------------------------------------------------------------------

def paged_rows(pool, block_table, n_rows, page_size):
    """The first n_rows[b] logical rows of every batch row, gathered from a
    page pool [n_pages, Hkv, P, D] through block_table [B, max_pages]: row r
    of batch row b is slot r % P of page block_table[b][r // P].  Returns
    [B, Hkv, max(n_rows), D] (rows past n_rows[b] are zero)."""
    pool = np.asarray(pool)
    bt = np.asarray(block_table)
    B = bt.shape[0]
    _, Hkv, P, D = pool.shape
    assert P == page_size
    n = np.asarray(n_rows, dtype=np.int64)
    R = int(n.max()) if B else 0
    out = np.zeros((B, Hkv, max(R, 1), D), dtype=pool.dtype)
    for b in range(B):
        for r in range(int(n[b])):
            out[b, :, r] = pool[int(bt[b, r // P]), :, r % P]
    return out


def paged_append(k_pool, v_pool, block_table, page_size, new_k, new_v, past_abs,
                 cos_cache=None, sin_cache=None):
    """Write S new rows per (b, kv head) in place: row i of batch row b
    (absolute position P_b + i) goes to slot (P_b + i) % P of page
    block_table[b][(P_b + i) // P]; K is rotated at its position first when
    the cos/sin tables are given."""
    B, Hkv, S, D = new_k.shape
    P = page_size
    nk = np.ascontiguousarray(new_k)
    Pb = np.asarray(past_abs, dtype=np.int64)
    if cos_cache is not None:
        pos = np.broadcast_to(Pb[:, None, None] + np.arange(S)[None, None, :], (B, Hkv, S))
        nk = rope_rows(nk, np.ascontiguousarray(pos).reshape(-1), cos_cache, sin_cache)
    for b in range(B):
        for i in range(S):
            r = int(Pb[b]) + i
            page = int(block_table[b][r // P])
            k_pool[page, :, r % P] = nk[b, :, i]
            v_pool[page, :, r % P] = new_v[b, :, i]


def paged_attention(q, k_pool, v_pool, block_table, page_size, n_rows, total_abs, window=0,
                    scale=None, cos_cache=None, sin_cache=None):
    """Attention of q [B, Hq, S, D] over the n_rows[b] logical rows of a paged
    cache (row r at absolute position total_abs[b] - n_rows[b] + r).  Returns
    (out, flags) like gqa_attention."""
    k = paged_rows(k_pool, block_table, n_rows, page_size)
    v = paged_rows(v_pool, block_table, n_rows, page_size)
    return gqa_attention(q, k, v, np.asarray(n_rows, np.int32), np.asarray(total_abs, np.int32),
                         window=window, scale=scale, cos_cache=cos_cache, sin_cache=sin_cache)


# ---------------------------------------------------------------------------
# affine page quantization ("Persistent input/output feedback", "Optional
# heterogeneous paged KV": selected-block quantization; roadmap "Phase 3")
# ---------------------------------------------------------------------------

PAGE_QUANT = 0x40000000  # block-table flag: the entry names a page of the int8 pools


def to_f32(a):
    """float32 values of 16-bit bit patterns (uint16 = bf16), float16 or float32."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32)
    return a.astype(np.float32)


def quantize_affine(x, scale, zero_point, unsigned=False):
    """Affine codes of float32 values: x / scale in float32, rounded to the
    nearest integer with ties to even, plus the zero point, saturated to the
    code range (INT8 [-128, 127], UINT8 [0, 255]).  Returns int32 codes."""
    t = np.asarray(x, dtype=np.float32) / np.float32(scale)
    r = np.rint(t).astype(np.float64)          # integral (or +-inf): ties to even
    lo, hi = (0, 255) if unsigned else (-128, 127)
    return np.clip(r + zero_point, lo, hi).astype(np.int32)


def dequantize_affine(codes, scale, zero_point):
    """Reconstruction (code - zero point) * scale in float32."""
    return ((np.asarray(codes, dtype=np.float32) - np.float32(zero_point)) *
            np.float32(scale)).astype(np.float32)


def quantize_page(page, scale, zero_point, unsigned=False):
    """One page (any shape) of 16-bit bits or float32 values -> (stored
    bytes as uint8, stored zero point).  The stored byte is the code plus an
    offset (128 for INT8, so that c in [-128, 127] becomes c + 128; 0 for
    UINT8) and the stored zero point is zero_point plus the same offset, so
    (stored - stored zero point) * scale is the reconstruction for either
    code type."""
    codes = quantize_affine(to_f32(page), scale, zero_point, unsigned)
    off = 0 if unsigned else 128
    return (codes + off).astype(np.uint8), int(zero_point) + off


def paged_rows_q(pool, qpool, qparams, which, block_table, n_rows, page_size):
    """float32 logical rows [B, Hkv, max(n_rows), D] of a paged cache whose
    table entries name either a page of the 16-bit pool or (flag PAGE_QUANT)
    a page of the int8 pool, reconstructed with that page's scale and stored
    zero point (qparams[page] = (k_scale, k_zp, v_scale, v_zp); which = 0 for
    K, 1 for V)."""
    bt = np.asarray(block_table)
    B = bt.shape[0]
    _, Hkv, P, D = pool.shape
    assert P == page_size
    n = np.asarray(n_rows, dtype=np.int64)
    R = int(n.max()) if B else 0
    out = np.zeros((B, Hkv, max(R, 1), D), dtype=np.float32)
    for b in range(B):
        for r in range(int(n[b])):
            e = int(bt[b, r // P])
            if e & PAGE_QUANT:
                page = e & (PAGE_QUANT - 1)
                sc, zp = qparams[page][2 * which], qparams[page][2 * which + 1]
                out[b, :, r] = dequantize_affine(qpool[page, :, r % P], sc, zp)
            else:
                out[b, :, r] = to_f32(pool[e, :, r % P])
    return out


def paged_attention_q(q, k_pool, v_pool, qk_pool, qv_pool, qparams, block_table, page_size,
                      n_rows, total_abs, window=0, scale=None, cos_cache=None, sin_cache=None):
    """Attention of q [B, Hq, S, D] (16-bit bits or float32) over a paged
    cache of 16-bit and int8 pages, in float32 over the reconstructed rows.
    Returns (out float32, flags)."""
    k = paged_rows_q(k_pool, qk_pool, qparams, 0, block_table, n_rows, page_size)
    v = paged_rows_q(v_pool, qv_pool, qparams, 1, block_table, n_rows, page_size)
    return gqa_attention(to_f32(q), k, v, np.asarray(n_rows, np.int32),
                         np.asarray(total_abs, np.int32), window=window, scale=scale,
                         cos_cache=cos_cache, sin_cache=sin_cache)
