"""The C-ABI library without a GPU: it loads, exports every entry point that
include/kvc.h declares, and rejects bad arguments on the host before any CUDA
call (the host checks return before a kernel is enqueued, so fake non-NULL
pointers are never touched)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvc():
    from persistent_kv_cache_gb300 import build as B
    B.build()
    from persistent_kv_cache_gb300 import kvc as K
    return K


def _declared():
    text = open(os.path.join(ROOT, "include", "kvc.h")).read()
    return sorted(set(re.findall(r"^\w[\w \*]*?\b(kvc_\w+)\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(kvc):
    names = _declared()
    assert "kvc_gqa_decode" in names and len(names) >= 8
    lib = kvc.library()
    for n in names:
        assert hasattr(lib, n), n
    assert set(kvc.EXPORTS) <= set(names)


def test_binding_rejects_host_tensors(kvc):
    """The binding passes device addresses only: a tensor in host memory is
    refused before anything reaches the library."""
    import torch
    x = torch.zeros(2, 2, 16, 8)
    with pytest.raises(ValueError, match="CUDA"):
        kvc.kvc_tensor_scatter(x, x, x[:, :, :1].contiguous())
    with pytest.raises(ValueError, match="CUDA"):
        kvc.kvc_seq_lengths(torch.zeros(2, dtype=torch.int32), 1, 16, 0)


def test_version_and_strings(kvc):
    assert kvc.kvc_abi_version() == 7
    assert kvc.kvc_status_string(0) == "ok"
    assert "window" in kvc.kvc_status_string(7)


FAKE = 0x10000  # 16-byte aligned, never dereferenced on the paths below
L5 = None


def _lengths(kvc):
    return kvc.KvcLengths(FAKE, FAKE, FAKE, FAKE, FAKE)


def test_scatter_host_checks(kvc):
    lib = kvc.library()
    shape = (ctypes.c_int64 * 4)(2, 2, 16, 8)
    f = lib.kvc_tensor_scatter
    assert f(None, FAKE, FAKE, None, 4, shape, 1, -2, 0, 4, None, None) == 1   # NULL
    assert f(FAKE, FAKE, FAKE, None, 4, shape, 1, 0, 0, 4, None, None) == 2   # axis 0
    assert f(FAKE, FAKE, FAKE, None, 4, shape, 1, 4, 0, 4, None, None) == 2   # axis out of range
    assert f(FAKE, FAKE, FAKE, None, 4, shape, 17, -2, 0, 4, None, None) == 2  # S > max_seq
    assert f(FAKE, FAKE, FAKE, None, 4, shape, 1, -2, 0, 3, None, None) == 3  # elem bytes
    assert f(FAKE, FAKE, FAKE, None, 4, shape, 1, -2, 2, 4, None, None) == 5  # mode
    assert f(FAKE, FAKE, FAKE, None, 1, shape, 1, -1, 0, 4, None, None) == 2  # rank 1
    # partial overlap of present and past
    assert f(FAKE, FAKE + 16, FAKE * 4, None, 4, shape, 1, -2, 0, 4, None, None) == 2


def test_lengths_host_checks(kvc):
    lib = kvc.library()
    f = lib.kvc_seq_lengths
    L = _lengths(kvc)
    assert f(FAKE, 4, 0, 128, 1, 128, L, None, None) == 2       # S < 1
    assert f(FAKE, 4, 1, 0, 1, 128, L, None, None) == 6         # C < 1
    assert f(FAKE, 4, 1, 128, 1, 129, L, None, None) == 7       # W > C
    assert f(FAKE, 4, 1, 128, 1, 0, L, None, None) == 7         # W missing
    assert f(None, 4, 1, 128, 1, 128, L, None, None) == 1
    assert f(FAKE, 0, 1, 128, 1, 128, L, None, None) == 0       # empty batch: nothing to do
    assert f(FAKE, 4, 1, 128, 4, 128, L, None, None) == 5       # unknown policy
    assert f(FAKE, 4, 1, 128, 2, 129, L, None, None) == 7       # drifting needs W <= C
    assert f(FAKE, 4, 1, 128, 2, 0, L, None, None) == 7


def test_append_host_checks(kvc):
    lib = kvc.library()
    f = lib.kvc_window_append
    L = _lengths(kvc)
    args = dict(kc=FAKE, vc=FAKE * 2, nk=FAKE * 3, nv=FAKE * 4, ks=None, vs=None)
    base = [args["kc"], args["vc"], args["nk"], args["nv"], None, None, L]
    assert f(*base, 2, 2, 1, 16, 8, 7, 1, 0, None, None, 0, None, None) == 3        # dtype
    assert f(*base, 2, 2, 1, 16, 7, 1, 1, 0, None, None, 0, None, None) == 2        # odd D
    assert f(*base, 2, 2, 4, 16, 8, 1, 1, 0, None, None, 0, None, None) == 1        # no stage
    assert f(*base, 2, 2, 1, 16, 8, 1, 1, 1, None, None, 0, None, None) == 5        # copy-back S=1
    assert f(*base, 2, 2, 1, 16, 8, 1, 4, 0, None, None, 0, None, None) == 5        # policy
    assert f(*base, 2, 2, 4, 16, 8, 1, 3, 1, None, None, 0, None, None) == 5        # ring copy-back
    assert f(*base, 2, 2, 1, 0, 8, 1, 1, 0, None, None, 0, None, None) == 6         # C < 1
    assert f(*base, 2, 2, 1, 16, 8, 1, 1, 0, FAKE, None, 16, None, None) == 1       # half a table
    unaligned = [FAKE + 2] + base[1:]
    assert f(*unaligned, 2, 2, 1, 16, 8, 1, 1, 0, None, None, 0, None, None) == 4   # alignment


def test_decode_host_checks(kvc):
    lib = kvc.library()
    f = lib.kvc_gqa_decode
    L = _lengths(kvc)
    base = [FAKE, FAKE * 2, FAKE * 3, FAKE * 4, L]
    assert f(*base, 2, 6, 4, 64, 128, 1, 0, 0.0, None, None, 0, FAKE, 1 << 20, None, None) == 2
    assert f(*base, 2, 8, 2, 64, 96, 1, 0, 0.0, None, None, 0, FAKE, 1 << 20, None, None) == 5
    assert f(*base, 2, 64, 2, 64, 128, 1, 0, 0.0, None, None, 0, FAKE, 1 << 20, None, None) == 5
    assert f(*base, 2, 8, 2, 8192, 128, 1, 0, 0.0, None, None, 0, None, 0, None, None) == 8
    need = lib.kvc_gqa_decode_workspace_size(2, 8, 2, 8192, 128, 1)
    assert need == 2 * 8 * 16 * 130 * 4
    assert f(*base, 2, 8, 2, 8192, 128, 1, 0, 0.0, None, None, 0, FAKE, need - 4, None, None) == 8
    bad = [FAKE + 8] + base[1:]
    assert f(*bad, 2, 8, 2, 64, 128, 1, 0, 0.0, None, None, 0, FAKE, 256, None, None) == 4
    assert lib.kvc_gqa_decode_workspace_size(2, 8, 2, 128, 64, 1) == 256
    # head_dim 256 is a supported 16-bit size: a missing workspace is the error
    assert f(*base, 2, 16, 8, 8192, 256, 1, 0, 0.0, None, None, 0, None, 0, None, None) == 8
    assert f(*base, 2, 16, 8, 8192, 256, 2, 0, 0.0, None, None, 0, None, 0, None, None) == 8


def test_decode_ring_host_checks(kvc):
    lib = kvc.library()
    f = lib.kvc_gqa_decode_ring
    L = _lengths(kvc)
    base = [FAKE, FAKE * 2, FAKE * 3, FAKE * 4, L]
    assert f(*base, 2, 6, 4, 64, 128, 1, 0, 0.0, None, None, 0, FAKE, 1 << 20, None, None) == 2
    assert f(*base, 2, 8, 2, 64, 96, 1, 0, 0.0, None, None, 0, FAKE, 1 << 20, None, None) == 5
    assert f(*base, 2, 8, 2, 8192, 128, 1, 0, 0.0, None, None, 0, None, 0, None, None) == 8
    bad = [FAKE + 8] + base[1:]
    assert f(*bad, 2, 8, 2, 64, 128, 1, 0, 0.0, None, None, 0, FAKE, 256, None, None) == 4


def test_decode_step_host_checks(kvc):
    lib = kvc.library()
    f = lib.kvc_decode_step
    none = kvc.KvcLengths(None, None, None, None, None)
    base = [FAKE, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 5, FAKE * 6, FAKE * 7]
    # policy: contiguous or ring only
    assert f(*base, none, 2, 8, 2, 128, 64, 1, 1, 0, 0.0, None, None, 0, FAKE, 1 << 20, None,
             None) == 5
    assert f(*base, none, 2, 8, 2, 128, 64, 0, 0, 0, 0.0, None, None, 0, FAKE, 1 << 20, None,
             None) == 5                                                      # fp32
    need = lib.kvc_decode_step_workspace_size(2, 8, 2, 8192, 128, 1)
    assert need == lib.kvc_gqa_decode_workspace_size(2, 8, 2, 8192, 128, 1)
    far = [FAKE, FAKE * 2, 1 << 32, 2 << 32, FAKE * 5, FAKE * 6, FAKE * 7]  # caches apart
    assert f(*far, none, 2, 8, 2, 8192, 128, 1, 0, 0, 0.0, None, None, 0, FAKE, need - 4,
             None, None) == 8
    half = kvc.KvcLengths(FAKE, None, None, None, None)
    assert f(*base, half, 2, 8, 2, 128, 64, 1, 3, 0, 0.0, None, None, 0, FAKE, 256, None,
             None) == 1
    assert f(*base, none, 0, 8, 2, 128, 64, 1, 3, 0, 0.0, None, None, 0, None, 0, None,
             None) == 0


def test_paged_host_checks(kvc):
    lib = kvc.library()
    L = _lengths(kvc)
    d = lib.kvc_gqa_decode_paged
    base = [FAKE, FAKE * 2, FAKE * 3, 1 << 32]
    # (out, q, k_pool, v_pool, table, max_pages, n_pages, page_size, len, B, Hq, Hkv, D, dtype, W,
    #  scale, cos, sin, rope_max, ws, ws_bytes, status, stream)
    ok = [FAKE * 4, 8, 64, 64, L, 2, 8, 2, 128, 1, 0, 0.0, None, None, 0, FAKE, 1 << 24, None, None]
    assert d(*base, *ok[:3], 48, *ok[4:]) == 2                      # page not a multiple of 64
    assert d(*base, *ok[:3], 0, *ok[4:]) == 2
    assert d(*base, *ok[:9], 0, *ok[10:]) == 5                      # fp32 not on this path
    assert d(*base, *ok[:9], 9, *ok[10:]) == 3                      # unknown dtype
    assert d(*base, None, *ok[1:]) == 1                             # no table
    assert d(FAKE + 8, *base[1:], *ok) == 4                         # alignment
    a = lib.kvc_paged_append
    okp = [FAKE * 4, 8, 64, 64, L, 2, 2, 1, 128, 1, None, None, 0, None, None]
    assert a(*base, *okp[:3], 0, *okp[4:]) == 2                     # page size
    assert a(*base, *okp[:9], 7, *okp[10:]) == 3                    # dtype
    assert a(*base, *okp[:7], 0, *okp[8:]) == 2                     # S = 0
    assert a(*base, None, *okp[1:]) == 1


def test_prefill_host_checks(kvc):
    lib = kvc.library()
    f = lib.kvc_gqa_prefill_chunk
    L = _lengths(kvc)
    base = [FAKE, FAKE * 2, FAKE * 3, FAKE * 4]
    ws = [None, 0, None, None]  # workspace, bytes, status, stream
    assert f(*base, 100, L, 2, 8, 2, 0, 64, 1, 0, 0.0, None, None, 0, *ws) == 2  # S = 0
    assert f(*base, 10, L, 2, 8, 2, 16, 64, 1, 0, 0.0, None, None, 0, *ws) == 6  # R < S
    assert f(*base, 100, L, 2, 8, 3, 16, 64, 1, 0, 0.0, None, None, 0, *ws) == 2  # heads
    assert f(*base, 100, L, 2, 8, 2, 16, 64, 9, 0, 0.0, None, None, 0, *ws) == 3  # dtype
    assert f(*base, 100, L, 2, 8, 2, 16, 64, 1, 0, 0.0, None, None, 0, FAKE + 16, 1 << 20,
             None, None) == 4                                                  # ws alignment
    assert f(*base, 100, L, 2, 8, 2, 16, 64, 1, 0, 0.0, FAKE * 5 + 4, FAKE * 6, 200,
             *ws) == 4                                                         # rope alignment
    assert f(*base, 100, L, 2, 8, 2, 16, 64, 1, 0, 0.0, FAKE * 5, FAKE * 6 + 8, 200,
             *ws) == 4
    wsz = lib.kvc_gqa_prefill_workspace_size
    assert wsz(8, 16, 8, 2048, 4096 + 2048, 256, 1, 4096) == 0   # a full grid: no split
    assert wsz(2, 8, 2, 64, 4096, 128, 0, 0) == 0                # fp32: never split


def test_binding_requires_library(monkeypatch, kvc):
    monkeypatch.setattr(kvc, "LIB_PATH", "/nonexistent/libkvc.so")
    monkeypatch.setattr(kvc, "_lib", None)
    with pytest.raises(kvc.KvcLibraryMissing):
        kvc.library()


def test_window_step_host_checks(kvc):
    lib = kvc.library()
    f = lib.kvc_window_decode_step
    wsz = lib.kvc_window_decode_step_workspace_size
    none = kvc.KvcLengths(None, None, None, None, None)
    base = [FAKE, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 5, FAKE * 6, FAKE * 7]
    nows = [None, 0, None, None]   # workspace, bytes, dev_status, stream
    for pol in (1, 2):
        assert f(*base, none, 2, 8, 2, 128, 64, 1, pol, 129, 0.0, None, None, 0, *nows) == 7
        assert f(*base, none, 2, 8, 2, 128, 64, 1, pol, 0, 0.0, None, None, 0, *nows) == 7
    assert f(*base, none, 2, 8, 2, 128, 64, 1, 0, 128, 0.0, None, None, 0, *nows) == 5  # contig
    assert f(*base, none, 2, 8, 2, 128, 64, 1, 4, 128, 0.0, None, None, 0, *nows) == 5  # policy
    assert f(*base, none, 2, 8, 2, 128, 64, 0, 1, 128, 0.0, None, None, 0, *nows) == 5  # fp32
    assert f(*base, none, 2, 8, 2, 128, 96, 1, 1, 128, 0.0, None, None, 0, *nows) == 5  # D
    half = kvc.KvcLengths(FAKE, None, None, None, None)
    assert f(*base, half, 2, 8, 2, 128, 64, 1, 2, 128, 0.0, None, None, 0, *nows) == 1
    assert f(*base, none, 0, 8, 2, 128, 64, 1, 2, 128, 0.0, None, None, 0, *nows) == 0
    # a window held on chip needs no workspace; a larger one needs the
    # lengths (5 x batch int32, 256-byte rounded) and the split partials
    assert wsz(2, 8, 2, 512, 64, 1) == 0 and wsz(2, 8, 2, 128, 256, 1) == 0
    assert wsz(2, 8, 2, 1024, 64, 1) == 256 + 256
    assert wsz(8, 16, 8, 4096, 256, 1) == 256 + 8 * 16 * 4 * (256 + 2) * 4   # 1024-row splits
    for pol in (1, 2, 3):
        assert f(*base, none, 8, 16, 8, 4096, 256, 1, pol, 4096, 0.0, None, None, 0,
                 *nows) == 8
        assert f(*base, none, 8, 16, 8, 4096, 256, 1, pol, 4096, 0.0, None, None, 0,
                 FAKE + 16, 1 << 24, None, None) == 4


def test_append_inplace_host_checks(kvc):
    lib = kvc.library()
    f = lib.kvc_window_append_inplace
    L = _lengths(kvc)
    far = [FAKE, 1 << 32, FAKE * 3, FAKE * 4, L]   # k rows, v rows far apart, new k, new v
    # (..., batch, kv_heads, S, capacity, rows_per_head, head_dim, dtype, policy, phase, cos, sin,
    #  rope_max, status, stream)
    ok = [2, 2, 16, 128, 144, 64, 1, 1, 0, None, None, 0, None, None]
    assert f(*far, *ok[:4], 143, *ok[5:]) == 6                      # rows_per_head < C + S
    assert f(*far, *ok[:7], 0, *ok[8:]) == 5                        # contiguous: no stage
    assert f(*far, *ok[:7], 3, *ok[8:]) == 5                        # ring: nothing moves
    assert f(*far, *ok[:8], 2, *ok[9:]) == 5                        # unknown phase
    assert f(*far, *ok[:5], 4, *ok[6:]) == 5                        # 8-byte rows: no bulk copies
    assert f(*far, *ok[:6], 7, *ok[7:]) == 3                        # dtype
    assert f(far[0], far[1], None, None, L, *ok) == 1               # append without new rows
    assert f(FAKE + 8, *far[1:], *ok) == 4                          # alignment
    assert f(FAKE, FAKE + 16, FAKE * 3, FAKE * 4, L, *ok) == 2      # K and V rows overlap
    assert f(*far, *ok[:9], FAKE, None, 16, None, None) == 1        # half a rope table
    assert f(*far, 0, *ok[1:]) == 0                                 # empty batch


def test_quantize_pages_host_checks(kvc):
    lib = kvc.library()
    f = lib.kvc_quantize_pages
    # (k, v, qk, qv, src, dst, n, n_pool, n_q, page, kv_heads, D, dtype, k_scale, k_zp, k_uns,
    #  v_scale, v_zp, v_uns, qparams, status, stream)
    ptr = [FAKE, 1 << 32, 2 << 32, 3 << 32, FAKE * 5, FAKE * 6]
    ok = [4, 8, 8, 64, 2, 128, 1, 0.01, 0, 0, 0.01, 128, 1, FAKE * 7, None, None]
    assert f(*ptr, *ok[:6], 0, *ok[7:]) == 5                        # fp32 pools
    assert f(*ptr, *ok[:6], 9, *ok[7:]) == 3                        # unknown dtype
    assert f(*ptr, *ok[:5], 12, *ok[6:]) == 2                       # head_dim not a multiple of 8
    assert f(*ptr, *ok[:7], 0.0, *ok[8:]) == 2                      # scale 0
    assert f(*ptr, *ok[:7], float("nan"), *ok[8:]) == 2             # scale NaN
    assert f(*ptr, *ok[:7], float("inf"), *ok[8:]) == 2
    assert f(*ptr, *ok[:8], 200, *ok[9:]) == 2                      # INT8 zero point 200
    assert f(*ptr, *ok[:11], -1, *ok[12:]) == 2                     # UINT8 zero point -1
    assert f(*ptr, 0, *ok[1:]) == 0                                 # nothing to convert
    assert f(None, *ptr[1:], *ok) == 1
    assert f(FAKE + 8, *ptr[1:], *ok) == 4                          # alignment
    assert f(*ptr[:2], FAKE * 9, FAKE * 9 + 16, *ptr[4:], *ok) == 2  # int8 pools overlap


def test_decode_paged_q_host_checks(kvc):
    lib = kvc.library()
    f = lib.kvc_gqa_decode_paged_q
    L = _lengths(kvc)
    # (out, q, k, v, qk, qv, qparams, n_q, table, max_pages, n_pool, page, len, B, Hq, Hkv, D,
    #  dtype, W, scale, cos, sin, rope_max, ws, ws_bytes, status, stream)
    pools = [FAKE, FAKE * 2, FAKE * 3, 1 << 32, 2 << 32, 3 << 32, FAKE * 4]
    tail = [FAKE * 5, 8, 64, 64, L, 2, 8, 2, 128, 1, 0, 0.0, None, None, 0, FAKE, 1 << 24, None,
            None]
    assert f(*pools, 0, *tail) == 2                                  # no int8 pages
    assert f(*pools[:4], None, *pools[5:], 8, *tail) == 1            # int8 pool missing
    assert f(*pools[:6], FAKE * 4 + 4, 8, *tail) == 4                # qparams alignment
    assert f(*pools[:4], 4 << 32, (4 << 32) + 16, pools[6], 8, *tail) == 2  # int8 pools overlap
    assert f(*pools, 8, *tail[:3], 48, *tail[4:]) == 2               # page not a multiple of 64


def test_window_prefill_step_host_checks(kvc):
    """kvc_window_prefill_step: policy, window, stage, shape and alignment
    checks return before anything is enqueued."""
    lib = kvc.library()
    f = lib.kvc_window_prefill_step
    L = _lengths(kvc)
    FAR = FAKE << 12  # the stage: far from the cache pointers
    # out, q, k_cache, v_cache, new_k, new_v, k_stage, v_stage
    ptrs = [FAKE, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 5, FAKE * 6, FAR, FAR * 2]
    # batch, q_heads, kv_heads, S, C, D, dtype, policy, W, scale, cos, sin, rmax
    ok = [2, 8, 2, 16, 64, 64, 1, 1, 48, 0.0, None, None, 0]
    tail = [None, 0, None, None]  # workspace, bytes, status, stream
    call = lambda p, a: f(*p, L, *a, *tail)
    assert call(ptrs, ok[:7] + [0] + ok[8:]) == 5                 # contiguous: not this call
    assert call(ptrs, ok[:7] + [3] + ok[8:]) == 5                 # ring: not this call
    assert call(ptrs, ok[:8] + [0] + ok[9:]) == 7                 # W < 1
    assert call(ptrs, ok[:8] + [65] + ok[9:]) == 7                # W > C
    assert call(ptrs[:6] + [None, None], ok) == 1                 # S > 1 without a stage
    assert call(ptrs, ok[:3] + [0] + ok[4:]) == 2                 # S = 0
    assert call(ptrs, ok[:6] + [9] + ok[7:]) == 3                 # dtype
    assert call(ptrs, ok[:5] + [96] + ok[6:]) == 5                # head_dim 96 (16-bit)
    assert call([FAKE + 8] + ptrs[1:], ok) == 4                   # out alignment
    assert call(ptrs, ok[:4] + [0] + ok[5:]) == 6                 # C < 1
    # the stage overlapping the cache
    assert call(ptrs[:6] + [FAKE * 3, FAR * 2], ok) == 2
    assert call(ptrs, [0] + ok[1:]) == 0                          # empty batch: nothing to do
