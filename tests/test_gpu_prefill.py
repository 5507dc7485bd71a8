"""GPU parity for kvc_gqa_prefill_chunk (tcgen05 path for bf16/fp16, CUDA-core
path for fp32) against the oracle, max-abs <= 2e-2 (16-bit) / 1e-4 (fp32).

Covers ragged chunks (S not a multiple of the query block, P = 0, S > C),
every supported head dim and GQA group, window masks, staged (windowed
cache) and contiguous rows, consecutive chunks on one windowed cache with
bit-exact stage/cache checks, and the full windowed chunked-prefill workload
(8 x 16/8 heads x 256, C = W = 4096, P ~ U[0, 20000], S in {64, 512, 2048})
with sampled queries checked one by one.
"""
import numpy as np
import pytest
import torch

from _gpu_helpers import assert_bytes_equal, assert_close, dev, status, tol
from persistent_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from persistent_kv_cache_gb300 import kvc
    return kvc


def _oracle_queries(orc, q, k_rows, v_rows, lens, S, window, cos, sin, idx):
    """Oracle output of the chunk's queries `idx` (each evaluated as the last
    query of a chunk ending at it: rows [0, Lp + i + 1), total P + i + 1)."""
    B = q.shape[0]
    outs = []
    for i in idx:
        n = (lens["cache_past"] + i + 1).astype(np.int32)
        T = (lens["past_abs"] + i + 1).astype(np.int32)
        o, _ = orc.gqa_attention(np.ascontiguousarray(q[:, :, i:i + 1]), k_rows, v_rows, n, T,
                                 window=window, cos_cache=cos, sin_cache=sin)
        outs.append(o)
    return np.concatenate(outs, axis=2)


def _chunk_case(K, orc, dtype, B, Hq, Hkv, D, C, S, P, window, windowed, rope, seed,
                sample=None, workspace="auto"):
    P = np.asarray(P, dtype=np.int64)
    T = P + S
    kc = synth.normal((B, Hkv, C, D), seed, 1, dtype)
    vc = synth.normal((B, Hkv, C, D), seed, 2, dtype)
    nk = synth.normal((B, Hkv, S, D), seed, 3, dtype)
    nv = synth.normal((B, Hkv, S, D), seed, 4, dtype)
    q = synth.normal((B, Hq, S, D), seed, 5, dtype)
    cos = sin = None
    rope_d = None
    if rope:
        cos, sin = synth.rope_cache(int(T.max()) + 1, D)
        rope_d = (cos.to(dev()), sin.to(dev()))
    sk = (T - 1).astype(np.int32)
    st = status()
    gk, gv = kc.to(dev()), vc.to(dev())
    L = K.kvc_seq_lengths(torch.from_numpy(sk).to(dev()), S, C, windowed,
                          local_window_size=window if windowed else 0, status=st)
    if windowed:
        # stage rows past Lp + S hold NaN: the kernel must never let them in
        ks = torch.full((B, Hkv, C + S, D), float("nan"), dtype=dtype, device=dev())
        vs = torch.full_like(ks, float("nan"))
        K.kvc_window_append(gk, gv, nk.to(dev()), nv.to(dev()), L, 1, K.KVC_APPEND, ks, vs,
                            rope=rope_d, status=st)
        rows_k, rows_v = ks, vs
    else:
        K.kvc_window_append(gk, gv, nk.to(dev()), nv.to(dev()), L, 0, rope=rope_d, status=st)
        rows_k, rows_v = gk, gv
    out = torch.full((B, Hq, S, D), float("nan"), dtype=dtype, device=dev())
    K.kvc_gqa_prefill_chunk(out, q.to(dev()), rows_k, rows_v, L, local_window_size=window,
                            rope=rope_d, status=st, workspace=workspace)
    if windowed:
        K.kvc_window_append(gk, gv, None, None, L, 1, K.KVC_COPY_BACK, ks, vs, rope=rope_d,
                            status=st)
    torch.cuda.synchronize()
    assert st.item() == 0, st.item()

    lens = orc.seq_lengths(sk, S, C, windowed)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    cn = None if cos is None else cos.numpy()
    sn = None if sin is None else sin.numpy()
    if windowed:
        wks = np.zeros((B, Hkv, C + S, D), dtype=wk.dtype)
        wvs = np.zeros_like(wks)
        orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 1, cn, sn, wks, wvs)
        for b in range(B):
            n = lens["cache_past"][b] + S
            assert_bytes_equal(ks[b, :, :n], np.ascontiguousarray(wks[b, :, :n]), "k stage")
            assert_bytes_equal(vs[b, :, :n], np.ascontiguousarray(wvs[b, :, :n]), "v stage")
        rk, rv = wks, wvs
    else:
        orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 0, cn, sn)
        rk, rv = wk, wv
    assert_bytes_equal(gk, wk, "k cache")
    assert_bytes_equal(gv, wv, "v cache")
    qn = synth.bits(q)
    if sample is None:
        want, _ = orc.gqa_attention(qn, rk, rv, (lens["cache_past"] + S).astype(np.int32),
                                    lens["total_abs"], window=window, cos_cache=cn,
                                    sin_cache=sn)
        return assert_close(out, want, tol(dtype), "prefill")
    want = _oracle_queries(orc, qn, rk, rv, lens, S, window, cn, sn, sample)
    return assert_close(out[:, :, list(sample)], want, tol(dtype), "prefill sampled")


@pytest.mark.parametrize("D,g,S,W", [(256, 2, 64, 4096), (128, 4, 100, 300), (64, 1, 33, 0)])
def test_kv_split_and_unsplit(K, orc, D, g, S, W):
    """Small grids split each query block's keys over several CTAs (the
    partials merged by a second launch); the same case without a workspace
    runs unsplit.  Both match the oracle."""
    Hkv, B = 2, 2
    C = max(W, 2048)
    P = [C + 700, 37] if W else [C - S - 5, 37]
    for ws in ("auto", None):
        _chunk_case(K, orc, torch.bfloat16, B, Hkv * g, Hkv, D, C, S, P, W, 1 if W else 0,
                    True, 600 + D, workspace=ws)


def test_kv_split_is_used(K):
    # the small-chunk workload shape asks for a split, the full one does not
    assert K.library().kvc_gqa_prefill_workspace_size(8, 16, 8, 64, 4096 + 64, 256, 1, 4096) > 0
    assert K.library().kvc_gqa_prefill_workspace_size(8, 16, 8, 2048, 6144, 256, 1, 4096) == 0


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("g", [1, 2, 16])
def test_windowed_chunk_bf16(K, orc, D, g):
    Hkv = 2
    P = [0, 5, 64, 100, 300]
    _chunk_case(K, orc, torch.bfloat16, len(P), Hkv * g, Hkv, D, 128, 70, P, 96, 1, True,
                100 + D + g)


@pytest.mark.parametrize("g", [4, 8])
def test_contiguous_chunk_bf16(K, orc, g):
    P = [0, 1, 63, 200]
    _chunk_case(K, orc, torch.bfloat16, len(P), 2 * g, 2, 128, 400, 133, P, 0, 0, True, 200 + g)
    # a window narrower than the chunk on a contiguous cache
    _chunk_case(K, orc, torch.bfloat16, len(P), 2 * g, 2, 128, 400, 133, P, 40, 0, True, 300 + g)


def test_chunk_longer_than_capacity(K, orc):
    _chunk_case(K, orc, torch.bfloat16, 3, 4, 2, 64, 48, 150, [0, 10, 500], 48, 1, True, 400)


def test_chunk_fp16_and_fp32(K, orc):
    P = [0, 7, 90]
    _chunk_case(K, orc, torch.float16, len(P), 8, 4, 128, 96, 40, P, 96, 1, True, 500)
    _chunk_case(K, orc, torch.float32, len(P), 8, 4, 64, 96, 40, P, 96, 1, True, 501)
    _chunk_case(K, orc, torch.float32, len(P), 4, 2, 8, 128, 17, P, 0, 0, False, 502)


def test_consecutive_chunks_small_slack(K, orc):
    """Chunks of 32 on C = W + 8 (the gap is smaller than the chunk): every
    output, the stage and the cache are checked after each chunk."""
    B, Hq, Hkv, D, W = 2, 4, 2, 64, 40
    C = W + 8
    cos, sin = synth.rope_cache(1024, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    kc = torch.zeros(B, Hkv, C, D, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    gk, gv = kc.to(dev()), vc.to(dev())
    st = status()
    T = 0
    for step, S in enumerate([32, 32, 1, 32, 5, 32, 32]):
        nk = synth.normal((B, Hkv, S, D), 9, 10 + step)
        nv = synth.normal((B, Hkv, S, D), 9, 20 + step)
        q = synth.normal((B, Hq, S, D), 9, 30 + step)
        sk = np.full(B, T + S - 1, np.int32)
        L = K.kvc_seq_lengths(torch.from_numpy(sk).to(dev()), S, C, 1, local_window_size=W,
                              status=st)
        lens = orc.seq_lengths(sk, S, C, 1)
        out = torch.empty(B, Hq, S, D, dtype=torch.bfloat16, device=dev())
        if S == 1:
            K.kvc_window_append(gk, gv, nk.to(dev()), nv.to(dev()), L, 1, rope=rope_d, status=st)
            K.kvc_gqa_decode(out, q.to(dev()), gk, gv, L, local_window_size=W, rope=rope_d,
                             status=st)
            orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 1, cos.numpy(),
                              sin.numpy())
            want, _ = orc.gqa_attention(synth.bits(q), wk, wv, lens["cache_total"],
                                        lens["total_abs"], window=W, cos_cache=cos.numpy(),
                                        sin_cache=sin.numpy())
        else:
            ks = torch.empty(B, Hkv, C + S, D, dtype=torch.bfloat16, device=dev())
            vs = torch.empty_like(ks)
            K.kvc_window_append(gk, gv, nk.to(dev()), nv.to(dev()), L, 1, K.KVC_APPEND, ks, vs,
                                rope=rope_d, status=st)
            K.kvc_gqa_prefill_chunk(out, q.to(dev()), ks, vs, L, local_window_size=W,
                                    rope=rope_d, status=st)
            K.kvc_window_append(gk, gv, None, None, L, 1, K.KVC_COPY_BACK, ks, vs, rope=rope_d,
                                status=st)
            wks = np.zeros((B, Hkv, C + S, D), np.uint16)
            wvs = np.zeros_like(wks)
            orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 1, cos.numpy(),
                              sin.numpy(), wks, wvs)
            want, _ = orc.gqa_attention(synth.bits(q), wks, wvs,
                                        (lens["cache_past"] + S).astype(np.int32),
                                        lens["total_abs"], window=W, cos_cache=cos.numpy(),
                                        sin_cache=sin.numpy())
        torch.cuda.synchronize()
        assert_bytes_equal(gk, wk, f"k cache step {step}")
        assert_bytes_equal(gv, wv, f"v cache step {step}")
        assert_close(out, want, 2e-2, f"step {step}")
        T += S
    assert st.item() == 0


@pytest.mark.parametrize("S", [64, 512, 2048])
def test_window_prefill_workload_full_size(K, orc, S):
    w = synth.WINDOW_PREFILL
    P = synth.randint(w.total_lo, w.total_hi + 1, (w.batch,), 0, S).numpy()
    P[0], P[1] = 0, w.capacity - S // 2  # from zero, and a chunk that starts evicting
    rng = np.random.default_rng(S)
    # the chunk's ends and middle, the edges of the 64-query blocks (the
    # group of two heads fills the 128-row tile with 64 queries) and three
    # queries at random
    edges = {0, 63, 64, 127, 128, S // 2 - 1, S // 2, S - 1}
    sample = sorted({i for i in edges if i < S} | set(rng.integers(0, S, size=3).tolist()))
    err = _chunk_case(K, orc, torch.bfloat16, w.batch, w.q_heads, w.kv_heads, w.head_dim,
                      w.capacity, S, P, w.window, 1, True, 600 + S, sample=sample)
    assert err <= 2e-2
