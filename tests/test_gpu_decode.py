"""GPU parity for kvc_gqa_decode (after kvc_seq_lengths + kvc_window_append)
against the oracle: max-abs error <= 2e-2 for bf16/fp16 and <= 1e-4 for fp32.

Covers the tiny fp32 scatter-then-decode workload, ragged lengths over
several TMA tiles and splits with partial tails, GQA groups 1..16, window
masks narrower than the resident rows, capacities whose rows need more
splits than the merge's fast path takes, the contiguous bf16 workload at full
size (32 x 32/8 heads x 128, capacity 8192, lengths U[512, 8192]; cache bytes
checked everywhere, attention sampled on several batch rows), the windowed
ring decode (64 x 64/8 x 64, C = W = 128) over consecutive one-token steps,
and a CUDA-graph capture of a whole step.
"""
import numpy as np
import pytest
import torch

from _gpu_helpers import assert_bytes_equal, assert_close, dev, lengths_np, status, tol
from persistent_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from persistent_kv_cache_gb300 import kvc
    return kvc


def test_tiny_f32_scatter_then_decode(K, orc):
    w = synth.TINY
    B, Hq, Hkv, D, C = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.capacity
    kc = torch.zeros(B, Hkv, C, D)
    vc = torch.zeros(B, Hkv, C, D)
    ku = synth.normal((B, Hkv, 1, D), 0, 1, torch.float32)
    vu = synth.normal((B, Hkv, 1, D), 0, 2, torch.float32)
    wi = synth.randint(0, C, (B,), 0, 3)
    q = synth.normal((B, Hq, 1, D), 0, 4, torch.float32)
    wk, _ = orc.tensor_scatter(kc.numpy(), ku.numpy(), wi.numpy())
    wv, _ = orc.tensor_scatter(vc.numpy(), vu.numpy(), wi.numpy())
    T = (wi.numpy() + 1).astype(np.int32)
    want, _ = orc.gqa_attention(q.numpy(), wk, wv, T, T)

    gk, gv = kc.to(dev()), vc.to(dev())
    K.kvc_tensor_scatter(gk, gk, ku.to(dev()), wi.to(dev()))
    K.kvc_tensor_scatter(gv, gv, vu.to(dev()), wi.to(dev()))
    st = status()
    L = K.kvc_seq_lengths(wi.to(dev()).to(torch.int32), 1, C, 0, status=st)
    out = torch.empty(B, Hq, 1, D, device=dev())
    K.kvc_gqa_decode(out, q.to(dev()), gk, gv, L, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert_bytes_equal(gk, wk, "k")
    assert_close(out, want, 1e-4, "tiny decode")


def _decode_case(K, orc, dtype, B, Hq, Hkv, D, C, T, window, windowed, rope, seed,
                 check_rows=None, untouched_check=False):
    """Append one token per row then decode; returns the max error."""
    T = np.asarray(T, dtype=np.int64)
    kc = synth.normal((B, Hkv, C, D), seed, 1, dtype)
    vc = synth.normal((B, Hkv, C, D), seed, 2, dtype)
    nk = synth.normal((B, Hkv, 1, D), seed, 3, dtype)
    nv = synth.normal((B, Hkv, 1, D), seed, 4, dtype)
    q = synth.normal((B, Hq, 1, D), seed, 5, dtype)
    cos = sin = None
    rope_d = None
    if rope:
        cos, sin = synth.rope_cache(int(T.max()) + 1, D)
        rope_d = (cos.to(dev()), sin.to(dev()))
    sk = (T - 1).astype(np.int32)
    st = status()
    gk, gv = kc.to(dev()), vc.to(dev())
    L = K.kvc_seq_lengths(torch.from_numpy(sk).to(dev()), 1, C, windowed,
                          local_window_size=window if windowed else 0, status=st)
    K.kvc_window_append(gk, gv, nk.to(dev()), nv.to(dev()), L, windowed, rope=rope_d, status=st)
    out = torch.full((B, Hq, 1, D), float("nan"), dtype=dtype, device=dev())
    K.kvc_gqa_decode(out, q.to(dev()), gk, gv, L, local_window_size=window, rope=rope_d,
                     status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    if untouched_check:
        # contiguous cache: only row T - 1 of every (b, head) may change
        ar = torch.arange(B, device=dev())
        idx = torch.from_numpy(T - 1).to(dev())
        for before, after in ((kc, gk), (vc, gv)):
            exp = before.to(dev())
            exp[ar, :, idx] = after[ar, :, idx]
            assert torch.equal(exp, after)
            del exp
    rows = list(range(B)) if check_rows is None else list(check_rows)
    lens = orc.seq_lengths(sk[rows], 1, C, windowed)
    wk = synth.bits(kc[rows]).copy()
    wv = synth.bits(vc[rows]).copy()
    cn = None if cos is None else cos.numpy()
    sn = None if sin is None else sin.numpy()
    orc.window_append(wk, wv, synth.bits(nk[rows]), synth.bits(nv[rows]), lens, windowed, cn, sn)
    assert_bytes_equal(gk[rows], wk, "k cache rows")
    assert_bytes_equal(gv[rows], wv, "v cache rows")
    want, _ = orc.gqa_attention(synth.bits(q[rows]), wk, wv, lens["cache_total"],
                                lens["total_abs"], window=window, cos_cache=cn, sin_cache=sn)
    return assert_close(out[rows], want, tol(dtype), "decode")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("g", [1, 4, 8])
def test_contiguous_ragged(K, orc, dtype, D, g):
    Hkv = 2
    T = [1, 2, 63, 64, 65, 130, 200, 256]
    _decode_case(K, orc, dtype, len(T), Hkv * g, Hkv, D, 256, T, 0, 0, True, 10 + g)


@pytest.mark.parametrize("g", [2, 16])
def test_multi_split_with_window(K, orc, g):
    """capacity >= 2048 uses 512-row splits merged by the combine pass; the
    window cuts the visible range at an unaligned row."""
    T = [1, 511, 512, 513, 1500, 2048, 3000, 4096]
    for window in (0, 700, 64, 1):
        _decode_case(K, orc, torch.bfloat16, len(T), 2 * g, 2, 128, 4096, T, window, 0, True,
                     20 + window)


@pytest.mark.parametrize("g", [1, 2, 16])
def test_head_dim_256_multi_split(K, orc, g):
    """head_dim 256 (tiles in a ring of three 32 KB slots, the query's
    fragments read from shared memory): 512-row splits merged by the
    combine pass, windows cutting rows at unaligned places."""
    T = [1, 63, 64, 65, 511, 513, 2048, 4096]
    for window in (0, 4096, 700, 1):
        for dtype in (torch.bfloat16, torch.float16):
            _decode_case(K, orc, dtype, len(T), 2 * g, 2, 256, 4096, T, window, 0, True,
                         50 + window + g)


def test_more_splits_than_the_fast_merge(K, orc):
    """capacity 12288 (512-row splits, up to 24 a row): the merge takes its
    general path; rows with one split, 16, 17 and 24, with and without a
    window."""
    T = [1, 512, 8192, 8193, 9000, 12288]
    for window in (0, 5000):
        _decode_case(K, orc, torch.bfloat16, len(T), 8, 2, 128, 12288, T, window, 0, True,
                     40 + window)


def test_windowed_cache_decode(K, orc):
    T = [1, 5, 127, 128, 129, 4000, 32768]
    for dtype in (torch.bfloat16, torch.float32):
        _decode_case(K, orc, dtype, len(T), 16, 2, 64, 128, T, 128, 1, True, 30)


def test_contiguous_workload_full_size(K, orc):
    """32 x 32/8 heads x 128, capacity 8192, T ~ U[512, 8192] (bf16); the
    appended row of every (b, head) and the attention of every batch row and
    head are checked against the oracle; every other cache byte must be
    unchanged."""
    w = synth.CONTIG_DECODE
    T = synth.randint(w.total_lo, w.total_hi + 1, (w.batch,), 0, 77).numpy()
    T[0], T[1] = w.total_lo, w.total_hi
    err = _decode_case(K, orc, torch.bfloat16, w.batch, w.q_heads, w.kv_heads, w.head_dim,
                       w.capacity, T, 0, 0, True, 40, untouched_check=True)
    assert err < 2e-2


def test_window_ring_consecutive_steps(K, orc):
    """64 x 64/8 x 64, C = W = 128, starting totals U[1, 32768], consecutive
    one-token steps with in-place compaction; the whole cache is compared
    every step and the attention every fourth step."""
    w = synth.WINDOW_DECODE
    B, Hq, Hkv, D, C, W = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.capacity, w.window
    steps = 24
    T0 = synth.randint(w.total_lo, w.total_hi + 1, (B,), 0, 1).numpy()
    T0[:3] = [1, 127, 128]
    cos, sin = synth.rope_cache(int(T0.max()) + steps + 1, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    kc = synth.normal((B, Hkv, C, D), 2, 1)
    vc = synth.normal((B, Hkv, C, D), 2, 2)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    gk, gv = kc.to(dev()), vc.to(dev())
    st = status()
    out = torch.empty(B, Hq, 1, D, dtype=torch.bfloat16, device=dev())
    ws = K.decode_workspace(out, gk)
    for s in range(steps):
        T = T0 + s
        sk = (T - 1).astype(np.int32)
        nk = synth.normal((B, Hkv, 1, D), 3, s)
        nv = synth.normal((B, Hkv, 1, D), 4, s)
        q = synth.normal((B, Hq, 1, D), 5, s)
        L = K.kvc_seq_lengths(torch.from_numpy(sk).to(dev()), 1, C, 1, local_window_size=W,
                              status=st)
        K.kvc_window_append(gk, gv, nk.to(dev()), nv.to(dev()), L, 1, rope=rope_d, status=st)
        K.kvc_gqa_decode(out, q.to(dev()), gk, gv, L, local_window_size=W, rope=rope_d,
                         workspace=ws, status=st)
        lens = orc.seq_lengths(sk, 1, C, 1)
        orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 1, cos.numpy(),
                          sin.numpy())
        torch.cuda.synchronize()
        assert_bytes_equal(gk, wk, f"k step {s}")
        assert_bytes_equal(gv, wv, f"v step {s}")
        if s % 4 == 3:
            want, _ = orc.gqa_attention(synth.bits(q), wk, wv, lens["cache_total"],
                                        lens["total_abs"], window=W, cos_cache=cos.numpy(),
                                        sin_cache=sin.numpy())
            assert_close(out, want, 2e-2, f"decode step {s}")
    assert st.item() == 0


def test_graph_captured_step(K, orc):
    """lengths + append + decode captured once in a CUDA graph and replayed:
    no host synchronisation or host read inside any call."""
    B, Hq, Hkv, D, C = 4, 16, 4, 128, 4096
    T = np.array([100, 700, 2500, 4096])
    kc = synth.normal((B, Hkv, C, D), 6, 1)
    vc = synth.normal((B, Hkv, C, D), 6, 2)
    nk = synth.normal((B, Hkv, 1, D), 6, 3)
    nv = synth.normal((B, Hkv, 1, D), 6, 4)
    q = synth.normal((B, Hq, 1, D), 6, 5)
    cos, sin = synth.rope_cache(C, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    gk, gv, gq, gnk, gnv = (t.to(dev()) for t in (kc, vc, q, nk, nv))
    sk = torch.from_numpy((T - 1).astype(np.int32)).to(dev())
    out = torch.empty(B, Hq, 1, D, dtype=torch.bfloat16, device=dev())
    ws = K.decode_workspace(out, gk)
    L = K.Lengths(B, dev())
    st = status()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            K.kvc_seq_lengths(sk, 1, C, 0, out=L, status=st)
            K.kvc_window_append(gk, gv, gnk, gnv, L, 0, rope=rope_d, status=st)
            K.kvc_gqa_decode(out, gq, gk, gv, L, rope=rope_d, workspace=ws, status=st)
    graph.replay()
    graph.replay()  # re-appending the same row is idempotent
    torch.cuda.synchronize()
    assert st.item() == 0
    lens = orc.seq_lengths((T - 1).astype(np.int32), 1, C, 0)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 0, cos.numpy(), sin.numpy())
    want, _ = orc.gqa_attention(synth.bits(q), wk, wv, lens["cache_total"], lens["total_abs"],
                                cos_cache=cos.numpy(), sin_cache=sin.numpy())
    assert_bytes_equal(gk, wk, "k")
    assert_close(out, want, 2e-2, "graph decode")


# --------------------------------------------------------------------------
# fused one-token step on a windowed cache (kvc_window_decode_step)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("D,g", [(64, 8), (128, 4), (128, 16)])
def test_window_step_fused_consecutive(K, orc, D, g):
    """Consecutive fused steps on a C = W cache: every cache byte and the
    written lengths match the oracle after each step, the attention every
    third step (window rows 1, 127, 128, 129 and long totals included)."""
    B, Hkv, C = 6, 2, 128
    W = C
    Hq = Hkv * g
    T0 = np.array([1, 127, 128, 129, 700, 30000])
    steps = 9
    cos, sin = synth.rope_cache(int(T0.max()) + steps + 1, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    kc = synth.normal((B, Hkv, C, D), 50 + D, 1)
    vc = synth.normal((B, Hkv, C, D), 50 + D, 2)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    gk, gv = kc.to(dev()), vc.to(dev())
    st = status()
    out = torch.empty(B, Hq, 1, D, dtype=torch.bfloat16, device=dev())
    Lg = K.Lengths(B, dev())
    for s in range(steps):
        T = T0 + s
        sk = (T - 1).astype(np.int32)
        nk = synth.normal((B, Hkv, 1, D), 51, s)
        nv = synth.normal((B, Hkv, 1, D), 52, s)
        q = synth.normal((B, Hq, 1, D), 53, s)
        K.kvc_window_decode_step(out, q.to(dev()), gk, gv, nk.to(dev()), nv.to(dev()),
                                 torch.from_numpy(sk).to(dev()), W, lengths=Lg, rope=rope_d,
                                 status=st)
        lens = orc.seq_lengths(sk, 1, C, 1)
        orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 1, cos.numpy(),
                          sin.numpy())
        torch.cuda.synchronize()
        assert_bytes_equal(gk, wk, f"k step {s}")
        assert_bytes_equal(gv, wv, f"v step {s}")
        got_len = lengths_np(Lg)
        for f in Lg.FIELDS:
            np.testing.assert_array_equal(got_len[f], lens[f], err_msg=f)
        if s % 3 == 2:
            want, _ = orc.gqa_attention(synth.bits(q), wk, wv, lens["cache_total"],
                                        lens["total_abs"], window=W, cos_cache=cos.numpy(),
                                        sin_cache=sin.numpy())
            assert_close(out, want, 2e-2, f"fused step {s}")
    assert st.item() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_window_step_fused_matches_unfused(K, orc, dtype):
    """Window narrower than the capacity (W = 90 < C = 200): the fused step
    and lengths + append + decode produce the same cache bytes and outputs
    within the attention tolerance."""
    B, Hq, Hkv, D, C, W = 5, 16, 4, 128, 200, 90
    T = np.array([1, 90, 150, 200, 5000])
    sk = torch.from_numpy((T - 1).astype(np.int32)).to(dev())
    cos, sin = synth.rope_cache(int(T.max()) + 1, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    kc = synth.normal((B, Hkv, C, D), 60, 1, dtype).to(dev())
    vc = synth.normal((B, Hkv, C, D), 60, 2, dtype).to(dev())
    nk = synth.normal((B, Hkv, 1, D), 60, 3, dtype).to(dev())
    nv = synth.normal((B, Hkv, 1, D), 60, 4, dtype).to(dev())
    q = synth.normal((B, Hq, 1, D), 60, 5, dtype).to(dev())
    st = status()
    k1, v1 = kc.clone(), vc.clone()
    o1 = torch.empty(B, Hq, 1, D, dtype=dtype, device=dev())
    K.kvc_window_decode_step(o1, q, k1, v1, nk, nv, sk, W, rope=rope_d, status=st)
    k2, v2 = kc.clone(), vc.clone()
    o2 = torch.empty_like(o1)
    L = K.kvc_seq_lengths(sk, 1, C, 1, local_window_size=W, status=st)
    K.kvc_window_append(k2, v2, nk, nv, L, 1, rope=rope_d, status=st)
    K.kvc_gqa_decode(o2, q, k2, v2, L, local_window_size=W, rope=rope_d, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    lens = orc.seq_lengths((T - 1).astype(np.int32), 1, C, 1)
    wk, wv = synth.bits(kc.cpu()).copy(), synth.bits(vc.cpu()).copy()
    orc.window_append(wk, wv, synth.bits(nk.cpu()), synth.bits(nv.cpu()), lens, 1, cos.numpy(),
                      sin.numpy())
    want, _ = orc.gqa_attention(synth.bits(q.cpu()), wk, wv, lens["cache_total"],
                                lens["total_abs"], window=W, cos_cache=cos.numpy(),
                                sin_cache=sin.numpy())
    assert_close(o1, want, 2e-2, "fused vs oracle")


def test_window_step_fused_rejects_bad_rows(K, orc):
    B, Hq, Hkv, D, C = 3, 8, 2, 64, 64
    sk = torch.tensor([-1, 10, 2**31 - 1], dtype=torch.int32, device=dev())
    kc = synth.normal((B, Hkv, C, D), 61, 1).to(dev())
    vc = synth.normal((B, Hkv, C, D), 61, 2).to(dev())
    before_k, before_v = kc.clone(), vc.clone()
    nk = synth.normal((B, Hkv, 1, D), 61, 3).to(dev())
    nv = synth.normal((B, Hkv, 1, D), 61, 4).to(dev())
    q = synth.normal((B, Hq, 1, D), 61, 5).to(dev())
    out = torch.zeros(B, Hq, 1, D, dtype=torch.bfloat16, device=dev())
    Lg = K.Lengths(B, dev())
    st = status()
    K.kvc_window_decode_step(out, q, kc, vc, nk, nv, sk, C, lengths=Lg, status=st)
    torch.cuda.synchronize()
    assert st.item() == K.KVC_DEV_SEQLEN_RANGE
    for b in (0, 2):
        assert torch.equal(kc[b], before_k[b]) and torch.equal(vc[b], before_v[b])
        assert (Lg.buf[:, b] == -1).all()
    assert not torch.equal(kc[1], before_k[1])
