"""Randomised GPU parity over the one-token decode entry points against the
oracle: seeded draws of head_dim {64, 128}, group {1..16}, capacities that
are not multiples of the 64-row tile, windows below a tile, totals at and
around the capacity and the window, for

* kvc_seq_lengths + kvc_window_append + kvc_gqa_decode (every policy),
* kvc_gqa_decode_ring after a ring append,
* kvc_paged_append + kvc_gqa_decode_paged,
* kvc_decode_step (contiguous and ring) and kvc_window_decode_step (every
  windowed policy, small windows);
* multi-token chunks (kvc_gqa_prefill_chunk over the stage or a contiguous
  cache, split and unsplit), sampled queries of every row;
* whole windowed steps through kvc_window_prefill_step (only hazardous rows
  staged), two in a row.

Every cache byte is compared; attention within 2e-2 (bf16/fp16).
"""
import numpy as np
import pytest
import torch

from _gpu_helpers import assert_bytes_equal, assert_close, dev, status
from persistent_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from persistent_kv_cache_gb300 import kvc
    return kvc


def _draw(rng, small_window_step=False):
    D = int(rng.choice([64, 128]))
    g = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
    Hkv = int(rng.integers(1, 4))
    B = int(rng.integers(1, 6))
    if small_window_step:
        C = int(rng.integers(2, 32768 // D + 1))
    else:
        C = int(rng.choice([int(rng.integers(2, 300)), int(rng.integers(300, 3000))]))
    W = int(rng.integers(1, C + 1))
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float16
    return D, g, Hkv, B, C, W, dtype


def _totals(rng, B, C, W, contiguous):
    cand = [1, 2, W, W + 1, C - 1, C, C + 1, 2 * C + 3, int(rng.integers(1, 5 * C + 2))]
    if contiguous:
        cand = [t for t in cand if 1 <= t <= C] + [int(rng.integers(1, C + 1))]
    cand = [t for t in cand if t >= 1]
    return np.array([cand[int(rng.integers(0, len(cand)))] for _ in range(B)], dtype=np.int64)


def _oracle_attention(orc, policy, q, wk, wv, lens, T, W, cos, sin):
    if policy == orc.RING:
        return orc.ring_attention(q, wk, wv, T, W, cos_cache=cos, sin_cache=sin)[0]
    return orc.gqa_attention(q, wk, wv, lens["cache_total"], lens["total_abs"], window=W,
                             cos_cache=cos, sin_cache=sin)[0]


@pytest.mark.parametrize("seed", range(12))
def test_fuzz_unfused_decode(K, orc, seed):
    rng = np.random.default_rng(7000 + seed)
    D, g, Hkv, B, C, W, dtype = _draw(rng)
    policy = int(rng.choice([0, 1, 2, 3]))
    Wd = W if policy else (0 if rng.random() < 0.5 else W)
    T = _totals(rng, B, C, W, policy == 0)
    Hq = Hkv * g
    cos, sin = synth.rope_cache(int(T.max()) + 1, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    kc = synth.normal((B, Hkv, C, D), seed, 1, dtype)
    vc = synth.normal((B, Hkv, C, D), seed, 2, dtype)
    nk = synth.normal((B, Hkv, 1, D), seed, 3, dtype)
    nv = synth.normal((B, Hkv, 1, D), seed, 4, dtype)
    q = synth.normal((B, Hq, 1, D), seed, 5, dtype)
    sk = torch.from_numpy((T - 1).astype(np.int32)).to(dev())
    gk, gv = kc.to(dev()), vc.to(dev())
    st = status()
    L = K.kvc_seq_lengths(sk, 1, C, policy, local_window_size=W if policy else 0, status=st)
    K.kvc_window_append(gk, gv, nk.to(dev()), nv.to(dev()), L, policy, rope=rope_d, status=st)
    out = torch.empty(B, Hq, 1, D, dtype=dtype, device=dev())
    if policy == K.KVC_RING:
        K.kvc_gqa_decode_ring(out, q.to(dev()), gk, gv, L, local_window_size=Wd, rope=rope_d,
                              status=st)
    else:
        K.kvc_gqa_decode(out, q.to(dev()), gk, gv, L, local_window_size=Wd, rope=rope_d,
                         status=st)
    torch.cuda.synchronize()
    assert st.item() == 0, (D, g, Hkv, B, C, W, policy, T)
    lens = orc.seq_lengths((T - 1).astype(np.int32), 1, C, policy, W)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    if policy == orc.RING:
        orc.ring_append(wk, wv, synth.bits(nk), synth.bits(nv), lens["past_abs"], cos.numpy(),
                        sin.numpy())
    else:
        orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 1 if policy else 0,
                          cos.numpy(), sin.numpy())
    assert_bytes_equal(gk, wk, f"k {(D, g, C, W, policy)}")
    assert_bytes_equal(gv, wv, f"v {(D, g, C, W, policy)}")
    want = _oracle_attention(orc, policy, synth.bits(q), wk, wv, lens, T, Wd, cos.numpy(),
                             sin.numpy())
    assert_close(out, want, 2e-2, f"decode {(D, g, Hkv, B, C, W, policy, T.tolist())}")


@pytest.mark.parametrize("seed", range(8))
def test_fuzz_fused_steps(K, orc, seed):
    rng = np.random.default_rng(7100 + seed)
    # kvc_decode_step: contiguous or ring, any capacity
    D, g, Hkv, B, C, W, dtype = _draw(rng)
    ring = rng.random() < 0.5
    Wd = W if (ring or rng.random() < 0.5) else 0
    T = _totals(rng, B, C, W, not ring)
    Hq = Hkv * g
    cos, sin = synth.rope_cache(int(T.max()) + 1, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    kc = synth.normal((B, Hkv, C, D), 50 + seed, 1, dtype)
    vc = synth.normal((B, Hkv, C, D), 50 + seed, 2, dtype)
    nk = synth.normal((B, Hkv, 1, D), 50 + seed, 3, dtype)
    nv = synth.normal((B, Hkv, 1, D), 50 + seed, 4, dtype)
    q = synth.normal((B, Hq, 1, D), 50 + seed, 5, dtype)
    sk = torch.from_numpy((T - 1).astype(np.int32)).to(dev())
    gk, gv = kc.to(dev()), vc.to(dev())
    st = status()
    out = torch.empty(B, Hq, 1, D, dtype=dtype, device=dev())
    K.kvc_decode_step(out, q.to(dev()), gk, gv, nk.to(dev()), nv.to(dev()), sk,
                      local_window_size=Wd, rope=rope_d, status=st,
                      windowed=K.KVC_RING if ring else K.KVC_CONTIGUOUS)
    torch.cuda.synchronize()
    assert st.item() == 0
    pol = orc.RING if ring else orc.CONTIGUOUS
    lens = orc.seq_lengths((T - 1).astype(np.int32), 1, C, pol, W)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    if ring:
        orc.ring_append(wk, wv, synth.bits(nk), synth.bits(nv), lens["past_abs"], cos.numpy(),
                        sin.numpy())
    else:
        orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 0, cos.numpy(),
                          sin.numpy())
    assert_bytes_equal(gk, wk, "step k")
    want = _oracle_attention(orc, pol, synth.bits(q), wk, wv, lens, T, Wd, cos.numpy(),
                             sin.numpy())
    assert_close(out, want, 2e-2, f"decode_step {(D, g, Hkv, B, C, W, ring, T.tolist())}")

    # kvc_window_decode_step: every windowed policy, windows that fit on chip
    D, g, Hkv, B, C, W, dtype = _draw(rng, small_window_step=True)
    policy = int(rng.choice([1, 2, 3]))
    T = _totals(rng, B, C, W, False)
    Hq = Hkv * g
    cos, sin = synth.rope_cache(int(T.max()) + 1, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    kc = synth.normal((B, Hkv, C, D), 60 + seed, 1, dtype)
    vc = synth.normal((B, Hkv, C, D), 60 + seed, 2, dtype)
    nk = synth.normal((B, Hkv, 1, D), 60 + seed, 3, dtype)
    nv = synth.normal((B, Hkv, 1, D), 60 + seed, 4, dtype)
    q = synth.normal((B, Hq, 1, D), 60 + seed, 5, dtype)
    sk = torch.from_numpy((T - 1).astype(np.int32)).to(dev())
    gk, gv = kc.to(dev()), vc.to(dev())
    out = torch.empty(B, Hq, 1, D, dtype=dtype, device=dev())
    K.kvc_window_decode_step(out, q.to(dev()), gk, gv, nk.to(dev()), nv.to(dev()), sk, W,
                             rope=rope_d, status=st, windowed=policy)
    torch.cuda.synchronize()
    assert st.item() == 0
    lens = orc.seq_lengths((T - 1).astype(np.int32), 1, C, policy, W)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    if policy == orc.RING:
        orc.ring_append(wk, wv, synth.bits(nk), synth.bits(nv), lens["past_abs"], cos.numpy(),
                        sin.numpy())
    else:
        orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 1, cos.numpy(),
                          sin.numpy())
    assert_bytes_equal(gk, wk, f"window step k {(D, g, C, W, policy, T.tolist())}")
    assert_bytes_equal(gv, wv, "window step v")
    want = _oracle_attention(orc, policy, synth.bits(q), wk, wv, lens, T, W, cos.numpy(),
                             sin.numpy())
    assert_close(out, want, 2e-2, f"window step {(D, g, Hkv, B, C, W, policy, T.tolist())}")


@pytest.mark.parametrize("seed", range(6))
def test_fuzz_paged(K, orc, seed):
    rng = np.random.default_rng(7200 + seed)
    D = int(rng.choice([64, 128]))
    g = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.integers(1, 3))
    B = int(rng.integers(1, 5))
    P = int(rng.choice([64, 128, 192]))
    max_pages = int(rng.integers(1, 12))
    C = P * max_pages
    W = int(rng.integers(0, C + 1))
    T = np.array([int(rng.integers(1, C + 1)) for _ in range(B)], dtype=np.int64)
    n_pool = B * max_pages + int(rng.integers(0, 4))
    table = rng.permutation(n_pool)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    Hq = Hkv * g
    cos, sin = synth.rope_cache(C + 1, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    kp = synth.normal((n_pool, Hkv, P, D), 70 + seed, 1)
    vp = synth.normal((n_pool, Hkv, P, D), 70 + seed, 2)
    nk = synth.normal((B, Hkv, 1, D), 70 + seed, 3)
    nv = synth.normal((B, Hkv, 1, D), 70 + seed, 4)
    q = synth.normal((B, Hq, 1, D), 70 + seed, 5)
    gk, gv = kp.to(dev()), vp.to(dev())
    tab = torch.from_numpy(table).to(dev())
    st = status()
    L = K.kvc_seq_lengths(torch.from_numpy((T - 1).astype(np.int32)).to(dev()), 1, C, 0,
                          status=st)
    K.kvc_paged_append(gk, gv, nk.to(dev()), nv.to(dev()), tab, L, rope=rope_d, status=st)
    out = torch.empty(B, Hq, 1, D, dtype=torch.bfloat16, device=dev())
    K.kvc_gqa_decode_paged(out, q.to(dev()), gk, gv, tab, L, local_window_size=W, rope=rope_d,
                           status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    wk, wv = synth.bits(kp).copy(), synth.bits(vp).copy()
    orc.paged_append(wk, wv, table, P, synth.bits(nk), synth.bits(nv), T - 1, cos.numpy(),
                     sin.numpy())
    assert_bytes_equal(gk, wk, "paged k")
    assert_bytes_equal(gv, wv, "paged v")
    want, _ = orc.paged_attention(synth.bits(q), wk, wv, table, P, T, T, W,
                                  cos_cache=cos.numpy(), sin_cache=sin.numpy())
    assert_close(out, want, 2e-2, f"paged {(D, g, Hkv, B, P, max_pages, W, T.tolist())}")


@pytest.mark.parametrize("seed", range(8))
def test_fuzz_prefill_chunks(K, orc, seed):
    """Random chunk steps: head_dim {64, 128, 256}, group {1, 2, 4, 8, 16},
    chunk lengths from 1 to past the capacity, contiguous / windowed /
    drifting caches, with and without the KV-split workspace."""
    rng = np.random.default_rng(7300 + seed)
    D = int(rng.choice([64, 128, 256]))
    g = int(rng.choice([1, 2, 4, 8, 16]))
    Hkv = int(rng.integers(1, 3))
    B = int(rng.integers(1, 4))
    policy = int(rng.choice([0, 1, 2]))
    C = int(rng.integers(64, 1500))
    W = int(rng.integers(1, C + 1))
    S = int(rng.choice([int(rng.integers(1, 40)), int(rng.integers(40, 300)), C + 5]))
    if policy:
        S = max(S, 2)  # a windowed one-token step compacts in place, with no stage
    if policy == 0:
        S = min(S, C - 1)
        P = np.array([int(rng.integers(0, C - S + 1)) for _ in range(B)], dtype=np.int64)
    else:
        P = np.array([int(rng.choice([0, int(rng.integers(0, 4 * C))])) for _ in range(B)],
                     dtype=np.int64)
    T = P + S
    Hq = Hkv * g
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float16
    ws = "auto" if rng.random() < 0.5 else None
    Wd = W if policy else (0 if rng.random() < 0.5 else W)
    cos, sin = synth.rope_cache(int(T.max()) + 1, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    kc = synth.normal((B, Hkv, C, D), 80 + seed, 1, dtype)
    vc = synth.normal((B, Hkv, C, D), 80 + seed, 2, dtype)
    nk = synth.normal((B, Hkv, S, D), 80 + seed, 3, dtype)
    nv = synth.normal((B, Hkv, S, D), 80 + seed, 4, dtype)
    q = synth.normal((B, Hq, S, D), 80 + seed, 5, dtype)
    sk = torch.from_numpy((T - 1).astype(np.int32)).to(dev())
    gk, gv = kc.to(dev()), vc.to(dev())
    st = status()
    L = K.kvc_seq_lengths(sk, S, C, policy, local_window_size=W if policy else 0, status=st)
    out = torch.empty(B, Hq, S, D, dtype=dtype, device=dev())
    if policy:
        ks = torch.full((B, Hkv, C + S, D), float("nan"), dtype=dtype, device=dev())
        vs = torch.full_like(ks, float("nan"))
        K.kvc_window_append(gk, gv, nk.to(dev()), nv.to(dev()), L, policy, K.KVC_APPEND, ks, vs,
                            rope=rope_d, status=st)
        K.kvc_gqa_prefill_chunk(out, q.to(dev()), ks, vs, L, local_window_size=Wd, rope=rope_d,
                                status=st, workspace=ws)
        K.kvc_window_append(gk, gv, None, None, L, policy, K.KVC_COPY_BACK, ks, vs, rope=rope_d,
                            status=st)
    else:
        K.kvc_window_append(gk, gv, nk.to(dev()), nv.to(dev()), L, 0, rope=rope_d, status=st)
        K.kvc_gqa_prefill_chunk(out, q.to(dev()), gk, gv, L, local_window_size=Wd, rope=rope_d,
                                status=st, workspace=ws)
    torch.cuda.synchronize()
    assert st.item() == 0, (D, g, Hkv, B, C, W, S, policy)
    lens = orc.seq_lengths((T - 1).astype(np.int32), S, C, policy, W)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    cn, sn = cos.numpy(), sin.numpy()
    if policy:
        wks = np.zeros((B, Hkv, C + S, D), dtype=wk.dtype)
        wvs = np.zeros_like(wks)
        orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 1, cn, sn, wks, wvs)
        rk, rv = wks, wvs
    else:
        orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 0, cn, sn)
        rk, rv = wk, wv
    assert_bytes_equal(gk, wk, "prefill k cache")
    assert_bytes_equal(gv, wv, "prefill v cache")
    # the last query and a few others of every row
    idx = sorted({0, S - 1, S // 2, int(rng.integers(0, S))})
    qb = synth.bits(q)
    for i in idx:
        qi = np.ascontiguousarray(qb[:, :, i:i + 1])
        # query i at P + i sees stage rows [0, Lp + i + 1)
        n = (lens["cache_past"] + i + 1).astype(np.int32)
        tot = (lens["past_abs"] + i + 1).astype(np.int32)
        want, _ = orc.gqa_attention(qi, rk, rv, n, tot, window=Wd, cos_cache=cn, sin_cache=sn)
        assert_close(out[:, :, i:i + 1], want, 2e-2,
                     f"prefill query {i} {(D, g, Hkv, B, C, W, S, policy, ws)}")


@pytest.mark.parametrize("seed", range(10))
def test_fuzz_window_prefill_step(K, orc, seed):
    """Random steps of kvc_window_prefill_step: head_dim {64, 128, 256},
    group {1, 2, 4, 8, 16}, windowed or drifting, capacities with and
    without slack above the window, chunks from 1 token to past the gap and
    the capacity, totals that fill, evict visibly and evict invisibly; two
    steps in a row, with and without the KV-split workspace."""
    rng = np.random.default_rng(9100 + seed)
    D = int(rng.choice([64, 128, 256]))
    g = int(rng.choice([1, 2, 4, 8, 16]))
    Hkv = int(rng.integers(1, 3))
    B = int(rng.integers(1, 5))
    policy = int(rng.choice([1, 2]))
    W = int(rng.integers(8, 600))
    C = W + int(rng.choice([0, int(rng.integers(1, 70)), int(rng.integers(70, 400))]))
    S = int(rng.choice([1, int(rng.integers(2, 20)), int(rng.integers(20, 200)), C + 3]))
    Hq = Hkv * g
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float16
    ws = "auto" if rng.random() < 0.5 else None
    T0 = np.array([int(rng.choice([0, int(rng.integers(0, C)), C - S // 2,
                                   int(rng.integers(C, 5 * C))])) for _ in range(B)])
    T0 = np.maximum(T0, 0)
    cos, sin = synth.rope_cache(int(T0.max()) + 2 * S + 2, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    cn, sn = cos.numpy(), sin.numpy()
    kc = synth.normal((B, Hkv, C, D), 90 + seed, 1, dtype)
    vc = synth.normal((B, Hkv, C, D), 90 + seed, 2, dtype)
    gk, gv = kc.to(dev()), vc.to(dev())
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    st = status()
    T = T0
    what = (D, g, Hkv, B, C, W, S, policy, ws, T0.tolist())
    for step in range(2):
        nk = synth.normal((B, Hkv, S, D), 90 + seed, 10 + step, dtype)
        nv = synth.normal((B, Hkv, S, D), 90 + seed, 20 + step, dtype)
        q = synth.normal((B, Hq, S, D), 90 + seed, 30 + step, dtype)
        sk = (T + S - 1).astype(np.int32)
        L = K.kvc_seq_lengths(torch.from_numpy(sk).to(dev()), S, C, policy,
                              local_window_size=W, status=st)
        ks = vs = None
        if S > 1:
            ks = torch.full((B, Hkv, C + S, D), float("nan"), dtype=dtype, device=dev())
            vs = torch.full_like(ks, float("nan"))
        out = torch.empty(B, Hq, S, D, dtype=dtype, device=dev())
        K.kvc_window_prefill_step(out, q.to(dev()), gk, gv, nk.to(dev()), nv.to(dev()), L,
                                  policy, W, ks, vs, rope=rope_d, status=st, workspace=ws)
        torch.cuda.synchronize()
        assert st.item() == 0, what
        lens = orc.seq_lengths(sk, S, C, policy, W)
        if S > 1:
            wks = np.zeros((B, Hkv, C + S, D), dtype=wk.dtype)
            wvs = np.zeros_like(wks)
            orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, policy, cn, sn, wks,
                              wvs)
            rk, rv = wks, wvs
        else:
            orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, policy, cn, sn)
            rk, rv = wk, wv
        assert_bytes_equal(gk, wk, f"step {step} k cache {what}")
        assert_bytes_equal(gv, wv, f"step {step} v cache {what}")
        qb = synth.bits(q)
        for i in sorted({0, S - 1, S // 2, int(rng.integers(0, S))}):
            if S > 1:
                n = (lens["cache_past"] + i + 1).astype(np.int32)
            else:
                n = lens["cache_total"]
            tot = (lens["past_abs"] + i + 1).astype(np.int32)
            want, _ = orc.gqa_attention(np.ascontiguousarray(qb[:, :, i:i + 1]), rk, rv, n, tot,
                                        window=W, cos_cache=cn, sin_cache=sn)
            assert_close(out[:, :, i:i + 1], want, 2e-2, f"step {step} query {i} {what}")
        T = T + S
