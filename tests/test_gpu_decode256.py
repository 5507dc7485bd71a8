"""GPU parity for one-token decode at head_dim 256 on the windowed-prefill
workload's cache (8 batch rows, 16 query / 8 KV heads, head_dim 256,
C = W = 4096; "GQA support sliding_window_cache", "Design": a windowed cache
alternates multi-token chunks through the C + S stage with one-token steps
over the same buffer).

* a 64-token chunk through the stage (seed, chunk attention, copy-back),
  then one-token steps (lengths, in-place compaction, split decode), under
  the compact-every-step layout (C = W) and the drifting layout
  (C = W + 64): every length, every cache byte after every call, and the
  attention of every batch row and head against the oracle (max-abs 2e-2);
* the fused one-token step (kvc_decode_step) on the same heads as a ring of
  C = W = 4096 slots and as a contiguous cache of 8192 rows.
Past lengths are drawn from U[0, 20000] as the workload's are, with the
edges (an empty cache, a cache one chunk short of full, one exactly full)
forced on three rows.
"""
import numpy as np
import pytest
import torch

from _gpu_helpers import assert_bytes_equal, assert_close, dev, lengths_np, status
from persistent_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from persistent_kv_cache_gb300 import kvc
    return kvc


def _check_lengths(L, lens, what):
    got = lengths_np(L)
    for f in L.FIELDS:
        np.testing.assert_array_equal(got[f], lens[f], err_msg=f"{what}: {f}")


@pytest.mark.parametrize("policy", ["windowed", "drifting"])
def test_chunk_then_one_token_steps(K, orc, policy):
    w = synth.WINDOW_PREFILL
    B, Hq, Hkv, D, W = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.window
    pol = K.KVC_WINDOWED if policy == "windowed" else K.KVC_DRIFTING
    opol = orc.WINDOWED if policy == "windowed" else orc.DRIFTING
    C = w.capacity if policy == "windowed" else w.capacity + 64
    S, steps = 64, 3
    seed = 256 + pol
    P = synth.randint(0, w.total_hi + 1, (B,), seed, 1).numpy()
    P[:3] = [0, C - S, C]
    cos, sin = synth.rope_cache(int(P.max()) + S + steps + 1, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    cn, sn = cos.numpy(), sin.numpy()
    kc = synth.normal((B, Hkv, C, D), seed, 2)
    vc = synth.normal((B, Hkv, C, D), seed, 3)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    gk, gv = kc.to(dev()), vc.to(dev())
    del kc, vc
    st = status()

    # the chunk through the stage
    nk = synth.normal((B, Hkv, S, D), seed, 4)
    nv = synth.normal((B, Hkv, S, D), seed, 5)
    q = synth.normal((B, Hq, S, D), seed, 6)
    sk = (P + S - 1).astype(np.int32)
    L = K.kvc_seq_lengths(torch.from_numpy(sk).to(dev()), S, C, pol, local_window_size=W,
                          status=st)
    ks = torch.empty(B, Hkv, C + S, D, dtype=torch.bfloat16, device=dev())
    vs = torch.empty_like(ks)
    out = torch.empty(B, Hq, S, D, dtype=torch.bfloat16, device=dev())
    K.kvc_window_append(gk, gv, nk.to(dev()), nv.to(dev()), L, pol, K.KVC_APPEND, ks, vs,
                        rope=rope_d, status=st)
    K.kvc_gqa_prefill_chunk(out, q.to(dev()), ks, vs, L, local_window_size=W, rope=rope_d,
                            status=st)
    K.kvc_window_append(gk, gv, None, None, L, pol, K.KVC_COPY_BACK, ks, vs, rope=rope_d,
                        status=st)
    lens = orc.seq_lengths(sk, S, C, opol, W)
    wks = np.zeros((B, Hkv, C + S, D), np.uint16)
    wvs = np.zeros_like(wks)
    orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 1, cn, sn, wks, wvs)
    del wks, wvs, ks, vs
    torch.cuda.synchronize()
    _check_lengths(L, lens, "chunk")
    assert_bytes_equal(gk, wk, "k cache after the chunk")
    assert_bytes_equal(gv, wv, "v cache after the chunk")
    P = P + S

    # one-token steps over the same cache
    out1 = torch.full((B, Hq, 1, D), float("nan"), dtype=torch.bfloat16, device=dev())
    for s in range(steps):
        nk = synth.normal((B, Hkv, 1, D), seed, 10 + s)
        nv = synth.normal((B, Hkv, 1, D), seed, 20 + s)
        q = synth.normal((B, Hq, 1, D), seed, 30 + s)
        sk = P.astype(np.int32)
        L = K.kvc_seq_lengths(torch.from_numpy(sk).to(dev()), 1, C, pol, local_window_size=W,
                              out=L, status=st)
        K.kvc_window_append(gk, gv, nk.to(dev()), nv.to(dev()), L, pol, rope=rope_d, status=st)
        K.kvc_gqa_decode(out1, q.to(dev()), gk, gv, L, local_window_size=W, rope=rope_d,
                         status=st)
        lens = orc.seq_lengths(sk, 1, C, opol, W)
        orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 1, cn, sn)
        want, _ = orc.gqa_attention(synth.bits(q), wk, wv, lens["cache_total"],
                                    lens["total_abs"], window=W, cos_cache=cn, sin_cache=sn)
        torch.cuda.synchronize()
        _check_lengths(L, lens, f"step {s}")
        assert_bytes_equal(gk, wk, f"k cache step {s}")
        assert_bytes_equal(gv, wv, f"v cache step {s}")
        assert_close(out1, want, 2e-2, f"{policy} decode step {s}")
        P = P + 1
    assert st.item() == 0


@pytest.mark.parametrize("ring", [True, False])
def test_fused_step_head_dim_256(K, orc, ring):
    w = synth.WINDOW_PREFILL
    B, Hq, Hkv, D = w.batch, w.q_heads, w.kv_heads, w.head_dim
    C = 4096 if ring else 8192
    W = 4096 if ring else 0
    seed = 300 + int(ring)
    T = synth.randint(1, (w.total_hi if ring else C) + 1, (B,), seed, 1).numpy()
    T[:3] = [1, C - 1, C]
    steps = 2 if ring else 1   # a contiguous cache of C rows holds T <= C only
    cos, sin = synth.rope_cache(int(T.max()) + steps + 1, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    cn, sn = cos.numpy(), sin.numpy()
    kc = synth.normal((B, Hkv, C, D), seed, 2)
    vc = synth.normal((B, Hkv, C, D), seed, 3)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    gk, gv = kc.to(dev()), vc.to(dev())
    del kc, vc
    st = status()
    Lg = K.Lengths(B, dev())
    out = torch.full((B, Hq, 1, D), float("nan"), dtype=torch.bfloat16, device=dev())
    pol = K.KVC_RING if ring else K.KVC_CONTIGUOUS
    for s in range(steps):
        Ts = T + s
        sk = (Ts - 1).astype(np.int32)
        nk = synth.normal((B, Hkv, 1, D), seed, 10 + s)
        nv = synth.normal((B, Hkv, 1, D), seed, 20 + s)
        q = synth.normal((B, Hq, 1, D), seed, 30 + s)
        K.kvc_decode_step(out, q.to(dev()), gk, gv, nk.to(dev()), nv.to(dev()),
                          torch.from_numpy(sk).to(dev()), W, lengths=Lg, rope=rope_d, status=st,
                          windowed=pol)
        if ring:
            lens = orc.seq_lengths(sk, 1, C, orc.RING, W)
            orc.ring_append(wk, wv, synth.bits(nk), synth.bits(nv), Ts - 1, cn, sn)
            want, _ = orc.ring_attention(synth.bits(q), wk, wv, Ts, W, cos_cache=cn,
                                         sin_cache=sn)
        else:
            lens = orc.seq_lengths(sk, 1, C, 0)
            orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 0, cn, sn)
            want, _ = orc.gqa_attention(synth.bits(q), wk, wv, lens["cache_total"],
                                        lens["total_abs"], cos_cache=cn, sin_cache=sn)
        torch.cuda.synchronize()
        _check_lengths(Lg, lens, f"step {s}")
        assert_bytes_equal(gk, wk, f"k cache step {s}")
        assert_bytes_equal(gv, wv, f"v cache step {s}")
        assert_close(out, want, 2e-2, f"{'ring' if ring else 'contiguous'} step {s}")
    assert st.item() == 0


@pytest.mark.parametrize("policy,D,g,C,W,own_len", [
    (1, 256, 2, 4096, 4096, True),     # the windowed-prefill workload's cache, compact every step
    (2, 256, 2, 4160, 4096, False),    # drifting, 65-row blocks
    (3, 256, 2, 4096, 4096, True),     # ring
    (1, 128, 4, 1024, 1000, False),
    (2, 64, 8, 2048, 2000, True),
])
def test_large_window_step(K, orc, policy, D, g, C, W, own_len):
    """kvc_window_decode_step above the on-chip limit (capacity * head_dim >
    32768): lengths, compaction and split decode for a windowed or drifting
    cache, the fused split step for a ring; lengths kept by the caller or in
    the call's workspace."""
    B, Hkv = 6, 2
    Hq = Hkv * g
    seed = 500 + policy + D
    T0 = np.array([1, C - 2, C, C + 1, 9000, 20000], dtype=np.int64)
    steps = 4 if policy != 2 else C - W + 3   # a drifting run passes a compaction
    steps = min(steps, 8)
    cos, sin = synth.rope_cache(int(T0.max()) + steps + 1, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    cn, sn = cos.numpy(), sin.numpy()
    kc = synth.normal((B, Hkv, C, D), seed, 1)
    vc = synth.normal((B, Hkv, C, D), seed, 2)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    gk, gv = kc.to(dev()), vc.to(dev())
    st = status()
    Lg = K.Lengths(B, dev()) if own_len else None
    out = torch.full((B, Hq, 1, D), float("nan"), dtype=torch.bfloat16, device=dev())
    for s in range(steps):
        T = T0 + s
        sk = (T - 1).astype(np.int32)
        nk = synth.normal((B, Hkv, 1, D), seed, 10 + s)
        nv = synth.normal((B, Hkv, 1, D), seed, 20 + s)
        q = synth.normal((B, Hq, 1, D), seed, 30 + s)
        K.kvc_window_decode_step(out, q.to(dev()), gk, gv, nk.to(dev()), nv.to(dev()),
                                 torch.from_numpy(sk).to(dev()), W, lengths=Lg, rope=rope_d,
                                 status=st, windowed=policy)
        lens = orc.seq_lengths(sk, 1, C, policy, W)
        if policy == 3:
            orc.ring_append(wk, wv, synth.bits(nk), synth.bits(nv), T - 1, cn, sn)
            want, _ = orc.ring_attention(synth.bits(q), wk, wv, T, W, cos_cache=cn, sin_cache=sn)
        else:
            orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, policy, cn, sn)
            want, _ = orc.gqa_attention(synth.bits(q), wk, wv, lens["cache_total"],
                                        lens["total_abs"], window=W, cos_cache=cn, sin_cache=sn)
        torch.cuda.synchronize()
        if Lg is not None:
            _check_lengths(Lg, lens, f"step {s}")
        assert_bytes_equal(gk, wk, f"k cache step {s}")
        assert_bytes_equal(gv, wv, f"v cache step {s}")
        assert_close(out, want, 2e-2, f"policy {policy} step {s}")
    assert st.item() == 0
