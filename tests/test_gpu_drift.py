"""GPU parity for the drifting windowed layout (the sliding-window PR's CPU
commit: gap = C - W + 1, resident rows [0, end(T)), a whole gap-sized block
reclaimed once every gap one-token steps) against the oracle.

* one-token steps through kvc_seq_lengths + kvc_window_append +
  kvc_gqa_decode and through the fused kvc_window_decode_step, on C = W + 8
  over more than three gaps, rows starting before the window fills, at the
  capacity and far past it: lengths and every cache byte after each step,
  attention within 2e-2 (bf16) on every step that compacts and every fourth
  one otherwise;
* a large gap (C = 256, W = 56, so 201 rows leave at once and the surviving
  55 rows do not overlap their old places);
* 32-token chunks at C = W + 8 (the gap is smaller than the chunk: the
  chunk stages from a drifted append point), interleaved with one-token
  steps;
* the three windowed decode workloads the benchmark times (compact every
  step, drifting, ring) at full size through the fused step.
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


def _one_token_run(K, orc, fused, B, g, Hkv, D, C, W, T0, steps, seed):
    Hq = Hkv * g
    T0 = np.asarray(T0, dtype=np.int64)
    cos, sin = synth.rope_cache(int(T0.max()) + steps + 1, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    kc = synth.normal((B, Hkv, C, D), seed, 1)
    vc = synth.normal((B, Hkv, C, D), seed, 2)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    gk, gv = kc.to(dev()), vc.to(dev())
    st = status()
    out = torch.empty(B, Hq, 1, D, dtype=torch.bfloat16, device=dev())
    Lg = K.Lengths(B, dev())
    compactions = 0
    for s in range(steps):
        T = T0 + s
        sk = (T - 1).astype(np.int32)
        skd = torch.from_numpy(sk).to(dev())
        nk = synth.normal((B, Hkv, 1, D), seed + 1, s)
        nv = synth.normal((B, Hkv, 1, D), seed + 2, s)
        q = synth.normal((B, Hq, 1, D), seed + 3, s)
        if fused:
            K.kvc_window_decode_step(out, q.to(dev()), gk, gv, nk.to(dev()), nv.to(dev()), skd,
                                     W, lengths=Lg, rope=rope_d, status=st,
                                     windowed=K.KVC_DRIFTING)
        else:
            K.kvc_seq_lengths(skd, 1, C, K.KVC_DRIFTING, local_window_size=W, out=Lg, status=st)
            K.kvc_window_append(gk, gv, nk.to(dev()), nv.to(dev()), Lg, K.KVC_DRIFTING,
                                rope=rope_d, status=st)
            K.kvc_gqa_decode(out, q.to(dev()), gk, gv, Lg, local_window_size=W, rope=rope_d,
                             status=st)
        lens = orc.seq_lengths(sk, 1, C, orc.DRIFTING, W)
        orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 1, cos.numpy(),
                          sin.numpy())
        torch.cuda.synchronize()
        got_len = lengths_np(Lg)
        for f in Lg.FIELDS:
            np.testing.assert_array_equal(got_len[f], lens[f], err_msg=f"{f} step {s}")
        assert_bytes_equal(gk, wk, f"k step {s}")
        assert_bytes_equal(gv, wv, f"v step {s}")
        compacting = bool((lens["evict"] > 0).any())
        compactions += int((lens["evict"] > 0).sum())
        if compacting or s % 4 == 3:
            want, _ = orc.gqa_attention(synth.bits(q), wk, wv, lens["cache_total"],
                                        lens["total_abs"], window=W, cos_cache=cos.numpy(),
                                        sin_cache=sin.numpy())
            assert_close(out, want, 2e-2, f"{'fused' if fused else 'unfused'} step {s}")
    assert st.item() == 0
    return compactions


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("D,g", [(64, 8), (128, 4), (256, 2)])
def test_drift_one_token_steps(K, orc, fused, D, g):
    W = 120
    C = W + 8
    # before the window fills, at the capacity, past it, far past it
    T0 = [1, 119, 127, 128, 129, 700, 30000]
    n = _one_token_run(K, orc, fused, len(T0), g, 2, D, C, W, T0, 30, 70 + D + fused)
    assert n >= 3 * (len(T0) - 2)   # several compactions on every row that passes C


@pytest.mark.parametrize("fused", [False, True])
def test_drift_large_gap(K, orc, fused):
    """gap = 201: the surviving rows move farther than their own extent."""
    W, C = 56, 256
    T0 = [250, 256, 257, 5000]
    n = _one_token_run(K, orc, fused, len(T0), 4, 2, 128, C, W, T0, 12, 90 + fused)
    assert n >= 2


def test_drift_chunks_small_slack(K, orc):
    """32-token chunks at C = W + 8 with one-token steps between them: the
    stage, the copy-back and the prefill attention under the drifting
    lengths."""
    B, Hq, Hkv, D, W = 2, 8, 2, 128, 40
    C = W + 8
    cos, sin = synth.rope_cache(1024, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    kc = torch.zeros(B, Hkv, C, D, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    gk, gv = kc.to(dev()), vc.to(dev())
    st = status()
    T = np.array([0, 3], dtype=np.int64)
    for step, S in enumerate([32, 32, 1, 1, 1, 32, 5, 1, 32, 32, 1]):
        nk = synth.normal((B, Hkv, S, D), 11, 10 + step)
        nv = synth.normal((B, Hkv, S, D), 11, 40 + step)
        q = synth.normal((B, Hq, S, D), 11, 70 + step)
        sk = (T + S - 1).astype(np.int32)
        L = K.kvc_seq_lengths(torch.from_numpy(sk).to(dev()), S, C, K.KVC_DRIFTING,
                              local_window_size=W, status=st)
        lens = orc.seq_lengths(sk, S, C, orc.DRIFTING, W)
        out = torch.empty(B, Hq, S, D, dtype=torch.bfloat16, device=dev())
        if S == 1:
            K.kvc_window_append(gk, gv, nk.to(dev()), nv.to(dev()), L, K.KVC_DRIFTING,
                                rope=rope_d, status=st)
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
            K.kvc_window_append(gk, gv, nk.to(dev()), nv.to(dev()), L, K.KVC_DRIFTING,
                                K.KVC_APPEND, ks, vs, rope=rope_d, status=st)
            K.kvc_gqa_prefill_chunk(out, q.to(dev()), ks, vs, L, local_window_size=W,
                                    rope=rope_d, status=st)
            K.kvc_window_append(gk, gv, None, None, L, K.KVC_DRIFTING, K.KVC_COPY_BACK, ks, vs,
                                rope=rope_d, status=st)
            wks = np.zeros((B, Hkv, C + S, D), np.uint16)
            wvs = np.zeros_like(wks)
            orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 1, cos.numpy(),
                              sin.numpy(), wks, wvs)
            want, _ = orc.gqa_attention(synth.bits(q), wks, wvs,
                                        (lens["cache_past"] + S).astype(np.int32),
                                        lens["total_abs"], window=W, cos_cache=cos.numpy(),
                                        sin_cache=sin.numpy())
        torch.cuda.synchronize()
        got_len = lengths_np(L)
        for f in L.FIELDS:
            np.testing.assert_array_equal(got_len[f], lens[f], err_msg=f"{f} step {step}")
        assert_bytes_equal(gk, wk, f"k cache step {step}")
        assert_bytes_equal(gv, wv, f"v cache step {step}")
        assert_close(out, want, 2e-2, f"step {step}")
        T += S
    assert st.item() == 0


@pytest.mark.parametrize("spec", ["WINDOW_DECODE", "WINDOW_DECODE_DRIFT", "WINDOW_DECODE_RING"])
def test_fused_window_workloads_full_size(K, orc, spec):
    """The three windowed decode workloads bench.py times (64 x 64/8 heads x
    64, W = 128; C = 128 compact-every-step, C = 144 drifting, C = 128 ring)
    at full size through the fused step, 20 consecutive steps from starting
    totals U[1, 32768]: every cache byte and the lengths after each step, the
    attention every fifth step and on every step where some row compacts."""
    w = getattr(synth, spec)
    policy = w.extra.get("policy", 1)
    B, Hq, Hkv, D, C, W = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.capacity, w.window
    steps = 20
    T0 = synth.randint(w.total_lo, w.total_hi + 1, (B,), 11, 1).numpy()
    T0[:4] = [1, W - 1, C, C + 1]
    cos, sin = synth.rope_cache(int(T0.max()) + steps + 1, D, w.theta)
    rope_d = (cos.to(dev()), sin.to(dev()))
    kc = synth.normal((B, Hkv, C, D), 12, 1)
    vc = synth.normal((B, Hkv, C, D), 12, 2)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    gk, gv = kc.to(dev()), vc.to(dev())
    st = status()
    out = torch.empty(B, Hq, 1, D, dtype=torch.bfloat16, device=dev())
    Lg = K.Lengths(B, dev())
    for s in range(steps):
        T = T0 + s
        sk = (T - 1).astype(np.int32)
        nk = synth.normal((B, Hkv, 1, D), 13, s)
        nv = synth.normal((B, Hkv, 1, D), 14, s)
        q = synth.normal((B, Hq, 1, D), 15, s)
        K.kvc_window_decode_step(out, q.to(dev()), gk, gv, nk.to(dev()), nv.to(dev()),
                                 torch.from_numpy(sk).to(dev()), W, lengths=Lg, rope=rope_d,
                                 status=st, windowed=policy)
        lens = orc.seq_lengths(sk, 1, C, policy, W)
        if policy == orc.RING:
            orc.ring_append(wk, wv, synth.bits(nk), synth.bits(nv), lens["past_abs"],
                            cos.numpy(), sin.numpy())
        else:
            orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 1, cos.numpy(),
                              sin.numpy())
        torch.cuda.synchronize()
        got_len = lengths_np(Lg)
        for f in Lg.FIELDS:
            np.testing.assert_array_equal(got_len[f], lens[f], err_msg=f"{f} step {s}")
        assert_bytes_equal(gk, wk, f"k step {s}")
        assert_bytes_equal(gv, wv, f"v step {s}")
        compacting = policy != orc.RING and bool((lens["evict"] > 0).any())
        if s % 5 == 4 or (policy == orc.DRIFTING and compacting):
            if policy == orc.RING:
                want, _ = orc.ring_attention(synth.bits(q), wk, wv, T, W, cos_cache=cos.numpy(),
                                             sin_cache=sin.numpy())
            else:
                want, _ = orc.gqa_attention(synth.bits(q), wk, wv, lens["cache_total"],
                                            lens["total_abs"], window=W, cos_cache=cos.numpy(),
                                            sin_cache=sin.numpy())
            assert_close(out, want, 2e-2, f"{spec} step {s}")
    assert st.item() == 0


def test_window_workload_256_steps_against_full_history(K, orc):
    """The windowed decode workload as stated (64 x 64/8 heads x 64, C = W =
    128, starting totals U[1, 32768], 256 consecutive one-token steps with
    in-place compaction) through the fused step, checked against attention
    over the full history: the cache starts as the rotated last min(T0, C)
    tokens of a per-row history, every new token is appended to that
    history, and the attention of the final step and of every 32nd step is
    compared with the attention over the whole history under the window
    mask (with the cache bytes against the oracle's compaction on every
    step)."""
    w = synth.WINDOW_DECODE
    B, Hq, Hkv, D, C, W = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.capacity, w.window
    steps = 256
    T0 = synth.randint(w.total_lo, w.total_hi + 1, (B,), 21, 1).numpy()
    T0[:3] = [1, C - 1, C]
    cos, sin = synth.rope_cache(int(T0.max()) + steps + 1, D, w.theta)
    cn, sn = cos.numpy(), sin.numpy()
    # per-row history of the last C tokens before the run (rotated K, V),
    # stored in the cache at [0, min(T0, C)); the rest of the cache is noise
    n0 = np.minimum(T0, C)
    hk = synth.bits(synth.normal((B, Hkv, C, D), 22, 1))
    hv = synth.bits(synth.normal((B, Hkv, C, D), 22, 2))
    kc = synth.bits(synth.normal((B, Hkv, C, D), 22, 3)).copy()
    vc = synth.bits(synth.normal((B, Hkv, C, D), 22, 4)).copy()
    hist_k = [[None] * 0 for _ in range(B)]
    hist_v = [[None] * 0 for _ in range(B)]
    for b in range(B):
        pos = np.arange(T0[b] - n0[b], T0[b])
        rk = orc.rope_rows(np.ascontiguousarray(hk[b, :, :n0[b]]),
                           np.tile(pos, Hkv), cn, sn).reshape(Hkv, n0[b], D)
        kc[b, :, :n0[b]] = rk
        vc[b, :, :n0[b]] = hv[b, :, :n0[b]]
        hist_k[b] = [rk[:, j] for j in range(n0[b])]
        hist_v[b] = [hv[b, :, j] for j in range(n0[b])]
    wk, wv = kc.copy(), vc.copy()
    gk = synth.from_bits(kc, torch.bfloat16).to(dev())
    gv = synth.from_bits(vc, torch.bfloat16).to(dev())
    rope_d = (cos.to(dev()), sin.to(dev()))
    st = status()
    out = torch.empty(B, Hq, 1, D, dtype=torch.bfloat16, device=dev())
    for s in range(steps):
        T = T0 + s + 1
        sk = (T - 1).astype(np.int32)
        nk = synth.normal((B, Hkv, 1, D), 23, s)
        nv = synth.normal((B, Hkv, 1, D), 24, s)
        q = synth.normal((B, Hq, 1, D), 25, s)
        K.kvc_window_decode_step(out, q.to(dev()), gk, gv, nk.to(dev()), nv.to(dev()),
                                 torch.from_numpy(sk).to(dev()), W, rope=rope_d, status=st)
        lens = orc.seq_lengths(sk, 1, C, orc.WINDOWED, W)
        orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 1, cn, sn)
        nkr = orc.rope_rows(synth.bits(nk)[:, :, 0], np.repeat(T - 1, Hkv), cn, sn)
        for b in range(B):
            hist_k[b].append(nkr[b])
            hist_v[b].append(synth.bits(nv)[b, :, 0])
        torch.cuda.synchronize()
        assert_bytes_equal(gk, wk, f"k step {s}")
        if s % 32 == 31 or s == steps - 1:
            # the full history's last W tokens are all a window can see
            n = np.minimum(W, [len(h) for h in hist_k])
            fk = np.zeros((B, Hkv, W, D), np.uint16)
            fv = np.zeros_like(fk)
            for b in range(B):
                fk[b, :, :n[b]] = np.stack(hist_k[b][-n[b]:], axis=1)
                fv[b, :, :n[b]] = np.stack(hist_v[b][-n[b]:], axis=1)
            want, _ = orc.gqa_attention(synth.bits(q), fk, fv, n.astype(np.int32),
                                        T.astype(np.int32), window=W, cos_cache=cn,
                                        sin_cache=sn)
            assert_close(out, want, 2e-2, f"step {s} against the full history")
    assert st.item() == 0
