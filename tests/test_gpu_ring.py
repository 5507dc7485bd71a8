"""GPU parity for ring-buffer addressing ("Stateful decode & KV cache",
"Sliding-window ring buffer": token p in slot p mod C, nothing moves)
against the oracle's ring_append / ring_attention.

* consecutive one-token steps through kvc_seq_lengths(KVC_RING) +
  kvc_window_append(KVC_RING) + kvc_gqa_decode_ring, and through the fused
  kvc_window_decode_step(KVC_RING): lengths and every slot byte after each
  step, attention within 2e-2 (bf16), for W = C and W < C, rows before the
  ring fills and far past it;
* a 4096-slot ring decoded with several splits, the visible range wrapping
  inside a split and inside a 64-row tile, with and without a window;
* a ring written by kvc_tensor_scatter in circular mode (the pairing the
  ring-buffer page describes) and read by kvc_gqa_decode_ring;
* multi-token ring appends, chunks longer than the ring included;
* the fp32 path.
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


def _steps(K, orc, fused, B, g, Hkv, D, C, W, T0, steps, seed):
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
    for s in range(steps):
        T = T0 + s
        sk = (T - 1).astype(np.int32)
        skd = torch.from_numpy(sk).to(dev())
        nk = synth.normal((B, Hkv, 1, D), seed + 1, s)
        nv = synth.normal((B, Hkv, 1, D), seed + 2, s)
        q = synth.normal((B, Hq, 1, D), seed + 3, s)
        if fused:
            K.kvc_window_decode_step(out, q.to(dev()), gk, gv, nk.to(dev()), nv.to(dev()), skd,
                                     W, lengths=Lg, rope=rope_d, status=st, windowed=K.KVC_RING)
        else:
            K.kvc_seq_lengths(skd, 1, C, K.KVC_RING, local_window_size=W, out=Lg, status=st)
            K.kvc_window_append(gk, gv, nk.to(dev()), nv.to(dev()), Lg, K.KVC_RING, rope=rope_d,
                                status=st)
            K.kvc_gqa_decode_ring(out, q.to(dev()), gk, gv, Lg, local_window_size=W,
                                  rope=rope_d, status=st)
        lens = orc.seq_lengths(sk, 1, C, orc.RING, W)
        orc.ring_append(wk, wv, synth.bits(nk), synth.bits(nv), T - 1, cos.numpy(), sin.numpy())
        torch.cuda.synchronize()
        got_len = lengths_np(Lg)
        for f in Lg.FIELDS:
            np.testing.assert_array_equal(got_len[f], lens[f], err_msg=f"{f} step {s}")
        assert_bytes_equal(gk, wk, f"k step {s}")
        assert_bytes_equal(gv, wv, f"v step {s}")
        want, _ = orc.ring_attention(synth.bits(q), wk, wv, T, W, cos_cache=cos.numpy(),
                                     sin_cache=sin.numpy())
        assert_close(out, want, 2e-2, f"{'fused' if fused else 'unfused'} step {s}")
    assert st.item() == 0


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("D,g,C,W", [(64, 8, 128, 128), (128, 4, 128, 100), (64, 16, 96, 40),
                                     (256, 2, 128, 128), (256, 8, 64, 50)])
def test_ring_one_token_steps(K, orc, fused, D, g, C, W):
    T0 = [1, C - 2, C, C + 1, 700, 30001]
    _steps(K, orc, fused, len(T0), g, 2, D, C, W, T0, 5, 110 + D + C + fused)


@pytest.mark.parametrize("W", [0, 3000])
def test_ring_large_splits(K, orc, W):
    """C = 4096 (512-row splits): totals chosen so the visible run wraps at
    slot C inside a split, inside a tile, at a tile edge, or not at all."""
    B, Hkv, g, D, C = 6, 2, 4, 128, 4096
    Hq = Hkv * g
    T = np.array([4096 + 200, 4096 + 64, 4096 * 3 + 1000, 17, 4096, 9000 + 33])
    cos, sin = synth.rope_cache(int(T.max()) + 1, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    kc = synth.normal((B, Hkv, C, D), 120, 1)
    vc = synth.normal((B, Hkv, C, D), 120, 2)
    q = synth.normal((B, Hq, 1, D), 120, 3)
    sk = torch.from_numpy((T - 1).astype(np.int32)).to(dev())
    st = status()
    L = K.kvc_seq_lengths(sk, 1, C, K.KVC_RING, local_window_size=W or C, status=st)
    out = torch.empty(B, Hq, 1, D, dtype=torch.bfloat16, device=dev())
    K.kvc_gqa_decode_ring(out, q.to(dev()), kc.to(dev()), vc.to(dev()), L, local_window_size=W,
                          rope=rope_d, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    want, _ = orc.ring_attention(synth.bits(q), synth.bits(kc), synth.bits(vc), T, W,
                                 cos_cache=cos.numpy(), sin_cache=sin.numpy())
    assert_close(out, want, 2e-2, "ring splits")


def test_ring_written_by_tensor_scatter(K, orc):
    """TensorScatter circular at write index P fills the ring; the ring decode
    reads it (no RoPE on either side)."""
    B, Hkv, g, D, C = 4, 2, 2, 64, 64
    Hq = Hkv * g
    kc = torch.zeros(B, Hkv, C, D, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    gk, gv = kc.to(dev()), vc.to(dev())
    st = status()
    T = np.array([0, 5, 63, 200], dtype=np.int64)
    for step, S in enumerate([7, 1, 1, 30, 1, 64, 1]):
        uk = synth.normal((B, Hkv, S, D), 130, step)
        uv = synth.normal((B, Hkv, S, D), 131, step)
        wi = torch.from_numpy(T.copy())
        K.kvc_tensor_scatter(gk, gk, uk.to(dev()), wi.to(dev()), mode=K.KVC_CIRCULAR, status=st)
        K.kvc_tensor_scatter(gv, gv, uv.to(dev()), wi.to(dev()), mode=K.KVC_CIRCULAR, status=st)
        orc.tensor_scatter(wk, synth.bits(uk), T, mode=orc.CIRCULAR, out=wk)
        orc.tensor_scatter(wv, synth.bits(uv), T, mode=orc.CIRCULAR, out=wv)
        T = T + S
        q = synth.normal((B, Hq, 1, D), 132, step)
        sk = torch.from_numpy((T - 1).astype(np.int32)).to(dev())
        L = K.kvc_seq_lengths(sk, 1, C, K.KVC_RING, local_window_size=C, status=st)
        out = torch.empty(B, Hq, 1, D, dtype=torch.bfloat16, device=dev())
        K.kvc_gqa_decode_ring(out, q.to(dev()), gk, gv, L, local_window_size=C, status=st)
        torch.cuda.synchronize()
        assert_bytes_equal(gk, wk, f"k step {step}")
        want, _ = orc.ring_attention(synth.bits(q), wk, wv, T, C)
        assert_close(out, want, 2e-2, f"scatter ring step {step}")
    assert st.item() == 0


def test_ring_chunk_appends(K, orc):
    """kvc_window_append(KVC_RING) with S > 1, including S > C (only the
    last C rows survive), every slot byte against the oracle."""
    B, Hkv, D, C = 3, 2, 128, 16
    cos, sin = synth.rope_cache(512, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    kc = synth.normal((B, Hkv, C, D), 140, 1)
    vc = synth.normal((B, Hkv, C, D), 140, 2)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    gk, gv = kc.to(dev()), vc.to(dev())
    st = status()
    T = np.array([0, 9, 100], dtype=np.int64)
    for step, S in enumerate([5, 16, 1, 19, 40, 3]):
        nk = synth.normal((B, Hkv, S, D), 141, step)
        nv = synth.normal((B, Hkv, S, D), 142, step)
        sk = torch.from_numpy((T + S - 1).astype(np.int32)).to(dev())
        L = K.kvc_seq_lengths(sk, S, C, K.KVC_RING, local_window_size=C, status=st)
        K.kvc_window_append(gk, gv, nk.to(dev()), nv.to(dev()), L, K.KVC_RING, rope=rope_d,
                            status=st)
        orc.ring_append(wk, wv, synth.bits(nk), synth.bits(nv), T, cos.numpy(), sin.numpy())
        torch.cuda.synchronize()
        assert_bytes_equal(gk, wk, f"k step {step} S={S}")
        assert_bytes_equal(gv, wv, f"v step {step} S={S}")
        T = T + S
    assert st.item() == 0


def test_ring_f32(K, orc):
    B, Hkv, g, D, C, W = 3, 2, 2, 32, 24, 10
    Hq = Hkv * g
    T = np.array([5, 24, 77])
    cos, sin = synth.rope_cache(128, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    kc = synth.normal((B, Hkv, C, D), 150, 1, torch.float32)
    vc = synth.normal((B, Hkv, C, D), 150, 2, torch.float32)
    q = synth.normal((B, Hq, 1, D), 150, 3, torch.float32)
    st = status()
    sk = torch.from_numpy((T - 1).astype(np.int32)).to(dev())
    for w in (0, W):
        L = K.kvc_seq_lengths(sk, 1, C, K.KVC_RING, local_window_size=C, status=st)
        out = torch.empty(B, Hq, 1, D, device=dev())
        K.kvc_gqa_decode_ring(out, q.to(dev()), kc.to(dev()), vc.to(dev()), L,
                              local_window_size=w, rope=rope_d, status=st)
        torch.cuda.synchronize()
        want, _ = orc.ring_attention(q.numpy(), kc.numpy(), vc.numpy(), T, w,
                                     cos_cache=cos.numpy(), sin_cache=sin.numpy())
        assert_close(out, want, 1e-4, f"f32 ring W={w}")
    assert st.item() == 0
