"""GPU parity for kvc_window_append_inplace: the C + S staging step with the
stage held in the cache's own rows (no seed copy; the copy-back is an in-place
shift), against the oracle's staged append and attention ("GQA support
sliding_window_cache", "Design").

* consecutive chunks of mixed sizes (1, 5, 32, 37, 200 and chunks longer than
  the capacity) on windowed and drifting caches, rows starting at different
  totals, every scratch row NaN at the start: rows [0, L) byte for byte after
  every step and every output against the oracle;
* the windowed chunked-prefill workload at full size (8 x 16/8 heads x 256,
  C = W = 4096, P ~ U[0, 20000], S in {64, 512}): rows [0, L) equal the
  oracle's and the staged pair's byte for byte, and the outputs equal the
  staged flow's bit for bit (the same attention kernel over the same rows);
* rows rejected by the lengths or by the RoPE range move nothing.
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


def _rows_equal(rows, cache_bits, lens, what):
    """Rows [0, L_b) of the in-place buffer against the oracle's cache."""
    for b in range(rows.shape[0]):
        n = int(lens["cache_total"][b])
        if n <= 0:
            continue
        assert_bytes_equal(rows[b, :, :n], np.ascontiguousarray(cache_bits[b, :, :n]),
                           f"{what} row {b}")


@pytest.mark.parametrize("policy,C,W", [(1, 256, 200), (2, 256, 200), (1, 96, 96)])
def test_consecutive_chunks(K, orc, policy, C, W):
    B, Hq, Hkv, D = 3, 8, 2, 64
    schedule = [37, 1, 200, 5, C + 44, 32, 1, 96, C + 7]
    R = C + max(schedule)
    cos, sin = synth.rope_cache(8192, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    cn, sn = cos.numpy(), sin.numpy()
    T = np.array([0, 50, 700], dtype=np.int64)
    # the cache a row starts with: rows [0, C) random (the oracle's cache of C rows)
    kc = synth.normal((B, Hkv, C, D), 40 + policy, 1)
    vc = synth.normal((B, Hkv, C, D), 40 + policy, 2)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    rows_k = torch.full((B, Hkv, R, D), float("nan"), dtype=torch.bfloat16, device=dev())
    rows_v = torch.full_like(rows_k, float("nan"))
    rows_k[:, :, :C] = kc.to(dev())
    rows_v[:, :, :C] = vc.to(dev())
    st = status()
    for step, S in enumerate(schedule):
        nk = synth.normal((B, Hkv, S, D), 41, step)
        nv = synth.normal((B, Hkv, S, D), 42, step)
        q = synth.normal((B, Hq, S, D), 43, step)
        sk = (T + S - 1).astype(np.int32)
        L = K.kvc_seq_lengths(torch.from_numpy(sk).to(dev()), S, C, policy, local_window_size=W,
                              status=st)
        lens = orc.seq_lengths(sk, S, C, policy, W)
        K.kvc_window_append_inplace(rows_k, rows_v, nk.to(dev()), nv.to(dev()), L, C, policy,
                                    K.KVC_APPEND, rope=rope_d, status=st)
        out = torch.full((B, Hq, S, D), float("nan"), dtype=torch.bfloat16, device=dev())
        K.kvc_gqa_prefill_chunk(out, q.to(dev()), rows_k, rows_v, L, local_window_size=W,
                                rope=rope_d, status=st)
        K.kvc_window_append_inplace(rows_k, rows_v, None, None, L, C, policy, K.KVC_COPY_BACK,
                                    new_tokens=S, rope=rope_d, status=st)
        if S == 1:
            orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 1, cn, sn)
            want, _ = orc.gqa_attention(synth.bits(q), wk, wv, lens["cache_total"],
                                        lens["total_abs"], window=W, cos_cache=cn, sin_cache=sn)
        else:
            wks = np.zeros((B, Hkv, C + S, D), np.uint16)
            wvs = np.zeros_like(wks)
            orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, 1, cn, sn, wks, wvs)
            want, _ = orc.gqa_attention(synth.bits(q), wks, wvs,
                                        (lens["cache_past"] + S).astype(np.int32),
                                        lens["total_abs"], window=W, cos_cache=cn, sin_cache=sn)
        torch.cuda.synchronize()
        assert st.item() == 0, (step, st.item())
        _rows_equal(rows_k, wk, lens, f"k step {step}")
        _rows_equal(rows_v, wv, lens, f"v step {step}")
        assert_close(out, want, 2e-2, f"step {step}")
        T = T + S


@pytest.mark.parametrize("S", [64, 512])
def test_window_prefill_workload_full_size(K, orc, S):
    w = synth.WINDOW_PREFILL
    B, Hq, Hkv, D, C, W = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.capacity, w.window
    P = synth.randint(w.total_lo, w.total_hi + 1, (B,), 0, S).numpy()
    P[0], P[1] = 0, C - S // 2
    T = P + S
    kc = synth.normal((B, Hkv, C, D), 700 + S, 1)
    vc = synth.normal((B, Hkv, C, D), 700 + S, 2)
    nk = synth.normal((B, Hkv, S, D), 700 + S, 3).to(dev())
    nv = synth.normal((B, Hkv, S, D), 700 + S, 4).to(dev())
    q = synth.normal((B, Hq, S, D), 700 + S, 5).to(dev())
    cos, sin = synth.rope_cache(int(T.max()) + 1, D, w.theta)
    rope_d = (cos.to(dev()), sin.to(dev()))
    sk = torch.from_numpy((T - 1).astype(np.int32)).to(dev())
    st = status()
    L = K.kvc_seq_lengths(sk, S, C, K.KVC_WINDOWED, local_window_size=W, status=st)
    # the staged pair on a copy
    gk, gv = kc.to(dev()), vc.to(dev())
    ks = torch.empty(B, Hkv, C + S, D, dtype=torch.bfloat16, device=dev())
    vs = torch.empty_like(ks)
    K.kvc_window_append(gk, gv, nk, nv, L, K.KVC_WINDOWED, K.KVC_APPEND, ks, vs, rope=rope_d,
                        status=st)
    o_staged = torch.empty(B, Hq, S, D, dtype=torch.bfloat16, device=dev())
    K.kvc_gqa_prefill_chunk(o_staged, q, ks, vs, L, local_window_size=W, rope=rope_d, status=st)
    K.kvc_window_append(gk, gv, None, None, L, K.KVC_WINDOWED, K.KVC_COPY_BACK, ks, vs,
                        rope=rope_d, status=st)
    # in place
    rows_k = torch.full((B, Hkv, C + S, D), float("nan"), dtype=torch.bfloat16, device=dev())
    rows_v = torch.full_like(rows_k, float("nan"))
    rows_k[:, :, :C] = kc.to(dev())
    rows_v[:, :, :C] = vc.to(dev())
    K.kvc_window_append_inplace(rows_k, rows_v, nk, nv, L, C, K.KVC_WINDOWED, K.KVC_APPEND,
                                rope=rope_d, status=st)
    o_inplace = torch.full_like(o_staged, float("nan"))
    K.kvc_gqa_prefill_chunk(o_inplace, q, rows_k, rows_v, L, local_window_size=W, rope=rope_d,
                            status=st)
    K.kvc_window_append_inplace(rows_k, rows_v, None, None, L, C, K.KVC_WINDOWED,
                                K.KVC_COPY_BACK, new_tokens=S, rope=rope_d, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(o_inplace, o_staged), "outputs differ from the staged flow"
    lens = orc.seq_lengths((T - 1).astype(np.int32), S, C, 1, W)
    Lh = lens["cache_total"]
    for b in range(B):
        n = int(Lh[b])
        assert torch.equal(rows_k[b, :, :n], gk[b, :, :n]), f"k rows {b}"
        assert torch.equal(rows_v[b, :, :n], gv[b, :, :n]), f"v rows {b}"
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    wks = np.zeros((B, Hkv, C + S, D), np.uint16)
    wvs = np.zeros_like(wks)
    orc.window_append(wk, wv, synth.bits(nk.cpu()), synth.bits(nv.cpu()), lens, 1, cos.numpy(),
                      sin.numpy(), wks, wvs)
    _rows_equal(rows_k, wk, lens, "k")
    _rows_equal(rows_v, wv, lens, "v")


def test_rejected_rows_move_nothing(K, orc):
    B, Hq, Hkv, D, C, W, S = 4, 4, 2, 64, 128, 128, 16
    R = C + S
    rows_k = synth.normal((B, Hkv, R, D), 50, 1).to(dev())
    rows_v = synth.normal((B, Hkv, R, D), 50, 2).to(dev())
    before_k, before_v = rows_k.clone(), rows_v.clone()
    nk = synth.normal((B, Hkv, S, D), 50, 3).to(dev())
    nv = synth.normal((B, Hkv, S, D), 50, 4).to(dev())
    # row 0: seqlens_k < S - 1 is not a valid total; row 2 runs past the rope table
    T = np.array([5, 300, 900, 40])
    sk = (T - 1).astype(np.int32)
    sk[0] = -2
    cos, sin = synth.rope_cache(600, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    st = status()
    L = K.kvc_seq_lengths(torch.from_numpy(sk).to(dev()), S, C, K.KVC_WINDOWED,
                          local_window_size=W, status=st)
    K.kvc_window_append_inplace(rows_k, rows_v, nk, nv, L, C, K.KVC_WINDOWED, K.KVC_APPEND,
                                rope=rope_d, status=st)
    K.kvc_window_append_inplace(rows_k, rows_v, None, None, L, C, K.KVC_WINDOWED,
                                K.KVC_COPY_BACK, new_tokens=S, rope=rope_d, status=st)
    torch.cuda.synchronize()
    assert st.item() == K.KVC_DEV_SEQLEN_RANGE | K.KVC_DEV_ROPE_RANGE
    for b in (0, 2):
        assert torch.equal(rows_k[b], before_k[b]) and torch.equal(rows_v[b], before_v[b]), b
    for b in (1, 3):
        assert not torch.equal(rows_k[b], before_k[b]), b
