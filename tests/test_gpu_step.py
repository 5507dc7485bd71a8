"""GPU parity for kvc_decode_step (lengths + one-token append + split decode
in one launch, plus the split merge) against the oracle.

* the contiguous decode workload at full size (32 x 32/8 heads x 128,
  capacity 8192, totals U[512, 8192]): every cache byte and the lengths,
  attention on sampled batch rows, and agreement with the unfused
  lengths + append + decode calls;
* consecutive steps sharing one workspace, also replayed from a CUDA graph;
* a 4096-slot ring wrapping inside splits, windows narrower than the rows,
  fp16 and head_dim 64;
* rejected rows (bad seqlens_k, a contiguous total beyond the capacity)
  leave their rows untouched, set the status bits and -1 lengths, and the
  next call on the same workspace is still right.
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


def _oracle_step(orc, ring, kc_bits, vc_bits, nk, nv, q, T, C, W, cos, sin, rows=None):
    """Append in place into the oracle's copies; attention for `rows`."""
    sk = (np.asarray(T) - 1).astype(np.int32)
    lens = orc.seq_lengths(sk, 1, C, orc.RING if ring else orc.CONTIGUOUS, W if W > 0 else C)
    if ring:
        orc.ring_append(kc_bits, vc_bits, synth.bits(nk), synth.bits(nv), lens["past_abs"], cos,
                        sin)
    else:
        orc.window_append(kc_bits, vc_bits, synth.bits(nk), synth.bits(nv), lens, 0, cos, sin)
    rows = list(range(len(T))) if rows is None else list(rows)
    qb = synth.bits(q)[rows]
    if ring:
        want, _ = orc.ring_attention(qb, kc_bits[rows], vc_bits[rows], np.asarray(T)[rows], W,
                                     cos_cache=cos, sin_cache=sin)
    else:
        want, _ = orc.gqa_attention(qb, kc_bits[rows], vc_bits[rows], lens["cache_total"][rows],
                                    lens["total_abs"][rows], window=W, cos_cache=cos,
                                    sin_cache=sin)
    return lens, want


def test_contiguous_workload_full_size(K, orc):
    w = synth.CONTIG_DECODE
    B, Hq, Hkv, D, C = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.capacity
    T = synth.randint(w.total_lo, w.total_hi + 1, (B,), 7, 1).numpy()
    T[:3] = [w.total_lo, C, 513]
    cos, sin = synth.rope_cache(C + 1, D, w.theta)
    rope_d = (cos.to(dev()), sin.to(dev()))
    kc = synth.normal((B, Hkv, C, D), 7, 2)
    vc = synth.normal((B, Hkv, C, D), 7, 3)
    nk = synth.normal((B, Hkv, 1, D), 7, 4)
    nv = synth.normal((B, Hkv, 1, D), 7, 5)
    q = synth.normal((B, Hq, 1, D), 7, 6)
    sk = torch.from_numpy((T - 1).astype(np.int32)).to(dev())
    st = status()
    gk, gv = kc.to(dev()), vc.to(dev())
    k2, v2 = gk.clone(), gv.clone()
    Lg = K.Lengths(B, dev())
    out = torch.full((B, Hq, 1, D), float("nan"), dtype=torch.bfloat16, device=dev())
    K.kvc_decode_step(out, q.to(dev()), gk, gv, nk.to(dev()), nv.to(dev()), sk, lengths=Lg,
                      rope=rope_d, status=st)
    # the unfused calls on a copy
    o2 = torch.empty_like(out)
    L2 = K.kvc_seq_lengths(sk, 1, C, K.KVC_CONTIGUOUS, status=st)
    K.kvc_window_append(k2, v2, nk.to(dev()), nv.to(dev()), L2, K.KVC_CONTIGUOUS, rope=rope_d,
                        status=st)
    K.kvc_gqa_decode(o2, q.to(dev()), k2, v2, L2, rope=rope_d, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(gk, k2) and torch.equal(gv, v2)
    assert (out.float() - o2.float()).abs().max().item() <= 2e-2
    rows = list(range(B))   # every batch row and head
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    lens, want = _oracle_step(orc, False, wk, wv, nk, nv, q, T, C, 0, cos.numpy(), sin.numpy(),
                              rows)
    assert_bytes_equal(gk, wk, "k cache")
    assert_bytes_equal(gv, wv, "v cache")
    got_len = lengths_np(Lg)
    for f in Lg.FIELDS:
        np.testing.assert_array_equal(got_len[f], lens[f], err_msg=f)
    assert_close(out[rows], want, 2e-2, "fused step")


@pytest.mark.parametrize("ring,dtype,D,g,C,W", [
    (False, torch.bfloat16, 128, 4, 3000, 0),
    (False, torch.float16, 64, 8, 2048, 700),
    (True, torch.bfloat16, 128, 4, 4096, 0),
    (True, torch.bfloat16, 64, 16, 4096, 3000),
    (True, torch.float16, 128, 2, 300, 300),
    # capacity 12288: up to 24 splits a row, past the merge's 16-split fast path
    (False, torch.bfloat16, 128, 4, 12288, 0),
    (True, torch.bfloat16, 128, 4, 12288, 5000),
    # head_dim 256 (three 32 KB ring slots a CTA)
    (False, torch.bfloat16, 256, 2, 4096, 0),
    (True, torch.float16, 256, 2, 4096, 4096),
    (True, torch.bfloat16, 256, 8, 300, 130),
])
def test_consecutive_steps_and_graph(K, orc, ring, dtype, D, g, C, W):
    B, Hkv = 5, 2
    Hq = Hkv * g
    if ring:
        T0 = np.array([1, C - 3, C, 3 * C + 700, 9000])
    else:
        T0 = np.array([1, C // 2, C - 6, 600, 64])
    steps = 4
    cos, sin = synth.rope_cache(int(T0.max()) + steps + 1, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    kc = synth.normal((B, Hkv, C, D), 8, 1, dtype)
    vc = synth.normal((B, Hkv, C, D), 8, 2, dtype)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    gk, gv = kc.to(dev()), vc.to(dev())
    st = status()
    pol = K.KVC_RING if ring else K.KVC_CONTIGUOUS
    out = torch.empty(B, Hq, 1, D, dtype=dtype, device=dev())
    ws = None
    for s in range(steps):
        T = T0 + s
        nk = synth.normal((B, Hkv, 1, D), 9, s, dtype)
        nv = synth.normal((B, Hkv, 1, D), 10, s, dtype)
        q = synth.normal((B, Hq, 1, D), 11, s, dtype)
        sk = torch.from_numpy((T - 1).astype(np.int32)).to(dev())
        if ws is None:
            ws = K.decode_step_workspace(q.to(dev()), gk)
        K.kvc_decode_step(out, q.to(dev()), gk, gv, nk.to(dev()), nv.to(dev()), sk,
                          local_window_size=W, rope=rope_d, workspace=ws, status=st, windowed=pol)
        _, want = _oracle_step(orc, ring, wk, wv, nk, nv, q, T, C, W, cos.numpy(), sin.numpy())
        torch.cuda.synchronize()
        assert_bytes_equal(gk, wk, f"k step {s}")
        assert_bytes_equal(gv, wv, f"v step {s}")
        assert_close(out, want, 2e-2, f"step {s}")
    # the same step captured once and replayed
    T = T0 + steps
    nk = synth.normal((B, Hkv, 1, D), 9, steps, dtype).to(dev())
    nv = synth.normal((B, Hkv, 1, D), 10, steps, dtype).to(dev())
    q = synth.normal((B, Hq, 1, D), 11, steps, dtype).to(dev())
    sk = torch.from_numpy((T - 1).astype(np.int32)).to(dev())
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            K.kvc_decode_step(out, q, gk, gv, nk, nv, sk, local_window_size=W, rope=rope_d,
                              workspace=ws, status=st, windowed=pol)
    torch.cuda.current_stream().wait_stream(side)
    _, want = _oracle_step(orc, ring, wk, wv, nk.cpu(), nv.cpu(), q.cpu(), T, C, W, cos.numpy(),
                           sin.numpy())
    for rep in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert_close(out, want, 2e-2, f"graph replay {rep}")
    assert_bytes_equal(gk, wk, "k after replays")
    assert st.item() == 0


def test_rejected_rows(K, orc):
    B, Hq, Hkv, D, C = 4, 8, 2, 128, 2048
    kc = synth.normal((B, Hkv, C, D), 12, 1).to(dev())
    vc = synth.normal((B, Hkv, C, D), 12, 2).to(dev())
    before_k, before_v = kc.clone(), vc.clone()
    nk = synth.normal((B, Hkv, 1, D), 12, 3).to(dev())
    nv = synth.normal((B, Hkv, 1, D), 12, 4).to(dev())
    q = synth.normal((B, Hq, 1, D), 12, 5).to(dev())
    sk = torch.tensor([-1, 1500, C, 700], dtype=torch.int32, device=dev())  # T = 0, ok, C + 1, ok
    out = torch.zeros(B, Hq, 1, D, dtype=torch.bfloat16, device=dev())
    Lg = K.Lengths(B, dev())
    st = status()
    ws = K.decode_step_workspace(q, kc)
    K.kvc_decode_step(out, q, kc, vc, nk, nv, sk, lengths=Lg, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == K.KVC_DEV_SEQLEN_RANGE | K.KVC_DEV_CAPACITY
    for b in (0, 2):
        assert torch.equal(kc[b], before_k[b]) and torch.equal(vc[b], before_v[b])
        assert (Lg.buf[:, b] == -1).all()
        assert (out[b] == 0).all()
    # the good rows, and a second call on the same workspace
    st.zero_()
    sk2 = torch.tensor([9, 1501, 100, 701], dtype=torch.int32, device=dev())
    K.kvc_decode_step(out, q, kc, vc, nk, nv, sk2, lengths=Lg, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    wk, wv = synth.bits(before_k.cpu()).copy(), synth.bits(before_v.cpu()).copy()
    T1 = np.array([1, 1501, 1, 701])   # rows 0 and 2 were rejected: nothing appended
    for b in (1, 3):
        wk[b, :, T1[b] - 1] = synth.bits(nk.cpu())[b, :, 0]
        wv[b, :, T1[b] - 1] = synth.bits(nv.cpu())[b, :, 0]
    T2 = sk2.cpu().numpy().astype(np.int64) + 1
    _, want = _oracle_step(orc, False, wk, wv, nk.cpu(), nv.cpu(), q.cpu(), T2, C, 0, None, None)
    assert_bytes_equal(kc, wk, "k after second call")
    assert_close(out, want, 2e-2, "second call")
