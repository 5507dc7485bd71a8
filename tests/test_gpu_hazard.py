"""GPU parity for kvc_window_prefill_step: a windowed (or drifting) step of S
new tokens that stages only the batch rows whose eviction the chunk would
see ("GQA support sliding_window_cache", CPU commit: staging for hazardous
steps), decided per row on the device.

After every step the cache is compared byte for byte with the oracle's
staged flow and the output with the oracle's attention (max-abs <= 2e-2,
1e-4 for fp32).  The stage starts each step filled with a sentinel: a row
the call stages must leave the oracle's stage there, a row it does not
stage must leave the sentinel untouched -- and which rows are staged is
checked against a brute-force reading of the lengths (does any query of the
chunk see a position the step evicts?), so the per-row decision itself is
pinned, not only its result.  Shapes: the page's small-slack chunked
prefill (chunks of 32 on C = W + 8) with batch rows at different offsets so
that every step mixes in-place and staged rows, chunks no longer than the
gap (evicting, yet in place), one-token steps, fp16 and fp32 (whose
CUDA-core path stages every row of a multi-token step), and the full
windowed chunked-prefill workload (8 x 16/8 heads x 256, C = W = 4096) at
S = 64 with sampled queries.
"""
import numpy as np
import pytest
import torch

from _gpu_helpers import assert_bytes_equal, assert_close, dev, status, tol
from persistent_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu

SENTINEL = 0x7f  # byte pattern of the stage before each step


@pytest.fixture(scope="module")
def K():
    from persistent_kv_cache_gb300 import kvc
    return kvc


def _hazardous(lens, S, W):
    """Rows whose step evicts a position one of its queries sees, read off
    the positions: stage row r holds position P - Lp + r, rows [0, E) are
    evicted, query i at P + i sees positions p with P + i - p < W."""
    out = []
    for b in range(len(lens["evict"])):
        P, Lp, E = int(lens["past_abs"][b]), int(lens["cache_past"][b]), int(lens["evict"][b])
        out.append(any(P + i - (P - Lp + r) < W for r in range(E) for i in range(S)))
    return np.array(out, dtype=bool)


def _step(K, orc, gk, gv, wk, wv, T, S, C, W, policy, dtype, seed, rope, Hq, sample=None):
    """One step on the device caches (gk, gv) and the oracle's (wk, wv).
    Returns (rows the call staged, lengths).  sample: check only these
    queries (each as the last of a chunk ending at it)."""
    B, Hkv, _, D = gk.shape
    nk = synth.normal((B, Hkv, S, D), seed, 1, dtype)
    nv = synth.normal((B, Hkv, S, D), seed, 2, dtype)
    q = synth.normal((B, Hq, S, D), seed, 3, dtype)
    sk = (np.asarray(T) + S - 1).astype(np.int32)
    st = status()
    L = K.kvc_seq_lengths(torch.from_numpy(sk).to(dev()), S, C, policy, local_window_size=W,
                          status=st)
    lens = orc.seq_lengths(sk, S, C, policy, W)
    ks = vs = None
    if S > 1:
        ks = torch.empty((B, Hkv, C + S, D), dtype=dtype, device=dev())
        ks.view(torch.uint8).fill_(SENTINEL)
        vs = ks.clone()
    out = torch.full((B, Hq, S, D), float("nan"), dtype=dtype, device=dev())
    cos, sin = rope
    K.kvc_window_prefill_step(out, q.to(dev()), gk, gv, nk.to(dev()), nv.to(dev()), L, policy, W,
                              ks, vs, rope=(cos.to(dev()), sin.to(dev())), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0, st.item()

    cn, sn = cos.numpy(), sin.numpy()
    qn = synth.bits(q)
    staged = np.zeros(B, dtype=bool)
    if S > 1:
        # fp32 runs on the CUDA-core path, which stages every row
        staged = np.ones(B, bool) if dtype == torch.float32 else _hazardous(lens, S, W)
        wks = np.zeros((B, Hkv, C + S, D), dtype=wk.dtype)
        wvs = np.zeros_like(wks)
        orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, policy, cn, sn, wks, wvs)
        sent = np.full(ks[0].numel() * ks.element_size(), SENTINEL, np.uint8)
        for b in range(B):
            if staged[b]:
                # the 16-bit path stages the new rows and the 127 old rows
                # below them (its attention reads older tiles from the
                # cache); fp32 stages the whole window
                Lp = int(lens["cache_past"][b])
                s0 = 0 if dtype == torch.float32 else max(0, Lp - 127)
                n = Lp + S
                assert_bytes_equal(ks[b, :, s0:n], np.ascontiguousarray(wks[b, :, s0:n]),
                                   f"k stage row {b}")
                assert_bytes_equal(vs[b, :, s0:n], np.ascontiguousarray(wvs[b, :, s0:n]),
                                   f"v stage row {b}")
                for s_ in (ks, vs):
                    got = s_[b, :, :s0].contiguous().view(torch.uint8).cpu().numpy().ravel()
                    assert (got == SENTINEL).all(), f"row {b} staged rows below Lp - 127"
            else:
                for s_ in (ks, vs):
                    got = s_[b].contiguous().view(torch.uint8).cpu().numpy().ravel()
                    assert np.array_equal(got, sent), f"row {b} wrote the stage"
        rk, rv, n_rows = wks, wvs, (lens["cache_past"] + S).astype(np.int32)
    else:
        orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, policy, cn, sn)
        rk, rv, n_rows = wk, wv, lens["cache_total"]
    assert_bytes_equal(gk, wk, "k cache")
    assert_bytes_equal(gv, wv, "v cache")
    if sample is None:
        want, _ = orc.gqa_attention(qn, rk, rv, n_rows, lens["total_abs"], window=W,
                                    cos_cache=cn, sin_cache=sn)
        assert_close(out, want, tol(dtype), f"step S={S}")
    else:
        for i in sample:
            n = (lens["cache_past"] + i + 1).astype(np.int32)
            Ti = (lens["past_abs"] + i + 1).astype(np.int32)
            want, _ = orc.gqa_attention(np.ascontiguousarray(qn[:, :, i:i + 1]), rk, rv, n, Ti,
                                        window=W, cos_cache=cn, sin_cache=sn)
            assert_close(out[:, :, i:i + 1], want, tol(dtype), f"query {i}")
    return staged, lens


def _run(K, orc, policy, dtype, B, Hkv, g, D, C, W, T0, schedule, seed):
    cos, sin = synth.rope_cache(int(max(T0)) + sum(schedule) + 1, D)
    kc = torch.zeros(B, Hkv, C, D, dtype=dtype)
    wk, wv = synth.bits(kc).copy(), synth.bits(kc).copy()
    gk, gv = kc.to(dev()), kc.clone().to(dev())
    T = np.asarray(T0)
    seen = set()
    for step, S in enumerate(schedule):
        staged, lens = _step(K, orc, gk, gv, wk, wv, T, S, C, W, policy, dtype,
                             seed + 10 * step, (cos, sin), Hkv * g)
        for b in range(B):
            seen.add("staged" if staged[b] else
                     ("moved" if int(lens["evict"][b]) > 0 else "append"))
        T = T + S
    return seen


@pytest.mark.parametrize("policy", [1, 2])
@pytest.mark.parametrize("D,g", [(64, 2), (128, 4)])
def test_small_slack_chunks(K, orc, policy, D, g):
    """Chunks of 32 (and shorter ones) on C = W + 8, batch rows started at
    different offsets: steps mix rows that still fill the cache, rows that
    evict only what no query sees and rows that must be staged."""
    W = 40
    seen = _run(K, orc, policy, torch.bfloat16, 4, 2, g, D, W + 8, W, [0, 20, 41, 300],
                [32, 32, 1, 32, 5, 32, 9, 32, 32, 8, 3, 32], 1000 * policy + D)
    assert seen == {"staged", "moved", "append"}, seen


def test_fp16_and_fp32(K, orc):
    # windowed, C = W + 16: once full, chunks of up to 17 tokens evict only
    # rows no query sees
    seen = _run(K, orc, 1, torch.float16, 3, 2, 2, 64, 40, 24, [0, 17, 90],
                [20, 12, 1, 30, 6, 40, 16], 700)
    assert seen == {"staged", "moved", "append"}, seen
    _run(K, orc, 2, torch.float32, 3, 2, 2, 32, 40, 24, [0, 17, 90], [20, 12, 1, 30, 6], 800)


def test_window_prefill_workload_s64(K, orc):
    """The windowed chunked-prefill workload at S = 64: rows that have not
    filled the cache append in place, the others stage; the cache is checked
    in full and the queries at the chunk's ends and the 64-query block edges
    one by one."""
    w = synth.WINDOW_PREFILL
    S = 64
    B, Hq, Hkv, D, C, W = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.capacity, w.window
    T = synth.randint(w.total_lo, w.total_hi + 1, (B,), 0, S).numpy()
    T[0], T[1], T[2] = 0, C - S - 3, C - S // 2
    kc = synth.normal((B, Hkv, C, D), 71, 1)
    vc = synth.normal((B, Hkv, C, D), 71, 2)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    gk, gv = kc.to(dev()), vc.to(dev())
    cos, sin = synth.rope_cache(int(T.max()) + S + 1, D)
    staged, _ = _step(K, orc, gk, gv, wk, wv, T, S, C, W, 1, torch.bfloat16, 72, (cos, sin), Hq,
                      sample=(0, 31, 32, 63))
    assert not staged[0] and not staged[1] and staged[2]


def test_rejected_rows_untouched(K, orc):
    """A row whose seqlens_k is out of range and a row past the rotary table
    are left as they were (cache and stage) and flagged; the valid rows of
    the same call are exact."""
    B, Hkv, g, D, C, W, S = 3, 2, 2, 64, 48, 40, 16
    kc = synth.normal((B, Hkv, C, D), 90, 1)
    vc = synth.normal((B, Hkv, C, D), 90, 2)
    nk = synth.normal((B, Hkv, S, D), 90, 3)
    nv = synth.normal((B, Hkv, S, D), 90, 4)
    q = synth.normal((B, Hkv * g, S, D), 90, 5)
    cos, sin = synth.rope_cache(200, D)
    sk = np.array([100 + S - 1, S - 2, 400 + S - 1], np.int32)  # valid, T < S, past the table
    st = status()
    gk, gv = kc.to(dev()), vc.to(dev())
    L = K.kvc_seq_lengths(torch.from_numpy(sk).to(dev()), S, C, 1, local_window_size=W, status=st)
    ks = torch.zeros(B, Hkv, C + S, D, dtype=torch.bfloat16, device=dev())
    vs = torch.zeros_like(ks)
    out = torch.zeros(B, Hkv * g, S, D, dtype=torch.bfloat16, device=dev())
    K.kvc_window_prefill_step(out, q.to(dev()), gk, gv, nk.to(dev()), nv.to(dev()), L, 1, W, ks,
                              vs, rope=(cos.to(dev()), sin.to(dev())), status=st)
    torch.cuda.synchronize()
    assert st.item() == K.KVC_DEV_SEQLEN_RANGE | K.KVC_DEV_ROPE_RANGE, st.item()
    for b in (1, 2):
        assert torch.equal(gk[b].cpu(), kc[b]) and torch.equal(gv[b].cpu(), vc[b]), b
        assert not ks[b].any() and not vs[b].any(), b
    # the valid row against the oracle
    lens = orc.seq_lengths(sk[:1], S, C, 1, W)
    wk, wv = synth.bits(kc[:1]).copy(), synth.bits(vc[:1]).copy()
    wks = np.zeros((1, Hkv, C + S, D), np.uint16)
    wvs = np.zeros_like(wks)
    orc.window_append(wk, wv, synth.bits(nk[:1]), synth.bits(nv[:1]), lens, 1, cos.numpy(),
                      sin.numpy(), wks, wvs)
    assert_bytes_equal(gk[:1], wk, "k cache row 0")
    assert_bytes_equal(gv[:1], wv, "v cache row 0")
    want, _ = orc.gqa_attention(synth.bits(q[:1]), wks, wvs,
                                (lens["cache_past"] + S).astype(np.int32), lens["total_abs"],
                                window=W, cos_cache=cos.numpy(), sin_cache=sin.numpy())
    assert_close(out[:1], want, 2e-2, "row 0")
