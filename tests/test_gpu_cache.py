"""GPU parity for kvc_seq_lengths and kvc_window_append against the oracle.

Lengths are compared exactly (random rows, int32 edges, contiguous and
windowed).  Appends are compared bit for bit over the WHOLE cache and stage
buffers (every shifted, evicted, untouched and new row): contiguous appends,
windowed one-token compaction (E = 0 and E = 1 rows mixed), windowed C + S
staging seed and copy-back (including S > C), with and without RoPE, for
fp32, bf16 and fp16, and the RoPE-range flag that leaves a row untouched.
"""
import numpy as np
import pytest
import torch

from _gpu_helpers import assert_bytes_equal, dev, lengths_np, status
from persistent_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu

INT32_MAX = 2**31 - 1


@pytest.fixture(scope="module")
def K():
    from persistent_kv_cache_gb300 import kvc
    return kvc


@pytest.mark.parametrize("windowed", [0, 1, 2])
def test_lengths(K, orc, windowed):
    rng = np.random.default_rng(7 + windowed)
    for S, C in [(1, 128), (5, 16), (64, 4096), (2048, 4096), (3, 1)]:
        sk = rng.integers(-3, 3 * C + S, size=97).astype(np.int32)
        sk[:4] = [-1, S - 1, INT32_MAX - 1, INT32_MAX]
        W = max(1, C - 8) if windowed == 2 else C
        want = orc.seq_lengths(sk, S, C, windowed, W)
        st = status()
        L = K.kvc_seq_lengths(torch.from_numpy(sk).to(dev()), S, C, windowed,
                              local_window_size=W, status=st)
        got = lengths_np(L)
        for f in L.FIELDS:
            np.testing.assert_array_equal(got[f], want[f], err_msg=f"{f} S={S} C={C}")
        flags = int(st.item())
        assert bool(flags & K.KVC_DEV_SEQLEN_RANGE) == bool((want["flags"] & 2).any())
        assert bool(flags & K.KVC_DEV_CAPACITY) == bool((want["flags"] & 4).any())


_DT = {torch.float32: np.float32, torch.bfloat16: np.uint16, torch.float16: np.float16}


def _rand(shape, seed, stream, dtype):
    return synth.normal(shape, seed, stream, dtype=dtype)


def _run_append(K, orc, dtype, windowed, S, C, T, rope, seed, D=16, Hkv=3):
    """One append step on GPU and oracle; compares every byte of the caches
    (and of the stages for windowed S > 1)."""
    B = len(T)
    T = np.asarray(T, dtype=np.int64)
    kc = _rand((B, Hkv, C, D), seed, 1, dtype)
    vc = _rand((B, Hkv, C, D), seed, 2, dtype)
    nk = _rand((B, Hkv, S, D), seed, 3, dtype)
    nv = _rand((B, Hkv, S, D), seed, 4, dtype)
    cos = sin = None
    if rope:
        cos, sin = synth.rope_cache(int(T.max()) + 8, D)
    staged = windowed and S > 1
    if staged:
        ks = _rand((B, Hkv, C + S, D), seed, 5, dtype)
        vs = _rand((B, Hkv, C + S, D), seed, 6, dtype)
    sk = (T - 1).astype(np.int32)
    lens = orc.seq_lengths(sk, S, C, windowed)
    w_kc, w_vc = synth.bits(kc).copy(), synth.bits(vc).copy()
    w_ks = synth.bits(ks).copy() if staged else None
    w_vs = synth.bits(vs).copy() if staged else None
    flags = orc.window_append(w_kc, w_vc, synth.bits(nk), synth.bits(nv), lens, windowed,
                              None if cos is None else cos.numpy(),
                              None if sin is None else sin.numpy(), w_ks, w_vs)

    st = status()
    g = {n: t.to(dev()) for n, t in dict(kc=kc, vc=vc, nk=nk, nv=nv).items()}
    if staged:
        g["ks"], g["vs"] = ks.to(dev()), vs.to(dev())
    rope_d = None if cos is None else (cos.to(dev()), sin.to(dev()))
    L = K.kvc_seq_lengths(torch.from_numpy(sk).to(dev()), S, C, windowed,
                          local_window_size=C, status=st)
    K.kvc_window_append(g["kc"], g["vc"], g["nk"], g["nv"], L, windowed, K.KVC_APPEND,
                        g.get("ks"), g.get("vs"), rope=rope_d, status=st)
    if staged:
        torch.cuda.synchronize()
        # the stage after seeding is what the chunk attention reads
        w_ks2, w_vs2 = synth.bits(ks).copy(), synth.bits(vs).copy()
        for b in range(B):
            if lens["cache_total"][b] < 0 or flags[b]:
                continue
            Lp = lens["cache_past"][b]
            w_ks2[b, :, :Lp + S] = w_ks[b, :, :Lp + S]
            w_vs2[b, :, :Lp + S] = w_vs[b, :, :Lp + S]
        assert_bytes_equal(g["ks"], w_ks2, "k stage")
        assert_bytes_equal(g["vs"], w_vs2, "v stage")
        K.kvc_window_append(g["kc"], g["vc"], None, None, L, windowed, K.KVC_COPY_BACK,
                            g["ks"], g["vs"], rope=rope_d, status=st)
    torch.cuda.synchronize()
    assert_bytes_equal(g["kc"], w_kc, "k cache")
    assert_bytes_equal(g["vc"], w_vc, "v cache")
    return int(st.item()), flags


DTYPES = [torch.float32, torch.bfloat16, torch.float16]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rope", [False, True])
def test_contiguous_append(K, orc, dtype, rope):
    st, _ = _run_append(K, orc, dtype, 0, 1, 40, [1, 17, 40, 33], rope, 1)
    assert st == 0
    st, _ = _run_append(K, orc, dtype, 0, 5, 40, [5, 17, 40, 6], rope, 2)
    assert st == 0


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rope", [False, True])
def test_windowed_decode_append(K, orc, dtype, rope):
    # rows with E = 0 (not yet full) and E = 1 (full) in one launch, C = 24 and 128
    st, _ = _run_append(K, orc, dtype, 1, 1, 24, [1, 5, 24, 25, 26, 1000], rope, 3)
    assert st == 0
    st, _ = _run_append(K, orc, dtype, 1, 1, 128, [1, 127, 128, 129, 30000], rope, 4, D=64)
    assert st == 0


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rope", [False, True])
def test_windowed_staging(K, orc, dtype, rope):
    for S, C, T in [(7, 24, [7, 10, 24, 31, 90]), (40, 24, [40, 41, 100]),
                    (64, 200, [64, 200, 263, 264, 5000])]:
        st, _ = _run_append(K, orc, dtype, 1, S, C, T, rope, 5 + S, D=32)
        assert st == 0


def test_rope_range_leaves_row(K, orc):
    st, flags = _run_append(K, orc, torch.bfloat16, 1, 1, 16, [5, 40, 9], True, 9)
    assert st == 0 and not flags.any()
    # tables cover positions < T.max() + 8; shrink by passing a short table
    B, Hkv, C, D, S = 2, 2, 16, 16, 3
    kc = synth.normal((B, Hkv, C, D), 3, 1)
    vc = synth.normal((B, Hkv, C, D), 3, 2)
    nk = synth.normal((B, Hkv, S, D), 3, 3)
    nv = synth.normal((B, Hkv, S, D), 3, 4)
    cos, sin = synth.rope_cache(20, D)
    sk = np.array([30, 10], dtype=np.int32)  # row 0 needs positions 28..30 >= 20
    gk, gv = kc.to(dev()), vc.to(dev())
    ks = torch.zeros(B, Hkv, C + S, D, dtype=torch.bfloat16, device=dev())
    vs = torch.zeros_like(ks)
    st = status()
    L = K.kvc_seq_lengths(torch.from_numpy(sk).to(dev()), S, C, 1, local_window_size=C, status=st)
    rope = (cos.to(dev()), sin.to(dev()))
    K.kvc_window_append(gk, gv, nk.to(dev()), nv.to(dev()), L, 1, K.KVC_APPEND, ks, vs, rope=rope,
                        status=st)
    K.kvc_window_append(gk, gv, None, None, L, 1, K.KVC_COPY_BACK, ks, vs, rope=rope, status=st)
    torch.cuda.synchronize()
    assert st.item() == K.KVC_DEV_ROPE_RANGE
    assert torch.equal(gk[0].cpu(), kc[0]) and torch.equal(gv[0].cpu(), vc[0])
    assert not torch.equal(gk[1].cpu(), kc[1])


def test_seqlen_errors_leave_rows(K, orc):
    # T < S and T > C (contiguous) rows are rejected; the others proceed
    st, flags = _run_append(K, orc, torch.bfloat16, 0, 2, 16, [1, 9, 17], False, 11)
    assert st == K.KVC_DEV_SEQLEN_RANGE | K.KVC_DEV_CAPACITY
