"""GPU parity for the one-token in-place compaction of large windowed slices
("GQA support sliding_window_cache", "Design": rows [E, Lp) move to
[0, Lp - E), the new row goes to Lp - E), which runs as a thread-block
cluster of up to eight CTAs per (batch row, kv head, K/V) once a slice holds
64 KB or more.

Each case runs consecutive one-token steps through kvc_seq_lengths +
kvc_window_append and compares the lengths and every cache byte with the
oracle after every step, on rows that start empty, below the capacity, at
it and far past it.  The shapes steer the kernel's paths:
  * cluster sizes 1, 2 and 8 (slices of 64 KB, 275 KB and 2 MB);
  * the drifting layout with a gap that fits the cluster's save buffer
    (E = 41 rows moved at once) and one that does not (E = 1949 rows, moved
    by the cluster's first CTA alone);
  * fp32, fp16 and bf16 rows, with and without RoPE.
"""
import numpy as np
import pytest
import torch

from _gpu_helpers import assert_bytes_equal, dev, lengths_np, status
from persistent_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from persistent_kv_cache_gb300 import kvc
    return kvc


@pytest.mark.parametrize("policy,dtype,D,C,W,steps", [
    (1, torch.bfloat16, 128, 256, 256, 6),      # 64 KB slices: a cluster of one
    (1, torch.bfloat16, 128, 1100, 900, 5),     # 275 KB: two CTAs
    (1, torch.float16, 256, 4096, 4096, 4),     # 2 MB: eight CTAs
    (1, torch.float32, 64, 512, 300, 5),        # fp32 rows, 128 KB
    (2, torch.bfloat16, 128, 1064, 1024, 45),   # drifting, 41-row blocks (in the save buffer)
    (2, torch.bfloat16, 128, 2048, 100, 4),     # drifting, 1949-row blocks (first CTA alone)
])
def test_compaction_steps(K, orc, policy, dtype, D, C, W, steps):
    B, Hkv = 5, 2
    seed = 400 + D + C + policy
    rope = dtype != torch.float32
    T0 = np.array([1, C // 2, C - 2, C, 30000 + C], dtype=np.int64)
    kc = synth.normal((B, Hkv, C, D), seed, 1, dtype)
    vc = synth.normal((B, Hkv, C, D), seed, 2, dtype)
    wk, wv = synth.bits(kc).copy(), synth.bits(vc).copy()
    gk, gv = kc.to(dev()), vc.to(dev())
    cos = sin = rope_d = None
    if rope:
        cos, sin = synth.rope_cache(int(T0.max()) + steps + 1, D)
        rope_d = (cos.to(dev()), sin.to(dev()))
    st = status()
    L = K.Lengths(B, dev())
    moved = 0
    for s in range(steps):
        T = T0 + s
        sk = (T - 1).astype(np.int32)
        nk = synth.normal((B, Hkv, 1, D), seed, 10 + s, dtype)
        nv = synth.normal((B, Hkv, 1, D), seed, 100 + s, dtype)
        K.kvc_seq_lengths(torch.from_numpy(sk).to(dev()), 1, C, policy, local_window_size=W,
                          out=L, status=st)
        K.kvc_window_append(gk, gv, nk.to(dev()), nv.to(dev()), L, policy, rope=rope_d,
                            status=st)
        lens = orc.seq_lengths(sk, 1, C, policy, W)
        orc.window_append(wk, wv, synth.bits(nk), synth.bits(nv), lens, policy,
                          None if cos is None else cos.numpy(),
                          None if sin is None else sin.numpy())
        torch.cuda.synchronize()
        got = lengths_np(L)
        for f in L.FIELDS:
            np.testing.assert_array_equal(got[f], lens[f], err_msg=f"{f} step {s}")
        assert_bytes_equal(gk, wk, f"k step {s}")
        assert_bytes_equal(gv, wv, f"v step {s}")
        moved += int((lens["evict"] > 0).sum())
    assert st.item() == 0
    assert moved >= 2   # the rows past the capacity moved
