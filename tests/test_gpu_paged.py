"""GPU parity for the paged cache (kvc_paged_append, kvc_gqa_decode_paged)
against the oracle's paged functions ("Persistent KV Cache and Decode
Performance Roadmap", Phase 2: fixed-size pages read through a page table).

* the contiguous decode workload at full size (32 x 32/8 heads x 128, 8192
  rows per sequence) held in 64-row pages scattered through a shuffled pool:
  the appended rows byte for byte, attention on sampled rows against the
  oracle and, for every row, equal to kvc_gqa_decode over the same rows laid
  out contiguously;
* windows that do not start on a tile boundary, page sizes 64/128/256, fp16
  and head_dim 64, multi-token appends that cross pages;
* a page id outside the pool: the append leaves the row alone and sets
  KVC_DEV_INDEX_OOB, the decode sets it without touching memory out of range.
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


def _pool_and_table(B, Hkv, D, P, max_pages, spare, seed, dtype=torch.bfloat16):
    n_pool = B * max_pages + spare
    rng = np.random.default_rng(seed)
    table = rng.permutation(n_pool)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    kp = synth.normal((n_pool, Hkv, P, D), seed, 1, dtype)
    vp = synth.normal((n_pool, Hkv, P, D), seed, 2, dtype)
    return kp, vp, table


def _contiguous_from_pool(pool, table, P):
    """[B, Hkv, max_pages * P, D] view of the pages in table order (torch)."""
    B, max_pages = table.shape
    idx = torch.from_numpy(table.astype(np.int64)).to(pool.device).reshape(-1)
    pages = pool.index_select(0, idx)                      # [B * max_pages, Hkv, P, D]
    Hkv, D = pool.shape[1], pool.shape[3]
    return pages.reshape(B, max_pages, Hkv, P, D).transpose(1, 2).reshape(
        B, Hkv, max_pages * P, D).contiguous()


def test_paged_workload_full_size(K, orc):
    w = synth.CONTIG_DECODE
    B, Hq, Hkv, D, C = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.capacity
    P = 64
    max_pages = C // P
    kp, vp, table = _pool_and_table(B, Hkv, D, P, max_pages, 17, 90)
    T = synth.randint(w.total_lo, w.total_hi + 1, (B,), 90, 3).numpy()
    T[:3] = [w.total_lo, C, 577]
    cos, sin = synth.rope_cache(C + 1, D, w.theta)
    rope_d = (cos.to(dev()), sin.to(dev()))
    nk = synth.normal((B, Hkv, 1, D), 90, 4)
    nv = synth.normal((B, Hkv, 1, D), 90, 5)
    q = synth.normal((B, Hq, 1, D), 90, 6)
    gk, gv = kp.to(dev()), vp.to(dev())
    tab = torch.from_numpy(table).to(dev())
    st = status()
    sk = torch.from_numpy((T - 1).astype(np.int32)).to(dev())
    L = K.kvc_seq_lengths(sk, 1, C, K.KVC_CONTIGUOUS, status=st)
    K.kvc_paged_append(gk, gv, nk.to(dev()), nv.to(dev()), tab, L, rope=rope_d, status=st)
    out = torch.full((B, Hq, 1, D), float("nan"), dtype=torch.bfloat16, device=dev())
    K.kvc_gqa_decode_paged(out, q.to(dev()), gk, gv, tab, L, rope=rope_d, status=st)
    # the same logical rows laid out contiguously, decoded by kvc_gqa_decode
    ck, cv = _contiguous_from_pool(gk, table, P), _contiguous_from_pool(gv, table, P)
    o2 = torch.empty_like(out)
    K.kvc_gqa_decode(o2, q.to(dev()), ck, cv, L, rope=rope_d, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(out, o2), "paged and contiguous decode differ"
    # appended rows against the oracle (only the new rows change)
    P_abs = T - 1
    wk, wv = synth.bits(kp).copy(), synth.bits(vp).copy()
    orc.paged_append(wk, wv, table, P, synth.bits(nk), synth.bits(nv), P_abs, cos.numpy(),
                     sin.numpy())
    for b in range(B):
        page = table[b, P_abs[b] // P]
        np.testing.assert_array_equal(synth.bits(gk[page].cpu()), wk[page])
        np.testing.assert_array_equal(synth.bits(gv[page].cpu()), wv[page])
    rows = [0, 1, 2, 20]
    want, _ = orc.paged_attention(synth.bits(q)[rows], wk, wv, table[rows], P, T[rows], T[rows],
                                  cos_cache=cos.numpy(), sin_cache=sin.numpy())
    assert_close(out[rows], want, 2e-2, "paged decode")


@pytest.mark.parametrize("P,D,g,W,dtype", [(64, 128, 4, 700, torch.bfloat16),
                                           (128, 64, 8, 100, torch.float16),
                                           (256, 128, 2, 0, torch.bfloat16),
                                           (64, 64, 16, 1, torch.bfloat16),
                                           (64, 256, 2, 1000, torch.bfloat16),
                                           (128, 256, 4, 0, torch.float16)])
def test_paged_steps(K, orc, P, D, g, W, dtype):
    """Chunks then one-token steps, window boundaries off the tiles."""
    B, Hkv = 4, 2
    Hq = Hkv * g
    max_pages = 24
    C = max_pages * P
    kp, vp, table = _pool_and_table(B, Hkv, D, P, max_pages, 5, 91 + P + D, dtype)
    wk, wv = synth.bits(kp).copy(), synth.bits(vp).copy()
    gk, gv = kp.to(dev()), vp.to(dev())
    tab = torch.from_numpy(table).to(dev())
    cos, sin = synth.rope_cache(C + 1, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    st = status()
    T = np.array([0, 5, 63, 700], dtype=np.int64)
    for step, S in enumerate([37, 1, 200, 1, 1, 64, 1]):
        nk = synth.normal((B, Hkv, S, D), 92, step, dtype)
        nv = synth.normal((B, Hkv, S, D), 93, step, dtype)
        sk = torch.from_numpy((T + S - 1).astype(np.int32)).to(dev())
        L = K.kvc_seq_lengths(sk, S, C, K.KVC_CONTIGUOUS, status=st)
        K.kvc_paged_append(gk, gv, nk.to(dev()), nv.to(dev()), tab, L, rope=rope_d, status=st)
        orc.paged_append(wk, wv, table, P, synth.bits(nk), synth.bits(nv), T, cos.numpy(),
                         sin.numpy())
        T = T + S
        torch.cuda.synchronize()
        assert_bytes_equal(gk, wk, f"k pool step {step}")
        assert_bytes_equal(gv, wv, f"v pool step {step}")
        if S == 1:
            q = synth.normal((B, Hq, 1, D), 94, step, dtype)
            out = torch.empty(B, Hq, 1, D, dtype=dtype, device=dev())
            K.kvc_gqa_decode_paged(out, q.to(dev()), gk, gv, tab, L, local_window_size=W,
                                   rope=rope_d, status=st)
            want, _ = orc.paged_attention(synth.bits(q), wk, wv, table, P, T, T, W,
                                          cos_cache=cos.numpy(), sin_cache=sin.numpy())
            torch.cuda.synchronize()
            assert_close(out, want, 2e-2, f"paged decode step {step}")
    assert st.item() == 0


def test_paged_bad_page(K, orc):
    B, Hq, Hkv, D, P, max_pages = 3, 8, 2, 128, 64, 4
    kp, vp, table = _pool_and_table(B, Hkv, D, P, max_pages, 0, 95)
    n_pool = B * max_pages
    table[1, 1] = n_pool + 3           # row 1's second page is outside the pool
    table[2, 0] = -1                   # row 2's first page too
    gk, gv = kp.to(dev()), vp.to(dev())
    before_k = gk.clone()
    tab = torch.from_numpy(table).to(dev())
    T = np.array([70, 70, 3])          # the new rows land in page 1, 1 and 0
    nk = synth.normal((B, Hkv, 1, D), 95, 4).to(dev())
    nv = synth.normal((B, Hkv, 1, D), 95, 5).to(dev())
    st = status()
    sk = torch.from_numpy((T - 1).astype(np.int32)).to(dev())
    L = K.kvc_seq_lengths(sk, 1, max_pages * P, K.KVC_CONTIGUOUS, status=st)
    K.kvc_paged_append(gk, gv, nk, nv, tab, L, status=st)
    torch.cuda.synchronize()
    assert st.item() == K.KVC_DEV_INDEX_OOB
    changed = [p for p in range(n_pool) if not torch.equal(gk[p], before_k[p])]
    assert changed == [int(table[0, 1])]    # only row 0 wrote its row
    st.zero_()
    out = torch.empty(B, Hq, 1, D, dtype=torch.bfloat16, device=dev())
    K.kvc_gqa_decode_paged(out, synth.normal((B, Hq, 1, D), 95, 6).to(dev()), gk, gv, tab, L,
                           status=st)
    torch.cuda.synchronize()
    assert st.item() == K.KVC_DEV_INDEX_OOB
