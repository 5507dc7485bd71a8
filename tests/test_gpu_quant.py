"""GPU parity for int8 pages: kvc_quantize_pages and kvc_gqa_decode_paged_q
against the oracle ("Persistent input/output feedback", "Optional
heterogeneous paged KV": selected-block affine quantization; roadmap
"Phase 3: cache quantization and fusion").

* quantization: the stored bytes (in the fragment order include/kvc.h
  specifies, restated here) and the per-page parameters bit for bit
  (bf16 and fp16 pools, INT8 and UINT8, a page full of exact ties, saturated
  values); pages not selected stay untouched; a pair outside a pool sets
  KVC_DEV_INDEX_OOB and is skipped;
* decode on values on the grid of a power-of-two scale: every page int8,
  the output equals the 16-bit paged decode bit for bit (the integers and the
  scales enter the MMAs exactly);
* the contiguous decode workload at full size (32 x 32/8 heads x 128, 8192
  rows) in 64-row pages with every full page quantized (the newest page of a
  row stays 16-bit): sampled rows against the oracle;
* mixed tables at small sizes, window masks, fp16, head_dim 64, UINT8 V;
* an int8 entry outside the int8 pool sets KVC_DEV_INDEX_OOB.
"""
import numpy as np
import pytest
import torch

from _gpu_helpers import assert_close, dev, status
from persistent_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from persistent_kv_cache_gb300 import kvc
    return kvc


def _positions(D, which):
    """[16, D] byte positions within a 16-row group of the payload's fragment
    order, restated from include/kvc.h."""
    j = np.arange(16)[:, None]
    d = np.arange(D)[None, :]
    if which == "k":
        lane = 4 * (j % 8) + (d % 16 % 8) // 2
        f = (2 * (d // 16) + d % 16 // 8) * 4 + 2 * (j // 8) + d % 2
    else:
        lane = 4 * (d % 16 % 8) + (j % 8) // 2
        f = (2 * (d // 16) + j // 8) * 4 + 2 * (d % 16 // 8) + j % 2
    return (f // 16) * 512 + lane * 16 + f % 16


def frag_order(a, which):
    """Natural [..., P, D] payload -> fragment order."""
    *lead, P, D = a.shape
    grp = a.reshape(-1, P // 16, 16, D)
    out = np.empty((grp.shape[0], P // 16, 16 * D), a.dtype)
    out[:, :, _positions(D, which)] = grp
    return out.reshape(a.shape)


def natural_order(a, which):
    """Fragment-order [..., P, D] payload -> natural order."""
    *lead, P, D = a.shape
    flat = a.reshape(-1, P // 16, 16 * D)
    return flat[:, :, _positions(D, which)].reshape(a.shape)


def _pools_np(qk, qv):
    return natural_order(qk.cpu().numpy(), "k"), natural_order(qv.cpu().numpy(), "v")


def _q8_pools(n_q, Hkv, P, D):
    qk = torch.full((n_q, Hkv, P, D), 77, dtype=torch.uint8, device=dev())
    qv = torch.full_like(qk, 77)
    qp = torch.zeros(n_q, 4, dtype=torch.float32, device=dev())
    return qk, qv, qp


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_quantize_bits(K, orc, dtype):
    n_pool, Hkv, P, D = 10, 2, 64, 64
    kp = (synth.normal((n_pool, Hkv, P, D), 60, 1, torch.float32) * 0.5).to(dtype)
    vp = (synth.normal((n_pool, Hkv, P, D), 60, 2, torch.float32) * 0.5).to(dtype)
    # page 3: exact ties for scale 0.25 (odd multiples of 0.125); page 4: saturating values
    ties = (torch.arange(P * D, dtype=torch.float32).reshape(P, D) % 31 - 15) * 0.125
    kp[3] = ties.to(dtype)
    vp[3] = ties.to(dtype)
    kp[4] = (synth.normal((Hkv, P, D), 60, 3, torch.float32) * 40).to(dtype)
    gk, gv = kp.to(dev()), vp.to(dev())
    n_q = 8
    qk, qv, qp = _q8_pools(n_q, Hkv, P, D)
    src = torch.tensor([3, 4, 0, 9, 5], dtype=torch.int32, device=dev())
    dst = torch.tensor([6, 1, 0, 2, 7], dtype=torch.int32, device=dev())
    st = status()
    ks, kz, vs, vz = 0.25, 0, 0.25, 128
    K.kvc_quantize_pages(gk, gv, qk, qv, src, dst, qp, ks, kz, False, vs, vz, True, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    kb, vb = synth.bits(kp), synth.bits(vp)
    for s_, d_ in zip(src.tolist(), dst.tolist()):
        want_k, zk = orc.quantize_page(kb[s_], ks, kz, False)
        want_v, zv = orc.quantize_page(vb[s_], vs, vz, True)
        assert np.array_equal(qk[d_].cpu().numpy(), frag_order(want_k, "k")), (s_, d_)
        assert np.array_equal(qv[d_].cpu().numpy(), frag_order(want_v, "v")), (s_, d_)
        assert qp[d_].tolist() == [ks, float(zk), vs, float(zv)]
    for d_ in set(range(n_q)) - set(dst.tolist()):
        assert (qk[d_] == 77).all() and (qv[d_] == 77).all() and (qp[d_] == 0).all()
    # the tie page holds exact ties: both roundings of a tie must not appear
    codes = orc.quantize_affine(orc.to_f32(kb[3]), 0.25, 0)
    assert np.array_equal(natural_order(qk[6].cpu().numpy(), "k").astype(np.int32) - 128, codes)
    # and the saturating page reaches both ends
    assert qk[1].max().item() == 255 and qk[1].min().item() == 0


def test_quantize_bad_pair(K):
    n_pool, Hkv, P, D = 4, 2, 64, 64
    gk = synth.normal((n_pool, Hkv, P, D), 61, 1).to(dev())
    gv = synth.normal((n_pool, Hkv, P, D), 61, 2).to(dev())
    qk, qv, qp = _q8_pools(3, Hkv, P, D)
    src = torch.tensor([0, 7, 1], dtype=torch.int32, device=dev())   # 7: outside the pool
    dst = torch.tensor([0, 1, 5], dtype=torch.int32, device=dev())   # 5: outside the int8 pool
    st = status()
    K.kvc_quantize_pages(gk, gv, qk, qv, src, dst, qp, 0.05, status=st)
    torch.cuda.synchronize()
    assert st.item() == K.KVC_DEV_INDEX_OOB
    assert not (qk[0] == 77).all()
    assert (qk[1] == 77).all() and (qk[2] == 77).all()


def _paged_setup(B, Hkv, D, P, max_pages, spare, seed, dtype, values=None):
    n_pool = B * max_pages + spare
    rng = np.random.default_rng(seed)
    table = rng.permutation(n_pool)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    if values is None:
        kp = synth.normal((n_pool, Hkv, P, D), seed, 1, dtype)
        vp = synth.normal((n_pool, Hkv, P, D), seed, 2, dtype)
    else:
        kp, vp = values
    return kp, vp, table


def _quantize_table(K, table, n_rows, P, kp_d, vp_d, qk, qv, qp, ks, kz, ku, vs, vz, vu,
                    keep_last=True):
    """Quantize every full page below each row's last (or every page holding
    rows), point the table at the int8 copies, return the new table."""
    B, max_pages = table.shape
    src, dst, new = [], [], table.copy()
    for b in range(B):
        n_used = (int(n_rows[b]) + P - 1) // P
        last = n_used - 1 if keep_last else n_used
        for j in range(last):
            src.append(int(table[b, j]))
            dst.append(len(dst))
            new[b, j] = K.KVC_PAGE_QUANT | (len(dst) - 1)
    st = status()
    if src:
        K.kvc_quantize_pages(kp_d, vp_d, qk, qv, torch.tensor(src, dtype=torch.int32, device=dev()),
                             torch.tensor(dst, dtype=torch.int32, device=dev()), qp, ks, kz, ku,
                             vs, vz, vu, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return new


@pytest.mark.parametrize("D,zp,uns,dtype,vsc,qsc", [(128, 0, False, torch.bfloat16, 1 / 32, 1),
                                                    (64, 128, True, torch.bfloat16, 1 / 32, 1),
                                                    (256, 3, False, torch.bfloat16, 1 / 32, 1),
                                                    (128, 0, False, torch.bfloat16, 1 / 32,
                                                     2.0**-20),
                                                    (64, 9, False, torch.bfloat16, 1 / 32,
                                                     2.0**17),
                                                    (128, 7, False, torch.float16, 1.0, 1),
                                                    (64, 150, True, torch.float16, 1.0, 1)])
def test_grid_values_equal_16bit_decode(K, D, zp, uns, dtype, vsc, qsc):
    """K values k * 2^-5 and V values k * vsc (|k| <= 100): the int8 pages
    reconstruct exactly and the int8 decode equals the 16-bit paged decode
    bit for bit.  Every code reaches an f16 MMA as the half 1024 + code
    minus the zero point; for bf16 pages the K codes meet an fp16 copy of
    the query and the V codes the bf16-rounded probabilities (times the V
    scale and a power of two) handed on as fp16.  The int8 path applies a
    page's V scale to the probabilities before they are packed; in fp16 a
    small product falls below the normal range and rounds differently from
    the unscaled probability of 16-bit pages, so the fp16 cases keep a V
    scale of 1.  qsc scales two query heads (of two groups) out of fp16's
    exact range, 2^-20 below it and 2^17 above it: those groups' K codes
    keep the bf16 route, and they still match bit for bit."""
    B, Hkv, g, P, max_pages = 4, 2, 4, 64, 8
    Hq = Hkv * g
    n_pool = B * max_pages + 3
    grid = lambda s, sc: (synth.randint(-100, 101, (n_pool, Hkv, P, D), 62, s).float() *
                          sc).to(dtype)
    kp, vp, table = _paged_setup(B, Hkv, D, P, max_pages, 3, 62, dtype,
                                 values=(grid(1, 1 / 32), grid(2, vsc)))
    gk, gv = kp.to(dev()), vp.to(dev())
    T = np.array([1, 64, 300, 512])
    qk, qv, qp = _q8_pools(B * max_pages, Hkv, P, D)
    qtab = _quantize_table(K, table, T, P, gk, gv, qk, qv, qp, 1 / 32, zp, uns, vsc, zp, uns,
                           keep_last=False)
    cos, sin = synth.rope_cache(1024, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    q = synth.normal((B, Hq, 1, D), 62, 3, dtype)
    q[0, 1] *= qsc
    q[2, g + 2] *= qsc
    q = q.to(dev())
    st = status()
    L = K.kvc_seq_lengths(torch.from_numpy((T - 1).astype(np.int32)).to(dev()), 1,
                          max_pages * P, K.KVC_CONTIGUOUS, status=st)
    o16 = torch.empty(B, Hq, 1, D, dtype=dtype, device=dev())
    o8 = torch.full_like(o16, float("nan"))
    K.kvc_gqa_decode_paged(o16, q, gk, gv, torch.from_numpy(table).to(dev()), L, rope=rope_d,
                           status=st)
    K.kvc_gqa_decode_paged_q(o8, q, gk, gv, qk, qv, qp, torch.from_numpy(qtab).to(dev()), L,
                             rope=rope_d, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.isfinite(o16).all()
    assert torch.equal(o8, o16)


def test_full_size_int8_cold_pages(K, orc):
    w = synth.CONTIG_DECODE
    B, Hq, Hkv, D, C = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.capacity
    P = 64
    max_pages = C // P
    kp, vp, table = _paged_setup(B, Hkv, D, P, max_pages, 5, 63, torch.bfloat16)
    gk, gv = kp.to(dev()), vp.to(dev())
    T = synth.randint(w.total_lo, w.total_hi + 1, (B,), 63, 3).numpy()
    T[:3] = [w.total_lo, C, 577]
    qk, qv, qp = _q8_pools(B * max_pages, Hkv, P, D)
    qtab = _quantize_table(K, table, T, P, gk, gv, qk, qv, qp, 0.04, 0, False, 0.04, 0, False)
    cos, sin = synth.rope_cache(C + 1, D, w.theta)
    rope_d = (cos.to(dev()), sin.to(dev()))
    q = synth.normal((B, Hq, 1, D), 63, 6)
    st = status()
    L = K.kvc_seq_lengths(torch.from_numpy((T - 1).astype(np.int32)).to(dev()), 1, C,
                          K.KVC_CONTIGUOUS, status=st)
    out = torch.full((B, Hq, 1, D), float("nan"), dtype=torch.bfloat16, device=dev())
    K.kvc_gqa_decode_paged_q(out, q.to(dev()), gk, gv, qk, qv, qp,
                             torch.from_numpy(qtab).to(dev()), L, rope=rope_d, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    rows = [0, 1, 2, 9, 31]
    nqk, nqv = _pools_np(qk, qv)
    want, _ = orc.paged_attention_q(synth.bits(q)[rows], synth.bits(kp), synth.bits(vp), nqk,
                                    nqv, qp.cpu().numpy(), qtab[rows], P, T[rows], T[rows],
                                    cos_cache=cos.numpy(), sin_cache=sin.numpy())
    assert_close(out[rows], want, 2e-2, "int8 cold pages")


@pytest.mark.parametrize("P,D,g,W,dtype,uns", [(64, 128, 4, 700, torch.bfloat16, False),
                                               (128, 64, 8, 100, torch.float16, True),
                                               (256, 128, 2, 0, torch.bfloat16, True),
                                               (64, 64, 16, 1, torch.bfloat16, False),
                                               (64, 256, 2, 1000, torch.bfloat16, False),
                                               (128, 256, 8, 0, torch.float16, True)])
def test_mixed_tables(K, orc, P, D, g, W, dtype, uns):
    B, Hkv, max_pages = 4, 2, 12
    Hq = Hkv * g
    kp, vp, table = _paged_setup(B, Hkv, D, P, max_pages, 4, 64 + P + D, dtype)
    gk, gv = kp.to(dev()), vp.to(dev())
    T = np.array([1, P + 5, 5 * P - 1, max_pages * P])
    qk, qv, qp = _q8_pools(B * max_pages, Hkv, P, D)
    zp = 128 if uns else -3
    qtab = _quantize_table(K, table, T, P, gk, gv, qk, qv, qp, 0.035, zp, uns, 0.03, zp, uns)
    # every other quantized page of row 3 goes back to its 16-bit original
    for j in range(0, max_pages - 1, 2):
        qtab[3, j] = table[3, j]
    cos, sin = synth.rope_cache(max_pages * P + 1, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    q = synth.normal((B, Hq, 1, D), 65, P, dtype)
    st = status()
    L = K.kvc_seq_lengths(torch.from_numpy((T - 1).astype(np.int32)).to(dev()), 1,
                          max_pages * P, K.KVC_CONTIGUOUS, status=st)
    out = torch.empty(B, Hq, 1, D, dtype=dtype, device=dev())
    K.kvc_gqa_decode_paged_q(out, q.to(dev()), gk, gv, qk, qv, qp,
                             torch.from_numpy(qtab).to(dev()), L, local_window_size=W,
                             rope=rope_d, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    nqk, nqv = _pools_np(qk, qv)
    want, _ = orc.paged_attention_q(synth.bits(q), synth.bits(kp), synth.bits(vp), nqk, nqv,
                                    qp.cpu().numpy(), qtab, P, T, T, window=W,
                                    cos_cache=cos.numpy(), sin_cache=sin.numpy())
    assert_close(out, want, 2e-2, "mixed table")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_page_scales_differ(K, orc, dtype):
    """Pages of one split quantized with V scales four decades apart (and K
    scales likewise), 16-bit pages among them: the decode scales each int8
    tile's probabilities by its own page's V scale (a bf16 cache by a common
    power of two on top, chosen from the split's largest V scale and taken
    out of the output again), so every page still meets the oracle."""
    B, Hkv, g, D, P, max_pages = 3, 2, 4, 128, 64, 10
    Hq = Hkv * g
    kp, vp, table = _paged_setup(B, Hkv, D, P, max_pages, 2, 67, dtype)
    gk, gv = kp.to(dev()), vp.to(dev())
    T = np.array([max_pages * P, 300, 7 * P + 5])
    qk, qv, qp = _q8_pools(B * max_pages, Hkv, P, D)
    v_scales = [0.0007, 0.013, 5.0, 0.04, 0.9]
    k_scales = [0.02, 0.3, 0.004, 0.05, 0.011]
    qtab, n_q = table.copy(), 0
    for i in range(len(v_scales)):
        src, dst = [], []
        for b in range(B):
            for j in range(i, (int(T[b]) + P - 1) // P - 1, len(v_scales)):
                if (b, j) == (0, 3):
                    continue                       # stays a 16-bit page
                src.append(int(table[b, j]))
                dst.append(n_q)
                qtab[b, j] = K.KVC_PAGE_QUANT | n_q
                n_q += 1
        if src:
            st = status()
            K.kvc_quantize_pages(gk, gv, qk, qv, torch.tensor(src, dtype=torch.int32,
                                                              device=dev()),
                                 torch.tensor(dst, dtype=torch.int32, device=dev()), qp,
                                 k_scales[i], 0, False, v_scales[i], 5, False, status=st)
            torch.cuda.synchronize()
            assert st.item() == 0
    cos, sin = synth.rope_cache(max_pages * P + 1, D)
    rope_d = (cos.to(dev()), sin.to(dev()))
    q = synth.normal((B, Hq, 1, D), 67, 9, dtype)
    st = status()
    L = K.kvc_seq_lengths(torch.from_numpy((T - 1).astype(np.int32)).to(dev()), 1,
                          max_pages * P, K.KVC_CONTIGUOUS, status=st)
    out = torch.full((B, Hq, 1, D), float("nan"), dtype=dtype, device=dev())
    K.kvc_gqa_decode_paged_q(out, q.to(dev()), gk, gv, qk, qv, qp,
                             torch.from_numpy(qtab).to(dev()), L, rope=rope_d, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    nqk, nqv = _pools_np(qk, qv)
    want, _ = orc.paged_attention_q(synth.bits(q), synth.bits(kp), synth.bits(vp), nqk, nqv,
                                    qp.cpu().numpy(), qtab, P, T, T,
                                    cos_cache=cos.numpy(), sin_cache=sin.numpy())
    assert_close(out, want, 2e-2, "per-page scales")


def test_bad_int8_entry(K):
    B, Hq, Hkv, D, P, max_pages = 2, 8, 2, 128, 64, 4
    kp, vp, table = _paged_setup(B, Hkv, D, P, max_pages, 0, 66, torch.bfloat16)
    gk, gv = kp.to(dev()), vp.to(dev())
    qk, qv, qp = _q8_pools(2, Hkv, P, D)
    qtab = table.copy()
    qtab[1, 0] = K.KVC_PAGE_QUANT | 9          # the int8 pool has two pages
    T = np.array([100, 100])
    st = status()
    L = K.kvc_seq_lengths(torch.from_numpy((T - 1).astype(np.int32)).to(dev()), 1,
                          max_pages * P, K.KVC_CONTIGUOUS, status=st)
    out = torch.empty(B, Hq, 1, D, dtype=torch.bfloat16, device=dev())
    K.kvc_gqa_decode_paged_q(out, synth.normal((B, Hq, 1, D), 66, 3).to(dev()), gk, gv, qk, qv,
                             qp, torch.from_numpy(qtab).to(dev()), L, status=st)
    torch.cuda.synchronize()
    assert st.item() == K.KVC_DEV_INDEX_OOB
