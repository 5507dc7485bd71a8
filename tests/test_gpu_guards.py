"""Out-of-bounds write guards for every kernel family that writes device
memory.  Each written operand is the middle of a larger buffer whose first
and last 4 KB hold a sentinel byte; after the call (or a run of calls) both
guard slabs must be byte-identical, so a write past either end of a cache,
stage, page pool, output, length array or workspace fails the test even
when every byte inside the operand is right.  (The parity tests compare the
operands themselves with the oracle; these check what lies around them.)

Families: seq_lengths; TensorScatter in place and functional; the append
(contiguous, ring, one-token compaction in its per-slice and cluster forms,
staging seed and copy-back); the in-place stage; the paged append and the
int8 page conversion; decode (plain, ring, paged, int8 pages, no-alloc) with
its workspace; the fused steps (contiguous, ring, small and large windows);
the chunk attention with its workspace; the windowed step that stages
only hazardous rows (kvc_window_prefill_step).  Tiny shapes, plus the full-size
workloads of the contiguous decode step, the chunked prefill (S = 64) and
the functional TensorScatter.
"""
import numpy as np
import pytest
import torch

from _gpu_helpers import dev, status
from persistent_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu

SENTINEL = 0xA5
G = 4096  # guard bytes on each side (a multiple of 256: alignment is kept)


@pytest.fixture(scope="module")
def K():
    from persistent_kv_cache_gb300 import kvc
    return kvc


class Guarded:
    """A tensor of `shape` placed between two guard slabs of SENTINEL bytes."""

    def __init__(self, shape, dtype, init=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((n + 2 * G,), SENTINEL, dtype=torch.uint8, device=dev())
        self.t = self.buf[G:G + n].view(dtype).view(tuple(shape))
        if init is not None:
            self.t.copy_(init)

    def check(self, what):
        torch.cuda.synchronize()
        for name, slab in (("before", self.buf[:G]), ("after", self.buf[-G:])):
            bad = int((slab != SENTINEL).sum().item())
            assert bad == 0, f"{what}: {bad} guard bytes {name} the operand changed"


def guarded(t, dtype=None):
    return Guarded(t.shape, dtype or t.dtype, init=t.to(dev()))


def glengths(K, B):
    """Lengths whose five arrays sit inside one guarded buffer."""
    g = Guarded((5, B), torch.int32)
    L = K.Lengths(B, dev())
    L.buf = g.t
    L._c = K.KvcLengths(*[g.t[i].data_ptr() for i in range(5)])
    return L, g


def rope(T, D):
    cos, sin = synth.rope_cache(int(T) + 2, D)
    return cos.to(dev()), sin.to(dev())


def test_seq_lengths_and_contiguous_append(K):
    B, Hkv, C, D = 3, 2, 96, 64
    T = np.array([1, 40, 96])
    L, gl = glengths(K, B)
    st = status()
    K.kvc_seq_lengths(torch.from_numpy((T - 1).astype(np.int32)).to(dev()), 1, C,
                      K.KVC_CONTIGUOUS, out=L, status=st)
    kc, vc = guarded(synth.normal((B, Hkv, C, D), 1, 1)), guarded(synth.normal((B, Hkv, C, D), 1, 2))
    nk, nv = synth.normal((B, Hkv, 1, D), 1, 3).to(dev()), synth.normal((B, Hkv, 1, D), 1, 4).to(dev())
    K.kvc_window_append(kc.t, vc.t, nk, nv, L, K.KVC_CONTIGUOUS, rope=rope(C, D), status=st)
    gl.check("lengths")
    kc.check("k cache")
    vc.check("v cache")
    assert st.item() == 0


@pytest.mark.parametrize("C,D", [(128, 64), (4096, 256)])   # per-slice and cluster compaction
def test_compaction_and_ring_append(K, C, D):
    B, Hkv = 3, 2
    T = np.array([1, C, 3 * C + 5])
    st = status()
    rd = rope(T.max(), D)
    for policy in (K.KVC_WINDOWED, K.KVC_DRIFTING, K.KVC_RING):
        W = C if policy != K.KVC_DRIFTING else C - 7
        L, gl = glengths(K, B)
        kc = guarded(synth.normal((B, Hkv, C, D), 2, 1))
        vc = guarded(synth.normal((B, Hkv, C, D), 2, 2))
        for s in range(3):
            sk = torch.from_numpy((T + s - 1).astype(np.int32)).to(dev())
            nk = synth.normal((B, Hkv, 1, D), 2, 10 + s).to(dev())
            nv = synth.normal((B, Hkv, 1, D), 2, 20 + s).to(dev())
            K.kvc_seq_lengths(sk, 1, C, policy, local_window_size=W, out=L, status=st)
            K.kvc_window_append(kc.t, vc.t, nk, nv, L, policy, rope=rd, status=st)
        gl.check(f"lengths, policy {policy}")
        kc.check(f"k cache, policy {policy}")
        vc.check(f"v cache, policy {policy}")
    assert st.item() == 0


def test_staging_seed_and_copy_back(K):
    B, Hkv, C, D, S, W = 3, 2, 96, 128, 40, 96
    P = np.array([0, 70, 500])
    st = status()
    rd = rope(P.max() + S, D)
    L = K.kvc_seq_lengths(torch.from_numpy((P + S - 1).astype(np.int32)).to(dev()), S, C,
                          K.KVC_WINDOWED, local_window_size=W, status=st)
    kc = guarded(synth.normal((B, Hkv, C, D), 3, 1))
    vc = guarded(synth.normal((B, Hkv, C, D), 3, 2))
    ks, vs = Guarded((B, Hkv, C + S, D), torch.bfloat16), Guarded((B, Hkv, C + S, D), torch.bfloat16)
    nk = synth.normal((B, Hkv, S, D), 3, 3).to(dev())
    nv = synth.normal((B, Hkv, S, D), 3, 4).to(dev())
    q = synth.normal((B, 2 * Hkv, S, D), 3, 5).to(dev())
    out = Guarded((B, 2 * Hkv, S, D), torch.bfloat16)
    K.kvc_window_append(kc.t, vc.t, nk, nv, L, K.KVC_WINDOWED, K.KVC_APPEND, ks.t, vs.t, rope=rd,
                        status=st)
    ws = K.prefill_workspace(out.t, ks.t, W)
    gws = None if ws is None else Guarded(ws.shape, torch.uint8)
    K.kvc_gqa_prefill_chunk(out.t, q, ks.t, vs.t, L, local_window_size=W, rope=rd, status=st,
                            workspace=None if gws is None else gws.t)
    K.kvc_window_append(kc.t, vc.t, None, None, L, K.KVC_WINDOWED, K.KVC_COPY_BACK, ks.t, vs.t,
                        rope=rd, status=st)
    for g, what in ((kc, "k cache"), (vc, "v cache"), (ks, "k stage"), (vs, "v stage"),
                    (out, "chunk output")):
        g.check(what)
    if gws is not None:
        gws.check("chunk workspace")
    assert st.item() == 0


def test_inplace_stage(K):
    B, Hkv, C, D, S, W = 3, 2, 128, 128, 64, 100
    P = np.array([0, 100, 900])
    st = status()
    rd = rope(P.max() + S, D)
    L = K.kvc_seq_lengths(torch.from_numpy((P + S - 1).astype(np.int32)).to(dev()), S, C,
                          K.KVC_WINDOWED, local_window_size=W, status=st)
    rk = guarded(synth.normal((B, Hkv, C + S, D), 4, 1))
    rv = guarded(synth.normal((B, Hkv, C + S, D), 4, 2))
    nk = synth.normal((B, Hkv, S, D), 4, 3).to(dev())
    nv = synth.normal((B, Hkv, S, D), 4, 4).to(dev())
    K.kvc_window_append_inplace(rk.t, rv.t, nk, nv, L, C, K.KVC_WINDOWED, K.KVC_APPEND, rope=rd,
                                status=st)
    K.kvc_window_append_inplace(rk.t, rv.t, None, None, L, C, K.KVC_WINDOWED, K.KVC_COPY_BACK,
                                new_tokens=S, rope=rd, status=st)
    rk.check("k rows")
    rv.check("v rows")
    assert st.item() == 0


@pytest.mark.parametrize("shape,S", [((2, 3, 16, 8), 5), ((2, 3, 4099, 2), 7)])
def test_tensor_scatter(K, shape, S):
    past = synth.normal(shape, 5, 1, torch.float16)
    ush = list(shape)
    ush[2] = S
    upd = synth.normal(ush, 5, 2, torch.float16).to(dev())
    wi = torch.tensor([shape[2] - 2, -1], dtype=torch.int64, device=dev())
    inplace = guarded(past)
    K.kvc_tensor_scatter(inplace.t, inplace.t, upd, wi, axis=2, mode=K.KVC_CIRCULAR)
    inplace.check("in place")
    present = Guarded(shape, torch.float16)
    K.kvc_tensor_scatter(present.t, past.to(dev()), upd, wi, axis=2, mode=K.KVC_CIRCULAR)
    present.check("functional")


def test_paged_append_quantize_and_decode(K):
    B, Hkv, g, D, P, max_pages = 3, 2, 4, 128, 64, 4
    Hq = Hkv * g
    n_pool = B * max_pages + 2
    st = status()
    kp = guarded(synth.normal((n_pool, Hkv, P, D), 6, 1))
    vp = guarded(synth.normal((n_pool, Hkv, P, D), 6, 2))
    table = torch.arange(B * max_pages, dtype=torch.int32, device=dev()).view(B, max_pages)
    T = np.array([1, 130, 256])
    rd = rope(T.max(), D)
    L = K.kvc_seq_lengths(torch.from_numpy((T - 1).astype(np.int32)).to(dev()), 1,
                          max_pages * P, K.KVC_CONTIGUOUS, status=st)
    nk = synth.normal((B, Hkv, 1, D), 6, 3).to(dev())
    nv = synth.normal((B, Hkv, 1, D), 6, 4).to(dev())
    K.kvc_paged_append(kp.t, vp.t, nk, nv, table, L, rope=rd, status=st)
    qk = Guarded((B * max_pages, Hkv, P, D), torch.uint8)
    qv = Guarded((B * max_pages, Hkv, P, D), torch.uint8)
    qp = Guarded((B * max_pages, 4), torch.float32)
    src = torch.tensor([0, 1, 4], dtype=torch.int32, device=dev())
    K.kvc_quantize_pages(kp.t, vp.t, qk.t, qv.t, src, src, qp.t, 0.05, status=st)
    q = synth.normal((B, Hq, 1, D), 6, 5).to(dev())
    out = Guarded((B, Hq, 1, D), torch.bfloat16)
    K.kvc_gqa_decode_paged(out.t, q, kp.t, vp.t, table, L, rope=rd, status=st)
    qtab = table.clone()
    qtab[:, 0] |= K.KVC_PAGE_QUANT
    out8 = Guarded((B, Hq, 1, D), torch.bfloat16)
    K.kvc_gqa_decode_paged_q(out8.t, q, kp.t, vp.t, qk.t, qv.t, qp.t, qtab, L, rope=rd,
                             status=st)
    for gd, what in ((kp, "k pool"), (vp, "v pool"), (qk, "int8 k pool"), (qv, "int8 v pool"),
                     (qp, "qparams"), (out, "paged out"), (out8, "int8-page out")):
        gd.check(what)
    assert st.item() == 0


@pytest.mark.parametrize("D,C", [(64, 256), (128, 4096), (256, 4096)])
def test_decode_entry_points(K, D, C):
    """kvc_gqa_decode, _ring and _noalloc: output and workspace (split
    partials for capacities of 2048 and more)."""
    B, Hkv, g = 3, 2, 4
    Hq = Hkv * g
    T = np.array([1, C // 2 + 3, C])
    st = status()
    rd = rope(T.max(), D)
    kc = synth.normal((B, Hkv, C, D), 7, 1).to(dev())
    vc = synth.normal((B, Hkv, C, D), 7, 2).to(dev())
    q = synth.normal((B, Hq, 1, D), 7, 3).to(dev())
    sk = torch.from_numpy((T - 1).astype(np.int32)).to(dev())
    for ring in (False, True):
        L = K.kvc_seq_lengths(sk, 1, C, K.KVC_RING if ring else K.KVC_CONTIGUOUS,
                              local_window_size=C, status=st)
        n = K.kvc_gqa_decode_workspace_size(B, Hq, Hkv, C, D, K.KVC_BF16)
        ws = Guarded((max(n, 256),), torch.uint8)
        out = Guarded((B, Hq, 1, D), torch.bfloat16)
        fn = K.kvc_gqa_decode_ring if ring else K.kvc_gqa_decode
        fn(out.t, q, kc, vc, L, local_window_size=C // 2, rope=rd, workspace=ws.t, status=st)
        out.check(f"out, ring={ring}")
        ws.check(f"workspace, ring={ring}")
    out = Guarded((B, Hq, 1, D), torch.bfloat16)
    K.kvc_gqa_decode_noalloc(out.t, q, kc, vc, L, rope=rd, status=st)
    out.check("no-alloc out")
    assert st.item() == 0


@pytest.mark.parametrize("policy,D,C", [(0, 128, 4096), (3, 256, 4096), (1, 64, 128),
                                        (2, 128, 256), (1, 256, 4096), (2, 128, 1100)])
def test_fused_steps(K, policy, D, C):
    """kvc_decode_step (contiguous, ring) and kvc_window_decode_step (small
    windows on chip; large ones through the workspace)."""
    B, Hkv, g = 3, 2, 4
    Hq = Hkv * g
    W = C if policy != 2 else C - 9
    T = np.array([1, C - 1, C]) if policy == 0 else np.array([1, C, 3 * C + 1])
    st = status()
    rd = rope(T.max() + 2, D)
    kc = guarded(synth.normal((B, Hkv, C, D), 8, 1))
    vc = guarded(synth.normal((B, Hkv, C, D), 8, 2))
    L, gl = glengths(K, B)
    out = Guarded((B, Hq, 1, D), torch.bfloat16)
    q = synth.normal((B, Hq, 1, D), 8, 3).to(dev())
    nk = synth.normal((B, Hkv, 1, D), 8, 4).to(dev())
    nv = synth.normal((B, Hkv, 1, D), 8, 5).to(dev())
    steps = 1 if policy == 0 else 2
    for s in range(steps):
        sk = torch.from_numpy((T + s - 1).astype(np.int32)).to(dev())
        if policy in (0, 3):
            ws = K.decode_step_workspace(out.t, kc.t)
            gws = Guarded(ws.shape, torch.uint8)
            K.kvc_decode_step(out.t, q, kc.t, vc.t, nk, nv, sk, W if policy == 3 else 0,
                              lengths=L, rope=rd, workspace=gws.t, status=st, windowed=policy)
        else:
            ws = K.window_step_workspace(out.t, kc.t)
            gws = None if ws is None else Guarded(ws.shape, torch.uint8)
            K.kvc_window_decode_step(out.t, q, kc.t, vc.t, nk, nv, sk, W, lengths=L, rope=rd,
                                     status=st, windowed=policy,
                                     workspace=None if gws is None else gws.t)
        if gws is not None:
            gws.check(f"workspace step {s}")
    for gd, what in ((kc, "k cache"), (vc, "v cache"), (gl, "lengths"), (out, "out")):
        gd.check(what)
    assert st.item() == 0


def test_full_size_contiguous_step(K):
    w = synth.CONTIG_DECODE
    B, Hq, Hkv, D, C = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.capacity
    T = synth.randint(w.total_lo, w.total_hi + 1, (B,), 9, 1).numpy()
    T[:2] = [w.total_lo, C]
    st = status()
    rd = rope(C, D)
    kc = Guarded((B, Hkv, C, D), torch.bfloat16, torch.randn(B, Hkv, C, D, device=dev()))
    vc = Guarded((B, Hkv, C, D), torch.bfloat16, torch.randn(B, Hkv, C, D, device=dev()))
    out = Guarded((B, Hq, 1, D), torch.bfloat16)
    L, gl = glengths(K, B)
    ws = K.decode_step_workspace(out.t, kc.t)
    gws = Guarded(ws.shape, torch.uint8)
    K.kvc_decode_step(out.t, synth.normal((B, Hq, 1, D), 9, 2).to(dev()), kc.t, vc.t,
                      synth.normal((B, Hkv, 1, D), 9, 3).to(dev()),
                      synth.normal((B, Hkv, 1, D), 9, 4).to(dev()),
                      torch.from_numpy((T - 1).astype(np.int32)).to(dev()), lengths=L, rope=rd,
                      workspace=gws.t, status=st)
    for gd, what in ((kc, "k cache"), (vc, "v cache"), (out, "out"), (gl, "lengths"),
                     (gws, "workspace")):
        gd.check(what)
    assert st.item() == 0


def test_full_size_prefill_chunk_64(K):
    w = synth.WINDOW_PREFILL
    B, Hq, Hkv, D, C, W, S = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.capacity, w.window, 64
    P = synth.randint(w.total_lo, w.total_hi + 1, (B,), 10, 1).numpy()
    P[:2] = [0, C - 10]
    st = status()
    rd = rope(P.max() + S, D)
    L, gl = glengths(K, B)
    K.kvc_seq_lengths(torch.from_numpy((P + S - 1).astype(np.int32)).to(dev()), S, C,
                      K.KVC_WINDOWED, local_window_size=W, out=L, status=st)
    kc = Guarded((B, Hkv, C, D), torch.bfloat16, torch.randn(B, Hkv, C, D, device=dev()))
    vc = Guarded((B, Hkv, C, D), torch.bfloat16, torch.randn(B, Hkv, C, D, device=dev()))
    ks = Guarded((B, Hkv, C + S, D), torch.bfloat16)
    vs = Guarded((B, Hkv, C + S, D), torch.bfloat16)
    out = Guarded((B, Hq, S, D), torch.bfloat16)
    nk = synth.normal((B, Hkv, S, D), 10, 2).to(dev())
    nv = synth.normal((B, Hkv, S, D), 10, 3).to(dev())
    q = synth.normal((B, Hq, S, D), 10, 4).to(dev())
    K.kvc_window_append(kc.t, vc.t, nk, nv, L, K.KVC_WINDOWED, K.KVC_APPEND, ks.t, vs.t, rope=rd,
                        status=st)
    ws = K.prefill_workspace(out.t, ks.t, W)
    gws = None if ws is None else Guarded(ws.shape, torch.uint8)
    K.kvc_gqa_prefill_chunk(out.t, q, ks.t, vs.t, L, local_window_size=W, rope=rd, status=st,
                            workspace=None if gws is None else gws.t)
    K.kvc_window_append(kc.t, vc.t, None, None, L, K.KVC_WINDOWED, K.KVC_COPY_BACK, ks.t, vs.t,
                        rope=rd, status=st)
    for gd, what in ((kc, "k cache"), (vc, "v cache"), (ks, "k stage"), (vs, "v stage"),
                     (out, "out"), (gl, "lengths")):
        gd.check(what)
    if gws is not None:
        gws.check("chunk workspace")
    assert st.item() == 0


def test_full_size_functional_scatter(K):
    w = synth.SCATTER
    shape = (w.batch, w.heads, w.max_seq, w.head_dim)
    past = torch.randn(*shape, device=dev(), dtype=torch.bfloat16)
    upd = synth.normal((w.batch, w.heads, 64, w.head_dim), 11, 1).to(dev())
    wi = synth.randint(0, w.max_seq, (w.batch,), 11, 2).to(dev())
    present = Guarded(shape, torch.bfloat16)
    K.kvc_tensor_scatter(present.t, past, upd, wi, mode=K.KVC_CIRCULAR)
    present.check("present")


@pytest.mark.parametrize("policy,D,C,W,S", [(1, 64, 48, 40, 32), (2, 128, 48, 40, 5),
                                           (1, 256, 4160, 4096, 64), (2, 64, 40, 24, 1)])
def test_window_prefill_step(K, policy, D, C, W, S):
    """kvc_window_prefill_step: the rows it stages (seed, attention,
    copy-back), the rows it moves and appends in place, and its workspace --
    batch rows that fill, that evict only what no query sees and that stage,
    over consecutive steps."""
    B, Hkv, g = 3, 2, 2
    Hq = Hkv * g
    T = np.array([0, C - S, 3 * C + 7])
    st = status()
    rd = rope(T.max() + 3 * S + 2, D)
    kc = guarded(synth.normal((B, Hkv, C, D), 12, 1))
    vc = guarded(synth.normal((B, Hkv, C, D), 12, 2))
    ks = Guarded((B, Hkv, C + S, D), torch.bfloat16) if S > 1 else None
    vs = Guarded((B, Hkv, C + S, D), torch.bfloat16) if S > 1 else None
    out = Guarded((B, Hq, S, D), torch.bfloat16)
    L, gl = glengths(K, B)
    n = K.library().kvc_gqa_prefill_workspace_size(B, Hq, Hkv, S, C, D, K.KVC_BF16, W)
    gws = Guarded((max(n, 256),), torch.uint8)
    for s in range(3):
        sk = torch.from_numpy((T + (s + 1) * S - 1).astype(np.int32)).to(dev())
        K.kvc_seq_lengths(sk, S, C, policy, local_window_size=W, out=L, status=st)
        K.kvc_window_prefill_step(out.t, synth.normal((B, Hq, S, D), 12, 10 + s).to(dev()),
                                  kc.t, vc.t, synth.normal((B, Hkv, S, D), 12, 20 + s).to(dev()),
                                  synth.normal((B, Hkv, S, D), 12, 30 + s).to(dev()), L, policy,
                                  W, None if ks is None else ks.t, None if vs is None else vs.t,
                                  rope=rd, status=st, workspace=gws.t if n else None)
    for gd, what in ((kc, "k cache"), (vc, "v cache"), (out, "out"), (gl, "lengths"),
                     (gws, "workspace")):
        gd.check(what)
    if ks is not None:
        ks.check("k stage")
        vs.check("v stage")
    assert st.item() == 0
