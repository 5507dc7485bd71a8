"""Pins for the oracle's RoPE rows and grouped-query attention.

RoPE (absolute-position rotary embedding; "GQA support sliding_window_cache"
and "Stateful decode & KV cache", "Sliding-window ring buffer"):
  * position 0 is the identity, bit for bit;
  * each rotated pair agrees with the complex product (lo + i hi) e^{i theta}
    in float64 to within one float32 rounding per output;
  * the inner product of a rotated query and key depends only on their
    distance (the property that lets the cache origin move), and norms are
    preserved.

Attention ("Persistent KV Cache and Decode Performance Roadmap", Phase 1, with
the PR's causal + local-window mask):
  * against torch's scaled_dot_product_attention in float64 (a library
    routine) with a boolean mask built from positions, GQA expanded by
    repeating KV heads, for decode and chunk shapes, with and without window;
  * closed forms: one visible key gives out = v exactly; a zero query gives
    the mean of the visible values; identical keys give the mean.
  * exactness claims: compacted-window attention equals full-history
    attention under the window mask after any S schedule (bit-exact inside the
    oracle); a width-W ring buffer written by TensorScatter circular equals the
    full cache for one-token decode and for from-zero prefill with chunks
    <= W; a chunk that wraps the ring is inexact for its non-final tokens and
    exact for its final token ("Stateful decode & KV cache").
"""
import numpy as np
import pytest
import torch

from persistent_kv_cache_gb300 import synth


def test_rope_position_zero_is_identity(orc):
    cos, sin = synth.rope_cache(4, 16)
    x = np.random.default_rng(0).standard_normal((3, 16)).astype(np.float32)
    out = orc.rope_rows(x, np.zeros(3, np.int64), cos.numpy(), sin.numpy())
    np.testing.assert_array_equal(out, x)


def test_rope_matches_complex_rotation(orc):
    D = 64
    cos, sin = synth.rope_cache(5000, D)
    cos, sin = cos.numpy(), sin.numpy()
    rng = np.random.default_rng(1)
    x = rng.standard_normal((200, D)).astype(np.float32)
    pos = rng.integers(0, 5000, size=200)
    out = orc.rope_rows(x, pos, cos, sin).astype(np.float64)
    z = (x[:, :D // 2].astype(np.float64) + 1j * x[:, D // 2:].astype(np.float64))
    w = cos[pos].astype(np.float64) + 1j * sin[pos].astype(np.float64)
    ref = z * w
    got = out[:, :D // 2] + 1j * out[:, D // 2:]
    # two products and one sum, each rounded to binary32
    bound = 3 * 2.0**-24 * (np.abs(z) * np.abs(w)) + 1e-30
    assert np.all(np.abs(got.real - ref.real) <= bound)
    assert np.all(np.abs(got.imag - ref.imag) <= bound)


def test_rope_relative_position_and_norm(orc):
    D = 32
    cos, sin = synth.rope_cache(1024, D)
    cos, sin = cos.numpy(), sin.numpy()
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, D)).astype(np.float32)
    k = rng.standard_normal((1, D)).astype(np.float32)

    def dot(pq, pk):
        a = orc.rope_rows(q, np.array([pq]), cos, sin).astype(np.float64)
        b = orc.rope_rows(k, np.array([pk]), cos, sin).astype(np.float64)
        return float((a * b).sum()), float(np.linalg.norm(a))

    base, n0 = dot(40, 13)
    for shift in (1, 7, 300, 900):
        d, n = dot(40 + shift, 13 + shift)
        assert abs(d - base) < 1e-4 * max(1.0, abs(base))
        assert abs(n - np.linalg.norm(q)) < 1e-5 * n
    # a sign error in the rotation would make this fail: distance matters
    other, _ = dot(41, 13)
    assert abs(other - base) > 1e-3


def _rotate_q_f64(q, pos, cos, sin):
    D = q.shape[-1]
    z = q[..., :D // 2].astype(np.float64) + 1j * q[..., D // 2:].astype(np.float64)
    w = cos[pos].astype(np.float64) + 1j * sin[pos].astype(np.float64)
    r = z * w
    return np.concatenate([r.real, r.imag], axis=-1)


def _sdpa_reference(q, k_rows, v_rows, n_rows, total, window, cos=None, sin=None):
    """float64 torch SDPA over the visible rows of each batch row."""
    B, Hq, S, D = q.shape
    Hkv = k_rows.shape[1]
    out = np.zeros((B, Hq, S, D))
    for b in range(B):
        n = int(n_rows[b])
        T = int(total[b])
        kpos = np.arange(T - n, T)
        qpos = np.arange(T - S, T)
        qb = q[b].astype(np.float64)
        if cos is not None:
            qb = _rotate_q_f64(qb, np.broadcast_to(qpos, (Hq, S)), cos, sin)
        vis = kpos[None, :] <= qpos[:, None]
        if window > 0:
            vis &= (qpos[:, None] - kpos[None, :]) < window
        kk = torch.from_numpy(k_rows[b, :, :n].astype(np.float64))
        vv = torch.from_numpy(v_rows[b, :, :n].astype(np.float64))
        kk = kk.repeat_interleave(Hq // Hkv, dim=0)
        vv = vv.repeat_interleave(Hq // Hkv, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(qb)[None], kk[None], vv[None],
            attn_mask=torch.from_numpy(vis)[None, None], scale=1.0 / np.sqrt(D))
        out[b] = o[0].numpy()
    return out


@pytest.mark.parametrize("S,window,g,rope", [(1, 0, 1, False), (1, 0, 4, True),
                                              (1, 5, 2, True), (6, 0, 2, False),
                                              (6, 4, 3, True), (9, 9, 1, True)])
def test_attention_against_sdpa(orc, S, window, g, rope):
    rng = np.random.default_rng(10 + S + window + g)
    B, Hkv, D, R = 3, 2, 16, 24
    Hq = Hkv * g
    q = rng.standard_normal((B, Hq, S, D)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, R, D)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, R, D)).astype(np.float32)
    n_rows = np.array([S, 13, R], dtype=np.int32)
    total = np.array([S, 40, 100], dtype=np.int32)
    cos = sin = None
    if rope:
        c, s = synth.rope_cache(128, D)
        cos, sin = c.numpy(), s.numpy()
    got, flags = orc.gqa_attention(q, k, v, n_rows, total, window=window, cos_cache=cos,
                                   sin_cache=sin)
    assert not flags.any()
    want = _sdpa_reference(q, k, v, n_rows, total, window, cos, sin)
    np.testing.assert_allclose(got, want, rtol=0, atol=2e-6)


def test_attention_closed_forms(orc):
    rng = np.random.default_rng(20)
    B, Hkv, g, D, R = 2, 2, 2, 8, 10
    q = rng.standard_normal((B, Hkv * g, 1, D)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, R, D)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, R, D)).astype(np.float32)
    n_rows = np.array([R, 7], dtype=np.int32)
    total = np.array([R, 30], dtype=np.int32)
    # window 1: only the query's own key (the last row) is visible -> out = v
    got, _ = orc.gqa_attention(q, k, v, n_rows, total, window=1)
    for b in range(B):
        for h in range(Hkv * g):
            np.testing.assert_array_equal(got[b, h, 0], v[b, h // g, n_rows[b] - 1])
    # zero query: uniform weights over the visible rows
    got, _ = orc.gqa_attention(np.zeros_like(q), k, v, n_rows, total, window=4)
    for b in range(B):
        n = n_rows[b]
        want = v[b, :, n - 4:n].astype(np.float64).mean(axis=1)
        np.testing.assert_allclose(got[b, ::g, 0], want, atol=1e-6)
    # identical keys: uniform weights again
    k_eq = np.broadcast_to(k[:, :, :1], k.shape).copy()
    got, _ = orc.gqa_attention(q, k_eq, v, n_rows, total)
    for b in range(B):
        want = v[b, :, :n_rows[b]].astype(np.float64).mean(axis=1)
        np.testing.assert_allclose(got[b, ::g, 0], want, atol=1e-6)


def _full_history_attention(orc, q, hist_k, hist_v, T, window, cos, sin):
    B = q.shape[0]
    n = np.asarray(T, dtype=np.int32)
    return orc.gqa_attention(q, hist_k, hist_v, n, n, window=window, cos_cache=cos,
                             sin_cache=sin)[0]


@pytest.mark.parametrize("seed,policy", [(s, p) for s in range(4) for p in (1, 2)])
def test_compacted_window_equals_full_history(orc, seed, policy):
    """Exactness: any S schedule on a windowed cache with C >= W gives exactly
    the full-history result under the window mask (decode and chunk queries),
    for the compact-every-step layout and for the drifting one."""
    rng = np.random.default_rng(30 + seed)
    B, Hkv, g, D = 2, 2, 2, 8
    W = int(rng.integers(2, 7))
    C = W + int(rng.integers(0, 4))
    cos, sin = [t.numpy() for t in synth.rope_cache(512, D)]
    schedule = [int(x) for x in rng.integers(1, 2 * C + 2, size=6)] + [1] * 8
    rng.shuffle(schedule)
    total_T = sum(schedule)
    k_cache = np.zeros((B, Hkv, C, D), np.uint16)
    v_cache = np.zeros((B, Hkv, C, D), np.uint16)
    hist_k = np.zeros((B, Hkv, total_T, D), np.uint16)
    hist_v = np.zeros((B, Hkv, total_T, D), np.uint16)
    T = 0
    for S in schedule:
        nk = synth.bits(synth.normal((B, Hkv, S, D), seed, 100 + T))
        nv = synth.bits(synth.normal((B, Hkv, S, D), seed, 200 + T))
        q = synth.bits(synth.normal((B, Hkv * g, S, D), seed, 300 + T))
        lens = orc.seq_lengths(np.full(B, T + S - 1, np.int32), S, C, policy, W)
        ks = vs = None
        if S > 1:
            ks = np.zeros((B, Hkv, C + S, D), np.uint16)
            vs = np.zeros((B, Hkv, C + S, D), np.uint16)
        orc.window_append(k_cache, v_cache, nk, nv, lens, True, cos, sin, ks, vs)
        # full history: the same rotated rows, never evicted
        hl = orc.seq_lengths(np.full(B, T + S - 1, np.int32), S, total_T, False)
        orc.window_append(hist_k, hist_v, nk, nv, hl, False, cos, sin)
        if S == 1:
            got = orc.gqa_attention(q, k_cache, v_cache, lens["cache_total"], lens["total_abs"],
                                    window=W, cos_cache=cos, sin_cache=sin)[0]
        else:
            got = orc.gqa_attention(q, ks, vs, lens["cache_past"] + S, lens["total_abs"],
                                    window=W, cos_cache=cos, sin_cache=sin)[0]
        want = _full_history_attention(orc, q, hist_k[:, :, :T + S], hist_v[:, :, :T + S],
                                       np.full(B, T + S), W, cos, sin)
        np.testing.assert_array_equal(got, want)
        T += S


def _ring_attention(orc, q, ring_k, ring_v, T, W, cos, sin):
    """Attend over a width-W ring by listing its slots in position order (slot
    r holds the latest position p < T with p = r mod W)."""
    B = q.shape[0]
    n = min(T, W)
    order = [(T - n + j) % W for j in range(n)]
    k = np.ascontiguousarray(ring_k[:, :, order])
    v = np.ascontiguousarray(ring_v[:, :, order])
    nn = np.full(B, n, np.int32)
    return orc.gqa_attention(q, k, v, nn, np.full(B, T, np.int32), window=W, cos_cache=cos,
                             sin_cache=sin)[0]


def test_ring_buffer_claims(orc):
    B, Hkv, g, D, W = 2, 2, 2, 8, 6
    cos, sin = [t.numpy() for t in synth.rope_cache(256, D)]
    steps = 20
    total = 4 + steps
    hist_k = synth.bits(synth.normal((B, Hkv, total, D), 5, 1))
    hist_v = synth.bits(synth.normal((B, Hkv, total, D), 5, 2))
    ring_k = np.zeros((B, Hkv, W, D), np.uint16)
    ring_v = np.zeros((B, Hkv, W, D), np.uint16)
    # from-zero prefill of 4 <= W tokens written at position 0, then decode
    T = 0
    for S in [4] + [1] * steps:
        wi = np.full(B, T, np.int64)
        ring_k, _ = orc.tensor_scatter(ring_k, np.ascontiguousarray(hist_k[:, :, T:T + S]), wi,
                                       mode=orc.CIRCULAR)
        ring_v, _ = orc.tensor_scatter(ring_v, np.ascontiguousarray(hist_v[:, :, T:T + S]), wi,
                                       mode=orc.CIRCULAR)
        q = synth.bits(synth.normal((B, Hkv * g, 1, D), 6, T))
        got = _ring_attention(orc, q, ring_k, ring_v, T + S, W, cos, sin)
        want = _full_history_attention(orc, q, hist_k[:, :, :T + S], hist_v[:, :, :T + S],
                                       np.full(B, T + S), W, cos, sin)
        np.testing.assert_array_equal(got, want)
        T += S
    # a chunk of S = 4 that wraps the ring: its queries see only the ring
    S = 4
    wi = np.full(B, T - S, np.int64)
    qs = synth.bits(synth.normal((B, Hkv * g, S, D), 7, 0))
    want = _full_history_attention(orc, qs, hist_k[:, :, :T], hist_v[:, :, :T], np.full(B, T),
                                   W, cos, sin)
    order = [(T - W + j) % W for j in range(W)]
    got = orc.gqa_attention(qs, np.ascontiguousarray(ring_k[:, :, order]),
                            np.ascontiguousarray(ring_v[:, :, order]), np.full(B, W, np.int32),
                            np.full(B, T, np.int32), window=W, cos_cache=cos, sin_cache=sin)[0]
    np.testing.assert_array_equal(got[:, :, -1], want[:, :, -1])   # final token exact
    for i in range(S - 1):                                         # earlier ones lose keys
        assert not np.array_equal(got[:, :, i], want[:, :, i])
