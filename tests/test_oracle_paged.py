"""Pins for the oracle's paged cache ("Persistent KV Cache and Decode
Performance Roadmap", Phase 2: fixed-size pages and a page table consumed by
attention).

* Gather: a pool built by cutting a contiguous cache into pages, with the
  pages shuffled and the table permuted to match, gives back the contiguous
  cache byte for byte (so the gather is a bijection of rows, not a copy of
  one page into several).
* Append: over a schedule of chunks and one-token steps, the gathered
  logical rows equal the history (K rotated at its absolute position) after
  every step, and no pool page outside the tables changes.
* Attention: decode and chunk queries over the paged rows equal full-history
  attention bit for bit, with and without a window.
"""
import numpy as np
import pytest

from persistent_kv_cache_gb300 import synth


def test_gather_is_the_contiguous_cache(orc):
    rng = np.random.default_rng(500)
    B, Hkv, P, D, pages_per_row = 3, 2, 4, 8, 5
    C = P * pages_per_row
    cache = rng.integers(0, 2**14, size=(B, Hkv, C, D)).astype(np.uint16)
    # pages in order: page (b, j) holds rows [jP, (j + 1)P) of row b
    pool = cache.reshape(B, Hkv, pages_per_row, P, D).transpose(0, 2, 1, 3, 4)
    pool = np.ascontiguousarray(pool.reshape(B * pages_per_row, Hkv, P, D))
    table = np.arange(B * pages_per_row).reshape(B, pages_per_row)
    perm = rng.permutation(B * pages_per_row)          # new slot of every page
    shuffled = np.empty_like(pool)
    shuffled[perm] = pool
    n = np.array([C, 7, 1])
    got = orc.paged_rows(shuffled, perm[table], n, P)
    for b in range(B):
        np.testing.assert_array_equal(got[b, :, :n[b]], cache[b, :, :n[b]])
    # a wrong page (one table entry moved) is visible
    bad = perm[table].copy()
    bad[0, 1], bad[0, 2] = bad[0, 2], bad[0, 1]
    assert not np.array_equal(orc.paged_rows(shuffled, bad, n, P)[0], got[0])


@pytest.mark.parametrize("seed", range(3))
def test_append_schedules(orc, seed):
    rng = np.random.default_rng(510 + seed)
    B, Hkv, P, D = 3, 2, 4, 8
    max_pages = 9
    n_pool = B * max_pages + 5
    cos, sin = [t.numpy() for t in synth.rope_cache(64, D)]
    table = rng.permutation(n_pool)[:B * max_pages].reshape(B, max_pages)
    k_pool = rng.integers(0, 2**14, size=(n_pool, Hkv, P, D)).astype(np.uint16)
    v_pool = rng.integers(0, 2**14, size=(n_pool, Hkv, P, D)).astype(np.uint16)
    unused = sorted(set(range(n_pool)) - set(table.reshape(-1).tolist()))
    before_unused = k_pool[unused].copy()
    hist_k = [[] for _ in range(B)]
    hist_v = [[] for _ in range(B)]
    T = np.zeros(B, dtype=np.int64)
    for step, S in enumerate([5, 1, 1, 3, 1, 7, 1, 2]):
        nk = synth.bits(synth.normal((B, Hkv, S, D), 20 + seed, step))
        nv = synth.bits(synth.normal((B, Hkv, S, D), 30 + seed, step))
        orc.paged_append(k_pool, v_pool, table, P, nk, nv, T, cos, sin)
        for b in range(B):
            for i in range(S):
                pos = int(T[b]) + i
                hist_k[b].append(orc.rope_rows(nk[b, :, i], np.full(Hkv, pos), cos, sin))
                hist_v[b].append(nv[b, :, i])
        T = T + S
        got_k = orc.paged_rows(k_pool, table, T, P)
        got_v = orc.paged_rows(v_pool, table, T, P)
        for b in range(B):
            np.testing.assert_array_equal(got_k[b, :, :T[b]],
                                          np.stack(hist_k[b], axis=1))
            np.testing.assert_array_equal(got_v[b, :, :T[b]],
                                          np.stack(hist_v[b], axis=1))
    np.testing.assert_array_equal(k_pool[unused], before_unused)


@pytest.mark.parametrize("W", [0, 6])
def test_attention_equals_full_history(orc, W):
    rng = np.random.default_rng(520 + W)
    B, Hkv, g, P, D = 2, 2, 3, 4, 8
    max_pages = 8
    n_pool = B * max_pages
    cos, sin = [t.numpy() for t in synth.rope_cache(64, D)]
    table = rng.permutation(n_pool).reshape(B, max_pages)
    k_pool = np.zeros((n_pool, Hkv, P, D), np.uint16)
    v_pool = np.zeros_like(k_pool)
    total = 30
    raw_k = synth.bits(synth.normal((B, Hkv, total, D), 40, 1))
    raw_v = synth.bits(synth.normal((B, Hkv, total, D), 40, 2))
    hist_k = np.zeros((B, Hkv, total, D), np.uint16)
    hist_v = np.zeros_like(hist_k)
    T = 0
    for S in [6, 1, 1, 4, 1]:
        sl = slice(T, T + S)
        orc.paged_append(k_pool, v_pool, table, P, np.ascontiguousarray(raw_k[:, :, sl]),
                         np.ascontiguousarray(raw_v[:, :, sl]), np.full(B, T), cos, sin)
        hl = orc.seq_lengths(np.full(B, T + S - 1, np.int32), S, total, orc.CONTIGUOUS)
        orc.window_append(hist_k, hist_v, np.ascontiguousarray(raw_k[:, :, sl]),
                          np.ascontiguousarray(raw_v[:, :, sl]), hl, 0, cos, sin)
        T += S
        q = synth.bits(synth.normal((B, Hkv * g, S, D), 41, T))
        n = np.full(B, T)
        got, flags = orc.paged_attention(q, k_pool, v_pool, table, P, n, n, W, cos_cache=cos,
                                         sin_cache=sin)
        assert not flags.any()
        want, _ = orc.gqa_attention(q, np.ascontiguousarray(hist_k[:, :, :T]),
                                    np.ascontiguousarray(hist_v[:, :, :T]), n.astype(np.int32),
                                    n.astype(np.int32), window=W, cos_cache=cos, sin_cache=sin)
        np.testing.assert_array_equal(got, want)
