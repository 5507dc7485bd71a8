"""Pins for the oracle's sequence lengths and cache append
("GQA support sliding_window_cache", onnxruntime PR 29904, section "Design").

* Lengths: a brute-force simulation of the resident window (a list of token
  positions that receives the S new tokens and then drops its oldest entries
  down to C) gives Lp, E and L for every P in [0, 3C], S in [1, 2C],
  C in [1, 8]; the invariant L = min(T, C) holds; seqlens_k near INT32_MAX is
  handled in 64-bit (the PR's int64 widening) and bad rows are rejected.
* Append: after every step of random S schedules the cache rows [0, L) equal
  the last L tokens of a plain history list byte for byte, rows [L, C) keep
  their previous bytes, and the staging buffer holds the old resident rows
  followed by the new ones.
* Drifting layout (the PR's CPU commit, gap = C - W + 1): a brute-force
  simulation that drops a whole gap-sized block when the list would overflow
  gives L and E for every C in [1, 11], W in [1, C] over 6C + 5 decode steps;
  the page's small-slack case (C = W + 8, 400 decode steps) compacts about 44
  times; gap 1 reduces to the compact-every-step layout; random S schedules
  keep the history invariant with W <= L <= C.
"""
import numpy as np
import pytest

INT32_MAX = 2**31 - 1


def _simulate(P, S, C):
    resident = list(range(P - min(P, C), P))
    Lp = len(resident)
    resident += list(range(P, P + S))
    evicted = 0
    while len(resident) > C:
        resident.pop(0)
        evicted += 1
    return Lp, evicted, len(resident), resident


def test_lengths_brute_force(orc):
    for C in range(1, 9):
        for S in range(1, 2 * C + 1):
            Ps = np.arange(0, 3 * C + 1)
            seqlens = (Ps + S - 1).astype(np.int32)
            out = orc.seq_lengths(seqlens, S, C, windowed=True)
            for j, P in enumerate(Ps):
                Lp, E, L, resident = _simulate(int(P), S, C)
                assert out["flags"][j] == 0
                assert out["past_abs"][j] == P and out["total_abs"][j] == P + S
                assert (out["cache_past"][j], out["evict"][j], out["cache_total"][j]) == (Lp, E, L)
                assert L == min(P + S, C)
                assert resident == list(range(P + S - L, P + S))


def test_lengths_contiguous(orc):
    seqlens = np.array([0, 5, 15, 16, 3], dtype=np.int32)
    out = orc.seq_lengths(seqlens, 1, 16, windowed=False)
    np.testing.assert_array_equal(out["total_abs"][:3], [1, 6, 16])
    np.testing.assert_array_equal(out["cache_past"][:3], [0, 5, 15])
    np.testing.assert_array_equal(out["cache_total"][:3], [1, 6, 16])
    np.testing.assert_array_equal(out["evict"][:3], [0, 0, 0])
    assert out["flags"][3] == orc.BAD_CAPACITY and out["cache_total"][3] == -1
    out2 = orc.seq_lengths(seqlens, 4, 16, windowed=False)
    assert out2["flags"][0] == orc.BAD_SEQLEN  # T = 1 < S = 4
    assert out2["cache_past"][4] == 0 and out2["cache_total"][4] == 4


def test_lengths_int32_edges(orc):
    seqlens = np.array([-1, 0, INT32_MAX - 1, INT32_MAX, -5], dtype=np.int32)
    out = orc.seq_lengths(seqlens, 1, 128, windowed=True)
    assert out["flags"][0] == orc.BAD_SEQLEN          # T = 0 < S
    assert out["flags"][1] == 0 and out["cache_total"][1] == 1
    assert out["flags"][2] == 0                       # T = INT32_MAX fits
    assert out["total_abs"][2] == INT32_MAX and out["cache_total"][2] == 128
    assert out["evict"][2] == 1 and out["cache_past"][2] == 128
    assert out["flags"][3] == orc.BAD_SEQLEN          # T = 2^31 does not
    assert out["flags"][4] == orc.BAD_SEQLEN
    assert all(out[k][3] == -1 for k in ("past_abs", "cache_total", "evict"))


def _run_schedule(orc, C, schedule, windowed, seed, Hkv=2, D=4, B=3, window=0):
    rng = np.random.default_rng(seed)
    k_cache = rng.integers(0, 2**16, size=(B, Hkv, C, D), dtype=np.uint16)
    v_cache = rng.integers(0, 2**16, size=(B, Hkv, C, D), dtype=np.uint16)
    # keep the values finite bf16 patterns so nothing special happens
    k_cache &= 0x3FFF
    v_cache &= 0x3FFF
    hist_k = [[[] for _ in range(Hkv)] for _ in range(B)]
    hist_v = [[[] for _ in range(Hkv)] for _ in range(B)]
    T = np.zeros(B, dtype=np.int64)
    for S in schedule:
        new_k = (rng.integers(0, 2**14, size=(B, Hkv, S, D))).astype(np.uint16)
        new_v = (rng.integers(0, 2**14, size=(B, Hkv, S, D))).astype(np.uint16)
        T_new = T + S
        lens = orc.seq_lengths((T_new - 1).astype(np.int32), S, C, windowed, window)
        assert not lens["flags"].any()
        before_k = k_cache.copy()
        before_v = v_cache.copy()
        k_st = v_st = None
        if windowed and S > 1:
            k_st = np.full((B, Hkv, C + S, D), 0x7FC0, dtype=np.uint16)
            v_st = np.full((B, Hkv, C + S, D), 0x7FC0, dtype=np.uint16)
        flags = orc.window_append(k_cache, v_cache, new_k, new_v, lens, windowed,
                                  k_stage=k_st, v_stage=v_st)
        assert not flags.any()
        for b in range(B):
            L = int(lens["cache_total"][b])
            Lp = int(lens["cache_past"][b])
            if windowed == 2:
                assert min(T_new[b], window) <= L <= C   # the window stays resident
            else:
                assert L == (min(T_new[b], C) if windowed else T_new[b])
            for h in range(Hkv):
                if k_st is not None:
                    np.testing.assert_array_equal(k_st[b, h, :Lp], before_k[b, h, :Lp])
                    np.testing.assert_array_equal(k_st[b, h, Lp:Lp + S], new_k[b, h])
                    np.testing.assert_array_equal(v_st[b, h, Lp:Lp + S], new_v[b, h])
                hist_k[b][h].extend(list(new_k[b, h]))
                hist_v[b][h].extend(list(new_v[b, h]))
                want_k = np.array(hist_k[b][h][len(hist_k[b][h]) - L:])
                want_v = np.array(hist_v[b][h][len(hist_v[b][h]) - L:])
                np.testing.assert_array_equal(k_cache[b, h, :L], want_k)
                np.testing.assert_array_equal(v_cache[b, h, :L], want_v)
                if windowed and S == 1 and int(lens["evict"][b]) >= 1:
                    pass  # a shift rewrote [0, L); rows past L keep stale bytes
                else:
                    # rows beyond the resident window are never written
                    np.testing.assert_array_equal(k_cache[b, h, L:], before_k[b, h, L:])
                    np.testing.assert_array_equal(v_cache[b, h, L:], before_v[b, h, L:])
        T = T_new


@pytest.mark.parametrize("seed", range(6))
def test_windowed_invariant_random_schedules(orc, seed):
    rng = np.random.default_rng(100 + seed)
    C = int(rng.integers(1, 9))
    schedule = [int(x) for x in rng.integers(1, 2 * C + 2, size=10)] + [1] * 12
    rng.shuffle(schedule)
    _run_schedule(orc, C, schedule, windowed=True, seed=seed)


def test_windowed_decode_only(orc):
    _run_schedule(orc, 5, [1] * 14, windowed=True, seed=7)


def test_contiguous_append(orc):
    _run_schedule(orc, 24, [3, 1, 1, 7, 1, 2, 5], windowed=False, seed=8)


def test_rope_applied_to_k_only_at_absolute_positions(orc):
    from persistent_kv_cache_gb300 import synth
    B, Hkv, C, D, S = 2, 2, 4, 8, 3
    cos, sin = synth.rope_cache(64, D)
    cos, sin = cos.numpy(), sin.numpy()
    rng = np.random.default_rng(9)
    k = rng.standard_normal((B, Hkv, C, D)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, C, D)).astype(np.float32)
    nk = rng.standard_normal((B, Hkv, S, D)).astype(np.float32)
    nv = rng.standard_normal((B, Hkv, S, D)).astype(np.float32)
    T = np.array([10, 3])
    lens = orc.seq_lengths((T - 1).astype(np.int32), S, C, True)
    ks = np.zeros((B, Hkv, C + S, D), np.float32)
    vs = np.zeros((B, Hkv, C + S, D), np.float32)
    orc.window_append(k, v, nk, nv, lens, True, cos, sin, ks, vs)
    for b in range(B):
        P = int(T[b]) - S
        L = int(lens["cache_total"][b])
        pos = np.arange(P, P + S)
        want = orc.rope_rows(nk[b], np.tile(pos, Hkv), cos, sin).reshape(Hkv, S, D)
        np.testing.assert_array_equal(k[b, :, L - S:L], want)
        np.testing.assert_array_equal(v[b, :, L - S:L], nv[b])
    # a position outside the cos/sin cache rejects the whole row
    k2, v2 = k.copy(), v.copy()
    lens = orc.seq_lengths(np.array([70, 5], dtype=np.int32), S, C, True)
    flags = orc.window_append(k2, v2, nk, nv, lens, True, cos, sin, ks, vs)
    assert flags[0] == orc.BAD_ROPE and flags[1] == 0
    np.testing.assert_array_equal(k2[0], k[0])
    np.testing.assert_array_equal(v2[0], v[0])


# --------------------------------------------------------------------------
# drifting layout ("GQA support sliding_window_cache", CPU commit: resident
# rows [0, end(T)) with gap = C - W + 1, compaction once every gap steps)
# --------------------------------------------------------------------------

def _drift_simulation(C, W, n_steps):
    """One-token steps on a list of resident positions: append the token;
    when the list would exceed C, drop the oldest gap = C - W + 1 entries
    first (a whole gap-sized block is reclaimed at once)."""
    gap = C - W + 1
    resident, out = [], []
    for T in range(1, n_steps + 1):
        evicted = 0
        if len(resident) + 1 > C:
            resident = resident[gap:]
            evicted = gap
        resident.append(T - 1)
        out.append((len(resident), evicted, list(resident)))
    return out


def test_drift_lengths_against_simulation(orc):
    for C in range(1, 12):
        for W in range(1, C + 1):
            sim = _drift_simulation(C, W, 6 * C + 5)
            sk = np.arange(0, len(sim), dtype=np.int32)
            out = orc.seq_lengths(sk, 1, C, orc.DRIFTING, W)
            for j, (L, E, resident) in enumerate(sim):
                T = j + 1
                assert (out["cache_total"][j], out["evict"][j]) == (L, E), (C, W, T)
                assert out["cache_past"][j] == L - 1 + E
                assert resident == list(range(T - L, T))
                assert L >= min(T, W) and L <= C


def test_drift_page_compaction_count(orc):
    """C = W + 8 over 400 decode steps: one compaction every gap = 9 steps,
    about 44 events (the page's small-slack test)."""
    W = 128
    C = W + 8
    T0 = 2048  # after a long prompt
    sk = np.arange(T0, T0 + 400, dtype=np.int32)
    out = orc.seq_lengths(sk, 1, C, orc.DRIFTING, W)
    events = int((out["evict"] > 0).sum())
    assert events in (44, 45)
    assert set(np.unique(out["evict"]).tolist()) == {0, C - W + 1}


def test_drift_gap_one_is_windowed(orc):
    """C = W gives gap = 1: the drifting layout is the compact-every-step one."""
    for C in (1, 5, 128):
        sk = np.arange(-1 + 1, 4 * C + 3, dtype=np.int32)
        for S in (1, 3):
            a = orc.seq_lengths(sk + S - 1, S, C, orc.DRIFTING, C)
            b = orc.seq_lengths(sk + S - 1, S, C, orc.WINDOWED)
            for f in ("past_abs", "total_abs", "cache_past", "cache_total", "evict"):
                np.testing.assert_array_equal(a[f], b[f])


def test_drift_rejects_bad_window(orc):
    sk = np.array([3, 40], dtype=np.int32)
    for W in (0, 17):
        out = orc.seq_lengths(sk, 1, 16, orc.DRIFTING, W)
        assert (out["flags"] == orc.BAD_CAPACITY).all()
        assert (out["cache_total"] == -1).all()


@pytest.mark.parametrize("seed", range(4))
def test_drift_invariant_random_schedules(orc, seed):
    rng = np.random.default_rng(300 + seed)
    C = int(rng.integers(3, 12))
    W = int(rng.integers(1, C + 1))
    schedule = [1] * 30 + [int(x) for x in rng.integers(2, 2 * C + 2, size=6)]
    rng.shuffle(schedule)
    _run_schedule(orc, C, schedule, 2, seed, window=W)
