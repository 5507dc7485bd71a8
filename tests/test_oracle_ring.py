"""Pins for the oracle's ring buffer ("Stateful decode & KV cache",
"Sliding-window ring buffer"; writes through "TensorScatter" circular mode).

* Slot positions: writing positions 0..T-1 one by one at slot p mod C (a
  plain list simulation) leaves slot r holding the newest p = r (mod C), for
  every C in [1, 9] and T in [0, 3C].
* Append: after random chunk schedules (chunks longer than the ring
  included) every slot holds the history row of the position the
  simulation assigns to it, byte for byte, K rotated at that position.
* Attention: decode over the ring equals full-history attention under the
  window mask bit for bit whenever W <= C (and, with no window, equals the
  full history restricted to the last C tokens); a window narrower than the
  ring uses only the newest W slots.
"""
import numpy as np
import pytest

from persistent_kv_cache_gb300 import synth


def _simulate_slots(T, C):
    slots = [-1] * C
    for p in range(T):
        slots[p % C] = p
    return slots


def test_slot_positions_brute_force(orc):
    for C in range(1, 10):
        for T in range(0, 3 * C + 1):
            assert orc.ring_slot_positions(T, C).tolist() == _simulate_slots(T, C), (C, T)


@pytest.mark.parametrize("seed", range(3))
def test_ring_append_schedules(orc, seed):
    rng = np.random.default_rng(400 + seed)
    B, Hkv, C, D = 2, 2, int(rng.integers(2, 9)), 8
    cos, sin = [t.numpy() for t in synth.rope_cache(512, D)]
    ring_k = np.full((B, Hkv, C, D), 0x7FC0, np.uint16)
    ring_v = np.full((B, Hkv, C, D), 0x7FC0, np.uint16)
    T = np.array([0, int(rng.integers(0, 20))], dtype=np.int64)
    hist_k = {b: {} for b in range(B)}
    hist_v = {b: {} for b in range(B)}
    for step, S in enumerate([int(x) for x in rng.integers(1, 2 * C + 3, size=8)] + [1] * 6):
        nk = synth.bits(synth.normal((B, Hkv, S, D), 40 + seed, step))
        nv = synth.bits(synth.normal((B, Hkv, S, D), 50 + seed, step))
        flags = orc.ring_append(ring_k, ring_v, nk, nv, T, cos, sin)
        assert not flags.any()
        for b in range(B):
            for i in range(S):
                p = int(T[b]) + i
                hist_k[b][p] = orc.rope_rows(nk[b, :, i], np.full(Hkv, p), cos, sin)
                hist_v[b][p] = nv[b, :, i]
        T = T + S
        for b in range(B):
            for r, p in enumerate(_simulate_slots(int(T[b]), C)):
                if p not in hist_k[b]:      # never written by this run: still the fill
                    assert (ring_k[b, :, r] == 0x7FC0).all() and (ring_v[b, :, r] == 0x7FC0).all()
                    continue
                np.testing.assert_array_equal(ring_k[b, :, r], hist_k[b][p])
                np.testing.assert_array_equal(ring_v[b, :, r], hist_v[b][p])


@pytest.mark.parametrize("C,W", [(6, 6), (6, 4), (5, 0)])
def test_ring_decode_equals_full_history(orc, C, W):
    B, Hkv, g, D = 2, 2, 3, 8
    cos, sin = [t.numpy() for t in synth.rope_cache(256, D)]
    total = 30
    raw_k = synth.bits(synth.normal((B, Hkv, total, D), 60, 1))
    raw_v = synth.bits(synth.normal((B, Hkv, total, D), 60, 2))
    ring_k = np.zeros((B, Hkv, C, D), np.uint16)
    ring_v = np.zeros((B, Hkv, C, D), np.uint16)
    hist_k = np.zeros((B, Hkv, total, D), np.uint16)
    hist_v = np.zeros((B, Hkv, total, D), np.uint16)
    T = 0
    for S in [3] + [1] * 20 + [2]:
        P = np.full(B, T, np.int64)
        orc.ring_append(ring_k, ring_v, np.ascontiguousarray(raw_k[:, :, T:T + S]),
                        np.ascontiguousarray(raw_v[:, :, T:T + S]), P, cos, sin)
        hl = orc.seq_lengths(np.full(B, T + S - 1, np.int32), S, total, orc.CONTIGUOUS)
        orc.window_append(hist_k, hist_v, np.ascontiguousarray(raw_k[:, :, T:T + S]),
                          np.ascontiguousarray(raw_v[:, :, T:T + S]), hl, 0, cos, sin)
        T += S
        q = synth.bits(synth.normal((B, Hkv * g, 1, D), 61, T))
        got, flags = orc.ring_attention(q, ring_k, ring_v, np.full(B, T), W, cos_cache=cos,
                                        sin_cache=sin)
        assert not flags.any()
        # the full history, keeping only what a C-slot ring can hold when
        # there is no window
        n = T if W > 0 else min(T, C)
        kk = np.ascontiguousarray(hist_k[:, :, T - n:T])
        vv = np.ascontiguousarray(hist_v[:, :, T - n:T])
        want, _ = orc.gqa_attention(q, kk, vv, np.full(B, n, np.int32), np.full(B, T, np.int32),
                                    window=W, cos_cache=cos, sin_cache=sin)
        np.testing.assert_array_equal(got, want)
