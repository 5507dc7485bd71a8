"""Pins for the rotary cos/sin table that feeds both the oracle and the CUDA
path (``synth.rope_cache``), and for the oracle's pairing of the rotation.

The pages fix RoPE by absolute position with base theta 10000 ("GQA support
sliding_window_cache": cos/sin caches indexed by absolute position;
workloads "RoPE theta 10000").  The table's angle for pair i at position p
is p * 10000^(-2i / D).  The values below come from that formula evaluated
with the ``math`` module, one point at a time, so that a wrong exponent
(-i / D), a wrong base, an off-by-one in i or a transposed table fails:

  * pair 0 turns by exactly one radian per position: cos(p), sin(p);
  * pair i = D / 4 turns by 10000^(-1/2) = 1/100 radian per position, for
    every head dimension;
  * the last pair, i = D/2 - 1, turns by 10000^(-(D - 2) / D) per position.

The rotation pairs element i with element i + D/2 (rotate-half): a one-hot
vector at i becomes cos(angle) at i and sin(angle) at i + D/2, one at
i + D/2 becomes -sin at i and cos at i + D/2, and nothing else moves.
"""
import math

import numpy as np
import pytest

from persistent_kv_cache_gb300 import synth

# one binary32 rounding of a value of magnitude <= 1
ULP1 = 2.0**-24


def _angle(p, i, D, theta=10000.0):
    return p * math.exp(-(2.0 * i / D) * math.log(theta))


@pytest.mark.parametrize("D", [8, 64, 128, 256])
def test_table_shape_and_type(D):
    cos, sin = synth.rope_cache(37, D)
    assert cos.shape == (37, D // 2) and sin.shape == (37, D // 2)
    assert str(cos.dtype) == "torch.float32" and str(sin.dtype) == "torch.float32"


def test_pair_zero_turns_one_radian_per_position():
    cos, sin = [t.numpy() for t in synth.rope_cache(4096, 64)]
    for p in (0, 1, 2, 3, 17, 1000, 4095):
        assert abs(float(cos[p, 0]) - math.cos(p)) <= ULP1
        assert abs(float(sin[p, 0]) - math.sin(p)) <= ULP1
    assert float(cos[1, 0]) == np.float32(math.cos(1.0))
    assert float(sin[1, 0]) == np.float32(math.sin(1.0))


@pytest.mark.parametrize("D", [8, 64, 128, 256])
def test_quarter_pair_turns_a_hundredth_radian(D):
    cos, sin = [t.numpy() for t in synth.rope_cache(20001, D)]
    i = D // 4
    for p in (1, 2, 100, 157, 4096, 8191, 20000):
        assert abs(float(cos[p, i]) - math.cos(p / 100.0)) <= 2 * ULP1, (D, p)
        assert abs(float(sin[p, i]) - math.sin(p / 100.0)) <= 2 * ULP1, (D, p)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_last_pair(D):
    cos, sin = [t.numpy() for t in synth.rope_cache(32769, D)]
    i = D // 2 - 1
    for p in (1, 5, 999, 32768):
        a = _angle(p, i, D)
        assert abs(float(cos[p, i]) - math.cos(a)) <= 2 * ULP1, (D, p)
        assert abs(float(sin[p, i]) - math.sin(a)) <= 2 * ULP1, (D, p)


def test_every_entry_against_the_formula():
    D, N = 32, 300
    cos, sin = [t.numpy() for t in synth.rope_cache(N, D)]
    for p in range(0, N, 7):
        for i in range(D // 2):
            a = _angle(p, i, D)
            assert abs(float(cos[p, i]) - math.cos(a)) <= 2 * ULP1
            assert abs(float(sin[p, i]) - math.sin(a)) <= 2 * ULP1


@pytest.mark.parametrize("D", [8, 64, 256])
def test_rotation_pairs_i_with_i_plus_half(orc, D):
    cos, sin = [t.numpy() for t in synth.rope_cache(64, D)]
    half = D // 2
    p = 37
    for i in (0, 1, half // 2, half - 1):
        for hot, sign_lo, which_lo, which_hi in ((i, 1.0, cos, sin), (i + half, -1.0, sin, cos)):
            x = np.zeros((1, D), np.float32)
            x[0, hot] = 1.0
            out = orc.rope_rows(x, np.array([p]), cos, sin)[0]
            want = np.zeros(D, np.float32)
            want[i] = sign_lo * which_lo[p, i]
            want[i + half] = which_hi[p, i]
            np.testing.assert_array_equal(out, want, err_msg=f"D={D} hot={hot}")
