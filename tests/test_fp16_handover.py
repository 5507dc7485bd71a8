"""Pins for the two numeric facts the int8-page decode of a bf16 cache rests
on when it hands bf16-rounded values to fp16 tensor-core MMAs (host-side
arithmetic only; the GPU tests check the decode itself).

  * A bf16 value that is 0 or of magnitude in [2^-17, 65504] is exactly
    representable in fp16: a bf16 value has 8 significant bits, fp16 keeps
    11 down to 2^-14 and then a fixed step of 2^-24, so 8 bits fit for
    magnitudes from 2^-17 on, and 65504 is fp16's largest finite value.
    Both bounds are tight (some bf16 values just below 2^-17, and every one
    above 65504, are not), while smaller values with few significant bits
    may still be exact: the test is sufficient, not necessary, which is
    all the decode needs.  It copies the query to fp16 only when every
    element passes, and rounds the scaled probabilities to bf16 before
    handing them on as fp16.
  * The per-CTA power of two 2^k, k = 6 - floor(log2 v) clamped to
    [-64, 64] for the largest V scale v of a split, takes v into
    [2^6, 2^7), so a probability P <= 2^8 (the lazy reference max moves
    past a margin of 8 in log2 units) times v * 2^k stays at or below 2^15,
    inside fp16's range; a smaller V scale gives a smaller product.

Every bf16 bit pattern is checked for the first fact, through torch's own
conversions, not by reasoning about bits.
"""
import math

import numpy as np
import torch


def _all_finite_bf16():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    return x[torch.isfinite(x.float())]


def test_bf16_in_range_is_exact_in_fp16_and_the_bounds_are_tight():
    x = _all_finite_bf16()
    f = x.float()
    back = f.half().float()
    exact = back == f
    a = f.abs()
    predicate = (a == 0) | ((a >= 2.0**-17) & (a <= 65504.0))
    assert bool(exact[predicate].all())
    # just below the lower bound some values lose bits; above 65504 all do
    assert not bool(exact[(a >= 2.0**-18) & (a < 2.0**-17)].all())
    assert not bool(exact[a > 65504.0].any())
    # the edges themselves: 8 significant bits fit from 2^-17 on, not one
    # binade lower (a power of two there still fits)
    for v, ok in ((2.0**-17, True), (2.0**-17 * (1 + 2.0**-7), True),
                  (2.0**-18 * (1 + 2.0**-7), False), (2.0**-18, True),
                  (65280.0, True), (65536.0, False)):
        b = torch.tensor([v], dtype=torch.bfloat16).float()
        assert (b.half().float() == b).item() == ok, v


def _pscale_exponent(v: float) -> int:
    """k of the decode's per-CTA scale 2^k for a largest V scale v > 0."""
    e = int((np.array([v], dtype=np.float32).view(np.uint32)[0] >> 23) & 0xFF) - 127
    return max(-64, min(64, 6 - e))


def test_power_of_two_scale_keeps_products_in_fp16_range():
    rng = np.random.default_rng(0)
    vs = np.concatenate([10.0 ** rng.uniform(-18, 18, 4000),
                         2.0 ** np.arange(-58, 70, dtype=np.float64),
                         [0.04, 1.0 / 32, 0.0007, 5.0, 0.9]]).astype(np.float32)
    for v in vs.tolist():
        k = _pscale_exponent(v)
        if -64 < k < 64:
            m = v * 2.0**k
            assert 2.0**6 <= m < 2.0**7, (v, k)
        # the largest product P * v * 2^k with P <= 2^8 stays finite in fp16
        top = 2.0**8 * v * 2.0**k
        assert top <= 2.0**15 or k == -64, (v, k)
        assert math.isfinite(float(np.float16(min(top, 65504.0))))


def test_scaled_probability_exact_range():
    """The hand-over of P * v * 2^k (rounded to bf16) is exact for every
    value from 2^-17 up to the 2^15 bound, and loses bits below 2^-17."""
    x = _all_finite_bf16().float()
    a = x.abs()
    inside = (a >= 2.0**-17) & (a <= 2.0**15)
    assert torch.equal(x[inside].half().float(), x[inside])
    below = (a > 0) & (a < 2.0**-17)
    assert not torch.equal(x[below].half().float(), x[below])
