"""Pins of the oracle's affine page quantization ("Persistent input/output
feedback", "Optional heterogeneous paged KV": selected-block quantization and
the paragraph on its rounding and fixtures; roadmap "Phase 3: cache
quantization and fusion").

* rounding: ties to even, values from a hand-made table;
* saturation to the INT8 / UINT8 code ranges;
* the pages' bound: a non-saturated reconstruction is within scale / 2 of its
  source (plus float32 rounding);
* UINT8 with zero point z stores the same bytes as INT8 with z - 128;
* values on the scale's grid reconstruct exactly, so attention over such a
  quantized page equals dense attention;
* the pages' four-step fixture: Q/K/V components +-0.173 * step, INT8 scale
  0.01 zero point 0 and UINT8 scale 0.01 zero point 128, attention within
  0.01 of unquantized dense attention;
* a paged cache with no quantized page is the paged attention of 16-bit rows.
"""
import numpy as np
import pytest

import oracle


def test_ties_to_even():
    x = np.array([0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 0.49, 0.51, -0.51], np.float32)
    want = [0, 2, 2, 4, 0, -2, -2, 0, 1, -1]
    assert oracle.quantize_affine(x, 1.0, 0).tolist() == want
    # the same ties through a scale: x / 0.25 = 0.5, 1.5, 2.5
    assert oracle.quantize_affine(np.float32([0.125, 0.375, 0.625]), 0.25, 0).tolist() == [0, 2, 2]
    # and with a zero point (added after rounding)
    assert oracle.quantize_affine(np.float32([0.5, 1.5]), 1.0, 10).tolist() == [10, 12]


def test_saturation():
    big = np.float32([1e4, -1e4, 1e30, -1e30])
    assert oracle.quantize_affine(big, 0.01, 0).tolist() == [127, -128, 127, -128]
    assert oracle.quantize_affine(big, 0.01, 128, unsigned=True).tolist() == [255, 0, 255, 0]
    # the edges themselves
    edge = np.float32([1.27, -1.28, 1.275, -1.285])
    assert oracle.quantize_affine(edge, 0.01, 0).tolist() == [127, -128, 127, -128]


@pytest.mark.parametrize("scale,zp,unsigned", [(0.01, 0, False), (0.05, 128, True),
                                               (0.003, -20, False), (1.0 / 64, 100, True)])
def test_reconstruction_bound(scale, zp, unsigned):
    rng = np.random.default_rng(1)
    lo, hi = (0, 255) if unsigned else (-128, 127)
    # values whose codes stay inside the range
    x = rng.uniform((lo - zp + 1) * scale, (hi - zp - 1) * scale, 20000).astype(np.float32)
    c = oracle.quantize_affine(x, scale, zp, unsigned)
    assert c.min() >= lo and c.max() <= hi
    err = np.abs(oracle.dequantize_affine(c, scale, zp).astype(np.float64) - x)
    assert err.max() <= scale / 2 * (1 + 1e-5) + 1e-7


def test_uint8_is_int8_with_shifted_zero_point():
    rng = np.random.default_rng(2)
    page = rng.normal(0, 0.5, (2, 64, 32)).astype(np.float32)
    s_u, z_u = oracle.quantize_page(page, 0.01, 128, unsigned=True)
    s_i, z_i = oracle.quantize_page(page, 0.01, 0, unsigned=False)
    assert z_u == z_i == 128
    assert np.array_equal(s_u, s_i)
    s_u, z_u = oracle.quantize_page(page, 0.02, 140, unsigned=True)
    s_i, z_i = oracle.quantize_page(page, 0.02, 12, unsigned=False)
    assert z_u == z_i == 140 and np.array_equal(s_u, s_i)


def _one_page_cache(k, v, P):
    """[1, 1, P, D] pools holding k, v ([n, D]) in page 0."""
    n, D = k.shape
    kp = np.zeros((1, 1, P, D), np.float32)
    vp = np.zeros_like(kp)
    kp[0, 0, :n], vp[0, 0, :n] = k, v
    return kp, vp


def _quant_pools(kp, vp, ks, kz, vs, vz, unsigned):
    qk, zk = oracle.quantize_page(kp, ks, kz, unsigned)
    qv, zv = oracle.quantize_page(vp, vs, vz, unsigned)
    return qk, qv, np.array([[ks, zk, vs, zv]], np.float32)


def test_grid_values_are_exact():
    """K and V on the grid of a power-of-two scale: the quantized page
    reconstructs exactly, so its attention equals dense attention."""
    rng = np.random.default_rng(3)
    n, D, P = 40, 16, 64
    scale = 1.0 / 32
    k = (rng.integers(-100, 100, (n, D)) * scale).astype(np.float32)
    v = (rng.integers(-100, 100, (n, D)) * scale).astype(np.float32)
    q = rng.normal(0, 1, (1, 2, 1, D)).astype(np.float32)
    kp, vp = _one_page_cache(k, v, P)
    qk, qv, qp = _quant_pools(kp, vp, scale, 0, scale, 0, False)
    table = np.array([[oracle.PAGE_QUANT | 0]], np.int32)
    got, _ = oracle.paged_attention_q(q, kp, vp, qk, qv, qp, table, P, [n], [n])
    want, _ = oracle.gqa_attention(q, kp, vp, np.int32([n]), np.int32([n]))
    assert np.array_equal(got, want)


@pytest.mark.parametrize("zp,unsigned", [(0, False), (128, True)])
def test_pages_four_step_fixture(zp, unsigned):
    """The pages' end-to-end fixture: four steps, each appending one token
    whose Q/K/V components are +-0.173 * step (sign alternating along the
    head dimension), K and V quantized with scale 0.01; every step's output
    is within 0.01 of unquantized dense attention."""
    D, P = 8, 16
    sign = np.where(np.arange(D) % 2 == 0, 1.0, -1.0).astype(np.float32)
    ks, vs = [], []
    for step in range(1, 5):
        comp = np.float32(0.173 * step) * sign
        ks.append(comp)
        vs.append(comp)
        q = comp.reshape(1, 1, 1, D)
        k, v = np.stack(ks), np.stack(vs)
        kp, vp = _one_page_cache(k, v, P)
        qk, qv, qp = _quant_pools(kp, vp, 0.01, zp, 0.01, zp, unsigned)
        table = np.array([[oracle.PAGE_QUANT | 0]], np.int32)
        got, _ = oracle.paged_attention_q(q, kp, vp, qk, qv, qp, table, P, [step], [step])
        want, _ = oracle.gqa_attention(q, kp, vp, np.int32([step]), np.int32([step]))
        assert np.abs(got - want).max() <= 0.01, step


def test_unquantized_table_is_paged_attention():
    rng = np.random.default_rng(4)
    B, Hkv, Hq, D, P, pages = 2, 2, 4, 16, 64, 6
    kp = (rng.normal(0, 1, (pages, Hkv, P, D)).astype(np.float32))
    vp = (rng.normal(0, 1, (pages, Hkv, P, D)).astype(np.float32))
    table = np.array([[3, 1, 5], [0, 2, 4]], np.int32)
    n = [150, 70]
    q = rng.normal(0, 1, (B, Hq, 1, D)).astype(np.float32)
    qk = np.zeros((1, Hkv, P, D), np.uint8)
    qp = np.zeros((1, 4), np.float32)
    got, _ = oracle.paged_attention_q(q, kp, vp, qk, qk, qp, table, P, n, n)
    want, _ = oracle.paged_attention(q, kp, vp, table, P, n, n)
    assert np.array_equal(got, want)
