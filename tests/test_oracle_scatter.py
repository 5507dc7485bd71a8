"""Pins for the oracle's TensorScatter ("TensorScatter" operator page, opset 24).

* The three worked examples printed on the page, matched exactly.
* An independent numpy restatement (vectorised over the prefix dimensions,
  unlike the oracle's scalar loop) on random small shapes: every axis, both
  modes, element sizes 1/2/4/8 bytes, in place and out of place.
* Invariants: rows that are not targeted keep their bytes; a linear write that
  does not fit leaves its batch row untouched and is flagged; an absent
  write_indices behaves as all zeros.
"""
import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tensorscatter_examples.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_printed_examples(orc, case):
    past = np.asarray(case["past_cache"], dtype=np.float32)
    upd = np.asarray(case["update"], dtype=np.float32)
    wi = np.asarray(case["write_indices"], dtype=np.int64)
    mode = orc.CIRCULAR if case["mode"] == "circular" else orc.LINEAR
    present, flags = orc.tensor_scatter(past, upd, wi, axis=case["axis"], mode=mode)
    np.testing.assert_array_equal(present, np.asarray(case["present_cache"], dtype=np.float32))
    assert not flags.any()
    # the same example run in place gives the same bytes
    buf = past.copy()
    orc.tensor_scatter(buf, upd, wi, axis=case["axis"], mode=mode, out=buf)
    np.testing.assert_array_equal(buf, present)


def _numpy_scatter(past, upd, wi, axis, circular):
    """Restatement vectorised over the prefix: view the cache as
    (batch, other prefix dims, max_seq, trailing) and assign whole columns."""
    ax = axis % past.ndim
    B = past.shape[0]
    M = past.shape[ax]
    S = upd.shape[ax]
    pre = int(np.prod(past.shape[1:ax], dtype=np.int64))
    tail = int(np.prod(past.shape[ax + 1:], dtype=np.int64))
    out = past.copy().reshape(B, pre, M, tail)
    u = upd.reshape(B, pre, S, tail)
    ok = np.ones(B, dtype=bool)
    for b in range(B):
        start = 0 if wi is None else int(wi[b])
        seq = np.arange(start, start + S)
        if circular:
            seq = np.mod(seq, M)
        elif start < 0 or start + S > M:
            ok[b] = False
            continue
        out[b][:, seq, :] = u[b]
    return out.reshape(past.shape), ok


@pytest.mark.parametrize("seed", range(12))
def test_random_shapes_against_numpy(orc, seed):
    rng = np.random.default_rng(seed)
    rank = int(rng.integers(2, 6))
    shape = [int(rng.integers(1, 5)) for _ in range(rank)]
    ax = int(rng.integers(1, rank))
    shape[ax] = int(rng.integers(1, 9))
    M = shape[ax]
    S = int(rng.integers(0, M + 1))
    ushape = list(shape)
    ushape[ax] = S
    circular = bool(seed % 2)
    dt = [np.uint8, np.float16, np.float32, np.float64][seed % 4]
    past = rng.integers(0, 250, size=shape).astype(dt)
    upd = rng.integers(0, 250, size=ushape).astype(dt)
    if circular:
        wi = rng.integers(-2 * M, 3 * M, size=shape[0])
    else:
        wi = rng.integers(0, M - S + 1, size=shape[0])
        if shape[0] > 1:
            wi[0] = M - S + 1  # does not fit: must be rejected for that row only
    axis_arg = ax if seed % 3 == 0 else ax - rank
    got, flags = orc.tensor_scatter(past, upd, wi, axis=axis_arg,
                                    mode=orc.CIRCULAR if circular else orc.LINEAR)
    want, ok = _numpy_scatter(past, upd, wi, ax, circular)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(flags != 0, ~ok)


def test_absent_indices_are_zero(orc):
    rng = np.random.default_rng(3)
    past = rng.standard_normal((3, 2, 6, 4)).astype(np.float32)
    upd = rng.standard_normal((3, 2, 2, 4)).astype(np.float32)
    a, _ = orc.tensor_scatter(past, upd, None)
    b, _ = orc.tensor_scatter(past, upd, np.zeros(3, dtype=np.int64))
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(a[:, :, 2:], past[:, :, 2:])
    np.testing.assert_array_equal(a[:, :, :2], upd)


def test_untargeted_rows_keep_bytes(orc):
    rng = np.random.default_rng(4)
    past = rng.integers(0, 2**16, size=(4, 3, 10, 8), dtype=np.uint16)
    upd = rng.integers(0, 2**16, size=(4, 3, 3, 8), dtype=np.uint16)
    wi = np.array([0, 7, 9, 4], dtype=np.int64)
    got, _ = orc.tensor_scatter(past, upd, wi, mode=orc.CIRCULAR)
    for b in range(4):
        hit = {(int(wi[b]) + s) % 10 for s in range(3)}
        for r in range(10):
            if r not in hit:
                np.testing.assert_array_equal(got[b, :, r], past[b, :, r])


def test_update_longer_than_cache_is_rejected(orc):
    past = np.zeros((1, 1, 4, 2), dtype=np.float32)
    upd = np.zeros((1, 1, 5, 2), dtype=np.float32)
    with pytest.raises(ValueError):
        orc.tensor_scatter(past, upd, np.zeros(1, dtype=np.int64), mode=orc.CIRCULAR)


def test_axis_zero_is_rejected(orc):
    past = np.zeros((2, 4), dtype=np.float32)
    with pytest.raises(ValueError):
        orc.tensor_scatter(past, past[:, :1], None, axis=0)
