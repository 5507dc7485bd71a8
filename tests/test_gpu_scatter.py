"""GPU parity for kvc_tensor_scatter against the oracle, bit for bit:
the page's three worked examples, random small shapes (every axis, both
modes, 1/2/4/8-byte elements, in place and functional, ragged sizes), the
full circular bf16 workload (16, 8, 4096, 128) with S in {1, 16, 64} for 100
seeded steps each plus a forced-wrap set, and the linear out-of-range flag."""
import json
import os

import numpy as np
import pytest
import torch

from _gpu_helpers import assert_bytes_equal, dev, status
from persistent_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tensorscatter_examples.json")


@pytest.fixture(scope="module")
def K():
    from persistent_kv_cache_gb300 import kvc
    return kvc


def test_printed_examples(K, orc):
    for case in json.load(open(GOLDEN))["cases"]:
        past = torch.tensor(case["past_cache"], dtype=torch.float32, device=dev())
        upd = torch.tensor(case["update"], dtype=torch.float32, device=dev())
        wi = torch.tensor(case["write_indices"], dtype=torch.int64, device=dev())
        mode = K.KVC_CIRCULAR if case["mode"] == "circular" else K.KVC_LINEAR
        want = np.asarray(case["present_cache"], dtype=np.float32)
        out = torch.empty_like(past)
        K.kvc_tensor_scatter(out, past, upd, wi, axis=case["axis"], mode=mode)
        assert_bytes_equal(out, want, case["name"] + " functional")
        K.kvc_tensor_scatter(past, past, upd, wi, axis=case["axis"], mode=mode)
        assert_bytes_equal(past, want, case["name"] + " in place")


_TORCH = {np.uint8: torch.uint8, np.float16: torch.float16, np.float32: torch.float32,
          np.float64: torch.float64}


@pytest.mark.parametrize("seed", range(16))
def test_random_shapes(K, orc, seed):
    rng = np.random.default_rng(1000 + seed)
    rank = int(rng.integers(2, 6))
    shape = [int(rng.integers(1, 6)) for _ in range(rank)]
    ax = int(rng.integers(1, rank))
    shape[ax] = int(rng.integers(1, 40))
    M = shape[ax]
    S = int(rng.integers(0, M + 1))
    ush = list(shape)
    ush[ax] = S
    circular = seed % 2 == 1
    npdt = [np.uint8, np.float16, np.float32, np.float64][seed % 4]
    past = rng.integers(0, 250, size=shape).astype(npdt)
    upd = rng.integers(0, 250, size=ush).astype(npdt)
    if circular:
        wi = rng.integers(-3 * M, 3 * M, size=shape[0])
    else:
        wi = rng.integers(0, M - S + 1, size=shape[0])
        if shape[0] > 1:
            wi[-1] = -1
    axis = ax if seed % 3 else ax - rank
    mode = K.KVC_CIRCULAR if circular else K.KVC_LINEAR
    want, flags = orc.tensor_scatter(past, upd, wi, axis=axis, mode=int(circular))
    tp = torch.from_numpy(past).to(dev())
    tu = torch.from_numpy(upd).to(dev())
    tw = torch.from_numpy(wi).to(dev())
    st = status()
    out = torch.full_like(tp, 77)
    K.kvc_tensor_scatter(out, tp, tu, tw, axis=axis, mode=mode, status=st)
    assert_bytes_equal(out, want, "functional")
    K.kvc_tensor_scatter(tp, tp, tu, tw, axis=axis, mode=mode, status=st)
    assert_bytes_equal(tp, want, "in place")
    bad = bool(flags.any())
    assert bool(st.item() & K.KVC_DEV_INDEX_OOB) == bad


def test_absent_write_indices(K, orc):
    rng = np.random.default_rng(5)
    past = rng.standard_normal((3, 4, 9, 6)).astype(np.float32)
    upd = rng.standard_normal((3, 4, 2, 6)).astype(np.float32)
    want, _ = orc.tensor_scatter(past, upd, None)
    t = torch.from_numpy(past).to(dev())
    K.kvc_tensor_scatter(t, t, torch.from_numpy(upd).to(dev()), None)
    assert_bytes_equal(t, want)


def test_strided_views_are_refused(K):
    """A non-contiguous view would be read as if it were dense: refused."""
    t = torch.zeros(2, 3, 16, 8, device=dev())
    upd = torch.zeros(2, 3, 1, 16, device=dev())[..., ::2]  # [2, 3, 1, 8], stride 2
    assert not upd.is_contiguous()
    with pytest.raises(ValueError, match="contiguous"):
        K.kvc_tensor_scatter(t, t, upd)


def test_unaligned_rows(K, orc):
    """Trailing slices of 3 bytes take the byte path."""
    rng = np.random.default_rng(6)
    past = rng.integers(0, 255, size=(2, 5, 7, 3)).astype(np.uint8)
    upd = rng.integers(0, 255, size=(2, 5, 4, 3)).astype(np.uint8)
    wi = np.array([5, -2])
    want, _ = orc.tensor_scatter(past, upd, wi, mode=1)
    t = torch.from_numpy(past).to(dev())
    K.kvc_tensor_scatter(t, t, torch.from_numpy(upd).to(dev()), torch.from_numpy(wi).to(dev()),
                         mode=K.KVC_CIRCULAR)
    assert_bytes_equal(t, want)


@pytest.mark.parametrize("S", [1, 16, 64])
def test_circular_bf16_workload(K, orc, S):
    """(16, 8, 4096, 128) bf16, 100 seeded steps of circular writes with
    wi ~ U[0, 4096), then 8 steps with every write wrapping; the whole cache
    is compared after each block of steps."""
    w = synth.SCATTER
    shape = (w.batch, w.heads, w.max_seq, w.head_dim)
    cache_cpu = synth.normal(shape, 0, 1)
    want = synth.bits(cache_cpu).copy()
    cache = cache_cpu.to(dev())
    st = status()
    for step in range(w.steps_per_len + 8):
        upd = synth.normal((w.batch, w.heads, S, w.head_dim), S, 10 + step)
        if step < w.steps_per_len:
            wi = synth.randint(0, w.max_seq, (w.batch,), S, 5000 + step)
        else:
            lo, hi = (w.max_seq - S + 1, w.max_seq) if S > 1 else (w.max_seq, 2 * w.max_seq)
            wi = synth.randint(lo, hi, (w.batch,), S, 9000 + step)
        K.kvc_tensor_scatter(cache, cache, upd.to(dev()), wi.to(dev()), mode=K.KVC_CIRCULAR,
                             status=st)
        orc.tensor_scatter(want, synth.bits(upd), wi.numpy(), mode=orc.CIRCULAR, out=want)
        if step in (w.steps_per_len - 1, w.steps_per_len + 7):
            torch.cuda.synchronize()
            assert_bytes_equal(cache, want, f"S={S} step {step}")
    assert st.item() == 0


def test_functional_full_size(K, orc):
    w = synth.SCATTER
    shape = (w.batch, w.heads, w.max_seq, w.head_dim)
    past = synth.normal(shape, 1, 1)
    upd = synth.normal((w.batch, w.heads, 64, w.head_dim), 1, 2)
    wi = synth.randint(0, w.max_seq, (w.batch,), 1, 3)
    want, _ = orc.tensor_scatter(synth.bits(past), synth.bits(upd), wi.numpy(), mode=1)
    out = torch.empty(shape, dtype=torch.bfloat16, device=dev())
    K.kvc_tensor_scatter(out, past.to(dev()), upd.to(dev()), wi.to(dev()), mode=K.KVC_CIRCULAR)
    assert_bytes_equal(out, want)


def test_linear_out_of_range_leaves_row(K, orc):
    past = torch.arange(2 * 3 * 8 * 4, dtype=torch.float32).reshape(2, 3, 8, 4)
    upd = -torch.ones(2, 3, 3, 4)
    wi = torch.tensor([6, 2])
    want, flags = orc.tensor_scatter(past.numpy(), upd.numpy(), wi.numpy())
    assert flags[0] != 0 and flags[1] == 0
    t = past.to(dev())
    st = status()
    K.kvc_tensor_scatter(t, t, upd.to(dev()), wi.to(dev()), status=st)
    assert_bytes_equal(t, want)
    assert st.item() == K.KVC_DEV_INDEX_OOB


@pytest.mark.parametrize("case", ["bytes3", "full_ring", "linear_oob", "no_indices",
                                  "many_prefixes", "long_prefix", "wide8_long", "wide4_long",
                                  "wide2_long", "wide1_long", "linear_oob_long"])
def test_functional_edges(K, orc, case):
    """The functional form (present != past) on the shapes that steer its
    path, vector width, grid and index arithmetic: prefixes shorter than one
    16 KB tile of the one-pass kernel take the copy + in-place scatter pair
    (the first five cases); longer ones take the one-pass kernel at 16-, 8-,
    4-, 2- and 1-byte vectors, each with a write that wraps the ring."""
    rng = np.random.default_rng(sum(map(ord, case)))
    npdt, shape, S, mode, wi = {
        # 3-byte rows: the byte-wide path
        "bytes3": (np.uint8, (2, 5, 7, 3), 4, 1, np.array([5, -2])),
        # every row rewritten, indices negative and beyond max_seq
        "full_ring": (np.float32, (3, 2, 9, 4), 9, 1, np.array([-4, 13, 0])),
        # batch row 0 out of range: it must come out equal to past
        "linear_oob": (np.float16, (2, 3, 8, 8), 3, 0, np.array([6, 2])),
        "no_indices": (np.float32, (3, 4, 9, 6), 2, 0, None),
        # more prefixes than one grid dimension holds
        "many_prefixes": (np.uint8, (2, 35000, 3, 16), 2, 1, np.array([1, 5])),
        # a single long prefix spread over many blocks, 16-byte rows
        "long_prefix": (np.float16, (1, 1, 20011, 8), 37, 1, np.array([20000])),
        # one-pass kernel at the narrower vector widths (8-, 4-, 6- and 3-byte rows)
        "wide8_long": (np.float16, (2, 3, 4100, 4), 9, 1, np.array([4095, -3])),
        "wide4_long": (np.float16, (2, 3, 4099, 2), 5, 1, np.array([4097, 7])),
        "wide2_long": (np.float16, (2, 2, 3001, 3), 4, 1, np.array([2999, 3000])),
        "wide1_long": (np.uint8, (2, 2, 1500, 3), 6, 1, np.array([1497, -1])),
        # batch row 0 out of range in the one-pass kernel
        "linear_oob_long": (np.float16, (2, 2, 5000, 8), 11, 0, np.array([4990, 10])),
    }[case]
    ush = list(shape)
    ush[2] = S
    past = rng.integers(0, 250, size=shape).astype(npdt)
    upd = rng.integers(0, 250, size=ush).astype(npdt)
    want, flags = orc.tensor_scatter(past, upd, wi, axis=2, mode=mode)
    tp = torch.from_numpy(past).to(dev())
    out = torch.full_like(tp, 77)
    st = status()
    K.kvc_tensor_scatter(out, tp, torch.from_numpy(upd).to(dev()),
                         None if wi is None else torch.from_numpy(wi).to(dev()), axis=2,
                         mode=K.KVC_CIRCULAR if mode else K.KVC_LINEAR, status=st)
    assert_bytes_equal(out, want, case)
    assert_bytes_equal(tp, past, case + ": past untouched")
    assert bool(st.item() & K.KVC_DEV_INDEX_OOB) == bool(flags.any())
    assert case.startswith("linear_oob") == bool(flags.any())
