"""Shared helpers for the GPU parity tests (inputs from the synth module, the
CUDA path through the C-ABI binding, expected values from the oracle)."""
import numpy as np
import torch

from persistent_kv_cache_gb300 import synth

BF16_TOL = 2e-2
F32_TOL = 1e-4


def dev():
    return torch.device("cuda")


def status():
    return torch.zeros(1, dtype=torch.int32, device=dev())


def lengths_np(L):
    """Lengths object (device) -> dict of numpy arrays for the oracle."""
    out = {f: getattr(L, f).cpu().numpy().copy() for f in L.FIELDS}
    return out


def tol(dtype):
    return F32_TOL if dtype == torch.float32 else BF16_TOL


def assert_bytes_equal(got: torch.Tensor, want_np: np.ndarray, what=""):
    g = synth.bits(got)
    if g.dtype != want_np.dtype:
        want_np = want_np.view(g.dtype)
    if not np.array_equal(g, want_np):
        diff = np.argwhere(g != want_np)
        raise AssertionError(f"{what}: {len(diff)} elements differ, first at {diff[:5].tolist()}")


def assert_close(got: torch.Tensor, want_np: np.ndarray, atol, what=""):
    g = got.detach().float().cpu().numpy()
    if want_np.dtype == np.uint16:
        w = synth.from_bits(want_np, torch.bfloat16).float().numpy()
    else:
        w = want_np.astype(np.float32)
    err = np.abs(g - w)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    assert err.max() <= atol, f"{what}: max abs error {err.max():.3g} > {atol}"
    return float(err.max())
