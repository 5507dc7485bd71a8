"""kvc_gqa_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (for example an operator inside a host framework that
owns all device memory through its own pool and gives its kernels no way to
ask for scratch).  It must return what kvc_gqa_decode returns with a
caller-allocated workspace, on two calls in a row (the second call finds the
first call's partials still in the library's scratch array), and it must
refuse sizes whose partials do not fit in that array.

This file is named to be collected last, so that a run that stops at the
first failure has already run every other test."""
import numpy as np
import pytest
import torch

from persistent_kv_cache_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = 2e-2  # the bf16 attention tolerance used by every decode test


def _inputs(seed, B=6, Hq=32, Hkv=8, D=128, C=8192):
    T = synth.randint(1, C + 1, (B,), seed, 1).numpy()
    T[0], T[1] = 1, C
    dev = torch.device("cuda")
    kc = synth.normal((B, Hkv, C, D), seed, 2).to(dev)
    vc = synth.normal((B, Hkv, C, D), seed, 3).to(dev)
    q = synth.normal((B, Hq, 1, D), seed, 4).to(dev)
    cos, sin = synth.rope_cache(C, D)
    sk = torch.from_numpy((T - 1).astype(np.int32)).to(dev)
    return kc, vc, q, (cos.to(dev), sin.to(dev)), sk


def test_noalloc_matches_decode_twice():
    from persistent_kv_cache_gb300 import kvc as K
    lib = K.library()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call, seed in enumerate((11, 12)):
        kc, vc, q, rope, sk = _inputs(seed)
        B, Hq, _, D = q.shape
        _, Hkv, C, _ = kc.shape
        # several 512-row splits per row: the partials live in the 16 MiB array
        need = K.kvc_gqa_decode_workspace_size(B, Hq, Hkv, C, D, K.KVC_BF16)
        assert 256 < need <= K.KVC_DECODE_STATIC_SCRATCH_BYTES
        L = K.kvc_seq_lengths(sk, 1, C, 0, status=st)
        want = torch.empty(B, Hq, 1, D, dtype=torch.bfloat16, device="cuda")
        K.kvc_gqa_decode(want, q, kc, vc, L, rope=rope, status=st)
        got = torch.full_like(want, float("nan"))
        rc = lib.kvc_gqa_decode_noalloc(
            got.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), L.c(), B, Hq, Hkv, C, D,
            K.KVC_BF16, 0, 0.0, rope[0].data_ptr(), rope[1].data_ptr(), rope[0].shape[0],
            st.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert rc == K.KVC_OK, f"call {call}: {K.kvc_status_string(rc)}"
        torch.cuda.synchronize()
        assert st.item() == 0
        err = (got.float() - want.float()).abs().max().item()
        assert err <= TOL, f"call {call}: max abs difference {err}"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from persistent_kv_cache_gb300 import kvc as K
    lib = K.library()
    B, Hq, Hkv, C, D = 64, 64, 8, 8192, 128
    assert K.kvc_gqa_decode_workspace_size(B, Hq, Hkv, C, D, K.KVC_BF16) > \
        K.KVC_DECODE_STATIC_SCRATCH_BYTES
    small = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    L = K.Lengths(B, torch.device("cuda"))
    p = small.data_ptr()
    rc = lib.kvc_gqa_decode_noalloc(p, p, p, p, L.c(), B, Hq, Hkv, C, D, K.KVC_BF16, 0, 0.0,
                                    None, None, 0, None, None)
    assert rc == 8  # KVC_ERR_WORKSPACE, nothing enqueued
