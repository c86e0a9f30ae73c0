"""The decode step that allocates nothing, called through the C ABI.

Callers that cannot allocate device memory while decoding (a fixed request
memory pool, a host that can pass only the tensors it owns) use
dilution_attn_decode_step_noalloc, whose scratch is a fixed array inside the
library.  Its results must match the ordinary decode step, which takes a
caller workspace, on consecutive calls (the array keeps the previous call's
contents).  This file is collected last so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from long_context_attention_gb300 import binding as b
from long_context_attention_gb300 import inputs
from tests._parity import BF16_OUT_ABS, host64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _state(B, H, T_cap, d, seed):
    kc = inputs.make_like((B, H, T_cap, d), seed=seed, dtype="bf16", device=DEV)
    vc = inputs.make_like((B, H, T_cap, d), seed=seed + 1, dtype="bf16", device=DEV)
    g = torch.Generator(device=DEV).manual_seed(seed + 2)
    dem = torch.rand(B, H, T_cap, generator=g, device=DEV) * 3.0
    return kc, vc, dem


def _raw_noalloc(lib, qn, kn, vn, kc, vc, dem, n_ctx, out, tau, eps):
    B, H, d = qn.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return lib.dilution_attn_decode_step_noalloc(p(qn), p(kn), p(vn), p(kc), p(vc), p(dem), n_ctx, kc.shape[2], p(out),
                                                 B, H, d, tau, eps, b.DA_BF16,
                                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_decode_on_consecutive_calls():
    lib = b.load()
    B, H, d, n0 = 2, 4, 64, 3000
    T_cap = n0 + 8
    tau, eps = 1.0990651, 1e-6
    assert b.dilution_attn_decode_workspace_size(B, H, T_cap, d) <= b.dilution_attn_decode_noalloc_scratch_bytes()
    kc, vc, dem = _state(B, H, T_cap, d, 81)
    kc2, vc2, dem2 = kc.clone(), vc.clone(), dem.clone()
    for step in range(2):
        n = n0 + step
        qn = inputs.make_like((B, H, d), std=1.5, seed=90 + step, dtype="bf16", device=DEV)
        kn = inputs.make_like((B, H, d), seed=100 + step, dtype="bf16", device=DEV)
        vn = inputs.make_like((B, H, d), seed=110 + step, dtype="bf16", device=DEV)
        ref = b.dilution_attn_decode_step(qn, kn, vn, kc, vc, dem, n, tau=tau, eps=eps)
        out = torch.empty_like(qn)
        assert _raw_noalloc(lib, qn, kn, vn, kc2, vc2, dem2, n, out, tau, eps) == b.DA_OK
        torch.cuda.synchronize()
        assert np.abs(host64(out) - host64(ref)).max() <= BF16_OUT_ABS
        rd, nd = host64(dem[:, :, :n + 1]), host64(dem2[:, :, :n + 1])
        assert np.all(np.abs(nd - rd) <= 1e-5 * np.maximum(rd, 1.0) + 1e-6)
        # the fixed array's status word: no error recorded, and reading it clears nothing else
        assert b.dilution_attn_decode_noalloc_get_error() == b.DA_OK
        assert torch.equal(kc2[:, :, n], kn) and torch.equal(vc2[:, :, n], vn)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = b.load()
    B, H, d = 8, 12, 64
    T_cap = 1 << 17    # 8 x 12 x 131072 needs ~50 MB of scratch
    assert b.dilution_attn_decode_workspace_size(B, H, T_cap, d) > b.dilution_attn_decode_noalloc_scratch_bytes()
    small = torch.zeros(16, dtype=torch.bfloat16, device=DEV)
    p = ctypes.c_void_p(small.data_ptr())
    st = lib.dilution_attn_decode_step_noalloc(p, p, p, p, p, p, 0, T_cap, p, B, H, d, 1.0, 1e-6, b.DA_BF16, None)
    assert st == b.DA_ERR_WORKSPACE
