"""The library's calls captured in CUDA graphs and replayed (the way a serving
loop drives them): the forward and the cached decode step launch only on the
caller's stream, allocate nothing and synchronise nothing, so a captured call
replays on new contents of the same buffers.  After a first ordinary call
(the one-time per-device set-up) each is captured once and replayed; the
forward is checked against the oracle, the decode step bit for bit against
the same step called directly (it is deterministic).

Operator: "DilutionAttention v0.1.0 · results", section "The operator" and
its cached-decoding paragraph.
"""
import numpy as np
import pytest
import torch

import oracle.dilution as od
from long_context_attention_gb300 import binding as b
from long_context_attention_gb300 import inputs
from tests._parity import BF16_OUT_ABS, host64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_forward_replayed_from_cuda_graph():
    B, H, T, d = 1, 4, 1500, 64
    q, k, v = inputs.make_qkv(B, H, T, d, q_std=1.5, pairs=8, seed=401, dtype="bf16", device=DEV)
    out = torch.empty_like(q)
    ws = torch.empty(b.dilution_attn_fwd_workspace_size(B, H, T, d, b.DA_BF16), dtype=torch.uint8, device=DEV)
    b.dilution_attn_fwd(q, k, v, out, workspace=ws)          # one-time set-up outside the capture
    assert b.dilution_attn_get_error(ws) == b.DA_OK
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        b.dilution_attn_fwd(q, k, v, out, workspace=ws)
    for seed in (402, 403):                                   # new inputs in the captured buffers
        q2, k2, v2 = inputs.make_qkv(B, H, T, d, q_std=1.5, pairs=8, seed=seed, dtype="bf16", device=DEV)
        q.copy_(q2), k.copy_(k2), v.copy_(v2)
        g.replay()
        assert b.dilution_attn_get_error(ws) == b.DA_OK
        ref = od.dilution_forward(host64(q), host64(k), host64(v), 1.0, 1e-6)["out"]
        assert np.abs(host64(out) - ref).max() <= BF16_OUT_ABS


def test_decode_step_replayed_from_cuda_graph():
    B, H, d, n_ctx = 2, 3, 64, 3000
    T_cap = n_ctx + 1
    tau, eps = 1.0990651, 1e-6
    kc0, vc0 = (inputs.make_like((B, H, T_cap, d), seed=s, dtype="bf16", device=DEV) for s in (411, 412))
    dem0 = torch.rand(B, H, T_cap, generator=torch.Generator(device=DEV).manual_seed(413), device=DEV) * 2.0
    tok = [inputs.make_like((B, H, d), std=s, seed=414 + i, dtype="bf16", device=DEV)
           for i, s in enumerate((1.5, 1.0, 1.0))]
    ws = torch.empty(b.dilution_attn_decode_workspace_size(B, H, T_cap, d), dtype=torch.uint8, device=DEV)
    # the direct call, on its own copy of the cache
    kd, vd, dd = kc0.clone(), vc0.clone(), dem0.clone()
    want = b.dilution_attn_decode_step(*tok, kd, vd, dd, n_ctx, tau=tau, eps=eps, workspace=ws).clone()
    assert b.dilution_attn_get_error(ws) == b.DA_OK
    # the captured call, on a fresh copy restored before each replay
    kc, vc, dem = kc0.clone(), vc0.clone(), dem0.clone()
    out = torch.empty(B, H, d, dtype=torch.bfloat16, device=DEV)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        b.dilution_attn_decode_step(*tok, kc, vc, dem, n_ctx, out, tau=tau, eps=eps, workspace=ws)
    for _ in range(2):
        kc.copy_(kc0), vc.copy_(vc0), dem.copy_(dem0)
        g.replay()
        assert b.dilution_attn_get_error(ws) == b.DA_OK
        assert torch.equal(out, want)
        assert torch.equal(dem, dd) and torch.equal(kc, kd) and torch.equal(vc, vd)
