"""GPU parity of dilution_attn_decode_step: against the float64 oracle's decode
step on the exact cache state, and against prefill ("decode step n reproduces
row n of a prefill of n+1 tokens")."""
import numpy as np
import pytest
import torch

import oracle.dilution as od
from long_context_attention_gb300 import binding as b
from long_context_attention_gb300 import inputs
from tests._parity import BF16_OUT_ABS, F32_OUT_REL, host64, row_rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"


def prefill_cache(q, k, v, T_cap, tau, eps):
    """GPU prefill of q/k/v [B,H,n,d]; returns caches with room for T_cap tokens."""
    B, H, n, d = q.shape
    dem = torch.zeros(B, H, T_cap, device=DEV)
    kc = torch.zeros(B, H, T_cap, d, dtype=q.dtype, device=DEV)
    vc = torch.zeros_like(kc)
    kc[:, :, :n] = k
    vc[:, :, :n] = v
    d_out = torch.empty(B, H, n, device=DEV)
    b.dilution_attn_fwd(q, k, v, None, None, None, d_out, tau=tau, eps=eps)
    dem[:, :, :n] = d_out
    return kc, vc, dem


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_equals_longer_prefill(dtype):
    B, H, N, d = 2, 3, 300, 64
    tau, eps = 1.1, 1e-6
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(B, H, N + 3, d, q_std=1.5, pairs=6, seed=41, dtype=dtype))
    kc, vc, dem = prefill_cache(q[:, :, :N].contiguous(), k[:, :, :N].contiguous(), v[:, :, :N].contiguous(),
                                N + 8, tau, eps)
    for step in range(3):
        n = N + step
        out = b.dilution_attn_decode_step(q[:, :, n].contiguous(), k[:, :, n].contiguous(),
                                          v[:, :, n].contiguous(), kc, vc, dem, n, tau=tau, eps=eps)
        full = torch.empty(B, H, n + 1, d, dtype=q.dtype, device=DEV)
        full_dem = torch.empty(B, H, n + 1, device=DEV)
        b.dilution_attn_fwd(q[:, :, :n + 1].contiguous(), k[:, :, :n + 1].contiguous(),
                            v[:, :, :n + 1].contiguous(), full, None, None, full_dem, tau=tau, eps=eps)
        o, fo = host64(out), host64(full[:, :, n])
        if dtype == "f32":
            assert row_rel_err(o, fo) <= 2 * F32_OUT_REL
            assert np.allclose(host64(dem[:, :, :n + 1]), host64(full_dem), rtol=1e-5, atol=1e-6)
        else:
            assert np.abs(o - fo).max() <= BF16_OUT_ABS
            assert np.allclose(host64(dem[:, :, :n + 1]), host64(full_dem), rtol=2e-3, atol=2e-4)
        # appended token landed in the cache
        assert torch.equal(kc[:, :, n], k[:, :, n]) and torch.equal(vc[:, :, n], v[:, :, n])


@pytest.mark.parametrize("n_ctx", [0, 1, 2047, 2048, 4095, 4096, 5000])
def test_decode_matches_oracle_step(n_ctx):
    """Arbitrary cache state (random positive demand) -> oracle decode step."""
    B, H, d, T_cap = 2, 2, 64, n_ctx + 16
    tau, eps = 1.0990651, 1e-6
    kc, vc = (x.to(DEV) for x in inputs.make_qkv(B, H, T_cap, d, seed=51, dtype="bf16")[1:])
    dem = (torch.rand(B, H, T_cap, generator=torch.Generator().manual_seed(5)) * 3).to(DEV)
    qn, kn, vn = (inputs.make_like((B, H, d), std=s, seed=60 + i, dtype="bf16").to(DEV)
                  for i, s in enumerate((1.5, 1.0, 1.0)))
    ref_out, ref_dem = od.dilution_decode_step(host64(qn), host64(kn), host64(vn), host64(kc), host64(vc),
                                               host64(dem), n_ctx, tau, eps)
    out = b.dilution_attn_decode_step(qn, kn, vn, kc, vc, dem, n_ctx, tau=tau, eps=eps)
    torch.cuda.synchronize()
    assert np.abs(host64(out) - ref_out).max() <= BF16_OUT_ABS
    assert np.all(np.abs(host64(dem[:, :, :n_ctx + 1]) - ref_dem) <= 1e-5 * np.maximum(ref_dem, 1.0) + 1e-6)


def test_decode_config_ctx131072_sampled():
    """8 caches of 131072 tokens (the decode workload's size); the oracle step
    runs on the exact cache state of sampled heads."""
    w = inputs.WORKLOADS["decode_bf16_ctx131072"]
    B, H, N, d = w.B, w.H, w.T, w.d
    T_cap = N + 256
    tau = od.yarn_tau(w.tau_scale)
    kc = inputs.make_like((B, H, T_cap, d), seed=71, dtype="bf16", device=DEV)
    vc = inputs.make_like((B, H, T_cap, d), seed=72, dtype="bf16", device=DEV)
    g = torch.Generator(device=DEV).manual_seed(73)
    dem = torch.rand(B, H, T_cap, generator=g, device=DEV) * 4.0
    qn = inputs.make_like((B, H, d), std=1.5, seed=74, dtype="bf16", device=DEV)
    kn = inputs.make_like((B, H, d), seed=75, dtype="bf16", device=DEV)
    vn = inputs.make_like((B, H, d), seed=76, dtype="bf16", device=DEV)
    heads = [(0, 0), (7, 11)]
    before = {hd: (host64(kc[hd]), host64(vc[hd]), host64(dem[hd])) for hd in heads}
    out = b.dilution_attn_decode_step(qn, kn, vn, kc, vc, dem, N, tau=tau, eps=w.eps)
    torch.cuda.synchronize()
    for hd in heads:
        kk, vv, dd = before[hd]
        ro, rd, _, _ = od.dilution_decode_step_head(host64(qn[hd]), host64(kn[hd]), host64(vn[hd]), kk, vv, dd, N,
                                                    tau, w.eps)
        assert np.abs(host64(out[hd]) - ro).max() <= BF16_OUT_ABS
        assert np.all(np.abs(host64(dem[hd][:N + 1]) - rd) <= 1e-5 * np.maximum(rd, 1.0) + 1e-6)
