"""GPU parity at head dimension 128 (the head size of every model on
"Learning to Focus: Focal Attention for Selective and Scalable Transformers",
its architecture table) against the float64 oracle: the fp32 and bf16
forward, the cached decode step and the backward, with the tolerances of the
d = 64 tests."""
import numpy as np
import pytest
import torch

import oracle.dilution as od
from long_context_attention_gb300 import binding as b
from long_context_attention_gb300 import inputs
from tests._parity import BF16_OUT_ABS, host64, oracle_forward, row_rel_err
from tests.test_gpu_forward import check_head, compare, run_fwd

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 128


@pytest.mark.parametrize("T", [1, 2, 129, 300])
def test_f32_d128(T):
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(2, 2, T, D, q_std=1.5, pairs=min(4, T - 1), seed=1100 + T))
    compare(q, k, v, tau=1.1, eps=1e-6)


@pytest.mark.parametrize("T", [1, 5, 127, 128, 255, 256, 257, 513, 1000])
def test_bf16_d128(T):
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(1, 3, T, D, q_std=1.5, pairs=min(4, T - 1), seed=1200 + T,
                                                   dtype="bf16"))
    compare(q, k, v, tau=1.0, eps=1e-6)


def test_bf16_d128_rows_of_A_sum_to_one():
    q, k, _ = (x.to(DEV) for x in inputs.make_qkv(1, 2, 700, D, q_std=1.5, pairs=4, seed=1301, dtype="bf16"))
    out = run_fwd(q, k, torch.ones_like(q))[0]
    assert torch.allclose(out.float(), torch.ones_like(out, dtype=torch.float32), atol=1e-5, rtol=0)


def test_bf16_d128_options():
    # per-head multipliers and the earlier-demand-only share at d = 128
    taus = np.array([[0.7, 1.0], [1.3, 2.0]])
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(2, 2, 400, D, q_std=1.5, pairs=4, seed=1302, dtype="bf16"))
    tau_bh = torch.tensor(taus, dtype=torch.float32, device=DEV)
    for flags in (0, b.DA_FLAG_EARLIER_DEMAND_ONLY):
        B, H, T, _ = q.shape
        out = torch.empty_like(q)
        side = [torch.empty(B, H, T, device=DEV) for _ in range(3)]
        b.dilution_attn_fwd_ex(q, k, v, out, *side, tau_bh=tau_bh, eps=1e-6, flags=flags)
        torch.cuda.synchronize()
        got = [host64(x) for x in [out] + side]
        qh, kh, vh = host64(q), host64(k), host64(v)
        for bb in range(B):
            for hh in range(H):
                ref = od.dilution_forward_head(qh[bb, hh], kh[bb, hh], vh[bb, hh], float(np.float32(taus[bb, hh])),
                                               1e-6, earlier_only=flags != 0)
                check_head([g[bb, hh] for g in got], ref, "bf16")


def test_bf16_d128_t4096_sampled():
    # several sweep spans and head groups; the oracle on sampled heads, all rows
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(2, 4, 4096, D, q_std=1.5, pairs=32, seed=1303, dtype="bf16"))
    got = [host64(x) for x in run_fwd(q, k, v)]
    ref = oracle_forward(q, k, v, 1.0, 1e-6, heads=[(0, 0), (1, 3)])
    for (bb, hh), r in ref.items():
        check_head([g[bb, hh] for g in got], r, "bf16")


def test_bf16_d128_config_t16384_full_heads():
    """The head-dimension-128 benchmark workload at full size (4 x 12 x 16384
    x 128), in the launch configuration the benchmark times: two whole heads
    (the first of the first head group of the row statistics and the sweep,
    and the last head) against the oracle row by row (out, lse2, row sums)
    and key by key (demand); the unit-demand invariant on every head."""
    w = inputs.WORKLOADS["fwd_bf16_t16384_d128"]
    q, k, v = (x.to(DEV) for x in inputs.make_workload(w, device=DEV))
    T = w.T
    out, lse2, rs, dem = run_fwd(q, k, v, 1.0, w.eps)
    assert torch.isfinite(out.float()).all()
    err = (dem.double().sum(-1) - T).abs().max().item()
    assert err <= 1e-5 * T, err
    ref = oracle_forward(q, k, v, 1.0, w.eps, heads=[(0, 0), (3, 11)])
    for (bb, hh), r in ref.items():
        check_head([host64(x[bb, hh]) for x in (out, lse2, rs, dem)], r, "bf16")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n_ctx", [0, 4095, 5000])
def test_decode_d128(dtype, n_ctx):
    B, H, T_cap = 2, 2, n_ctx + 16
    tau, eps = 1.0990651, 1e-6
    kc, vc = (x.to(DEV) for x in inputs.make_qkv(B, H, T_cap, D, seed=1400, dtype=dtype)[1:])
    dem = (torch.rand(B, H, T_cap, generator=torch.Generator().manual_seed(14)) * 3).to(DEV)
    qn, kn, vn = (inputs.make_like((B, H, D), std=s, seed=1410 + i, dtype=dtype).to(DEV)
                  for i, s in enumerate((1.5, 1.0, 1.0)))
    ref_out, ref_dem = od.dilution_decode_step(host64(qn), host64(kn), host64(vn), host64(kc), host64(vc),
                                               host64(dem), n_ctx, tau, eps)
    out = b.dilution_attn_decode_step(qn, kn, vn, kc, vc, dem, n_ctx, tau=tau, eps=eps)
    torch.cuda.synchronize()
    if dtype == "f32":
        assert row_rel_err(host64(out), ref_out) <= 2e-5
    else:
        assert np.abs(host64(out) - ref_out).max() <= BF16_OUT_ABS
    assert np.all(np.abs(host64(dem[:, :, :n_ctx + 1]) - ref_dem) <= 1e-5 * np.maximum(ref_dem, 1.0) + 1e-6)
    assert torch.equal(kc[:, :, n_ctx], kn) and torch.equal(vc[:, :, n_ctx], vn)


@pytest.mark.parametrize("dtype,T,tol", [("f32", 200, 2e-4), ("bf16", 129, 1.5e-2), ("bf16", 700, 1.5e-2)])
def test_bwd_d128(dtype, T, tol):
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(1, 2, T, D, q_std=1.5, pairs=4, seed=1500 + T, dtype=dtype))
    g = inputs.make_like((1, 2, T, D), seed=1600 + T, dtype=dtype, device=DEV)
    lse2 = torch.empty(1, 2, T, device=DEV)
    b.dilution_attn_fwd(q, k, v, None, lse2, tau=1.1, eps=1e-6)
    got = b.dilution_attn_bwd(q, k, v, g, lse2, tau=1.1, eps=1e-6)
    torch.cuda.synchronize()
    ref = od.dilution_backward(host64(q), host64(k), host64(v), host64(g), 1.1, 1e-6)
    for gg, rr in zip(got, ref):
        assert float(np.abs(host64(gg) - rr).max() / np.abs(rr).max()) <= tol


def test_bwd_d128_options():
    # tensor-core backward at d = 128 with per-head multipliers and the
    # earlier-demand-only share
    taus = np.array([[0.7, 1.3]])
    B, H, T = 1, 2, 300
    flags = b.DA_FLAG_EARLIER_DEMAND_ONLY
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(B, H, T, D, q_std=1.5, pairs=4, seed=1700, dtype="bf16"))
    g = inputs.make_like((B, H, T, D), seed=1701, dtype="bf16", device=DEV)
    tau_bh = torch.tensor(taus, dtype=torch.float32, device=DEV)
    lse2 = torch.empty(B, H, T, device=DEV)
    b.dilution_attn_fwd_ex(q, k, v, None, lse2, tau_bh=tau_bh, eps=1e-6, flags=flags)
    got = b.dilution_attn_bwd_ex(q, k, v, g, lse2, tau_bh=tau_bh, eps=1e-6, flags=flags)
    torch.cuda.synchronize()
    ref = od.dilution_backward(host64(q), host64(k), host64(v), host64(g), taus.astype(np.float32).astype(np.float64),
                               1e-6, earlier_only=True)
    for gg, rr in zip(got, ref):
        assert float(np.abs(host64(gg) - rr).max() / np.abs(rr).max()) <= 1.5e-2
