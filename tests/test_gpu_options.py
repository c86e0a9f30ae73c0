"""GPU parity of the *_ex entry points against the float64 oracle: the
earlier-demand-only variant (share = p / (committed + eps), "DilutionAttention
v0.1.0 · results", paragraph after "The operator") and per-(batch, head) logit
multipliers (the per-head temperature of "Learning to Focus: Focal Attention
for Selective and Scalable Transformers", section "Transformer with Learned
Temperature").  Tolerances are those of the default operator's tests."""
import numpy as np
import pytest
import torch

import oracle.dilution as od
from long_context_attention_gb300 import binding as b
from long_context_attention_gb300 import inputs
from tests._parity import BF16_OUT_ABS, F32_OUT_REL, host64, row_rel_err
from tests.test_gpu_forward import check_head

pytestmark = pytest.mark.gpu
DEV = "cuda"
EARLY = b.DA_FLAG_EARLIER_DEMAND_ONLY
TAUS = np.array([[0.0, 0.5, 1.0], [1.5, 2.2, 3.0]])   # [B=2, H=3], tau = 0 included


def run_fwd_ex(q, k, v, tau=1.0, tau_bh=None, eps=1e-6, flags=0):
    B, H, T, _ = q.shape
    out = torch.empty_like(q)
    side = [torch.empty(B, H, T, device=DEV) for _ in range(3)]
    ws = torch.empty(b.dilution_attn_fwd_workspace_size(B, H, T, q.shape[-1], b._dtype_code(q)), dtype=torch.uint8,
                     device=DEV)
    b.dilution_attn_fwd_ex(q, k, v, out, *side, tau=tau, tau_bh=tau_bh, eps=eps, flags=flags, workspace=ws)
    assert b.dilution_attn_get_error(ws) == b.DA_OK
    torch.cuda.synchronize()
    return [host64(x) for x in [out] + side]


def compare_ex(q, k, v, taus, eps, earlier):
    """taus: [B, H] multipliers, passed as a device tensor; oracle per head."""
    dtype = "f32" if q.dtype == torch.float32 else "bf16"
    tau_bh = torch.tensor(taus, dtype=torch.float32, device=DEV).contiguous()
    got = run_fwd_ex(q, k, v, tau=1.0, tau_bh=tau_bh, eps=eps, flags=EARLY if earlier else 0)
    qh, kh, vh = host64(q), host64(k), host64(v)
    B, H = taus.shape
    for bb in range(B):
        for hh in range(H):
            # the oracle takes the multiplier the GPU read: the fp32 value
            tau = float(np.float32(taus[bb, hh]))
            ref = od.dilution_forward_head(qh[bb, hh], kh[bb, hh], vh[bb, hh], tau, eps, earlier_only=earlier)
            # fp32 logits x = tau q.k log2(e) / sqrt(d) carry ~|x| 2^-24 of
            # rounding, a relative error of ~4e-8 |x| in each bid and so in
            # the demand sums: the 1e-6 demand bound widens with the head's
            # largest |x| (planted pairs at tau = 3 reach |x| ~ 80)
            x_max = tau * np.abs(qh[bb, hh] @ kh[bb, hh].T).max() / 8.0 / np.log(2.0)
            check_head([g[bb, hh] for g in got], ref, dtype, dem_rel=max(1e-6, 8e-8 * x_max))
    return got


# ------------------------------------------------------------------ forward
@pytest.mark.parametrize("T", [1, 7, 129, 300])
def test_f32_earlier_only(T):
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(1, 2, T, 64, q_std=1.5, pairs=min(4, T - 1), seed=300 + T))
    compare_ex(q, k, v, np.full((1, 2), 1.2), 1e-6, earlier=True)


@pytest.mark.parametrize("T", [1, 5, 128, 257, 640])
def test_bf16_earlier_only(T):
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(1, 2, T, 64, q_std=1.5, pairs=min(4, T - 1), seed=400 + T,
                                                   dtype="bf16"))
    compare_ex(q, k, v, np.full((1, 2), 1.0), 1e-6, earlier=True)


def test_bf16_earlier_only_tiny_eps():
    # eps = 1e-12: diagonal shares near p_ii / eps ~ 1e12 go through the bf16
    # value product and the fp32 accumulators; most rows are close to v_i
    # (keys whose earlier demand is itself tiny keep large shares too)
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(1, 2, 520, 64, q_std=1.5, pairs=4, seed=77, dtype="bf16"))
    got = compare_ex(q, k, v, np.full((1, 2), 1.0), 1e-12, earlier=True)
    assert np.median(np.abs(got[0] - host64(v))) <= 1e-2


@pytest.mark.parametrize("dtype,T", [("f32", 200), ("bf16", 300), ("bf16", 777)])
def test_tau_per_head(dtype, T):
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(2, 3, T, 64, q_std=1.5, pairs=4, seed=500 + T, dtype=dtype))
    compare_ex(q, k, v, TAUS, 1e-6, earlier=False)


def test_tau_per_head_with_earlier_only():
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(2, 3, 400, 64, q_std=1.5, pairs=4, seed=601, dtype="bf16"))
    compare_ex(q, k, v, TAUS, 1e-6, earlier=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tau_per_head_equal_values_match_scalar(dtype):
    # every entry equal to the scalar: same outputs as the scalar entry point
    # (up to the one rounding of tau * log2(e) / sqrt(d) done on the device)
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(2, 3, 300, 64, q_std=1.5, pairs=4, seed=602, dtype=dtype))
    a = run_fwd_ex(q, k, v, tau=1.25)
    c = run_fwd_ex(q, k, v, tau=1.0, tau_bh=torch.full((6,), 1.25, device=DEV))
    tol = 1e-5 if dtype == "f32" else BF16_OUT_ABS
    assert np.abs(a[0] - c[0]).max() <= tol


def test_tau_per_head_bad_entry_reports_invalid():
    # a NaN multiplier cannot be seen on the host before the launch; the
    # kernels record DA_ERR_INVALID in the status word instead
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(1, 2, 256, 64, seed=603, dtype="bf16"))
    tau_bh = torch.tensor([1.0, float("nan")], device=DEV)
    ws = torch.empty(b.dilution_attn_fwd_workspace_size(1, 2, 256, 64, b.DA_BF16), dtype=torch.uint8, device=DEV)
    b.dilution_attn_fwd_ex(q, k, v, tau_bh=tau_bh, workspace=ws)
    assert b.dilution_attn_get_error(ws) == b.DA_ERR_INVALID
    # the status word was cleared by the read; a good array runs clean again
    b.dilution_attn_fwd_ex(q, k, v, tau_bh=torch.ones(2, device=DEV), workspace=ws)
    assert b.dilution_attn_get_error(ws) == b.DA_OK


def test_tau_bh_wrong_size_rejected_by_binding():
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(1, 2, 16, 64, seed=604, dtype="bf16"))
    with pytest.raises(ValueError):
        b.dilution_attn_fwd_ex(q, k, v, tau_bh=torch.ones(3, device=DEV))


# ------------------------------------------------------------------- decode
@pytest.mark.parametrize("n_ctx", [0, 1, 4095, 5000])
def test_decode_ex_matches_oracle_step(n_ctx):
    B, H, d, T_cap = 2, 3, 64, n_ctx + 16
    eps = 1e-6
    kc, vc = (x.to(DEV) for x in inputs.make_qkv(B, H, T_cap, d, seed=700, dtype="bf16")[1:])
    dem = (torch.rand(B, H, T_cap, generator=torch.Generator().manual_seed(7)) * 3).to(DEV)
    qn, kn, vn = (inputs.make_like((B, H, d), std=s, seed=710 + i, dtype="bf16").to(DEV)
                  for i, s in enumerate((1.5, 1.0, 1.0)))
    taus32 = TAUS.astype(np.float32).astype(np.float64)
    ref_out, ref_dem = od.dilution_decode_step(host64(qn), host64(kn), host64(vn), host64(kc), host64(vc),
                                               host64(dem), n_ctx, taus32, eps, earlier_only=True)
    out = b.dilution_attn_decode_step_ex(qn, kn, vn, kc, vc, dem, n_ctx,
                                         tau_bh=torch.tensor(TAUS, dtype=torch.float32, device=DEV),
                                         eps=eps, flags=EARLY)
    torch.cuda.synchronize()
    assert np.abs(host64(out) - ref_out).max() <= BF16_OUT_ABS
    assert np.all(np.abs(host64(dem[:, :, :n_ctx + 1]) - ref_dem) <= 1e-5 * np.maximum(ref_dem, 1.0) + 1e-6)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_ex_continues_flagged_prefill(dtype):
    # prefill n tokens with the flag, decode token n with the flag: row n of a
    # flagged prefill of n + 1 tokens
    B, H, N, d = 2, 3, 300, 64
    eps = 1e-6
    tau_bh = torch.tensor(TAUS, dtype=torch.float32, device=DEV)
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(B, H, N + 1, d, q_std=1.5, pairs=6, seed=720, dtype=dtype))
    T_cap = N + 8
    kc = torch.zeros(B, H, T_cap, d, dtype=q.dtype, device=DEV)
    vc = torch.zeros_like(kc)
    kc[:, :, :N], vc[:, :, :N] = k[:, :, :N], v[:, :, :N]
    dem = torch.zeros(B, H, T_cap, device=DEV)
    d_out = torch.empty(B, H, N, device=DEV)
    b.dilution_attn_fwd_ex(q[:, :, :N].contiguous(), k[:, :, :N].contiguous(), v[:, :, :N].contiguous(), None,
                           None, None, d_out, tau_bh=tau_bh, eps=eps, flags=EARLY)
    dem[:, :, :N] = d_out
    out = b.dilution_attn_decode_step_ex(q[:, :, N].contiguous(), k[:, :, N].contiguous(), v[:, :, N].contiguous(),
                                         kc, vc, dem, N, tau_bh=tau_bh, eps=eps, flags=EARLY)
    full = b.dilution_attn_fwd_ex(q, k, v, tau_bh=tau_bh, eps=eps, flags=EARLY)
    torch.cuda.synchronize()
    o, fo = host64(out), host64(full[:, :, N])
    if dtype == "f32":
        assert row_rel_err(o, fo) <= 2 * F32_OUT_REL
    else:
        assert np.abs(o - fo).max() <= BF16_OUT_ABS


# ----------------------------------------------------------------- backward
def _rel_to_max(got, ref):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


@pytest.mark.parametrize("dtype,T,earlier,tol", [("f32", 200, True, 2e-4), ("f32", 130, False, 2e-4),
                                                  ("bf16", 129, True, 1.5e-2), ("bf16", 300, False, 1.5e-2)])
def test_bwd_ex_matches_oracle(dtype, T, earlier, tol):
    B, H = TAUS.shape
    eps = 1e-6
    flags = EARLY if earlier else 0
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(B, H, T, 64, q_std=1.5, pairs=4, seed=800 + T, dtype=dtype))
    g = inputs.make_like((B, H, T, 64), seed=900 + T, dtype=dtype, device=DEV)
    tau_bh = torch.tensor(TAUS, dtype=torch.float32, device=DEV)
    lse2 = torch.empty(B, H, T, device=DEV)
    b.dilution_attn_fwd_ex(q, k, v, None, lse2, tau_bh=tau_bh, eps=eps, flags=flags)
    got = b.dilution_attn_bwd_ex(q, k, v, g, lse2, tau_bh=tau_bh, eps=eps, flags=flags)
    torch.cuda.synchronize()
    taus32 = TAUS.astype(np.float32).astype(np.float64)
    ref = od.dilution_backward(host64(q), host64(k), host64(v), host64(g), taus32, eps, earlier_only=earlier)
    for gg, rr in zip(got, ref):
        assert _rel_to_max(host64(gg), rr) <= tol
