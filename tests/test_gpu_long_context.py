"""GPU parity at the long-context sizes: the prefill at 1 x 12 x 131072 with the
YaRN multiplier for s = 8, a chain of cached decode steps that starts from a
real prefill, and decode steps at 8 x 12 caches of 131072 tokens whose demand
has the heavy tail a prefill leaves.

Operator: "DilutionAttention v0.1.0 · results", section "The operator" (the
causal softmax, the exclusive column cumsum of the bids, share, renormalised
value product) and its cached-decoding paragraph (one running demand total per
key and head).  tau = sqrt(0.1 ln s + 1): "YaRN › Attention Temperature
Scaling", its temperature formula and table.
"""
import numpy as np
import pytest
import torch

import oracle.dilution as od
from long_context_attention_gb300 import binding as b
from long_context_attention_gb300 import inputs
from tests._parity import BF16_OUT_ABS, LOG2E, host64, oracle_forward

pytestmark = pytest.mark.gpu
DEV = "cuda"

# demand tolerances of the bf16 path (see tests/_parity.py)
DEM_REL, DEM_ABS = 1e-3, 1e-4


def _fwd_all(q, k, v, tau, eps):
    B, H, T, d = q.shape
    out = torch.empty_like(q)
    lse2, rs, dem = (torch.empty(B, H, T, device=DEV) for _ in range(3))
    ws = torch.empty(b.dilution_attn_fwd_workspace_size(B, H, T, d, b.DA_BF16), dtype=torch.uint8, device=DEV)
    b.dilution_attn_fwd(q, k, v, out, lse2, rs, dem, tau=tau, eps=eps, workspace=ws)
    assert b.dilution_attn_get_error(ws) == b.DA_OK
    torch.cuda.synchronize()
    return out, lse2, rs, dem


def _late_rows_exact(qh, kh, rows, c):
    """lse (natural log) of the given query rows and the bids p [len(rows), T]
    over every key, straight from the definition (causal softmax)."""
    T = kh.shape[0]
    s = c * (qh[rows] @ kh.T)
    mask = np.arange(T)[None, :] <= rows[:, None]
    s = np.where(mask, s, -np.inf)
    m = s.max(1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(1)
    return m[:, 0] + np.log(l), e / l[:, None]


def test_prefill_config_t131072():
    """1 x 12 x 131072, tau = yarn_tau(8), 16 planted pairs per head, in the
    benchmark's launch configuration.  Checked against the oracle: out, lse2
    and the row sums of the first 4096 rows of two heads; lse2 of the last 256
    rows and of 256 random rows; the demand of the last 256 keys (only the
    last 256 queries bid on them, so it follows exactly from those rows); the
    unit-demand invariant on every head."""
    w = inputs.WORKLOADS["prefill_bf16_t131072"]
    tau = od.yarn_tau(w.tau_scale)
    q, k, v = inputs.make_workload(w, device=DEV)
    T = w.T
    out, lse2, rs, dem = _fwd_all(q, k, v, tau, w.eps)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse2).all()
    # Unit demand per query: each head's demand totals T.  The totals are fp32
    # running sums over up to T bids, and a bid below half an ulp of its key's
    # running total is absorbed, so the sum falls short by a margin that grows
    # with T: a CPU replay of exact bids added in fp32 in query order loses
    # 1.3e-5 T on this workload (at most 3e-4 of any key's total, inside the
    # per-key demand tolerance of 1e-3).  The bound is ten times below that
    # per-key tolerance.
    err = (dem.double().sum(-1) - T).abs().max().item()
    assert err <= 1e-4 * T, err
    heads = [(0, 0), (0, 11)]
    n = 4096
    ref = oracle_forward(q, k, v, tau, w.eps, rows=n, heads=heads)
    c = od.logit_scale(w.d, tau)
    rng = np.random.default_rng(1234)
    for (bb, hh) in heads:
        r = ref[(bb, hh)]
        o, l2, rsum = (host64(x[bb, hh][:n]) for x in (out, lse2, rs))
        assert np.abs(o - r["out"]).max() <= BF16_OUT_ABS
        assert np.abs(l2 - r["lse"] * LOG2E).max() <= 2e-3
        assert np.abs(rsum / r["rowsum"] - 1).max() <= 2e-2
        qh, kh = host64(q[bb, hh]), host64(k[bb, hh])
        tail = np.arange(T - 256, T)
        lse_t, p_t = _late_rows_exact(qh, kh, tail, c)
        assert np.abs(host64(lse2[bb, hh])[tail] - lse_t * LOG2E).max() <= 2e-3
        d_tail = p_t[:, T - 256:].sum(0)
        g_tail = host64(dem[bb, hh])[T - 256:]
        assert np.all(np.abs(g_tail - d_tail) <= DEM_REL * np.maximum(d_tail, 1) + DEM_ABS)
        mid = np.sort(rng.choice(np.arange(n, T - 256), 256, replace=False))
        lse_m, _ = _late_rows_exact(qh, kh, mid, c)
        assert np.abs(host64(lse2[bb, hh])[mid] - lse_m * LOG2E).max() <= 2e-3


def _prefill_cache(q, k, v, T_cap, tau, eps):
    """GPU prefill of q, k, v [B, H, n, d]: caches with room for T_cap tokens
    and the prefill's demand (the decode cache)."""
    B, H, n, d = q.shape
    kc = torch.zeros(B, H, T_cap, d, dtype=q.dtype, device=DEV)
    vc = torch.zeros_like(kc)
    kc[:, :, :n] = k
    vc[:, :, :n] = v
    dem = torch.zeros(B, H, T_cap, device=DEV)
    d_out = torch.empty(B, H, n, device=DEV)
    b.dilution_attn_fwd(q, k, v, None, None, None, d_out, tau=tau, eps=eps)
    dem[:, :, :n] = d_out
    return kc, vc, dem


def test_decode_chain_from_prefill():
    """A prefill of 8192 tokens at the long-context multiplier, then 64 cached
    decode steps on the GPU; the oracle runs its own prefill and its own decode
    chain on the same tokens.  Every step's output and the final demand of
    every key are compared on four heads."""
    B, H, N, d, steps = 2, 12, 8192, 64, 64
    tau, eps = od.yarn_tau(8.0), 1e-6
    q, k, v = inputs.make_qkv(B, H, N + steps, d, q_std=1.5, pairs=16, seed=3, dtype="bf16", device=DEV)
    kc, vc, dem = _prefill_cache(q[:, :, :N].contiguous(), k[:, :, :N].contiguous(), v[:, :, :N].contiguous(),
                                 N + steps, tau, eps)
    ws = torch.empty(b.dilution_attn_decode_workspace_size(B, H, N + steps, d), dtype=torch.uint8, device=DEV)
    outs = []
    for t in range(steps):
        n = N + t
        o = b.dilution_attn_decode_step(q[:, :, n].contiguous(), k[:, :, n].contiguous(), v[:, :, n].contiguous(),
                                        kc, vc, dem, n, tau=tau, eps=eps, workspace=ws)
        outs.append(o.clone())
    assert b.dilution_attn_get_error(ws) == b.DA_OK
    torch.cuda.synchronize()
    got = torch.stack(outs, 2)   # [B, H, steps, d]
    for (bb, hh) in [(0, 0), (0, 5), (1, 7), (1, 11)]:
        qh, kh, vh = (host64(x[bb, hh]) for x in (q, k, v))
        D = od.dilution_forward_rowblocked_head(qh[:N], kh[:N], vh[:N], tau, eps)["demand"]
        ref = []
        for t in range(steps):
            n = N + t
            o, D, _, _ = od.dilution_decode_step_head(qh[n], kh[n], vh[n], kh[:n], vh[:n], D, n, tau, eps)
            ref.append(o)
        err = np.abs(host64(got[bb, hh]) - np.stack(ref)).max()
        assert err <= BF16_OUT_ABS, err
        gd = host64(dem[bb, hh])
        assert np.all(np.abs(gd - D) <= DEM_REL * np.maximum(D, 1) + DEM_ABS)
        # the appended tokens landed in the cache
        assert torch.equal(kc[bb, hh, N:N + steps], k[bb, hh, N:N + steps])


def test_decode_ctx131072_heavy_tailed_demand():
    """8 x 12 caches of 131072 tokens (the decode workload's size) whose
    demand has the shape a prefill leaves: the column totals of uniform bids,
    sum_{i >= k} 1 / (i + 1) (from ~12.3 on the first key down to 1/N on the
    last), plus 16 keys per head that won a large bid (+0.5 .. 1).  Eight
    consecutive steps; each step's output and the final demand compared with
    the oracle's decode chain on two heads."""
    w = inputs.WORKLOADS["decode_bf16_ctx131072"]
    B, H, N, d = w.B, w.H, w.T, w.d
    steps = 8
    T_cap = N + steps
    tau = od.yarn_tau(w.tau_scale)
    kc = inputs.make_like((B, H, T_cap, d), seed=171, dtype="bf16", device=DEV)
    vc = inputs.make_like((B, H, T_cap, d), seed=172, dtype="bf16", device=DEV)
    # input recipe: harmonic tail + spikes (float64 on the host, stored fp32)
    tail = np.concatenate([np.cumsum((1.0 / np.arange(1, N + 1))[::-1])[::-1], np.zeros(steps)])
    rng = np.random.default_rng(173)
    dem0 = np.broadcast_to(tail, (B, H, T_cap)).copy()
    for bb in range(B):
        for hh in range(H):
            dem0[bb, hh, rng.choice(N, 16, replace=False)] += rng.uniform(0.5, 1.0, 16)
    dem = torch.from_numpy(dem0.astype(np.float32)).to(DEV)
    heads = [(0, 3), (7, 11)]
    before = {hd: (host64(kc[hd]), host64(vc[hd]), host64(dem[hd])) for hd in heads}
    toks = [tuple(inputs.make_like((B, H, d), std=s, seed=180 + 3 * t + i, dtype="bf16", device=DEV)
                  for i, s in enumerate((1.5, 1.0, 1.0))) for t in range(steps)]
    ws = torch.empty(b.dilution_attn_decode_workspace_size(B, H, T_cap, d), dtype=torch.uint8, device=DEV)
    outs = [b.dilution_attn_decode_step(qn, kn, vn, kc, vc, dem, N + t, tau=tau, eps=w.eps, workspace=ws).clone()
            for t, (qn, kn, vn) in enumerate(toks)]
    assert b.dilution_attn_get_error(ws) == b.DA_OK
    torch.cuda.synchronize()
    for hd in heads:
        kk, vv, D = before[hd]
        D = D[:N]
        for t, (qn, kn, vn) in enumerate(toks):
            o, D, K, V = od.dilution_decode_step_head(host64(qn[hd]), host64(kn[hd]), host64(vn[hd]), kk, vv, D,
                                                      N + t, tau, w.eps)
            kk, vv = K, V
            err = np.abs(host64(outs[t][hd]) - o).max()
            assert err <= BF16_OUT_ABS, (t, err)
        gd = host64(dem[hd])[:N + steps]
        assert np.all(np.abs(gd - D) <= 1e-5 * np.maximum(D, 1.0) + 1e-6)


def test_prefill_t131072_per_head_tau():
    """1 x 4 x 131072 with a different multiplier per head (the YaRN value for
    s = 2, 4, 8, 16): at this length the row statistics take heads in groups
    of 3 and the sweep one head at a time, so each CTA's head comes from the
    grouped launch order and its multiplier from the per-head array.  Checked
    against the oracle with each head's own multiplier: out, lse2 and row sums
    of the first 2048 rows, lse2 of the last 128 rows, the last 128 keys'
    demand, and the unit-demand invariant."""
    B, H, T, d = 1, 4, 131072, 64
    taus = [od.yarn_tau(s) for s in (2.0, 4.0, 8.0, 16.0)]
    q, k, v = inputs.make_qkv(B, H, T, d, q_std=1.5, pairs=16, seed=701, dtype="bf16", device=DEV)
    out = torch.empty_like(q)
    lse2, rs, dem = (torch.empty(B, H, T, device=DEV) for _ in range(3))
    ws = torch.empty(b.dilution_attn_fwd_workspace_size(B, H, T, d, b.DA_BF16), dtype=torch.uint8, device=DEV)
    tau_bh = torch.tensor(taus, dtype=torch.float32, device=DEV)
    b.dilution_attn_fwd_ex(q, k, v, out, lse2, rs, dem, tau_bh=tau_bh, eps=1e-6, workspace=ws)
    assert b.dilution_attn_get_error(ws) == b.DA_OK
    torch.cuda.synchronize()
    err = (dem.double().sum(-1) - T).abs().max().item()
    assert err <= 1e-4 * T, err            # fp32 demand totals at this length: see test_prefill_config_t131072
    n = 2048
    for hh in range(H):
        tau = float(np.float32(taus[hh]))   # the multiplier as the kernels read it
        qh, kh, vh = (host64(x[0, hh]) for x in (q, k, v))
        r = od.dilution_forward_rowblocked_head(qh, kh, vh, tau, 1e-6, rows=n)
        assert np.abs(host64(out[0, hh][:n]) - r["out"]).max() <= BF16_OUT_ABS
        assert np.abs(host64(lse2[0, hh][:n]) - r["lse"] * LOG2E).max() <= 2e-3
        assert np.abs(host64(rs[0, hh][:n]) / r["rowsum"] - 1).max() <= 2e-2
        c = od.logit_scale(d, tau)
        tail = np.arange(T - 128, T)
        lse_t, p_t = _late_rows_exact(qh, kh, tail, c)
        assert np.abs(host64(lse2[0, hh])[tail] - lse_t * LOG2E).max() <= 2e-3
        d_tail = p_t[:, T - 128:].sum(0)
        g_tail = host64(dem[0, hh])[T - 128:]
        assert np.all(np.abs(g_tail - d_tail) <= DEM_REL * np.maximum(d_tail, 1) + DEM_ABS)
