"""GPU parity of dilution_attn_fwd (through the C ABI) against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle.dilution as od
from long_context_attention_gb300 import binding as b
from long_context_attention_gb300 import inputs
from tests._parity import BF16_OUT_ABS, F32_OUT_REL, LOG2E, host64, oracle_forward, row_rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_fwd(q, k, v, tau=1.0, eps=1e-6):
    B, H, T, _ = q.shape
    out = torch.empty_like(q)
    lse2 = torch.empty(B, H, T, device=DEV)
    rs = torch.empty(B, H, T, device=DEV)
    dem = torch.empty(B, H, T, device=DEV)
    ws = torch.empty(b.dilution_attn_fwd_workspace_size(B, H, T, q.shape[-1], b._dtype_code(q)), dtype=torch.uint8,
                     device=DEV)
    b.dilution_attn_fwd(q, k, v, out, lse2, rs, dem, tau=tau, eps=eps, workspace=ws)
    assert b.dilution_attn_get_error(ws) == b.DA_OK
    torch.cuda.synchronize()
    return out, lse2, rs, dem


def check_head(got, ref, dtype, rows=None, dem_rel=1e-6):
    out, lse2, rs, dem = got
    n = rows if rows is not None else out.shape[0]
    o_ref = ref["out"][:n]
    if dtype == "f32":
        assert row_rel_err(out[:n], o_ref) <= F32_OUT_REL
        assert np.abs(lse2[:n] - ref["lse"][:n] * LOG2E).max() <= 1e-5 * max(1.0, np.abs(lse2[:n]).max())
        assert np.abs(rs[:n] / ref["rowsum"][:n] - 1).max() <= 1e-5
        if rows is None:
            assert np.all(np.abs(dem - ref["demand"]) <= dem_rel * np.maximum(ref["demand"], 1.0))
    else:
        assert np.abs(out[:n] - o_ref).max() <= BF16_OUT_ABS
        assert np.abs(lse2[:n] - ref["lse"][:n] * LOG2E).max() <= 2e-3
        assert np.abs(rs[:n] / ref["rowsum"][:n] - 1).max() <= 2e-2
        if rows is None:
            assert np.all(np.abs(dem - ref["demand"]) <= 1e-3 * np.maximum(ref["demand"], 1.0) + 1e-4)


def compare(q, k, v, tau=1.0, eps=1e-6, heads=None, rows=None):
    dtype = "f32" if q.dtype == torch.float32 else "bf16"
    got = [host64(x) for x in run_fwd(q, k, v, tau, eps)]
    ref = oracle_forward(q, k, v, tau, eps, rows=rows, heads=heads)
    for (bb, hh), r in ref.items():
        check_head([g[bb, hh] for g in got], r, dtype, rows)
    return got, ref


# ----------------------------------------------------------------------------- fp32
def test_f32_config_t256():
    w = inputs.WORKLOADS["fwd_f32_t256"]
    q, k, v = (x.to(DEV) for x in inputs.make_workload(w))
    got, ref = compare(q, k, v, 1.0, w.eps)
    # the unit-demand invariant on the GPU's own demand output
    assert abs(got[3][0, 0].sum() - 256) < 1e-3


@pytest.mark.parametrize("T", [1, 2, 3, 7, 8, 127, 129, 255, 300])
def test_f32_ragged(T):
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(2, 3, T, 64, q_std=1.5, pairs=min(4, T - 1) if T > 1 else 0,
                                                   seed=T))
    compare(q, k, v, tau=1.3, eps=1e-6)


def test_f32_single_token_is_v():
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(3, 2, 1, 64, seed=11))
    out = run_fwd(q, k, v)[0]
    assert torch.allclose(out, v, rtol=1e-6, atol=1e-6)


def test_f32_tau_zero_uniform_bids():
    # tau = 0: every visible bid is 1/(i+1); committed = H_i - H_k (harmonic numbers)
    T = 100
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(1, 1, T, 64, seed=12))
    out, lse2, rs, dem = (host64(x)[0, 0] for x in run_fwd(q, k, v, tau=0.0, eps=1e-6))
    Hn = np.concatenate([[0.0], np.cumsum(1.0 / np.arange(1, T + 2))])
    share = np.array([[1.0 / ((i + 1) * (Hn[i + 1] - Hn[kk] + 1e-6)) if kk <= i else 0.0 for kk in range(T)]
                      for i in range(T)])
    ref = (share / share.sum(1, keepdims=True)) @ host64(v)[0, 0]
    assert row_rel_err(out, ref) <= F32_OUT_REL
    assert np.abs(lse2 - np.log2(np.arange(1, T + 1))).max() < 1e-5


# ----------------------------------------------------------------------------- bf16
@pytest.mark.parametrize("T", [1, 2, 5, 127, 128, 129, 255, 256, 257, 300, 640])
def test_bf16_ragged(T):
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(1, 2, T, 64, q_std=1.5, pairs=min(8, max(T - 1, 0)), seed=T,
                                                   dtype="bf16"))
    compare(q, k, v, tau=1.0, eps=1e-6)


def test_bf16_tau_and_eps():
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(2, 2, 700, 64, q_std=1.5, pairs=8, seed=21, dtype="bf16"))
    compare(q, k, v, tau=od.yarn_tau(8), eps=1e-6)
    compare(q, k, v, tau=2.5, eps=1e-3)


def test_bf16_sharp_logits_rescale():
    # tau = 6 multiplies the planted logits (~26 in log2 units at tau = 1) to
    # ~150: a row whose planted key lies beyond its first 32 keys then scores
    # far above that chunk's maximum, overflows the unchecked running sum and
    # is recomputed by the fix-up pass.
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(1, 2, 700, 64, q_std=1.5, pairs=8, seed=41, dtype="bf16"))
    compare(q, k, v, tau=6.0, eps=1e-6)


def test_bf16_rows_of_A_sum_to_one():
    q, k, _ = inputs.make_qkv(2, 3, 1000, 64, q_std=1.5, pairs=16, seed=22, dtype="bf16")
    q, k = q.to(DEV), k.to(DEV)
    ones = torch.ones_like(q)
    out = run_fwd(q, k, ones)[0].float()
    assert (out - 1).abs().max().item() <= 1e-5


def test_bf16_config_t4096():
    w = inputs.WORKLOADS["fwd_bf16_t4096"]
    q, k, v = (x.to(DEV) for x in inputs.make_workload(w))
    got, _ = compare(q, k, v, 1.0, w.eps, heads=[(0, 0), (0, 7), (1, 3), (1, 11)])
    dem = got[3]
    assert np.abs(dem.sum(axis=-1) - w.T).max() < 0.05 * 1e-3 * w.T + 0.1


def test_bf16_planted_pairs_retrieved():
    # a planted key k_j = q_i carries a logit of about |q|^2/8 ~ 18: query i's
    # output is close to v_j.
    w = inputs.WORKLOADS["fwd_bf16_t4096"]
    q, k, v = (x.to(DEV) for x in inputs.make_workload(w, B=1))
    out = run_fwd(q, k, v)[0].float()
    pp = inputs.planted_pairs(1, w.H, w.T, w.pairs, w.seed)
    hits = 0
    for (_, h, i, j) in pp:
        hits += int(torch.nn.functional.cosine_similarity(out[0, h, i], v[0, h, j].float(), dim=0) > 0.5)
    assert hits >= 0.9 * len(pp)


def test_bf16_config_t16384_full_heads():
    """The benchmark's workload at full size (4 x 12 x 16384), in the launch
    configuration the benchmark times: two whole heads, one from the first
    sweep head group and the last head of the last group, against the oracle
    row by row (out, lse2, row sums) and key by key (demand); the unit-demand
    invariant on every head."""
    w = inputs.WORKLOADS["fwd_bf16_t16384"]
    q, k, v = (x.to(DEV) for x in inputs.make_workload(w, device=DEV))
    T = w.T
    out, lse2, rs, dem = run_fwd(q, k, v, 1.0, w.eps)
    assert torch.isfinite(out.float()).all()
    # invariant: every query adds exactly one unit of demand (the bids of a
    # row sum to 1), so each head's demand totals T
    err = (dem.double().sum(-1) - T).abs().max().item()
    assert err <= 1e-5 * T, err
    heads = [(0, 0), (3, 11)]
    ref = oracle_forward(q, k, v, 1.0, w.eps, heads=heads)
    for (bb, hh), r in ref.items():
        check_head([host64(x[bb, hh]) for x in (out, lse2, rs, dem)], r, "bf16")


def test_error_status_clean_and_invalid_args():
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(1, 1, 64, 64, dtype="bf16", seed=3))
    with pytest.raises(b.DilutionAttnError) as ei:
        b.dilution_attn_fwd(q, k, v, eps=0.0)
    assert ei.value.status == b.DA_ERR_INVALID
    with pytest.raises(b.DilutionAttnError) as ei:
        b.dilution_attn_fwd(q, k, v, workspace=torch.empty(16, dtype=torch.uint8, device=DEV))
    assert ei.value.status == b.DA_ERR_WORKSPACE
    ws = torch.empty(b.dilution_attn_fwd_workspace_size(1, 1, 64, 64, 1), dtype=torch.uint8, device=DEV)
    b.dilution_attn_fwd(q, k, v, workspace=ws)
    assert b.dilution_attn_get_error(ws) == b.DA_OK


def test_repeatable_and_stream_ordered():
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(1, 4, 1500, 64, q_std=1.5, pairs=8, seed=31, dtype="bf16"))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o1 = b.dilution_attn_fwd(q, k, v, stream=s)
        o2 = b.dilution_attn_fwd(q, k, v, stream=s)
    s.synchronize()
    # fp32 reductions in L2 may add partials in any order: equal to rounding
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2


def test_bf16_tau_zero_uniform_bids():
    # tau = 0: every visible bid is 1/(i+1), whatever q and k
    T = 300
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(1, 2, T, 64, q_std=1.5, seed=13, dtype="bf16"))
    got = [host64(x) for x in run_fwd(q, k, v, tau=0.0, eps=1e-6)]
    ref = oracle_forward(q, k, v, 0.0, 1e-6)
    for (bb, hh), r in ref.items():
        check_head([x[bb, hh] for x in got], r, "bf16")
    assert np.abs(got[1][0, 0] - np.log2(np.arange(1, T + 1))).max() < 2e-3


def _status_words(ws):
    torch.cuda.synchronize()
    return ws[:32].view(torch.int32).cpu().tolist()


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_overflowing_rows_recomputed(d):
    """The row-statistics pass sums each row against the maximum of its first
    32 keys without further checks; a row whose later logit lies far above that
    (here ~185 log2 units at d = 64) overflows the running sum, is marked, and
    is recomputed exactly by the fix-up pass (status word 4 counts the marked
    rows).  Marked and ordinary rows both match the oracle."""
    B, H, T = 1, 2, 300
    g = torch.Generator().manual_seed(70 + d)
    q = torch.randn(B, H, T, d, generator=g) * 1.5
    k = torch.randn(B, H, T, d, generator=g)
    v = torch.randn(B, H, T, d, generator=g)
    big = [50, 100, 200, 299]
    k[:, :, 40] = 4.0          # key 40 sits in the second 32-key chunk of every row
    for i in big:
        q[:, :, i] = 4.0       # q_i . k_40 = 16 d
    q, k, v = (x.to(torch.bfloat16).to(DEV) for x in (q, k, v))
    out = torch.empty_like(q)
    lse2, rs, dem = (torch.empty(B, H, T, device=DEV) for _ in range(3))
    ws = torch.empty(b.dilution_attn_fwd_workspace_size(B, H, T, d, b._dtype_code(q)), dtype=torch.uint8,
                     device=DEV)
    b.dilution_attn_fwd(q, k, v, out, lse2, rs, dem, workspace=ws)
    words = _status_words(ws)
    assert words[0] == b.DA_OK
    assert words[4] == B * H * len(big)
    got = [host64(x) for x in (out, lse2, rs, dem)]
    ref = oracle_forward(q, k, v, 1.0, 1e-6)
    for (bb, hh), r in ref.items():
        check_head([x[bb, hh] for x in got], r, "bf16")
    assert np.all(got[1][0, :, big] > 150.0)


def test_bf16_ordinary_rows_not_marked():
    """Planted retrieval pairs at tau = 1 stay well inside the unchecked range:
    no row is marked for recomputation."""
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(1, 4, 1500, 64, q_std=1.5, pairs=16, seed=33, dtype="bf16"))
    ws = torch.empty(b.dilution_attn_fwd_workspace_size(1, 4, 1500, 64, 1), dtype=torch.uint8, device=DEV)
    b.dilution_attn_fwd(q, k, v, workspace=ws)
    words = _status_words(ws)
    assert words[0] == b.DA_OK and words[4] == 0
