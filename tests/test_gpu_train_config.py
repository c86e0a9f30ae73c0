"""GPU parity of the backward at the training configuration, 4 x 12 x 16384 x
64 bf16 (q, k, v and dout drawn as the benchmark draws them), and at the same
shape with head dimension 128 (the benchmark's d = 128 training line), in the
benchmark's launch configuration: the forward keeps its demand checkpoints in
the backward's workspace (DA_FLAG_KEEP_FOR_BACKWARD) and the backward starts
from them.

* Two full heads, the first and the last (launched in the first and the last
  head group), against the row-blocked float64 oracle backward: dQ, dK and dV
  element by element, with the bf16 backward bound the other backward tests
  use (1.5 % of the largest |reference| of each tensor).
* Every head through identities of the exact gradients that hold at any size:
    sum_k dV_k = sum_i dout_i   every row of A sums to 1;
    sum_k dK_k = 0              each row of ds sums to 0 (the bids of a row sum
                                to 1), i.e. a constant added to every key
                                leaves the softmax and the loss unchanged;
    <Q, dQ> = <K, dK>           both equal c sum_jk ds_jk (q_j . k_k).
  Their tolerances come from the bf16 arithmetic: each output element carries
  a rounding error of at most 2^-9 of itself, independent across elements, so
  a sum over the 16384 keys of one column is off by about 2^-9 of the
  column's 2-norm; the bounds below allow 2^-5 of the norms (16 x) for dV and
  the inner products.  dK = c (sum u q - sum p rho q) comes from two bf16
  products, each rounded on its own: up to ~0.4 % of max |dK| per element,
  and max |dK| reaches ~16 x its root mean square here, so an element's
  error is up to ~6 % of the rms and a sum of 16384 of them, with independent
  signs, ~3.5 % of the column's 2-norm; the bound is 2^-3.

Operator and gradients: "DilutionAttention v0.1.0 · results", section "The
operator" (the forward), and its line that the operator has exact gradients
for training; the chain rule is the oracle's (dilution_backward_head).
"""
import numpy as np
import pytest
import torch

import oracle.dilution as od
from long_context_attention_gb300 import binding as b
from long_context_attention_gb300 import inputs
from tests._parity import host64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_training_config_t16384(d):
    w = inputs.WORKLOADS["train_bf16_t16384"]
    B, H, T = w.B, w.H, w.T
    q, k, v = inputs.make_qkv(B, H, T, d, q_std=w.q_std, pairs=w.pairs, seed=w.seed, dtype=w.dtype, device=DEV)
    g = inputs.make_like((B, H, T, d), seed=w.seed + 1, dtype=w.dtype, device=DEV)
    keep = b.DA_FLAG_KEEP_FOR_BACKWARD
    ws = torch.empty(b.dilution_attn_bwd_workspace_size(B, H, T, d, b.DA_BF16), dtype=torch.uint8, device=DEV)
    out = torch.empty_like(q)
    lse2 = torch.empty(B, H, T, device=DEV)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    b.dilution_attn_fwd_ex(q, k, v, out, lse2, flags=keep, workspace=ws)
    b.dilution_attn_bwd_ex(q, k, v, g, lse2, dq, dk, dv, flags=keep, workspace=ws)
    assert b.dilution_attn_get_error(ws) == b.DA_OK
    torch.cuda.synchronize()
    for x in (dq, dk, dv):
        assert torch.isfinite(x.float()).all()

    # identities, every head (float64 sums of the bf16 outputs)
    Q, K, G = (x.double() for x in (q, k, g))
    dQ, dK, dV = (x.double() for x in (dq, dk, dv))
    tol_v = 2.0 ** -5 * (dV.norm(dim=2) + G.norm(dim=2))
    assert ((dV.sum(2) - G.sum(2)).abs() <= tol_v).all()
    assert (dK.sum(2).abs() <= 2.0 ** -3 * dK.norm(dim=2)).all()
    qdq = (Q * dQ).sum(-1)
    kdk = (K * dK).sum(-1)
    scale = qdq.abs().sum(-1) + kdk.abs().sum(-1)
    assert ((qdq.sum(-1) - kdk.sum(-1)).abs() <= 2.0 ** -5 * scale).all()

    # two full heads against the oracle (about 10 s of CPU each at d = 64)
    for bb, hh in [(0, 0), (B - 1, H - 1)]:
        ref = od.dilution_backward_rowblocked_head(host64(q[bb, hh]), host64(k[bb, hh]), host64(v[bb, hh]),
                                                   host64(g[bb, hh]), 1.0, w.eps)
        for got, r in zip((dq, dk, dv), ref):
            err = np.abs(host64(got[bb, hh]) - r).max()
            assert err <= 1.5e-2 * max(np.abs(r).max(), 1e-3), (bb, hh, err)
