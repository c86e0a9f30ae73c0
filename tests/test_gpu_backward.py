"""GPU parity of dilution_attn_bwd (through the C ABI): against the float64
oracle's backward on the same inputs, and against central finite differences
of the GPU's own fp32 forward.

Tolerances: fp32 inputs, max |error| <= 2e-4 x max |oracle gradient|;
bf16 inputs (gradients rounded to bf16 at the end), <= 1.5e-2 x max |oracle|.
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


def gpu_grads(q, k, v, g, tau, eps):
    B, H, T, _ = q.shape
    lse2 = torch.empty(B, H, T, device=DEV)
    b.dilution_attn_fwd(q, k, v, None, lse2, tau=tau, eps=eps)
    dq, dk, dv = b.dilution_attn_bwd(q, k, v, g, lse2, tau=tau, eps=eps)
    torch.cuda.synchronize()
    return [host64(x) for x in (dq, dk, dv)]


def oracle_grads(q, k, v, g, tau, eps):
    return od.dilution_backward(host64(q), host64(k), host64(v), host64(g), tau, eps)


def rel_to_max(got, ref):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


@pytest.mark.parametrize("T", [1, 2, 17, 128, 200, 300])
def test_bwd_f32_matches_oracle(T):
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(2, 2, T, 64, q_std=1.5, pairs=min(4, max(T - 1, 0)), seed=T))
    g = inputs.make_like((2, 2, T, 64), seed=1000 + T, device=DEV)
    for got, ref in zip(gpu_grads(q, k, v, g, 1.1, 1e-6), oracle_grads(q, k, v, g, 1.1, 1e-6)):
        assert rel_to_max(got, ref) <= 2e-4


@pytest.mark.parametrize("T", [5, 129, 256])
def test_bwd_bf16_matches_oracle(T):
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(1, 2, T, 64, q_std=1.5, pairs=4, seed=T, dtype="bf16"))
    g = inputs.make_like((1, 2, T, 64), seed=2000 + T, dtype="bf16", device=DEV)
    for got, ref in zip(gpu_grads(q, k, v, g, 1.0, 1e-6), oracle_grads(q, k, v, g, 1.0, 1e-6)):
        assert rel_to_max(got, ref) <= 1.5e-2


def test_bwd_training_recipe_slice_t512():
    """The training workload's recipe (q, k, v, dout all N(0,1)) on a T = 512 slice."""
    w = inputs.WORKLOADS["train_bf16_t16384"]
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(1, 2, 512, 64, q_std=w.q_std, pairs=0, seed=w.seed, dtype="bf16"))
    g = inputs.make_like((1, 2, 512, 64), seed=w.seed + 1, dtype="bf16", device=DEV)
    for got, ref in zip(gpu_grads(q, k, v, g, 1.0, w.eps), oracle_grads(q, k, v, g, 1.0, w.eps)):
        assert rel_to_max(got, ref) <= 1.5e-2


def test_bwd_finite_differences_of_gpu_forward():
    """T = 16, fp32: central differences of L = sum(dout * out) through the
    GPU forward, at 24 random coordinates of q, k and v."""
    T, d = 16, 64
    q, k, v = (x.to(DEV).double().float() for x in inputs.make_qkv(1, 1, T, d, seed=5))
    g = inputs.make_like((1, 1, T, d), seed=6, device=DEV)
    tau, eps, h = 1.3, 1e-3, 2e-3
    grads = gpu_grads(q, k, v, g, tau, eps)

    def loss(qq, kk, vv):
        out = b.dilution_attn_fwd(qq.contiguous(), kk.contiguous(), vv.contiguous(), tau=tau, eps=eps)
        return float((out.double() * g.double()).sum())

    rng = np.random.default_rng(7)
    for which, X in enumerate((q, k, v)):
        for _ in range(8):
            i, t = int(rng.integers(0, T)), int(rng.integers(0, d))
            Xp, Xm = X.clone(), X.clone()
            Xp[0, 0, i, t] += h
            Xm[0, 0, i, t] -= h
            args_p, args_m = [q, k, v], [q, k, v]
            args_p[which], args_m[which] = Xp, Xm
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            an = grads[which][0, 0, i, t]
            assert abs(fd - an) <= 2e-3 * max(1.0, abs(an)), (which, i, t, fd, an)


def test_bwd_argument_errors():
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(1, 1, 64, 64, dtype="bf16", seed=3))
    lse2 = torch.empty(1, 1, 64, device=DEV)
    with pytest.raises(b.DilutionAttnError) as ei:
        b.dilution_attn_bwd(q, k, v, q, lse2, eps=0.0)
    assert ei.value.status == b.DA_ERR_INVALID


@pytest.mark.parametrize("d,T", [(64, 300), (64, 1000), (128, 300)])
def test_bwd_with_forward_state(d, T):
    """DA_FLAG_KEEP_FOR_BACKWARD: the forward leaves its demand checkpoints and
    accumulators in a backward-sized workspace and the backward skips its own
    forward pass; same gradients as the stand-alone backward."""
    keep = b.DA_FLAG_KEEP_FOR_BACKWARD
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(1, 2, T, d, q_std=1.5, pairs=4, seed=T + d, dtype="bf16"))
    g = inputs.make_like((1, 2, T, d), seed=3000 + T, dtype="bf16", device=DEV)
    lse2 = torch.empty(1, 2, T, device=DEV)
    ws = torch.empty(b.dilution_attn_bwd_workspace_size(1, 2, T, d, b.DA_BF16), dtype=torch.uint8, device=DEV)
    out = b.dilution_attn_fwd_ex(q, k, v, None, lse2, flags=keep, workspace=ws)
    kept = b.dilution_attn_bwd_ex(q, k, v, g, lse2, flags=keep, workspace=ws)
    assert b.dilution_attn_get_error(ws) == b.DA_OK
    alone = b.dilution_attn_bwd(q, k, v, g, lse2)
    plain_out = b.dilution_attn_fwd(q, k, v)
    torch.cuda.synchronize()
    # the flag changes nothing the forward returns (up to the order of the
    # accumulator reductions across key spans, which is not fixed)
    assert (out.float() - plain_out.float()).abs().max().item() <= 1e-2
    ref = od.dilution_backward(host64(q), host64(k), host64(v), host64(g), 1.0, 1e-6)
    for gk, ga, rr in zip(kept, alone, ref):
        assert rel_to_max(host64(gk), rr) <= 1.5e-2
        assert rel_to_max(host64(gk), host64(ga)) <= 1e-2
