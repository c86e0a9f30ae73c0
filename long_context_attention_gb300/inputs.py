"""Seeded synthetic inputs for dilution attention workloads.

Shared by the tests, the benchmark and the smoke check; holds none of the
operator's arithmetic.  Inputs stand in for the text workloads of the
"DilutionAttention v0.1.0 · results" page (FineWeb-Edu training, PG-19 and
keyword-retrieval haystacks) with the head layout of its 24-layer decoders:
d_model = 768 split into H = 12 heads of d = 64.

Recipe (all draws from one ``torch.Generator`` seeded with ``seed`` on the
device where the tensors are made, in this order):
  q ~ N(0, q_std^2), k ~ N(0, 1), v ~ N(0, 1), each [B, H, T, d], float32;
  then ``pairs`` planted retrieval targets per (b, h): a query index i is drawn
  uniformly from [1, T) and a key index j uniformly from [0, i), rejecting a j
  already used in that head, and k[b, h, j] is overwritten with q[b, h, i].
  The planted indices come from ``numpy.random.default_rng(seed)``.
  bf16 workloads round once, to nearest even, after planting; both the CUDA
  path and the oracle see the rounded values.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    d: int
    dtype: str            # "f32" or "bf16"
    q_std: float
    pairs: int
    seed: int
    tau_scale: float = 1.0   # YaRN extension factor s; tau = sqrt(0.1 ln s + 1) (1 -> tau = 1)
    eps: float = 1e-6
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    # fp32 correctness anchor: 1 x 1 x 256 x 64, N(0,1) inputs, seed 0.
    "fwd_f32_t256": Workload("fwd_f32_t256", 1, 1, 256, 64, "f32", 1.0, 0, 0),
    # bf16 in / fp32 accumulate: 2 x 12 x 4096 x 64, 32 planted pairs per head.
    "fwd_bf16_t4096": Workload("fwd_bf16_t4096", 2, 12, 4096, 64, "bf16", 1.5, 32, 1),
    # training context: 4 x 12 x 16384 x 64, 128 planted pairs per head (headline shape).
    "fwd_bf16_t16384": Workload("fwd_bf16_t16384", 4, 12, 16384, 64, "bf16", 1.5, 128, 2),
    # long-context prefill at 8x the training context with the YaRN multiplier for s = 8.
    "prefill_bf16_t131072": Workload("prefill_bf16_t131072", 1, 12, 131072, 64, "bf16", 1.5, 16, 3,
                                     tau_scale=8.0),
    # cached decode: 8 independent 128K caches, 256 appended tokens each.
    "decode_bf16_ctx131072": Workload("decode_bf16_ctx131072", 8, 12, 131072, 64, "bf16", 1.5, 16, 3,
                                      tau_scale=8.0, extra={"steps": 256}),
    # training step shape: all N(0,1), upstream gradient N(0,1).
    "train_bf16_t16384": Workload("train_bf16_t16384", 4, 12, 16384, 64, "bf16", 1.0, 0, 4),
    # the headline shape at head dimension 128 (the head size of the focal-
    # attention models), same distributions and planted pairs.
    "fwd_bf16_t16384_d128": Workload("fwd_bf16_t16384_d128", 4, 12, 16384, 128, "bf16", 1.5, 128, 5),
}


def planted_pairs(B: int, H: int, T: int, pairs: int, seed: int):
    """List of (b, h, i, j) with k[b,h,j] := q[b,h,i]; distinct j per head."""
    rng = np.random.default_rng(seed)
    out = []
    if T < 2 or pairs <= 0:
        return out
    for b in range(B):
        for h in range(H):
            used = set()
            n = min(pairs, T - 1)
            while len(used) < n:
                i = int(rng.integers(1, T))
                j = int(rng.integers(0, i))
                if j in used:
                    continue
                used.add(j)
                out.append((b, h, i, j))
    return out


def torch_dtype(name: str):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def make_qkv(B, H, T, d, *, q_std=1.0, pairs=0, seed=0, dtype="f32", device="cpu"):
    """Seeded q, k, v of shape [B, H, T, d] (contiguous) on ``device``."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    shape = (B, H, T, d)
    q = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * q_std
    k = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    pp = planted_pairs(B, H, T, pairs, seed)
    if pp:
        idx = torch.tensor(pp, dtype=torch.long, device=device)
        b, h, i, j = idx.unbind(1)
        k[b, h, j] = q[b, h, i]
    td = torch_dtype(dtype)
    return q.to(td).contiguous(), k.to(td).contiguous(), v.to(td).contiguous()


def make_workload(w: Workload, device="cpu", B=None, T=None):
    """q, k, v for a named workload (optionally with a smaller B or T)."""
    return make_qkv(B or w.B, w.H, T or w.T, w.d, q_std=w.q_std, pairs=w.pairs, seed=w.seed,
                    dtype=w.dtype, device=device)


def make_like(shape, *, std=1.0, seed=0, dtype="f32", device="cpu"):
    """One seeded N(0, std^2) tensor (decode tokens, upstream gradients)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std
    return x.to(torch_dtype(dtype)).contiguous()
