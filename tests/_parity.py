"""Shared helpers for the GPU parity tests: run the oracle on the exact inputs
the CUDA path saw and compare with the tolerances of the spec.

Tolerances (written here, used by every parity test):
  fp32 inputs : per-row relative error of out, max_i ||g_i - o_i||_inf /
                max(||o_i||_inf, 1e-30) <= 1e-5.
  bf16 inputs : max abs error of out <= 2e-2 against the oracle run on the same
                bf16-rounded inputs (fp32 accumulation on the GPU);
                rows of A sum to 1 within 1e-5 (checked with v = 1).
  lse2        : |dlse2| <= 1e-5 * max(1, |lse2|) (fp32), 2e-3 (bf16 products).
  demand      : |dD| <= 1e-6 * max(D, 1) (fp32), 1e-3 * max(D, 1) + 1e-4 (bf16).
  rowsum      : relative 1e-5 (fp32), 2e-2 (bf16: shares are rounded to bf16).
"""
import math

import numpy as np
import torch

import oracle.dilution as od

LOG2E = 1.0 / math.log(2.0)

F32_OUT_REL = 1e-5
BF16_OUT_ABS = 2e-2


def host64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def row_rel_err(got, ref):
    """max over rows of ||got_i - ref_i||_inf / max(||ref_i||_inf, 1e-30)."""
    num = np.abs(got - ref).max(axis=-1)
    den = np.maximum(np.abs(ref).max(axis=-1), 1e-30)
    return float((num / den).max())


def oracle_forward(q, k, v, tau, eps, rows=None, heads=None):
    """Oracle outputs for [B,H,T,d] tensors.  ``heads`` = list of (b, h) to
    evaluate (default all); ``rows`` limits each head to queries [0, rows)."""
    qh, kh, vh = host64(q), host64(k), host64(v)
    B, H, T, _ = qh.shape
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    res = {}
    for (b, h) in heads:
        if rows is None and T <= 4096:
            r = od.dilution_forward_head(qh[b, h], kh[b, h], vh[b, h], tau, eps)
        else:
            r = od.dilution_forward_rowblocked_head(qh[b, h], kh[b, h], vh[b, h], tau, eps, rows=rows)
        res[(b, h)] = r
    return res
