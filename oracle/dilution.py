"""Float64 CPU oracle for dilution attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA path.

What it computes, and where each step comes from:

* The operator, per (batch, head), follows the pseudocode in
  "DilutionAttention v0.1.0 · results", section "The operator":

      p         = causal softmax of the scaled logits       (the bids)
      committed = exclusive cumulative sum of p down each key column,
                  i.e. the demand that earlier queries placed on the key
      share     = p / (committed + p + eps)
      A         = share / rowsum(share),   out = A @ v

* The logit multiplier ``tau`` (default 1) is the temperature of
  "Focal Attention" (arXiv 2511.06818), section "Transformer with Constant
  Temperature", eq. focal-const, written as a multiplier: tau = 1/t.  The
  YaRN value tau = sqrt(0.1 ln s + 1) is from "YaRN › Attention Temperature
  Scaling", the temperature formula and its table of scaling factors.

* Cached decoding keeps, per key and head, the running total of the bids the
  key has received; "DilutionAttention v0.1.0 · results", section "The
  operator", last paragraph.  Reading taken here: the total is inclusive of
  every query processed so far and is updated after the step's output is
  formed; a newly appended key starts at zero.

* The "earlier demand only" variant (``earlier_only=True``): the results
  page, in the paragraph after "The operator", describes dividing each bid
  by the earlier demand alone, which lets every key win its own first query
  (the key itself) outright.  Reading taken: share = p / (committed + eps);
  eps keeps the diagonal entry defined.  The page trained a model this way,
  so the backward takes the flag too.

* ``tau`` may be a scalar or an array broadcastable to [B, H] in the batched
  functions: one logit multiplier per (batch, head), the per-head
  temperature of "Learning to Focus: Focal Attention for Selective and
  Scalable Transformers", section "Transformer with Learned Temperature"
  (learned there, given here as an input).

* The backward pass is not written out on any page (the results page only
  says exact gradients exist).  ``dilution_backward`` is the chain rule through
  the forward above, derived by hand: softmax, exclusive column cumsum,
  share, renormalisation and the value product.

All arithmetic is float64 NumPy.  Masked entries (key after query) carry
p = 0, committed = 0 and share = 0 exactly.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, brute force, finite differences, the YaRN table).
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "yarn_temperature",
    "yarn_tau",
    "logit_scale",
    "dilution_forward_head",
    "dilution_forward",
    "dilution_forward_rowblocked_head",
    "dilution_decode_step_head",
    "dilution_decode_step",
    "dilution_backward_head",
    "dilution_backward",
    "dilution_backward_rowblocked_head",
]


# ---------------------------------------------------------------------------
# Temperature
# ---------------------------------------------------------------------------
def yarn_temperature(scale: float) -> float:
    """YaRN attention temperature t = 0.1 * ln(s) + 1 for an extension factor s.

    Source: "YaRN › Attention Temperature Scaling", the temperature formula.
    """
    return 0.1 * math.log(scale) + 1.0


def yarn_tau(scale: float) -> float:
    """Logit multiplier sqrt(t) that YaRN applies before the softmax.

    Source: "YaRN › Attention Temperature Scaling" (the sqrt(t) column of its
    table of scaling factors).
    """
    return math.sqrt(yarn_temperature(scale))


def logit_scale(d: int, tau: float) -> float:
    """Scale applied to q.k: tau / sqrt(d).

    sqrt(d) is the softmax temperature of scaled dot-product attention
    ("Focal Attention", section "Transformer with Constant Temperature");
    tau multiplies the logits (tau = 1/t for the focal constant t).
    """
    return tau / math.sqrt(d)


# ---------------------------------------------------------------------------
# Forward, one head, full T x T matrices
# ---------------------------------------------------------------------------
def _causal_softmax(s: np.ndarray) -> np.ndarray:
    """Row softmax over keys k <= i (diagonal included), max-subtracted.

    Entries with k > i are exactly 0.
    """
    T = s.shape[0]
    mask = np.tril(np.ones((T, T), dtype=bool))
    z = np.where(mask, s, -np.inf)
    m = z.max(axis=1, keepdims=True)
    e = np.where(mask, np.exp(z - m), 0.0)
    return e / e.sum(axis=1, keepdims=True)


def _exclusive_cumsum_cols(p: np.ndarray) -> np.ndarray:
    """committed[i, k] = sum_{j < i} p[j, k]: demand from strictly earlier queries.

    The cumulative sum runs down each key column over the query axis
    ("DilutionAttention v0.1.0 · results", section "The operator").
    """
    committed = np.zeros_like(p)
    if p.shape[0] > 1:
        committed[1:] = np.cumsum(p, axis=0)[:-1]
    return committed


def dilution_forward_head(q, k, v, tau: float = 1.0, eps: float = 1e-6, full: bool = False,
                          earlier_only: bool = False):
    """Dilution attention forward for one (batch, head) slice.

    q, k: [T, d]; v: [T, dv].  Returns a dict with
      out [T, dv], rowsum [T] (sum_k share_ik), demand [T] (column totals of p,
      the decode cache after the last query), lse [T] (natural-log normaliser
      m_i + log(sum_k exp(s_ik - m_i)) of the scaled logits),
    and, when ``full``: p, committed, share, A (all [T, T]).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, d = q.shape
    if eps <= 0:
        raise ValueError("eps must be > 0")
    s = logit_scale(d, tau) * (q @ k.T)
    mask = np.tril(np.ones((T, T), dtype=bool))
    z = np.where(mask, s, -np.inf)
    m = z.max(axis=1)
    lse = m + np.log(np.where(mask, np.exp(z - m[:, None]), 0.0).sum(axis=1))
    p = _causal_softmax(s)
    committed = _exclusive_cumsum_cols(p)
    share = p / (committed + eps) if earlier_only else p / (committed + p + eps)
    rowsum = share.sum(axis=1)
    A = share / rowsum[:, None]
    out = A @ v
    res = {"out": out, "rowsum": rowsum, "demand": p.sum(axis=0), "lse": lse}
    if full:
        res.update(p=p, committed=committed, share=share, A=A)
    return res


def dilution_forward(q, k, v, tau=1.0, eps: float = 1e-6, earlier_only: bool = False):
    """Batched forward over [B, H, T, d] inputs; heads are independent.
    ``tau``: scalar or array broadcastable to [B, H].

    Returns dict of out [B,H,T,dv], rowsum [B,H,T], demand [B,H,T], lse [B,H,T].
    """
    q = np.asarray(q, dtype=np.float64)
    B, H, T, _ = q.shape
    taus = np.broadcast_to(np.asarray(tau, dtype=np.float64), (B, H))
    dv = np.shape(v)[-1]
    out = np.empty((B, H, T, dv))
    rowsum = np.empty((B, H, T))
    demand = np.empty((B, H, T))
    lse = np.empty((B, H, T))
    for b in range(B):
        for h in range(H):
            r = dilution_forward_head(q[b, h], k[b, h], v[b, h], float(taus[b, h]), eps, earlier_only=earlier_only)
            out[b, h], rowsum[b, h], demand[b, h], lse[b, h] = r["out"], r["rowsum"], r["demand"], r["lse"]
    return {"out": out, "rowsum": rowsum, "demand": demand, "lse": lse}


# ---------------------------------------------------------------------------
# Forward, one head, row-blocked (for T too large for T x T matrices)
# ---------------------------------------------------------------------------
def dilution_forward_rowblocked_head(q, k, v, tau: float = 1.0, eps: float = 1e-6,
                                     rows: int | None = None, block: int = 1024, earlier_only: bool = False):
    """Same operator as ``dilution_forward_head``, evaluated block of queries by
    block of queries, carrying the column demand of all earlier blocks.

    Only queries [0, rows) are produced (default: all).  Memory is
    O(block * T); the arithmetic per entry is the same as the full version.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, d = q.shape
    n = T if rows is None else int(rows)
    c = logit_scale(d, tau)
    carried = np.zeros(T)          # sum of p over all queries before the block
    out = np.empty((n, v.shape[1]))
    rowsum = np.empty(n)
    lse = np.empty(n)
    for i0 in range(0, n, block):
        i1 = min(n, i0 + block)
        kk = i1                      # keys 0 .. i1-1 are visible to some query of the block
        s = c * (q[i0:i1] @ k[:kk].T)
        qi = np.arange(i0, i1)[:, None]
        mask = np.arange(kk)[None, :] <= qi
        z = np.where(mask, s, -np.inf)
        m = z.max(axis=1)
        e = np.where(mask, np.exp(z - m[:, None]), 0.0)
        l = e.sum(axis=1)
        p = e / l[:, None]
        lse[i0:i1] = m + np.log(l)
        committed = carried[None, :kk] + _exclusive_cumsum_cols(p)
        share = p / (committed + eps) if earlier_only else p / (committed + p + eps)
        rs = share.sum(axis=1)
        out[i0:i1] = (share / rs[:, None]) @ v[:kk]
        rowsum[i0:i1] = rs
        carried[:kk] += p.sum(axis=0)
    return {"out": out, "rowsum": rowsum, "lse": lse, "demand": carried}


# ---------------------------------------------------------------------------
# Cached decode
# ---------------------------------------------------------------------------
def dilution_decode_step_head(q_new, k_new, v_new, k_cache, v_cache, demand, n_ctx: int,
                              tau: float = 1.0, eps: float = 1e-6, earlier_only: bool = False):
    """One cached-decode step for one (batch, head).

    The cache holds keys/values 0 .. n_ctx-1 and their running demand totals.
    The new key/value are appended at position n_ctx (its demand starts at 0);
    the new query attends to keys 0 .. n_ctx.  Returns (out [dv], demand_new
    [n_ctx+1], k_all, v_all) where demand_new = demand + p for this query.
    """
    q_new = np.asarray(q_new, dtype=np.float64)
    K = np.concatenate([np.asarray(k_cache, np.float64)[:n_ctx], np.asarray(k_new, np.float64)[None]], axis=0)
    V = np.concatenate([np.asarray(v_cache, np.float64)[:n_ctx], np.asarray(v_new, np.float64)[None]], axis=0)
    D = np.concatenate([np.asarray(demand, np.float64)[:n_ctx], [0.0]])
    s = logit_scale(q_new.shape[0], tau) * (K @ q_new)
    e = np.exp(s - s.max())
    p = e / e.sum()
    share = p / (D + eps) if earlier_only else p / (D + p + eps)
    out = (share @ V) / share.sum()
    return out, D + p, K, V


def dilution_decode_step(q_new, k_new, v_new, k_cache, v_cache, demand, n_ctx: int,
                         tau=1.0, eps: float = 1e-6, earlier_only: bool = False):
    """Batched decode step: q_new/k_new/v_new [B,H,d]; caches [B,H,>=n_ctx,d];
    demand [B,H,>=n_ctx]; ``tau`` scalar or broadcastable to [B, H].
    Returns (out [B,H,dv], demand_new [B,H,n_ctx+1])."""
    q_new = np.asarray(q_new, np.float64)
    B, H, _ = q_new.shape
    taus = np.broadcast_to(np.asarray(tau, dtype=np.float64), (B, H))
    out = np.empty((B, H, np.shape(v_new)[-1]))
    dn = np.empty((B, H, n_ctx + 1))
    for b in range(B):
        for h in range(H):
            o, dd, _, _ = dilution_decode_step_head(q_new[b, h], k_new[b, h], v_new[b, h], k_cache[b, h],
                                                   v_cache[b, h], demand[b, h], n_ctx, float(taus[b, h]), eps,
                                                   earlier_only)
            out[b, h], dn[b, h] = o, dd
    return out, dn


# ---------------------------------------------------------------------------
# Backward, one head (hand-derived chain rule; no page states it)
# ---------------------------------------------------------------------------
def _reverse_exclusive_cumsum_cols(x: np.ndarray) -> np.ndarray:
    """out[j, k] = sum_{i > j} x[i, k]: the adjoint of the exclusive column cumsum."""
    out = np.zeros_like(x)
    if x.shape[0] > 1:
        out[:-1] = np.cumsum(x[::-1], axis=0)[::-1][1:]
    return out


def dilution_backward_head(q, k, v, dout, tau: float = 1.0, eps: float = 1e-6, earlier_only: bool = False):
    """Gradients (dq, dk, dv) of sum(dout * out) for one head.

    With c = tau/sqrt(d), r = share, R = rowsum(share), D = committed + p + eps:
      dV_k   = sum_i A_ik dout_i
      dr_ik  = (dout_i . v_k - dout_i . out_i) / R_i            (k <= i)
      dC_ik  = -dr_ik p_ik / D_ik^2                              (d share / d committed)
      dp_jk  = dr_jk (committed_jk + eps) / D_jk^2 + sum_{i > j} dC_ik
      ds_jk  = p_jk (dp_jk - sum_k' p_jk' dp_jk')                (softmax)
      dq     = c ds k,   dk = c ds^T q
    With ``earlier_only`` (share = p / (committed + eps)) D = committed + eps
    and the direct term of dp is dr_jk / D_jk instead.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(dout, np.float64)
    T, d = q.shape
    c = logit_scale(d, tau)
    f = dilution_forward_head(q, k, v, tau, eps, full=True, earlier_only=earlier_only)
    p, C, A, out, R = f["p"], f["committed"], f["A"], f["out"], f["rowsum"]
    mask = np.tril(np.ones((T, T), dtype=bool))
    Dn = C + eps if earlier_only else C + p + eps
    dv = A.T @ g
    dA = g @ v.T
    delta = np.sum(g * out, axis=1)
    dr = np.where(mask, (dA - delta[:, None]) / R[:, None], 0.0)
    dC = -dr * p / Dn**2
    direct = dr / Dn if earlier_only else dr * (C + eps) / Dn**2
    dp = direct + _reverse_exclusive_cumsum_cols(dC)
    ds = p * (dp - np.sum(p * dp, axis=1, keepdims=True))
    dq = c * (ds @ k)
    dk = c * (ds.T @ q)
    return dq, dk, dv


def dilution_backward(q, k, v, dout, tau=1.0, eps: float = 1e-6, earlier_only: bool = False):
    """Batched backward over [B,H,T,d]; ``tau`` scalar or broadcastable to
    [B, H]; returns (dq, dk, dv)."""
    q = np.asarray(q, np.float64)
    B, H, T, d = q.shape
    taus = np.broadcast_to(np.asarray(tau, dtype=np.float64), (B, H))
    dq = np.empty_like(q)
    dk = np.empty((B, H, T, d))
    dv = np.empty((B, H, T, np.shape(v)[-1]))
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = dilution_backward_head(q[b, h], k[b, h], v[b, h], dout[b, h],
                                                                  float(taus[b, h]), eps, earlier_only)
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Backward, one head, row-blocked (for T too large for T x T matrices)
# ---------------------------------------------------------------------------
def dilution_backward_rowblocked_head(q, k, v, dout, tau: float = 1.0, eps: float = 1e-6, block: int = 1024,
                                      earlier_only: bool = False):
    """Same gradients as ``dilution_backward_head``, with O(block * T) memory.

    The chain rule needs, for every (query j, key k), committed_jk (a sum over
    the queries before j) and sum_{i > j} dC_ik (a sum over the queries
    after j).  Blocks of queries are taken twice: ascending, as the row-blocked
    forward, to get lse, R and out of every row and the column demand carried
    into each block; then descending, carrying sum_i dC_ik of the blocks
    already visited, to form dp, rho, ds and the three gradients block by
    block.  Each entry goes through the same formulas as the full version.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(dout, np.float64)
    T, d = q.shape
    c = logit_scale(d, tau)
    starts = list(range(0, T, block))
    lse = np.empty(T)
    R = np.empty(T)
    out = np.empty((T, v.shape[1]))
    carried_in = []                  # column demand before each block
    carried = np.zeros(T)

    def block_bids(i0, i1):
        kk = i1
        s = c * (q[i0:i1] @ k[:kk].T)
        mask = np.arange(kk)[None, :] <= np.arange(i0, i1)[:, None]
        return s, mask, kk

    for i0 in starts:
        i1 = min(T, i0 + block)
        s, mask, kk = block_bids(i0, i1)
        z = np.where(mask, s, -np.inf)
        m = z.max(axis=1)
        e = np.where(mask, np.exp(z - m[:, None]), 0.0)
        l = e.sum(axis=1)
        p = e / l[:, None]
        lse[i0:i1] = m + np.log(l)
        committed = carried[None, :kk] + _exclusive_cumsum_cols(p)
        share = p / (committed + eps) if earlier_only else p / (committed + p + eps)
        R[i0:i1] = share.sum(axis=1)
        out[i0:i1] = (share / R[i0:i1, None]) @ v[:kk]
        carried_in.append(carried.copy())
        carried[:kk] += p.sum(axis=0)

    dq = np.empty((T, d))
    dk = np.zeros((T, d))
    dv = np.zeros((T, v.shape[1]))
    delta = np.sum(g * out, axis=1)
    rev = np.zeros(T)                # sum of dC over the queries of the blocks after this one
    for bi in range(len(starts) - 1, -1, -1):
        i0 = starts[bi]
        i1 = min(T, i0 + block)
        s, mask, kk = block_bids(i0, i1)
        p = np.where(mask, np.exp(np.where(mask, s, -np.inf) - lse[i0:i1, None]), 0.0)
        C = carried_in[bi][None, :kk] + _exclusive_cumsum_cols(p)
        Dn = C + eps if earlier_only else C + p + eps
        share = p / Dn
        A = share / R[i0:i1, None]
        gb = g[i0:i1]
        dv[:kk] += A.T @ gb
        dA = gb @ v[:kk].T
        dr = np.where(mask, (dA - delta[i0:i1, None]) / R[i0:i1, None], 0.0)
        dC = -dr * p / Dn**2
        direct = dr / Dn if earlier_only else dr * (C + eps) / Dn**2
        dp = direct + _reverse_exclusive_cumsum_cols(dC) + rev[None, :kk]
        ds = p * (dp - np.sum(p * dp, axis=1, keepdims=True))
        dq[i0:i1] = c * (ds @ k[:kk])
        dk[:kk] += c * (ds.T @ q[i0:i1])
        rev[:kk] += dC.sum(axis=0)
    return dq, dk, dv

