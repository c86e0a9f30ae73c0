"""Host-side checks of the seeded input generator (no operator arithmetic here
except through the oracle)."""
import numpy as np
import torch

import oracle.dilution as od
from long_context_attention_gb300 import inputs, yarn_tau


def test_seeded_and_reproducible():
    a = inputs.make_qkv(1, 2, 33, 8, q_std=1.5, pairs=4, seed=5)
    b = inputs.make_qkv(1, 2, 33, 8, q_std=1.5, pairs=4, seed=5)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    c = inputs.make_qkv(1, 2, 33, 8, q_std=1.5, pairs=4, seed=6)
    assert not torch.equal(a[0], c[0])


def test_planted_pairs_distinct_and_causal():
    pp = inputs.planted_pairs(2, 3, 100, 32, seed=1)
    assert len(pp) == 2 * 3 * 32
    for b in range(2):
        for h in range(3):
            js = [j for (bb, hh, i, j) in pp if (bb, hh) == (b, h)]
            assert len(js) == len(set(js))
    assert all(0 <= j < i < 100 for (_, _, i, j) in pp)


def test_planted_key_copies_query_and_dominates_bid():
    q, k, v = inputs.make_qkv(1, 1, 128, 64, q_std=1.5, pairs=8, seed=3, dtype="bf16")
    pp = inputs.planted_pairs(1, 1, 128, 8, seed=3)
    r = od.dilution_forward_head(q[0, 0].double().numpy(), k[0, 0].double().numpy(),
                                 v[0, 0].double().numpy(), 1.0, 1e-6, full=True)
    for (_, _, i, j) in pp:
        assert torch.equal(k[0, 0, j], q[0, 0, i])
        # |q|^2/8 ~ 18 versus N(0, 1.5^2) background logits: the planted key wins the row.
        assert r["p"][i].argmax() == j or r["p"][i, j] > 0.5


def test_bf16_rounding_is_nearest_even():
    x = inputs.make_like((1000,), std=3.0, seed=9)
    xb = x.to(torch.bfloat16).float()
    bits = x.view(torch.int32).numpy().astype(np.int64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) >> 16) << 16
    assert np.array_equal(xb.view(torch.int32).numpy().astype(np.int64) & 0xFFFFFFFF, rounded & 0xFFFFFFFF)


def test_workload_table():
    w = inputs.WORKLOADS["fwd_bf16_t16384"]
    assert (w.B, w.H, w.T, w.d, w.pairs) == (4, 12, 16384, 64, 128)
    assert inputs.WORKLOADS["fwd_f32_t256"].dtype == "f32"
    assert abs(yarn_tau(inputs.WORKLOADS["prefill_bf16_t131072"].tau_scale) - od.yarn_tau(8)) < 1e-15
