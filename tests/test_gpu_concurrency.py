"""Concurrent use of the library on one GPU.

* Two forwards in flight at once on two streams, each with its own
  workspace: both match the oracle (no state is shared between calls but the
  per-device one-time set-up).
* A fresh process whose first calls of the forward, the decode step and the
  backward come from four host threads at the same moment, each on its own
  stream: the per-device one-time set-up (shared-memory opt-ins, the
  register-split check) is guarded, so every thread's results match the
  oracle.

Operator: "DilutionAttention v0.1.0 · results", section "The operator" and
its cached-decoding paragraph.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

import oracle.dilution as od
from long_context_attention_gb300 import binding as b
from long_context_attention_gb300 import inputs
from tests._parity import BF16_OUT_ABS, host64

pytestmark = pytest.mark.gpu
DEV = "cuda"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_two_streams_in_flight():
    B, H, T, d = 1, 3, 2000, 64
    runs = []
    for seed in (501, 502):
        q, k, v = inputs.make_qkv(B, H, T, d, q_std=1.5, pairs=8, seed=seed, dtype="bf16", device=DEV)
        ws = torch.empty(b.dilution_attn_fwd_workspace_size(B, H, T, d, b.DA_BF16), dtype=torch.uint8, device=DEV)
        runs.append((q, k, v, torch.empty_like(q), ws, torch.cuda.Stream()))
    torch.cuda.synchronize()
    for q, k, v, out, ws, s in runs:          # both enqueued before either is waited on
        b.dilution_attn_fwd(q, k, v, out, workspace=ws, stream=s)
    for q, k, v, out, ws, s in runs:
        assert b.dilution_attn_get_error(ws, s) == b.DA_OK
        ref = od.dilution_forward(host64(q), host64(k), host64(v), 1.0, 1e-6)["out"]
        assert np.abs(host64(out) - ref).max() <= BF16_OUT_ABS


CHILD = textwrap.dedent("""
    import sys, threading
    import numpy as np, torch
    sys.path.insert(0, {root!r})
    import oracle.dilution as od
    from long_context_attention_gb300 import binding as b, inputs
    from tests._parity import BF16_OUT_ABS, host64
    DEV = "cuda"
    torch.cuda.init()
    go = threading.Barrier(4)
    results, errors = {{}}, []

    def work(i):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            B, H, T, d = 1, 2, 300, 64
            with torch.cuda.stream(s):
                q, k, v = inputs.make_qkv(B, H, T, d, q_std=1.5, pairs=4, seed=600 + i, dtype="bf16", device=DEV)
                g = inputs.make_like((B, H, T, d), seed=610 + i, dtype="bf16", device=DEV)
                kc = torch.zeros(B, H, T + 1, d, dtype=torch.bfloat16, device=DEV)
                vc = torch.zeros_like(kc)
                kc[:, :, :T], vc[:, :, :T] = k, v
                dem = torch.zeros(B, H, T + 1, device=DEV)
                d_out = torch.empty(B, H, T, device=DEV)
                lse2 = torch.empty(B, H, T, device=DEV)
                tok = [inputs.make_like((B, H, d), std=1.5 if j == 0 else 1.0, seed=620 + 3 * i + j,
                                        dtype="bf16", device=DEV) for j in range(3)]
                s.synchronize()
                go.wait()                       # first calls of every entry point at the same moment
                out = b.dilution_attn_fwd(q, k, v, None, lse2, None, d_out, stream=s)
                dem[:, :, :T] = d_out
                dem0 = dem.clone()
                o1 = b.dilution_attn_decode_step(*tok, kc, vc, dem, T, stream=s)
                dq, dk, dv = b.dilution_attn_bwd(q, k, v, g, lse2, stream=s)
                s.synchronize()
            kc0 = kc.clone()
            kc0[:, :, T] = 0
            vc0 = vc.clone()
            vc0[:, :, T] = 0
            results[i] = [host64(x) for x in (q, k, v, g, out, dq, dk, dv, *tok, kc0, vc0, dem0, o1)]
        except Exception as e:                  # reported by the parent
            errors.append(repr(e))

    ts = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    for t in ts: t.start()
    for t in ts: t.join()
    assert not errors, errors
    for i, (q, k, v, g, out, dq, dk, dv, qn, kn, vn, kc0, vc0, dem0, o1) in results.items():
        ref = od.dilution_forward(q, k, v, 1.0, 1e-6)["out"]
        assert np.abs(out - ref).max() <= BF16_OUT_ABS, i
        o_ref, _ = od.dilution_decode_step(qn, kn, vn, kc0, vc0, dem0, q.shape[2], 1.0, 1e-6)
        assert np.abs(o1 - o_ref).max() <= BF16_OUT_ABS, i
        for got, r in zip((dq, dk, dv), od.dilution_backward(q, k, v, g, 1.0, 1e-6)):
            assert np.abs(got - r).max() <= 1.5e-2 * max(np.abs(r).max(), 1e-3), i
    print("ok", len(results))
""")


def test_first_calls_from_threads_in_a_fresh_process():
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT)], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert r.stdout.strip().endswith("ok 4")
