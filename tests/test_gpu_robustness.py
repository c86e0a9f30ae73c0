"""GPU checks of the library's failure handling and memory discipline:

* a bounded wait that runs out (the decode test hook keeps one ring slot from
  being handed back) reports DA_ERR_TIMEOUT with its place, the call
  completes, and the next ordinary call is correct;
* a decode cache (keys, values, demand) saved to host memory and restored into
  fresh buffers continues exactly as the uninterrupted cache does;
* guard bands around every output buffer (forward, decode, backward) and after
  the workspace stay untouched at ragged sizes, the stand-in for a bounds
  checker of the kernels' stores, copy-engine stores and bulk reductions.
"""
import numpy as np
import pytest
import torch

import oracle.dilution as od
from long_context_attention_gb300 import binding as b
from long_context_attention_gb300 import inputs
from tests._parity import BF16_OUT_ABS, host64

pytestmark = pytest.mark.gpu
DEV = "cuda"


# ------------------------------------------------------------------ timeouts
def test_decode_wait_timeout_reported_and_recovered():
    B, H, d, n_ctx = 1, 3, 64, 5000          # key chunk 1 (keys 2048 .. 4095) streams 8 ring stages
    T_cap = n_ctx + 8
    tau, eps = 1.0990651, 1e-6
    kc, vc = (inputs.make_like((B, H, T_cap, d), seed=s, dtype="bf16", device=DEV) for s in (301, 302))
    g = torch.Generator(device=DEV).manual_seed(303)
    dem = torch.rand(B, H, T_cap, generator=g, device=DEV) * 2.0
    qn, kn, vn = (inputs.make_like((B, H, d), std=s, seed=310 + i, dtype="bf16", device=DEV)
                  for i, s in enumerate((1.5, 1.0, 1.0)))
    saved = (kc.clone(), vc.clone(), dem.clone())
    ws = torch.empty(b.dilution_attn_decode_workspace_size(B, H, T_cap, d), dtype=torch.uint8, device=DEV)

    # argument checks of the hook itself
    for bad in (dict(wait_limit_ns=10), dict(wait_limit_ns=2_000_000_000), dict(stall_bh=3), dict(stall_chunk=-1)):
        args = dict(stall_chunk=1, stall_bh=1, wait_limit_ns=2_000_000)
        args.update(bad)
        st, _ = b.dilution_attn_debug_decode_stall(qn, kn, vn, kc, vc, dem, n_ctx, tau=tau, eps=eps, workspace=ws,
                                                   **args)
        assert st == b.DA_ERR_INVALID, bad

    st, _ = b.dilution_attn_debug_decode_stall(qn, kn, vn, kc, vc, dem, n_ctx, tau=tau, eps=eps, workspace=ws,
                                               stall_chunk=1, stall_bh=1, wait_limit_ns=2_000_000)
    assert st == b.DA_OK                                  # launched; the failure is on the device
    words = b.dilution_attn_debug_last_timeout(ws)        # synchronises: the call completed
    assert words[0] == b.DA_ERR_TIMEOUT
    assert words[2] == 1                                  # the stalled chunk's block
    assert 0 <= words[3] < 288                            # a thread of that block (256 consumers + producer warp)
    assert words[1] > 0                                   # a barrier's shared-memory offset
    assert b.dilution_attn_get_error(ws) == b.DA_ERR_TIMEOUT
    assert b.dilution_attn_get_error(ws) == b.DA_OK       # read and cleared

    # the device is still usable: an ordinary step on the restored cache is correct
    kc.copy_(saved[0]), vc.copy_(saved[1]), dem.copy_(saved[2])
    ref_out, ref_dem = od.dilution_decode_step(host64(qn), host64(kn), host64(vn), host64(kc), host64(vc),
                                               host64(dem), n_ctx, tau, eps)
    out = b.dilution_attn_decode_step(qn, kn, vn, kc, vc, dem, n_ctx, tau=tau, eps=eps, workspace=ws)
    assert b.dilution_attn_get_error(ws) == b.DA_OK
    assert np.abs(host64(out) - ref_out).max() <= BF16_OUT_ABS
    assert np.all(np.abs(host64(dem[:, :, :n_ctx + 1]) - ref_dem) <= 1e-5 * np.maximum(ref_dem, 1.0) + 1e-6)


# ------------------------------------------------------------ checkpoint/resume
def test_decode_cache_resume_is_bit_exact():
    """Save the decode cache after 5 steps, restore it into fresh buffers and
    continue for 5 more: outputs, keys, values and demand equal those of the
    uninterrupted cache bit for bit (the step is deterministic)."""
    B, H, N, d = 2, 3, 3000, 64
    T_cap = N + 16
    tau, eps = 1.0990651, 1e-6
    q, k, v = inputs.make_qkv(B, H, N + 10, d, q_std=1.5, pairs=8, seed=320, dtype="bf16", device=DEV)
    kc = torch.zeros(B, H, T_cap, d, dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    kc[:, :, :N], vc[:, :, :N] = k[:, :, :N], v[:, :, :N]
    dem = torch.zeros(B, H, T_cap, device=DEV)
    d_out = torch.empty(B, H, N, device=DEV)
    b.dilution_attn_fwd(q[:, :, :N].contiguous(), k[:, :, :N].contiguous(), v[:, :, :N].contiguous(), None, None,
                        None, d_out, tau=tau, eps=eps)
    dem[:, :, :N] = d_out

    def step(kc, vc, dem, n):
        return b.dilution_attn_decode_step(q[:, :, n].contiguous(), k[:, :, n].contiguous(), v[:, :, n].contiguous(),
                                           kc, vc, dem, n, tau=tau, eps=eps).clone()

    for t in range(5):
        step(kc, vc, dem, N + t)
    torch.cuda.synchronize()
    host = [x.to("cpu").pin_memory() for x in (kc, vc, dem)]          # the checkpoint
    straight = [step(kc, vc, dem, N + 5 + t) for t in range(5)]
    kc2, vc2, dem2 = (torch.empty_like(x, device=DEV) for x in host)
    for dst, src in zip((kc2, vc2, dem2), host):
        dst.copy_(src, non_blocking=True)
    resumed = [step(kc2, vc2, dem2, N + 5 + t) for t in range(5)]
    torch.cuda.synchronize()
    for a, r in zip(straight, resumed):
        assert torch.equal(a, r)
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2) and torch.equal(dem, dem2)


# ---------------------------------------------------------------- guard bands
GUARD = 4096          # bytes before and after each buffer (keeps 16-byte alignment)
PAT = 0xA5


class Guarded:
    """A device tensor view of `shape`/`dtype` inside a byte buffer whose
    guard bands hold PAT."""

    def __init__(self, shape, dtype, fill=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.n = n
        self.raw = torch.full((GUARD + n + GUARD,), PAT, dtype=torch.uint8, device=DEV)
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def intact(self):
        torch.cuda.synchronize()
        return bool((self.raw[:GUARD] == PAT).all()) and bool((self.raw[GUARD + self.n:] == PAT).all())


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T", [1, 127, 129, 300])
def test_forward_writes_stay_inside_buffers(T, dtype):
    B, H, d = 1, 2, 64
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(B, H, T, d, q_std=1.5, pairs=min(4, T - 1), seed=330 + T,
                                                   dtype=dtype))
    td = q.dtype
    out = Guarded((B, H, T, d), td)
    lse2, rs, dem = (Guarded((B, H, T), torch.float32) for _ in range(3))
    wsz = b.dilution_attn_fwd_workspace_size(B, H, T, d, b._dtype_code(q))
    ws = Guarded((wsz,), torch.uint8)
    b.dilution_attn_fwd(q, k, v, out.t, lse2.t, rs.t, dem.t, workspace=ws.t)
    assert b.dilution_attn_get_error(ws.t) == b.DA_OK
    for g in (out, lse2, rs, dem, ws):
        assert g.intact()
    ref = od.dilution_forward(host64(q), host64(k), host64(v), 1.0, 1e-6)
    assert np.abs(host64(out.t) - ref["out"]).max() <= (BF16_OUT_ABS if dtype == "bf16" else 1e-4)


@pytest.mark.parametrize("T", [1, 127, 129, 300])
def test_backward_writes_stay_inside_buffers(T):
    B, H, d = 1, 2, 64
    q, k, v = (x.to(DEV) for x in inputs.make_qkv(B, H, T, d, seed=340 + T, dtype="bf16"))
    g = inputs.make_like((B, H, T, d), seed=350 + T, dtype="bf16", device=DEV)
    lse2 = torch.empty(B, H, T, device=DEV)
    b.dilution_attn_fwd(q, k, v, None, lse2)
    grads = [Guarded((B, H, T, d), torch.bfloat16) for _ in range(3)]
    wsz = b.dilution_attn_bwd_workspace_size(B, H, T, d, b.DA_BF16)
    ws = Guarded((wsz,), torch.uint8)
    b.dilution_attn_bwd(q, k, v, g, lse2, *(x.t for x in grads), workspace=ws.t)
    assert b.dilution_attn_get_error(ws.t) == b.DA_OK
    for x in grads + [ws]:
        assert x.intact()
    refs = od.dilution_backward(*(host64(t) for t in (q, k, v, g)), 1.0, 1e-6)
    for x, r in zip(grads, refs):
        assert np.abs(host64(x.t) - r).max() <= 1.5e-2 * max(np.abs(r).max(), 1e-3)


@pytest.mark.parametrize("n_ctx", [0, 127, 129, 2300])
def test_decode_writes_stay_inside_buffers(n_ctx):
    B, H, d = 2, 2, 64
    T_cap = n_ctx + 1                              # the new token fills the cache exactly
    kc0, vc0 = (inputs.make_like((B, H, T_cap, d), seed=s, dtype="bf16", device=DEV) for s in (361, 362))
    dem0 = torch.rand(B, H, T_cap, generator=torch.Generator(device=DEV).manual_seed(363), device=DEV)
    kc, vc = Guarded(kc0.shape, torch.bfloat16, kc0), Guarded(vc0.shape, torch.bfloat16, vc0)
    dem = Guarded(dem0.shape, torch.float32, dem0)
    qn, kn, vn = (inputs.make_like((B, H, d), std=s, seed=370 + i, dtype="bf16", device=DEV)
                  for i, s in enumerate((1.5, 1.0, 1.0)))
    out = Guarded((B, H, d), torch.bfloat16)
    wsz = b.dilution_attn_decode_workspace_size(B, H, T_cap, d)
    ws = Guarded((wsz,), torch.uint8)
    ref_out, _ = od.dilution_decode_step(host64(qn), host64(kn), host64(vn), host64(kc0), host64(vc0), host64(dem0),
                                         n_ctx, 1.0, 1e-6)
    b.dilution_attn_decode_step(qn, kn, vn, kc.t, vc.t, dem.t, n_ctx, out.t, workspace=ws.t)
    assert b.dilution_attn_get_error(ws.t) == b.DA_OK
    for x in (kc, vc, dem, out, ws):
        assert x.intact()
    assert np.abs(host64(out.t) - ref_out).max() <= BF16_OUT_ABS
