"""CPU-only checks of the C-ABI library: it loads, exports every symbol the
header declares, validates arguments before touching the GPU, and its integer
artefacts (tile schedules, causal mask) match independent CPU generators bit
for bit."""
import ctypes

import numpy as np
import pytest

from long_context_attention_gb300 import binding as b


@pytest.fixture(scope="module")
def lib():
    return b.load()


def test_exports_every_header_symbol(lib):
    names = b.header_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert b.status_string(b.DA_OK) == "DA_OK"
    for s in range(1, 6):
        assert b.status_string(s).startswith("DA_ERR_")
    assert b.status_string(99) == "unknown status"
    assert b.dilution_attn_version() >= 100


def _groups(BH, hg):
    # group sizes: the remainder (BH mod hg, if any) first, then full groups
    sizes = ([BH % hg] if BH % hg else []) + [hg] * (BH // hg)
    starts = np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(int)
    return zip(starts, sizes)


def _sched_rowstats(BH, T, d=64):
    # pairs of 128-row query tiles; heads grouped so their Q and K total ~96 MB
    Tp = -(-T // 256) * 256
    npairs = Tp // 256
    hg = min(BH, max(1, (96 << 20) // (Tp * d * 4)))
    rows = []
    for h0, n in _groups(BH, hg):
        for pair in range(npairs - 1, -1, -1):
            for bh in range(h0, h0 + n):
                rows.append((bh, 2 * pair, 2, 0))
    return np.array(rows, dtype=np.int32).reshape(-1, 4)


def _sched_sweep(BH, T, d=64):
    # spans of 384 keys (three key tiles) at d = 64, 256 (two) at d = 128;
    # heads grouped so their fp32 accumulators (Tp rows of d + 4) total ~64 MB
    span_keys = 384 if d == 64 else 256
    Tp = -(-T // 256) * 256
    nqt, nspan = Tp // 128, -(-Tp // span_keys)
    hg = min(BH, max(1, (64 << 20) // (Tp * (d + 4) * 4)))
    rows = []
    for h0, n in _groups(BH, hg):
        heads = list(range(h0, h0 + n))
        for span in range(nspan):
            for bh in heads:
                q0 = span_keys * span // 128
                rows.append((bh, q0, nqt - q0, span_keys * span))
    return np.array(rows, dtype=np.int32).reshape(-1, 4)


def _sched_bwd(BH, T, d, pass_):
    # one CTA per (head, 128-key tile) for the reverse (0) and light dK (1)
    # passes, per (head, 128-query tile) for the dQ pass (2); heads grouped
    # so their two streamed [Tp x d] bf16 operands total ~96 MB, except the
    # reverse pass at d = 64 (every head's tile 0, then tile 1, ...)
    Tp = -(-T // 256) * 256
    nt = Tp // 128
    hg = min(BH, max(1, (96 << 20) // (Tp * d * 4)))
    if pass_ == 0 and d == 64:
        order = [(c % BH, c // BH) for c in range(BH * nt)]
    else:
        order = [(bh, i) for h0, n in _groups(BH, hg) for i in range(nt) for bh in range(h0, h0 + n)]
    rows = [(bh, nt - 1 - i, 1, 0) if pass_ == 2 else (bh, i, nt - i, 128 * i) for bh, i in order]
    return np.array(rows, dtype=np.int32).reshape(-1, 4)


# (5, 131072) and (7, 65536): head groups that do not divide the heads (the
# remainder group first) in the row statistics and the backward
@pytest.mark.parametrize("BH,T", [(1, 1), (2, 255), (3, 256), (5, 257), (48, 16384), (12, 131072), (5, 131072),
                                  (7, 65536)])
def test_tile_schedules_bit_exact(lib, BH, T):
    assert np.array_equal(b.dilution_attn_debug_tile_schedule(BH, T, 0), _sched_rowstats(BH, T))
    assert np.array_equal(b.dilution_attn_debug_tile_schedule(BH, T, 1), _sched_sweep(BH, T))
    assert np.array_equal(b.dilution_attn_debug_tile_schedule(BH, T, 2), _sched_sweep(BH, T, 128))
    assert np.array_equal(b.dilution_attn_debug_tile_schedule(BH, T, 3), _sched_rowstats(BH, T, 128))
    for pass_ in range(3):
        for d in (64, 128):
            got = b.dilution_attn_debug_tile_schedule(BH, T, 4 + 2 * pass_ + (d == 128))
            assert np.array_equal(got, _sched_bwd(BH, T, d, pass_)), (pass_, d)


@pytest.mark.parametrize("BH,T", [(3, 1000), (5, 131072), (7, 65536)])
def test_backward_and_rowstats_schedules_cover_once(BH, T):
    # every (head, key tile) once in the key-tile passes, every (head, query
    # tile) once in the dQ pass and the row statistics, at both head sizes
    Tp = -(-T // 256) * 256
    nt = Tp // 128
    everything = sorted((bh, t) for bh in range(BH) for t in range(nt))
    for d in (64, 128):
        for pass_ in range(3):
            s = b.dilution_attn_debug_tile_schedule(BH, T, 4 + 2 * pass_ + (d == 128))
            if pass_ == 2:
                assert sorted((int(r[0]), int(r[1])) for r in s) == everything
                assert all(int(r[2]) == 1 for r in s)
            else:
                assert sorted((int(r[0]), int(r[3]) // 128) for r in s) == everything
                assert all(int(r[1]) == int(r[3]) // 128 and int(r[1]) + int(r[2]) == nt for r in s)
        rs = b.dilution_attn_debug_tile_schedule(BH, T, 0 if d == 64 else 3)
        assert sorted((int(r[0]), int(r[1]) + i) for r in rs for i in range(r[2])) == everything


@pytest.mark.parametrize("kernel,tiles_per_span", [(1, 3), (2, 2)])
def test_tile_schedules_cover_triangle_once(kernel, tiles_per_span):
    # every (head, key, query) pair with key <= query < Tp is visited by exactly
    # one sweep CTA (128-key tiles x 128-query tiles; kernel 1: d = 64, 2:
    # d = 128), every 128-row query tile by one row-statistics CTA
    BH, T = 3, 1000
    Tp = 1024
    seen = {}
    for bh, q0, n, key0 in b.dilution_attn_debug_tile_schedule(BH, T, kernel):
        for kt in range(key0 // 128, key0 // 128 + tiles_per_span):
            for qt in range(q0, q0 + n):
                if kt * 128 < Tp and kt * 128 <= qt * 128 + 127:
                    seen[(bh, kt, qt)] = seen.get((bh, kt, qt), 0) + 1
    want = {(bh, kt, qt) for bh in range(BH) for qt in range(Tp // 128) for kt in range(Tp // 128)
            if kt * 128 <= qt * 128 + 127}
    assert set(seen) == want and all(v == 1 for v in seen.values())
    for k in (0, 3):
        rs = b.dilution_attn_debug_tile_schedule(BH, T, k)
        tiles = sorted((int(r[0]), int(r[1]) + i) for r in rs for i in range(r[2]))
        assert tiles == sorted((bh, qt) for bh in range(BH) for qt in range(Tp // 128))


@pytest.mark.parametrize("T,qt,kt", [(256, 0, 0), (256, 1, 0), (200, 1, 1), (130, 1, 1), (1000, 3, 5), (5, 0, 0)])
def test_tile_mask_bit_exact(lib, T, qt, kt):
    r = np.arange(128)[:, None] + qt * 128
    c = np.arange(128)[None, :] + kt * 128
    want = ((c <= r) & (r < T)).astype(np.uint8)
    assert np.array_equal(b.dilution_attn_debug_tile_mask(T, qt, kt), want)


def test_workspace_sizes(lib):
    Tp = 16384
    for d in (64, 128):
        want = 256 + 48 * Tp * 4
        want = -(-want // 256) * 256 + 48 * Tp * (d + 4) * 4
        assert b.dilution_attn_fwd_workspace_size(4, 12, 16384, d, b.DA_BF16) == want
    assert b.dilution_attn_fwd_workspace_size(4, 12, 16384, 96, b.DA_BF16) == 0   # unsupported d
    assert b.dilution_attn_bwd_workspace_size(1, 1, 100, 128, 1) > 100 * 128 * 4
    assert b.dilution_attn_fwd_workspace_size(0, 12, 16384, 64, b.DA_BF16) == 256
    assert b.dilution_attn_decode_workspace_size(8, 12, 131328, 64) > 8 * 12 * 131328 * 4


# Argument validation happens before any CUDA call, so it runs without a GPU.
FAKE = ctypes.c_void_p(0x10000)
MIS = ctypes.c_void_p(0x10004)


def _fwd(lib, q=FAKE, out=FAKE, B=1, H=1, T=8, d=64, tau=1.0, eps=1e-6, dtype=1, ws=FAKE, wsb=1 << 30):
    return lib.dilution_attn_fwd(q, FAKE, FAKE, out, None, None, None, B, H, T, d, tau, eps, dtype, ws, wsb, None)


def test_fwd_argument_validation(lib):
    assert _fwd(lib, eps=0.0) == b.DA_ERR_INVALID
    assert _fwd(lib, eps=-1.0) == b.DA_ERR_INVALID
    assert _fwd(lib, eps=float("nan")) == b.DA_ERR_INVALID
    assert _fwd(lib, tau=-0.5) == b.DA_ERR_INVALID
    assert _fwd(lib, tau=float("inf")) == b.DA_ERR_INVALID
    assert _fwd(lib, d=96) == b.DA_ERR_UNSUPPORTED
    assert _fwd(lib, d=256) == b.DA_ERR_UNSUPPORTED
    assert _fwd(lib, d=128, ws=None) == b.DA_ERR_WORKSPACE      # d = 128 is supported
    assert _fwd(lib, eps=1e-20) == b.DA_ERR_UNSUPPORTED        # bf16 path: eps >= 1e-18
    assert _fwd(lib, eps=1e-20, dtype=0, ws=None) == b.DA_ERR_WORKSPACE   # fp32 path accepts it
    assert _fwd(lib, T=(1 << 24) + 1) == b.DA_ERR_UNSUPPORTED
    assert _fwd(lib, B=-1) == b.DA_ERR_INVALID
    assert _fwd(lib, dtype=7) == b.DA_ERR_INVALID
    assert _fwd(lib, q=None) == b.DA_ERR_INVALID
    assert _fwd(lib, out=MIS) == b.DA_ERR_INVALID
    assert _fwd(lib, ws=None) == b.DA_ERR_WORKSPACE
    assert _fwd(lib, wsb=1024) == b.DA_ERR_WORKSPACE
    # empty problems are valid no-ops, whatever the pointers
    assert _fwd(lib, q=None, T=0) == b.DA_OK
    assert _fwd(lib, q=None, B=0) == b.DA_OK


def _dec(lib, n_ctx=4, T_cap=16, d=64, eps=1e-6, dtype=1, ws=FAKE, wsb=1 << 30, k_cache=FAKE):
    return lib.dilution_attn_decode_step(FAKE, FAKE, FAKE, k_cache, FAKE, FAKE, n_ctx, T_cap, FAKE, 1, 1, d, 1.0, eps,
                                         dtype, ws, wsb, None)


def test_decode_argument_validation(lib):
    assert _dec(lib, n_ctx=16) == b.DA_ERR_INVALID          # no room for the new token
    assert _dec(lib, n_ctx=-1) == b.DA_ERR_INVALID
    assert _dec(lib, eps=0.0) == b.DA_ERR_INVALID
    assert _dec(lib, d=32) == b.DA_ERR_UNSUPPORTED
    assert _dec(lib, k_cache=None) == b.DA_ERR_INVALID
    assert _dec(lib, k_cache=MIS) == b.DA_ERR_INVALID
    assert _dec(lib, wsb=16) == b.DA_ERR_WORKSPACE


def test_noalloc_decode_checks_arguments_before_its_scratch_size(lib):
    # a call that is both malformed and too large for the fixed scratch array
    # reports the malformed argument; a well-formed oversize call reports the
    # size (both before any CUDA call)
    big = 1 << 17   # 8 x 12 heads of 131072 keys need ~50 MB of scratch

    def call(n_ctx=4, T_cap=big, dtype=1, q=FAKE, d=64, eps=1e-6):
        return lib.dilution_attn_decode_step_noalloc(q, FAKE, FAKE, FAKE, FAKE, FAKE, n_ctx, T_cap, FAKE, 8, 12, d,
                                                     1.0, eps, dtype, None)

    assert call(dtype=7) == b.DA_ERR_INVALID
    assert call(n_ctx=big) == b.DA_ERR_INVALID
    assert call(q=None) == b.DA_ERR_INVALID
    assert call(q=MIS) == b.DA_ERR_INVALID
    assert call(eps=0.0) == b.DA_ERR_INVALID
    assert call(d=96) == b.DA_ERR_UNSUPPORTED
    assert call() == b.DA_ERR_WORKSPACE


def test_get_error_rejects_null(lib):
    assert lib.dilution_attn_get_error(None, None) == b.DA_ERR_INVALID


def test_bwd_argument_validation(lib):
    def bwd(eps=1e-6, d=64, q=FAKE, ws=FAKE, wsb=1 << 30):
        return lib.dilution_attn_bwd(q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 32, d, 1.0, eps, 1, ws, wsb, None)
    assert bwd(eps=0.0) == b.DA_ERR_INVALID
    assert bwd(d=96) == b.DA_ERR_UNSUPPORTED
    assert bwd(d=128, ws=None) == b.DA_ERR_WORKSPACE
    assert bwd(q=None) == b.DA_ERR_INVALID
    assert bwd(ws=None) == b.DA_ERR_WORKSPACE
    assert b.dilution_attn_bwd_workspace_size(4, 12, 16384, 64, 1) > 4 * 12 * 16384 * 64 * 4


def test_ex_option_validation(lib):
    # flags other than DA_FLAG_EARLIER_DEMAND_ONLY and a tau_bh that is not
    # 4-byte aligned are argument errors; valid options pass on to the
    # workspace check (the first check that would need a real buffer)
    MIS2 = ctypes.c_void_p(0x10002)
    EARLY = b.DA_FLAG_EARLIER_DEMAND_ONLY

    def fwd(tau_bh=None, flags=0, ws=None):
        return lib.dilution_attn_fwd_ex(FAKE, FAKE, FAKE, FAKE, None, None, None, 1, 2, 8, 64, 1.0, tau_bh, 1e-6,
                                        flags, 1, ws, 1 << 30, None, None)

    def bwd(tau_bh=None, flags=0):
        return lib.dilution_attn_bwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 8, 64, 1.0, tau_bh,
                                        1e-6, flags, 1, None, 1 << 30, None)

    def dec(tau_bh=None, flags=0):
        return lib.dilution_attn_decode_step_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 3, 16, FAKE, 1, 2, 64, 1.0,
                                                tau_bh, 1e-6, flags, 1, None, 1 << 30, None)

    for call in (fwd, bwd, dec):
        assert call(flags=4) == b.DA_ERR_INVALID
        assert call(flags=-1) == b.DA_ERR_INVALID
        assert call(tau_bh=MIS2) == b.DA_ERR_INVALID
        assert call(flags=EARLY) == b.DA_ERR_WORKSPACE
        assert call(tau_bh=MIS, flags=EARLY) == b.DA_ERR_WORKSPACE   # 4-byte aligned is enough
    assert fwd(flags=EARLY, ws=MIS) == b.DA_ERR_INVALID              # workspace must be 256-byte aligned


def test_keep_for_backward_validation(lib):
    # the forward-state flag: bf16 only, and the forward then needs a
    # backward-sized workspace; a decode step rejects it
    KEEP = b.DA_FLAG_KEEP_FOR_BACKWARD

    def fwd(dtype=1, wsb=1 << 40, ws=FAKE):
        return lib.dilution_attn_fwd_ex(FAKE, FAKE, FAKE, FAKE, None, None, None, 1, 2, 1000, 64, 1.0, None, 1e-6,
                                        KEEP, dtype, ws, wsb, None, None)

    assert fwd(dtype=0) == b.DA_ERR_UNSUPPORTED
    need_bwd = b.dilution_attn_bwd_workspace_size(1, 2, 1000, 64, 1)
    need_fwd = b.dilution_attn_fwd_workspace_size(1, 2, 1000, 64, 1)
    assert need_bwd > need_fwd
    assert fwd(wsb=need_fwd) == b.DA_ERR_WORKSPACE
    assert fwd(ws=None) == b.DA_ERR_WORKSPACE
    assert lib.dilution_attn_bwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 8, 64, 1.0, None, 1e-6,
                                    KEEP, 0, FAKE, 1 << 30, None) == b.DA_ERR_UNSUPPORTED
    assert lib.dilution_attn_decode_step_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 3, 16, FAKE, 1, 2, 64, 1.0, None,
                                            1e-6, KEEP, 1, FAKE, 1 << 30, None) == b.DA_ERR_INVALID


def test_header_is_plain_c(lib, tmp_path):
    """The public header is a C ABI: it compiles as C99 (and C++) on its own,
    with no CUDA or PyTorch types, and a C program links against the library's
    exported version symbol."""
    import os
    import shutil
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cc = shutil.which("gcc")
    if cc is None:
        pytest.skip("gcc not available")
    hdr = os.path.join(root, "include", "dilution_attn.h")
    src = tmp_path / "use.c"
    src.write_text('#include "%s"\nint main(void) { return dilution_attn_version() > 0 ? 0 : 1; }\n' % hdr)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-c", str(src), "-o", str(tmp_path / "use.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    lib = b.lib_path()
    r = subprocess.run([cc, str(tmp_path / "use.o"), lib, "-o", str(tmp_path / "use"),
                        "-Wl,-rpath," + os.path.dirname(lib)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    if shutil.which("g++"):
        r = subprocess.run(["g++", "-std=c++17", "-Wall", "-Werror", "-x", "c++", "-c", str(src), "-o",
                            str(tmp_path / "use_cpp.o")], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
