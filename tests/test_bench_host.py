"""Host-side arithmetic of the benchmark, checked on the CPU.

The reported numbers are algorithmic work divided by measured time, so the
work formulas, the special-function-unit peak and the rule that a committed
DRAM-traffic figure is used only while the kernel source is unchanged are
pinned here against values worked out by hand.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_forward_work_counts_three_contractions_over_causal_pairs():
    # 4 x 12 heads of T = 16384, d = 64: causal pairs 16384 * 16385 / 2 per head,
    # 2 d FLOP per pair per contraction, three contractions
    pairs = 16384 * 16385 // 2 * 48
    assert bench.fwd_flops(4, 12, 16384, 64) == 3 * 2 * 64 * pairs == 2474052157440
    assert bench.sweep_flops(4, 12, 16384, 64) * 3 == bench.fwd_flops(4, 12, 16384, 64) * 2
    assert bench.fwd_flops(1, 1, 1, 64) == 3 * 2 * 64   # one query, one pair


def test_backward_work_is_five_contractions():
    assert bench.bwd_flops(4, 12, 16384, 64) * 3 == bench.fwd_flops(4, 12, 16384, 64) * 5


def test_sfu_peak_and_fractions():
    # 32 results per SM per clock x 152 SMs x 2070 MHz = 10.06848 T/s
    r = bench.sfu_report(1, 1, 3, {"rowstats": 1.0, "sweep": 2.0}, 152, 2070.0)
    assert abs(r["peak"] - 10.06848) < 1e-9
    pairs = 6   # T = 3: 3 * 4 / 2
    assert abs(r["rowstats"]["achieved"] - 1.0 * pairs / 1e-3 / 1e12) < 1e-18
    assert abs(r["sweep"]["achieved"] - 1.5 * pairs / 2e-3 / 1e12) < 1e-18
    assert abs(r["achieved"] - 2.5 * pairs / 3e-3 / 1e12) < 1e-18
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-15


def test_traffic_figure_only_for_the_profiled_source(tmp_path):
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    rel = os.path.relpath(src, bench.ROOT)
    prof = tmp_path / "p.md"
    prof.write_text("kernel_source_hash: `%s`\n\ntraffic_bytes_per_launch_full_size: `12345`\n"
                    % bench.sources_hash([rel]))
    assert bench.profiled_traffic(str(prof), [rel]) == 12345.0
    src.write_text("kernel v2\n")          # the kernel changed since the capture
    assert bench.profiled_traffic(str(prof), [rel]) is None
    assert bench.profiled_traffic(str(tmp_path / "missing.md"), [rel]) is None


def test_traffic_figure_only_for_the_profiled_workload(tmp_path):
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    rel = os.path.relpath(src, bench.ROOT)
    prof = tmp_path / "p.md"
    prof.write_text("kernel_source_hash: `%s`\nprofile_workload: `fwd_x B=4 H=12 T=16384 d=64`\n\n"
                    "traffic_bytes_per_launch_full_size: `12345`\n" % bench.sources_hash([rel]))
    assert bench.profiled_traffic(str(prof), [rel], "fwd_x B=4 H=12 T=16384 d=64") == 12345.0
    assert bench.profiled_traffic(str(prof), [rel], "fwd_x B=2 H=12 T=16384 d=64") is None   # another batch
    assert bench.profiled_traffic(str(prof), [rel], "fwd_y B=4 H=12 T=16384 d=128") is None



def test_cpu_baseline_reports_parity_of_a_gpu_forward(monkeypatch):
    # the CPU-baseline leg compares a forward on its own sample with the
    # oracle's output there (the oracle replaced here by a fast stand-in that
    # returns zeros): a forward that returns the same passes, one that is off
    # by 0.05 somewhere fails, none gives no parity entry
    import numpy as np
    monkeypatch.setattr(bench, "oracle_sample", lambda q, k, v, rows: (1, 1.0, np.zeros((rows, q.shape[1]))))

    def same(q, k, v):
        return np.zeros(tuple(q.shape))

    def off(q, k, v):
        o = same(q, k, v)
        o[0, 1, 7, 3] += 0.05
        return o

    base, par = bench.cpu_baseline(2, gpu_forward=same)
    assert base["kind"] == "oracle" and par["ok"] and par["max_abs_err_out"] == 0.0 and par["heads"] == 2
    _, par = bench.cpu_baseline(2, gpu_forward=off)
    assert not par["ok"] and abs(par["max_abs_err_out"] - 0.05) < 1e-12
    assert bench.cpu_baseline(2)[1] is None
