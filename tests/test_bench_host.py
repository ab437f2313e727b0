"""Host-side logic of bench.py on the CPU: the clock record that decides
whether a timed run is kept (throttle reasons, median SM clock under load)
and the algorithmic bytes / FLOPs the roofline divides by."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def _sampler(lines):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc, s.lines = None, lines
    return s


def _line(sm, hw="Not Active", hw_th="Not Active", sw_th="Not Active", cap="Not Active"):
    # index, clocks.sm, clocks.max.sm, power.draw, reasons.active, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
    return f"0, {sm}, 2070, 900.5, 0x0000000000000000, {hw}, {hw_th}, {sw_th}, {cap}"


def test_clock_summary_median_under_load_and_no_reasons():
    s = _sampler([_line(345), _line(1980), _line(1965), _line(2010), _line(400)]).summary()
    assert s["sm_max_mhz"] == 2070.0
    assert s["sm_mhz"] == 1980.0  # idle samples (below half the maximum) are left out
    assert s["reasons"] == [] and s["samples"] == 5


def test_clock_summary_reports_every_active_throttle_reason():
    lines = [_line(1900), _line(1500, cap="Active"), _line(1400, hw_th="Active"), _line(1800, sw_th="Active"),
             _line(1850, hw="Active")]
    s = _sampler(lines).summary()
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap", "sw_thermal_slowdown"]


def test_clock_summary_skips_malformed_lines_and_handles_no_samples():
    s = _sampler(["", "[N/A], [N/A]", "0, [N/A], 2070, 1, 0x0, Not Active, Not Active, Not Active, Not Active"])
    out = s.summary()
    assert out["sm_mhz"] is None and out["samples"] == 0


def test_algorithmic_bytes_match_the_stated_weight_sizes():
    # every expert active: w13 + w2 codes are 3*H*I bytes per expert (one byte per code)
    cfg = synth.config("oss20b_decode")
    counts = np.full(cfg.E, cfg.T * cfg.top_k // cfg.E)
    a = bench.algorithmic(cfg, counts)
    H, I, E, R = cfg.H, cfg.I, cfg.E, cfg.T * cfg.top_k
    hb = ib = -(-2880 // 128)
    codes = E * 3 * H * I
    assert codes == pytest.approx(0.796e9, rel=1e-3)  # 32 experts x 3 x 2880^2 bytes
    scales = E * 4 * (2 * ib * hb + hb * ib)
    biases = E * 2 * (2 * I + H)
    assert a["step_bytes"] == codes + scales + biases + E * H * 2 + E * 2 + 2 * cfg.T * H * 2
    assert a["gemm1_flops"] == 2 * R * 2 * I * H and a["gemm2_flops"] == 2 * R * H * I
    assert a["active"] == E


def test_algorithmic_counts_only_active_experts_and_halves_fp4_codes():
    cfg = synth.config("oss120b_decode")
    counts = np.zeros(cfg.E, np.int64)
    counts[:10] = cfg.T * cfg.top_k // 10
    a8 = bench.algorithmic(cfg, counts, mx=True)
    a4 = bench.algorithmic(cfg, counts, mx=True, fp4=True)
    assert a8["active"] == a4["active"] == 10
    H, I = cfg.H, cfg.I
    # the MXFP4 weights carry half a byte per code, the same scale bytes and biases
    assert (a8["gemm1_bytes"] - a4["gemm1_bytes"]) == 10 * H * I  # 2*I*H codes at 1/2 byte saved
    assert (a8["gemm2_bytes"] - a4["gemm2_bytes"]) == 10 * H * I // 2


def test_prefill_flops_of_the_stated_workloads():
    cfg = synth.config("oss120b_prefill")
    a = bench.algorithmic(cfg, np.full(cfg.E, cfg.T * cfg.top_k // cfg.E))
    assert a["gemm1_flops"] + a["gemm2_flops"] == pytest.approx(1.631e12, rel=1e-3)
    cfg = synth.config("qwen235b_prefill")
    a = bench.algorithmic(cfg, np.full(cfg.E, cfg.T * cfg.top_k // cfg.E))
    assert a["gemm1_flops"] + a["gemm2_flops"] == pytest.approx(4.948e12, rel=1e-3)


def test_flush_writes_one_buffer_and_reads_the_other():
    import torch
    w = torch.zeros(1 << 12, dtype=torch.uint8)
    r = torch.zeros(1 << 9, dtype=torch.int64)
    bench.flush_l2(w, r, 0x1A5)
    assert int(w.min()) == int(w.max()) == 0xA5  # the step index's low byte, every byte written
    assert int(r.abs().sum()) == 0  # the read buffer is only read


def test_baseline_sample_includes_the_extreme_experts():
    rng = np.random.default_rng(3)
    idx = rng.integers(0, 8, (200, 2))
    idx[:, 1] = np.where(idx[:, 1] == idx[:, 0], (idx[:, 0] + 1) % 8, idx[:, 1])  # two distinct experts per token
    counts = np.bincount(idx.ravel(), minlength=8)
    nz = np.nonzero(counts)[0]
    most, least = nz[np.argmax(counts[nz])], nz[np.argmin(counts[nz])]
    tokens, desc = bench.sample_for_baseline(idx, 8, 40)
    assert len(tokens) == 40 and np.all(np.diff(tokens) > 0)
    for e in (most, least):
        assert (idx[tokens] == e).any(), e
    assert f"expert {least}" in desc and f"expert {most}" in desc
    all_tokens, _ = bench.sample_for_baseline(idx, 8, 10 ** 6)  # a budget above the batch takes all of it
    assert np.array_equal(all_tokens, np.arange(200))
