"""Host-side pieces of bench.py (CPU only): every workload describes its config
without a device, the ncu figures count only while the kernel's sources match
the summary, and the two rooflines are the arithmetic they claim."""

import json

import pytest

import bench


def test_every_workload_describes_itself():
    for name in bench._workload_table(0):
        cfg = bench.describe_workload(name)
        json.dumps(cfg)
        assert cfg["numel"] > 0 and cfg["bytes_per_param"] > 0, name
        assert "workload" in cfg and "l2" in cfg, name
        assert name in bench.CPU_SAMPLES, name


def test_ncu_figures_need_matching_sources(monkeypatch):
    assert bench.ncu_traffic("gpt2_small") is not None
    monkeypatch.setattr(bench, "kernel_source_sha", lambda workload="gpt2_small": "0" * 16)
    assert bench.ncu_traffic("gpt2_small") is None
    assert bench.ncu_figure("gpt2_small", "warp_instructions_per_element") is None
    assert bench.issue_roofline("gpt2_small", 1e11, 2070.0, sms=152) is None


def test_issue_roofline_arithmetic():
    wpe = bench.ncu_figure("q8", "warp_instructions_per_element")
    rate = (1 << 30) / 3.11e-3
    r = bench.issue_roofline("q8", rate, 2070.0, sms=152)
    assert r["bound"] == "issue" and r["unit"] == "warp-inst/s"
    assert r["peak"] == pytest.approx(152 * 4 * 2070e6)
    assert r["achieved"] == pytest.approx(wpe * rate)
    assert r["frac"] == pytest.approx(wpe * rate / (152 * 4 * 2070e6))
    assert 0.5 < r["frac"] < 1.0     # the 8-bit step runs close to its issue bound
    assert bench.issue_roofline("adam_mini_llama3", rate, 2070.0, sms=152) is None   # no summary
