"""Host-side parts of bench.py (no GPU): the clock sampler's parsing of
nvidia-smi output, the flop and byte accounting of the metric, and the rule
that a committed ncu traffic figure is reported only for the kernel sources
it was measured on."""
import os
import shutil
import stat
import time
import types

import pytest
import torch

import bench


def _fake_smi(tmp_path, lines):
    d = tmp_path / "bin"
    d.mkdir()
    script = d / "nvidia-smi"
    body = "".join(f"echo '{ln}'\n" for ln in lines)
    script.write_text("#!/bin/bash\n" + body + "exec sleep 30\n")
    script.chmod(script.stat().st_mode | stat.S_IXUSR)
    return str(d)


def test_clock_sampler_parses_clocks_and_throttle_reasons(tmp_path, monkeypatch):
    lines = ["0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Active",
             "0, 1980, 2070, 1000.0, 0x4, Not Active, Not Active, Not Active, Active",
             "0, 2070, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "garbage line"]
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, lines) + os.pathsep + os.environ["PATH"])
    s = bench.ClockSampler(0)
    s.start()
    deadline = time.monotonic() + 10
    while time.monotonic() < deadline and open(s.path).read().count("\n") < len(lines):
        time.sleep(0.05)
    path = s.path
    got = s.stop()
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert not os.path.exists(path)


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))
    s = bench.ClockSampler(0)
    s.start()
    got = s.stop()
    assert got["sm_mhz"] is None and got["reasons"] == ["nvidia-smi unavailable"]


@pytest.mark.parametrize("fp8,rope_bf16,per_tok", [(False, False, 1152), (True, False, 596), (True, True, 656)])
def test_work_counts_visible_keys_and_cache_bytes(fp8, rope_bf16, per_tok):
    # seqlens 3, 0, 70 with s_q = 2: rows see 2+3, 0+0 and 69+70 keys
    inp = types.SimpleNamespace(seqlens=torch.tensor([3, 0, 70], dtype=torch.int32), s_q=2, heads=4,
                                kv_fp8=fp8, rope_bf16=rope_bf16)
    flops, kv_bytes = bench.work_of(inp)
    assert flops == 4 * (5 + 0 + 139) * (2 * 576 + 2 * 512)
    assert kv_bytes == (3 + 0 + 70) * per_tok


def test_traffic_is_withheld_when_the_kernel_sources_change(tmp_path, monkeypatch):
    root = tmp_path / "repo"
    for f in bench.KERNEL_SOURCES + (bench.NCU_SUMMARY["decode"],):
        (root / f).parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, f), root / f)
    monkeypatch.setattr(bench, "ROOT", str(root))
    first = bench.measured_traffic("decode")
    assert first is None or first > 0
    assert bench.measured_traffic("mtp") is None            # no summary for that workload
    with open(root / bench.KERNEL_SOURCES[0], "a") as fh:  # any edit of a kernel source
        fh.write("\n")
    assert bench.measured_traffic("decode") is None
