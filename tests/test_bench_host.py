"""Host-side pieces of bench.py that decide what its JSON line may claim:
the ncu traffic figure is reported only while the GEMM sources still hash
to the values recorded beside it; the clock summary flags throttle reasons;
the algorithmic flop counts match the per-token closed forms.  CPU only."""
import shutil
import tempfile
from pathlib import Path

import pytest

import bench


def _profile_value(root: Path) -> int:
    for line in (root / "profiles" / "traffic_gate_up_fwd_T8192.md").read_text().splitlines():
        if line.startswith("traffic_bytes_per_launch:"):
            return int(line.split(":")[1])
    raise AssertionError("no traffic line")


def _tree(tmp: Path):
    (tmp / "profiles").mkdir()
    shutil.copy(bench.ROOT / "profiles" / "traffic_gate_up_fwd_T8192.md", tmp / "profiles")
    csrc = tmp / "moe_expert_layer_topk_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in ("gemm_tc.cu", "tc_common.cuh"):
        shutil.copy(bench.ROOT / "moe_expert_layer_topk_gb300" / "csrc" / name, csrc / name)
    return csrc


def test_recorded_traffic_follows_the_sources(tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    assert bench.recorded_traffic() == _profile_value(tmp_path)
    with open(csrc / "gemm_tc.cu", "a") as f:
        f.write("\n// changed\n")
    assert bench.recorded_traffic() is None


def test_recorded_traffic_of_this_tree():
    v = bench.recorded_traffic()
    assert v is None or v == _profile_value(bench.ROOT)


class _Running:
    def terminate(self):
        pass


def _summary(lines):
    s = bench.ClockSampler(0)
    s.proc = _Running()
    s.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
    s.f.write("\n".join(lines) + "\n")
    return s.summary()


def test_clock_summary():
    na = "Not Active"
    rows = [f"0, {mhz}, 2070, 300.0, 0x0, {na}, {na}, {na}, {cap}"
            for mhz, cap in ((2070, na), (2055, "Active"), (2070, na))]
    out = _summary(rows)
    assert out["sm_mhz"] == 2070 and out["sm_max_mhz"] == 2070 and out["samples"] == 3
    assert out["reasons"] == ["sw_power_cap"]
    hot = _summary([f"0, 1500, 2070, 900.0, 0x0, {na}, Active, {na}, {na}"])
    assert hot["reasons"] == ["hw_thermal_slowdown"] and hot["sm_mhz"] == 1500
    assert _summary([])["reasons"] == ["no samples"]


@pytest.mark.parametrize("T", [4096, 8192])
def test_layer_flops_closed_forms(T):
    """Per token at H=2048, I=768, E=128, k=8: gate/up 50.33 MFLOP, down
    25.17 MFLOP, router 0.52 MFLOP forward; the backward doubles each."""
    fwd, bwd = bench.layer_flops(T, 2048, 768, 128, 8)
    assert fwd["gate_up"] == T * 2 * 8 * 2048 * 2 * 768
    assert fwd["down"] == T * 2 * 8 * 768 * 2048
    assert fwd["router"] == T * 2 * 2048 * 128
    assert abs((fwd["gate_up"] + fwd["down"]) / T / 1e6 - 75.5) < 0.05
    assert all(bwd[k + "_bwd"] == 2 * fwd[k] for k in fwd)
