"""Host-side pieces of bench.py that decide what its JSON line may claim:
the ncu traffic figure is reported only while the GEMM sources still hash
to the values recorded beside it; the clock summary flags throttle reasons;
the algorithmic flop and byte counts match their closed forms; the roofline
of each call picks the larger of its compute and memory times.  CPU only."""
import shutil
import tempfile
from pathlib import Path

import pytest

import bench


def _tree(tmp: Path, value=123456789):
    """A repository tree with the GEMM sources and a traffic record whose
    hashes are those of the copied sources."""
    import hashlib
    (tmp / "profiles").mkdir()
    csrc = tmp / "moe_expert_layer_topk_gb300" / "csrc"
    csrc.mkdir(parents=True)
    lines = ["# record", "", f"traffic_bytes_per_launch: {value}"]
    for name in ("gemm_tc.cu", "tc_common.cuh"):
        shutil.copy(bench.ROOT / "moe_expert_layer_topk_gb300" / "csrc" / name, csrc / name)
        lines.append(f"source_sha256 {name}: {hashlib.sha256((csrc / name).read_bytes()).hexdigest()}")
    for call, fname in bench.TRAFFIC_PROFILES.items():
        (tmp / "profiles" / fname).write_text("\n".join(lines) + "\n")
    return csrc


def test_recorded_traffic_follows_the_sources(tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    for call in bench.TRAFFIC_PROFILES:
        assert bench.recorded_traffic(call) == 123456789
    assert bench.recorded_traffic("combine") is None  # no record for that call
    with open(csrc / "gemm_tc.cu", "a") as f:
        f.write("\n// changed\n")
    for call in bench.TRAFFIC_PROFILES:
        assert bench.recorded_traffic(call) is None


def test_recorded_traffic_of_this_tree():
    for call, fname in bench.TRAFFIC_PROFILES.items():
        v = bench.recorded_traffic(call)
        prof = bench.ROOT / "profiles" / fname
        if v is not None:
            assert f"traffic_bytes_per_launch: {v}" in prof.read_text()


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


def test_call_costs_closed_forms():
    """At T=8192, H=2048, I=768, E=128, k=8: the four GEMM halves of the
    backward add up to twice the forward GEMM flops; dW_gate/up writes
    1.61 GB of fp32 and reads dgu and x_perm (2.08 GB in all); dispatch
    reads x once and writes 8 rows per token."""
    c = bench.call_costs(8192, 2048, 768, 128, 8)
    fwd, bwd = bench.layer_flops(8192, 2048, 768, 128, 8)
    assert c["down_bwd_dx"]["flops"] + c["down_bwd_dw"]["flops"] == bwd["down_bwd"]
    assert c["gate_up_bwd_dx"]["flops"] + c["gate_up_bwd_dw"]["flops"] == bwd["gate_up_bwd"]
    assert c["gate_up"]["flops"] == fwd["gate_up"] and c["route"]["flops"] == fwd["router"]
    R = 8192 * 8
    assert c["gate_up_bwd_dw"]["bytes"] == 2 * 128 * 768 * 2048 * 4 + R * 1536 * 2 + R * 2048 * 2
    assert abs(c["gate_up_bwd_dw"]["bytes"] / 1e9 - 2.08) < 0.01
    assert c["dispatch"]["bytes"] == 8192 * 2048 * 2 + R * 2048 * 2 + 3 * R * 4


def test_rooflines_pick_the_bound():
    pk = {"hbm_gbs": 1000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1000.0}
    costs = {"a": {"flops": 2e12, "bytes": 1e9}, "b": {"flops": 1e9, "bytes": 4e9},
             "r": {"flops": 2e12, "bytes": 1e6, "pipe": "fma"}}
    r = bench.rooflines({"a": 4.0, "b": 8.0, "r": 100.0}, costs, pk, fma_tfma=20.0)   # ms
    assert r["a"]["bound"] == "tensor" and abs(r["a"]["frac"] - 0.5) < 1e-9    # 2 ms at peak of 4
    assert r["a"]["unit"] == "TFLOP/s" and abs(r["a"]["achieved"] - 500.0) < 1e-6
    assert r["b"]["bound"] == "hbm" and abs(r["b"]["frac"] - 0.5) < 1e-9       # 4 ms of 8
    assert r["r"]["bound"] == "alu" and abs(r["r"]["frac"] - 0.5) < 1e-9       # 1e12 FMA at 20 T/s: 50 of 100 ms


def test_host_cpu():
    h = bench.host_cpu()
    assert h["nproc"] >= 1 and isinstance(h["model"], str) and h["model"]
