"""Host logic of bench.py (no GPU): algorithmic bytes per expert, the tensor-peak ratios, the
rule that ties a recorded DRAM-traffic figure to the kernel sources it was captured on, and the
parsing of the nvidia-smi clock record taken during the timed region."""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_per_expert_bytes(bench):
    H, I = 2048, 768
    # (gate/up, down) packed bytes of one expert: codes + scales (+ global scale for NVFP4)
    assert bench.per_expert_bytes("fp8", H, I) == (2 * I * H + (2 * I // 128) * (H // 128) * 4,
                                                   H * I + (H // 128) * (I // 128) * 4)
    assert bench.per_expert_bytes("fp8_w8a8", H, I) == bench.per_expert_bytes("fp8", H, I)
    assert sum(bench.per_expert_bytes("fp8", H, I)) == 4_719_744
    assert sum(bench.per_expert_bytes("int4", H, I)) == 2_433_024
    assert sum(bench.per_expert_bytes("nvfp4_w4a16", H, I)) == 2_654_216
    assert sum(bench.per_expert_bytes("bf16", H, I)) == 3 * H * I * 2  # [2I, H] + [H, I] bf16


def test_tensor_peak_ratios(bench):
    # nominal dense rates relative to bf16: FP4 13.5 / 2.25, FP8 4.5 / 2.25; bf16-operand paths 1
    assert bench.TENSOR_RATIO["nvfp4_w4a4"] == pytest.approx(6.0)
    assert bench.TENSOR_RATIO["fp8_w8a8"] == pytest.approx(2.0)
    for f in ("fp8", "int4", "nvfp4_w4a16", "bf16"):
        assert bench.TENSOR_RATIO[f] == 1.0
    assert set(bench.TENSOR_RATIO) == set(bench.FMT_ID)


def test_recorded_traffic_needs_the_captured_sources(bench, tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    digest = bench.source_digest(["k.cu"])
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# format tokens bytes sources digest\n"
        f"nvfp4_w4a4 16384 550128384 k.cu {digest}\n"
        "fp8 16 1000 missing.cu 0123456789abcdef\n")
    assert bench.recorded_traffic("nvfp4_w4a4", 16384) == 550128384.0
    assert bench.recorded_traffic("nvfp4_w4a4", 4096) is None  # another workload
    assert bench.recorded_traffic("fp8", 16) is None            # its source is gone
    src.write_text("kernel v2\n")                              # the kernel changed since the capture
    assert bench.recorded_traffic("nvfp4_w4a4", 16384) is None


class _Done:
    def terminate(self):
        pass

    def wait(self):
        return 0


def _clocks_from(bench, rows, monkeypatch):
    monkeypatch.setattr(bench.time, "sleep", lambda s: None)
    c = bench.Clocks(0)
    c.proc = _Done()
    c.file.write("".join(rows))
    c.file.flush()
    return c.stop()


def test_clock_record_median_and_reasons(bench, monkeypatch):
    row = "0, {sm}, 2070, 1100.5, 0x{a}, {hw}, Not Active, Not Active, {pc}\n"
    rows = [row.format(sm=s, a="00", hw="Not Active", pc="Not Active") for s in (2070, 2055, 2070)]
    rows.append(row.format(sm=1980, a="04", hw="Not Active", pc="Active"))
    rows.append("garbled line\n")
    r = _clocks_from(bench, rows, monkeypatch)
    assert r["sm_mhz"] == 2062.5 and r["sm_max_mhz"] == 2070.0 and r["samples"] == 4
    assert r["reasons"] == ["sw_power_cap"]
    r = _clocks_from(bench, [row.format(sm=1500, a="08", hw="Active", pc="Not Active")], monkeypatch)
    assert r["reasons"] == ["hw_slowdown"]


def test_clock_record_without_samples(bench, monkeypatch):
    assert _clocks_from(bench, [], monkeypatch)["reasons"] == ["no samples"]
    c = bench.Clocks(0)
    c.proc = None  # nvidia-smi could not be started
    assert c.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_reference_arm_runs_the_w8a8_workload():
    """`bench.py --impl reference --config 8` times the oracle's W8A8 layer on a bounded sample and
    prints one JSON line naming that workload."""
    import json
    import subprocess
    import sys

    env = dict(os.environ)
    env.pop("CUDA_VISIBLE_DEVICES", None)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "8",
                        "--layers", "1", "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                       timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["config"]["format"] == "fp8_w8a8" and line["cpu_baseline"]["kind"] == "oracle"
