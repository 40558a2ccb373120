"""CPU checks of the benchmark's bookkeeping: the committed ncu summaries under profiles/
are text, give the command that made them (ncu always with --clock-control none), and
their per-launch DRAM traffic lines name a known workload with a source hash the
benchmark can match; the oracle's per-layer wall-time estimates scale a bounded sample
to the whole layer, take the transposed oracle for a transposed layer, and report a
failure instead of raising."""
import importlib.util
import os
import re

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_profiles_are_text_with_their_commands():
    pdir = os.path.join(ROOT, "profiles")
    names = sorted(os.listdir(pdir))
    assert names, "no ncu summaries committed"
    for name in names:
        assert name.endswith((".md", ".txt")), name
        text = open(os.path.join(pdir, name)).read()
        assert len(text) < 16384, name  # a short summary, not a raw report
        ncu_lines = [ln for ln in text.splitlines() if re.search(r"(^|\s)ncu\s", ln)]
        assert ncu_lines, "%s gives no ncu command" % name
        for ln in ncu_lines:
            assert "--clock-control none" in ln, (name, ln)


def test_traffic_lines_name_known_workloads():
    bench = _bench()
    traffic = bench.load_traffic()
    assert {"body", "dw"} <= set(traffic), sorted(traffic)
    for key, (nbytes, digest) in traffic.items():
        assert key in bench.KERNEL_SOURCES, key
        assert nbytes > 0
        assert re.fullmatch(r"[0-9a-f]{12}", digest), (key, digest)
        assert len(bench.kernel_source_hash(key)) == 12


def test_both_arms_report_one_metric():
    bench = _bench()
    src = open(os.path.join(ROOT, "bench.py")).read()
    assert src.count('"metric": METRIC') == 2  # the GPU arm and the reference arm
    assert "TFLOP/s" in bench.METRIC


def test_oracle_beside_layers_scales_samples_and_skips_composites():
    bench = _bench()
    gpu_ms = {"tiny_f32": 0.01, "upsample": 0.05, "block": 0.1}
    out = bench.oracle_beside_layers(gpu_ms, seconds=0.05)
    assert set(out) == {"tiny_f32", "upsample"}  # the two-kernel block has no single oracle call
    for key, est in out.items():
        assert "error" not in est, est  # the transposed layer goes through its own oracle
        assert est["full_layer_s"] > 0 and est["tflops"] > 0 and est["cores"] >= 1
        assert abs(est["gpu_speedup"] - est["full_layer_s"] / (gpu_ms[key] * 1e-3)) < 1e-9 * est["gpu_speedup"]
    s = bench.WORKLOADS["tiny_f32"].shape
    assert "scaled to the layer's %d outputs" % (s.pixels * s.C_out) in out["tiny_f32"]["sample"]


def test_oracle_beside_layers_reports_a_failure_without_raising():
    bench = _bench()

    class Broken:
        def full_layer(self, seconds):
            raise RuntimeError("no oracle here")

    out = bench.oracle_beside_layers({"stem": 0.02}, samplers={"stem": Broken()})
    assert out == {"stem": {"error": "RuntimeError: no oracle here"}}
