"""CPU checks of the benchmark's bookkeeping: the committed ncu summaries under profiles/
are text, give the command that made them (ncu always with --clock-control none), and
their per-launch DRAM traffic lines name a known workload with a source hash the
benchmark can match."""
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
