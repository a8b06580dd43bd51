"""The benchmark's output contract, checked on the CPU: the reference arm (the float64 oracle
timed on the host cores) prints one JSON line with the metric, unit and config of the
default workload, a cpu_baseline describing that run and an e2e object with no transfers;
the config names the workload by its shape and states the launch mode."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    # (a warm-up below three is raised to three)
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    sys.path.insert(0, ROOT)
    import bench
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3 and d["data"] == "synthetic"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["vs_baseline"] is None
    assert d["config"]["workload"] == bench.WORKLOADS["pages_shape"]["desc"]
    assert d["config"]["batch"] == 32 and d["config"]["layers"] == 36 and "launch" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == "GB/s"
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0



def test_traffic_is_taken_only_for_the_kernel_source_it_was_captured_on(tmp_path):
    """roofline.traffic comes from profiles/traffic.json only when the entry's source hash is
    the hash of the decode sources as the production library compiles them: blocks that only
    the tests' library builds are left out of the hash (an #else branch is kept), every other
    change to the sources changes it."""
    sys.path.insert(0, ROOT)
    import bench
    src = (b"a\n#ifdef EKV_TEST_WAIT_TIMEOUT\nx\n#endif\n\nb\n"
           b"#ifdef EKV_TEST_WAIT_TIMEOUT\ny\n#else\nz\n#endif\nc\n")
    assert bench._production_source(src) == b"a\nb\nz\nc\n"
    assert bench._production_source(b"a\n#ifdef OTHER\nx\n#endif\n") == b"a\n#ifdef OTHER\nx\n#endif\n"
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))["decode_split_mma"]
    entry = rec["pages_shape"]
    if entry["kernel_source_hash"] == bench.kernel_source_hash():
        assert bench.profiled_traffic("pages_shape") == float(entry["traffic_bytes_per_launch"])
    else:
        assert bench.profiled_traffic("pages_shape") is None
    for name, e in rec.items():
        if e.get("kernel_source_hash") is None:
            assert bench.profiled_traffic(name) is None
