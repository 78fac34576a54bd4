"""The benchmark's evidence links, checked on the CPU: every `bench:` hook in
profiles/*.md parses, names a workload the benchmark knows, and the headline
workload (the default `python bench.py` line) has DRAM traffic recorded for
the current kernel source, so the JSON line's roofline.traffic is not null.
A kernel change needs a fresh 1-pass ncu capture (profiles/) to pass."""
import glob
import json
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def hooks():
    out = []
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path) as f:
            for line in f:
                if line.startswith("<!-- bench:"):
                    out.append((os.path.basename(path), json.loads(line[len("<!-- bench:"):].rsplit("-->", 1)[0])))
    return out


def test_profile_hooks_parse_and_name_known_workloads():
    from safetensors_materialization_gb300 import synth
    names = {f().name for f in synth.WORKLOADS.values()}
    hs = hooks()
    assert len(hs) >= 8
    for path, h in hs:
        assert set(h) == {"workload", "kernel_sha256", "traffic_per_launch"}, path
        assert h["workload"] in names, (path, h["workload"])
        assert isinstance(h["traffic_per_launch"], int) and h["traffic_per_launch"] > 0, path


def test_headline_workload_has_traffic_for_the_current_kernel():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from safetensors_materialization_gb300 import synth
    headline = synth.WORKLOADS["unet"]().name
    assert bench.profiled_traffic(headline) is not None, \
        "st_kernels.cu changed since the last ncu capture: re-take the 1-pass DRAM bytes into profiles/"
