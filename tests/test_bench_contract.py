"""The benchmark's evidence links and launch rules, checked on the CPU:
profiles/traffic.json parses, names workloads the benchmark knows, and holds
DRAM traffic for the headline workload (the default `python bench.py` line)
taken on the current kernel source, so that the JSON line's roofline.traffic
is not null (a kernel change needs a fresh 1-pass ncu capture to pass); and
--gpus is either honoured or refused, never silently ignored."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def test_traffic_record_parses_and_names_known_workloads():
    from safetensors_materialization_gb300 import synth
    import bench
    names = {f().name for f in synth.WORKLOADS.values()}
    with open(bench.TRAFFIC) as f:
        rec = json.load(f)
    assert set(rec) >= {"command", "workloads"}
    assert len(rec["workloads"]) >= 8
    for w, r in rec["workloads"].items():
        assert w in names, w
        assert set(r) == {"kernel_sha256", "traffic_per_launch"}, w
        assert isinstance(r["traffic_per_launch"], int) and r["traffic_per_launch"] > 0, w


def test_headline_workload_has_traffic_for_the_current_kernel():
    import bench
    from safetensors_materialization_gb300 import synth
    assert bench.HEADLINE == "scaled_fp8"
    assert bench.parse_args([]).workload == bench.HEADLINE
    headline = synth.WORKLOADS[bench.HEADLINE]().name
    assert bench.profiled_traffic(headline) is not None, \
        "st_kernels.cu changed since the last ncu capture: re-take the 1-pass DRAM bytes into profiles/traffic.json"


def test_config_rows_cover_every_configuration():
    import bench
    from safetensors_materialization_gb300 import synth
    rows = {bench.HEADLINE, *bench.CONFIG_ROWS}
    assert {"tiny", "unet", "scaled_fp8", "llm8b", "llm8b_f16", "stress"} <= rows
    assert all(r in synth.WORKLOADS for r in rows)


def test_gpus_flag_is_honoured_or_refused(monkeypatch):
    import bench
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    assert bench.launch_command(bench.parse_args([]), 1, []) is None
    # more GPUs than this machine has: a clear refusal, not a one-GPU run
    import torch
    have = torch.cuda.device_count() if torch.cuda.is_available() else 0
    n = str(max(2, have + 1))
    with pytest.raises(SystemExit, match="needs"):
        bench.launch_command(bench.parse_args(["--gpus", n]), 1, ["--gpus", n])
    # the reference arm runs on the host: it is re-launched under torchrun
    cmd = bench.launch_command(bench.parse_args(["--impl", "reference", "--gpus", "2"]), 1,
                               ["--impl", "reference", "--gpus", "2"])
    assert cmd[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"] and "--nproc-per-node=2" in cmd
    # under torchrun, --gpus must match WORLD_SIZE
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.launch_command(bench.parse_args(["--gpus", "2"]), 2, []) is None
    with pytest.raises(SystemExit, match="WORLD_SIZE"):
        bench.launch_command(bench.parse_args(["--gpus", "4"]), 2, [])


def test_traffic_key_ignores_comments_only():
    """A traffic record stays valid across comment edits and is voided by any
    code edit."""
    import bench
    src = 'int f(int a) { // add one\n  return a + 1; /* "x" */ }\nconst char *s = "a // b";\n'
    assert bench.kernel_code(src) == 'int f(int a) { return a + 1; } const char *s = "a // b";'
    assert bench.kernel_code(src.replace("add one", "plus 1")) == bench.kernel_code(src)
    assert bench.kernel_code(src.replace("a + 1", "a + 2")) != bench.kernel_code(src)
    assert bench.kernel_code(src.replace('"a // b"', '"a // c"')) != bench.kernel_code(src)
