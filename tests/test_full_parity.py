"""Full-size parity: every element of every output of the large workloads
against the oracle, 0 ULP, in the launch configuration the benchmark times.

The workloads are the UNet-shaped F16 checkpoint (716 tensors, 2.67 GB, rename
view, BF16 out), the scaled-FP8 checkpoint (57 blocks, 570 E4M3 weights with
per-tensor F32 scales, 11.8 GB in, 23.7 GB BF16 out) and the 8B-LLM-shaped
BF16 checkpoint (4 shard files joined into one arena, 16.06 GB, one launch)
copied to BF16 and cast to F16.  Each is materialized by the planner's own
choice of kernel build (what the benchmark runs) and, where it differs, by the
TMA build, each into a guard-banded arena; one pass of the oracle on every
host core (tests/oracle_compare.py) then checks every byte of both.  After the
launches the guard bytes must be untouched and the device data section equal
to its host copy.

Source: "Disk tier safetensors streaming design audit (ComfyUI)", "Tests and
docs" (metadata correctness, single-tensor loading, load behaviour) and the
scaled-FP8 conversion of "ComfyUI load path + eager materialization sites".
"""
import numpy as np
import pytest

from oracle_compare import GuardedOutputs, assert_device_equals_host, compare_full

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def materialize_builds(stmat, ix, data_ptr, dst, kernels, **sel):
    """{label: GuardedOutputs} of one launch per kernel build (0 = the
    planner's choice), each checked for flags and untouched guard bytes."""
    res = {}
    for k in kernels:
        plan = ix.plan(dst=dst, kernel=k, **sel)
        label = f"kernel {k} ({plan.stats()['kernel']})"
        outs = GuardedOutputs(plan)
        plan.materialize(data_ptr, outs.ptrs)
        torch.cuda.synchronize()
        assert plan.check() == 0, label
        outs.check_guards()
        res[label] = outs
        res[label].plan = plan
    return res


def single_file_case(stmat, oracle, name, kernels):
    from safetensors_materialization_gb300 import synth
    w = synth.WORKLOADS[name]()
    lay = w.files[0]
    img = synth.build_workload_file(w, 0)
    data = img[lay.data_start:]
    ix = w.view(stmat.Index.from_header(lay.header, lay.data_bytes))
    dev = torch.empty(lay.data_bytes + 256, dtype=torch.uint8, device="cuda")
    dev[:lay.data_bytes].copy_(torch.from_numpy(data))
    res = materialize_builds(stmat, ix, dev.data_ptr(), w.dst[0], kernels, scale_suffix=w.scale_suffix,
                             **w.selection(ix))
    assert_device_equals_host(dev[:lay.data_bytes], data)
    oix = w.view(oracle.parse_header(lay.header, lay.data_bytes))
    sel = oix.select(dst=w.dst[0], scale_suffix=w.scale_suffix, **w.selection(oix))
    for r in res.values():
        assert [o["name"] for o in r.plan.outputs()] == [o["name"] for o in sel.outputs()]
    n = compare_full(sel, data, res)
    assert n == sum(o["bytes"] for o in sel.outputs())
    return n


def test_full_parity_unet(stmat, oracle):
    """716 F16 tensors -> BF16 through the rename view, every element."""
    assert single_file_case(stmat, oracle, "unet", kernels=[0, 3]) == 2_668_385_920


def test_full_parity_scaled_fp8(stmat, oracle):
    """570 E4M3 weights x per-tensor F32 scale -> BF16, every element."""
    assert single_file_case(stmat, oracle, "scaled_fp8", kernels=[0, 3]) == 23_668_457_472


@pytest.fixture(scope="module")
def llm(stmat, oracle):
    """The 8B LLM checkpoint: 4 shard files, 16.06 GB, joined into one arena
    (library and oracle) and resident on the device."""
    from safetensors_materialization_gb300 import synth
    w = synth.llm8b()
    ix, bases = stmat.Index.concat([stmat.Index.from_header(l.header, l.data_bytes) for l in w.files])
    oix, obases = oracle.concat([oracle.parse_header(l.header, l.data_bytes) for l in w.files])
    assert bases == obases
    arena = np.zeros(ix.sizes()[1], np.uint8)
    for k, lay in enumerate(w.files):
        synth.build_workload_data(w, k, arena[bases[k]:bases[k] + lay.data_bytes])
    dev = torch.from_numpy(arena).cuda()
    yield ix, oix, arena, dev
    del dev
    torch.cuda.empty_cache()


def test_full_parity_llm8b_bf16(stmat, oracle, llm):
    """BF16 -> BF16 over all 4 shards in one launch: every element equals the
    oracle's, and (a raw copy) its own source bytes."""
    ix, oix, arena, dev = llm
    res = materialize_builds(stmat, ix, dev.data_ptr(), "BF16", [0])
    (outs,) = res.values()
    for i, o in enumerate(outs.plan.outputs()):
        assert torch.equal(outs.raw(i), dev[o["begin"]:o["begin"] + o["bytes"]]), o["name"]
    sel = oix.select(dst="BF16")
    assert compare_full(sel, arena, res) == 16_060_522_496
    assert_device_equals_host(dev, arena)


def test_full_parity_llm8b_f16(stmat, oracle, llm):
    """BF16 -> F16 over all 4 shards in one launch, every element, by the
    planner's build and the TMA build."""
    ix, oix, arena, dev = llm
    res = materialize_builds(stmat, ix, dev.data_ptr(), "F16", [0, 3])
    sel = oix.select(dst="F16")
    assert compare_full(sel, arena, res) == 16_060_522_496
    assert_device_equals_host(dev, arena)
