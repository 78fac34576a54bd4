"""Pins for the oracle's header parse, views, selection and materialization
(CPU only), against hand-built files with hand-computed expectations
(tests/golden/), round trips of generated files, and invariants.

The metadata-only index and the Prefix/Filter/Rename views are those of
"Disk tier safetensors streaming design audit (ComfyUI)", sections
"FastSageTensors (fastsafetensors) capability audit" and "Strategy summary
(implemented)"; the rename semantics are those of state_dict_prefix_replace
("ComfyUI load path + eager materialization sites").
"""
import numpy as np
import pytest

from conftest import golden, golden_file, small_file

CASES = golden("format_errors.json")["cases"]


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_golden_status(oracle, case):
    f = golden_file(case)
    if case["expect"] == "OK":
        ix = oracle.parse(f)
        assert len(ix) == case["count"]
        if "names" in case:
            assert [e["name"] for e in ix.entries()] == case["names"]
    else:
        with pytest.raises(oracle.OracleError) as e:
            oracle.parse(f)
        assert e.value.status == case["expect"]


def test_small_file_index(oracle):
    g, f = small_file()
    ix = oracle.parse(f)
    assert ix.header_len == len(g["header"].encode()) + g["pad"]
    assert ix.data_bytes == len(bytes.fromhex(g["data_hex"]))
    assert [e["name"] for e in ix.entries()] == g["index_order"]
    for e in ix.entries():
        want = g["entries"][e["name"]]
        assert (e["dtype"], e["shape"], e["begin"], e["end"]) == \
            (want["dtype"], want["shape"], want["begin"], want["end"])
    assert ix.metadata() == g["metadata"]


def test_small_file_views(oracle):
    g, f = small_file()
    ix = oracle.parse(f)
    assert [e["name"] for e in ix.view_prefix("c.").entries()] == g["views"]["prefix c."]
    assert [e["name"] for e in ix.view_filter(["f", "a"]).entries()] == g["views"]["filter [f, a]"]
    r = ix.view_rename([("c.", "layer.c."), ("a", "A")])
    assert [e["name"] for e in r.entries()] == g["views"]["rename [c. -> layer.c., a -> A]"]
    # a view keeps the parent's offsets
    assert r.entries()[2]["begin"] == ix.entries()[2]["begin"]


@pytest.mark.parametrize("dst", ["BF16", "F16", "F32"])
def test_small_file_materialize(oracle, dst):
    g, f = small_file()
    ix = oracle.parse(f)
    data = np.frombuffer(f, dtype=np.uint8)[8 + ix.header_len:]
    plan = ix.select(dst=dst, scale_suffix=(".weight", ".scale_weight"))
    outs = plan.outputs()
    assert [o["name"] for o in outs] == g["scaled_outputs"]
    assert outs[2]["scale"] == "c.scale_weight"
    for i, o in enumerate(outs):
        assert plan.materialize(i, data).tobytes().hex() == g["expect"][dst][o["name"]], o["name"]


def test_small_file_keep_is_raw(oracle):
    g, f = small_file()
    ix = oracle.parse(f)
    data = np.frombuffer(f, dtype=np.uint8)[8 + ix.header_len:]
    plan = ix.select(dst="KEEP")
    for i, o in enumerate(plan.outputs()):
        assert o["dtype"] == o["src_dtype"]
        np.testing.assert_array_equal(plan.materialize(i, data), data[o["begin"]:o["begin"] + o["bytes"]])
    with pytest.raises(oracle.OracleError) as e:
        ix.select(dst="KEEP", scale_suffix=(".weight", ".scale_weight"))
    assert e.value.status == "UNSUPPORTED_CAST"


def test_selection_rules(oracle):
    g, f = small_file()
    ix = oracle.parse(f)
    p = ix.select(names=["f", "a"], dst="BF16")
    assert [o["name"] for o in p.outputs()] == ["f", "a"]
    # explicit scale names; the scale tensor is consumed even if selected
    p = ix.select(names=["c.scale_weight", "c.weight"], dst="BF16", scale_names=[None, "c.scale_weight"])
    assert [o["name"] for o in p.outputs()] == ["c.weight"]
    for bad, status in [(dict(names=["nope"]), "NOT_FOUND"),
                        (dict(names=["a", "a"]), "DUP_KEY"),
                        (dict(names=["a"], scale_names=["c.scale_weight"]), "INVAL"),     # not fp8
                        (dict(names=["c.weight"], scale_names=["a"]), "INVAL"),           # not 1-elem
                        (dict(names=["c.weight"], scale_names=["nope"]), "NOT_FOUND"),
                        (dict(dst="I32"), "UNSUPPORTED_CAST")]:
        with pytest.raises(oracle.OracleError) as e:
            ix.select(**{"dst": "BF16", **bad})
        assert e.value.status == status, bad


def test_rename_collision(oracle):
    g, f = small_file()
    ix = oracle.parse(f)
    with pytest.raises(oracle.OracleError) as e:
        ix.view_rename([("a", "b")])
    assert e.value.status == "DUP_KEY"
    with pytest.raises(oracle.OracleError) as e:
        ix.view_filter(["a", "missing"])
    assert e.value.status == "NOT_FOUND"


def test_first_rename_rule_wins(oracle):
    g, f = small_file()
    ix = oracle.parse(f)
    r = ix.view_rename([("c.s", "S."), ("c.", "C."), ("c.w", "never.")])
    names = [e["name"] for e in r.entries()]
    assert names == ["a", "b", "C.weight", "S.cale_weight", "d", "e", "f", "z"]


@pytest.mark.parametrize("wl", ["tiny", "stress"])
def test_generated_file_round_trip(oracle, wl):
    """Generator layout == oracle index, and KEEP returns each tensor's bytes."""
    from safetensors_materialization_gb300 import synth
    w = synth.WORKLOADS[wl]()
    lay = w.files[0]
    buf = synth.build_workload_file(w, 0)
    ix = oracle.parse(buf)
    ents = ix.entries()
    assert [e["name"] for e in ents] == [e.name for e in lay.entries]
    assert [(e["begin"], e["end"]) for e in ents] == [(e.begin, e.end) for e in lay.entries]
    data = buf[lay.data_start:]
    plan = ix.select(dst="KEEP")
    rng = np.random.Generator(np.random.PCG64(0))
    for i in rng.choice(len(plan), size=min(len(plan), 200), replace=False):
        o = plan.output(int(i))
        np.testing.assert_array_equal(plan.materialize(int(i), data), data[o["begin"]:o["begin"] + o["bytes"]])
    if wl == "stress":
        # every tensor starts 1..15 bytes off a 16-byte boundary of the file image
        starts = np.array([lay.data_start + e["begin"] for e in ents])
        assert np.all(starts % 16 != 0)


def _zero_image(lay):
    return np.concatenate([np.frombuffer(lay.header, dtype=np.uint8), np.zeros(lay.data_bytes, np.uint8)])


@pytest.mark.parametrize("nparts", [1, 2, 3, 7])
def test_partition_covers_outputs_once(oracle, nparts):
    """Parts are disjoint, contiguous in output order, cover every output, and
    each part's bytes are within one output of the ideal share."""
    from safetensors_materialization_gb300 import synth
    lay = synth.tiny().files[0]
    ix = oracle.parse(_zero_image(lay))
    full = [o["name"] for o in ix.select(dst="BF16").outputs()]
    sizes = {o["name"]: o["bytes"] for o in ix.select(dst="BF16").outputs()}
    parts = [[o["name"] for o in ix.select(dst="BF16", part=k, nparts=nparts).outputs()] for k in range(nparts)]
    assert sum(parts, []) == full
    total = sum(sizes.values())
    biggest = max(sizes.values())
    for p in parts:
        assert abs(sum(sizes[n] for n in p) - total / nparts) <= biggest
    with pytest.raises(oracle.OracleError):
        ix.select(dst="BF16", part=nparts, nparts=nparts)
