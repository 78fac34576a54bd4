"""One index over several shard files (st_index_concat / the oracle's
or_concat): the checkpoint split over shard files of "Disk tier safetensors
streaming design audit (ComfyUI)", "Strategy summary (implemented)", loaded
through one mapping, one plan and one launch.

The oracle's join is pinned against a single file that holds the same
tensors at the same offsets: the shards' entries packed in order with a U8
filler tensor in every gap, parsed by the oracle's own (separately pinned)
parser and narrowed by its filter view.  The library is then compared with
the oracle.
"""
import numpy as np
import pytest

from safetensors_materialization_gb300 import synth


def shards(seed=11):
    """Three small shard files with mixed dtypes and odd sizes, so that the
    joined bases need rounding."""
    rng = np.random.Generator(np.random.PCG64(seed))
    dts = ["F32", "F16", "BF16", "F8_E4M3", "I64", "BOOL"]
    lays = []
    for k in range(3):
        ents = [synth.Entry(f"s{k}.t{i}", dts[int(rng.integers(0, len(dts)))], [int(rng.integers(1, 300))])
                for i in range(5 + k)]
        ents.append(synth.Entry(f"s{k}.w.weight", "F8_E4M3", [7, 9]))
        ents.append(synth.Entry(f"s{k}.w.scale_weight", "F32", []))
        lays.append(synth.make_layout(ents, metadata={"format": "pt", "shard": str(k)}))
    return lays


def shard_data(lays, seed=11):
    out = []
    for k, lay in enumerate(lays):
        d = np.empty(lay.data_bytes, np.uint8)
        synth.fill(lay, d, seed * 10 + k)
        synth.fill_scales(lay, d, seed * 10 + k)
        out.append(d)
    return out


def merged_file(lays, datas, align):
    """One file whose data section is the joined arena: the shards' entries in
    order, a U8 filler where the next shard's start is rounded up."""
    ents, arena, at = [], [], 0
    for k, (lay, d) in enumerate(zip(lays, datas)):
        base = -(-at // align) * align
        if base > at:
            ents.append(synth.Entry(f"__gap{k}", "U8", [base - at]))
            arena.append(np.zeros(base - at, np.uint8))
        ents += [synth.Entry(e.name, e.dtype, list(e.shape)) for e in lay.entries]
        arena.append(d)
        at = base + lay.data_bytes
    m = synth.make_layout(ents)
    data = np.concatenate(arena)
    assert data.size == m.data_bytes
    img = np.concatenate([np.frombuffer(m.header, np.uint8), data])
    real = [e.name for lay in lays for e in lay.entries]
    return img, data, real


def image(lay, d):
    return np.concatenate([np.frombuffer(lay.header, np.uint8), d])


@pytest.mark.parametrize("align", [1, 16, 256, 4096])
def test_oracle_concat_equals_merged_file(oracle, align):
    lays = shards()
    datas = shard_data(lays)
    joined, bases = oracle.concat([oracle.parse(image(l, d)) for l, d in zip(lays, datas)], align)
    img, data, real = merged_file(lays, datas, align)
    merged = oracle.parse(img).view_filter(real)
    assert joined.entries() == merged.entries()
    assert joined.data_bytes == data.size
    end = 0
    for b, lay in zip(bases, lays):
        assert b % align == 0 and end <= b < end + align
        end = b + lay.data_bytes
    for dst in ("BF16", "F32", "KEEP"):
        sfx = (".weight", ".scale_weight") if dst != "KEEP" else None
        a = joined.select(dst=dst, scale_suffix=sfx)
        b = merged.select(dst=dst, scale_suffix=sfx)
        assert a.outputs() == b.outputs()
        for i in range(len(a)):
            assert np.array_equal(a.materialize(i, data), b.materialize(i, data)), (dst, i)


def test_oracle_concat_rules(oracle):
    lays = shards()
    datas = shard_data(lays)
    parts = [oracle.parse(image(l, d)) for l, d in zip(lays, datas)]
    # metadata: first occurrence of each key in part order
    joined, _ = oracle.concat(parts)
    assert joined.metadata() == {"format": "pt", "shard": "0"}
    assert joined.header_len == 0
    # a name in two parts
    with pytest.raises(oracle.OracleError) as e:
        oracle.concat([parts[0], parts[1], parts[0]])
    assert e.value.status == "DUP_KEY"
    # renaming one copy resolves it
    joined, bases = oracle.concat([parts[0], parts[0].view_prefix("s0.").view_rename([("", "x.")])])
    assert len(joined) == 2 * len(parts[0])
    for align in (0, 3, 24):
        with pytest.raises(oracle.OracleError) as e:
            oracle.concat(parts, align)
        assert e.value.status == "INVAL"
    # one part: the same index
    one, b = oracle.concat(parts[:1], 256)
    assert b == [0] and one.entries() == parts[0].entries()


def status_of(fn):
    try:
        fn()
        return "OK"
    except Exception as e:  # noqa: BLE001
        s = getattr(e, "status", None) or getattr(e, "name", None) or str(e)
        return s.replace("ST_E_", "")


@pytest.mark.parametrize("align", [1, 256, 4096])
def test_library_concat_matches_oracle(stmat, oracle, align):
    lays = shards()
    datas = shard_data(lays)
    ojoined, obases = oracle.concat([oracle.parse(image(l, d)) for l, d in zip(lays, datas)], align)
    joined, bases = stmat.Index.concat([stmat.Index.from_header(l.header, l.data_bytes) for l in lays], align)
    assert bases == obases
    assert joined.entries() == ojoined.entries()
    assert joined.sizes() == (0, ojoined.data_bytes)
    assert joined.metadata() == ojoined.metadata()
    for dst in ("BF16", "F16", "KEEP"):
        sfx = (".weight", ".scale_weight") if dst != "KEEP" else None
        p = joined.plan(dst=dst, scale_suffix=sfx, workers=37, host_only=True)
        o = ojoined.select(dst=dst, scale_suffix=sfx)
        assert [(x["name"], x["dtype"], x["bytes"], x["begin"]) for x in p.outputs()] == \
               [(x["name"], x["dtype"], x["bytes"], x["begin"]) for x in o.outputs()]


def test_library_concat_errors_match_oracle(stmat, oracle):
    lays = shards()
    datas = shard_data(lays)
    sp = [stmat.Index.from_header(l.header, l.data_bytes) for l in lays]
    op = [oracle.parse(image(l, d)) for l, d in zip(lays, datas)]
    assert status_of(lambda: stmat.Index.concat([sp[0], sp[1], sp[0]])) == \
        status_of(lambda: oracle.concat([op[0], op[1], op[0]])) == "DUP_KEY"
    for align in (0, 3):
        assert status_of(lambda: stmat.Index.concat(sp, align)) == \
            status_of(lambda: oracle.concat(op, align)) == "INVAL"
    assert status_of(lambda: stmat.Index.concat([])) == "INVAL"
    # views of shards join under their view names; parts may be freed afterwards
    v = [x.view_rename([(f"s{k}.", f"layer{k}.")]) for k, x in enumerate(sp)]
    joined, _ = stmat.Index.concat(v)
    del v, sp
    assert [e["name"] for e in joined.entries()][:2] == ["layer0.t0", "layer0.t1"]


def test_llm_shards_join_in_one_plan(stmat, oracle):
    """The 4-shard LLM layout: one joined index whose outputs are every
    shard's, in shard order, with pieces covering the joined arena."""
    w = synth.llm8b(layers=4, hidden=128, inter=320, vocab=500, kv=32, shards=4)
    assert len(w.files) == 4
    parts = [stmat.Index.from_header(l.header, l.data_bytes) for l in w.files]
    joined, bases = stmat.Index.concat(parts)
    names = [e.name for l in w.files for e in l.entries]
    assert [e["name"] for e in joined.entries()] == names
    plan = joined.plan(dst="F16", workers=64, host_only=True)
    outs = plan.outputs()
    assert [o["name"] for o in outs] == names
    st = plan.stats()
    for k in range(st["pieces"]):
        p = plan.piece(k)
        o = outs[p["output"]]
        shard = max(i for i, b in enumerate(bases) if b <= o["begin"])
        assert bases[shard] <= p["src"] and p["src"] + 2 * p["count"] <= bases[shard] + w.files[shard].data_bytes
