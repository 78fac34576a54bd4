"""Host side of libstmat against the oracle (CPU only, no GPU calls).

Covers: the C ABI exports every symbol include/stmat.h declares; the header
parser returns the oracle's status on every golden case and on randomized
corruptions of real headers; indexes, views and selections match the
oracle's on the synthetic workloads; and the planner's pieces cover every
output exactly once, respect chunk readiness and balance the warps.
"""
import os
import re

import numpy as np
import pytest

from conftest import ROOT, golden, golden_file, small_file

CASES = golden("format_errors.json")["cases"]


def status_of(fn):
    try:
        fn()
        return "OK"
    except Exception as e:  # noqa: BLE001 - both error types carry .status
        s = getattr(e, "status", None)
        if s is None:
            raise
        return s.replace("ST_E_", "")


def header_decls():
    txt = open(os.path.join(ROOT, "include", "stmat.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(st_[a-z0-9_]+)\s*\(", txt)))


def test_library_exports_every_declared_symbol(stmat):
    decls = header_decls()
    assert len(decls) >= 30
    missing = [n for n in decls if not hasattr(stmat.lib(), n)]
    assert not missing, missing
    assert sorted(stmat.EXPORTS) == decls
    assert stmat.lib().st_version() == 0x000100


def test_status_and_dtype_names(stmat):
    L = stmat.lib()
    for i, n in enumerate(stmat.STATUS):
        assert L.st_status_name(i).decode() == n
    for i, n in enumerate(stmat.DTYPES):
        assert L.st_dtype_name(i).decode() == n
    assert [L.st_dtype_size(i) for i in range(16)] == [1, 1, 1, 2, 2, 4, 4, 8, 8, 2, 2, 4, 8, 1, 1, 0]


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_golden_status_matches(stmat, oracle, case):
    f = golden_file(case)
    assert status_of(lambda: stmat.Index.from_file(f)) == case["expect"]
    assert status_of(lambda: oracle.parse(f)) == case["expect"]
    if case["expect"] == "OK" and "names" in case:
        assert [e["name"] for e in stmat.Index.from_file(f).entries()] == case["names"]


def test_header_only_build(stmat):
    g, f = small_file()
    n = stmat.header_size(f[:8])
    ix = stmat.Index.from_header(f[:8 + n], len(f) - 8 - n)
    assert [e["name"] for e in ix.entries()] == g["index_order"]
    with pytest.raises(stmat.StmatError) as e:
        stmat.Index.from_header(f[:8 + n - 1], len(f) - 8 - n)
    assert e.value.status == "ST_E_TRUNCATED"


def same_index(a, b):
    ea, eb = a.entries(), b.entries()
    assert len(ea) == len(eb)
    for x, y in zip(ea, eb):
        assert (x["name"], x["dtype"], x["shape"], x["begin"], x["end"]) == \
            (y["name"], y["dtype"], y["shape"], y["begin"], y["end"])


@pytest.mark.parametrize("wl", ["tiny", "unet", "scaled_fp8", "llm8b", "stress"])
def test_index_matches_oracle_on_workloads(stmat, oracle, wl):
    from safetensors_materialization_gb300 import synth
    w = synth.WORKLOADS[wl]()
    for lay in w.files[:2]:
        lib_ix = stmat.Index.from_header(lay.header, lay.data_bytes)
        same_index(lib_ix, oracle.parse_header(lay.header, lay.data_bytes))
        assert [e["name"] for e in lib_ix.entries()] == [e.name for e in lay.entries]
        assert lib_ix.sizes() == (lay.header_len, lay.data_bytes)


def test_views_match_oracle(stmat, oracle):
    g, f = small_file()
    L, O = stmat.Index.from_file(f), oracle.parse(f)
    same_index(L.view_prefix("c."), O.view_prefix("c."))
    same_index(L.view_filter(["f", "a"]), O.view_filter(["f", "a"]))
    rules = [("c.s", "S."), ("c.", "C."), ("a", "A")]
    same_index(L.view_rename(rules), O.view_rename(rules))
    same_index(L.view_rename(rules).view_prefix("C."), O.view_rename(rules).view_prefix("C."))
    for fn in (lambda ix: ix.view_rename([("a", "b")]), lambda ix: ix.view_filter(["zz"])):
        assert status_of(lambda: fn(L)) == status_of(lambda: fn(O))
    # a view outlives its parent
    v = L.view_prefix("c.")
    del L
    assert [e["name"] for e in v.entries()] == ["weight", "scale_weight"]
    assert v.find("scale_weight") == 1


def test_views_on_unet_match_oracle(stmat, oracle):
    from safetensors_materialization_gb300 import synth
    lay = synth.unet().files[0]
    L = stmat.Index.from_header(lay.header, lay.data_bytes)
    O = oracle.parse_header(lay.header, lay.data_bytes)
    rules = [("model.diffusion_model.", "unet.")]
    same_index(L.view_rename(rules), O.view_rename(rules))
    same_index(L.view_prefix("model.diffusion_model.attn_"), O.view_prefix("model.diffusion_model.attn_"))


def outputs_key(outs):
    return [(o["name"], o["dtype"], o["src_dtype"], o["shape"], o["bytes"], o["scale"]) for o in outs]


SELECTIONS = [
    dict(dst="BF16"), dict(dst="F16"), dict(dst="F32"), dict(dst="KEEP"),
    dict(dst="BF16", scale_suffix=(".weight", ".scale_weight")),
    dict(dst="F32", scale_suffix=(".weight", ".scale_weight")),
    dict(dst="BF16", names=["f", "a", "c.weight"]),
    dict(dst="BF16", names=["c.scale_weight", "c.weight"], scale_names=[None, "c.scale_weight"]),
    dict(dst="BF16", part=1, nparts=3), dict(dst="BF16", part=0, nparts=2),
    # errors
    dict(dst="BF16", names=["nope"]), dict(dst="BF16", names=["a", "a"]),
    dict(dst="BF16", names=["a"], scale_names=["c.scale_weight"]),
    dict(dst="BF16", names=["c.weight"], scale_names=["a"]),
    dict(dst="KEEP", scale_suffix=(".weight", ".scale_weight")), dict(dst="I32"),
    dict(dst="BF16", part=3, nparts=3),
]


@pytest.mark.parametrize("sel", SELECTIONS, ids=[str(i) for i in range(len(SELECTIONS))])
def test_selection_matches_oracle(stmat, oracle, sel):
    g, f = small_file()
    L, O = stmat.Index.from_file(f), oracle.parse(f)
    kw = dict(sel)
    nparts = kw.pop("nparts", 1)
    lib_kw = dict(kw, n_parts=nparts, workers=8, host_only=True)
    so = status_of(lambda: O.select(**kw, nparts=nparts))
    sl = status_of(lambda: L.plan(**lib_kw))
    assert sl == so
    if so == "OK":
        assert outputs_key(L.plan(**lib_kw).outputs()) == outputs_key(O.select(**kw, nparts=nparts).outputs())


@pytest.mark.parametrize("wl,nparts", [("scaled_fp8", 1), ("stress", 1), ("unet", 4), ("stress", 3)])
def test_workload_selection_matches_oracle(stmat, oracle, wl, nparts):
    from safetensors_materialization_gb300 import synth
    w = synth.WORKLOADS[wl]()
    lay = w.files[0]
    L = stmat.Index.from_header(lay.header, lay.data_bytes)
    O = oracle.parse_header(lay.header, lay.data_bytes)
    if w.rename:
        L, O = L.view_rename(w.rename), O.view_rename(w.rename)
    for part in range(nparts):
        a = L.plan(dst=w.dst[0], scale_suffix=w.scale_suffix, part=part, n_parts=nparts, workers=64,
                   host_only=True)
        b = O.select(dst=w.dst[0], scale_suffix=w.scale_suffix, part=part, nparts=nparts)
        assert outputs_key(a.outputs()) == outputs_key(b.outputs())


# ------------------------------------------------------------- fuzzing

MUTATION_BYTES = b'{}[],:"\\ 0123456789-.eEtrufalsn_/x\x00\x1f\x7f\xc3\xa9\xff'


def mutate(rng, h):
    h = bytearray(h)
    for _ in range(int(rng.integers(1, 4))):
        op = int(rng.integers(0, 4))
        i = int(rng.integers(0, max(1, len(h))))
        if op == 0 and h:
            del h[i]
        elif op == 1:
            h.insert(i, MUTATION_BYTES[int(rng.integers(0, len(MUTATION_BYTES)))])
        elif op == 2 and h:
            h[i] = MUTATION_BYTES[int(rng.integers(0, len(MUTATION_BYTES)))]
        else:
            j = int(rng.integers(0, max(1, len(h))))
            h[i:i] = h[j:j + int(rng.integers(1, 12))]
    return bytes(h)


def test_parser_fuzz_matches_oracle(stmat, oracle):
    """Randomly corrupted headers: libstmat and the oracle agree on the status
    (and on the entries when both accept)."""
    import struct
    g, f = small_file()
    base = g["header"].encode()
    data = bytes.fromhex(g["data_hex"])
    rng = np.random.Generator(np.random.PCG64(2024))
    seen = {}
    for _ in range(4000):
        h = mutate(rng, base)
        for extra in (0, 1):
            img = struct.pack("<Q", len(h)) + h + data + bytes(extra)
            sl = status_of(lambda: stmat.Index.from_file(img))
            so = status_of(lambda: oracle.parse(img))
            assert sl == so, (h, sl, so)
            seen[sl] = seen.get(sl, 0) + 1
            if sl == "OK":
                same_index(stmat.Index.from_file(img), oracle.parse(img))
    # the corpus reaches several distinct outcomes
    assert len(seen) >= 4, seen


def test_deep_nesting_matches_oracle(stmat, oracle):
    import struct
    for depth in (62, 63, 64, 65, 200):
        meta = '{"__metadata__":{"k":"v"},"x":' + "[" * depth + "]" * depth + "}"
        img = struct.pack("<Q", len(meta)) + meta.encode()
        assert status_of(lambda: stmat.Index.from_file(img)) == status_of(lambda: oracle.parse(img)), depth


# ------------------------------------------------------------- planner

def piece_table(plan):
    st = plan.stats()
    return [plan.piece(k) for k in range(st["pieces"])], st


CLS_SIZES = {0: (1, 1), 1: (4, 2), 2: (4, 2), 3: (2, 2), 4: (2, 4), 5: (2, 2), 6: (2, 4),
             7: (1, 2), 8: (1, 2), 9: (1, 4), 10: (1, 2), 11: (1, 2), 12: (1, 4)}


@pytest.mark.parametrize("wl,workers,chunk", [("tiny", 7, 0), ("tiny", 64, 1 << 16), ("unet", 1216, 0),
                                              ("unet", 300, 64 << 20), ("scaled_fp8", 4864, 0),
                                              ("stress", 4864, 0), ("stress", 1000, 50 << 20)])
def test_pieces_cover_outputs_once(stmat, wl, workers, chunk):
    from safetensors_materialization_gb300 import synth
    w = synth.WORKLOADS[wl]()
    lay = w.files[0]
    ix = stmat.Index.from_header(lay.header, lay.data_bytes)
    if w.rename:
        ix = ix.view_rename(w.rename)
    if w.prefix:
        ix = ix.view_prefix(w.prefix)
    plan = ix.plan(dst=w.dst[0], scale_suffix=w.scale_suffix, workers=workers, chunk_bytes=chunk,
                   host_only=True)
    outs = plan.outputs()
    pieces, st = piece_table(plan)
    assert st["workers"] <= workers
    covered = [[] for _ in outs]
    cls_of = {}
    for chunk_i in range(st["chunks"]):
        prev = None
        for wk in range(st["workers"] + 1):    # the warps' own shares, then the claimed pieces
            a, b = plan.worker(chunk_i, wk)
            assert prev is None or a == prev   # workers' ranges are consecutive
            prev = b
            for p in pieces[a:b]:
                o = outs[p["output"]]
                si, so = CLS_SIZES[p["cls"]]
                assert cls_of.setdefault(p["output"], p["cls"]) == p["cls"]
                u0, rem = divmod(p["src"] - o["begin"], si)
                assert rem == 0 and p["dst"] == u0 * so
                covered[p["output"]].append((u0, u0 + p["count"]))
                if chunk:
                    # every byte the piece reads is staged by the end of its chunk
                    assert p["src"] + p["count"] * si <= (chunk_i + 1) * chunk
                    if p["scale"] != (1 << 64) - 1:
                        assert p["scale"] + 4 <= (chunk_i + 1) * chunk
    for i, o in enumerate(outs):
        if o["bytes"] == 0:
            assert not covered[i]
            continue
        total = o["bytes"] if cls_of[i] == 0 else o["numel"]   # copies count bytes
        pos = 0
        for a, b in sorted(covered[i]):
            assert a == pos, o["name"]
            pos = b
        assert pos == total, o["name"]


def test_worker_balance(stmat):
    """Each warp's share of bytes is within one piece cost of the mean."""
    from safetensors_materialization_gb300 import synth
    for wl, W in (("unet", 1216), ("stress", 2432)):
        w = synth.WORKLOADS[wl]()
        lay = w.files[0]
        plan = stmat.Index.from_header(lay.header, lay.data_bytes).plan(dst="BF16", workers=W, host_only=True)
        pieces, st = piece_table(plan)
        loads = []
        for wk in range(st["workers"]):
            a, b = plan.worker(0, wk)
            loads.append(sum(1024 + p["count"] * sum(CLS_SIZES[p["cls"]]) for p in pieces[a:b]))
        mean = sum(loads) / len(loads)
        biggest_unsplit = 1024 + 4096 * 12
        assert max(loads) <= mean + biggest_unsplit + 2048, (wl, max(loads), mean)


def test_tma_claimed_tail_is_cut_into_segment_pieces(stmat):
    """The TMA build's claimed tail holds pieces of at most 2 KiB of source
    (one segment: its warps claim two or more at a time), while its own
    shares keep whole 16 KiB units; the streaming build's claimed tail keeps
    whole units.  (test_pieces_cover_outputs_once checks that TMA plans of
    this workload still cover every output once.)"""
    from safetensors_materialization_gb300 import synth
    lay = synth.stress().files[0]
    ix = stmat.Index.from_header(lay.header, lay.data_bytes)
    W = 2432

    def src_bytes(p):
        return p["count"] * CLS_SIZES[p["cls"]][0]

    plan = ix.plan(dst="BF16", workers=W, host_only=True)
    assert plan.stats()["kernel"] == "tma"
    pieces, st = piece_table(plan)
    a, b = plan.worker(0, st["workers"])
    tail, own = pieces[a:b], pieces[:a]
    assert len(tail) > 1000
    assert all(p["rows"] == 1 and 1 <= src_bytes(p) <= 2048 for p in tail)
    assert max(src_bytes(p) for p in own) > 8192
    stream = ix.plan(dst="BF16", workers=W, host_only=True, kernel=1)
    spieces, sst = piece_table(stream)
    a, b = stream.worker(0, sst["workers"])
    assert b > a and max(src_bytes(p) for p in spieces[a:b]) > 8192


# ------------------------------------------------------------- slicing

def sliced_layout(seed):
    import json
    import struct
    rng = np.random.Generator(np.random.PCG64(seed))
    shapes = [[64, 300], [9, 40, 33], [3, 5, 7, 11], [4096, 96], [2, 700], [12]]
    dts = ["F32", "F16", "F8_E4M3", "BF16", "I64", "F8_E5M2"]
    isz = {"F32": 4, "F16": 2, "BF16": 2, "F8_E4M3": 1, "F8_E5M2": 1, "I64": 8}
    ents, off = {}, 0
    for i, (shp, dt) in enumerate(zip(shapes, dts)):
        n = int(np.prod(shp))
        ents[f"s{i}"] = {"dtype": dt, "shape": shp, "data_offsets": [off, off + n * isz[dt]]}
        off += n * isz[dt]
    h = json.dumps(ents).encode()
    return struct.pack("<Q", len(h)) + h, off, shapes, rng


def test_slicing_outputs_match_oracle(stmat, oracle):
    header, data_bytes, shapes, rng = sliced_layout(1)
    L = stmat.Index.from_header(header, data_bytes)
    O = oracle.parse(np.concatenate([np.frombuffer(header, dtype=np.uint8), np.zeros(data_bytes, np.uint8)]))
    names = [f"s{i}" for i in range(len(shapes))]
    for trial in range(20):
        slices = []
        for shp in shapes:
            if rng.integers(0, 4) == 0:
                slices.append(None)
                continue
            d = int(rng.integers(0, len(shp)))
            a = int(rng.integers(0, shp[d]))
            slices.append((d, a, int(rng.integers(a, shp[d] + 1))))
        for dst in ("BF16", "KEEP"):
            for nparts, part in ((1, 0), (2, 1)):
                a_ = L.plan(dst=dst, names=names, slices=slices, workers=16, host_only=True, n_parts=nparts,
                            part=part)
                b_ = O.select(dst=dst, names=names, slices=slices, nparts=nparts, part=part)
                assert outputs_key(a_.outputs()) == outputs_key(b_.outputs())
    for bad in [(2, 0, 1), (0, 5, 4), (1, 0, 301), (-1, 0, 0)]:
        sl = [bad] + [None] * (len(shapes) - 1)
        sa = status_of(lambda: L.plan(dst="BF16", names=names, slices=sl, workers=4, host_only=True))
        so = status_of(lambda: O.select(dst="BF16", names=names, slices=sl))
        assert sa == so
    assert status_of(lambda: L.plan(dst="BF16", slices=[(0, 0, 1)] * 6, workers=4, host_only=True)) == "INVAL"


@pytest.mark.parametrize("chunk", [0, 20000])
def test_sliced_pieces_cover_each_output_once(stmat, chunk):
    header, data_bytes, shapes, rng = sliced_layout(2)
    ix = stmat.Index.from_header(header, data_bytes)
    names = [f"s{i}" for i in range(len(shapes))]
    slices = [(1, 7, 250), (1, 3, 30), (2, 2, 5), (1, 16, 48), (1, 100, 101), (0, 2, 9)]
    plan = ix.plan(dst="BF16", names=names, slices=slices, workers=37, host_only=True, chunk_bytes=chunk,
                   unit_bytes=2048)
    outs = plan.outputs()
    st = plan.stats()
    covered = [set() for _ in outs]
    multi = 0
    for k in range(st["pieces"]):
        p = plan.piece(k)
        si, so = CLS_SIZES[p["cls"]]
        multi += p["rows"] > 1
        for r in range(p["rows"]):
            u0 = p["dst"] // so + r * p["count"]
            for u in range(u0, u0 + p["count"]):
                assert u not in covered[p["output"]]
                covered[p["output"]].add(u)
    for i, o in enumerate(outs):
        isz = {"I64": 8, "F32": 4, "F16": 2, "BF16": 2, "F8_E4M3": 1, "F8_E5M2": 1}[o["src_dtype"]]
        units = o["numel"] * (1 if o["dtype"] != o["src_dtype"] else isz)   # copies count bytes
        assert len(covered[i]) == units, o["name"]
    assert multi > 0


def test_plan_copy_bytes_of_a_tensor_parallel_rank(stmat):
    """A tensor-parallel rank's plan copies only the byte ranges it reads
    (under three quarters of the data section); a whole-checkpoint plan
    copies everything.  Host-only plans, no GPU."""
    from safetensors_materialization_gb300 import synth
    w = synth.llm8b(seed=8, layers=2, hidden=1024, inter=2816, vocab=4000, kv=256, shards=1)
    lay = w.files[0]
    ix = stmat.Index.from_header(lay.header, lay.data_bytes)
    full = ix.plan(dst="BF16", workers=64, host_only=True)
    assert full.copy_bytes() == (lay.data_bytes, 1)
    tp = synth.tp_slices(lay.entries, 4, 1)
    names = list(tp)
    part = ix.plan(dst="BF16", names=names, slices=[tp[n] for n in names], workers=64, host_only=True)
    b, r = part.copy_bytes()
    ents = {e["name"]: e for e in ix.entries()}
    want = 0   # each output's source extent: a dim-0 slice its rows; a dim-1 slice from its first row's
    for n in names:   # first column to its last row's last column (BF16: 2 bytes an element)
        (rows, cols), (dim, start, stop) = ents[n]["shape"], tp[n]
        want += (stop - start) * cols * 2 if dim == 0 else ((rows - 1) * cols + (stop - start)) * 2
    assert r > 1 and want <= b < lay.data_bytes * 3 // 4
    assert b <= want + r * 65536                    # plus at most the merged gaps


def test_plan_copy_ranges_merge_and_threshold(stmat):
    """The ranges a sparse plan copies: one per output extent, merged when the
    gap between them is at most 64 KiB; a plan reading three quarters or more
    of the data section copies all of it."""
    import json
    import struct
    n = 100_000
    ents = {name: {"dtype": "U8", "shape": [n], "data_offsets": [k * n, (k + 1) * n]}
            for k, name in enumerate(["a", "b", "c", "d"])}
    h = json.dumps(ents).encode()
    img = np.frombuffer(struct.pack("<Q", len(h)) + h + bytes(4 * n), dtype=np.uint8)
    ix = stmat.Index.from_file(img)

    def copied(sl):
        names = list(sl)
        return ix.plan(dst="KEEP", names=names, slices=[sl[k] for k in names], workers=8,
                       host_only=True).copy_bytes()

    # a[99000:100000] ends at 100000; b's slice starts 65536 (merged) or 65537 (separate) bytes later
    assert copied({"a": (0, 99_000, n), "b": (0, 65_536, 66_536)}) == (100_000 + 66_536 - 99_000, 1)
    assert copied({"a": (0, 99_000, n), "b": (0, 65_537, 66_537)}) == (2_000, 2)
    # three quarters of the data section or more: everything
    assert copied({"a": (0, 0, n), "b": (0, 0, n), "c": (0, 0, n)}) == (4 * n, 1)
    assert copied({"a": (0, 0, n), "b": (0, 0, n), "c": (0, 0, n - 1)}) == (3 * n - 1, 1)
