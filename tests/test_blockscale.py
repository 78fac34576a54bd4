"""Block-scaled weights (block FP8, NVFP4) through the library: the host side
against the oracle (CPU) and the TMA kernel build against the oracle, byte
for byte (GPU).  The formats are the readings stated in include/stmat.h
(st_block_quant) and pinned in tests/test_oracle_blockscale.py."""
import json
import struct

import numpy as np
import pytest

from oracle_compare import GuardedOutputs, compare_full
from safetensors_materialization_gb300 import synth


def image(ents_data, lead=0):
    """File image from [(name, dtype, shape, raw bytes)]; `lead` spacer bytes
    in front of the first tensor shift every later offset."""
    ents, parts, off = {}, [], 0
    if lead:
        ents["_lead"] = {"dtype": "U8", "shape": [lead], "data_offsets": [0, lead]}
        parts.append(bytes(lead))
        off = lead
    for name, dt, shape, raw in ents_data:
        ents[name] = {"dtype": dt, "shape": list(shape), "data_offsets": [off, off + len(raw)]}
        parts.append(raw)
        off += len(raw)
    h = json.dumps(ents).encode()
    return np.frombuffer(struct.pack("<Q", len(h)) + h + b"".join(parts), dtype=np.uint8).copy()


def quant_file(seed, lead=0, fp8=("F8_E4M3", 257, 300, (128, 128)), nv=(33, 200)):
    """One block-FP8 weight and one NVFP4 weight (with their scales) plus an
    ordinary F16 tensor in between, at odd sizes so offsets are unaligned."""
    rng = np.random.Generator(np.random.PCG64(seed))
    dt, M, N, (br, bc) = fp8
    w = rng.integers(0, 256, size=M * N, dtype=np.uint8)
    sc = rng.uniform(1e-3, 1e-1, size=(-(-M // br)) * (-(-N // bc))).astype(np.float32)
    Mn, Nn = nv
    wn = rng.integers(0, 256, size=Mn * Nn // 2, dtype=np.uint8)
    sn = rng.integers(0x08, 0x48, size=Mn * (-(-Nn // 16)), dtype=np.uint8)
    sn[::37] = 0x7F                                     # some NaN block scales
    g = np.float32(rng.uniform(1e-4, 1e-2))
    h16 = rng.standard_normal(77).astype(np.float16)
    ents = [("a.weight", dt, [M, N], w.tobytes()),
            ("a.weight_scale_inv", "F32", [-(-M // br), -(-N // bc)], sc.tobytes()),
            ("mid", "F16", [77], h16.tobytes()),
            ("b.weight", "U8", [Mn, Nn // 2], wn.tobytes()),
            ("b.weight_scale", "F8_E4M3", [Mn, -(-Nn // 16)], sn.tobytes()),
            ("b.weight_scale_2", "F32", [], g.tobytes())]
    quant = {"a.weight": ("block_fp8", "a.weight_scale_inv", None, (br, bc)),
             "b.weight": ("nvfp4", "b.weight_scale", "b.weight_scale_2", None)}
    return image(ents, lead), quant


def selection(ix, quant):
    names = [e["name"] for e in ix.entries()]
    return names, [quant.get(n) for n in names]


def outputs_key(outs):
    return [(o["name"], o["dtype"], o["shape"], o["bytes"], o["scale"], o["quant"]) for o in outs]


@pytest.mark.parametrize("dst", ["BF16", "F16", "F32"])
def test_library_selection_matches_oracle(stmat, oracle, dst):
    img, quant = quant_file(1, lead=3)
    ix, oix = stmat.Index.from_file(img), oracle.parse(img)
    names, q = selection(ix, quant)
    plan = ix.plan(dst=dst, names=names, quant=q, workers=64, host_only=True)
    sel = oix.select(dst=dst, names=names, quant=q)
    assert outputs_key(plan.outputs()) == outputs_key(sel.outputs())
    assert plan.stats()["kernel"] == "tma_wide"
    assert [o["name"] for o in plan.outputs()] == ["_lead", "a.weight", "mid", "b.weight"]


def test_library_errors_match_oracle(stmat, oracle):
    img = image([("w", "F8_E4M3", [4, 32], bytes(128)), ("s", "F32", [1, 1], struct.pack("<f", 1.0)),
                 ("s2", "F32", [1, 2], bytes(8)), ("h", "F16", [4, 32], bytes(256)),
                 ("u", "U8", [4, 16], bytes(64)), ("e", "F8_E4M3", [4, 2], bytes(8)),
                 ("g", "F32", [], bytes(4)), ("g2", "F32", [2], bytes(8))])
    ix, oix = stmat.Index.from_file(img), oracle.parse(img)

    def lib(**kw):
        try:
            ix.plan(workers=8, host_only=True, **kw)
            return "OK"
        except stmat.StmatError as e:
            return e.status.replace("ST_E_", "")

    def orc(**kw):
        try:
            oix.select(**kw)
            return "OK"
        except oracle.OracleError as e:
            return e.status

    cases = [dict(names=["w"], quant=[("block_fp8", "s", None, (128, 128))]),
             dict(names=["w"], quant=[("block_fp8", "s2", None, (128, 16))]),
             dict(names=["w"], quant=[("block_fp8", "s", None, (128, 8))]),
             dict(names=["w"], quant=[("block_fp8", "s", None, (96, 128))]),
             dict(names=["w"], quant=[("block_fp8", "s2", None, (128, 128))]),
             dict(names=["h"], quant=[("block_fp8", "s", None, None)]),
             dict(names=["w"], quant=[("block_fp8", "nope", None, None)]),
             dict(names=["w"], dst="KEEP", quant=[("block_fp8", "s", None, None)]),
             dict(names=["w"], quant=[("block_fp8", "s", None, None)], slices=[(0, 0, 1)]),
             dict(names=["w"], quant=[("block_fp8", "s", None, None)], scale_names=["g"]),
             dict(names=["w"], quant=[("other", "s", None, None)]),
             dict(names=["u"], quant=[("nvfp4", "e", "g", None)]),
             dict(names=["u"], quant=[("nvfp4", "e", "g", (2, 16))]),
             dict(names=["u"], quant=[("nvfp4", "e", None, None)]),
             dict(names=["u"], quant=[("nvfp4", "e", "g2", None)]),
             dict(names=["u"], quant=[("nvfp4", "s", "g", None)]),
             dict(names=["w"], quant=[("nvfp4", "e", "g", None)]),
             dict(names=["u"], quant=[("nvfp4", "e", "nope", None)])]
    for kw in cases:
        assert lib(**kw) == orc(**kw), kw
    # the register builds refuse block-scaled outputs
    for kernel in (1, 2):
        with pytest.raises(stmat.StmatError) as e:
            ix.plan(names=["w"], quant=[("block_fp8", "s", None, (128, 128))], workers=8, host_only=True, kernel=kernel)
        assert e.value.status == "ST_E_INVAL"


def test_synthetic_workloads_select_like_the_oracle(stmat, oracle):
    for name in ("block_fp8_4l", "nvfp4_4l"):
        w = synth.WORKLOADS[name]()
        lay = w.files[0]
        ix = stmat.Index.from_header(lay.header, lay.data_bytes)
        oix = oracle.parse_header(lay.header, lay.data_bytes)
        names, q = selection(ix, w.quant)
        plan = ix.plan(dst="BF16", names=names, quant=q, workers=64, host_only=True)
        sel = oix.select(dst="BF16", names=names, quant=q)
        assert outputs_key(plan.outputs()) == outputs_key(sel.outputs())
        assert len(plan.outputs()) == len(w.quant)


# ------------------------------------------------------------------ GPU

def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return torch


def run_gpu(stmat, img, quant, dst, shift=0, **kw):
    torch = _gpu()
    ix = stmat.Index.from_file(img)
    names, q = selection(ix, quant)
    plan = ix.plan(dst=dst, names=names, quant=q, **kw)
    hlen, dbytes = ix.sizes()
    data = img[8 + hlen:]
    buf = torch.zeros(data.size + 32, dtype=torch.uint8, device="cuda")
    buf[shift:shift + data.size].copy_(torch.from_numpy(data.copy()))
    outs = GuardedOutputs(plan)
    plan.materialize(buf.data_ptr() + shift, outs.ptrs)
    torch.cuda.synchronize()
    assert plan.check() == 0
    return plan, outs, names, q


def assert_outputs(plan, outs, want):
    """Every output equals the oracle's bytes; guard bytes untouched."""
    outs.check_guards()
    for i, o in enumerate(plan.outputs()):
        got = outs.raw(i).cpu().numpy()
        if not np.array_equal(got, want[i]):
            bad = np.nonzero(got != want[i])[0]
            raise AssertionError(f"{o['name']}: {bad.size} bytes differ, first at {bad[0]}")


@pytest.mark.gpu
@pytest.mark.parametrize("dst", ["BF16", "F16", "F32"])
@pytest.mark.parametrize("lead,shift,kernel", [(0, 0, 0), (3, 0, 3), (1, 7, 0), (13, 9, 3)])
def test_gpu_blockscaled_matches_oracle(stmat, oracle, dst, lead, shift, kernel):
    """Both formats, unaligned weight and scale offsets, the data section at
    several device misalignments, ragged rows and blocks, on both TMA builds."""
    img, quant = quant_file(10 + lead, lead=lead)
    plan, outs, names, q = run_gpu(stmat, img, quant, dst, shift=shift, kernel=kernel)
    assert plan.stats()["kernel"] == {0: "tma_wide", 3: "tma"}[kernel]
    oix = oracle.parse(img)
    sel = oix.select(dst=dst, names=names, quant=q)
    data = img[8 + oix.header_len:]
    assert_outputs(plan, outs, [sel.materialize(i, data) for i in range(len(sel))])


@pytest.mark.gpu
@pytest.mark.parametrize("fp8", [("F8_E5M2", 64, 48, (16, 16)), ("F8_E4M3", 3, 2000, (1, 16)),
                                 ("F8_E4M3", 1000, 17, (256, 16)), ("F8_E4M3", 130, 1030, (64, 512)),
                                 ("F8_E4M3", 9, 40000, (1, 16))])
def test_gpu_block_shapes(stmat, oracle, fp8):
    img, quant = quant_file(20, lead=5, fp8=fp8, nv=(7, 2064))
    for dst in ("BF16", "F32"):
        plan, outs, names, q = run_gpu(stmat, img, quant, dst, workers=[1, 9, 0][len(fp8[0]) % 3])
        oix = oracle.parse(img)
        sel = oix.select(dst=dst, names=names, quant=q)
        data = img[8 + oix.header_len:]
        assert_outputs(plan, outs, [sel.materialize(i, data) for i in range(len(sel))])


@pytest.mark.gpu
@pytest.mark.parametrize("kernel", [0, 3])
@pytest.mark.parametrize("dst", ["F32", "BF16", "F16"])
def test_gpu_outputs_at_itemsize_alignment(stmat, oracle, kernel, dst):
    """Outputs aligned to their itemsize only (4 mod 8 for F32, 2 mod 4 for
    BF16/F16): an NVFP4 output's two-element units then never reach vector
    alignment, so every unit is written element by element; the bytes equal
    the oracle's."""
    torch = _gpu()
    img, quant = quant_file(60, lead=3)
    ix = stmat.Index.from_file(img)
    names, q = selection(ix, quant)
    plan = ix.plan(dst=dst, names=names, quant=q, kernel=kernel)
    data = img[8 + ix.sizes()[0]:]
    dbuf = torch.from_numpy(data.copy()).cuda()
    infos = plan.outputs()
    at, offs = 0, []
    for o in infos:
        at = (at + 255) // 256 * 256 + (4 if dst == "F32" else 2)
        offs.append(at)
        at += o["bytes"]
    arena = torch.full((at + 256,), 0xA5, dtype=torch.uint8, device="cuda")
    ptrs = torch.tensor([arena.data_ptr() + x for x in offs], dtype=torch.int64, device="cuda")
    plan.materialize(dbuf, ptrs)
    torch.cuda.synchronize()
    assert plan.check() == 0
    oix = oracle.parse(img)
    sel = oix.select(dst=dst, names=names, quant=q)
    host = arena.cpu().numpy()
    for i, o in enumerate(infos):
        assert np.array_equal(host[offs[i]:offs[i] + o["bytes"]], sel.materialize(i, data)), o["name"]


@pytest.mark.gpu
def test_gpu_blockscaled_noalloc(stmat, oracle):
    torch = _gpu()
    img, quant = quant_file(30, lead=2)
    ix = stmat.Index.from_file(img)
    names, q = selection(ix, quant)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = ix.plan(dst="BF16", names=names, quant=q, workers=sms * 16, host_only=True)
    hlen, _ = ix.sizes()
    buf = torch.from_numpy(img[8 + hlen:].copy()).cuda()
    outs = GuardedOutputs(plan)
    plan.materialize_noalloc(buf.data_ptr(), outs.ptrs)
    torch.cuda.synchronize()
    oix = oracle.parse(img)
    sel = oix.select(dst="BF16", names=names, quant=q)
    assert_outputs(plan, outs, [sel.materialize(i, img[8 + hlen:]) for i in range(len(sel))])


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["block_fp8", "nvfp4"])
def test_gpu_blockscaled_workloads(stmat, oracle, name):
    """The full synthetic checkpoints (40 layers), every element of every
    weight against the oracle (all host cores)."""
    torch = _gpu()
    w = synth.WORKLOADS[name]()
    lay = w.files[0]
    img = synth.build_workload_file(w, 0)
    plan, outs, names, q = run_gpu(stmat, img, w.quant, "BF16")
    outs.check_guards()
    sel = oracle.parse_header(lay.header, lay.data_bytes).select(dst="BF16", names=names, quant=q)
    assert compare_full(sel, img[lay.data_start:], {name: outs}) == sum(o["bytes"] for o in plan.outputs())
    del torch


@pytest.mark.parametrize("chunk", [4096, 65536])
def test_chunked_plans_wait_for_block_scales(stmat, chunk):
    """With st_load's chunks, a block-scaled piece runs only after the chunk
    holding the end of its scale tensors (and its global scale)."""
    img, quant = quant_file(40, lead=11)
    ix = stmat.Index.from_file(img)
    names, q = selection(ix, quant)
    ents = {e["name"]: e for e in ix.entries()}
    plan = ix.plan(dst="BF16", names=names, quant=q, workers=16, chunk_bytes=chunk, host_only=True)
    outs = plan.outputs()
    st = plan.stats()
    for c in range(st["chunks"]):
        for w in range(st["workers"] + 1):   # own shares and the claimed pieces
            a, b = plan.worker(c, w)
            for k in range(a, b):
                p = plan.piece(k)
                o = outs[p["output"]]
                assert p["src"] + p["count"] <= (c + 1) * chunk or not o["quant"]
                if o["quant"]:
                    assert ents[o["scale"]]["end"] <= (c + 1) * chunk
                    if o["quant"] == "nvfp4":
                        assert ents[quant[o["name"]][2]]["end"] <= (c + 1) * chunk


@pytest.mark.gpu
@pytest.mark.parametrize("dst", ["BF16", "F16", "F32"])
def test_gpu_special_scales(stmat, oracle, dst):
    """Every fp8 code (E5M2 infinities and NaNs included) against block
    scales of 0, -0, inf, NaN, tiny and huge values, and NVFP4 with the same
    global/block scale specials: 0 x inf and NaN products must come out as
    the canonical NaN, the rest exactly as the oracle."""
    specials = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, 3.4e38, 1.0], dtype=np.float32)
    w = np.tile(np.arange(256, dtype=np.uint8), 8)                     # [8, 256]: each row every code
    sc = np.repeat(specials, 16).reshape(8, 16)                        # 16 x 16 blocks, one special per row
    for fmt in ("F8_E5M2", "F8_E4M3"):
        ents = [("a.weight", fmt, [8, 256], w.tobytes()), ("a.s", "F32", [8, 16], sc.astype(np.float32).tobytes())]
        nb = np.tile(np.arange(256, dtype=np.uint8), 2)                # NVFP4 [4, 128]: 256 elements per row
        ns = np.array([0x00, 0x80, 0x7F, 0x38, 0x01, 0x7E, 0xFE, 0x08] * 8, dtype=np.uint8)   # [4, 16]
        for g in (0.0, np.inf, np.nan, 2.5e-3):
            img = image(ents + [("b.weight", "U8", [4, 128], nb.tobytes()), ("b.s", "F8_E4M3", [4, 16], ns.tobytes()),
                                ("b.g", "F32", [], np.float32(g).tobytes())], lead=1)
            quant = {"a.weight": ("block_fp8", "a.s", None, (1, 16)), "b.weight": ("nvfp4", "b.s", "b.g", None)}
            plan, outs, names, q = run_gpu(stmat, img, quant, dst)
            oix = oracle.parse(img)
            sel = oix.select(dst=dst, names=names, quant=q)
            data = img[8 + oix.header_len:]
            assert_outputs(plan, outs, [sel.materialize(i, data) for i in range(len(sel))])


@pytest.mark.gpu
@pytest.mark.parametrize("chunk", [4096, 5000, 1 << 16])
def test_gpu_chunked_loads_wait_for_block_scales(stmat, oracle, tmp_path, chunk):
    """Block-scaled weights through the chunked pipelines, st_load from pinned
    memory and st_load_files through a pinned ring: a chunk's pieces run only
    once the chunk holding their block scales has landed; the bytes equal
    the oracle's."""
    import os
    torch = _gpu()
    img, quant = quant_file(77, lead=9)
    path = os.path.join(str(tmp_path), "q.safetensors")
    img.tofile(path)
    oix = oracle.parse(img)
    data = img[8 + oix.header_len:]
    files, ix = stmat.Files.of_checkpoint([path])
    names, q = selection(ix, quant)
    sel = oix.select(dst="BF16", names=names, quant=q)
    want = [sel.materialize(i, data) for i in range(len(sel))]
    for mode in ("pinned", "ring"):
        plan = ix.plan(dst="BF16", names=names, quant=q, chunk_bytes=chunk)
        assert plan.stats()["chunks"] > 1
        dev = torch.full((data.size,), 0xA5, dtype=torch.uint8, device="cuda")
        outs = GuardedOutputs(plan)
        copy = torch.cuda.Stream()
        if mode == "pinned":
            host = torch.from_numpy(data.copy()).pin_memory()
            plan.load(host, dev, outs.ptrs, copy_stream=copy, compute_stream=torch.cuda.current_stream())
        else:
            ring = torch.empty(3 * chunk, dtype=torch.uint8).pin_memory()
            plan.load_files(files, dev, outs.ptrs, ring, threads=3, copy_stream=copy,
                            compute_stream=torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert plan.check() == 0
        assert_outputs(plan, outs, want)
    files.close()
