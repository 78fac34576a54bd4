"""GPU parity: libstmat's CUDA path against the oracle, byte for byte (0 ULP).

Every test calls the product through the C ABI (ctypes binding) and compares
with the oracle on the same seeded bytes, in full (the large workloads are
compared in full in test_full_parity.py).  Every destination arena is filled
with a guard value first, and every byte that no output owns (alignment
padding, gaps between packed outputs, the tail) must still hold it after the
launch; the device copy of the source must be unchanged.
"""
import json
import struct

import numpy as np
import pytest

from conftest import golden, small_file
from oracle_compare import FILL, GuardedOutputs, assert_device_equals_host, assert_guards, compare_full

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def to_device(image, offset=0, whole=True, data_start=None):
    """Copies a file image (uint8 numpy) to the GPU.  whole=True keeps the
    header in front (so the data section keeps the file's alignment) and adds
    `offset` bytes before the image; returns (buffer, data pointer)."""
    if whole:
        buf = torch.empty(image.size + offset + 16, dtype=torch.uint8, device="cuda")
        buf[offset:offset + image.size].copy_(torch.from_numpy(image))
        return buf, buf.data_ptr() + offset + data_start
    data = image[data_start:]
    buf = torch.empty(max(1, data.size), dtype=torch.uint8, device="cuda")
    if data.size:
        buf[:data.size].copy_(torch.from_numpy(np.ascontiguousarray(data)))
    return buf, buf.data_ptr()


class Packed:
    """Outputs packed back to back, each aligned only to its itemsize."""

    def __init__(self, plan, shift=0):
        self.infos = plan.outputs()
        offs, at = [], 0
        for o in self.infos:
            isz = max(1, o["bytes"] // max(1, o["numel"]))
            at = (at + isz - 1) // isz * isz
            if (at // isz) % 2 == 0:
                at += isz  # keep it off 2*itemsize alignment
            offs.append(at)
            at += o["bytes"]
        self.offsets = offs
        self.arena = torch.full((at + 64,), FILL, dtype=torch.uint8, device="cuda")
        self.ptrs = torch.tensor([self.arena.data_ptr() + o for o in offs] or [0], dtype=torch.int64,
                                 device="cuda")

    def raw(self, i):
        return self.arena[self.offsets[i]:self.offsets[i] + self.infos[i]["bytes"]]

    def check_guards(self):
        assert_guards(self.arena, self.offsets, [o["bytes"] for o in self.infos])


def run(stmat, image, dst="BF16", view=None, scale_suffix=None, whole=True, offset=0, packed=False,
        workers=0, scales=None, kernel=0):
    ix = stmat.Index.from_file(image)
    if view:
        ix = view(ix)
    plan = ix.plan(dst=dst, scale_suffix=scale_suffix, workers=workers, kernel=kernel)
    hlen, dbytes = ix.sizes()
    buf, data_ptr = to_device(image, offset, whole, 8 + hlen)
    outs = Packed(plan) if packed else GuardedOutputs(plan)
    plan.materialize(data_ptr, outs.ptrs, scales=scales)
    torch.cuda.synchronize()
    assert plan.check() == 0
    outs.check_guards()
    if whole:
        assert_device_equals_host(buf[offset:offset + image.size], image)
    else:
        assert_device_equals_host(buf[:image.size - 8 - hlen], image[8 + hlen:])
    return plan, outs, buf


def oracle_all(oracle, image, dst="BF16", view=None, scale_suffix=None):
    ix = oracle.parse(image)
    if view:
        ix = view(ix)
    sel = ix.select(dst=dst, scale_suffix=scale_suffix)
    data = image[8 + ix.header_len:]
    return sel, [sel.materialize(i, data) for i in range(len(sel))]


def assert_same(plan, outs, sel, expected):
    """Every output equals the oracle's bytes; guard bytes untouched."""
    assert [o["name"] for o in plan.outputs()] == [o["name"] for o in sel.outputs()]
    if hasattr(outs, "check_guards"):
        outs.check_guards()
    for i, want in enumerate(expected):
        got = outs.raw(i).cpu().numpy()
        if not np.array_equal(got, want):
            bad = np.nonzero(got != want)[0]
            raise AssertionError(f"output {plan.output(i)['name']}: {bad.size} bytes differ, first at {bad[0]}: "
                                 f"got {got[bad[0]:bad[0] + 8].tobytes().hex()} want {want[bad[0]:bad[0] + 8].tobytes().hex()}")


def image_of(ents, data, pad=0):
    h = json.dumps(ents).encode() + b" " * pad
    return np.frombuffer(struct.pack("<Q", len(h)) + h + data, dtype=np.uint8).copy()


# ------------------------------------------------------------------ golden

@pytest.mark.parametrize("dst", ["BF16", "F16", "F32"])
def test_golden_small_file(stmat, oracle, dst):
    g, f = small_file()
    img = np.frombuffer(f, dtype=np.uint8).copy()
    plan, outs, _ = run(stmat, img, dst=dst, scale_suffix=(".weight", ".scale_weight"))
    for i, o in enumerate(plan.outputs()):
        assert outs.raw(i).cpu().numpy().tobytes().hex() == g["expect"][dst][o["name"]], o["name"]


# -------------------------------------------------- exhaustive special values

def special_image(seed=0):
    """Every f16, bf16 and fp8 bit pattern, a structured f32 sweep, and fp8
    tensors under special scales (2^k, random, subnormal-producing, overflowing,
    zero, negative, NaN, +inf, -inf)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    parts, ents, off = [], {}, 0

    def add(name, dt, arr):
        nonlocal off
        b = np.ascontiguousarray(arr).view(np.uint8).reshape(-1)
        isz = {"F32": 4, "F16": 2, "BF16": 2, "F8_E4M3": 1, "F8_E5M2": 1}[dt]
        ents[name] = {"dtype": dt, "shape": [b.size // isz], "data_offsets": [off, off + b.size]}
        parts.append(b.tobytes())
        off += b.size

    all16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    add("f16_all", "F16", all16)
    add("bf16_all", "BF16", all16)
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0, 1, 0x0FFF, 0x1000, 0x1001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    add("f32_grid", "F32", (hi[:, None] | lows[None, :]).reshape(-1))
    add("f32_rand", "F32", rng.integers(0, 1 << 32, size=1 << 18, dtype=np.uint64).astype(np.uint32))
    all8 = np.arange(256, dtype=np.uint8)
    scales = [1.0, 0.5, 2.0 ** -7, 1024.0, 0.0371, float(np.float32(rng.uniform(1e-3, 1e-1))), 3.0e-39,
              1.7e38, 0.0, -0.25, float("nan"), float("inf"), float("-inf")]
    for fmt in ("F8_E4M3", "F8_E5M2"):
        add(f"{fmt}.raw.weight", fmt, all8)
        for j, s in enumerate(scales):
            # 767 values: the second copy is shifted by one, so every pattern
            # lands in both halves of an element pair
            add(f"{fmt}.s{j}.weight", fmt, np.concatenate([all8, all8[1:], all8]))
            add(f"{fmt}.s{j}.scale_weight", "F32", np.array([s], dtype=np.float32).view(np.uint32))
            ents[f"{fmt}.s{j}.scale_weight"]["shape"] = []
    return image_of(ents, b"".join(parts), pad=3)


@pytest.mark.parametrize("dst", ["BF16", "F16", "F32"])
@pytest.mark.parametrize("packed", [False, True])
@pytest.mark.parametrize("kernel", [1, 2, 3, 4])
def test_every_bit_pattern(stmat, oracle, dst, packed, kernel):
    img = special_image()
    sfx = (".weight", ".scale_weight")
    plan, outs, _ = run(stmat, img, dst=dst, scale_suffix=sfx, packed=packed, kernel=kernel)
    assert plan.stats()["kernel"] == {1: "stream", 2: "latency", 3: "tma", 4: "tma_wide"}[kernel]
    sel, want = oracle_all(oracle, img, dst=dst, scale_suffix=sfx)
    assert_same(plan, outs, sel, want)


# ------------------------------------------------------- alignment sweep

def sweep_image(residue_pad, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    dts = ["F32", "F16", "BF16", "F8_E4M3", "F8_E5M2", "I64", "BOOL", "U8", "I32"]
    isz = {"F32": 4, "F16": 2, "BF16": 2, "F8_E4M3": 1, "F8_E5M2": 1, "I64": 8, "BOOL": 1, "U8": 1, "I32": 4}
    ents, parts, off = {}, [], 0
    lengths = [1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257,
               511, 1000, 4095, 4096, 4097, 12345, 100003]
    i = 0
    for n in lengths:
        for dt in dts:
            raw = rng.integers(0, 256, size=n * isz[dt], dtype=np.uint8)
            if dt == "BOOL":
                raw = raw & 1
            ents[f"t{i:04d}"] = {"dtype": dt, "shape": [n], "data_offsets": [off, off + raw.size]}
            parts.append(raw.tobytes())
            off += raw.size
            i += 1
            # a one-byte tensor between others shifts every later start by one
            ents[f"t{i:04d}"] = {"dtype": "U8", "shape": [1], "data_offsets": [off, off + 1]}
            parts.append(bytes([i & 255]))
            off += 1
            i += 1
    return image_of(ents, b"".join(parts), pad=residue_pad)


@pytest.mark.parametrize("residue", list(range(16)))
def test_alignment_sweep(stmat, oracle, residue):
    """Every class at every source misalignment (1-byte spacers shift the
    starts; the device copy is offset by `residue`) into 256-byte-aligned and
    into packed (itemsize-aligned) outputs."""
    img = sweep_image(residue % 8, seed=residue)
    for dst in ("BF16", "F16", "F32", "KEEP"):
        sel, want = oracle_all(oracle, img, dst=dst)
        for packed in (False, True):
            for kernel in (1, 2, 3, 4):
                plan, outs, _ = run(stmat, img, dst=dst, offset=residue, packed=packed,
                                    workers=[0, 7, 333][residue % 3], kernel=kernel)
                assert_same(plan, outs, sel, want)


def test_data_section_edges(stmat, oracle):
    """Misaligned tensors that start at the first byte and end at the last
    byte of an unaligned, exactly sized device data section."""
    rng = np.random.Generator(np.random.PCG64(5))
    for n0, n1 in [(1, 1), (33, 70), (1000, 4097), (17, 3)]:
        a = rng.integers(0, 1 << 32, size=n0, dtype=np.uint64).astype(np.uint32)
        b = rng.integers(0, 1 << 16, size=n1, dtype=np.uint64).astype(np.uint16)
        ents = {"first": {"dtype": "F32", "shape": [n0], "data_offsets": [0, 4 * n0]},
                "last": {"dtype": "F16", "shape": [n1], "data_offsets": [4 * n0, 4 * n0 + 2 * n1]}}
        img = image_of(ents, a.tobytes() + b.tobytes())
        sel, want = oracle_all(oracle, img, dst="BF16")
        ix = stmat.Index.from_file(img)
        data = img[8 + ix.sizes()[0]:]
        for kernel in (1, 2, 3, 4):
            plan = ix.plan(dst="BF16", kernel=kernel)
            for shift in (1, 5, 9, 15):
                buf = torch.zeros(data.size + 32, dtype=torch.uint8, device="cuda")
                buf[shift:shift + data.size].copy_(torch.from_numpy(data.copy()))
                outs = GuardedOutputs(plan)
                plan.materialize(buf.data_ptr() + shift, outs.ptrs)
                torch.cuda.synchronize()
                assert plan.check() == 0
                assert_same(plan, outs, sel, want)


# ------------------------------------------------------------- workloads

def workload_case(stmat, oracle, name, kernel=0):
    """A whole workload through run() (guard-banded outputs, source checked
    unchanged), every element against the oracle on all host cores."""
    from safetensors_materialization_gb300 import synth
    w = synth.WORKLOADS[name]()
    lay = w.files[0]
    img = synth.build_workload_file(w, 0)
    dst = w.dst[0]
    plan, outs, buf = run(stmat, img, dst=dst, view=w.view, scale_suffix=w.scale_suffix,
                          whole=w.whole_file_on_device, kernel=kernel)
    sel = w.view(oracle.parse_header(lay.header, lay.data_bytes)).select(dst=dst, scale_suffix=w.scale_suffix)
    assert [o["name"] for o in plan.outputs()] == [o["name"] for o in sel.outputs()]
    assert compare_full(sel, img[lay.data_start:], {f"kernel {kernel}": outs}) == \
        sum(o["bytes"] for o in sel.outputs())
    return plan, outs, buf, lay, img


def test_tiny_workload_full(stmat, oracle):
    workload_case(stmat, oracle, "tiny")


@pytest.mark.parametrize("kernel", [0, 2])
def test_stress_workload_full(stmat, oracle, kernel):
    """100k tensors, 7 dtypes, every source 1-15 bytes off 16-byte alignment."""
    workload_case(stmat, oracle, "stress", kernel=kernel)


def joined(stmat, oracle, w, align=256):
    """Every shard of `w` under one joined index (library and oracle) and one
    host arena holding each shard's data section at its base."""
    from safetensors_materialization_gb300 import synth
    ix, bases = stmat.Index.concat([stmat.Index.from_header(l.header, l.data_bytes) for l in w.files], align)
    oix, obases = oracle.concat([oracle.parse_header(l.header, l.data_bytes) for l in w.files], align)
    assert bases == obases
    arena = np.zeros(ix.sizes()[1], np.uint8)
    for k, lay in enumerate(w.files):
        synth.build_workload_data(w, k, arena[bases[k]:bases[k] + lay.data_bytes])
    return ix, oix, arena


@pytest.mark.parametrize("align", [1, 256])
@pytest.mark.parametrize("kernel", [1, 2, 3])
def test_joined_shards_one_launch(stmat, oracle, align, kernel):
    """A 4-shard checkpoint joined into one arena and materialized by one
    launch; align=1 packs the shards back to back, so later shards' sources
    lose their alignment."""
    from safetensors_materialization_gb300 import synth
    w = synth.llm8b(seed=5, layers=4, hidden=256, inter=704, vocab=1000, kv=64, shards=4)
    ix, oix, arena = joined(stmat, oracle, w, align)
    dev = torch.from_numpy(arena).cuda()
    for dst in ("BF16", "F16", "F32"):
        plan = ix.plan(dst=dst, kernel=kernel)
        assert plan.stats()["chunks"] == 1
        outs = GuardedOutputs(plan)
        plan.materialize(dev.data_ptr(), outs.ptrs)
        torch.cuda.synchronize()
        assert plan.check() == 0
        sel = oix.select(dst=dst)
        assert_same(plan, outs, sel, [sel.materialize(i, arena) for i in range(len(sel))])


# ------------------------------------------------------ pipeline and misc

@pytest.mark.parametrize("chunk", [1 << 20, 48 << 20])
def test_load_pipeline_matches_materialize(stmat, oracle, chunk):
    """st_load (chunked pinned H2D copies overlapped with per-chunk kernels)
    produces the oracle's bytes."""
    from safetensors_materialization_gb300 import synth
    w = synth.stress()
    lay = w.files[0]
    img = synth.build_workload_file(w, 0)
    ix = stmat.Index.from_file(img)
    plan = ix.plan(dst="BF16", chunk_bytes=chunk)
    assert plan.stats()["chunks"] == (lay.data_bytes + chunk - 1) // chunk
    host = torch.from_numpy(img[lay.data_start:].copy()).pin_memory()
    dev = torch.empty(lay.data_bytes, dtype=torch.uint8, device="cuda")
    outs = GuardedOutputs(plan)
    copy = torch.cuda.Stream()
    plan.load(host, dev, outs.ptrs, copy_stream=copy, compute_stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert plan.check() == 0
    outs.check_guards()
    sel = oracle.parse_header(lay.header, lay.data_bytes).select(dst="BF16")
    assert compare_full(sel, img[lay.data_start:], {f"chunk {chunk}": outs}) == sum(o["bytes"] for o in sel.outputs())
    assert torch.equal(dev.cpu(), host)


def test_stage_h2d(stmat):
    src = torch.randint(0, 256, (10_000_019,), dtype=torch.uint8).pin_memory()
    dst = torch.zeros_like(src, device="cuda")
    ev = torch.cuda.Event()
    stmat.stage_h2d(dst, src, src.numel(), chunk_bytes=1 << 20, done_event=ev)
    ev.synchronize()
    assert torch.equal(dst.cpu(), src)


def test_scale_override(stmat, oracle):
    img = special_image()
    sfx = (".weight", ".scale_weight")
    ix = stmat.Index.from_file(img)
    plan = ix.plan(dst="BF16", scale_suffix=sfx)
    hlen = ix.sizes()[0]
    buf, data_ptr = to_device(img, 0, True, 8 + hlen)
    outs = GuardedOutputs(plan)
    scales = torch.full((len(plan),), 0.125, dtype=torch.float32, device="cuda")
    plan.materialize(data_ptr, outs.ptrs, scales=scales)
    torch.cuda.synchronize()
    for i, o in enumerate(plan.outputs()):
        if o["src_dtype"] in ("F8_E4M3", "F8_E5M2"):
            raw = img[8 + hlen + o["begin"]:8 + hlen + o["begin"] + o["numel"]]
            want = oracle.convert(o["src_dtype"], "BF16", raw, scale=0.125)
            assert np.array_equal(outs.raw(i).cpu().numpy(), want), o["name"]
    outs.check_guards()


def test_bad_destinations_are_flagged_and_skipped(stmat, oracle):
    g, f = small_file()
    img = np.frombuffer(f, dtype=np.uint8).copy()
    ix = stmat.Index.from_file(img)
    plan = ix.plan(dst="BF16")
    buf, data_ptr = to_device(img, 0, True, 8 + ix.sizes()[0])
    outs = GuardedOutputs(plan)
    outs.arena.fill_(0xA5)
    ptrs = outs.ptrs.clone()
    ptrs[0] = 0                      # NULL destination for "a"
    ptrs[1] = outs.ptrs[1] + 1       # odd address for the BF16 output "b"
    plan.materialize(data_ptr, ptrs)
    torch.cuda.synchronize()
    assert plan.check() == 1
    assert plan.check() == 0         # reading clears the flags
    assert torch.all(outs.arena[:outs.offsets[2]] == 0xA5)   # nothing written for "a" or "b"
    sel, want = oracle_all(oracle, img, dst="BF16")
    for i in range(2, len(want)):
        assert np.array_equal(outs.raw(i).cpu().numpy(), want[i])


def test_empty_cases(stmat):
    img = image_of({}, b"")
    ix = stmat.Index.from_file(img)
    plan = ix.plan(dst="BF16")
    assert len(plan) == 0 and plan.stats()["pieces"] == 0
    scratch = torch.zeros(16, dtype=torch.uint8, device="cuda")
    plan.materialize(scratch, torch.zeros(1, dtype=torch.int64, device="cuda"))  # no work, no launch
    ents = {"z": {"dtype": "F32", "shape": [0], "data_offsets": [0, 0]},
            "s": {"dtype": "F16", "shape": [], "data_offsets": [0, 2]}}
    img = image_of(ents, b"\x00\x3c")
    plan, outs, _ = run(stmat, img, dst="F32")
    assert outs.raw(1).cpu().numpy().view(np.float32)[0] == 1.0


# ---------------------------------------------------------------- slicing

def sliced_image(seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    shapes = [[64, 300], [9, 40, 33], [3, 5, 7, 11], [512, 96], [2, 7000], [12], [33, 17]]
    dts = ["F32", "F16", "F8_E4M3", "BF16", "I64", "F8_E5M2", "BOOL"]
    isz = {"F32": 4, "F16": 2, "BF16": 2, "F8_E4M3": 1, "F8_E5M2": 1, "I64": 8, "BOOL": 1}
    ents, parts, off = {}, [], 0
    for i, (shp, dt) in enumerate(zip(shapes, dts)):
        n = int(np.prod(shp))
        raw = rng.integers(0, 256, size=n * isz[dt], dtype=np.uint8)
        if dt == "BOOL":
            raw &= 1
        ents[f"s{i}"] = {"dtype": dt, "shape": shp, "data_offsets": [off, off + raw.size]}
        parts.append(raw.tobytes())
        off += raw.size
    return image_of(ents, b"".join(parts), pad=5), shapes, rng


def test_data_section_in_host_memory(stmat, oracle):
    """A data section in page-locked host memory, which the kernel reads over
    the host link: the register builds materialize it exactly (the L2
    prefetch of small plans, which targets only this GPU's memory, is left
    out), and the TMA builds refuse it with ST_E_INVAL before any launch."""
    g, f = small_file()
    img = np.frombuffer(f, dtype=np.uint8).copy()
    host = torch.empty(img.size, dtype=torch.uint8, pin_memory=True)
    host.numpy()[:] = img
    ix = stmat.Index.from_file(img)
    hlen, _ = ix.sizes()
    data_ptr = host.data_ptr() + 8 + hlen
    suffix = (".weight", ".scale_weight")
    sel, expected = oracle_all(oracle, img, dst="BF16", scale_suffix=suffix)
    for kernel in (1, 2):
        plan = ix.plan(dst="BF16", scale_suffix=suffix, kernel=kernel)
        outs = GuardedOutputs(plan)
        plan.materialize(data_ptr, outs.ptrs)
        torch.cuda.synchronize()
        assert plan.check() == 0
        assert_same(plan, outs, sel, expected)
    for kernel in (3, 4):
        plan = ix.plan(dst="BF16", scale_suffix=suffix, kernel=kernel)
        outs = GuardedOutputs(plan)
        with pytest.raises(stmat.StmatError) as e:
            plan.materialize(data_ptr, outs.ptrs)
        assert e.value.status == "ST_E_INVAL"
        outs.check_guards()
    assert np.array_equal(host.numpy(), img)


@pytest.mark.parametrize("kernel", [1, 2, 3, 4])
def test_sliced_outputs(stmat, oracle, kernel):
    """Slices on every dimension (contiguous and strided runs) at misaligned
    sources, into aligned and packed outputs."""
    img, shapes, rng = sliced_image(21 + kernel)
    names = [f"s{i}" for i in range(len(shapes))]
    ix = stmat.Index.from_file(img)
    hlen = ix.sizes()[0]
    oix = oracle.parse(img)
    data = img[8 + hlen:]
    for trial in range(8):
        slices = []
        for shp in shapes:
            d = int(rng.integers(0, len(shp)))
            a = int(rng.integers(0, shp[d]))
            slices.append((d, a, int(rng.integers(a, shp[d] + 1))))
        dst = ["BF16", "F16", "F32", "KEEP"][trial % 4]
        sel = oix.select(dst=dst, names=names, slices=slices)
        want = [sel.materialize(i, data) for i in range(len(sel))]
        plan = ix.plan(dst=dst, names=names, slices=slices, kernel=kernel, unit_bytes=[2048, 32768][trial % 2])
        buf, data_ptr = to_device(img, trial % 16, True, 8 + hlen)
        outs = Packed(plan) if trial % 3 == 0 else GuardedOutputs(plan)
        plan.materialize(data_ptr, outs.ptrs)
        torch.cuda.synchronize()
        assert plan.check() == 0
        assert [o["shape"] for o in plan.outputs()] == [o["shape"] for o in sel.outputs()]
        assert_same(plan, outs, sel, want)


def test_tensor_parallel_shard_load(stmat, oracle):
    """Rank 0 of 4 tensor-parallel ranks of an LLM shard file at full size:
    every sliced output equals torch's slice of the source tensor (a byte
    copy) and, every element, the oracle's."""
    from safetensors_materialization_gb300 import synth
    w = synth.llm8b_tp4()
    lay = w.files[0]
    img = synth.build_workload_file(w, 0)
    ix = stmat.Index.from_file(img)
    names = [e["name"] for e in ix.entries()]
    slices = [w.slices.get(n) for n in names]
    plan = ix.plan(dst="BF16", names=names, slices=slices)
    buf, data_ptr = to_device(img, 0, False, lay.data_start)
    outs = GuardedOutputs(plan)
    plan.materialize(data_ptr, outs.ptrs)
    torch.cuda.synchronize()
    assert plan.check() == 0
    ents = {e["name"]: e for e in ix.entries()}
    for i, o in enumerate(plan.outputs()):
        e = ents[o["name"]]
        src = buf[e["begin"]:e["end"]].view(torch.bfloat16).view(e["shape"])
        if o["slice"]:
            d, a, b = o["slice"]
            src = src.narrow(d, a, b - a)
        assert torch.equal(outs.tensor(i).view(torch.int16), src.contiguous().view(torch.int16)), o["name"]
    oix = oracle.parse(img)
    sel = oix.select(dst="BF16", names=names, slices=slices)
    outs.check_guards()
    assert compare_full(sel, img[lay.data_start:], {"tp rank 0": outs}) == sum(o["bytes"] for o in plan.outputs())


@pytest.mark.parametrize("name", ["unet_small", "stress"])
def test_partition_parts_load_only_their_bytes(stmat, oracle, name):
    """The multi-GPU split on one GPU: each of 3 parts (st_selection.part /
    n_parts) is loaded by st_load from pinned host memory into a device data
    buffer that holds garbage everywhere else; a part copies only its own
    byte ranges (st_plan_copy_range), and its outputs equal the oracle's
    selection of the same part, every element."""
    from safetensors_materialization_gb300 import synth
    w = synth.WORKLOADS[name]()
    lay = w.files[0]
    img = synth.build_workload_file(w, 0)
    data = img[lay.data_start:]
    ix = w.view(stmat.Index.from_header(lay.header, lay.data_bytes))
    oix = w.view(oracle.parse_header(lay.header, lay.data_bytes))
    host = torch.from_numpy(data.copy()).pin_memory()
    names = []
    for part in range(3):
        plan = ix.plan(dst="BF16", part=part, n_parts=3, chunk_bytes=64 << 20)
        ranges = plan.copy_ranges()
        assert sum(b - a for a, b in ranges) == plan.copy_bytes()[0] < lay.data_bytes
        dev = torch.full((lay.data_bytes,), 0x7F, dtype=torch.uint8, device="cuda")
        outs = GuardedOutputs(plan)
        plan.load(host, dev, outs.ptrs, copy_stream=torch.cuda.Stream(), compute_stream=torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert plan.check() == 0
        outs.check_guards()
        copied = torch.zeros(lay.data_bytes, dtype=torch.bool, device="cuda")
        for a, b in ranges:
            copied[a:b] = True
            assert torch.equal(dev[a:b], host[a:b].cuda())
        assert torch.all(dev[~copied] == 0x7F)              # nothing outside the ranges was copied
        sel = oix.select(dst="BF16", part=part, nparts=3)
        assert compare_full(sel, data, {f"part {part}": outs}) == sum(o["bytes"] for o in sel.outputs())
        names += [o["name"] for o in plan.outputs()]
    assert names == [o["name"] for o in oix.select(dst="BF16").outputs()]   # the parts cover every output once


@pytest.mark.parametrize("kernel", [1, 3, 4])
def test_claimed_tail_on_every_launch(stmat, oracle, kernel):
    """Warps claim a plan's tail through two words that the last warp of each
    launch zeroes: five launches of one plan in a row (and a chunked st_load
    whose chunk launches share the words) each produce every output, equal to
    the oracle's, with the arena cleared in between."""
    img = sweep_image(3, seed=40 + kernel)
    ix = stmat.Index.from_file(img)
    hlen = ix.sizes()[0]
    sel, want = oracle_all(oracle, img, dst="BF16")
    buf, data_ptr = to_device(img, 0, True, 8 + hlen)
    plan = ix.plan(dst="BF16", kernel=kernel, workers=64, unit_bytes=2048)
    st = plan.stats()
    tail = plan.worker(0, st["workers"])
    assert tail[1] > tail[0], "the plan has a claimed tail"
    outs = GuardedOutputs(plan)
    for _ in range(5):
        outs.arena.fill_(0xA5)
        plan.materialize(data_ptr, outs.ptrs)
        torch.cuda.synchronize()
        assert plan.check() == 0
        assert_same(plan, outs, sel, want)
    data = img[8 + hlen:]
    chunked = ix.plan(dst="BF16", kernel=kernel, workers=64, unit_bytes=2048, chunk_bytes=1 << 16)
    cst = chunked.stats()
    assert cst["chunks"] > 1 and any(chunked.worker(c, cst["workers"])[1] > chunked.worker(c, cst["workers"])[0]
                                     for c in range(cst["chunks"]))
    host = torch.from_numpy(data.copy()).pin_memory()
    dev = torch.empty(data.size, dtype=torch.uint8, device="cuda")
    couts = GuardedOutputs(chunked)
    for _ in range(2):
        couts.arena.fill_(0xA5)
        chunked.load(host, dev, couts.ptrs, copy_stream=torch.cuda.Stream(), compute_stream=torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert chunked.check() == 0
        assert_same(chunked, couts, sel, want)
