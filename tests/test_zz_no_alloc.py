"""The allocation-free entry point (st_materialize_noalloc) against the
regular one (st_materialize), through the C ABI.

st_materialize_noalloc serves callers that cannot allocate device memory
(a stream capture that forbids cudaMalloc, or device memory fully held by
another allocator): the plan is built host-only and its tables go into the
library's static device scratch.  Its output must equal st_materialize's
byte for byte (the same tolerance as every parity test here: 0 ULP), also on
two calls in a row that reuse the scratch with different plans.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import json
import struct

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def mixed_image(seed, n):
    """n tensors of mixed dtypes and lengths, most of them at misaligned offsets."""
    rng = np.random.Generator(np.random.PCG64(seed))
    isz = {"F32": 4, "F16": 2, "BF16": 2, "F8_E4M3": 1, "F8_E5M2": 1, "I64": 8, "BOOL": 1}
    dts = list(isz)
    ents, parts, off = {}, [], 0
    for i in range(n):
        dt = dts[int(rng.integers(0, len(dts)))]
        cnt = int(rng.integers(1, 9000))
        raw = rng.integers(0, 256, size=cnt * isz[dt], dtype=np.uint8)
        if dt == "BOOL":
            raw &= 1
        ents[f"w.{i:04d}"] = {"dtype": dt, "shape": [cnt], "data_offsets": [off, off + raw.size]}
        parts.append(raw.tobytes())
        off += raw.size
    h = json.dumps(ents).encode() + b" " * 5
    return np.frombuffer(struct.pack("<Q", len(h)) + h + b"".join(parts), dtype=np.uint8).copy()


def case(stmat, image, dst, workers, kernel=0):
    """(device data pointer holder, host-only plan, device plan, outputs for each)."""
    ix = stmat.Index.from_file(image)
    hlen, dbytes = ix.sizes()
    buf = torch.empty(image.size + 16, dtype=torch.uint8, device="cuda")
    buf[:image.size].copy_(torch.from_numpy(image))
    data = buf.data_ptr() + 8 + hlen          # keeps the file's misalignment
    host_plan = ix.plan(dst=dst, workers=workers, host_only=True, kernel=kernel)
    dev_plan = ix.plan(dst=dst)
    return buf, data, host_plan, dev_plan


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def test_noalloc_matches_materialize_on_two_calls(stmat):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    stream = torch.cuda.current_stream()
    cases = [case(stmat, mixed_image(1, 300), "BF16", sms * 3 * 8),
             case(stmat, mixed_image(2, 120), "F32", sms * 6 * 8),
             case(stmat, mixed_image(3, 200), "F16", sms * 2 * 8, kernel=3)]
    results = []
    for buf, data, host_plan, dev_plan in cases:
        outs = stmat.Outputs(host_plan)
        outs.arena.fill_(0x5A)
        host_plan.materialize_noalloc(data, outs.ptrs, stream=stream)   # no sync between the two calls
        results.append(outs)
    torch.cuda.synchronize()
    for (buf, data, host_plan, dev_plan), outs in zip(cases, results):
        ref = stmat.Outputs(dev_plan)
        dev_plan.materialize(data, ref.ptrs, stream=stream)
        torch.cuda.synchronize()
        assert dev_plan.check() == 0
        assert [o["name"] for o in host_plan.outputs()] == [o["name"] for o in dev_plan.outputs()]
        for i in range(len(ref.infos)):
            assert torch.equal(outs.raw(i), ref.raw(i)), host_plan.output(i)["name"]


def test_noalloc_rejects_a_plan_larger_than_its_scratch(stmat):
    """A plan whose tables exceed the 4 MiB static scratch is refused on the
    host before anything is queued (so the small stand-in buffers below are
    never touched)."""
    from safetensors_materialization_gb300 import synth
    lay = synth.stress().files[0]
    ix = stmat.Index.from_header(lay.header, lay.data_bytes)
    big = ix.plan(dst="BF16", workers=7296, unit_bytes=1024, host_only=True)
    assert big.stats()["pieces"] * 48 > 4 << 20
    data = torch.zeros(16, dtype=torch.uint8, device="cuda")
    ptrs = torch.zeros(1, dtype=torch.int64, device="cuda")
    with pytest.raises(stmat.StmatError) as e:
        big.materialize_noalloc(data, ptrs)
    assert e.value.status == "ST_E_INVAL"
    assert "static scratch" in str(e.value)


def test_noalloc_under_stream_capture(stmat):
    """Captured into a CUDA graph (after a first call outside the capture, as
    the header asks) and replayed: the outputs equal st_materialize's.  The
    captured table copies read the plan's host memory when the graph runs."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    buf, data, host_plan, dev_plan = case(stmat, mixed_image(4, 250), "BF16", sms * 3 * 8)
    outs = stmat.Outputs(host_plan)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        host_plan.materialize_noalloc(data, outs.ptrs, stream=side)
    torch.cuda.synchronize()
    ref = stmat.Outputs(dev_plan)
    dev_plan.materialize(data, ref.ptrs)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        host_plan.materialize_noalloc(data, outs.ptrs, stream=torch.cuda.current_stream())
    for _ in range(2):
        outs.arena.fill_(0x5A)
        graph.replay()
        torch.cuda.synchronize()
        for i in range(len(ref.infos)):
            assert torch.equal(outs.raw(i), ref.raw(i)), host_plan.output(i)["name"]
