"""The allocation-free entry point (st_materialize_noalloc), through the C ABI.

Some callers cannot allocate device memory: a plugin running inside an
application whose device memory is all held by that application's own pool,
or code that must not allocate once it runs because cudaMalloc can block and
fail where nothing can recover.  For them the plan is built host-only and its
tables go into the library's static device scratch.  Its output must equal
the regular entry point's (st_materialize) and the oracle's byte for byte
(the tolerance of every parity test here: 0 ULP) on two calls in a row that
reuse the scratch with different plans; free device memory must not change
across a call; the scratch's error word must report a skipped destination
through st_static_check.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import json
import struct

import numpy as np
import pytest

from oracle_compare import GuardedOutputs

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
    """(device copy of the image, data pointer, host-only plan, device plan)."""
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


def test_noalloc_matches_materialize_and_oracle_on_two_calls(stmat, oracle):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    stream = torch.cuda.current_stream()
    specs = [(mixed_image(1, 300), "BF16", sms * 3 * 8, 0),
             (mixed_image(2, 120), "F32", sms * 6 * 8, 0),
             (mixed_image(3, 200), "F16", sms * 2 * 8, 3)]
    cases = [case(stmat, img, dst, workers, kernel) for img, dst, workers, kernel in specs]
    # a first call of every plan on this device (the library's one-time set-up
    # and the first launch of each kernel build, which may load its code onto
    # the device), then every buffer the calls below use
    for buf, data, host_plan, dev_plan in cases:
        warm = GuardedOutputs(host_plan)
        host_plan.materialize_noalloc(data, warm.ptrs, stream=stream)
        torch.cuda.synchronize()
        del warm
    results = [GuardedOutputs(host_plan) for _, _, host_plan, _ in cases]
    torch.cuda.synchronize()
    assert stmat.static_check(stream) == 0
    free0 = torch.cuda.mem_get_info()[0]
    for (buf, data, host_plan, dev_plan), outs in zip(cases, results):
        host_plan.materialize_noalloc(data, outs.ptrs, stream=stream)   # no sync between the calls
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "free device memory changed across the calls"
    assert stmat.static_check(stream) == 0
    for (img, dst, _, _), (buf, data, host_plan, dev_plan), outs in zip(specs, cases, results):
        outs.check_guards()
        ref = GuardedOutputs(dev_plan)
        dev_plan.materialize(data, ref.ptrs, stream=stream)
        torch.cuda.synchronize()
        assert dev_plan.check() == 0
        assert [o["name"] for o in host_plan.outputs()] == [o["name"] for o in dev_plan.outputs()]
        oix = oracle.parse(img)
        sel = oix.select(dst=dst)
        data_host = img[8 + oix.header_len:]
        for i in range(len(ref.infos)):
            assert torch.equal(outs.raw(i), ref.raw(i)), host_plan.output(i)["name"]
            assert np.array_equal(outs.raw(i).cpu().numpy(), sel.materialize(i, data_host)), \
                host_plan.output(i)["name"]


def test_noalloc_reports_a_skipped_destination(stmat):
    """A NULL destination is skipped and its flag stays in the scratch's
    error word until st_static_check reads (and clears) it; the other
    outputs are still written."""
    buf, data, host_plan, dev_plan = case(stmat, mixed_image(5, 40), "BF16", 1024)
    outs = GuardedOutputs(host_plan)
    ref = GuardedOutputs(dev_plan)
    dev_plan.materialize(data, ref.ptrs)
    ptrs = outs.ptrs.clone()
    ptrs[3] = 0
    stream = torch.cuda.current_stream()
    host_plan.materialize_noalloc(data, ptrs, stream=stream)
    host_plan.materialize_noalloc(data, outs.ptrs, stream=stream)   # a clean call does not clear it
    assert stmat.static_check(stream) == 1
    assert stmat.static_check(stream) == 0
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
