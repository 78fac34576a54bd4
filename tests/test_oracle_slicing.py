"""Pins for the oracle's tensor slicing (CPU only): hand-computed sliced
outputs (tests/golden/slicing.json), equality with numpy's slicing of the
full output on generated tensors, and the invalid-slice status.

Slicing follows the TensorFrame slicing metadata of "Disk tier safetensors
streaming design audit (ComfyUI)", section "FastSageTensors (fastsafetensors)
capability audit": an output keeps [start, stop) along one dimension.
"""
import json
import struct

import numpy as np
import pytest

from conftest import golden

G = golden("slicing.json")


def small():
    h = G["header"].encode()
    return struct.pack("<Q", len(h)) + h + bytes.fromhex(G["data_hex"])


@pytest.mark.parametrize("case", G["cases"], ids=[f"{c['name']}-{c['slice']}-{c['dst']}" for c in G["cases"]])
def test_golden_slices(oracle, case):
    f = small()
    ix = oracle.parse(f)
    sel = ix.select(names=[case["name"]], dst=case["dst"], slices=[tuple(case["slice"])])
    o = sel.output(0)
    assert o["shape"] == case["shape"]
    data = np.frombuffer(f, dtype=np.uint8)[8 + ix.header_len:]
    assert sel.materialize(0, data).tobytes().hex() == case["hex"], case["why"]


@pytest.mark.parametrize("case", G["errors"], ids=[e["why"] for e in G["errors"]])
def test_invalid_slices(oracle, case):
    ix = oracle.parse(small())
    with pytest.raises(oracle.OracleError) as e:
        ix.select(names=[case["name"]], dst="BF16", slices=[tuple(case["slice"])])
    assert e.value.status == case["expect"]
    with pytest.raises(oracle.OracleError) as e:   # slices need explicit names
        ix.select(dst="BF16", slices=[(0, 0, 1), None])
    assert e.value.status == "INVAL"


def image(shapes, dts, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    isz = {"F32": 4, "F16": 2, "BF16": 2, "F8_E4M3": 1, "I64": 8}
    ents, parts, off = {}, [], 0
    for i, (shp, dt) in enumerate(zip(shapes, dts)):
        n = int(np.prod(shp))
        raw = rng.integers(0, 256, size=n * isz[dt], dtype=np.uint8)
        if dt == "F8_E4M3":
            raw[(raw & 0x7F) == 0x7F] = 0x11
        ents[f"x{i}"] = {"dtype": dt, "shape": list(shp), "data_offsets": [off, off + raw.size]}
        parts.append(raw.tobytes())
        off += raw.size
    h = json.dumps(ents).encode()
    return np.frombuffer(struct.pack("<Q", len(h)) + h + b"".join(parts), dtype=np.uint8).copy()


def test_slices_equal_numpy_slicing_of_the_full_output(oracle):
    """For every dimension and several ranges, the sliced output equals the
    full output (reshaped) sliced with numpy."""
    shapes = [[6, 5], [4, 3, 5], [2, 3, 4, 5], [7]]
    dts = ["F32", "F16", "F8_E4M3", "I64"]
    img = image(shapes, dts, 1)
    ix = oracle.parse(img)
    data = img[8 + ix.header_len:]
    rng = np.random.Generator(np.random.PCG64(2))
    for i, shp in enumerate(shapes):
        full = ix.select(names=[f"x{i}"], dst="F32" if dts[i] != "I64" else "KEEP")
        fo = full.output(0)
        isz = fo["bytes"] // fo["numel"]
        arr = full.materialize(0, data).view({4: np.uint32, 8: np.uint64}[isz]).reshape(shp)
        for d in range(len(shp)):
            for _ in range(3):
                a = int(rng.integers(0, shp[d] + 1))
                b = int(rng.integers(a, shp[d] + 1))
                sel = ix.select(names=[f"x{i}"], dst="F32" if dts[i] != "I64" else "KEEP", slices=[(d, a, b)])
                got = sel.materialize(0, data).view(arr.dtype)
                want = np.ascontiguousarray(np.take(arr, np.arange(a, b), axis=d)).reshape(-1)
                np.testing.assert_array_equal(got, want)
                assert sel.output(0)["shape"] == list(np.take(arr, np.arange(a, b), axis=d).shape)


def test_slice_windows_match_whole_output(oracle):
    img = image([[9, 7, 3]], ["BF16"], 3)
    ix = oracle.parse(img)
    data = img[8 + ix.header_len:]
    sel = ix.select(names=["x0"], dst="F32", slices=[(1, 2, 6)])
    whole = sel.materialize(0, data)
    n = sel.output(0)["numel"]
    for first, count in [(0, n), (5, 17), (11, 1), (n - 4, 4), (30, 0)]:
        np.testing.assert_array_equal(sel.materialize_range(0, data, first, count), whole[first * 4:(first + count) * 4])


def test_partition_counts_sliced_bytes(oracle):
    """The part rule weighs outputs by their sliced bytes."""
    img = image([[8, 4], [8, 4], [8, 4]], ["F32", "F32", "F32"], 4)
    ix = oracle.parse(img)
    names = ["x0", "x1", "x2"]
    slices = [(0, 0, 8), (0, 0, 1), (0, 0, 1)]   # 128, 16, 16 bytes as F32
    parts = [[o["name"] for o in ix.select(names=names, dst="F32", slices=slices, part=k, nparts=2).outputs()]
             for k in range(2)]
    assert parts == [["x0"], ["x1", "x2"]]
