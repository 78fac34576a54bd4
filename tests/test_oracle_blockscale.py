"""Pins for the oracle's block-scaled weights (CPU only).

The pages name the formats only (block-FP8 and NVFP4 checkpoints, "Current
Backend Boundary" of the resident-LLM architecture page); the layouts are the
readings stated in the oracle.  Pinned here against:
  - the OCP MX E2M1 value table (all 16 codes) and the nibble order;
  - the separately pinned per-tensor scaled-FP8 path: block FP8 with every
    block scale equal to s gives the same bytes as one per-tensor scale s;
  - an independent reconstruction: torch's float8 decode, numpy broadcasting
    of the block scales, numpy binary32 products and torch's rounding to the
    output dtype, on ragged shapes;
  - hand-worked examples (tests/golden/blockscale.json);
  - the invalid forms and their status.
"""
import json
import struct

import numpy as np
import pytest

from conftest import golden

torch = pytest.importorskip("torch")

# OCP Microscaling Formats (MX) v1.0, FP4 E2M1: codes 0..7 and their negatives.
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def image(ents_data):
    """File image from [(name, dtype, shape, raw bytes)]."""
    ents, parts, off = {}, [], 0
    for name, dt, shape, raw in ents_data:
        ents[name] = {"dtype": dt, "shape": list(shape), "data_offsets": [off, off + len(raw)]}
        parts.append(raw)
        off += len(raw)
    h = json.dumps(ents).encode()
    return np.frombuffer(struct.pack("<Q", len(h)) + h + b"".join(parts), dtype=np.uint8).copy()


def run(oracle, img, name, dst, quant):
    ix = oracle.parse(img)
    sel = ix.select(names=[name], dst=dst, quant=[quant])
    return sel, sel.materialize(0, img[8 + ix.header_len:])


def as_dtype(raw, dst):
    return raw.view({"F32": np.float32, "F16": np.uint16, "BF16": np.uint16}[dst])


def to_dst_bits(x32, dst):
    """Reference rounding of binary32 values to the output dtype (torch CPU),
    NaN as the canonical quiet NaN."""
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32))
    if dst == "F32":
        out = t.view(torch.int32).numpy().view(np.uint32).copy()
        out[np.isnan(x32)] = 0x7FC00000
        return out
    out = t.to(torch.bfloat16 if dst == "BF16" else torch.float16).view(torch.int16).numpy().view(np.uint16).copy()
    out[np.isnan(x32)] = 0x7FC0 if dst == "BF16" else 0x7E00
    return out


def test_e2m1_table_and_nibble_order(oracle):
    # every byte: element 2c is the low nibble, 2c+1 the high nibble; scales 1.0
    w = np.arange(256, dtype=np.uint8)
    M, K = 8, 32
    img = image([("w", "U8", [M, K], w.tobytes()),
                 ("s", "F8_E4M3", [M, 4], bytes([0x38]) * (M * 4)),
                 ("g", "F32", [], struct.pack("<f", 1.0))])
    _, out = run(oracle, img, "w", "F32", ("nvfp4", "s", "g", None))
    vals = out.view(np.float32)
    want = np.array([[E2M1[b & 15], E2M1[b >> 4]] for b in range(256)], dtype=np.float32).reshape(-1)
    assert np.array_equal(vals.view(np.uint32), want.view(np.uint32))   # -0.0 kept


@pytest.mark.parametrize("dst", ["BF16", "F16", "F32"])
@pytest.mark.parametrize("fmt", ["F8_E4M3", "F8_E5M2"])
def test_uniform_blocks_equal_the_per_tensor_scale(oracle, dst, fmt):
    rng = np.random.Generator(np.random.PCG64(3))
    M, N = 37, 70
    w = rng.integers(0, 256, size=M * N, dtype=np.uint8).tobytes()
    for s in (1.0, 0.0123, 3.5e-3, 448.0, 1e-30, 7.0e30):
        sc = np.full((M + 15) // 16 * ((N + 31) // 32), s, dtype=np.float32)
        img = image([("w", fmt, [M, N], w), ("s", "F32", [(M + 15) // 16, (N + 31) // 32], sc.tobytes()),
                     ("t", "F32", [], struct.pack("<f", s))])
        _, got = run(oracle, img, "w", dst, ("block_fp8", "s", None, (16, 32)))
        ix = oracle.parse(img)
        per_tensor = ix.select(names=["w"], dst=dst, scale_names=["t"])
        assert np.array_equal(got, per_tensor.materialize(0, img[8 + ix.header_len:])), s


@pytest.mark.parametrize("dst", ["BF16", "F16", "F32"])
@pytest.mark.parametrize("shape,block", [((300, 260), (128, 128)), ((5, 48), (1, 16)), ((129, 17), (64, 16)),
                                         ((1, 1), (128, 128))])
def test_block_fp8_matches_reconstruction(oracle, dst, shape, block):
    rng = np.random.Generator(np.random.PCG64(shape[0] * 1000 + shape[1]))
    M, N = shape
    br, bc = block
    w = rng.integers(0, 256, size=M * N, dtype=np.uint8)
    SM, SN = -(-M // br), -(-N // bc)
    sc = (rng.uniform(1e-3, 1e-1, size=SM * SN) * rng.choice([1, -1, 1e20, 1e-20], size=SM * SN)).astype(np.float32)
    img = image([("w", "F8_E4M3", [M, N], w.tobytes()), ("s", "F32", [SM, SN], sc.tobytes())])
    _, got = run(oracle, img, "w", dst, ("block_fp8", "s", None, block))
    v = torch.from_numpy(w).view(torch.float8_e4m3fn).float().numpy().reshape(M, N)
    S = np.repeat(np.repeat(sc.reshape(SM, SN), br, axis=0), bc, axis=1)[:M, :N]
    x = (v.astype(np.float32) * S.astype(np.float32)).astype(np.float32).reshape(-1)
    assert np.array_equal(as_dtype(got, dst).view(to_dst_bits(x, dst).dtype), to_dst_bits(x, dst))


@pytest.mark.parametrize("dst", ["BF16", "F16", "F32"])
@pytest.mark.parametrize("M,N", [(4, 64), (3, 50), (17, 2), (64, 1024)])
def test_nvfp4_matches_reconstruction(oracle, dst, M, N):
    rng = np.random.Generator(np.random.PCG64(M * 7 + N))
    K = N // 2
    w = rng.integers(0, 256, size=M * K, dtype=np.uint8)
    SN = -(-N // 16)
    s8 = rng.integers(0, 256, size=M * SN, dtype=np.uint8)
    s8[(s8 & 0x7F) == 0x7F] = 0x38                        # NaN scales are tested below
    g = np.float32(rng.uniform(1e-4, 1.0))
    img = image([("w", "U8", [M, K], w.tobytes()), ("s", "F8_E4M3", [M, SN], s8.tobytes()),
                 ("g", "F32", [], g.tobytes())])
    sel, got = run(oracle, img, "w", dst, ("nvfp4", "s", "g", None))
    assert sel.output(0)["shape"] == [M, N]
    codes = np.stack([w & 15, w >> 4], axis=1).reshape(M, N)
    v = np.array(E2M1, dtype=np.float32)[codes]
    sb = torch.from_numpy(s8).view(torch.float8_e4m3fn).float().numpy().reshape(M, SN)
    s = (np.repeat(sb, 16, axis=1)[:, :N].astype(np.float32) * g).astype(np.float32)
    x = (v * s).astype(np.float32).reshape(-1)
    assert np.array_equal(as_dtype(got, dst).view(to_dst_bits(x, dst).dtype), to_dst_bits(x, dst))


def test_nan_scales_give_canonical_nan(oracle):
    img = image([("w", "U8", [1, 16], bytes([0x22]) * 16), ("s", "F8_E4M3", [1, 2], bytes([0x7F, 0x38])),
                 ("g", "F32", [], struct.pack("<f", 1.0))])
    _, got = run(oracle, img, "w", "BF16", ("nvfp4", "s", "g", None))
    bits = got.view(np.uint16)
    assert (bits[:16] == 0x7FC0).all() and (bits[16:] == 0x3F80).all()


@pytest.mark.parametrize("case", golden("blockscale.json")["cases"], ids=lambda c: c["name"])
def test_golden_blockscale(oracle, case):
    h = json.dumps(case["header"]).encode()
    img = np.frombuffer(struct.pack("<Q", len(h)) + h + bytes.fromhex(case["data_hex"]), dtype=np.uint8).copy()
    q = case["quant"]
    _, got = run(oracle, img, "w", case["dst"], (q[0], q[1], q[2], tuple(q[3]) if q[3] else None))
    bits = got.view(np.uint16)
    for k, hexv in case["expect"].items():
        assert int(bits[int(k)]) == int(hexv, 16), (case["why"], k)


def test_invalid_forms(oracle):
    fp8 = image([("w", "F8_E4M3", [4, 32], bytes(128)), ("s", "F32", [1, 1], struct.pack("<f", 1.0)),
                 ("s2", "F32", [1, 2], bytes(8)), ("h", "F16", [4, 32], bytes(256)),
                 ("u", "U8", [4, 16], bytes(64)), ("e", "F8_E4M3", [4, 2], bytes(8)),
                 ("g", "F32", [], bytes(4)), ("g2", "F32", [2], bytes(8))])
    ix = oracle.parse(fp8)

    def status(**kw):
        try:
            ix.select(**kw)
            return "OK"
        except oracle.OracleError as e:
            return e.status

    assert status(names=["w"], quant=[("block_fp8", "s", None, (128, 128))]) == "OK"
    assert status(names=["w"], quant=[("block_fp8", "s2", None, (128, 16))]) == "OK"
    assert status(names=["w"], quant=[("block_fp8", "s", None, (128, 8))]) == "INVAL"       # bc < 16
    assert status(names=["w"], quant=[("block_fp8", "s", None, (96, 128))]) == "INVAL"      # not a power of two
    assert status(names=["w"], quant=[("block_fp8", "s2", None, (128, 128))]) == "INVAL"    # scale shape
    assert status(names=["h"], quant=[("block_fp8", "s", None, None)]) == "INVAL"           # not fp8
    assert status(names=["w"], quant=[("block_fp8", "nope", None, None)]) == "NOT_FOUND"
    assert status(names=["w"], dst="KEEP", quant=[("block_fp8", "s", None, None)]) == "UNSUPPORTED_CAST"
    assert status(names=["w"], quant=[("block_fp8", "s", None, None)], slices=[(0, 0, 1)]) == "INVAL"
    assert status(names=["w"], quant=[("block_fp8", "s", None, None)], scale_names=["g"]) == "INVAL"
    assert status(names=["w"], quant=[("other", "s", None, None)]) == "INVAL"
    assert status(names=["u"], quant=[("nvfp4", "e", "g", None)]) == "OK"
    assert status(names=["u"], quant=[("nvfp4", "e", "g", (2, 16))]) == "INVAL"
    assert status(names=["u"], quant=[("nvfp4", "e", None, None)]) == "INVAL"               # no global scale
    assert status(names=["u"], quant=[("nvfp4", "e", "g2", None)]) == "INVAL"               # global not scalar
    assert status(names=["u"], quant=[("nvfp4", "s", "g", None)]) == "INVAL"                # scale dtype
    assert status(names=["w"], quant=[("nvfp4", "e", "g", None)]) == "INVAL"                # weight dtype
    # scale tensors are consumed: selecting everything with the pairing leaves them out
    sel = ix.select(names=["u", "e", "g"], quant=[("nvfp4", "e", "g", None), None, None])
    assert [o["name"] for o in sel.outputs()] == ["u"]
