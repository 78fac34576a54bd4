"""Pins for the oracle's element conversions (CPU only).

The oracle decodes every float format from its definition and rounds to
nearest, ties to even.  These tests tie it to things other than itself:
  * brute force: the result is the nearest value of the target format found
    by searching a table of all 65,536 bf16 / f16 values;
  * independent libraries on the CPU: torch's float8/bfloat16 casts and
    numpy's binary16 cast;
  * closed forms: fp8 x 2^k is exact in bf16/f16, special values from the
    IEEE 754 and OCP OFP8 definitions, textbook tie cases.
The scaled-fp8 reading (decode, one binary32 multiply by the per-tensor scale,
then round) follows the scaled-FP8 conversion named in "Disk tier safetensors
streaming design audit (ComfyUI)", section "ComfyUI load path + eager
materialization sites".
"""
import numpy as np
import pytest
import torch

CANON = {"BF16": 0x7FC0, "F16": 0x7E00, "F32": 0x7FC00000}
UINT = {"BF16": np.uint16, "F16": np.uint16, "F32": np.uint32}


def conv(O, src, out, bits, scale=None):
    raw = np.ascontiguousarray(bits).view(np.uint8)
    return O.convert(src, out, raw, scale).view(UINT[out])


def f32_sweep():
    """All 65,536 upper halves x low halves around every rounding position,
    plus random patterns."""
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x0FFF, 0x1000, 0x1001, 0x1FFF, 0x2000, 0x3000, 0x5000,
                     0x7FFF, 0x8000, 0x8001, 0xC000, 0xFFFF], dtype=np.uint32)
    grid = (hi[:, None] | lows[None, :]).reshape(-1)
    rnd = np.random.Generator(np.random.PCG64(12345)).integers(0, 1 << 32, size=1 << 20,
                                                                  dtype=np.uint64).astype(np.uint32)
    return np.concatenate([grid, rnd])


def table(fmt):
    """Positive finite values of a 16-bit format, sorted, with their patterns,
    followed by +inf placed at 2^(emax+1) (its pattern is even, so a tie at
    the overflow threshold goes to infinity, as IEEE round-to-nearest-even says)."""
    pats = np.arange(0, 1 << 15, dtype=np.uint32)
    if fmt == "BF16":
        with np.errstate(invalid="ignore"):
            vals = (pats << 16).view(np.float32).astype(np.float64)
        inf_pat, inf_val = 0x7F80, 2.0 ** 128
    else:
        vals = pats.astype(np.uint16).view(np.float16).astype(np.float64)
        inf_pat, inf_val = 0x7C00, 2.0 ** 16
    keep = np.isfinite(vals)
    pats, vals = pats[keep], vals[keep]
    order = np.argsort(vals, kind="stable")
    return np.append(vals[order], inf_val), np.append(pats[order], inf_pat)


def nearest_even(x, fmt):
    """Brute-force round-to-nearest-even of float64 values x (no NaN)."""
    vals, pats = table(fmt)
    a = np.abs(x)
    idx = np.searchsorted(vals, a, side="left")
    idx = np.minimum(idx, len(vals) - 1)
    hi_v, hi_p = vals[idx], pats[idx]
    lo_i = np.maximum(idx - 1, 0)
    lo_v, lo_p = vals[lo_i], pats[lo_i]
    d_hi, d_lo = hi_v - a, a - lo_v
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi_p % 2 == 0))
    pick_hi |= (a == hi_v)
    pick_hi |= a >= vals[-1]
    res = np.where(pick_hi, hi_p, lo_p).astype(np.uint32)
    sign = np.signbit(x).astype(np.uint32) << 15
    return (res | sign).astype(np.uint16)


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("out", ["BF16", "F16"])
def test_f32_rounding_is_nearest_even_bruteforce(oracle, out):
    bits = f32_sweep()
    x = bits.view(np.float32)
    ok = ~np.isnan(x)
    got = conv(oracle, "F32", out, bits)
    want = nearest_even(x[ok].astype(np.float64), out)
    np.testing.assert_array_equal(got[ok], want)
    assert np.all(got[~ok] == CANON[out])


@pytest.mark.parametrize("src,out", [("F16", "BF16"), ("BF16", "F16")])
def test_16bit_cross_rounding_bruteforce(oracle, src, out):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    if src == "F16":
        x = bits.view(np.float16).astype(np.float64)
    else:
        with np.errstate(invalid="ignore"):
            x = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ok = ~np.isnan(x)
    got = conv(oracle, src, out, bits)
    np.testing.assert_array_equal(got[ok], nearest_even(x[ok], out))
    assert np.all(got[~ok] == CANON[out])


# ---------------------------------------------------------- library checks

def torch_bits(t, out):
    t = t.to({"BF16": torch.bfloat16, "F16": torch.float16, "F32": torch.float32}[out])
    return t.view({"BF16": torch.int16, "F16": torch.int16, "F32": torch.int32}[out]).numpy().view(UINT[out])


@pytest.mark.parametrize("out", ["BF16", "F16"])
def test_f32_matches_torch(oracle, out):
    bits = f32_sweep()
    x = torch.from_numpy(bits.view(np.float32).copy())
    got = conv(oracle, "F32", out, bits)
    want = torch_bits(x, out)
    nan = torch.isnan(x).numpy()
    np.testing.assert_array_equal(got[~nan], want[~nan])


def test_f32_to_f16_matches_numpy(oracle):
    bits = f32_sweep()
    x = bits.view(np.float32)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    got = conv(oracle, "F32", "F16", bits)
    nan = np.isnan(x)
    np.testing.assert_array_equal(got[~nan], want[~nan])


@pytest.mark.parametrize("src,out", [("F16", "BF16"), ("F16", "F32"), ("BF16", "F16"), ("BF16", "F32")])
def test_16bit_exhaustive_matches_torch(oracle, src, out):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.float16 if src == "F16" else torch.bfloat16)
    got = conv(oracle, src, out, bits)
    want = torch_bits(t, out)
    nan = torch.isnan(t).numpy()
    np.testing.assert_array_equal(got[~nan], want[~nan])
    assert np.all(got[nan] == CANON[out])


FP8 = {"F8_E4M3": torch.float8_e4m3fn, "F8_E5M2": torch.float8_e5m2}


@pytest.mark.parametrize("src", ["F8_E4M3", "F8_E5M2"])
def test_fp8_decode_matches_torch(oracle, src):
    bits = np.arange(256, dtype=np.uint8)
    t = torch.from_numpy(bits.copy()).view(FP8[src]).float()
    got = conv(oracle, src, "F32", bits)
    nan = torch.isnan(t).numpy()
    np.testing.assert_array_equal(got[~nan], t.numpy().view(np.uint32)[~nan])
    assert np.all(got[nan] == CANON["F32"])
    assert nan.sum() == (2 if src == "F8_E4M3" else 6)


@pytest.mark.parametrize("src", ["F8_E4M3", "F8_E5M2"])
@pytest.mark.parametrize("out", ["BF16", "F16", "F32"])
def test_fp8_scaled_random_matches_torch(oracle, src, out):
    bits = np.arange(256, dtype=np.uint8)
    rng = np.random.Generator(np.random.PCG64(7))
    # random scales, a subnormal and a near-overflow one, then the special scales (zero, negative,
    # NaN and both infinities: IEEE binary32 products, NaN results canonical)
    scales = list(rng.uniform(1e-3, 1e-1, size=24).astype(np.float32)) + [np.float32(3.0e-39),
                                                                            np.float32(1.7e38)]
    scales += [np.float32(x) for x in (0.0, -0.25, "nan", "inf", "-inf")]
    for s in scales:
        x = torch.from_numpy(bits.copy()).view(FP8[src]).float() * torch.tensor(float(s), dtype=torch.float32)
        got = conv(oracle, src, out, bits, scale=float(s))
        want = torch_bits(x, out)
        nan = torch.isnan(x).numpy()
        np.testing.assert_array_equal(got[~nan], want[~nan])
        assert np.all(got[nan] == CANON[out])


# --------------------------------------------------------------- closed forms

OCP_E4M3 = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3C: 1.5,
            0x7E: 448.0, 0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0}
OCP_E5M2 = {0x00: 0.0, 0x01: 2.0 ** -16, 0x03: 3 * 2.0 ** -16, 0x04: 2.0 ** -14, 0x3C: 1.0,
            0x7B: 57344.0, 0x7C: float("inf"), 0xFC: float("-inf"), 0xBC: -1.0}


@pytest.mark.parametrize("src,tab,nans", [("F8_E4M3", OCP_E4M3, [0x7F, 0xFF]),
                                         ("F8_E5M2", OCP_E5M2, [0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF])])
def test_fp8_ocp_definition_values(oracle, src, tab, nans):
    bits = np.array(list(tab), dtype=np.uint8)
    got = conv(oracle, src, "F32", bits).view(np.float32)
    for b, g in zip(bits, got):
        assert g == np.float32(tab[int(b)]) and np.signbit(g) == np.signbit(tab[int(b)]), hex(b)
    assert np.all(conv(oracle, src, "F32", np.array(nans, dtype=np.uint8)) == CANON["F32"])


@pytest.mark.parametrize("src", ["F8_E4M3", "F8_E5M2"])
@pytest.mark.parametrize("k", [-12, -5, -1, 0, 1, 4, 9])
def test_fp8_times_power_of_two_is_exact(oracle, src, k):
    """x * 2^k has at most 4 significant bits, so bf16/f16/f32 hold it exactly:
    the expected bits are the exact product's bits (no rounding involved)."""
    bits = np.arange(256, dtype=np.uint8)
    x = torch.from_numpy(bits.copy()).view(FP8[src]).double().numpy()
    ok = ~np.isnan(x)
    exact = x[ok] * 2.0 ** k
    got32 = conv(oracle, src, "F32", bits, scale=2.0 ** k)[ok]
    np.testing.assert_array_equal(got32, exact.astype(np.float32).view(np.uint32))
    gotb = conv(oracle, src, "BF16", bits, scale=2.0 ** k)[ok]
    w = exact.astype(np.float32).view(np.uint32)
    assert np.all(w & 0xFFFF == 0)
    np.testing.assert_array_equal(gotb, (w >> 16).astype(np.uint16))
    finite16 = np.abs(exact) <= 65504
    goth = conv(oracle, src, "F16", bits, scale=2.0 ** k)[ok]
    sub = np.abs(exact) < 2.0 ** -24  # would not be exact in binary16
    sel = finite16 & ~sub
    np.testing.assert_array_equal(goth[sel], exact[sel].astype(np.float16).view(np.uint16))


TEXTBOOK = [
    # (src, out, input bits, expected bits, why)
    ("F32", "BF16", 0x3F808000, 0x3F80, "1+2^-8: tie between 1 and 1+2^-7 -> even"),
    ("F32", "BF16", 0x3F818000, 0x3F82, "1+3*2^-8: tie -> even (up)"),
    ("F32", "BF16", 0x3F808001, 0x3F81, "just above the tie -> up"),
    ("F32", "BF16", 0x7F7F7FFF, 0x7F7F, "just below the overflow threshold -> max finite"),
    ("F32", "BF16", 0x7F7F8000, 0x7F80, "tie at max finite + half ulp -> infinity"),
    ("F32", "BF16", 0x00000001, 0x0000, "2^-149 is far below half of the smallest bf16 subnormal 2^-133 -> +0"),
    ("F32", "BF16", 0x00008000, 0x0000, "2^-134: tie between 0 and 2^-133 -> even 0"),
    ("F32", "BF16", 0x00018000, 0x0002, "3*2^-134: tie between 2^-133 and 2^-132 -> even"),
    ("F32", "BF16", 0x80000000, 0x8000, "-0 keeps its sign"),
    ("F32", "BF16", 0xFF800000, 0xFF80, "-inf"),
    ("F32", "F16", 0x477FE000, 0x7BFF, "65504 exact"),
    ("F32", "F16", 0x477FEFFF, 0x7BFF, "just below 65520 -> 65504"),
    ("F32", "F16", 0x477FF000, 0x7C00, "65520: tie -> infinity"),
    ("F32", "F16", 0x33800000, 0x0001, "2^-24: smallest subnormal"),
    ("F32", "F16", 0x33000000, 0x0000, "2^-25: tie between 0 and 2^-24 -> 0"),
    ("F32", "F16", 0x33000001, 0x0001, "just above 2^-25 -> 2^-24"),
    ("F32", "F16", 0x33C00000, 0x0002, "1.5*2^-24: tie -> even 2*2^-24"),
    ("F32", "F16", 0x387FE000, 0x0400, "2^-14 - 2^-25: tie between the largest subnormal (odd) and the smallest normal -> normal"),
    ("F32", "F16", 0xB3000000, 0x8000, "-2^-25 -> -0"),
    ("BF16", "F16", 0x4780, 0x7C00, "65536 -> infinity"),
    ("BF16", "F16", 0x477F, 0x7BF8, "65280 exact"),
    ("F16", "BF16", 0x3C01, 0x3F80, "1+2^-10 -> 1 (below the tie)"),
    ("F16", "BF16", 0x3C02, 0x3F80, "1+2^-9: below the tie at 1+2^-8 -> 1"),
    ("F16", "BF16", 0x3C04, 0x3F80, "1+2^-8: tie -> even 1"),
    ("F16", "BF16", 0x3C0C, 0x3F82, "1+3*2^-8: tie -> even 1+2^-6"),
]


@pytest.mark.parametrize("src,out,inp,want,why", TEXTBOOK)
def test_textbook_rounding(oracle, src, out, inp, want, why):
    dt = np.uint32 if src == "F32" else np.uint16
    assert int(conv(oracle, src, out, np.array([inp], dtype=dt))[0]) == want, why


@pytest.mark.parametrize("src,bits", [("F32", [0x7FC00000, 0xFFC00000, 0x7F800001, 0xFFFFFFFF]),
                                      ("F16", [0x7E00, 0xFE00, 0x7C01, 0xFFFF]),
                                      ("BF16", [0x7FC0, 0xFFC0, 0x7F81, 0xFFFF])])
@pytest.mark.parametrize("out", ["BF16", "F16", "F32"])
def test_nan_becomes_positive_quiet_nan(oracle, src, bits, out):
    """Reading: every converted NaN is the target's positive quiet NaN."""
    if src == out:
        pytest.skip("same dtype is a byte copy")
    dt = np.uint32 if src == "F32" else np.uint16
    assert np.all(conv(oracle, src, out, np.array(bits, dtype=dt)) == CANON[out])


def test_same_dtype_and_integers_copy_bytes(oracle):
    rng = np.random.Generator(np.random.PCG64(3))
    for dt in ["BOOL", "U8", "I8", "I16", "U16", "I32", "U32", "I64", "U64", "F16", "BF16", "F32",
               "F64", "F8_E4M3", "F8_E5M2"]:
        raw = rng.integers(0, 256, size=8 * 37, dtype=np.uint8)
        assert oracle.out_dtype(dt, "KEEP") == dt
        np.testing.assert_array_equal(oracle.convert(dt, dt, raw), raw)


OUT_RULES = [
    ("F32", "BF16", "BF16"), ("F16", "BF16", "BF16"), ("BF16", "F16", "F16"), ("F8_E4M3", "F32", "F32"),
    ("I64", "BF16", "I64"), ("BOOL", "F16", "BOOL"), ("U8", "F32", "U8"), ("F64", "BF16", None),
    ("F64", "KEEP", "F64"), ("F32", "KEEP", "F32"), ("F8_E5M2", "KEEP", "F8_E5M2"), ("F32", "I32", None),
]


@pytest.mark.parametrize("src,req,want", OUT_RULES)
def test_output_dtype_rules(oracle, src, req, want):
    """Integers and bool are copied raw; floats take the requested float dtype."""
    assert oracle.out_dtype(src, req) == want


def test_unsupported_cast_is_rejected(oracle):
    with pytest.raises(oracle.OracleError) as e:
        oracle.convert("F64", "BF16", np.zeros(8, np.uint8))
    assert e.value.status == "UNSUPPORTED_CAST"
    with pytest.raises(oracle.OracleError) as e:
        oracle.convert("F16", "BF16", np.zeros(2, np.uint8), scale=2.0)
    assert e.value.status == "INVAL"
