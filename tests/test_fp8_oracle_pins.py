"""Pins of the FP8 (E4M3) storage oracle to facts fixed outside it (no GPU).

Each ``check_*`` compares ``oracle.fp8_oracle`` against something it does not
share code with:
* the OCP E4M3 ("fn") bit layout, decoded here by explicit enumeration of the
  sign, exponent and mantissa fields;
* PyTorch's ``float8_e4m3fn`` dtype (a library routine) for decoding and for
  float32 -> E4M3 rounding (round to nearest, ties to even);
* closed-form rows whose scale and codes are known.
``test_planted_*`` plant plausible mistakes in copies of the oracle's
functions and require that some check fails.

Source of the storage scheme: "Inference-Time Hyper-Scaling with KV Cache
Compression", paper-notes page, "Related work" (quantization is orthogonal to
DMS and combinable); the scheme itself (per-row absmax scale, E4M3 codes) is
a reading of that remark, stated in the oracle's docstring.
"""
import numpy as np
import pytest
import torch

import oracle.fp8_oracle as F

ALL_CODES = np.arange(256, dtype=np.uint8)
FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def _spec_value(c: int) -> float:
    """E4M3 value of one code, field by field (OCP 8-bit formats)."""
    s = -1.0 if c >> 7 else 1.0
    e = (c >> 3) & 0xF
    m = c & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * m / 8.0 * 2.0 ** (1 - 7)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def _torch_round_codes(y32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(y32, dtype=np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


# --------------------------------------------------------------------------
# checks (each takes the functions under test)
# --------------------------------------------------------------------------

def check_decode(value_fn):
    got = value_fn(ALL_CODES)
    spec = np.array([_spec_value(int(c)) for c in ALL_CODES])
    lib = torch.from_numpy(ALL_CODES.copy()).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(spec)
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(np.isnan(lib), nan)
    assert np.array_equal(got[~nan], spec[~nan]), "decode differs from the bit layout"
    assert np.array_equal(got[~nan], lib[~nan]), "decode differs from torch float8_e4m3fn"
    assert np.nanmax(got) == 448.0 and np.nanmin(got) == -448.0


def check_round_trip(round_fn, encode_fn, value_fn):
    v = value_fn(FINITE)
    assert np.array_equal(encode_fn(round_fn(v)), FINITE), "finite codes do not round-trip"


def check_rounding_vs_library(round_fn, encode_fn, seed=0):
    rng = np.random.default_rng(seed)
    # magnitudes across every binade, subnormals included, plus exact midpoints
    mags = np.exp2(rng.uniform(-12.0, np.log2(448.0), 20000)).astype(np.float32)
    y = (mags * rng.choice([-1.0, 1.0], mags.size)).astype(np.float32)
    vals = F.e4m3_value(FINITE)
    vals = np.sort(np.unique(vals))
    mids = ((vals[1:] + vals[:-1]) / 2.0).astype(np.float32)  # exact in float32
    y = np.concatenate([y, mids, -mids, np.float32([0.0, -0.0, 448.0, -448.0, 2.0 ** -10, -2.0 ** -10])])
    got = encode_fn(round_fn(y))
    assert np.array_equal(got, _torch_round_codes(y)), "rounding differs from torch float8_e4m3fn"


def check_quantize_rows(quant_fn):
    # constant row c: amax = |c|, every code is +-448
    x = np.full((3, 16), 0.375, np.float32)
    x[1] = -2.5
    x[2, ::2] = 1.0e-3
    codes, scale = quant_fn(x)
    assert scale[0] == np.float32(0.375) / np.float32(448) and np.all(codes[0] == 0x7E)
    assert np.all(codes[1] == 0xFE)
    # zero row: scale 1, codes +0
    codes, scale = quant_fn(np.zeros((1, 8), np.float32))
    assert scale[0] == 1.0 and np.all(codes == 0)
    # rows of E4M3 values times a power of two whose max is 448 * 2^k: lossless
    rng = np.random.default_rng(3)
    vals = F.e4m3_value(FINITE)
    for k in (-5, 0, 3):
        row = rng.choice(vals, 64)
        row[7] = 448.0
        x = (row * 2.0 ** k).astype(np.float32)
        codes, scale = quant_fn(x[None])
        assert scale[0] == np.float32(2.0 ** k)
        assert np.array_equal(F.dequantize_rows(codes, scale)[0], x.astype(np.float64))
    # general rows: the codes equal the library rounding of the float32 quotient;
    # the last rows hold values whose float32 quotient lands on a midpoint between
    # two E4M3 values while the exact quotient does not (the code depends on
    # taking the quotient in float32)
    x = np.concatenate([rng.standard_normal((50, 128)).astype(np.float32), _quotient_sensitive_rows()])
    codes, scale = quant_fn(x)
    amax = np.abs(x).max(axis=1)
    assert np.array_equal(scale, (amax / np.float32(448)).astype(np.float32))
    y = np.clip((x / scale[:, None]).astype(np.float32), -448, 448)
    assert np.array_equal(codes, _torch_round_codes(y))
    # the dequantized row is within half a quantum of the input: relative 2^-4
    # for normal codes, 2^-10 * scale for subnormal ones (plus the float32
    # rounding of the quotient)
    err = np.abs(F.dequantize_rows(codes, scale) - x)
    assert np.all(err <= (np.abs(x) * 2.0 ** -4 + scale[:, None] * 2.0 ** -10) * (1 + 2.0 ** -16))


def _quotient_sensitive_rows(n_rows=4, D=128):
    """Rows [amax, x1, x2, ..., 0 ...] where float32(x_i / scale) is an exact
    midpoint M of two E4M3 values but x_i / scale (exactly) is not, so rounding
    the float32 quotient and rounding the exact quotient give different codes."""
    vals = np.sort(np.unique(F.e4m3_value(FINITE)))
    vals = vals[vals > 0]
    mids = (vals[1:] + vals[:-1]) / 2.0
    rng = np.random.default_rng(11)
    rows = []
    for _ in range(200):  # bounded search over row maxima
        amax = np.float32(rng.uniform(0.5, 4.0))
        scale = np.float32(amax / np.float32(448))
        found = []
        for m in mids:
            base = np.float32(m * np.float64(scale))
            for cand in (base, np.nextafter(base, np.float32(0)), np.nextafter(base, np.float32(np.inf))):
                if (np.float32(cand / scale) == np.float32(m) and np.float64(cand) / np.float64(scale) != m
                        and abs(cand) < amax):
                    found.append(cand)
                    break
        if len(found) >= 4:
            row = np.zeros(D, np.float32)
            row[0] = amax
            k = min(len(found), (D - 1) // 2)
            row[1:1 + k] = found[:k]
            row[1 + k:1 + 2 * k] = -np.float32(found[:k])
            rows.append(row)
        if len(rows) == n_rows:
            break
    assert len(rows) == n_rows, "no quotient-sensitive rows found"
    return np.stack(rows)


# --------------------------------------------------------------------------
# the real oracle
# --------------------------------------------------------------------------

def test_decode_all_codes():
    check_decode(F.e4m3_value)


def test_round_trip_every_finite_code():
    check_round_trip(F.e4m3_round, F.e4m3_encode, F.e4m3_value)


def test_rounding_matches_library():
    check_rounding_vs_library(F.e4m3_round, F.e4m3_encode)


def test_quantize_rows_closed_forms():
    check_quantize_rows(F.quantize_rows)


# --------------------------------------------------------------------------
# planted mistakes: each must be caught by at least one check
# --------------------------------------------------------------------------

def _round_half_up(y):
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    _, ex = np.frexp(np.where(a >= 2.0 ** -6, a, 1.0))
    q = np.where(a >= 2.0 ** -6, np.exp2(ex - 4.0), 2.0 ** -9)
    return np.copysign(np.floor(a / q + 0.5) * q, y)


def _round_no_subnormals(y):
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    q = np.exp2(ex - 4.0)
    return np.copysign(np.rint(a / q) * q, y)


def _value_bias_8(code):
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    v = np.where(e == 0, m * 2.0 ** -10, (1 + m / 8) * np.exp2(e - 8.0))
    v = np.where((e == 15) & ((c & 7) == 7), np.nan, v)
    return np.where(c & 0x80, -v, v)


def _quant_scale_447(x):
    x = np.asarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=-1)
    scale = np.where(amax > 0, amax / np.float32(447), 1).astype(np.float32)
    y = np.clip(x / scale[..., None], -448, 448)
    return F.e4m3_encode(F.e4m3_round(y)), scale


def _quant_float64_quotient(x):
    x = np.asarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=-1)
    scale = np.where(amax > 0, amax / np.float32(448), 1).astype(np.float32)
    y = np.clip(x.astype(np.float64) / scale[..., None].astype(np.float64), -448, 448)
    return F.e4m3_encode(F.e4m3_round(y)), scale


def _quant_zero_row_scale_0(x):
    x = np.asarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=-1)
    scale = (amax / np.float32(448)).astype(np.float32)
    with np.errstate(invalid="ignore", divide="ignore"):
        y = np.nan_to_num(np.clip(x / scale[..., None], -448, 448))
    return F.e4m3_encode(F.e4m3_round(y)), scale


def _fails(fn, *args):
    try:
        fn(*args)
    except (AssertionError, ValueError):
        return True
    return False


@pytest.mark.parametrize("bad_round", [_round_half_up, _round_no_subnormals])
def test_planted_rounding_mistakes_are_caught(bad_round):
    assert _fails(check_rounding_vs_library, bad_round, F.e4m3_encode) or _fails(
        check_round_trip, bad_round, F.e4m3_encode, F.e4m3_value)


def test_planted_decode_mistake_is_caught():
    assert _fails(check_decode, _value_bias_8)


@pytest.mark.parametrize("bad_quant", [_quant_scale_447, _quant_float64_quotient, _quant_zero_row_scale_0])
def test_planted_quantize_mistakes_are_caught(bad_quant):
    assert _fails(check_quantize_rows, bad_quant)
