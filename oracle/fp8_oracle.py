"""CPU oracle for the FP8 (E4M3) storage of the compacted KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU legs of ``bench.py`` may import or run this module; the product path never
does.  It shares no code with the CUDA path.

Source: "Inference-Time Hyper-Scaling with KV Cache Compression", paper-notes
page, section "Related work" (KVQuant / KIVI): quantization compresses the KV
cache along an axis orthogonal to DMS's sparsification, and the two can be
combined.  The pages fix no quantization scheme.  The reading used here is
the plainest one with native hardware support:

* every retained K row and every V row (one token, one KV head, D values) is
  stored as D FP8 E4M3 codes and one float32 scale;
* ``scale = amax / 448`` in float32 (448 is the largest finite E4M3 value),
  where amax is the largest magnitude in the row; a row of zeros gets scale 1;
* ``code = E4M3(x / scale)``: the float32 quotient (IEEE division, round to
  nearest even) rounded to the nearest E4M3 value, ties to even, and clamped
  to +-448 (saturation; the quotient can exceed 448 by float32 rounding);
* the stored row stands for ``code_value * scale``, and attention runs over
  those dequantized rows exactly as over bf16 rows.

So the quantization decision (an integer code) is made in float32 on both
sides, and the attention is compared against the float64 oracle evaluated on
the dequantized rows.

E4M3 ("fn" variant) as defined by the OCP 8-bit floating point formats: 1 sign
bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 encodes
subnormals m * 2^-9; exponent field 15 with mantissa 7 is NaN; there is no
infinity; the largest finite magnitude is 1.75 * 2^8 = 448.

Parity status: pinned by ``tests/test_fp8_oracle_pins.py``: the
decoding of all 256 codes against the format definition written out bit by
bit and against PyTorch's float8_e4m3fn type, the rounding against PyTorch's
float32 -> float8_e4m3fn conversion on random and tie inputs, the encode /
decode round trip of every finite code, and the row scale on closed-form
rows.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
_MIN_NORMAL = 2.0 ** -6
_SUB_QUANTUM = 2.0 ** -9


def e4m3_value(code) -> np.ndarray:
    """float64 value of E4M3 codes (uint8); NaN for the two NaN codes."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = (c & 0x7).astype(np.float64)
    val = np.where(exp == 0, man * _SUB_QUANTUM, (1.0 + man / 8.0) * np.exp2(exp - 7.0))
    val = np.where((exp == 15) & ((c & 0x7) == 7), np.nan, val)
    return sign * val


def e4m3_round(y) -> np.ndarray:
    """Round float values (|y| <= 448) to the nearest E4M3 value, ties to even,
    in float64.  The sign of zero is kept (a negative input that rounds to zero
    gives -0)."""
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    # binade exponent e with 2^e <= a < 2^(e+1), for normal magnitudes
    _, ex = np.frexp(np.where(a >= _MIN_NORMAL, a, 1.0))
    quantum = np.where(a >= _MIN_NORMAL, np.exp2(ex - 1 - 3.0), _SUB_QUANTUM)
    r = np.rint(a / quantum) * quantum  # np.rint rounds half to even
    return np.copysign(r, y)


def e4m3_encode(v) -> np.ndarray:
    """uint8 codes of float64 values that are exact E4M3 values (output of
    e4m3_round), sign of zero included."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    sign = np.signbit(v).astype(np.int64) << 7
    _, ex = np.frexp(np.where(a >= _MIN_NORMAL, a, 1.0))
    e = ex - 1  # a = 1.m * 2^e
    normal = a >= _MIN_NORMAL
    exp_field = np.where(normal, e + 7, 0)
    man = np.where(normal, (a / np.exp2(e) - 1.0) * 8.0, a / _SUB_QUANTUM)
    if not np.all(man == np.rint(man)):
        raise ValueError("value is not an E4M3 value")
    return (sign | (exp_field.astype(np.int64) << 3) | np.rint(man).astype(np.int64)).astype(np.uint8)


def quantize_rows(x):
    """Quantize rows (last axis) of float32 values (bf16 inputs widened).

    Returns (codes uint8 [..., D], scale float32 [...]).  Every operation that
    decides a code is float32, as stated in the module docstring."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1).astype(np.float32)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    y = (x / scale[..., None]).astype(np.float32)
    y = np.clip(y, np.float32(-E4M3_MAX), np.float32(E4M3_MAX))
    return e4m3_encode(e4m3_round(y)), scale


def dequantize_rows(codes, scale) -> np.ndarray:
    """float64 rows ``code_value * scale`` (exact in float64)."""
    return e4m3_value(codes) * np.asarray(scale, dtype=np.float64)[..., None]
