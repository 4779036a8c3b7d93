"""Oracle for the fp8 GEMM variant: E4M3 rounding, per-row quantisation and the quantised
linear layer.  Test infrastructure only (float64 / float32 NumPy); nothing on the product path
imports it.

The pages name no fp8 arithmetic: the variant is a knob of the block's projections (lower
precision GEMMs), and every constant here is the plainest reading of the E4M3 format
(1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities, largest finite value
448, subnormals down to 2^-9) with round-to-nearest-even and saturation to +-448:

* a row's scale is s = amax / 448 in float32 (s = 1 for an all-zero row), the quantised code
  of element x is E4M3(x / s) with the division done in float32 (correctly rounded);
* the quantised linear layer is y = (A_q B_q^T) * s_a[row] * s_b[col] + bias, evaluated here
  in float64 from the dequantised codes.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_MIN_SUBNORMAL = 2.0 ** -9


def e4m3_round(v):
    """Nearest E4M3 value of float64 v, ties to even mantissa, saturating to +-448 (NaN stays
    NaN).  Returns float64 values that are exactly representable in E4M3."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    # quantum: 2^(e - 3) in the normal range (3 mantissa bits), 2^-9 below the smallest normal
    e = np.floor(np.log2(np.where(a >= E4M3_MIN_NORMAL, a, E4M3_MIN_NORMAL)))
    q = np.where(a >= E4M3_MIN_NORMAL, 2.0 ** (e - 3), E4M3_MIN_SUBNORMAL)
    r = np.round(a / q) * q              # np.round rounds halves to even; a / q is exact here
    r = np.minimum(r, E4M3_MAX)
    return np.where(np.isnan(v), np.nan, np.copysign(r, v))


def e4m3_code(v):
    """The 8-bit E4M3 code of values that are exactly representable (e.g. e4m3_round output)."""
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros(v.shape, dtype=np.uint8)
    sign = (np.signbit(v)).astype(np.uint8) << 7
    a = np.abs(v)
    sub = a < E4M3_MIN_NORMAL
    m_sub = np.rint(a / E4M3_MIN_SUBNORMAL).astype(np.int64)            # 0..7
    e = np.floor(np.log2(np.where(sub, 1.0, a))).astype(np.int64)
    m_norm = np.rint((np.where(sub, 1.0, a) / 2.0 ** e - 1.0) * 8).astype(np.int64)
    code = np.where(sub, m_sub, ((e + 7) << 3) | m_norm)
    out[...] = (code.astype(np.uint8) | sign)
    return out


def e4m3_decode(code):
    """float64 value of E4M3 codes (0x7f / 0xff are NaN)."""
    c = np.asarray(code, dtype=np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return s * val


def quantize_rows(x):
    """Per-row E4M3 quantisation of float32-representable x [M][K]: (codes uint8 [M][K],
    scales float32 [M]) with s = amax / 448 (float32), codes of E4M3(float32(x) / s)."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.abs(x32).max(axis=1) if x32.shape[1] else np.zeros(len(x32), np.float32)
    s = np.where(amax > 0, (amax / np.float32(E4M3_MAX)).astype(np.float32), np.float32(1.0))
    s = s.astype(np.float32)
    scaled = (x32 / s[:, None]).astype(np.float32)                     # float32 division
    return e4m3_code(e4m3_round(scaled.astype(np.float64))), s


def linear_fp8(a_codes, a_scale, b_codes, b_scale, bias=None):
    """y = (A_q B_q^T) * s_a[:, None] * s_b[None, :] + bias in float64."""
    a = e4m3_decode(a_codes)
    b = e4m3_decode(b_codes)
    y = (a @ b.T) * np.asarray(a_scale, np.float64)[:, None] * np.asarray(b_scale, np.float64)[None, :]
    if bias is not None:
        y = y + np.asarray(bias, np.float64)[None, :]
    return y


def bf16_round(x):
    """float64 values rounded to the nearest bfloat16 (ties to even), as float64: the value a
    bf16 activation buffer holds."""
    f = np.asarray(x, dtype=np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def linear_fp8_act(x, w8: dict, name: str, bias):
    """The fp8 variant's projection of activations x (float64 [L][K]): x is stored in bf16,
    quantised per row, and multiplied with the weight codes w8['q_' + name] and scales
    w8['s_' + name] (quantised per output row from the bf16 weights)."""
    codes, s = quantize_rows(bf16_round(x).astype(np.float32))
    return linear_fp8(codes, s, w8["q_" + name], w8["s_" + name], bias)


def quantize_weights(bw_stream: dict):
    """E4M3 codes and row scales of one stream's four projection matrices (float32 arrays
    exactly representable in bf16)."""
    out = {}
    for name, key in (("qkv", "w_qkv"), ("o", "w_o"), ("1", "w_1"), ("2", "w_2")):
        out["q_" + name], out["s_" + name] = quantize_rows(np.asarray(bw_stream[key], np.float32))
    return out
