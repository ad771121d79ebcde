"""Number formats of the MoE layer, written from their definitions.

Test infrastructure only (see oracle/__init__.py).

The pages fix FP8 only in passing (the SGLang/H20 article, section "FP8 MLA",
and the DeepGEMM swapAB section, which run DeepSeek-R1 in FP8); the layout
used here is the one the R1-shaped workload states: e4m3 weights with one
fp32 scale per 128x128 block, activations with one fp32 scale per token and
128-column group.  Readings taken where the pages say nothing:
  * e4m3 is the OCP "fn" variant (max finite 448, no infinity);
  * encoding rounds to nearest, ties to even, and saturates to +-448;
  * a group scale is amax / 448 in fp32 (not a power of two); a group whose
    amax is 0 gets scale 1 and codes 0;
  * value / scale is one IEEE fp32 division.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
GROUP = 128


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """fp64 value of each e4m3 code: S.EEEE.MMM, bias 7, subnormals at E=0."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = np.ldexp((8 + m).astype(np.float64), (e - 10).astype(np.int64))
    sub = np.ldexp(m.astype(np.float64), -9)
    v = np.where(e == 0, sub, normal)
    v = np.where((e == 0xF) & (m == 0x7), np.nan, v)
    return sign * v


def e4m3_encode(values) -> np.ndarray:
    """Round fp32 values to e4m3 codes: nearest, ties to even, saturating.

    Works in fp64, where dividing by a power of two is exact: the value is
    scaled to units of its e4m3 quantum (2^(e-3) in binade e >= -6, 2^-9
    below), rounded half-to-even, and re-encoded.  |v| > 448 gives 448.
    """
    v = np.asarray(values, dtype=np.float32).astype(np.float64)
    neg = np.signbit(v)
    a = np.abs(v)
    sat = a > E4M3_MAX
    a = np.where(sat, E4M3_MAX, a)
    # binade of a (floor(log2 a)); clamp to the subnormal quantum below 2^-6
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.maximum(ex.astype(np.int64) - 1, -6)
    quantum = np.ldexp(1.0, e - 3)
    r = np.rint(a / quantum) * quantum          # rint: half to even
    r = np.minimum(r, E4M3_MAX)
    # re-encode the rounded magnitude
    _, ex2 = np.frexp(np.where(r > 0, r, 1.0))
    e2 = ex2.astype(np.int64) - 1
    is_sub = r < 2.0 ** -6
    m_sub = np.rint(r / 2.0 ** -9).astype(np.int64)
    m_norm = np.rint(r / np.ldexp(1.0, e2) * 8.0).astype(np.int64) - 8
    code = np.where(is_sub, m_sub, ((e2 + 7) << 3) | m_norm)
    code = np.where(r == 0, 0, code)
    code = code | np.where(neg, 0x80, 0)
    return code.astype(np.uint8)


def bf16_round(values) -> np.ndarray:
    """Round to the nearest bf16 value (8-bit significand), ties to even.

    Input fp32 or fp64; result fp64 holding bf16 values.  Rounding is direct
    (one rounding from the input's own precision), in units of the quantum
    2^(e-7) of the input's binade e (clamped at the smallest normal binade).
    """
    v = np.asarray(values, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.maximum(ex.astype(np.int64) - 1, -126)
    quantum = np.ldexp(1.0, e - 7)
    return np.copysign(np.rint(a / quantum) * quantum, v)


def bf16_bits(values_bf16_exact) -> np.ndarray:
    """uint16 bit patterns of values that are already exact bf16 values."""
    f = np.asarray(values_bf16_exact, dtype=np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(bits) -> np.ndarray:
    """fp32 value of bf16 bit patterns (the upper half of a binary32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def quant_groups_fp8(values_f32) -> tuple[np.ndarray, np.ndarray]:
    """Per-row, per-128-column FP8 quantisation of an fp32 matrix.

    For each row and group g of 128 columns: amax = max |v|, scale = amax/448
    (fp32 division; 1 when amax is 0), code = e4m3(v / scale) with the
    division in fp32.  Returns (codes uint8 [rows, cols], scales fp32
    [rows, cols/128]).
    """
    v = np.ascontiguousarray(values_f32, dtype=np.float32)
    rows, cols = v.shape
    assert cols % GROUP == 0, "columns must be a multiple of 128"
    g = v.reshape(rows, cols // GROUP, GROUP)
    amax = np.max(np.abs(g), axis=2)
    scale = np.where(amax == 0, np.float32(1.0),
                     amax / np.float32(E4M3_MAX)).astype(np.float32)
    scaled = (g / scale[:, :, None]).astype(np.float32)
    codes = e4m3_encode(scaled).reshape(rows, cols)
    return codes, scale


def dequant_groups_fp8(codes, scales) -> np.ndarray:
    """fp64 values code * scale for a [rows, cols] matrix with per-128 scales."""
    c = np.asarray(codes, dtype=np.uint8)
    rows, cols = c.shape
    s = np.asarray(scales, dtype=np.float32).astype(np.float64)
    v = e4m3_decode(c).reshape(rows, cols // GROUP, GROUP)
    return (v * s[:, :, None]).reshape(rows, cols)
