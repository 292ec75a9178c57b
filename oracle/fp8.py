"""CPU oracle for the FP8 (e4m3) row-wise input projection -- TEST INFRASTRUCTURE.

Only the tests may import this module; it shares no code with the CUDA path.  The pages
run quantized variants of the projections (SGLang cookbook FLUX.3, section 7
"Quantization": FP8 and NVFP4 checkpoints of the DiT; the Miles page, section 3:
"fp8 rowwise" among the precisions); the block's arithmetic is unchanged except that
the input projection multiplies e4m3 codes:

  a_q, s_a = quantize_rows(a)            per token: s_a = amax / 448, a ~ a_q * s_a
  W_q, s_w = quantize_rows(W_in)         per output channel (row of W_in)
  P = s_a[:, None] * (a_q W_q^T) * s_w[None, :] + b_in

Quantization decisions are fixed in fp32, the way the device takes them: amax of the row
(exact on bf16 inputs), inv = fp32(448 / amax), one fp32 product x * inv, then
round-to-nearest-even to e4m3 (saturating at +-448).  Readings: 448 (the largest finite
e4m3) maps to the row's amax; an all-zero row quantizes to zeros with scale 0.

Pins (tests/test_oracle_fp8.py): the rounding against torch's float8_e4m3fn cast; the
row quantizer's exactness on representable inputs, its power-of-two equivariance and
error bound; the linear map's exactness when quantization is lossless.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
F64 = np.float64
E4M3_MAX = 448.0


def e4m3_round(v) -> np.ndarray:
    """Round float values (fp32-representable) to the nearest e4m3 value, ties to even,
    saturating at +-448 (float64 result)."""
    v = np.asarray(v, dtype=F64)
    a = np.abs(v)
    # binade exponent of normals; the subnormal step 2^-9 below 2^-6
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    step = np.where(a >= 2.0 ** -6, 2.0 ** (e - 3), 2.0 ** -9)
    q = np.round(a / step) * step                       # np.round: ties to even
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, v)


def quantize_rows(x):
    """Per-row e4m3 quantization: returns (codes as float64 values, scale per row, fp32
    values in float64) with x ~ codes * scale."""
    x32 = np.asarray(x, dtype=F32)
    amax = np.max(np.abs(x32), axis=1)
    safe = np.where(amax > 0, amax, F32(1))
    inv = np.where(amax > 0, F32(E4M3_MAX) / safe, F32(0)).astype(F32)
    codes = e4m3_round((x32 * inv[:, None]).astype(F32))
    scale = np.where(amax > 0, amax / F32(E4M3_MAX), F32(0)).astype(F32)
    return codes, scale.astype(F64)


def fp8_linear(a, w) -> np.ndarray:
    """a W^T with both operands quantized row-wise to e4m3 (a per token, W per output
    channel), products and sums exact in float64."""
    qa, sa = quantize_rows(a)
    qw, sw = quantize_rows(w)
    return (qa @ qw.T) * sa[:, None] * sw[None, :]
