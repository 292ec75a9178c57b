"""CPU oracle for the NVFP4 input projection -- TEST INFRASTRUCTURE.

Only the tests may import this module; it shares no code with the CUDA path.  The pages
ship an NVFP4 variant of the DiT (SGLang cookbook FLUX.3, section 3 "Checkpoints and
precision", Quantized checkpoints: FP4 (E2M1) weights with FP8 block scales, which needs
a Blackwell GPU and a matching GEMM).  E2M1 is 1 sign, 2 exponent (bias 1) and 1
mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.  Blocks of 16 consecutive elements
along K share one e4m3 scale.

Readings where the pages are silent (listed in the design notes with the rest):
  - both operands are NVFP4 (the FP4 tensor-core product the pages' "Blackwell GPU"
    requirement points to): W_in offline, the modulated activations on the fly;
  - above the block scales sits one fp32 scale per row (per token for the activations,
    per output channel for W_in), chosen so that the row's amax maps to 6 x 448, the
    largest E2M1 magnitude times the largest e4m3 value;
  - decisions are fixed in fp32, the way the device takes them:
        amax = max |x| over the row (exact on bf16 inputs)
        g    = fp32(2688 / amax),  s_row = fp32(amax / 2688)        (2688 = 6 * 448)
        per block: sb = e4m3(fp32(fp32(bmax * g) / 6))              bmax = max |x| in block
        per element: code = e2m1(fp32(x * fp32(g / sb)))            (code 0 where sb = 0)
    each rounding to nearest even, e4m3 and E2M1 saturating (at 448 and 6); the sign of
    an element that rounds to zero is kept (code 8 is -0); an all-zero row, and a row so
    small that g overflows fp32, quantizes to zeros with s_row = 0;
  - then x ~ e2m1(code) * e4m3(sb) * s_row and
        P = s_a[token] * sum_k (e2m1(a) sb_a)(e2m1(w) sb_w) * s_w[out] + b_in.
Storage (a contract between the quantizer and the GEMM, not arithmetic): two codes per
byte, the even element in the low nibble; the block scales of 128 rows x 64 elements
(4 scales per row) form one 512-byte tile, row r's scale j at byte
(r % 32) * 16 + (r // 32) * 4 + j, tiles ordered by row tile, then by 64-element step,
rows padded to a multiple of 256 (a pair of 128-row tiles) with zero scales.

Pins (tests/test_oracle_nvfp4.py): E2M1 values from the bit-field formula; the rounding
against a brute-force nearest search with ties to the even code; the quantizer's zero row,
exact round trip on representable rows, power-of-two equivariance and error bound; the
linear map's exactness when quantization is lossless; the storage layout's inverse.
"""
from __future__ import annotations

import numpy as np

from .fp8 import e4m3_round   # nearest e4m3, ties to even, saturating (pinned to torch's cast)

F32 = np.float32
F64 = np.float64
E2M1_MAX = 6.0
E4M3_MAX = 448.0
ROW_TARGET = E2M1_MAX * E4M3_MAX   # 2688
BLOCK = 16


def e2m1_value(codes) -> np.ndarray:
    """Value of 4-bit E2M1 codes: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0;
    exponent 0 is subnormal (m * 0.5)."""
    c = np.asarray(codes, dtype=np.int64)
    s = np.where(c & 8, -1.0, 1.0)
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, 0.5 * m, 2.0 ** (e - 1) * (1.0 + 0.5 * m))
    return s * mag


_MAGS = e2m1_value(np.arange(8))   # 0, 0.5, 1, 1.5, 2, 3, 4, 6


def e2m1_round(v) -> np.ndarray:
    """Codes of the nearest E2M1 values (ties to the even code, i.e. mantissa bit 0),
    saturating at +-6, sign kept for values that round to zero."""
    v = np.asarray(v, dtype=F64)
    a = np.abs(v)
    # midpoints between consecutive magnitudes; at a tie pick the even code
    mids = (_MAGS[:-1] + _MAGS[1:]) / 2
    idx = np.searchsorted(mids, a, side="left")        # a <= mid -> lower candidate
    at_mid = np.isin(a, mids)
    lower_even = (np.searchsorted(mids, a, side="left") % 2) == 0
    # for a tie a == mids[i]: candidates i (lower) and i + 1; take the even one
    tie_idx = np.where(lower_even, idx, idx + 1)
    idx = np.where(at_mid, tie_idx, idx)
    idx = np.minimum(idx, 7)
    sign = np.signbit(v).astype(np.int64) * 8
    return (sign | idx).astype(np.uint8)


def e4m3_code(v) -> np.ndarray:
    """The e4m3 bit pattern of e4m3-representable non-negative values."""
    v = np.asarray(v, dtype=F64)
    out = np.zeros(v.shape, dtype=np.uint8)
    nz = v > 0
    e = np.floor(np.log2(np.where(nz, v, 1.0)))
    sub = nz & (v < 2.0 ** -6)
    nrm = nz & ~sub
    m_sub = np.round(v / 2.0 ** -9)
    m_nrm = np.round((v / 2.0 ** e - 1.0) * 8)
    out[sub] = m_sub[sub].astype(np.uint8)
    out[nrm] = (((e[nrm] + 7).astype(np.int64) << 3) | m_nrm[nrm].astype(np.int64)).astype(np.uint8)
    return out


def e4m3_value(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.int64)
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, m * 2.0 ** -9, 2.0 ** (e - 7) * (1.0 + m / 8.0))
    return np.where(c & 0x80, -mag, mag)


def quantize_rows(x):
    """NVFP4 quantization of the rows of x ([rows, k], k % 16 == 0, fp32-representable).
    Returns (codes uint8 [rows, k] in 0..15, block-scale codes uint8 [rows, k / 16],
    row scales float32 [rows])."""
    x32 = np.asarray(x, dtype=F32)
    rows, k = x32.shape
    amax = np.max(np.abs(x32), axis=1)
    safe = np.where(amax > 0, amax, F32(1))
    with np.errstate(over="ignore"):
        g_raw = (F32(ROW_TARGET) / safe).astype(F32)
    pos = (amax > 0) & np.isfinite(g_raw)
    g = np.where(pos, g_raw, F32(0)).astype(F32)
    s_row = np.where(pos, safe / F32(ROW_TARGET), F32(0)).astype(F32)
    blocks = x32.reshape(rows, k // BLOCK, BLOCK)
    bmax = np.max(np.abs(blocks), axis=2)
    t = (bmax * g[:, None]).astype(F32)
    u = (t / F32(6)).astype(F32)
    sbv = e4m3_round(u)                                    # values >= 0
    sb = e4m3_code(sbv)
    sbf = sbv.astype(F32)
    ok = sbf > 0
    r = np.where(ok, g[:, None] / np.where(ok, sbf, F32(1)), F32(0)).astype(F32)
    v = (blocks * r[:, :, None]).astype(F32)
    codes = e2m1_round(v)
    codes = np.where(ok[:, :, None], codes, np.uint8(0)).astype(np.uint8)
    return codes.reshape(rows, k), sb, s_row


def dequantize(codes, sb, s_row) -> np.ndarray:
    """x^ = e2m1(code) * e4m3(sb) * s_row, float64."""
    codes = np.asarray(codes)
    rows, k = codes.shape
    vals = e2m1_value(codes).reshape(rows, k // BLOCK, BLOCK) * e4m3_value(sb)[:, :, None]
    return vals.reshape(rows, k) * np.asarray(s_row, dtype=F64)[:, None]


def nvfp4_linear(a, w) -> np.ndarray:
    """a W^T with both operands quantized row-wise to NVFP4; the block-scaled products
    and their sums exact in float64, then the two row scales."""
    ca, sba, sa = quantize_rows(a)
    cw, sbw, sw = quantize_rows(w)
    ka = dequantize(ca, sba, np.ones_like(sa))
    kw = dequantize(cw, sbw, np.ones_like(sw))
    return (ka @ kw.T) * sa.astype(F64)[:, None] * sw.astype(F64)[None, :]


# ------------------------------------------------------------------ storage
def pack_codes(codes) -> np.ndarray:
    """Two codes per byte, the even element in the low nibble: [rows, k] -> [rows, k / 2]."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def unpack_codes(packed) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], p.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = p & 15
    out[:, 1::2] = p >> 4
    return out


def scale_tile_offset(r, j, k: int) -> np.ndarray:
    """Byte offset of block scale j (0 .. k/16 - 1) of row r in the tiled storage."""
    r = np.asarray(r, dtype=np.int64)
    j = np.asarray(j, dtype=np.int64)
    steps = k // 64
    tile = (r // 128) * steps + j // 4
    return tile * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (j % 4)


def scale_bytes(rows: int, k: int) -> int:
    return (rows + 255) // 256 * 256 * (k // BLOCK)


def tile_scales(sb, rows_padded: int = None) -> np.ndarray:
    """Block-scale codes [rows, k / 16] -> the tiled byte layout (zero-padded rows)."""
    sb = np.asarray(sb, dtype=np.uint8)
    rows, nb = sb.shape
    k = nb * BLOCK
    out = np.zeros(scale_bytes(rows, k), dtype=np.uint8)
    r, j = np.meshgrid(np.arange(rows), np.arange(nb), indexing="ij")
    out[scale_tile_offset(r, j, k)] = sb
    return out


def untile_scales(buf, rows: int, k: int) -> np.ndarray:
    r, j = np.meshgrid(np.arange(rows), np.arange(k // BLOCK), indexing="ij")
    return np.asarray(buf, dtype=np.uint8)[scale_tile_offset(r, j, k)]
