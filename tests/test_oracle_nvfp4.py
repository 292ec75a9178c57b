"""Pins of the NVFP4 oracle (oracle/nvfp4.py) against the format's definition and the
mathematics: E2M1 from its bit fields, round-to-nearest-even by brute force, the row
quantizer's special cases, round trip, equivariance and error bound, and the linear
map on losslessly quantized operands."""
import numpy as np
import pytest

from oracle import nvfp4 as Q

F32 = np.float32


def test_e2m1_values_from_bit_fields():
    # 1 sign, 2 exponent bits with bias 1, 1 mantissa bit; exponent 0 is subnormal
    mags = Q.e2m1_value(np.arange(8))
    assert mags.tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert (Q.e2m1_value(np.arange(8, 16)) == -mags).all()


def _brute_round(v):
    """Nearest of the 15 E2M1 values by exhaustive search; on a tie the code whose
    mantissa bit is 0; beyond 6 the largest magnitude; the sign kept at zero."""
    mags = Q.e2m1_value(np.arange(8))
    out = []
    for x in np.asarray(v, dtype=np.float64).ravel():
        a = min(abs(x), 6.0)
        d = np.abs(mags - a)
        best = np.flatnonzero(d == d.min())
        if len(best) > 1:
            best = [b for b in best if b % 2 == 0]
        out.append(int(best[0]) | (8 if np.signbit(x) else 0))
    return np.array(out, dtype=np.uint8)


def test_e2m1_round_matches_brute_force():
    grid = np.arange(-7.5, 7.5, 1 / 64, dtype=np.float64)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    extra = np.concatenate([mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 10),
                            [0.0, -0.0, 1e-30, -1e-30, 6.0, 6.5, 100.0, -100.0]])
    v = np.concatenate([grid, extra]).astype(F32)
    assert (Q.e2m1_round(v) == _brute_round(v)).all()
    # ties: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    assert Q.e2m1_value(Q.e2m1_round(mids)).tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def test_e4m3_code_round_trips():
    v = np.unique(np.abs(Q.e4m3_round(np.linspace(0, 448, 20001))))
    assert (Q.e4m3_value(Q.e4m3_code(v)) == v).all()
    assert Q.e4m3_code(np.array([448.0]))[0] == 0x7E and Q.e4m3_code(np.array([2.0 ** -9]))[0] == 1


def _rng(seed):
    return np.random.default_rng(seed)


def test_zero_row_and_zero_block():
    x = np.zeros((3, 64), dtype=F32)
    x[1, 16:32] = _rng(1).standard_normal(16)
    x[2, 5] = F32(1e-40)                 # a subnormal row maximum: 2688 / amax overflows fp32
    codes, sb, s = Q.quantize_rows(x)
    assert (codes[0] == 0).all() and (sb[0] == 0).all() and s[0] == 0
    assert (codes[2] == 0).all() and (sb[2] == 0).all() and s[2] == 0
    assert (codes[1, :16] == 0).all() and (codes[1, 32:] == 0).all() and sb[1, 0] == 0 and sb[1, 1] > 0


def _representable_rows(rng, rows, k, j):
    """Rows whose blocks are E2M1 values times an e4m3 block scale times 2^j, with the
    block maximum 6 and one block reaching the row maximum 6 * 448 * 2^j."""
    codes = rng.integers(0, 16, size=(rows, k)).astype(np.uint8)
    codes[:, ::16] = 7                                  # every block holds a 6
    sbv = Q.e4m3_round(rng.uniform(0.05, 448, size=(rows, k // 16)))
    sbv[:, 0] = 448.0
    x = Q.e2m1_value(codes).reshape(rows, k // 16, 16) * sbv[:, :, None] * 2.0 ** j
    return x.reshape(rows, k), codes, sbv


@pytest.mark.parametrize("j", [-20, -3, 0, 5])
def test_round_trip_on_representable_rows(j):
    x, codes, sbv = _representable_rows(_rng(2), 4, 256, j)
    c, sb, s = Q.quantize_rows(x)
    assert (Q.e2m1_value(c) == Q.e2m1_value(codes)).all()   # -0 and +0 compare equal
    assert (Q.e4m3_value(sb) == sbv).all()
    assert (s == F32(2.0 ** j)).all()
    assert (Q.dequantize(c, sb, s) == x).all()


def test_power_of_two_equivariance():
    x = (_rng(3).standard_normal((6, 512)) * _rng(4).uniform(0.1, 10, size=(6, 1))).astype(F32)
    c0, sb0, s0 = Q.quantize_rows(x)
    for j in (-7, 4, 11):
        c, sb, s = Q.quantize_rows(x * F32(2.0 ** j))
        assert (c == c0).all() and (sb == sb0).all() and (s == s0 * F32(2.0 ** j)).all()


def test_error_bound():
    x = (_rng(5).standard_normal((8, 1024)) ** 3).astype(F32)
    c, sb, s = Q.quantize_rows(x)
    xh = Q.dequantize(c, sb, s)
    # per block: the step of E2M1 at the element's magnitude is at most 2 (between 4 and 6),
    # so |x - x^| <= 1 block unit, where one unit is e4m3(sb) * s_row (plus fp32 slack);
    # the block scale rounds bmax / 6 to within 1/16, so saturation costs at most 6/16 units
    unit = (Q.e4m3_value(sb) * s[:, None].astype(np.float64))
    err = np.abs(x.astype(np.float64) - xh).reshape(8, 64, 16)
    assert (err <= unit[:, :, None] * (1.0 + 1e-5) + 1e-30).all()
    # and relative to the row: a typical element is far finer than the row maximum
    assert np.linalg.norm(x - xh) / np.linalg.norm(x) < 0.1


def test_linear_is_exact_when_quantization_is_lossless():
    rng = _rng(6)
    a, _, _ = _representable_rows(rng, 5, 256, -4)
    w, _, _ = _representable_rows(rng, 7, 256, -9)
    assert np.allclose(Q.nvfp4_linear(a, w), a @ w.T, rtol=1e-12, atol=0)


def test_storage_layout_inverse_and_packing():
    rng = _rng(7)
    sb = rng.integers(0, 127, size=(200, 768 // 16)).astype(np.uint8)
    buf = Q.tile_scales(sb)
    assert buf.size == 256 * 48          # rows padded to a pair of 128-row tiles
    assert (Q.untile_scales(buf, 200, 768) == sb).all()
    assert (buf.reshape(-1)[np.setdiff1d(np.arange(buf.size), Q.scale_tile_offset(*np.meshgrid(
        np.arange(200), np.arange(48), indexing="ij"), 768).ravel())] == 0).all()   # padding rows are zero
    codes = rng.integers(0, 16, size=(3, 64)).astype(np.uint8)
    assert (Q.unpack_codes(Q.pack_codes(codes)) == codes).all()
    assert Q.pack_codes(np.array([[1, 2]], dtype=np.uint8))[0, 0] == 0x21


def _tiny_block_args():
    import oracle as O
    from flow_matching_image_flux3_b300 import synth
    case = synth.config(0, bias=True)
    d = case.dims
    ang = O.rope_angles(case.pos.numpy(), d.rope_theta)
    w = [O.Weights(*(synth.as_f64(t) for t in (wi.w_in, wi.b_in, wi.q_norm, wi.k_norm, wi.w_out, wi.b_out)))
         for wi in case.weights]
    return O, (synth.as_f64(case.x), w, case.seg_off, synth.as_f64(case.mod), ang, d.heads)


@pytest.mark.parametrize("quant", ["fp8", "nvfp4"])
def test_quantized_block_rows_match_quantized_block(quant):
    # the sampled-rows path takes the same steps as the whole block, both projections quantized
    O, args = _tiny_block_args()
    kw = dict(rounding="bf16", out_proj_quant=quant, **({"fp8_in_proj": True} if quant == "fp8" else {"nvfp4_in_proj": True}))
    full = O.block_forward(*args, **kw)
    rows = [0, 5, 63, 64, 143]
    part = O.block_forward_rows(*args, rows, **kw)
    np.testing.assert_allclose(part["x_out"], full.x_out[rows], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("quant", ["fp8", "nvfp4"])
def test_quantized_block_is_close_to_the_bf16_block(quant):
    # not a pin of the arithmetic (the tests above are): quantizing both projections moves y
    # by a few percent (fp8) to ~10-20% (nvfp4) and x' by far less, since x dominates it
    O, args = _tiny_block_args()
    ref = O.block_forward(*args, rounding="bf16")
    kw = {"fp8_in_proj": True} if quant == "fp8" else {"nvfp4_in_proj": True}
    qb = O.block_forward(*args, rounding="bf16", out_proj_quant=quant, **kw)
    e_y = np.linalg.norm(qb.y - ref.y) / np.linalg.norm(ref.y)
    assert 1e-3 < e_y < (0.1 if quant == "fp8" else 0.3)
    assert np.linalg.norm(qb.x_out - ref.x_out) / np.linalg.norm(ref.x_out) < (2e-2 if quant == "fp8" else 0.1)
