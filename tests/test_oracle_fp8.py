"""Pins for the FP8 oracle (oracle/fp8.py).  Expected values come from torch's own
float8_e4m3fn cast, from exactness on representable inputs, and from invariants."""
import numpy as np
import pytest
import torch

import oracle as O
from oracle import fp8 as Q
from flow_matching_image_flux3_b300 import synth
from tests.common import rel_l2, oracle_block

rng = np.random.default_rng(8)


def test_e4m3_round_matches_torch_cast():
    mag = 2.0 ** rng.uniform(-12, np.log2(448.0), 50000)
    v = (np.sign(rng.standard_normal(50000)) * mag).astype(np.float32)
    # exact ties between neighbouring codes, the largest values, zero and subnormals
    ties = np.array([1.0625, 1.1875, 0.0029296875, 440.0, 448.0, 464.0 - 1e-3, 0.0, -0.0, 2 ** -9, 3 * 2 ** -10],
                    dtype=np.float32)
    v = np.concatenate([v, ties, -ties])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(Q.e4m3_round(v.astype(np.float64)), ref)
    assert Q.e4m3_round(np.array([1e6, -500.0])).tolist() == [448.0, -448.0]   # saturation


def test_quantize_rows_exact_on_representable_rows():
    # rows already e4m3 codes times a power of two, with 448 present: lossless
    codes = torch.randint(-126, 127, (8, 64), dtype=torch.int8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    codes = np.nan_to_num(codes)
    codes[:, 0] = 448.0
    x = codes * (2.0 ** rng.integers(-8, 8, (8, 1)))
    q, s = Q.quantize_rows(x)
    np.testing.assert_array_equal(q * s[:, None], x)
    np.testing.assert_array_equal(np.abs(q).max(1), 448.0)


def test_quantize_rows_invariants_and_error_bound():
    x = rng.standard_normal((16, 256)).astype(np.float32).astype(np.float64)
    q, s = Q.quantize_rows(x)
    q2, s2 = Q.quantize_rows(x * 8.0)
    np.testing.assert_array_equal(q2, q)            # power-of-two scaling commutes
    np.testing.assert_array_equal(s2, s * 8.0)
    # a normal e4m3 value is within 2^-4 of its input relatively, a subnormal within 2^-10 * scale
    err = np.abs(q * s[:, None] - x)
    assert np.all(err <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * s[:, None]) * (1 + 1e-6))
    z, sz = Q.quantize_rows(np.zeros((2, 32)))
    assert np.all(z == 0) and np.all(sz == 0)


def test_fp8_linear_exact_when_quantization_is_lossless():
    codes = lambda shape: np.nan_to_num(torch.randint(-126, 127, shape, dtype=torch.int8)
                                        .view(torch.float8_e4m3fn).to(torch.float64).numpy())
    a, w = codes((6, 128)), codes((10, 128))
    a[:, 3] = 448.0
    w[:, 5] = -448.0
    a *= 2.0 ** -5
    np.testing.assert_array_equal(Q.fp8_linear(a, w), a @ w.T)


def test_fp8_block_is_close_to_the_bf16_block():
    # not a pin of the arithmetic (the tests above are): the quantized projection changes
    # the block's output by a few percent of y, far less than x itself
    case = synth.config(0, bias=True)
    ref = oracle_block(case, rounding="bf16")
    d = case.dims
    ang = O.rope_angles(case.pos.numpy(), d.rope_theta)
    w = [O.Weights(*(synth.as_f64(t) for t in (wi.w_in, wi.b_in, wi.q_norm, wi.k_norm, wi.w_out, wi.b_out)))
         for wi in case.weights]
    f8 = O.block_forward(synth.as_f64(case.x), w, case.seg_off, synth.as_f64(case.mod), ang, d.heads,
                         rounding="bf16", fp8_in_proj=True)
    assert 1e-3 < rel_l2(f8.y, ref.y) < 0.1
    assert rel_l2(f8.x_out, ref.x_out) < 2e-2


def test_fp8_rows_match_fp8_block():
    case = synth.config(0, bias=True)
    d = case.dims
    ang = O.rope_angles(case.pos.numpy(), d.rope_theta)
    w = [O.Weights(*(synth.as_f64(t) for t in (wi.w_in, wi.b_in, wi.q_norm, wi.k_norm, wi.w_out, wi.b_out)))
         for wi in case.weights]
    args = (synth.as_f64(case.x), w, case.seg_off, synth.as_f64(case.mod), ang, d.heads)
    full = O.block_forward(*args, rounding="bf16", fp8_in_proj=True)
    rows = [0, 5, 63, 64, 143]
    part = O.block_forward_rows(*args, rows, rounding="bf16", fp8_in_proj=True)
    np.testing.assert_allclose(part["x_out"], full.x_out[rows], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(part["k"], full.k, rtol=1e-12, atol=1e-12)
