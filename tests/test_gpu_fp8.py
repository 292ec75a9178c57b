"""Parity of the FP8 (e4m3) row-wise input projection (through the C-ABI) with the oracle:
the quantizer's codes bit for bit, the FP8 projection on the same codes, and the block."""
import numpy as np
import pytest
import torch

import oracle as O
from oracle import fp8 as Q8
from flow_matching_image_flux3_b300 import synth
from tests.common import assert_close, f64, DevWeights, oracle_weights
from tests import test_gpu_parity as TP

pytestmark = pytest.mark.gpu
B = None


@pytest.fixture(scope="module", autouse=True)
def lib():
    global B
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from flow_matching_image_flux3_b300 import build
    build.build()
    from flow_matching_image_flux3_b300 import binding
    B = binding
    TP.B = binding
    yield binding
    assert binding.device_error(reset=True) == 0, "a device-side wait timed out"


def _codes(q: torch.Tensor) -> np.ndarray:
    return q.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_quantize_rows_bitwise():
    g = torch.Generator("cpu").manual_seed(31)
    x = torch.randn(300, 3072, generator=g) * (10.0 ** torch.randint(-3, 3, (300, 1), generator=g))
    x[7] = 0.0                     # an all-zero row
    x[8, 100] = 5e4                # one outlier dominates its row's scale
    x = x.to(torch.bfloat16)
    q, sc = B.quantize_rows_fp8(x.cuda())
    rq, rs = Q8.quantize_rows(f64(x))
    np.testing.assert_array_equal(_codes(q), rq)
    np.testing.assert_array_equal(sc.cpu().numpy().astype(np.float64), rs)


def test_quantize_full_size_weight_rows_bitwise():
    w = synth.draw_weights(torch.Generator("cpu").manual_seed(32), synth.FULL).w_in   # [27648, 3072]
    q, sc = B.quantize_rows_fp8(w.cuda())
    rows = np.random.default_rng(0).choice(w.shape[0], 64, replace=False)
    rq, rs = Q8.quantize_rows(f64(w[rows]))
    np.testing.assert_array_equal(_codes(q[rows]), rq)
    np.testing.assert_array_equal(sc.cpu().numpy()[rows].astype(np.float64), rs)


@pytest.mark.parametrize("streams,stage", [
    ([synth.Stream("image", 64, (8, 8)), synth.text_stream(80)], 2),
    ([synth.Stream("image", 130, (10, 13)), synth.text_stream(160)], 2),
    ([synth.Stream("image", 48, (6, 8)), synth.text_stream(80), synth.Stream("ref", 35, (5, 7), t=1)], 1),
], ids=["tiny", "ragged", "stage1"])
def test_in_proj_fp8(streams, stage):
    case = synth.make_case(synth.TINY, streams, seed=33, stage=stage, bias=True)
    dims, n = case.dims, case.n
    a = (torch.randn(n, dims.width, generator=torch.Generator("cpu").manual_seed(34))).to(torch.bfloat16)
    dw = [B.Fp8Weights(DevWeights(w)) for w in case.weights]
    rope = B.rope_build(dims, case.pos.cuda())
    a8, sa = B.quantize_rows_fp8(a.cuda())
    q, k, vt, y = B.in_proj_fp8_fwd(dims, dw, case.seg_off, a8, sa, rope)
    rq, rk, rv, ract = TP._in_proj_oracle(f64(a), [oracle_weights(w) for w in case.weights], case.seg_off,
                                          case.pos.numpy(), dims, stage, fp8=True)
    assert_close("q", f64(q).transpose(1, 0, 2), rq)
    assert_close("k", f64(k).transpose(1, 0, 2), rk)
    assert_close("v", f64(vt)[:, :, :n].transpose(2, 0, 1), rv)
    assert_close("act", f64(y)[:, dims.width:], ract)


def test_block_fp8_tiny():
    case = synth.config(0, bias=True)
    d = case.dims
    w = B.Fp8Weights(DevWeights(case.weights[0]))
    rope = B.rope_build(d, case.pos.cuda())
    out = B.block_fp8_fwd(d, w, case.seg_off, case.mod.cuda(), case.x.cuda(), rope)
    ang = O.rope_angles(case.pos.numpy(), d.rope_theta)
    ref = O.block_forward(synth.as_f64(case.x), [oracle_weights(case.weights[0])], case.seg_off,
                          synth.as_f64(case.mod), ang, d.heads, rounding="bf16", fp8_in_proj=True)
    assert_close("x_out (fp8 projection)", f64(out), ref.x_out)


def test_block_fp8_full_size_sampled():
    case = synth.config(1)
    d, n = case.dims, case.n
    w = B.Fp8Weights(DevWeights(case.weights[0], bias=False))
    rope = B.rope_build(d, case.pos.cuda())
    out = B.block_fp8_fwd(d, w, case.seg_off, case.mod.cuda(), case.x.cuda(), rope)
    torch.cuda.synchronize()
    rows = TP._sample_rows(case)
    ang = O.rope_angles(case.pos.numpy(), d.rope_theta)
    ref = O.block_forward_rows(synth.as_f64(case.x), [oracle_weights(case.weights[0])], case.seg_off,
                               synth.as_f64(case.mod), ang, d.heads, rows, rounding="bf16", fp8_in_proj=True)
    assert_close("x_out (rows, fp8 projection)", f64(out[rows]), ref["x_out"])


@pytest.mark.parametrize("cfg", [0, 1])
def test_block_fp8_both_projections(cfg):
    """Both projections on row-wise e4m3 operands: tiny (every row) and the full 4,256-token
    block (sampled rows)."""
    case = synth.config(cfg, bias=cfg == 0)
    d = case.dims
    w = B.Fp8Weights(DevWeights(case.weights[0], bias=cfg == 0), quantize_out=True)
    rope = B.rope_build(d, case.pos.cuda())
    out = B.block_fp8_fwd(d, w, case.seg_off, case.mod.cuda(), case.x.cuda(), rope)
    torch.cuda.synchronize()
    ang = O.rope_angles(case.pos.numpy(), d.rope_theta)
    args = (synth.as_f64(case.x), [oracle_weights(case.weights[0])], case.seg_off, synth.as_f64(case.mod), ang, d.heads)
    kw = dict(rounding="bf16", fp8_in_proj=True, out_proj_quant="fp8")
    if cfg == 0:
        assert_close("x_out (fp8 projections)", f64(out), O.block_forward(*args, **kw).x_out)
    else:
        rows = TP._sample_rows(case)
        ref = O.block_forward_rows(*args, rows, **kw)
        assert_close("x_out (rows, fp8 projections)", f64(out[rows]), ref["x_out"])
