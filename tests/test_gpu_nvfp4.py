"""Parity of the NVFP4 input projection (through the C-ABI) with the oracle: the
quantizer's codes, tiled block scales and row scales bit for bit, the block-scaled
projection on the same codes, and the block."""
import numpy as np
import pytest
import torch

import oracle as O
from oracle import nvfp4 as Q4
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


def _check_quantized(x_bf16, q, sf, sc, rows=None):
    """Device codes / scales against the oracle on the same bf16 values (rows: a sample)."""
    xs = x_bf16 if rows is None else x_bf16[rows]
    codes, sb, s = Q4.quantize_rows(f64(xs))
    qd = q.cpu().numpy() if rows is None else q.cpu().numpy()[rows]
    np.testing.assert_array_equal(qd, Q4.pack_codes(codes))
    n, k = x_bf16.shape
    buf = sf.cpu().numpy()
    assert buf.size == Q4.scale_bytes(n, k)
    if rows is None:
        np.testing.assert_array_equal(buf, Q4.tile_scales(sb))
    else:
        r, j = np.meshgrid(np.asarray(rows), np.arange(k // 16), indexing="ij")
        np.testing.assert_array_equal(buf[Q4.scale_tile_offset(r, j, k)], sb)
    scd = sc.cpu().numpy() if rows is None else sc.cpu().numpy()[rows]
    np.testing.assert_array_equal(scd, s)


@pytest.mark.parametrize("rows,k", [(300, 3072), (1, 256), (129, 768)])
def test_quantize_rows_bitwise(rows, k):
    g = torch.Generator("cpu").manual_seed(41 + rows)
    x = torch.randn(rows, k, generator=g) * (10.0 ** torch.randint(-3, 3, (rows, 1), generator=g))
    if rows > 10:
        x[7] = 0.0                      # an all-zero row
        x[8, 100] = 5e4                 # one outlier: most of the row's blocks get tiny scales
        x[9, :16] = 0.0                 # a zero block inside a live row
        x[10] = 0.0
        x[10, 3] = 1e-39                # a subnormal row maximum: g overflows, a zero row
    x = x.to(torch.bfloat16)
    q, sf, sc = B.quantize_rows_nvfp4(x.cuda())
    _check_quantized(x, q, sf, sc)


def test_quantize_full_size_weight_rows_bitwise():
    w = synth.draw_weights(torch.Generator("cpu").manual_seed(42), synth.FULL).w_in   # [27648, 3072]
    q, sf, sc = B.quantize_rows_nvfp4(w.cuda())
    rows = np.sort(np.random.default_rng(0).choice(w.shape[0], 64, replace=False))
    _check_quantized(w, q, sf, sc, rows)


@pytest.mark.parametrize("streams", [
    [synth.Stream("image", 64, (8, 8)), synth.text_stream(80)],
    [synth.Stream("image", 1, (1, 1))],
    [synth.Stream("image", 130, (10, 13)), synth.text_stream(160)],
], ids=["tiny", "n1", "ragged"])
def test_in_proj_nvfp4(streams):
    case = synth.make_case(synth.TINY, streams, seed=43, stage=2, bias=True)
    dims, n = case.dims, case.n
    a = (torch.randn(n, dims.width, generator=torch.Generator("cpu").manual_seed(44))).to(torch.bfloat16)
    w = B.Nvfp4Weights(DevWeights(case.weights[0]))
    rope = B.rope_build(dims, case.pos.cuda())
    a4, asf, sa = B.quantize_rows_nvfp4(a.cuda())
    q, k, vt, y = B.in_proj_nvfp4_fwd(dims, w, a4, asf, sa, rope)
    rq, rk, rv, ract = TP._in_proj_oracle(f64(a), [oracle_weights(case.weights[0])], case.seg_off,
                                          case.pos.numpy(), dims, 2, nvfp4=True)
    assert_close("q", f64(q).transpose(1, 0, 2), rq)
    assert_close("k", f64(k).transpose(1, 0, 2), rk)
    assert_close("v", f64(vt)[:, :, :n].transpose(2, 0, 1), rv)
    assert_close("act", f64(y)[:, dims.width:], ract)
    assert torch.all(y[:, :dims.width] == 0)  # attention columns untouched


def test_in_proj_nvfp4_full_size_sampled():
    # the full input projection (4,256 tokens x 27,648 outputs) against the oracle's
    # projection of sampled rows: values of V (no normalisation) and of the SwiGLU output
    case = synth.config(1)
    dims, n = case.dims, case.n
    D, F = dims.width, dims.ffn_hidden
    a = (torch.randn(n, D, generator=torch.Generator("cpu").manual_seed(45))).to(torch.bfloat16)
    w = B.Nvfp4Weights(DevWeights(case.weights[0], bias=False))
    rope = B.rope_build(dims, case.pos.cuda())
    a4, asf, sa = B.quantize_rows_nvfp4(a.cuda())
    q, k, vt, y = B.in_proj_nvfp4_fwd(dims, w, a4, asf, sa, rope)
    torch.cuda.synchronize()
    rows = TP._sample_rows(case)
    ow = oracle_weights(case.weights[0])
    p = Q4.nvfp4_linear(f64(a)[rows], ow.w_in)
    assert_close("v (rows)", f64(vt)[:, :, rows].transpose(2, 0, 1).reshape(len(rows), D), p[:, 2 * D:3 * D])
    assert_close("act (rows)", f64(y)[rows, D:], O.swiglu(p[:, 3 * D:3 * D + F], p[:, 3 * D + F:]))


def test_block_nvfp4_tiny():
    case = synth.config(0, bias=True)
    d = case.dims
    w = B.Nvfp4Weights(DevWeights(case.weights[0]))
    rope = B.rope_build(d, case.pos.cuda())
    out = B.block_nvfp4_fwd(d, w, case.seg_off, case.mod.cuda(), case.x.cuda(), rope)
    ang = O.rope_angles(case.pos.numpy(), d.rope_theta)
    ref = O.block_forward(synth.as_f64(case.x), [oracle_weights(case.weights[0])], case.seg_off,
                          synth.as_f64(case.mod), ang, d.heads, rounding="bf16", nvfp4_in_proj=True)
    assert_close("x_out (nvfp4 projection)", f64(out), ref.x_out)


def test_block_nvfp4_full_size_sampled():
    case = synth.config(1)
    d = case.dims
    w = B.Nvfp4Weights(DevWeights(case.weights[0], bias=False))
    rope = B.rope_build(d, case.pos.cuda())
    out = B.block_nvfp4_fwd(d, w, case.seg_off, case.mod.cuda(), case.x.cuda(), rope)
    torch.cuda.synchronize()
    rows = TP._sample_rows(case)
    ang = O.rope_angles(case.pos.numpy(), d.rope_theta)
    ref = O.block_forward_rows(synth.as_f64(case.x), [oracle_weights(case.weights[0])], case.seg_off,
                               synth.as_f64(case.mod), ang, d.heads, rows, rounding="bf16", nvfp4_in_proj=True)
    assert_close("x_out (rows, nvfp4 projection)", f64(out[rows]), ref["x_out"])


@pytest.mark.parametrize("cfg", [0, 1])
def test_block_nvfp4_both_projections(cfg):
    """Both projections on NVFP4 operands: tiny (every row) and the full 4,256-token block
    (sampled rows)."""
    case = synth.config(cfg, bias=cfg == 0)
    d = case.dims
    w = B.Nvfp4Weights(DevWeights(case.weights[0], bias=cfg == 0), quantize_out=True)
    rope = B.rope_build(d, case.pos.cuda())
    out = B.block_nvfp4_fwd(d, w, case.seg_off, case.mod.cuda(), case.x.cuda(), rope)
    torch.cuda.synchronize()
    ang = O.rope_angles(case.pos.numpy(), d.rope_theta)
    args = (synth.as_f64(case.x), [oracle_weights(case.weights[0])], case.seg_off, synth.as_f64(case.mod), ang, d.heads)
    kw = dict(rounding="bf16", nvfp4_in_proj=True, out_proj_quant="nvfp4")
    if cfg == 0:
        assert_close("x_out (nvfp4 projections)", f64(out), O.block_forward(*args, **kw).x_out)
    else:
        rows = TP._sample_rows(case)
        ref = O.block_forward_rows(*args, rows, **kw)
        assert_close("x_out (rows, nvfp4 projections)", f64(out[rows]), ref["x_out"])
