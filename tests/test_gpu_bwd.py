"""Parity of the joint block's backward pass (flux3_block_bwd, through the C-ABI) with the
backward oracle (float64, pinned to finite differences of the forward oracle)."""
import numpy as np
import pytest
import torch

import oracle as O
from oracle.backward import block_backward
from flow_matching_image_flux3_b300 import synth
from tests.common import f64, DevWeights, oracle_weights, rel_l2

pytestmark = pytest.mark.gpu
B = None

# The bar, per gradient: relative L2 error.  The device path keeps the forward pass's bf16
# tensors (a, q, k, the projections, [O | act]) and rounds the backward's GEMM operands to
# bf16 (dy, d[O | act], the attention probabilities and dS, dP); each rounding is a relative
# error of at most 2^-9 per element, and a gradient is a sum over many such products, so
# its relative L2 error stays near that scale; 2e-2 leaves a margin of about ten.
GRAD_REL_L2 = 2e-2
KEYS = ["dx", "dw_in", "db_in", "dq_norm", "dk_norm", "dw_out", "db_out", "dmod"]


@pytest.fixture(scope="module", autouse=True)
def lib():
    global B
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from flow_matching_image_flux3_b300 import build
    build.build()
    from flow_matching_image_flux3_b300 import binding
    B = binding
    yield binding
    assert binding.device_error(reset=True) == 0, "a device-side wait timed out"


def _run(case, bias, seed):
    d = case.dims
    dxo = torch.randn(case.n, d.width, generator=torch.Generator("cpu").manual_seed(seed))
    w = DevWeights(case.weights[0], bias=bias)
    rope = B.rope_build(d, case.pos.cuda())
    got = B.block_bwd(d, w, case.seg_off, case.mod.cuda(), case.x.cuda(), rope, dxo.cuda())
    torch.cuda.synchronize()
    ow = oracle_weights(case.weights[0])
    if not bias:
        ow.b_in = np.zeros_like(ow.b_in)
        ow.b_out = np.zeros_like(ow.b_out)
    ang = O.rope_angles(case.pos.numpy(), d.rope_theta)
    ref = block_backward(synth.as_f64(case.x), ow, case.seg_off, synth.as_f64(case.mod), ang, d.heads,
                         dxo.double().numpy(), ln_eps=d.ln_eps, rms_eps=d.rms_eps)
    return got, ref


@pytest.mark.parametrize("streams,bias", [
    ([synth.Stream("image", 64, (8, 8)), synth.text_stream(80)], True),
    ([synth.Stream("image", 130, (10, 13)), synth.text_stream(160), synth.Stream("ref", 35, (5, 7), t=1)], False),
], ids=["tiny", "ragged3"])
def test_block_backward(streams, bias):
    case = synth.make_case(synth.TINY, streams, seed=51, stage=2, bias=bias)
    got, ref = _run(case, bias, 52)
    errs = {k: rel_l2(f64(got[k]), ref[k]) for k in KEYS}
    print(errs)
    for k in KEYS:
        assert np.all(np.isfinite(f64(got[k]))), k
        assert errs[k] <= GRAD_REL_L2, (k, errs[k])


def test_block_backward_full_size():
    case = synth.config(1)
    got, ref = _run(case, False, 53)
    errs = {k: rel_l2(f64(got[k]), ref[k]) for k in KEYS}
    print(errs)
    for k in KEYS:
        assert errs[k] <= GRAD_REL_L2, (k, errs[k])


def test_stream_block_backward_stage1():
    """The stage-1 block (a weight set per stream, attention inside each stream): every
    stream's gradients against the backward oracle run on that stream alone, dx on all rows."""
    streams = [synth.Stream("image", 130, (10, 13)), synth.text_stream(160), synth.Stream("ref", 35, (5, 7), t=1)]
    case = synth.make_case(synth.TINY, streams, seed=54, stage=1, bias=True)
    d = case.dims
    dxo = torch.randn(case.n, d.width, generator=torch.Generator("cpu").manual_seed(55))
    ws = [DevWeights(w) for w in case.weights]
    rope = B.rope_build(d, case.pos.cuda())
    got = B.stream_block_bwd(d, ws, case.seg_off, case.mod.cuda(), case.x.cuda(), rope, dxo.cuda())
    torch.cuda.synchronize()
    ang = O.rope_angles(case.pos.numpy(), d.rope_theta)
    x64, mod64 = synth.as_f64(case.x), synth.as_f64(case.mod)
    dx_ref = np.empty(x64.shape)
    for g in range(len(case.seg_off) - 1):
        lo, hi = case.seg_off[g], case.seg_off[g + 1]
        ref = block_backward(x64[lo:hi], oracle_weights(case.weights[g]), [0, hi - lo], mod64[g:g + 1], ang[lo:hi],
                             d.heads, dxo[lo:hi].double().numpy(), ln_eps=d.ln_eps, rms_eps=d.rms_eps)
        dx_ref[lo:hi] = ref["dx"]
        for k in KEYS[1:]:
            e = rel_l2(f64(got[k][g]), ref[k] if k != "dmod" else ref[k][0])
            assert e <= GRAD_REL_L2, (g, k, e)
    assert rel_l2(f64(got["dx"]), dx_ref) <= GRAD_REL_L2
