"""Pins of the backward oracle (oracle/backward.py): every gradient against central finite
differences of the forward oracle in float64, along random directions, plus special cases."""
import copy

import numpy as np
import pytest
import torch

import oracle as O
from oracle.backward import block_backward
from flow_matching_image_flux3_b300 import synth
from tests.common import oracle_weights


def _case(seed=0, n_img=(4, 6), n_txt=20):
    dims = synth.TINY
    g = torch.Generator("cpu").manual_seed(seed)
    streams = [synth.Stream("image", n_img[0] * n_img[1], n_img), synth.text_stream(n_txt)]
    seg = [0, streams[0].n, streams[0].n + n_txt]
    pos = synth.positions(streams).numpy()
    w = oracle_weights(synth.draw_weights(g, dims, True))
    w.b_in = np.random.default_rng(seed).standard_normal(w.b_in.shape) * 0.1
    w.b_out = np.random.default_rng(seed + 1).standard_normal(w.b_out.shape) * 0.1
    mod = synth.as_f64(synth.draw_mod(g, 2, dims.width))
    x = np.random.default_rng(seed + 2).standard_normal((seg[-1], dims.width))
    dxo = np.random.default_rng(seed + 3).standard_normal(x.shape)
    ang = O.rope_angles(pos, dims.rope_theta)
    return dims, x, w, seg, mod, ang, dxo


def _loss(dims, x, w, seg, mod, ang, dxo):
    out = O.block_forward(x, [w], seg, mod, ang, dims.heads, ln_eps=dims.ln_eps, rms_eps=dims.rms_eps, stage=2)
    return float((out.x_out * dxo).sum())


# (gradient key, how to perturb the inputs along direction v by eps)
def _perturb(name, eps, v, x, w, mod):
    x2, w2, m2 = x, copy.copy(w), mod
    if name == "dx":
        x2 = x + eps * v
    elif name == "dmod":
        m2 = mod + eps * v
    else:
        attr = {"dw_in": "w_in", "db_in": "b_in", "dq_norm": "q_norm", "dk_norm": "k_norm", "dw_out": "w_out",
                "db_out": "b_out"}[name]
        setattr(w2, attr, getattr(w, attr) + eps * v)
    return x2, w2, m2


@pytest.mark.parametrize("name", ["dx", "dw_in", "db_in", "dq_norm", "dk_norm", "dw_out", "db_out", "dmod"])
def test_gradient_matches_finite_differences(name):
    dims, x, w, seg, mod, ang, dxo = _case()
    grads = block_backward(x, w, seg, mod, ang, dims.heads, dxo, ln_eps=dims.ln_eps, rms_eps=dims.rms_eps)
    rng = np.random.default_rng(hash(name) % 2 ** 32)
    gr = grads[name]
    for _ in range(2):
        v = rng.standard_normal(gr.shape)
        eps = 1e-5
        xp, wp, mp = _perturb(name, eps, v, x, w, mod)
        xm, wm, mm = _perturb(name, -eps, v, x, w, mod)
        fd = (_loss(dims, xp, wp, seg, mp, ang, dxo) - _loss(dims, xm, wm, seg, mm, ang, dxo)) / (2 * eps)
        an = float((gr * v).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_zero_gate_stops_the_weight_gradients():
    dims, x, w, seg, mod, ang, dxo = _case(1)
    mod = mod.copy()
    mod[:, 2] = 0.0
    gr = block_backward(x, w, seg, mod, ang, dims.heads, dxo, ln_eps=dims.ln_eps, rms_eps=dims.rms_eps)
    for k in ("dw_in", "db_in", "dq_norm", "dk_norm", "dw_out", "db_out"):
        assert np.all(gr[k] == 0.0), k
    assert np.array_equal(gr["dx"], dxo)            # x' = x: the gradient passes straight through
    assert np.all(gr["dmod"][:, :2] == 0.0) and np.any(gr["dmod"][:, 2] != 0.0)


def test_single_token_attention_passes_v_through():
    # one token: softmax over one key is 1, so dv = dO and no gradient reaches q or k
    dims, x, w, seg, mod, ang, dxo = _case(2, n_img=(1, 1), n_txt=0)
    seg = [0, 1]
    mod = mod[:1]
    gr = block_backward(x, w, seg, mod, ang, dims.heads, dxo, ln_eps=dims.ln_eps, rms_eps=dims.rms_eps)
    D = dims.width
    assert np.allclose(gr["dp"][:, 0:2 * D], 0.0, atol=1e-12)
    assert np.allclose(gr["dp"][:, 2 * D:3 * D], gr["dycat"][:, 0:D], rtol=1e-12, atol=1e-12)
