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


def test_stage1_backward_is_the_per_stream_joint_backward():
    """The stage-1 block gives every stream its own weights and attention inside the stream,
    so its gradients are the joint block's gradients of each stream on its own rows: checked
    against central finite differences of the stage-1 forward oracle."""
    dims = synth.TINY
    g = torch.Generator("cpu").manual_seed(8)
    streams = [synth.Stream("image", 24, (4, 6)), synth.text_stream(20), synth.Stream("ref", 12, (3, 4), t=1)]
    seg = [0, 24, 44, 56]
    pos = synth.positions(streams).numpy()
    ws = [oracle_weights(synth.draw_weights(g, dims, True)) for _ in range(3)]
    mod = synth.as_f64(synth.draw_mod(g, 3, dims.width))
    rng = np.random.default_rng(9)
    x = rng.standard_normal((56, dims.width))
    dxo = rng.standard_normal(x.shape)
    ang = O.rope_angles(pos, dims.rope_theta)

    def loss(xx, wl):
        out = O.block_forward(xx, wl, seg, mod, ang, dims.heads, ln_eps=dims.ln_eps, rms_eps=dims.rms_eps, stage=1)
        return float((out.x_out * dxo).sum())

    dx = np.empty_like(x)
    dwin = []
    for s in range(3):
        lo, hi = seg[s], seg[s + 1]
        gr = block_backward(x[lo:hi], ws[s], [0, hi - lo], mod[s:s + 1], ang[lo:hi], dims.heads, dxo[lo:hi],
                            ln_eps=dims.ln_eps, rms_eps=dims.rms_eps)
        dx[lo:hi] = gr["dx"]
        dwin.append(gr["dw_in"])
    eps = 1e-5
    v = rng.standard_normal(x.shape)
    fd = (loss(x + eps * v, ws) - loss(x - eps * v, ws)) / (2 * eps)
    assert abs(fd - float((dx * v).sum())) <= 1e-6 * max(1.0, abs(fd))
    for s in range(3):   # each stream's W_in
        vw = rng.standard_normal(ws[s].w_in.shape)
        wp, wm = list(ws), list(ws)
        wp[s], wm[s] = copy.copy(ws[s]), copy.copy(ws[s])
        wp[s].w_in = ws[s].w_in + eps * vw
        wm[s].w_in = ws[s].w_in - eps * vw
        fd = (loss(x, wp) - loss(x, wm)) / (2 * eps)
        assert abs(fd - float((dwin[s] * vw).sum())) <= 1e-6 * max(1.0, abs(fd)), s
