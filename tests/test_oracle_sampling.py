"""Pins for the sampling-loop oracle (oracle/sampling.py).  None re-uses the oracle's own
code for the expected value: the pages' own numbers, closed forms, and exact integration."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import sampling as S

GOLD = os.path.join(os.path.dirname(__file__), "golden")
FACTS = json.load(open(os.path.join(GOLD, "page_facts.json")))
rng = np.random.default_rng(77)


def test_44_of_50_steps_run_above_half_sigma():
    # "Welcome FLUX.3 Image Klein in Diffusers", 'How it works': time shift 6.93, so 44 of
    # 50 steps run above sigma = 0.5 (a step runs at the level it starts from)
    alpha, n, above = FACTS["time_shift"]["value"], FACTS["steps_base"]["value"], FACTS["steps_above_half_sigma"]["value"]
    s = S.sigma_schedule(n, alpha)
    assert len(s) == n + 1 and s[0] == 1.0 and s[-1] == 0.0
    assert int(np.sum(s[:n] > 0.5)) == above
    # the statement pins the grid: a 50-point linspace(1, 0) grid would give 43, no shift 25
    lin = 1.0 - np.arange(n) / (n - 1)
    shifted = alpha * lin / (1 + (alpha - 1) * lin)
    assert int(np.sum(shifted > 0.5)) == 43
    assert int(np.sum(S.sigma_schedule(n, 1.0)[:n] > 0.5)) == 25


def test_time_shift_closed_forms():
    for alpha in (1.0, 3.0, 6.93):
        assert S.time_shift(0.0, alpha) == 0.0 and S.time_shift(1.0, alpha) == 1.0
        # sigma' = 1/2 exactly at sigma = 1 / (alpha + 1)
        assert S.time_shift(1.0 / (alpha + 1.0), alpha) == pytest.approx(0.5, abs=1e-15)
    sig = rng.random(1000)
    np.testing.assert_array_equal(S.time_shift(sig, 1.0), sig)
    assert np.all(np.diff(S.time_shift(np.sort(sig), 6.93)) >= 0)
    # shifting by alpha then by beta is one shift by alpha * beta
    np.testing.assert_allclose(S.time_shift(S.time_shift(sig, 2.5), 3.0), S.time_shift(sig, 7.5), rtol=1e-14)


def test_cfg_special_cases():
    vp, vn = rng.standard_normal((5, 7)), rng.standard_normal((5, 7))
    # exact in real arithmetic; v_neg + 1 * (v_pos - v_neg) may differ from v_pos by an ulp
    np.testing.assert_allclose(S.cfg(vp, vn, 1.0), vp, rtol=0, atol=1e-15)
    np.testing.assert_array_equal(S.cfg(vp, vn, 0.0), vn)
    np.testing.assert_allclose(S.cfg(vp, vn, 2.0), 2 * vp - vn, rtol=1e-15)
    np.testing.assert_allclose(S.cfg(vp, vn, 3.5), vn + 3.5 * vp - 3.5 * vn, rtol=1e-14, atol=1e-14)


def test_embed_matches_torch_linear():
    x, w, b = rng.standard_normal((9, 128)), rng.standard_normal((64, 128)), rng.standard_normal(64)
    ref = torch.nn.functional.linear(torch.from_numpy(x), torch.from_numpy(w), torch.from_numpy(b)).numpy()
    np.testing.assert_allclose(S.embed(x, w, b), ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("cfg_scale", [1.0, 3.5])
def test_loop_integrates_the_straight_flow_exactly(cfg_scale):
    # along x(sigma) = (1 - sigma) d + sigma e the velocity e - d is constant, so Euler on
    # any grid from sigma = 1 (pure noise e) to 0 lands exactly on the data d
    d, e = rng.standard_normal((16, 128)), rng.standard_normal((16, 128))
    calls = []

    def velocity(x, i, prompted):
        calls.append((i, prompted))
        return (e - d) if prompted else (e - d) * 0.25 + 1.0  # negative branch differs

    guided = S.cfg(e - d, (e - d) * 0.25 + 1.0, cfg_scale)
    xs = S.sample(e, S.sigma_schedule(50, 6.93), velocity, cfg_scale)
    assert len(xs) == 51
    np.testing.assert_allclose(xs[-1], e - guided, rtol=1e-12, atol=1e-12)
    if cfg_scale == 1.0:
        np.testing.assert_allclose(xs[-1], d, rtol=1e-12, atol=1e-12)
        assert calls == [(i, True) for i in range(50)]
    else:
        assert calls == [(i, p) for i in range(50) for p in (True, False)]


def test_context_stage1_does_not_depend_on_the_image():
    """Welcome FLUX.3 Image Klein in Diffusers, "How it works": in stage 1 every stream runs
    its own blocks and attends only to itself, and text (and references) get the t = 0
    modulation at every step.  So the text rows after stage 1 are the same whatever the
    image tokens (that is, at every sigma): bit for bit in the oracle, which is what lets
    the sampling loop compute them once per prompt."""
    import oracle as O
    from flow_matching_image_flux3_b300 import synth
    from tests.common import oracle_weights

    dims = synth.TINY
    g = torch.Generator("cpu").manual_seed(17)
    streams = [synth.Stream("image", 64, (8, 8)), synth.text_stream(80)]
    seg = [0, 64, 144]
    pos = synth.positions(streams).numpy()
    s1 = [[oracle_weights(synth.draw_weights(g, dims, True)) for _ in range(2)] for _ in range(2)]
    m1 = [synth.as_f64(synth.draw_mod(g, 2, dims.width)) for _ in range(2)]
    text = synth.as_f64(torch.randn(80, dims.width, generator=g).to(torch.bfloat16))
    outs = []
    for sigma in (0.9, 0.3):   # two image inputs, as at two noise levels
        img = synth.as_f64(torch.randn(64, dims.width, generator=g).to(torch.bfloat16)) * sigma
        x = np.concatenate([img, text])
        _, h = O.dit_forward(x, seg, pos, s1, m1, [], [], np.zeros((2, dims.width)), np.zeros((128, dims.width)),
                             np.zeros(128), heads=dims.heads, theta=1e4, rounding="bf16")
        outs.append(h)
    assert np.array_equal(outs[0][64:], outs[1][64:])
    assert not np.allclose(outs[0][:64], outs[1][:64])
    assert not np.allclose(outs[0][64:], text)    # stage 1 did change the text rows
