"""Pins for the CPU oracle.  None of these re-uses the oracle's own code for the expected
value: each checks a closed form, an invariant, a library routine for a special case, a
worked example derived by hand, or a brute-force loop on a tiny input."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from flow_matching_image_flux3_b300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


# ------------------------------------------------------------------ bf16 rounding
def test_round_bf16_matches_torch_cast():
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.005859375, 65504.0, 1e-40]])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_bf16(x), ref)


# ------------------------------------------------------------------ LayerNorm + modulation
def test_layer_norm_worked_example():
    # mean 2.5 and biased variance 1.25 worked out by hand
    n = O.layer_norm(np.array([[1.0, 2.0, 3.0, 4.0]]), 1e-6)[0]
    s = math.sqrt(1.25 + 1e-6)
    np.testing.assert_allclose(n, [-1.5 / s, -0.5 / s, 0.5 / s, 1.5 / s], rtol=1e-15)


def test_layer_norm_matches_torch_and_invariants():
    x = rng.standard_normal((7, 256)) * 3 + 1
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (256,), eps=1e-6).numpy()
    np.testing.assert_allclose(O.layer_norm(x, 1e-6), ref, rtol=1e-12, atol=1e-12)
    n = O.layer_norm(x, 0.0)
    np.testing.assert_allclose(n.mean(1), 0, atol=1e-13)
    np.testing.assert_allclose((n ** 2).mean(1), 1, rtol=1e-12)
    np.testing.assert_allclose(O.layer_norm(2.5 * x - 7.0, 0.0), n, atol=1e-12)


def test_ada_ln_selects_stream_vectors():
    x = rng.standard_normal((10, 256))
    mod = np.zeros((2, 3, 256))
    seg = [0, 4, 10]
    # scale = shift = 0: plain LayerNorm
    np.testing.assert_allclose(O.ada_ln(x, seg, mod, 1e-6), O.layer_norm(x, 1e-6), rtol=0, atol=0)
    # stream 0: scale = -1 kills the normalized part, leaving the shift; stream 1: doubled
    mod[0, 1] = -1.0
    mod[0, 0] = np.arange(256)
    mod[1, 1] = 1.0
    a = O.ada_ln(x, seg, mod, 1e-6)
    np.testing.assert_allclose(a[:4], np.broadcast_to(np.arange(256.0), (4, 256)), atol=1e-12)
    np.testing.assert_allclose(a[4:], 2 * O.layer_norm(x[4:], 1e-6), rtol=1e-14)


# ------------------------------------------------------------------ RoPE
def test_rope_frequencies_golden():
    rows = [l.split() for l in open(os.path.join(GOLD, "rope_frequencies.txt")) if l.strip() and l[0] != "#"]
    for axis in range(4):
        pos = np.zeros((1, 4), dtype=np.int64)
        pos[0, axis] = 3
        ang = O.rope_angles(pos, 10000.0)[0]
        for j, f in rows:
            assert ang[16 * axis + int(j)] == pytest.approx(3 * float(f), rel=1e-14)
        others = np.delete(ang, np.arange(16 * axis, 16 * axis + 16))
        assert np.all(others == 0)


def test_rope_rotation_convention_quarter_turn():
    # angle pi/2 on pair (2j, 2j+1) maps (1, 0) -> (0, 1) and (0, 1) -> (-1, 0)
    x = np.zeros((1, 1, 128))
    x[0, 0, 34] = 1.0      # axis h, pair j=1: dims 34, 35
    x[0, 0, 37] = 1.0      # axis h, pair j=2: dims 36, 37
    ang = np.zeros((1, 64))
    ang[0, 17] = ang[0, 18] = math.pi / 2
    y = O.rope_rotate(x, ang)[0, 0]
    exp = np.zeros(128)
    exp[35] = 1.0
    exp[36] = -1.0
    np.testing.assert_allclose(y, exp, atol=1e-15)


def test_rope_matches_complex_multiplication():
    x = rng.standard_normal((5, 3, 128))
    pos = rng.integers(0, 100, (5, 4))
    ang = O.rope_angles(pos, 10000.0)
    z = (x[..., 0::2] + 1j * x[..., 1::2]) * np.exp(1j * ang)[:, None, :]
    y = O.rope_rotate(x, ang)
    np.testing.assert_allclose(y[..., 0::2], z.real, atol=1e-12)
    np.testing.assert_allclose(y[..., 1::2], z.imag, atol=1e-12)


def test_rope_norm_preservation_and_identity():
    x = rng.standard_normal((9, 2, 128))
    pos = rng.integers(0, 4096, (9, 4))
    y = O.rope_rotate(x, O.rope_angles(pos, 10000.0))
    np.testing.assert_allclose(np.linalg.norm(y[..., 0::2] + 1j * y[..., 1::2], axis=-1, ord=None),
                               np.linalg.norm(x[..., 0::2] + 1j * x[..., 1::2], axis=-1), rtol=1e-12)
    pair_norm_x = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    pair_norm_y = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    np.testing.assert_allclose(pair_norm_y, pair_norm_x, rtol=1e-10, atol=1e-12)
    z = O.rope_rotate(x, O.rope_angles(np.zeros((9, 4)), 10000.0))
    np.testing.assert_array_equal(z, x)


@pytest.mark.parametrize("axis", [0, 1, 2, 3])
def test_rope_relative_position_invariance(axis):
    q = rng.standard_normal((6, 2, 128))
    k = rng.standard_normal((6, 2, 128))
    pos = rng.integers(0, 64, (6, 4))
    pos2 = pos.copy()
    pos2[:, axis] += 37
    s1 = np.einsum("nhd,mhd->hnm", O.rope_rotate(q, O.rope_angles(pos, 1e4)), O.rope_rotate(k, O.rope_angles(pos, 1e4)))
    s2 = np.einsum("nhd,mhd->hnm", O.rope_rotate(q, O.rope_angles(pos2, 1e4)), O.rope_rotate(k, O.rope_angles(pos2, 1e4)))
    np.testing.assert_allclose(s2, s1, rtol=1e-10, atol=1e-10)
    # and a shift of only some tokens does change the scores (the pin is not vacuous)
    pos3 = pos.copy()
    pos3[:3, axis] += 5
    s3 = np.einsum("nhd,mhd->hnm", O.rope_rotate(q, O.rope_angles(pos3, 1e4)), O.rope_rotate(k, O.rope_angles(pos3, 1e4)))
    assert np.abs(s3 - s1).max() > 1e-3


# ------------------------------------------------------------------ RMSNorm, SwiGLU
def test_rms_norm_matches_torch_and_invariants():
    x = rng.standard_normal((4, 3, 128)) * 5
    g = 1 + 0.1 * rng.standard_normal(128)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (128,), torch.from_numpy(g), eps=1e-6).numpy()
    np.testing.assert_allclose(O.rms_norm(x, g, 1e-6), ref, rtol=1e-12)
    y = O.rms_norm(x, np.ones(128), 0.0)
    np.testing.assert_allclose(np.sqrt((y ** 2).mean(-1)), 1, rtol=1e-12)
    np.testing.assert_allclose(O.rms_norm(7.0 * x, g, 0.0), O.rms_norm(x, g, 0.0), rtol=1e-12)


def test_swiglu_matches_torch_silu():
    g = rng.standard_normal(1000) * 8
    u = rng.standard_normal(1000)
    ref = (torch.nn.functional.silu(torch.from_numpy(g)) * torch.from_numpy(u)).numpy()
    np.testing.assert_allclose(O.swiglu(g, u), ref, rtol=1e-13, atol=1e-300)


# ------------------------------------------------------------------ attention
def _attention_loops(q, k, v, groups):
    n, h, d = q.shape
    out = np.zeros((n, h * d))
    for a, b in groups:
        for hh in range(h):
            for i in range(a, b):
                s = [sum(q[i, hh, t] * k[j, hh, t] for t in range(d)) / math.sqrt(d) for j in range(a, b)]
                m = max(s)
                e = [math.exp(z - m) for z in s]
                tot = sum(e)
                for t in range(d):
                    out[i, hh * d + t] = sum(e[j - a] * v[j, hh, t] for j in range(a, b)) / tot
    return out


def test_attention_brute_force_tiny():
    q = rng.standard_normal((7, 2, 128)); k = rng.standard_normal((7, 2, 128)); v = rng.standard_normal((7, 2, 128))
    np.testing.assert_allclose(O.attention(q, k, v), _attention_loops(q, k, v, [(0, 7)]), rtol=1e-12, atol=1e-13)
    g = [(0, 3), (3, 7)]
    np.testing.assert_allclose(O.attention(q, k, v, g), _attention_loops(q, k, v, g), rtol=1e-12, atol=1e-13)


def test_attention_matches_torch_sdpa():
    q = rng.standard_normal((50, 3, 128)); k = rng.standard_normal((50, 3, 128)); v = rng.standard_normal((50, 3, 128))
    t = lambda a: torch.from_numpy(a).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v)).permute(1, 0, 2).reshape(50, -1).numpy()
    np.testing.assert_allclose(O.attention(q, k, v), ref, rtol=1e-10, atol=1e-12)


def test_attention_special_cases():
    v = rng.standard_normal((1, 2, 128))
    np.testing.assert_array_equal(O.attention(rng.standard_normal((1, 2, 128)), rng.standard_normal((1, 2, 128)), v),
                                  v.reshape(1, -1))
    q = rng.standard_normal((5, 2, 128))
    k = np.broadcast_to(rng.standard_normal((1, 2, 128)), (5, 2, 128))
    v = rng.standard_normal((5, 2, 128))
    np.testing.assert_allclose(O.attention(q, k, v), np.broadcast_to(v.mean(0).reshape(1, -1), (5, 256)), atol=1e-14)


def test_attention_groups_are_independent_runs():
    q = rng.standard_normal((12, 2, 128)); k = rng.standard_normal((12, 2, 128)); v = rng.standard_normal((12, 2, 128))
    o = O.attention(q, k, v, [(0, 5), (5, 12)])
    np.testing.assert_allclose(o[:5], O.attention(q[:5], k[:5], v[:5]), rtol=0, atol=0)
    np.testing.assert_allclose(o[5:], O.attention(q[5:], k[5:], v[5:]), rtol=0, atol=0)


# ------------------------------------------------------------------ the block
def _tiny_case(stage=2, streams=None, bias=True, seed=5):
    streams = streams or [synth.Stream("image", 16, (4, 4)), synth.text_stream(8)]
    return synth.make_case(synth.TINY, streams, seed=seed, stage=stage, bias=bias)


def _run(case, rounding=None, x=None, mod=None):
    d = case.dims
    w = [O.Weights(*(synth.as_f64(t) for t in (wi.w_in, wi.b_in, wi.q_norm, wi.k_norm, wi.w_out, wi.b_out)))
         for wi in case.weights]
    ang = O.rope_angles(case.pos.numpy(), d.rope_theta)
    return O.block_forward(synth.as_f64(case.x) if x is None else x, w, case.seg_off,
                           synth.as_f64(case.mod) if mod is None else mod, ang, d.heads,
                           stage=case.stage, rounding=rounding)


def _block_loops(x, w, seg_off, mod, pos, H, stage, theta=1e4, eps=1e-6):
    """The block written as explicit per-token, per-head loops with the math module."""
    n, D = x.shape
    d = 128
    F = (w[0].w_in.shape[0] - 3 * D) // 2
    seg = [s for s in range(len(seg_off) - 1) for _ in range(seg_off[s], seg_off[s + 1])]
    a = []
    for i in range(n):
        row = list(x[i]); mu = sum(row) / D
        var = sum((t - mu) ** 2 for t in row) / D
        a.append([(row[c] - mu) / math.sqrt(var + eps) * (1 + mod[seg[i], 1, c]) + mod[seg[i], 0, c] for c in range(D)])
    a = np.array(a)
    wsel = [w[0] if stage == 2 else w[seg[i]] for i in range(n)]
    p = np.array([[float(np.dot(wsel[i].w_in[o], a[i])) + wsel[i].b_in[o] for o in range(w[0].w_in.shape[0])] for i in range(n)])
    q = np.zeros((n, H, d)); k = np.zeros((n, H, d)); v = np.zeros((n, H, d))
    for i in range(n):
        for h in range(H):
            for tgt, off, g in ((q, 0, wsel[i].q_norm), (k, D, wsel[i].k_norm)):
                vec = p[i, off + h * d: off + (h + 1) * d]
                r = math.sqrt(sum(t * t for t in vec) / d + eps)
                vec = [vec[c] / r * g[c] for c in range(d)]
                for axis in range(4):
                    for j in range(16):
                        th = pos[i, axis] * theta ** (-j / 16)
                        c0 = 32 * axis + 2 * j
                        tgt[i, h, c0] = vec[c0] * math.cos(th) - vec[c0 + 1] * math.sin(th)
                        tgt[i, h, c0 + 1] = vec[c0] * math.sin(th) + vec[c0 + 1] * math.cos(th)
            v[i, h] = p[i, 2 * D + h * d: 2 * D + (h + 1) * d]
    groups = [(0, n)] if stage == 2 else [(seg_off[s], seg_off[s + 1]) for s in range(len(seg_off) - 1)]
    attn = _attention_loops(q, k, v, groups)
    act = np.array([[p[i, 3 * D + c] / (1 + math.exp(-p[i, 3 * D + c])) * p[i, 3 * D + F + c] for c in range(F)] for i in range(n)])
    ycat = np.concatenate([attn, act], 1)
    out = np.zeros_like(x)
    for i in range(n):
        for c in range(D):
            yv = float(np.dot(wsel[i].w_out[c], ycat[i])) + wsel[i].b_out[c]
            out[i, c] = x[i, c] + mod[seg[i], 2, c] * yv
    return out


@pytest.mark.parametrize("stage", [2, 1])
def test_block_matches_loop_version(stage):
    dims = synth.Dims(width=256, heads=2, ffn_hidden=64)
    streams = [synth.Stream("image", 4, (2, 2), t=3), synth.text_stream(3)]
    case = synth.make_case(dims, streams, seed=11, stage=stage, bias=True)
    got = _run(case).x_out
    w = [O.Weights(*(synth.as_f64(t) for t in (wi.w_in, wi.b_in, wi.q_norm, wi.k_norm, wi.w_out, wi.b_out)))
         for wi in case.weights]
    ref = _block_loops(synth.as_f64(case.x), w, case.seg_off, synth.as_f64(case.mod), case.pos.numpy(), 2, stage)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-11)


def test_block_gate_zero_is_identity():
    case = _tiny_case()
    mod = synth.as_f64(case.mod)
    mod[:, 2] = 0.0
    out = _run(case, mod=mod).x_out
    np.testing.assert_array_equal(out, synth.as_f64(case.x))


def test_stage1_streams_do_not_mix():
    case = _tiny_case(stage=1)
    x = synth.as_f64(case.x)
    base = _run(case, x=x).x_out
    x2 = x.copy()
    x2[16:] += rng.standard_normal(x2[16:].shape)
    pert = _run(case, x=x2).x_out
    np.testing.assert_array_equal(pert[:16], base[:16])
    assert np.abs(pert[16:] - base[16:]).max() > 1e-3


def test_stage2_streams_do_mix():
    case = _tiny_case(stage=2)
    x = synth.as_f64(case.x)
    x2 = x.copy()
    x2[16:] += rng.standard_normal(x2[16:].shape)
    assert np.abs(_run(case, x=x2).x_out[:16] - _run(case, x=x).x_out[:16]).max() > 1e-6


def test_stage2_permutation_equivariance():
    case = _tiny_case(stage=2)
    n = case.n
    perm = rng.permutation(n)
    x = synth.as_f64(case.x)
    w = [O.Weights(*(synth.as_f64(t) for t in (wi.w_in, wi.b_in, wi.q_norm, wi.k_norm, wi.w_out, wi.b_out)))
         for wi in case.weights]
    # the stream of each row must travel with it: give every row its own modulation segment
    mod_rows = synth.as_f64(case.mod)[O.segment_ids(case.seg_off)]
    seg_rows = list(range(n + 1))
    ang = O.rope_angles(case.pos.numpy(), 1e4)
    ref = O.block_forward(x, w, seg_rows, mod_rows, ang, 2).x_out
    got = O.block_forward(x[perm], w, seg_rows, mod_rows[perm], ang[perm], 2).x_out
    np.testing.assert_allclose(got, ref[perm], rtol=1e-12, atol=1e-12)


def test_stage1_single_stream_equals_joint_block():
    streams = [synth.Stream("image", 24, (4, 6))]
    c1 = synth.make_case(synth.TINY, streams, seed=3, stage=1, bias=True)
    c2 = synth.make_case(synth.TINY, streams, seed=3, stage=2, bias=True)
    np.testing.assert_array_equal(_run(c1).x_out, _run(c2).x_out)


def test_block_relative_position_invariance():
    case = _tiny_case(stage=2)
    base = _run(case).x_out
    case.pos[:, 1] += 11          # shift h for every token
    np.testing.assert_allclose(_run(case).x_out, base, rtol=1e-10, atol=1e-10)


def test_block_bf16_rounding_model_is_close():
    case = _tiny_case(stage=2)
    a = _run(case).x_out
    b = _run(case, rounding="bf16").x_out
    rel = np.linalg.norm(a - b) / np.linalg.norm(a)
    assert 1e-5 < rel < 1e-2


# ------------------------------------------------------------------ stack, final layer, Euler
def test_dit_with_zero_gates_reduces_to_final_layer():
    dims = synth.TINY
    g = torch.Generator().manual_seed(9)
    streams = [synth.Stream("image", 8, (2, 4)), synth.text_stream(5)]
    seg = [0, 8, 13]
    x = synth.as_f64(torch.randn(13, 256, generator=g).to(torch.bfloat16))
    pos = synth.positions(streams).numpy()
    mk = lambda: O.Weights(*(synth.as_f64(t) for t in (lambda w: (w.w_in, w.b_in, w.q_norm, w.k_norm, w.w_out, w.b_out))(synth.draw_weights(g, dims, True))))
    s1 = [[mk(), mk()] for _ in range(2)]
    j = [mk() for _ in range(2)]
    zmod = np.zeros((2, 3, 256))
    zmod[:, :2] = rng.standard_normal((2, 2, 256))
    fm = rng.standard_normal((2, 256)) * 0.1
    wf = rng.standard_normal((128, 256)) / 16
    bf = rng.standard_normal(128)
    vel, xo = O.dit_forward(x, seg, pos, s1, [zmod, zmod], j, [zmod, zmod], fm, wf, bf, heads=2, theta=1e4)
    np.testing.assert_array_equal(xo, x)
    n = torch.nn.functional.layer_norm(torch.from_numpy(x[:8]), (256,), eps=1e-6).numpy()
    np.testing.assert_allclose(vel, (n * (1 + fm[1]) + fm[0]) @ wf.T + bf, rtol=1e-12, atol=1e-12)


def test_euler_step_integrates_constant_velocity_exactly():
    x0 = rng.standard_normal((4, 128)); v = rng.standard_normal((4, 128))
    sig = [1.0, 0.75, 0.5, 0.125, 0.0]
    x = x0
    for s, sn in zip(sig[:-1], sig[1:]):
        x = O.euler_step(x, v, s, sn)
    np.testing.assert_allclose(x, x0 - v, atol=1e-14)


# ------------------------------------------------------------------ the input recipe
def test_synth_recipe_matches_page_facts():
    facts = json.load(open(os.path.join(GOLD, "page_facts.json")))
    img = synth.image_stream(1024, 1024)
    assert img.n == facts["tokens_1024"]["value"]
    assert 1024 // img.grid[0] == facts["px_per_token"]["value"]
    assert synth.FULL.width == facts["width"]["value"]
    assert synth.FULL.heads * synth.FULL.head_dim == synth.FULL.width
    assert synth.FULL.heads == facts["heads"]["value"]
    assert facts["rope_dims_per_axis"]["value"] * len(facts["rope_axes"]["value"]) == facts["head_dim"]["value"]
    for idx in (0,):
        c = synth.config(idx)
        assert (c.seg_off[-1] - c.seg_off[-2]) % facts["text_pad_multiple"]["value"] == 0
    c = synth.config(0)
    assert c.pos.shape == (144, 4)
    assert c.pos[:64, 3].abs().sum() == 0 and c.pos[64:, :3].abs().sum() == 0
    assert list(c.pos[64:, 3]) == list(range(80))


@pytest.mark.parametrize("stage", [2, 1])
def test_block_rows_match_full_block(stage):
    case = _tiny_case(stage=stage, streams=[synth.Stream("image", 20, (4, 5)), synth.text_stream(9),
                                            synth.Stream("ref", 6, (2, 3), t=1)])
    full = _run(case, rounding="bf16")
    w = [O.Weights(*(synth.as_f64(t) for t in (wi.w_in, wi.b_in, wi.q_norm, wi.k_norm, wi.w_out, wi.b_out)))
         for wi in case.weights]
    rows = [0, 7, 19, 20, 28, 29, 34]
    r = O.block_forward_rows(synth.as_f64(case.x), w, case.seg_off, synth.as_f64(case.mod),
                             O.rope_angles(case.pos.numpy(), 1e4), 2, rows, stage=stage, rounding="bf16")
    np.testing.assert_allclose(r["x_out"], full.x_out[rows], rtol=0, atol=1e-2)
    assert np.mean(r["x_out"] == full.x_out[rows]) > 0.97
    np.testing.assert_allclose(r["k"], full.k, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["v"], full.v, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["q"], full.q[rows], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["act"], full.act[rows], rtol=0, atol=1e-2)


def test_block_keys_values_of_some_rows_match_all_rows():
    case = _tiny_case(stage=1, streams=[synth.Stream("image", 20, (4, 5)), synth.text_stream(9)])
    w = [O.Weights(*(synth.as_f64(t) for t in (wi.w_in, wi.b_in, wi.q_norm, wi.k_norm, wi.w_out, wi.b_out)))
         for wi in case.weights]
    args = (synth.as_f64(case.x), w, case.seg_off, synth.as_f64(case.mod), O.rope_angles(case.pos.numpy(), 1e4), 2)
    k, v = O.block_keys_values(*args, stage=1)
    rows = [3, 19, 20, 28]
    k2, v2 = O.block_keys_values(*args, rows=rows, stage=1)
    np.testing.assert_allclose(k2, k[rows], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(v2, v[rows], rtol=1e-13, atol=1e-13)
    full = _run(case)
    np.testing.assert_allclose(k, full.k, rtol=1e-12, atol=1e-12)


def test_attention_rows_match_full_attention():
    # the sampled-rows form of attention against the full (pinned) one, joint and per range
    q, k, v = (rng.standard_normal((150, 3, 128)) for _ in range(3))
    rows = [0, 1, 63, 64, 100, 149]
    np.testing.assert_allclose(O.attention_rows(q, k, v, rows), O.attention(q, k, v)[rows], rtol=1e-12, atol=1e-12)
    groups = [(0, 64), (64, 140), (140, 150)]
    np.testing.assert_allclose(O.attention_rows(q, k, v, rows, groups), O.attention(q, k, v, groups)[rows],
                               rtol=1e-12, atol=1e-12)
