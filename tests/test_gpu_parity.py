"""Parity of the CUDA path (through the C-ABI) with the CPU oracle, step by step and for
whole blocks, on seeded inputs: small sizes element by element (several tiles plus a
ragged tail), full sizes on sampled rows."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from oracle import fp8 as Q8
from oracle import nvfp4 as Q4
from flow_matching_image_flux3_b300 import synth
from tests.common import (REL_L2, MAX_ABS, REL_L2_F32, assert_close, rel_l2, max_abs, f64, DevWeights,
                          oracle_weights, oracle_block)

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
    yield binding
    assert binding.device_error(reset=True) == 0, "a device-side wait timed out"


def gen(seed):
    return torch.Generator("cpu").manual_seed(seed)


def randn_bf16(shape, seed, std=1.0):
    return (torch.randn(*shape, generator=gen(seed)) * std).to(torch.bfloat16)


def case_to_dev(case, bias=True):
    return ([DevWeights(w, bias=bias) for w in case.weights], case.x.cuda(), case.mod.cuda(), case.pos.cuda())


# ------------------------------------------------------------------ a1 RoPE table
def test_rope_table():
    pos = torch.cat([synth.config(0).pos,
                     torch.tensor([[10, 255, 255, 8191], [3, 0, 4095, 17], [0, 0, 0, 0]], dtype=torch.int32)])
    rope = B.rope_build(synth.TINY, pos.cuda()).cpu().numpy()
    ang = O.rope_angles(pos.numpy(), 1e4)
    # fp32 rounding of the reduced angle (<= pi * 2^-24) plus a 2-ulp sincosf: < 5e-7
    np.testing.assert_allclose(rope[..., 0], np.cos(ang), atol=5e-7, rtol=0)
    np.testing.assert_allclose(rope[..., 1], np.sin(ang), atol=5e-7, rtol=0)


# ------------------------------------------------------------------ a2+a3 LayerNorm + modulation
@pytest.mark.parametrize("n,seg", [(144, [0, 64, 144]), (1, [0, 1]), (300, [0, 77, 200, 300])])
@pytest.mark.parametrize("dims", [synth.TINY, synth.FULL], ids=["D256", "D3072"])
def test_adaln(n, seg, dims):
    g = gen(7)
    x = (torch.randn(n, dims.width, generator=g) * 2 + 0.5).to(torch.bfloat16)
    mod = synth.draw_mod(g, len(seg) - 1, dims.width)
    a = B.adaln_fwd(dims, x.cuda(), seg, mod.cuda())
    ref = O.ada_ln(f64(x), seg, f64(mod), dims.ln_eps)
    assert_close("adaln", f64(a), ref, rl2=4e-3, ma=MAX_ABS)
    # against the oracle's own bf16 rounding: equal up to one bf16 step
    diff = np.abs(f64(a) - O.round_bf16(ref))
    assert np.all(diff <= np.abs(ref) * 2.0 ** -7 + 1e-6)


# ------------------------------------------------------------------ a4..a7 input projection
def _in_proj_oracle(a, weights, seg_off, pos, dims, stage, fp8=False, nvfp4=False):
    D, H, F = dims.width, dims.heads, dims.ffn_hidden
    n = a.shape[0]
    ang = O.rope_angles(pos, dims.rope_theta)
    q = np.empty((n, H, 128)); k = np.empty((n, H, 128)); v = np.empty((n, H, 128)); act = np.empty((n, F))
    ranges = [(0, n, weights[0])] if stage == 2 else [(seg_off[s], seg_off[s + 1], weights[s]) for s in range(len(seg_off) - 1)]
    for lo, hi, w in ranges:
        if nvfp4:
            p = Q4.nvfp4_linear(a[lo:hi], w.w_in) + w.b_in
        else:
            p = (Q8.fp8_linear(a[lo:hi], w.w_in) if fp8 else a[lo:hi] @ w.w_in.T) + w.b_in
        q[lo:hi] = O.rope_rotate(O.rms_norm(p[:, :D].reshape(-1, H, 128), w.q_norm, dims.rms_eps), ang[lo:hi])
        k[lo:hi] = O.rope_rotate(O.rms_norm(p[:, D:2 * D].reshape(-1, H, 128), w.k_norm, dims.rms_eps), ang[lo:hi])
        v[lo:hi] = p[:, 2 * D:3 * D].reshape(-1, H, 128)
        act[lo:hi] = O.swiglu(p[:, 3 * D:3 * D + F], p[:, 3 * D + F:])
    return q, k, v, act


@pytest.mark.parametrize("streams,stage", [
    ([synth.Stream("image", 64, (8, 8)), synth.text_stream(80)], 2),
    ([synth.Stream("image", 1, (1, 1))], 2),
    ([synth.Stream("image", 130, (10, 13)), synth.text_stream(160)], 2),
    ([synth.Stream("image", 48, (6, 8)), synth.text_stream(80), synth.Stream("ref", 35, (5, 7), t=1)], 1),
], ids=["tiny", "n1", "ragged", "stage1"])
def test_in_proj(streams, stage):
    case = synth.make_case(synth.TINY, streams, seed=21, stage=stage, bias=True)
    dims, n = case.dims, case.n
    a = randn_bf16((n, dims.width), 22)
    ws, _, _, pos = case_to_dev(case)
    rope = B.rope_build(dims, pos)
    q, k, vt, y = B.in_proj_fwd(dims, ws, case.seg_off, a.cuda(), rope)
    rq, rk, rv, ract = _in_proj_oracle(f64(a), [oracle_weights(w) for w in case.weights], case.seg_off,
                                       case.pos.numpy(), dims, stage)
    assert_close("q", f64(q).transpose(1, 0, 2), rq)
    assert_close("k", f64(k).transpose(1, 0, 2), rk)
    assert_close("v", f64(vt)[:, :, :n].transpose(2, 0, 1), rv)
    assert_close("act", f64(y)[:, dims.width:], ract)
    assert torch.all(y[:, :dims.width] == 0)  # attention columns untouched


# ------------------------------------------------------------------ a8 attention
def _attn_inputs(n, H, seed):
    q = randn_bf16((H, n, 128), seed)
    k = randn_bf16((H, n, 128), seed + 1)
    v = randn_bf16((H, n, 128), seed + 2)
    ldv = B.ld_vt(n)
    vt = torch.zeros(H, 128, ldv, dtype=torch.bfloat16)
    vt[:, :, :n] = v.transpose(1, 2)
    return q, k, v, vt


@pytest.mark.parametrize("n,seg", [
    (1, None), (79, None), (80, None), (81, None), (127, None), (128, None), (129, None), (144, None),
    (1000, None), (333, [0, 77, 200, 333]), (300, [0, 1, 129, 300]), (256, [0, 128, 256]), (90, [0, 0, 90]),
])
def test_attention(n, seg):
    H = 2
    q, k, v, vt = _attn_inputs(n, H, seed=n)
    groups = None if seg is None else [(seg[i], seg[i + 1]) for i in range(len(seg) - 1)]
    ref = O.attention(f64(q).transpose(1, 0, 2), f64(k).transpose(1, 0, 2), f64(v).transpose(1, 0, 2), groups)
    out = B.attn_fwd(synth.TINY, q.cuda(), k.cuda(), vt.cuda(), seg)
    assert_close("attn", f64(out), ref)
    out32 = B.attn_fwd(synth.TINY, q.cuda(), k.cuda(), vt.cuda(), seg, fp32_debug=True)
    e = rel_l2(f64(out32), ref)
    assert e <= REL_L2_F32, e


def test_attention_peaked_scores_and_out_stride():
    # large scores stress the running-max rescaling; output into a wider buffer
    H, n = 2, 700
    q, k, v, vt = _attn_inputs(n, H, seed=5)
    q = (q.float() * 6).to(torch.bfloat16)
    out = torch.full((n, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    B.attn_fwd(synth.TINY, q.cuda(), k.cuda(), vt.cuda(), None, out=out)
    ref = O.attention(f64(q).transpose(1, 0, 2), f64(k).transpose(1, 0, 2), f64(v).transpose(1, 0, 2))
    assert_close("attn", f64(out[:, :256]), ref)
    assert torch.all(out[:, 256:] == 7.0)


@pytest.mark.parametrize("stage", [2, 1])
def test_attention_ten_references_sampled(stage):
    # multi-reference editing: a 1024^2 image, ten 1024^2 references (one stream) and 160
    # text tokens = 45,216 tokens; the whole sequence runs on the device, sampled query rows
    # (tile and stream boundaries, the last row, random rows) are checked against all keys
    H, N = 24, 4096 + 40960 + 160
    seg = [0, 4096, 45056, N]
    g = torch.Generator(device="cuda").manual_seed(100 + stage)
    q, k, v = (torch.randn(H, N, 128, generator=g, device="cuda").to(torch.bfloat16) for _ in range(3))
    vt = torch.zeros(H, 128, B.ld_vt(N), dtype=torch.bfloat16, device="cuda")
    vt[:, :, :N] = v.transpose(1, 2)
    out = B.attn_fwd(synth.FULL, q, k, vt, None if stage == 2 else seg)
    rows = sorted({0, 1, 127, 128, 255, 256, 4095, 4096, 4097, 20000, 44999, 45055, 45056, 45100, N - 1} |
                  set(np.random.default_rng(stage).choice(N, 8, replace=False).tolist()))
    groups = None if stage == 2 else [(seg[i], seg[i + 1]) for i in range(3)]
    cpu = [t.float().cpu().transpose(0, 1).numpy() for t in (q, k, v)]   # [N, H, 128], exact bf16 values
    ref = O.attention_rows(cpu[0], cpu[1], cpu[2], rows, groups)
    assert_close("attn (10 references)", f64(out[rows]), ref)


# ------------------------------------------------------------------ a9 output projection
@pytest.mark.parametrize("n,seg,stage", [(144, [0, 64, 144], 2), (1, [0, 1], 2), (290, [0, 130, 290], 2),
                                         (200, [0, 50, 120, 200], 1)])
def test_out_proj(n, seg, stage):
    dims = synth.TINY
    g = gen(31)
    nw = 1 if stage == 2 else len(seg) - 1
    wts = [synth.draw_weights(g, dims, bias=True) for _ in range(nw)]
    mod = synth.draw_mod(g, len(seg) - 1, dims.width)
    y = randn_bf16((n, dims.width + dims.ffn_hidden), 32)
    x = randn_bf16((n, dims.width), 33)
    xo = B.out_proj_fwd(dims, [DevWeights(w) for w in wts], seg, mod.cuda(), y.cuda(), x.cuda())
    ow = [oracle_weights(w) for w in wts]
    ref = np.empty((n, dims.width))
    sid = O.segment_ids(seg)
    for r in range(n):
        w = ow[0] if stage == 2 else ow[sid[r]]
        ref[r] = f64(x)[r] + f64(mod)[sid[r], 2] * (f64(y)[r] @ w.w_out.T + w.b_out)
    assert_close("x_out", f64(xo), ref)
    # in place (x_out aliases x)
    xd = x.cuda()
    B.out_proj_fwd(dims, [DevWeights(w) for w in wts], seg, mod.cuda(), y.cuda(), xd, x_out=xd)
    assert torch.equal(xd.cpu(), xo.cpu())


# ------------------------------------------------------------------ whole blocks, small sizes
def _run_block(case, bias=True, x=None, mod=None):
    ws, xd, md, pos = case_to_dev(case, bias)
    if x is not None:
        xd = x.cuda()
    if mod is not None:
        md = mod.cuda()
    rope = B.rope_build(case.dims, pos)
    if case.stage == 2:
        return B.block_fwd(case.dims, ws[0], case.seg_off, md, xd, rope)
    return B.stream_block_fwd(case.dims, ws, case.seg_off, md, xd, rope)


BLOCK_CASES = {
    "cfg0": lambda: synth.config(0, bias=True),
    "cfg0_nobias": lambda: synth.config(0, bias=False),
    "n1": lambda: synth.make_case(synth.TINY, [synth.Stream("image", 1, (1, 1))], 40, 2, True),
    "n79": lambda: synth.make_case(synth.TINY, [synth.text_stream(79)], 41, 2, True),
    "n81": lambda: synth.make_case(synth.TINY, [synth.Stream("image", 1, (1, 1)), synth.text_stream(80)], 42, 2, True),
    "n129": lambda: synth.make_case(synth.TINY, [synth.Stream("image", 49, (7, 7)), synth.text_stream(80)], 43, 2, True),
    "joint_ref": lambda: synth.make_case(synth.TINY, [synth.Stream("image", 64, (8, 8)), synth.Stream("ref", 64, (8, 8), t=1),
                                                      synth.text_stream(160)], 44, 2, True),
    "stage1": lambda: synth.make_case(synth.TINY, [synth.Stream("image", 64, (8, 8)), synth.Stream("ref", 64, (8, 8), t=1),
                                                   synth.text_stream(240)], 45, 1, True),
    "stage1_ragged": lambda: synth.make_case(synth.TINY, [synth.Stream("image", 63, (7, 9)), synth.text_stream(80),
                                                          synth.Stream("ref", 15, (3, 5), t=1)], 46, 1, True),
}


@pytest.mark.parametrize("name", list(BLOCK_CASES))
def test_block(name):
    case = BLOCK_CASES[name]()
    got = f64(_run_block(case, bias=True))
    ref = oracle_block(case).x_out
    assert_close(f"{name} x_out", got, ref)
    # the residual update alone (x' - x) is what the block computes; check it too
    x = synth.as_f64(case.x)
    assert rel_l2(got - x, ref - x) <= 2e-2, rel_l2(got - x, ref - x)


def test_block_gate_zero_is_identity_bitwise():
    case = synth.config(0, bias=True)
    mod = case.mod.clone()
    mod[:, 2] = 0
    got = _run_block(case, mod=mod).cpu()
    assert torch.equal(got, case.x)


def test_stage1_streams_isolated_bitwise():
    case = BLOCK_CASES["stage1_ragged"]()
    base = _run_block(case).cpu()
    x2 = case.x.clone()
    x2[63:] = randn_bf16((x2.shape[0] - 63, x2.shape[1]), 99)
    pert = _run_block(case, x=x2).cpu()
    assert torch.equal(pert[:63], base[:63])
    assert not torch.equal(pert[63:], base[63:])


def test_block_in_place_matches_out_of_place():
    case = synth.config(0, bias=True)
    ws, xd, md, pos = case_to_dev(case)
    rope = B.rope_build(case.dims, pos)
    ref = B.block_fwd(case.dims, ws[0], case.seg_off, md, xd, rope)
    B.block_fwd(case.dims, ws[0], case.seg_off, md, xd, rope, x_out=xd)
    assert torch.equal(ref, xd)


def test_block_is_deterministic():
    case = synth.config(0, bias=True)
    a = _run_block(case)
    b = _run_block(case)
    assert torch.equal(a, b)


# ------------------------------------------------------------------ full sizes, sampled rows
def _ws_views(dims, n, ws):
    D, H, F = dims.width, dims.heads, dims.ffn_hidden
    up = lambda b: (b + 255) // 256 * 256
    ldv = (n + 7) // 8 * 8
    sizes = [n * D * 2, H * n * 128 * 2, H * n * 128 * 2, H * 128 * ldv * 2, n * (D + F) * 2]
    offs = np.cumsum([0] + [up(s) for s in sizes])
    view = lambda i, shape: ws[offs[i]:offs[i] + sizes[i]].view(torch.bfloat16).view(*shape)
    return {"a": view(0, (n, D)), "q": view(1, (H, n, 128)), "k": view(2, (H, n, 128)),
            "vt": view(3, (H, 128, ldv)), "y": view(4, (n, D + F))}


def _sample_rows(case, extra=()):
    n = case.n
    rows = set(extra) | {0, 1, 127, 128, n - 1, n - 2}
    for a in case.seg_off[1:-1]:
        rows |= {a - 1, a}
    rng = np.random.default_rng(case.n)
    rows |= set(rng.choice(n, 20, replace=False).tolist())
    return sorted(r for r in rows if 0 <= r < n)


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_full_size_block_sampled(cfg):
    case = synth.config(cfg)
    dims, n = case.dims, case.n
    ws_dev, xd, md, pos = case_to_dev(case, bias=False)
    rope = B.rope_build(dims, pos)
    ws = B.workspace(B.block_workspace_size(dims, n))
    if case.stage == 2:
        xo = B.block_fwd(dims, ws_dev[0], case.seg_off, md, xd, rope, ws=ws)
    else:
        xo = B.stream_block_fwd(dims, ws_dev, case.seg_off, md, xd, rope, ws=ws)
    torch.cuda.synchronize()
    views = _ws_views(dims, n, ws)
    rows = _sample_rows(case)
    ang = O.rope_angles(case.pos.numpy(), dims.rope_theta)
    ref = O.block_forward_rows(synth.as_f64(case.x), [oracle_weights(w) for w in case.weights], case.seg_off,
                               synth.as_f64(case.mod), ang, dims.heads, rows, stage=case.stage, rounding="bf16")
    assert_close("k (all rows)", f64(views["k"]).transpose(1, 0, 2), ref["k"])
    assert_close("v (all rows)", f64(views["vt"])[:, :, :n].transpose(2, 0, 1), ref["v"])
    assert_close("q (rows)", f64(views["q"][:, rows]).transpose(1, 0, 2), ref["q"])
    assert_close("attn (rows)", f64(views["y"][rows, :dims.width]), ref["attn"])
    assert_close("act (rows)", f64(views["y"][rows, dims.width:]), ref["act"])
    assert_close("x_out (rows)", f64(xo[rows]), ref["x_out"])


# ------------------------------------------------------------------ final layer and the stack
def test_final_layer():
    dims = synth.TINY
    g = gen(51)
    x = randn_bf16((200, dims.width), 52, std=3.0)
    wf = (torch.randn(256, dims.width, generator=g) / 16).to(torch.bfloat16)
    bf = torch.randn(256, generator=g)
    fm = torch.randn(2, dims.width, generator=g) * 0.1
    out = B.final_fwd(dims, wf.cuda(), bf.cuda(), fm.cuda(), x.cuda())
    ref = O.final_layer(f64(x), f64(fm)[0], f64(fm)[1], f64(wf), f64(bf), rounding="bf16")
    assert_close("velocity", f64(out), ref)


def _tiny_dit(n_stage1=2, n_joint=3, n_img=64, n_ref=0, n_txt=80, seed=61):
    dims = synth.TINY
    g = gen(seed)
    streams = [synth.Stream("image", n_img, (8, n_img // 8))]
    if n_ref:
        streams.append(synth.Stream("ref", n_ref, (8, n_ref // 8), t=1))
    streams.append(synth.text_stream(n_txt))
    ns = len(streams)
    x = torch.randn(sum(s.n for s in streams), dims.width, generator=g).to(torch.bfloat16)
    s1 = [[synth.draw_weights(g, dims, True) for _ in range(ns)] for _ in range(n_stage1)]
    jw = [synth.draw_weights(g, dims, True) for _ in range(n_joint)]
    m1 = torch.stack([synth.draw_mod(g, ns, dims.width) for _ in range(n_stage1)]) if n_stage1 else None
    mj = torch.stack([synth.draw_mod(g, ns, dims.width) for _ in range(n_joint)]) if n_joint else None
    fm = torch.randn(2, dims.width, generator=g) * 0.1
    wf = (torch.randn(128, dims.width, generator=g) / 16).to(torch.bfloat16)
    bf = torch.randn(128, generator=g) * 0.1
    return dims, streams, x, s1, jw, m1, mj, fm, wf, bf


@pytest.mark.parametrize("n_ref", [0, 64])
def test_dit_stack_tiny(n_ref):
    dims, streams, x, s1, jw, m1, mj, fm, wf, bf = _tiny_dit(n_ref=n_ref)
    pos = synth.positions(streams)
    seg = [0]
    for s in streams:
        seg.append(seg[-1] + s.n)
    keep = dict(s1=[[DevWeights(w) for w in blk] for blk in s1], j=[DevWeights(w) for w in jw])
    args = B.DitArgs(keep["s1"], keep["j"], wf.cuda(), bf.cuda(), m1.cuda(), mj.cuda(), fm.cuda(), len(streams))
    tok = x.cuda()
    vel = B.dit_fwd(dims, args, tok, streams[0].n, n_ref, streams[-1].n, pos.cuda())
    rv, rx = O.dit_forward(synth.as_f64(x), seg, pos.numpy(), [[oracle_weights(w) for w in blk] for blk in s1],
                           [synth.as_f64(m) for m in m1], [oracle_weights(w) for w in jw], [synth.as_f64(m) for m in mj],
                           synth.as_f64(fm), synth.as_f64(wf), synth.as_f64(bf), heads=dims.heads, theta=1e4,
                           rounding="bf16")
    assert_close("velocity", f64(vel), rv, rl2=REL_L2, ma=0.1)
    assert rel_l2(f64(tok), rx) <= REL_L2


def test_euler_step():
    g = gen(71)
    lat = torch.randn(4096, 128, generator=g)
    v = torch.randn(4096, 128, generator=g)
    d = lat.cuda()
    B.euler_step(d, v.cuda(), 0.8, 0.75)
    np.testing.assert_allclose(f64(d), O.euler_step(f64(lat), f64(v), 0.8, 0.75), rtol=1e-6, atol=1e-6)


# ------------------------------------------------------------------ the bounded-wait failure path
def test_bounded_wait_times_out_and_the_context_stays_usable():
    # a device wait on a barrier nothing completes: it must give up after its limit, set
    # the error flag the host reads, and leave the context working
    assert B.device_error(reset=True) == 0
    B.selftest_timeout(20000)                      # 20 ms
    assert B.device_error(reset=True) == 1         # bit 0: a bounded wait ran out
    assert B.device_error(reset=True) == 0         # reset
    case = synth.config(0, bias=True)
    out = _run_block(case)
    assert_close("x_out after a timed-out wait", f64(out), oracle_block(case).x_out)
