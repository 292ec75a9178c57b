"""Parity of the sampling loop's device pieces (through the C-ABI) with the oracle: the
token embedders, the guided Euler step and the whole loop on a tiny denoiser."""
import numpy as np
import pytest
import torch

import oracle as O
from oracle import sampling as S
from flow_matching_image_flux3_b300 import synth
from tests.common import REL_L2, assert_close, f64, DevWeights, oracle_weights

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


@pytest.mark.parametrize("rows,k", [(300, 640), (1, 128), (128, 20480)])
def test_linear_into_token_rows(rows, k):
    dims = synth.TINY if k != 20480 else synth.FULL
    D = dims.width
    g = gen(rows + k)
    x = torch.randn(rows, k, generator=g).to(torch.bfloat16)
    w = (torch.randn(D, k, generator=g) / k ** 0.5).to(torch.bfloat16)
    b = torch.randn(D, generator=g) * 0.1
    buf = torch.full((rows + 70, D), 3.0, dtype=torch.bfloat16, device="cuda")
    B.linear_fwd(dims, x.cuda(), w.cuda(), b.cuda(), out=buf[50:50 + rows])
    ref = O.round_bf16(S.embed(synth.as_f64(x), synth.as_f64(w), synth.as_f64(b)))
    assert_close("embed", f64(buf[50:50 + rows]), ref)
    assert torch.all(buf[:50] == 3.0) and torch.all(buf[50 + rows:] == 3.0)


@pytest.mark.parametrize("guided", [True, False])
def test_cfg_euler_step(guided):
    g = gen(5)
    lat = torch.randn(4096, 128, generator=g)
    vp, vn = torch.randn(4096, 128, generator=g), torch.randn(4096, 128, generator=g)
    dl = lat.cuda()
    lb = torch.empty(4096, 128, dtype=torch.bfloat16, device="cuda")
    B.cfg_euler_step(dl, vp.cuda(), vn.cuda() if guided else None, 3.5, 0.8, 0.55, latent_bf16=lb)
    v = S.cfg(vp.double().numpy(), vn.double().numpy(), 3.5) if guided else vp.double().numpy()
    ref = O.euler_step(lat.double().numpy(), v, 0.8, 0.55)
    np.testing.assert_allclose(f64(dl), ref, rtol=1e-5, atol=1e-5)
    assert torch.equal(lb.cpu(), dl.cpu().to(torch.bfloat16))   # the bf16 copy of the new latent


def _tiny_loop(n_ref, n_steps, cfg_scale, seed=91, cache=None):
    """The loop on the device and in the oracle.  cache=None: per-step modulation for every
    stream, uncached loop.  cache=True/False: the stage-1 reference and text entries are
    step 0's at every step (the clean-context reading) and the device loop runs with
    cache_context set/cleared.  Returns (device latent, oracle latent, initial latent)."""
    dims = synth.TINY
    D = dims.width
    g = gen(seed)
    n_img, n_txt, C, T = 64, 80, 128, 640
    streams = [synth.Stream("image", n_img, (8, 8))]
    if n_ref:
        streams.append(synth.Stream("ref", n_ref, (8, n_ref // 8), t=1))
    streams.append(synth.text_stream(n_txt))
    ns = len(streams)
    seg = [0]
    for s in streams:
        seg.append(seg[-1] + s.n)
    pos = synth.positions(streams)
    s1 = [[synth.draw_weights(g, dims, True) for _ in range(ns)] for _ in range(2)]
    jw = [synth.draw_weights(g, dims, True) for _ in range(2)]
    wf = (torch.randn(C, D, generator=g) / 16).to(torch.bfloat16)
    bf = torch.randn(C, generator=g) * 0.1
    w_img = (torch.randn(D, C, generator=g) / C ** 0.5).to(torch.bfloat16)
    b_img = torch.randn(D, generator=g) * 0.1
    w_txt = (torch.randn(D, T, generator=g) / T ** 0.5).to(torch.bfloat16)
    b_txt = torch.randn(D, generator=g) * 0.1
    t_pos = torch.randn(n_txt, T, generator=g).to(torch.bfloat16)
    t_neg = torch.randn(n_txt, T, generator=g).to(torch.bfloat16)
    ref = torch.randn(n_ref, C, generator=g).to(torch.bfloat16) if n_ref else None
    mods = [(torch.stack([synth.draw_mod(g, ns, D) for _ in range(2)]),
             torch.stack([synth.draw_mod(g, ns, D) for _ in range(2)]),
             torch.randn(2, D, generator=g) * 0.1) for _ in range(n_steps)]
    if cache is not None:
        for m in mods[1:]:
            m[0][:, 1:] = mods[0][0][:, 1:]
    lat0 = torch.randn(n_img, C, generator=g)

    # ---- device, through flux3_sample_fwd
    keep = dict(s1=[[DevWeights(w) for w in blk] for blk in s1], j=[DevWeights(w) for w in jw])
    dmods = [tuple(m.cuda() for m in ms) for ms in mods]
    dit = B.DitArgs(keep["s1"], keep["j"], wf.cuda(), bf.cuda(), dmods[0][0], dmods[0][1], dmods[0][2], ns)
    args = B.SampleArgs(n_img, n_ref, n_txt, w_img.cuda(), b_img.cuda(), w_txt.cuda(), b_txt.cuda(), t_pos.cuda(),
                        t_neg.cuda() if cfg_scale != 1.0 else None, pos.cuda(), dmods, n_steps, 6.93, cfg_scale,
                        ref_latent=ref.cuda() if n_ref else None, cache_context=bool(cache))
    lat = lat0.cuda()
    B.sample_fwd(dims, dit, args, lat)
    torch.cuda.synchronize()

    # ---- oracle
    a64 = synth.as_f64
    ow1 = [[oracle_weights(w) for w in blk] for blk in s1]
    owj = [oracle_weights(w) for w in jw]
    ctx = {}
    for name, feats in (("pos", t_pos), ("neg", t_neg)):
        parts = []
        if n_ref:
            parts.append(O.round_bf16(S.embed(a64(ref), a64(w_img), a64(b_img))))
        parts.append(O.round_bf16(S.embed(a64(feats), a64(w_txt), a64(b_txt))))
        ctx[name] = np.concatenate(parts, axis=0)

    def velocity(x, i, prompted):
        img = O.round_bf16(S.embed(x, a64(w_img), a64(b_img)))
        tok = np.concatenate([img, ctx["pos" if prompted else "neg"]], axis=0)
        m1, mj, fm = mods[i]
        v, _ = O.dit_forward(tok, seg, pos.numpy(), ow1, [a64(m) for m in m1], owj, [a64(m) for m in mj], a64(fm),
                             a64(wf), a64(bf), heads=dims.heads, theta=1e4, rounding="bf16")
        return v

    sig = S.sigma_schedule(n_steps, float(np.float32(6.93)))
    xs = S.sample(a64(lat0), sig, velocity, cfg_scale, round_latent=O.round_bf16)
    return f64(lat), xs[-1], a64(lat0)


# The bf16 bar on the relative L2 error; the largest single-element error gets the same
# 0.1 as the denoiser-stack test: each step runs one or two stacks whose velocities may
# differ from the oracle's by up to that much element-wise (bf16 rounding decisions taken
# differently inside the stack), guidance scales those differences by up to
# |s| + |s - 1| = 6 at s = 3.5, and the Euler sum integrates them with weights summing to 1.
LOOP_MAX_ABS = 0.1


@pytest.mark.parametrize("n_ref,n_steps,cfg_scale", [(0, 3, 3.5), (0, 2, 1.0), (64, 2, 3.5)])
def test_sampling_loop_tiny(n_ref, n_steps, cfg_scale):
    got, ref, lat0 = _tiny_loop(n_ref, n_steps, cfg_scale)
    assert_close("latent after the loop", got, ref, rl2=REL_L2, ma=LOOP_MAX_ABS)
    # the loop moved the latent by far more than the tolerance (the comparison is not vacuous)
    assert np.linalg.norm(ref - lat0) > 10 * REL_L2 * np.linalg.norm(ref)


@pytest.mark.parametrize("n_ref,n_steps,cfg_scale", [(0, 3, 3.5), (64, 2, 3.5), (64, 2, 1.0)])
def test_sampling_loop_cached_context(n_ref, n_steps, cfg_scale):
    """The loop that runs the context streams' stage 1 once per prompt against the oracle
    loop (which recomputes every stream at every step) and against the uncached device
    loop on the same inputs."""
    got, ref, lat0 = _tiny_loop(n_ref, n_steps, cfg_scale, cache=True)
    assert_close("latent after the cached loop", got, ref, rl2=REL_L2, ma=LOOP_MAX_ABS)
    assert np.linalg.norm(ref - lat0) > 10 * REL_L2 * np.linalg.norm(ref)
    plain, _, _ = _tiny_loop(n_ref, n_steps, cfg_scale, cache=False)
    assert_close("cached vs uncached loop", got, plain, rl2=REL_L2, ma=LOOP_MAX_ABS)
