"""Shared helpers for the parity tests: moving seeded cases to the device, running the
oracle on the same values, and the error measures."""
import numpy as np
import torch

import oracle as O
from flow_matching_image_flux3_b300 import synth

# the bf16-path bar: relative L2 error and largest absolute error per output
REL_L2 = 1e-2
MAX_ABS = 5e-2
# the fp32 attention check path
REL_L2_F32 = 1e-5


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def max_abs(got, ref) -> float:
    return float(np.max(np.abs(np.asarray(got, dtype=np.float64) - np.asarray(ref, dtype=np.float64)))) if np.size(ref) else 0.0


def assert_close(name, got, ref, rl2=REL_L2, ma=MAX_ABS):
    e1, e2 = rel_l2(got, ref), max_abs(got, ref)
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{name}: non-finite values"
    assert e1 <= rl2 and e2 <= ma, f"{name}: rel_l2={e1:.3e} (<= {rl2}), max_abs={e2:.3e} (<= {ma})"
    return e1, e2


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


class DevWeights:
    def __init__(self, w: synth.BlockWeights, dev="cuda", bias=True):
        self.w_in = w.w_in.to(dev).contiguous()
        self.b_in = w.b_in.to(dev).contiguous() if bias else None
        self.q_norm = w.q_norm.to(dev).contiguous()
        self.k_norm = w.k_norm.to(dev).contiguous()
        self.w_out = w.w_out.to(dev).contiguous()
        self.b_out = w.b_out.to(dev).contiguous() if bias else None


def oracle_weights(w: synth.BlockWeights):
    return O.Weights(*(synth.as_f64(t) for t in (w.w_in, w.b_in, w.q_norm, w.k_norm, w.w_out, w.b_out)))


def oracle_block(case: synth.BlockCase, rounding="bf16"):
    d = case.dims
    ang = O.rope_angles(case.pos.numpy(), d.rope_theta)
    return O.block_forward(synth.as_f64(case.x), [oracle_weights(w) for w in case.weights], case.seg_off,
                           synth.as_f64(case.mod), ang, d.heads, ln_eps=d.ln_eps, rms_eps=d.rms_eps,
                           stage=case.stage, rounding=rounding)
