"""CPU oracle for the backward pass of the joint (stage-2) transformer block -- TEST
INFRASTRUCTURE.

Only the tests and the benchmark's CPU-baseline leg may import this module; it shares no
code with the CUDA path.  Float64 NumPy.  The forward pass is the one in flux3_block.py
("Welcome FLUX.3 Image Klein in Diffusers", section "How it works"; the Miles page,
section 1, for fine-tuning the base checkpoint); this module is the chain rule of that
forward pass written out step by step, for a loss L whose gradient with respect to the
block output x' is given (dxo):

  forward                                         backward
  ln  = LN(x)                                     dx  = dxo + LN^T(dln)
  a   = ln (1 + scale_s) + shift_s                dln = da (1 + scale_s); dscale_s = sum da ln; dshift_s = sum da
  P   = a W_in^T + b_in                           da = dP W_in; dW_in = dP^T a; db_in = sum dP
  q   = rope(rms(Pq) g_q), k likewise             dPq = rms^T(rope^T(dq) ...), dg_q = sum ...
  O   = softmax(q k^T / sqrt(d)) v                dv = S^T dO; dq, dk from dS = S (dS' - rowsum(dO O))
  act = silu(G) U                                 dG = dact U silu'(G); dU = dact silu(G)
  y   = [O | act] W_out^T + b_out                 d[O | act] = dy W_out; dW_out = dy^T [O | act]
  x'  = x + gate_s y                              dy = gate_s dxo; dgate_s = sum dxo y

Readings: the same as the forward oracle's; the block is the joint one (one weight set,
attention over all tokens, modulation per stream).  The gradient of the modulation
vectors is summed over the rows of their stream.

Pins (tests/test_oracle_backward.py): every gradient against central finite differences
of the forward oracle (flux3_block.block_forward in float64) along random directions,
and the special cases gate = 0 (nothing flows into the block's weights) and a single
token (attention passes v through).
"""
from __future__ import annotations

import math
from typing import Dict, List, Sequence

import numpy as np

from .flux3_block import Weights, layer_norm, segment_ids, rope_rotate

F64 = np.float64


def _rms_forward(x, g, eps):
    r = 1.0 / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)
    return x * r * g, r


def _rms_backward(dz, x, r, g):
    """z = x r g, r = (mean(x^2) + eps)^(-1/2) over the last axis: returns (dx, dg)."""
    d = x.shape[-1]
    dzg = dz * g
    dx = r * dzg - x * r ** 3 * (dzg * x).sum(axis=-1, keepdims=True) / d
    dg = (dz * x * r).reshape(-1, d).sum(axis=0)
    return dx, dg


def _ln_backward(dln, x, eps):
    """ln = (x - mu) rstd over the last axis: returns dx."""
    mu = x.mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(((x - mu) ** 2).mean(axis=-1, keepdims=True) + eps)
    ln = (x - mu) * rstd
    return rstd * (dln - dln.mean(axis=-1, keepdims=True) - ln * (dln * ln).mean(axis=-1, keepdims=True))


def block_backward(x: np.ndarray, w: Weights, seg_off: Sequence[int], mod: np.ndarray, angles: np.ndarray,
                   heads: int, dxo: np.ndarray, head_dim: int = 128, ln_eps: float = 1e-6,
                   rms_eps: float = 1e-6) -> Dict[str, np.ndarray]:
    """Gradients of sum(x' * dxo) for the joint block x' = block(x): returns dx [N, D],
    dw_in [3D + 2F, D], db_in, dq_norm [d], dk_norm [d], dw_out [D, D + F], db_out and
    dmod [n_seg, 3, D] (shift, scale, gate)."""
    x = np.asarray(x, dtype=F64)
    dxo = np.asarray(dxo, dtype=F64)
    n, D = x.shape
    H, d = heads, head_dim
    F = (w.w_in.shape[0] - 3 * D) // 2
    seg = segment_ids(seg_off)
    shift, scale, gate = mod[seg, 0], mod[seg, 1], mod[seg, 2]

    # ---- forward, keeping what the backward needs
    ln = layer_norm(x, ln_eps)
    a = ln * (1.0 + scale) + shift
    p = a @ w.w_in.T + w.b_in
    pq = p[:, 0:D].reshape(n, H, d)
    pk = p[:, D:2 * D].reshape(n, H, d)
    v = p[:, 2 * D:3 * D].reshape(n, H, d)
    g, u = p[:, 3 * D:3 * D + F], p[:, 3 * D + F:]
    qn, rq = _rms_forward(pq, w.q_norm, rms_eps)
    kn, rk = _rms_forward(pk, w.k_norm, rms_eps)
    q = rope_rotate(qn, angles)
    k = rope_rotate(kn, angles)
    sc = 1.0 / math.sqrt(d)

    def probs(h):
        s = q[:, h] @ k[:, h].T * sc
        s = np.exp(s - s.max(axis=1, keepdims=True))
        return s / s.sum(axis=1, keepdims=True)

    o = np.empty((n, H, d))
    for h in range(H):
        o[:, h] = probs(h) @ v[:, h]
    sig = 1.0 / (1.0 + np.exp(-g))
    act = g * sig * u
    ycat = np.concatenate([o.reshape(n, D), act], axis=1)
    y = ycat @ w.w_out.T + w.b_out

    # ---- backward
    n_seg = len(seg_off) - 1
    dmod = np.zeros((n_seg, 3, D))
    dy = gate * dxo
    for s in range(n_seg):
        lo, hi = seg_off[s], seg_off[s + 1]
        dmod[s, 2] = (dxo[lo:hi] * y[lo:hi]).sum(axis=0)
    db_out = dy.sum(axis=0)
    dw_out = dy.T @ ycat
    dycat = dy @ w.w_out
    do = dycat[:, :D].reshape(n, H, d)
    dact = dycat[:, D:]
    dg = dact * u * sig * (1.0 + g * (1.0 - sig))
    du = dact * g * sig
    dq = np.empty((n, H, d)); dk = np.empty((n, H, d)); dv = np.empty((n, H, d))
    for h in range(H):
        pr = probs(h)
        dv[:, h] = pr.T @ do[:, h]
        dpr = do[:, h] @ v[:, h].T
        delta = (do[:, h] * o[:, h]).sum(axis=1, keepdims=True)
        ds = pr * (dpr - delta)
        dq[:, h] = ds @ k[:, h] * sc
        dk[:, h] = ds.T @ q[:, h] * sc
    dqn = rope_rotate(dq, -angles)
    dkn = rope_rotate(dk, -angles)
    dpq, dq_norm = _rms_backward(dqn, pq, rq, w.q_norm)
    dpk, dk_norm = _rms_backward(dkn, pk, rk, w.k_norm)
    dp = np.concatenate([dpq.reshape(n, D), dpk.reshape(n, D), dv.reshape(n, D), dg, du], axis=1)
    db_in = dp.sum(axis=0)
    dw_in = dp.T @ a
    da = dp @ w.w_in
    for s in range(n_seg):
        lo, hi = seg_off[s], seg_off[s + 1]
        dmod[s, 0] = da[lo:hi].sum(axis=0)
        dmod[s, 1] = (da[lo:hi] * ln[lo:hi]).sum(axis=0)
    dln = da * (1.0 + scale)
    dx = dxo + _ln_backward(dln, x, ln_eps)
    return {"dx": dx, "dw_in": dw_in, "db_in": db_in, "dq_norm": dq_norm, "dk_norm": dk_norm,
            "dw_out": dw_out, "db_out": db_out, "dmod": dmod,
            # intermediates a device implementation may be compared against stage by stage
            "dp": dp, "dycat": dycat, "dy": dy, "da": da}
