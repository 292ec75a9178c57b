"""CPU oracle for the FLUX.3 Image Klein transformer block -- TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import this
module.  It is a plain, slow, float64 NumPy restatement of what the block computes,
written from the model description "Welcome FLUX.3 Image Klein in Diffusers" (section
"How it works") and the Miles page "FLUX 3 Image Klein" (section 1 "Model
introduction" and section 3 "Family config").  It shares no code with the CUDA path.

Each step is the definition written out, in the order the description gives it:

  a = LN(x) * (1 + scale_s) + shift_s            per-stream modulation, LN without affine
  P = a W_in^T + b_in = [Q | K | V | gate | up]   one projection of the normalized input
  q, k <- RMSNorm(q) * g  then  RoPE(t, h, w, l)  per token and head
  O    = softmax(q k^T / sqrt(d)) v              all tokens (joint) or own stream only
  act  = silu(gate) * up                         SwiGLU, in parallel with attention
  x'   = x + gate_s * ([O | act] W_out^T + b_out)

Readings where the pages are silent (every one is listed in the design notes):
LN eps 1e-6 without affine; RMSNorm eps 1e-6, before RoPE, learned scale after the
normalisation; RoPE pairs are adjacent dims (2j, 2j+1) inside each axis's 32-dim
slice, axes in the listed order t, h, w, l, frequency theta^(-2j/32); softmax scale
1/sqrt(128); SwiGLU takes silu of the first F rows of the feed-forward part; W_in rows
are Q | K | V | gate | up with each head's 128 dims contiguous.

Parity status: every function below is pinned by a test that does not re-use it
(closed forms, invariants, brute force on tiny inputs, library routines).  Whole-model
agreement with the released FLUX.3 weights is "parity unpinned": the pages give no
weights and no golden outputs.
"""
from __future__ import annotations

import math
from typing import List, Optional, Sequence, Tuple

import numpy as np

F64 = np.float64


# ---------------------------------------------------------------------------------
# rounding model of the device path (optional): fp32 -> bf16 round-to-nearest-even
# ---------------------------------------------------------------------------------
def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even) through fp32, return float64.

    Used only when the oracle is asked to round its intermediates at the points where
    the device path stores bf16 tensors.  Pinned against torch's own bf16 cast."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    b = f.view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    r = ((b + 0x7FFF + lsb) & 0xFFFF0000).astype(np.uint32)
    return r.view(np.float32).astype(F64)


def _maybe_round(x: np.ndarray, rounding: Optional[str]) -> np.ndarray:
    if rounding is None:
        return x
    if rounding == "bf16":
        return round_bf16(x)
    raise ValueError(rounding)


# ---------------------------------------------------------------------------------
# normalisation and modulation ("How it works": each block's attention and SwiGLU
# read the same normalized input; scale, shift, gate come per stream)
# ---------------------------------------------------------------------------------
def layer_norm(x: np.ndarray, eps: float) -> np.ndarray:
    """LayerNorm over the last axis, biased variance, no affine parameters."""
    x = np.asarray(x, dtype=F64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def segment_ids(seg_off: Sequence[int]) -> np.ndarray:
    """Segment index of every row for contiguous segments [seg_off[s], seg_off[s+1])."""
    n = seg_off[-1]
    ids = np.empty(n, dtype=np.int64)
    for s in range(len(seg_off) - 1):
        ids[seg_off[s]:seg_off[s + 1]] = s
    return ids


def modulate(n: np.ndarray, shift: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """(1 + scale) * n + shift, broadcast over rows."""
    return n * (1.0 + scale) + shift


def ada_ln(x: np.ndarray, seg_off: Sequence[int], mod: np.ndarray, eps: float) -> np.ndarray:
    """Per-stream modulated LayerNorm.  mod[s] = (shift, scale, gate) of stream s."""
    n = layer_norm(x, eps)
    out = np.empty_like(n)
    for s in range(len(seg_off) - 1):
        a, b = seg_off[s], seg_off[s + 1]
        out[a:b] = modulate(n[a:b], mod[s, 0], mod[s, 1])
    return out


# ---------------------------------------------------------------------------------
# RoPE over four axes (t, h, w, l), 32 of the 128 head dims each ("How it works")
# ---------------------------------------------------------------------------------
def rope_angles(pos: np.ndarray, theta: float, head_dim: int = 128, n_axes: int = 4) -> np.ndarray:
    """Rotation angle of every (token, pair): [N, head_dim // 2].

    Pair p = 16 a + j (axis a, j = 0..15) rotates dims (32 a + 2 j, 32 a + 2 j + 1) by
    pos[:, a] * theta ** (-2 j / 32)."""
    pos = np.asarray(pos, dtype=F64)
    per_axis = head_dim // n_axes
    n_pairs = per_axis // 2
    ang = np.empty((pos.shape[0], n_axes * n_pairs), dtype=F64)
    for a in range(n_axes):
        for j in range(n_pairs):
            freq = theta ** (-2.0 * j / per_axis)
            ang[:, a * n_pairs + j] = pos[:, a] * freq
    return ang


def rope_rotate(x: np.ndarray, angles: np.ndarray) -> np.ndarray:
    """Rotate adjacent pairs of the last axis of x [N, H, d] by angles [N, d/2]."""
    c = np.cos(angles)[:, None, :]
    s = np.sin(angles)[:, None, :]
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis (per token, per head)."""
    ms = (x * x).mean(axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


# ---------------------------------------------------------------------------------
# attention: full bidirectional, no padding mask; optionally one group per stream
# ---------------------------------------------------------------------------------
def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
              groups: Optional[Sequence[Tuple[int, int]]] = None) -> np.ndarray:
    """softmax(q k^T / sqrt(d)) v per head; q, k, v [N, H, d] -> [N, H*d].

    groups: list of [a, b) token ranges; a query attends to the keys of its own range.
    None means one range over all tokens (the joint stage)."""
    n, h, d = q.shape
    if groups is None:
        groups = [(0, n)]
    out = np.zeros((n, h, d), dtype=F64)
    scale = 1.0 / math.sqrt(d)
    for a, b in groups:
        if b <= a:
            continue
        for hh in range(h):
            s = q[a:b, hh] @ k[a:b, hh].T * scale
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p = p / p.sum(axis=1, keepdims=True)
            out[a:b, hh] = p @ v[a:b, hh]
    return out.reshape(n, h * d)


def attention_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, rows: Sequence[int],
                   groups: Optional[Sequence[Tuple[int, int]]] = None) -> np.ndarray:
    """Rows `rows` of attention(q, k, v, groups), for sequences too long for the full
    score matrix: each sampled query row attends to the keys of its own range, one head
    at a time.  q, k, v [N, H, d] (any float dtype; computed in float64) -> [len(rows), H*d]."""
    n, h, d = k.shape
    if groups is None:
        groups = [(0, n)]
    rows = list(rows)
    own = []
    for r in rows:
        rng = [(a, b) for a, b in groups if a <= r < b]
        assert len(rng) == 1, "every sampled row must fall in exactly one range"
        own.append(rng[0])
    out = np.zeros((len(rows), h, d), dtype=F64)
    scale = 1.0 / math.sqrt(d)
    for hh in range(h):
        kh = np.asarray(k[:, hh], dtype=F64)
        vh = np.asarray(v[:, hh], dtype=F64)
        for i, r in enumerate(rows):
            a, b = own[i]
            s = kh[a:b] @ np.asarray(q[r, hh], dtype=F64) * scale
            p = np.exp(s - s.max())
            out[i, hh] = (p / p.sum()) @ vh[a:b]
    return out.reshape(len(rows), h * d)


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """silu(g) * u with silu(g) = g / (1 + exp(-g))."""
    return g / (1.0 + np.exp(-g)) * u


# ---------------------------------------------------------------------------------
# the block
# ---------------------------------------------------------------------------------
class Weights:
    """One block's parameters as float64 arrays (row layouts as in the C-ABI)."""

    def __init__(self, w_in, b_in, q_norm, k_norm, w_out, b_out):
        self.w_in = np.asarray(w_in, dtype=F64)      # [3D+2F, D]: Q | K | V | gate | up
        self.b_in = np.asarray(b_in, dtype=F64)      # [3D+2F]
        self.q_norm = np.asarray(q_norm, dtype=F64)  # [d]
        self.k_norm = np.asarray(k_norm, dtype=F64)  # [d]
        self.w_out = np.asarray(w_out, dtype=F64)    # [D, D+F]: columns attn | act
        self.b_out = np.asarray(b_out, dtype=F64)    # [D]


class BlockOut:
    """Intermediates kept for stage-by-stage comparisons."""
    a: np.ndarray; q: np.ndarray; k: np.ndarray; v: np.ndarray
    attn: np.ndarray; act: np.ndarray; y: np.ndarray; x_out: np.ndarray


def _in_proj(a: np.ndarray, w: "Weights", quant: Optional[str]) -> np.ndarray:
    """P = a W_in^T + b_in; quant "fp8": the product on row-wise e4m3 operands
    (oracle/fp8.py); "nvfp4": on NVFP4 operands (oracle/nvfp4.py)."""
    if quant == "fp8":
        from .fp8 import fp8_linear
        return fp8_linear(a, w.w_in) + w.b_in
    if quant == "nvfp4":
        from .nvfp4 import nvfp4_linear
        return nvfp4_linear(a, w.w_in) + w.b_in
    assert quant is None
    return a @ w.w_in.T + w.b_in


def _out_proj(ycat: np.ndarray, w: "Weights", quant: Optional[str]) -> np.ndarray:
    """y = [attn | act] W_out^T + b_out; quant "fp8" / "nvfp4": the product on quantized
    operands (the rows of [attn | act] and of W_out, as for the input projection)."""
    if quant == "fp8":
        from .fp8 import fp8_linear
        return fp8_linear(ycat, w.w_out) + w.b_out
    if quant == "nvfp4":
        from .nvfp4 import nvfp4_linear
        return nvfp4_linear(ycat, w.w_out) + w.b_out
    assert quant is None
    return ycat @ w.w_out.T + w.b_out


def _quant(fp8_in_proj: bool, nvfp4_in_proj: bool) -> Optional[str]:
    assert not (fp8_in_proj and nvfp4_in_proj)
    return "fp8" if fp8_in_proj else ("nvfp4" if nvfp4_in_proj else None)


def block_forward(x: np.ndarray, weights: List[Weights], seg_off: Sequence[int], mod: np.ndarray,
                  angles: np.ndarray, heads: int, head_dim: int = 128, ln_eps: float = 1e-6,
                  rms_eps: float = 1e-6, stage: int = 2, rounding: Optional[str] = None,
                  fp8_in_proj: bool = False, nvfp4_in_proj: bool = False,
                  out_proj_quant: Optional[str] = None) -> BlockOut:
    """One transformer block.

    stage 2 (joint): one weight set, attention over all tokens, modulation per stream.
    stage 1 (per stream): weights[s] for stream s, attention inside each stream.
    rounding="bf16" rounds to bf16 where the device stores bf16 tensors (the modulated
    input, q, k, v, the attention output, the SwiGLU output and x'); None keeps fp64.
    fp8_in_proj: the input projection on row-wise e4m3 operands (oracle/fp8.py);
    nvfp4_in_proj: on NVFP4 operands (oracle/nvfp4.py); out_proj_quant "fp8" / "nvfp4":
    the output projection on quantized operands too."""
    x = np.asarray(x, dtype=F64)
    n, D = x.shape
    H, d = heads, head_dim
    nseg = len(seg_off) - 1
    if stage == 2:
        assert len(weights) == 1
        rows = [(0, n, weights[0])]
        groups = None
    else:
        assert len(weights) == nseg
        rows = [(seg_off[s], seg_off[s + 1], weights[s]) for s in range(nseg)]
        groups = [(seg_off[s], seg_off[s + 1]) for s in range(nseg)]
    F = (weights[0].w_in.shape[0] - 3 * D) // 2

    r = BlockOut()
    a = _maybe_round(ada_ln(x, seg_off, mod, ln_eps), rounding)
    q = np.empty((n, H, d)); k = np.empty((n, H, d)); v = np.empty((n, H, d))
    g = np.empty((n, F)); u = np.empty((n, F))
    for lo, hi, w in rows:
        p = _in_proj(a[lo:hi], w, _quant(fp8_in_proj, nvfp4_in_proj))
        q[lo:hi] = rope_rotate(rms_norm(p[:, 0:D].reshape(-1, H, d), w.q_norm, rms_eps), angles[lo:hi])
        k[lo:hi] = rope_rotate(rms_norm(p[:, D:2 * D].reshape(-1, H, d), w.k_norm, rms_eps), angles[lo:hi])
        v[lo:hi] = p[:, 2 * D:3 * D].reshape(-1, H, d)
        g[lo:hi] = p[:, 3 * D:3 * D + F]
        u[lo:hi] = p[:, 3 * D + F:3 * D + 2 * F]
    q = _maybe_round(q, rounding); k = _maybe_round(k, rounding); v = _maybe_round(v, rounding)
    attn = _maybe_round(attention(q, k, v, groups), rounding)
    act = _maybe_round(swiglu(g, u), rounding)
    ycat = np.concatenate([attn, act], axis=1)
    y = np.empty((n, D))
    for lo, hi, w in rows:
        y[lo:hi] = _out_proj(ycat[lo:hi], w, out_proj_quant)
    gate = mod[segment_ids(seg_off), 2]
    x_out = _maybe_round(x + gate * y, rounding)
    r.a, r.q, r.k, r.v, r.attn, r.act, r.y, r.x_out = a, q, k, v, attn, act, y, x_out
    return r


# ---------------------------------------------------------------------------------
# the denoiser stack ("How it works": 5 blocks per stream with their own weights,
# concatenation, 28 shared joint blocks, output layers on image tokens only)
# ---------------------------------------------------------------------------------
def final_layer(x_img: np.ndarray, shift: np.ndarray, scale: np.ndarray, w_final: np.ndarray,
                b_final: np.ndarray, ln_eps: float = 1e-6, rounding: Optional[str] = None) -> np.ndarray:
    """Output layer on image tokens: LN, (1+scale)*x+shift, linear to the patch channels."""
    a = _maybe_round(modulate(layer_norm(x_img, ln_eps), shift, scale), rounding)
    return a @ np.asarray(w_final, dtype=F64).T + np.asarray(b_final, dtype=F64)


def dit_forward(x: np.ndarray, seg_off: Sequence[int], pos: np.ndarray,
                stage1: List[List[Weights]], stage1_mod: List[np.ndarray],
                joint: List[Weights], joint_mod: List[np.ndarray],
                final_mod: np.ndarray, w_final: np.ndarray, b_final: np.ndarray,
                heads: int, theta: float, head_dim: int = 128, ln_eps: float = 1e-6,
                rms_eps: float = 1e-6, rounding: Optional[str] = None):
    """Stage 1: for b in blocks, every stream s runs stage1[b][s] on its own tokens.
    Stage 2: the same contiguous token buffer runs the joint blocks.  The first stream
    is the image; the velocity is the final layer on its rows.  Returns (velocity, x)."""
    x = np.asarray(x, dtype=F64)
    ang = rope_angles(pos, theta, head_dim)
    for b in range(len(stage1)):
        x = block_forward(x, stage1[b], seg_off, stage1_mod[b], ang, heads, head_dim, ln_eps,
                          rms_eps, stage=1, rounding=rounding).x_out
    for b in range(len(joint)):
        x = block_forward(x, [joint[b]], seg_off, joint_mod[b], ang, heads, head_dim, ln_eps,
                          rms_eps, stage=2, rounding=rounding).x_out
    n_img = seg_off[1]
    vel = final_layer(x[:n_img], final_mod[0], final_mod[1], w_final, b_final, ln_eps, rounding)
    return vel, x


def euler_step(latent: np.ndarray, velocity: np.ndarray, sigma: float, sigma_next: float) -> np.ndarray:
    """One explicit Euler step of the flow ODE: x <- x + (sigma_next - sigma) * v."""
    return np.asarray(latent, dtype=F64) + (sigma_next - sigma) * np.asarray(velocity, dtype=F64)


def block_keys_values(x: np.ndarray, weights: List[Weights], seg_off: Sequence[int], mod: np.ndarray,
                      angles: np.ndarray, heads: int, rows: Optional[Sequence[int]] = None, head_dim: int = 128,
                      ln_eps: float = 1e-6, rms_eps: float = 1e-6, stage: int = 2,
                      rounding: Optional[str] = None, fp8_in_proj: bool = False, nvfp4_in_proj: bool = False):
    """Keys and values [len(rows), H, d] of the given rows (all rows by default): the
    same steps as block_forward up to k and v, row by row (row-wise quantization keeps a
    row's projection independent of the other rows and of W_in's other rows)."""
    x = np.asarray(x, dtype=F64)
    n, D = x.shape
    H, d = heads, head_dim
    seg = segment_ids(seg_off)
    rows = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    a = _maybe_round(modulate(layer_norm(x[rows], ln_eps), mod[seg[rows], 0], mod[seg[rows], 1]), rounding)
    k = np.empty((len(rows), H, d)); v = np.empty((len(rows), H, d))
    wsel = np.zeros(len(rows), dtype=np.int64) if stage == 2 else seg[rows]
    for wi in np.unique(wsel):
        m = wsel == wi
        w = weights[wi]
        kw = Weights(w.w_in[D:3 * D], w.b_in[D:3 * D], w.q_norm, w.k_norm, w.w_out, w.b_out)
        pkv = _in_proj(a[m], kw, _quant(fp8_in_proj, nvfp4_in_proj))
        pk, pv = pkv[:, 0:D], pkv[:, D:2 * D]
        k[m] = rope_rotate(rms_norm(pk.reshape(-1, H, d), w.k_norm, rms_eps), angles[rows[m]])
        v[m] = pv.reshape(-1, H, d)
    return _maybe_round(k, rounding), _maybe_round(v, rounding)


def block_forward_rows(x: np.ndarray, weights: List[Weights], seg_off: Sequence[int], mod: np.ndarray,
                       angles: np.ndarray, heads: int, rows: Sequence[int], head_dim: int = 128,
                       ln_eps: float = 1e-6, rms_eps: float = 1e-6, stage: int = 2,
                       rounding: Optional[str] = None, kv=None, fp8_in_proj: bool = False,
                       nvfp4_in_proj: bool = False, out_proj_quant: Optional[str] = None) -> dict:
    """The block's outputs for a few rows, at sizes where the whole block is too slow.

    A row's output needs its own q, gate/up and the keys and values of every token it
    attends to, so k and v are computed for all tokens (unless given as kv = (k, v) from
    block_keys_values) and q, the attention, the SwiGLU output and x' only for `rows`.
    Same steps and rounding points as block_forward.  Returns k, v [N, H, d] and, per
    sampled row, q, attn, act and x_out (arrays indexed like `rows`)."""
    x = np.asarray(x, dtype=F64)
    n, D = x.shape
    H, d = heads, head_dim
    seg = segment_ids(seg_off)
    F = (weights[0].w_in.shape[0] - 3 * D) // 2
    if kv is None:
        kv = block_keys_values(x, weights, seg_off, mod, angles, heads, None, head_dim, ln_eps, rms_eps, stage,
                               rounding, fp8_in_proj, nvfp4_in_proj)
    k, v = kv
    rows = list(rows)
    out = {"k": k, "v": v}
    kh = np.ascontiguousarray(k.transpose(1, 0, 2))   # [H, N, d]
    vh = np.ascontiguousarray(v.transpose(1, 0, 2))
    scale = 1.0 / math.sqrt(d)
    res = {key: [None] * len(rows) for key in ("q", "attn", "act", "x_out")}
    # rows that share a weight set and an attended range are computed together
    groups = {}
    for i, r in enumerate(rows):
        s = int(seg[r])
        groups.setdefault(0 if stage == 2 else s, []).append(i)
    for gkey, idx in groups.items():
        w = weights[0] if stage == 2 else weights[gkey]
        lo, hi = (0, n) if stage == 2 else (seg_off[gkey], seg_off[gkey + 1])
        rr = np.array([rows[i] for i in idx])
        a = _maybe_round(modulate(layer_norm(x[rr], ln_eps), mod[seg[rr], 0], mod[seg[rr], 1]), rounding)
        p = _in_proj(a, w, _quant(fp8_in_proj, nvfp4_in_proj))
        q = rope_rotate(rms_norm(p[:, 0:D].reshape(-1, H, d), w.q_norm, rms_eps), angles[rr])
        q = _maybe_round(q, rounding)
        o = np.empty((len(rr), H, d))
        for h in range(H):
            sc = q[:, h] @ kh[h, lo:hi].T * scale
            sc = sc - sc.max(axis=1, keepdims=True)
            e = np.exp(sc)
            o[:, h] = (e / e.sum(axis=1, keepdims=True)) @ vh[h, lo:hi]
        o = _maybe_round(o.reshape(len(rr), -1), rounding)
        act = _maybe_round(swiglu(p[:, 3 * D:3 * D + F], p[:, 3 * D + F:3 * D + 2 * F]), rounding)
        y = _out_proj(np.concatenate([o, act], axis=1), w, out_proj_quant)
        xo = _maybe_round(x[rr] + mod[seg[rr], 2] * y, rounding)
        for j, i in enumerate(idx):
            res["q"][i], res["attn"][i], res["act"][i], res["x_out"][i] = q[j], o[j], act[j], xo[j]
    for key in res:
        out[key] = np.array(res[key])
    return out
