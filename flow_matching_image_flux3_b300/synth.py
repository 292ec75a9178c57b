"""Seeded synthetic inputs for the FLUX.3 Image Klein transformer block.

This module only draws random numbers and lays out position ids; it holds none of
the block's arithmetic.  Both the CUDA path (through the C-ABI) and the CPU oracle
consume the tensors it returns, so the two sides see bit-identical inputs.

Value recipe (same for every configuration):
  * activations x ~ N(0, 1), drawn in fp32 and rounded to bf16;
  * projection weights ~ N(0, 1/fan_in) (fan_in = width for W_in, width + ffn_hidden
    for W_out), drawn in fp32 and rounded to bf16; biases are zero unless asked for;
  * QK RMSNorm scales ~ 1 + N(0, 0.1), fp32;
  * per-stream modulation shift ~ N(0, 0.1), scale ~ N(0, 0.1), gate ~ N(0, 0.5), fp32.
Draw order from one CPU generator: x, then per weight set (W_in, [b_in], g_q, g_k,
W_out, [b_out]), then modulation per segment.

Token layout (the pages' description of the model, "Welcome FLUX.3 Image Klein in
Diffusers", section "How it works"): one image token per 2x2 packed latent patch, i.e.
per 16x16 pixels, so 1024x1024 gives a 64x64 grid = 4,096 tokens; text is padded to a
multiple of 80 tokens; references keep their own grid and share (h, w) with the image.
Position ids are (t, h, w, l): image (t_img, h, w, 0), reference k (k+1, h, w, 0), text
(0, 0, 0, l) with l counting through the padding.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np
import torch

HEAD_DIM = 128


@dataclasses.dataclass
class Dims:
    width: int
    heads: int
    ffn_hidden: int
    head_dim: int = HEAD_DIM
    ln_eps: float = 1e-6
    rms_eps: float = 1e-6
    rope_theta: float = 10000.0

    @property
    def n_in(self) -> int:
        """Rows of the fused input projection: Q | K | V | gate | up."""
        return 3 * self.width + 2 * self.ffn_hidden

    @property
    def k_out(self) -> int:
        """Columns of the fused output projection: attention out | SwiGLU act."""
        return self.width + self.ffn_hidden


TINY = Dims(width=256, heads=2, ffn_hidden=768)
FULL = Dims(width=3072, heads=24, ffn_hidden=9216)


@dataclasses.dataclass
class Stream:
    kind: str            # "image", "ref" or "text"
    n: int               # tokens
    grid: Optional[tuple] = None   # (rows, cols) for image/ref
    t: int = 0           # t coordinate for image/ref tokens


@dataclasses.dataclass
class BlockWeights:
    w_in: torch.Tensor      # bf16 [3D+2F, D]
    b_in: torch.Tensor      # fp32 [3D+2F]
    q_norm: torch.Tensor    # fp32 [128]
    k_norm: torch.Tensor    # fp32 [128]
    w_out: torch.Tensor     # bf16 [D, D+F]
    b_out: torch.Tensor     # fp32 [D]


@dataclasses.dataclass
class BlockCase:
    dims: Dims
    x: torch.Tensor                 # bf16 [N, D]
    pos: torch.Tensor               # int32 [N, 4]
    seg_off: List[int]              # [n_seg + 1]
    mod: torch.Tensor               # fp32 [n_seg, 3, D]: shift, scale, gate
    weights: List[BlockWeights]     # 1 (joint block) or n_seg (per-stream block)
    stage: int                      # 2 = joint block, 1 = per-stream block
    streams: List[Stream]

    @property
    def n(self) -> int:
        return int(self.x.shape[0])


def positions(streams: Sequence[Stream]) -> torch.Tensor:
    """Position ids (t, h, w, l) for the concatenated streams, int32 [N, 4]."""
    rows = []
    for s in streams:
        p = torch.zeros(s.n, 4, dtype=torch.int32)
        if s.kind in ("image", "ref"):
            gh, gw = s.grid
            assert gh * gw == s.n
            hh = torch.arange(gh, dtype=torch.int32).repeat_interleave(gw)
            ww = torch.arange(gw, dtype=torch.int32).repeat(gh)
            p[:, 0] = s.t
            p[:, 1] = hh
            p[:, 2] = ww
        elif s.kind == "text":
            p[:, 3] = torch.arange(s.n, dtype=torch.int32)
        else:
            raise ValueError(s.kind)
        rows.append(p)
    return torch.cat(rows, 0)


def _randn(g: torch.Generator, shape, std: float = 1.0, mean: float = 0.0) -> torch.Tensor:
    return torch.randn(*shape, generator=g, dtype=torch.float32) * std + mean


def draw_weights(g: torch.Generator, dims: Dims, bias: bool = False) -> BlockWeights:
    D, F = dims.width, dims.ffn_hidden
    w_in = _randn(g, (dims.n_in, D), std=D ** -0.5).to(torch.bfloat16)
    b_in = (_randn(g, (dims.n_in,), std=0.1) if bias else torch.zeros(dims.n_in))
    q_norm = _randn(g, (dims.head_dim,), std=0.1, mean=1.0)
    k_norm = _randn(g, (dims.head_dim,), std=0.1, mean=1.0)
    w_out = _randn(g, (D, D + F), std=(D + F) ** -0.5).to(torch.bfloat16)
    b_out = (_randn(g, (D,), std=0.1) if bias else torch.zeros(D))
    return BlockWeights(w_in, b_in.float(), q_norm, k_norm, w_out, b_out.float())


def draw_mod(g: torch.Generator, n_seg: int, D: int) -> torch.Tensor:
    m = torch.empty(n_seg, 3, D)
    for s in range(n_seg):
        m[s, 0] = _randn(g, (D,), std=0.1)
        m[s, 1] = _randn(g, (D,), std=0.1)
        m[s, 2] = _randn(g, (D,), std=0.5)
    return m


def make_case(dims: Dims, streams: Sequence[Stream], seed: int, stage: int = 2,
              bias: bool = False) -> BlockCase:
    """One block's inputs. stage 2: one weight set shared by all tokens; stage 1: one
    weight set per stream. Modulation is always per stream."""
    g = torch.Generator("cpu").manual_seed(seed)
    n = sum(s.n for s in streams)
    x = _randn(g, (n, dims.width)).to(torch.bfloat16)
    n_w = 1 if stage == 2 else len(streams)
    weights = [draw_weights(g, dims, bias) for _ in range(n_w)]
    mod = draw_mod(g, len(streams), dims.width)
    seg_off = [0]
    for s in streams:
        seg_off.append(seg_off[-1] + s.n)
    return BlockCase(dims, x, positions(streams), seg_off, mod, weights, stage, list(streams))


def image_stream(px_h: int, px_w: int, t: int = 0, kind: str = "image") -> Stream:
    """A 16-px-per-token grid (8x VAE downsampling, 2x2 latent packing)."""
    gh, gw = px_h // 16, px_w // 16
    return Stream(kind, gh * gw, (gh, gw), t)


def text_stream(n_tokens: int) -> Stream:
    return Stream("text", n_tokens)


def config(idx: int, bias: bool = False) -> BlockCase:
    """The block-level workloads: 0 tiny joint block, 1 joint block at 1024^2,
    2 per-stream blocks (image | ref | text), 3 joint block with one reference."""
    if idx == 0:
        return make_case(TINY, [image_stream(128, 128), text_stream(80)], seed=0, stage=2, bias=bias)
    if idx == 1:
        return make_case(FULL, [image_stream(1024, 1024), text_stream(160)], seed=1, stage=2, bias=bias)
    if idx == 2:
        return make_case(FULL, [image_stream(1024, 1024), image_stream(1024, 1024, t=1, kind="ref"),
                                text_stream(240)], seed=2, stage=1, bias=bias)
    if idx == 3:
        return make_case(FULL, [image_stream(1024, 1024), image_stream(1024, 1024, t=1, kind="ref"),
                                text_stream(160)], seed=3, stage=2, bias=bias)
    raise ValueError(idx)


def config_refs(n_refs: int, stage: int, seed: int, bias: bool = False) -> BlockCase:
    """Multi-reference editing at 1024^2: the image, n_refs references of 4,096 tokens each
    (reference k at t = k + 1 on the image's (h, w) grid) and 160 text tokens.  The
    references form one stream: one segment for modulation and, in stage 1, one
    self-attending range and weight set."""
    img = image_stream(1024, 1024)
    refs = [image_stream(1024, 1024, t=k + 1, kind="ref") for k in range(n_refs)]
    txt = text_stream(160)
    g = torch.Generator("cpu").manual_seed(seed)
    dims = FULL
    n = img.n + sum(r.n for r in refs) + txt.n
    x = _randn(g, (n, dims.width)).to(torch.bfloat16)
    weights = [draw_weights(g, dims, bias) for _ in range(1 if stage == 2 else 3)]
    mod = draw_mod(g, 3, dims.width)
    seg_off = [0, img.n, img.n + sum(r.n for r in refs), n]
    return BlockCase(dims, x, positions([img] + refs + [txt]), seg_off, mod, weights, stage, [img] + refs + [txt])


def as_f64(t: torch.Tensor) -> np.ndarray:
    """Exact upcast of a CPU tensor (bf16 or fp32) to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()
