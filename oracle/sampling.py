"""CPU oracle for the base-model sampling loop around the denoiser -- TEST INFRASTRUCTURE.

Only the tests may import this module; it shares no code with the CUDA path.  Float64
NumPy, written from:

  "Welcome FLUX.3 Image Klein in Diffusers", section "How it works": image tokens are the
  2x2 patches of the 32-channel latents packed into 128 channels; text is 8 Qwen3-VL
  hidden-state layers stacked into a 20,480-dim vector per token and projected to the
  width 3072; the scheduler applies a time shift of 6.93 so that 44 of 50 steps run
  above sigma = 0.5; section "What it claims": the base checkpoint runs 50 steps with
  classifier-free guidance.
  DiffSynth-Studio FLUX.3 page, pipeline arguments: cfg_scale (1.0 = off; the Base
  examples use 3.5), alpha = the rational-shift coefficient of the flow-matching
  schedule, 6.93.

Readings where the pages are silent (listed in the design notes with the rest):
  - the unshifted grid is sigma_i = 1 - i / n, i = 0..n (n + 1 values, the last 0);
  - the rational shift is sigma' = alpha sigma / (1 + (alpha - 1) sigma);
  - the velocity points from data to noise, so a step is x <- x + (sigma' - sigma) v;
  - guidance is v = v_neg + s (v_pos - v_neg);
  - both embedders are plain linear maps with a bias;
  - the timestep -> modulation map is not on the pages: modulation vectors are inputs,
    one set per step (the same for the prompted and the negative forward).

Pins (tests/test_oracle_sampling.py): the 44-of-50 statement, which fixes the grid and
the shift together; closed forms of the shift; the guidance's special cases; the
embedders against torch's linear; the loop against exact integration of a constant
velocity.
"""
from __future__ import annotations

from typing import Callable, List, Sequence

import numpy as np

F64 = np.float64


def time_shift(sigma, alpha: float):
    """Rational shift of a noise level: sigma' = alpha sigma / (1 + (alpha - 1) sigma)."""
    sigma = np.asarray(sigma, dtype=F64)
    return alpha * sigma / (1.0 + (alpha - 1.0) * sigma)


def sigma_schedule(n_steps: int, alpha: float) -> np.ndarray:
    """The n_steps + 1 noise levels of a sampling run, from 1 down to 0, shifted."""
    base = 1.0 - np.arange(n_steps + 1, dtype=F64) / n_steps
    return time_shift(base, alpha)


def cfg(v_pos: np.ndarray, v_neg: np.ndarray, scale: float) -> np.ndarray:
    """Classifier-free guidance: v_neg + s (v_pos - v_neg)."""
    v_pos = np.asarray(v_pos, dtype=F64)
    v_neg = np.asarray(v_neg, dtype=F64)
    return v_neg + scale * (v_pos - v_neg)


def embed(x: np.ndarray, w: np.ndarray, b: np.ndarray) -> np.ndarray:
    """A token embedder: x W^T + b (image: 128 -> width, text: 20,480 -> width)."""
    return np.asarray(x, dtype=F64) @ np.asarray(w, dtype=F64).T + np.asarray(b, dtype=F64)


def sample(latent: np.ndarray, sigmas: Sequence[float],
           velocity: Callable[[np.ndarray, int, bool], np.ndarray], cfg_scale: float,
           round_latent: Callable[[np.ndarray], np.ndarray] = lambda a: a) -> List[np.ndarray]:
    """The Euler sampling loop.  velocity(latent, step, prompted) runs the denoiser on the
    image tokens embedded from `latent` (with the prompt's text tokens when prompted is
    True, the negative prompt's otherwise) and returns its velocity for the image rows.
    With cfg_scale == 1 the negative forward is skipped (guidance is off).  round_latent
    models how the device feeds the latent to the image embedder (bf16).  Returns the
    latent after every step (step 0 = the input)."""
    x = np.asarray(latent, dtype=F64).copy()
    out = [x.copy()]
    for i in range(len(sigmas) - 1):
        xin = round_latent(x)
        v = velocity(xin, i, True)
        if cfg_scale != 1.0:
            v = cfg(v, velocity(xin, i, False), cfg_scale)
        x = x + (sigmas[i + 1] - sigmas[i]) * v
        out.append(x.copy())
    return out
