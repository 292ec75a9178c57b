"""ctypes binding of libflux3.so (include/flux3.h).

Argument marshalling only: torch tensors provide device memory and the current CUDA
stream; every step of the block runs in the library's CUDA kernels.  There is no CPU
fallback: if the library cannot be loaded, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libflux3.so")

c_i32, c_f32, c_vp, c_size = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(6)
MAX_SEGMENTS = 16
KERNEL_NAMES = {1: "rope", 2: "adaln", 3: "in_proj", 4: "attn", 5: "out_proj", 6: "final", 7: "euler", 8: "attn_f32",
                9: "linear", 10: "cfg_euler", 11: "to_bf16", 12: "quantize", 13: "bwd_gemm", 14: "bwd_elem"}


class flux3_dims(ctypes.Structure):
    _fields_ = [("width", c_i32), ("heads", c_i32), ("head_dim", c_i32), ("ffn_hidden", c_i32),
                ("ln_eps", c_f32), ("rms_eps", c_f32), ("rope_theta", c_f32)]


class flux3_block_weights(ctypes.Structure):
    _fields_ = [("w_in", c_vp), ("b_in", c_vp), ("q_norm", c_vp), ("k_norm", c_vp), ("w_out", c_vp), ("b_out", c_vp)]


class flux3_block_weights_fp8(ctypes.Structure):
    _fields_ = [("w_in", c_vp), ("s_in", c_vp), ("b_in", c_vp), ("q_norm", c_vp), ("k_norm", c_vp), ("w_out", c_vp),
                ("b_out", c_vp), ("w_out_q", c_vp), ("s_out", c_vp)]


class flux3_block_weights_nvfp4(ctypes.Structure):
    _fields_ = [("w_in", c_vp), ("w_sf", c_vp), ("s_in", c_vp), ("b_in", c_vp), ("q_norm", c_vp), ("k_norm", c_vp),
                ("w_out", c_vp), ("b_out", c_vp), ("w_out_q", c_vp), ("w_out_sf", c_vp), ("s_out", c_vp)]


class flux3_segments(ctypes.Structure):
    _fields_ = [("n_seg", c_i32), ("seg_off", ctypes.POINTER(c_i32)), ("mod", c_vp)]


class flux3_dit_weights(ctypes.Structure):
    _fields_ = [("n_streams", c_i32), ("n_stage1", c_i32), ("n_joint", c_i32),
                ("stage1", ctypes.POINTER(flux3_block_weights)), ("joint", ctypes.POINTER(flux3_block_weights)),
                ("w_final", c_vp), ("b_final", c_vp), ("out_channels", c_i32)]


class flux3_dit_mod(ctypes.Structure):
    _fields_ = [("stage1", c_vp), ("joint", c_vp), ("final", c_vp)]


class flux3_sample_args(ctypes.Structure):
    _fields_ = [("n_img", c_i32), ("n_ref", c_i32), ("n_txt", c_i32), ("latent_channels", c_i32), ("text_dim", c_i32),
                ("w_img", c_vp), ("b_img", c_vp), ("w_txt", c_vp), ("b_txt", c_vp), ("ref_latent", c_vp),
                ("text_pos", c_vp), ("text_neg", c_vp), ("pos", c_vp), ("mod", ctypes.POINTER(flux3_dit_mod)),
                ("n_steps", c_i32), ("alpha", c_f32), ("cfg_scale", c_f32), ("cache_context", c_i32)]


class Flux3Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {lib.flux3_status_string(status).decode()} (status {status})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libflux3.so is not built ({LIB_PATH}); run __graft_entry__.build() or "
                          f"python -m flow_matching_image_flux3_b300.build")
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    sig = {
        "flux3_status_string": (ctypes.c_char_p, [c_i32]),
        "flux3_version": (ctypes.c_char_p, []),
        "flux3_rope_build": (c_i32, [P(flux3_dims), c_vp, c_i32, c_vp, c_vp]),
        "flux3_adaln_fwd": (c_i32, [P(flux3_dims), P(flux3_segments), c_vp, c_i32, c_vp, c_vp]),
        "flux3_in_proj_fwd": (c_i32, [P(flux3_dims), P(flux3_block_weights), c_i32, P(flux3_segments), c_vp, c_i32,
                                      c_vp, c_vp, c_vp, c_vp, c_i32, c_vp, c_vp]),
        "flux3_attn_fwd": (c_i32, [P(flux3_dims), c_vp, c_vp, c_vp, c_i32, c_i32, P(c_i32), c_i32, c_vp, c_i32,
                                   c_i32, c_vp]),
        "flux3_out_proj_fwd": (c_i32, [P(flux3_dims), P(flux3_block_weights), c_i32, P(flux3_segments), c_vp, c_vp,
                                       c_vp, c_i32, c_vp]),
        "flux3_block_workspace_size": (c_size, [P(flux3_dims), c_i32]),
        "flux3_block_fwd": (c_i32, [P(flux3_dims), P(flux3_block_weights), P(flux3_segments), c_vp, c_vp, c_i32,
                                    c_vp, c_vp, c_size, c_vp]),
        "flux3_stream_block_fwd": (c_i32, [P(flux3_dims), P(flux3_block_weights), P(flux3_segments), c_vp, c_vp,
                                           c_i32, c_vp, c_vp, c_size, c_vp]),
        "flux3_final_fwd": (c_i32, [P(flux3_dims), c_vp, c_vp, c_i32, c_vp, c_vp, c_i32, c_vp, c_vp, c_size, c_vp]),
        "flux3_dit_workspace_size": (c_size, [P(flux3_dims), c_i32, c_i32, c_i32]),
        "flux3_dit_fwd": (c_i32, [P(flux3_dims), P(flux3_dit_weights), P(flux3_dit_mod), c_vp, c_i32, c_i32, c_i32,
                                  c_vp, c_vp, c_vp, c_size, c_vp]),
        "flux3_euler_step": (c_i32, [c_vp, c_vp, ctypes.c_int64, c_f32, c_f32, c_vp]),
        "flux3_sigma_schedule": (c_i32, [c_i32, c_f32, P(c_f32)]),
        "flux3_linear_fwd": (c_i32, [P(flux3_dims), c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_i32, c_vp]),
        "flux3_cfg_euler_step": (c_i32, [c_vp, c_vp, c_vp, ctypes.c_int64, c_f32, c_f32, c_f32, c_vp, c_vp]),
        "flux3_sample_workspace_size": (c_size, [P(flux3_dims), P(flux3_sample_args)]),
        "flux3_quantize_rows_fp8": (c_i32, [c_vp, c_i32, c_i32, c_vp, c_vp, c_vp]),
        "flux3_in_proj_fp8_fwd": (c_i32, [P(flux3_dims), P(flux3_block_weights_fp8), c_i32, P(flux3_segments), c_vp,
                                          c_vp, c_i32, c_vp, c_vp, c_vp, c_vp, c_i32, c_vp, c_vp]),
        "flux3_block_fp8_workspace_size": (c_size, [P(flux3_dims), c_i32]),
        "flux3_block_fp8_fwd": (c_i32, [P(flux3_dims), P(flux3_block_weights_fp8), P(flux3_segments), c_vp, c_vp,
                                        c_i32, c_vp, c_vp, c_size, c_vp]),
        "flux3_sample_fwd": (c_i32, [P(flux3_dims), P(flux3_dit_weights), P(flux3_sample_args), c_vp, c_vp, c_size,
                                     c_vp]),
        "flux3_block_bwd_workspace_size": (c_size, [P(flux3_dims), c_i32]),
        "flux3_block_bwd": (c_i32, [P(flux3_dims), P(flux3_block_weights), P(flux3_segments), c_vp, c_vp, c_vp, c_i32,
                                    c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_size, c_vp]),
        "flux3_stream_block_bwd_workspace_size": (c_size, [P(flux3_dims), P(flux3_segments)]),
        "flux3_stream_block_bwd": (c_i32, [P(flux3_dims), P(flux3_block_weights), P(flux3_segments), c_vp, c_vp, c_vp,
                                           c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_size, c_vp]),
        "flux3_nvfp4_scale_bytes": (c_size, [c_i32, c_i32]),
        "flux3_quantize_rows_nvfp4": (c_i32, [c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp]),
        "flux3_in_proj_nvfp4_fwd": (c_i32, [P(flux3_dims), P(flux3_block_weights_nvfp4), c_vp, c_vp, c_vp, c_i32, c_vp,
                                            c_vp, c_vp, c_vp, c_i32, c_vp, c_vp]),
        "flux3_block_nvfp4_workspace_size": (c_size, [P(flux3_dims), c_i32]),
        "flux3_block_nvfp4_fwd": (c_i32, [P(flux3_dims), P(flux3_block_weights_nvfp4), P(flux3_segments), c_vp, c_vp,
                                          c_i32, c_vp, c_vp, c_size, c_vp]),
        "flux3_block_fwd_static": (c_i32, [P(flux3_dims), P(flux3_block_weights), P(flux3_segments), c_vp, c_vp,
                                           c_i32, c_vp, c_vp]),
        "flux3_device_error": (c_i32, [P(ctypes.c_uint32), c_i32]),
        "flux3_selftest_timeout": (c_i32, [ctypes.c_uint32]),
        "flux3_profile_begin": (c_i32, [c_i32]),
        "flux3_profile_end": (c_i32, [P(c_f32), P(c_i32), c_i32, P(c_i32)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


lib = _load()
EXPORTED = [
    "flux3_status_string", "flux3_version", "flux3_rope_build", "flux3_adaln_fwd", "flux3_in_proj_fwd",
    "flux3_attn_fwd", "flux3_out_proj_fwd", "flux3_block_workspace_size", "flux3_block_fwd",
    "flux3_stream_block_fwd", "flux3_final_fwd", "flux3_dit_workspace_size", "flux3_dit_fwd", "flux3_euler_step",
    "flux3_device_error", "flux3_profile_begin", "flux3_profile_end", "flux3_block_fwd_static",
    "flux3_sigma_schedule", "flux3_linear_fwd", "flux3_cfg_euler_step", "flux3_sample_workspace_size",
    "flux3_sample_fwd", "flux3_quantize_rows_fp8", "flux3_in_proj_fp8_fwd", "flux3_block_fp8_workspace_size",
    "flux3_block_fp8_fwd", "flux3_selftest_timeout", "flux3_nvfp4_scale_bytes", "flux3_quantize_rows_nvfp4",
    "flux3_in_proj_nvfp4_fwd", "flux3_block_nvfp4_workspace_size", "flux3_block_nvfp4_fwd",
    "flux3_block_bwd_workspace_size", "flux3_block_bwd", "flux3_stream_block_bwd_workspace_size",
    "flux3_stream_block_bwd",
]
STATIC_SCRATCH_BYTES = 64 << 20


def _check(fn: str, st: int) -> None:
    if st != OK:
        raise Flux3Error(fn, st)


# ----------------------------------------------------------------- marshalling helpers
def make_dims(d) -> flux3_dims:
    return flux3_dims(d.width, d.heads, getattr(d, "head_dim", 128), d.ffn_hidden, getattr(d, "ln_eps", 1e-6),
                      getattr(d, "rms_eps", 1e-6), getattr(d, "rope_theta", 1e4))


def _ptr(t: Optional[torch.Tensor], dtype=None) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _offsets(seg_off: Sequence[int]):
    arr = (c_i32 * len(seg_off))(*[int(v) for v in seg_off])
    return arr


class Segments:
    """Keeps the host offset array alive for the duration of a call."""

    def __init__(self, seg_off: Sequence[int], mod: Optional[torch.Tensor]):
        self.off = _offsets(seg_off)
        self.s = flux3_segments(len(seg_off) - 1, ctypes.cast(self.off, ctypes.POINTER(c_i32)),
                                _ptr(mod, torch.float32))


def block_weights(w) -> flux3_block_weights:
    """w: object with w_in, b_in, q_norm, k_norm, w_out, b_out device tensors (b_* may be None)."""
    return flux3_block_weights(_ptr(w.w_in, torch.bfloat16), _ptr(getattr(w, "b_in", None), torch.float32),
                               _ptr(w.q_norm, torch.float32), _ptr(w.k_norm, torch.float32),
                               _ptr(w.w_out, torch.bfloat16), _ptr(getattr(w, "b_out", None), torch.float32))


def _weights_array(ws: Sequence) -> ctypes.Array:
    return (flux3_block_weights * len(ws))(*[block_weights(w) for w in ws])


# ----------------------------------------------------------------- entry points
def version() -> str:
    return lib.flux3_version().decode()


def rope_build(dims, pos: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    n = pos.shape[0]
    out = out if out is not None else torch.empty(n, 64, 2, dtype=torch.float32, device=pos.device)
    d = make_dims(dims)
    _check("flux3_rope_build", lib.flux3_rope_build(ctypes.byref(d), _ptr(pos, torch.int32), n, _ptr(out, torch.float32),
                                                    _stream(stream)))
    return out


def adaln_fwd(dims, x: torch.Tensor, seg_off: Sequence[int], mod: torch.Tensor, out=None, stream=None) -> torch.Tensor:
    out = out if out is not None else torch.empty_like(x)
    d, s = make_dims(dims), Segments(seg_off, mod)
    _check("flux3_adaln_fwd", lib.flux3_adaln_fwd(ctypes.byref(d), ctypes.byref(s.s), _ptr(x, torch.bfloat16), x.shape[0],
                                                  _ptr(out, torch.bfloat16), _stream(stream)))
    return out


def ld_vt(n: int) -> int:
    return (n + 7) // 8 * 8


def in_proj_fwd(dims, weights: Sequence, seg_off: Sequence[int], a: torch.Tensor, rope: torch.Tensor, stream=None):
    """Returns q, k [H, N, 128], vt [H, 128, ld_vt], y [N, D + F] (act in columns D..)."""
    n = a.shape[0]
    D, H, F = dims.width, dims.heads, dims.ffn_hidden
    dev = a.device
    q = torch.empty(H, n, 128, dtype=torch.bfloat16, device=dev)
    k = torch.empty_like(q)
    ldv = ld_vt(n)
    vt = torch.zeros(H, 128, ldv, dtype=torch.bfloat16, device=dev)
    y = torch.zeros(n, D + F, dtype=torch.bfloat16, device=dev)
    d, s = make_dims(dims), Segments(seg_off, None)
    wa = _weights_array(weights)
    _check("flux3_in_proj_fwd", lib.flux3_in_proj_fwd(ctypes.byref(d), wa, len(weights), ctypes.byref(s.s),
                                                      _ptr(a, torch.bfloat16), n, _ptr(rope, torch.float32), _ptr(q),
                                                      _ptr(k), _ptr(vt), ldv, _ptr(y), _stream(stream)))
    return q, k, vt, y


def attn_fwd(dims, q, k, vt, seg_off: Optional[Sequence[int]] = None, out: Optional[torch.Tensor] = None,
             fp32_debug: bool = False, stream=None) -> torch.Tensor:
    H, n, _ = q.shape
    if out is None:
        out = torch.zeros(n, H * 128, dtype=torch.float32 if fp32_debug else torch.bfloat16, device=q.device)
    d = make_dims(dims)
    off = _offsets(seg_off) if seg_off is not None else None
    n_seg = len(seg_off) - 1 if seg_off is not None else 1
    _check("flux3_attn_fwd", lib.flux3_attn_fwd(ctypes.byref(d), _ptr(q, torch.bfloat16), _ptr(k, torch.bfloat16),
                                                _ptr(vt, torch.bfloat16), vt.shape[2], n,
                                                ctypes.cast(off, ctypes.POINTER(c_i32)) if off is not None else None,
                                                n_seg, _ptr(out), out.stride(0), 1 if fp32_debug else 0, _stream(stream)))
    return out


def out_proj_fwd(dims, weights: Sequence, seg_off: Sequence[int], mod: torch.Tensor, y: torch.Tensor, x: torch.Tensor,
                 x_out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    x_out = x_out if x_out is not None else torch.empty_like(x)
    d, s = make_dims(dims), Segments(seg_off, mod)
    wa = _weights_array(weights)
    _check("flux3_out_proj_fwd", lib.flux3_out_proj_fwd(ctypes.byref(d), wa, len(weights), ctypes.byref(s.s),
                                                        _ptr(y, torch.bfloat16), _ptr(x, torch.bfloat16),
                                                        _ptr(x_out, torch.bfloat16), x.shape[0], _stream(stream)))
    return x_out


def block_workspace_size(dims, n: int) -> int:
    d = make_dims(dims)
    return int(lib.flux3_block_workspace_size(ctypes.byref(d), n))


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def block_fwd(dims, weights, seg_off: Sequence[int], mod: torch.Tensor, x: torch.Tensor, rope: torch.Tensor,
              x_out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Stage-2 joint block (one weight set) or, with a list of one weight set per
    segment, use stream_block_fwd."""
    n = x.shape[0]
    x_out = x_out if x_out is not None else torch.empty_like(x)
    need = block_workspace_size(dims, n)
    ws = ws if ws is not None else workspace(need, x.device)
    d, s = make_dims(dims), Segments(seg_off, mod)
    w = block_weights(weights)
    _check("flux3_block_fwd", lib.flux3_block_fwd(ctypes.byref(d), ctypes.byref(w), ctypes.byref(s.s),
                                                  _ptr(x, torch.bfloat16), _ptr(x_out, torch.bfloat16), n,
                                                  _ptr(rope, torch.float32), _ptr(ws), ws.numel(), _stream(stream)))
    return x_out


def block_fwd_static(dims, weights, seg_off: Sequence[int], mod: torch.Tensor, x: torch.Tensor, rope: torch.Tensor,
                     x_out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """block_fwd for callers that cannot allocate device memory: the scratch is the
    library's own static device array (at most STATIC_SCRATCH_BYTES), so no workspace is
    passed.  Calls share that array; do not overlap them on the GPU."""
    x_out = x_out if x_out is not None else torch.empty_like(x)
    d, s = make_dims(dims), Segments(seg_off, mod)
    w = block_weights(weights)
    _check("flux3_block_fwd_static", lib.flux3_block_fwd_static(ctypes.byref(d), ctypes.byref(w), ctypes.byref(s.s),
                                                                _ptr(x, torch.bfloat16), _ptr(x_out, torch.bfloat16),
                                                                x.shape[0], _ptr(rope, torch.float32), _stream(stream)))
    return x_out


def stream_block_fwd(dims, weights: Sequence, seg_off: Sequence[int], mod: torch.Tensor, x: torch.Tensor,
                     rope: torch.Tensor, x_out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
    n = x.shape[0]
    x_out = x_out if x_out is not None else torch.empty_like(x)
    ws = ws if ws is not None else workspace(block_workspace_size(dims, n), x.device)
    d, s = make_dims(dims), Segments(seg_off, mod)
    wa = _weights_array(weights)
    _check("flux3_stream_block_fwd", lib.flux3_stream_block_fwd(ctypes.byref(d), wa, ctypes.byref(s.s),
                                                                _ptr(x, torch.bfloat16), _ptr(x_out, torch.bfloat16), n,
                                                                _ptr(rope, torch.float32), _ptr(ws), ws.numel(),
                                                                _stream(stream)))
    return x_out


def final_fwd(dims, w_final: torch.Tensor, b_final: Optional[torch.Tensor], mod_final: torch.Tensor, x: torch.Tensor,
              out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    n = x.shape[0]
    oc = w_final.shape[0]
    out = out if out is not None else torch.empty(n, oc, dtype=torch.float32, device=x.device)
    ws = ws if ws is not None else workspace((n * dims.width * 2 + 255) // 256 * 256, x.device)
    d = make_dims(dims)
    _check("flux3_final_fwd", lib.flux3_final_fwd(ctypes.byref(d), _ptr(w_final, torch.bfloat16),
                                                  _ptr(b_final, torch.float32), oc, _ptr(mod_final, torch.float32),
                                                  _ptr(x, torch.bfloat16), n, _ptr(out, torch.float32), _ptr(ws),
                                                  ws.numel(), _stream(stream)))
    return out


def dit_workspace_size(dims, n_img: int, n_ref: int, n_txt: int) -> int:
    d = make_dims(dims)
    return int(lib.flux3_dit_workspace_size(ctypes.byref(d), n_img, n_ref, n_txt))


class DitArgs:
    """Host structs of a denoiser stack; keeps the weight arrays alive."""

    def __init__(self, stage1: Sequence[Sequence], joint: Sequence, w_final: torch.Tensor,
                 b_final: Optional[torch.Tensor], mod_stage1: Optional[torch.Tensor], mod_joint: Optional[torch.Tensor],
                 mod_final: torch.Tensor, n_streams: int):
        # the structs hold raw device addresses: keep every tensor alive with this object
        self._keep = [stage1, joint, w_final, b_final, mod_stage1, mod_joint, mod_final]
        flat = [w for blk in stage1 for w in blk]
        self.s1 = _weights_array(flat) if flat else None
        self.j = _weights_array(joint) if joint else None
        P = ctypes.POINTER(flux3_block_weights)
        self.w = flux3_dit_weights(n_streams, len(stage1), len(joint),
                                   ctypes.cast(self.s1, P) if self.s1 is not None else None,
                                   ctypes.cast(self.j, P) if self.j is not None else None,
                                   _ptr(w_final, torch.bfloat16), _ptr(b_final, torch.float32), w_final.shape[0])
        self.m = flux3_dit_mod(_ptr(mod_stage1, torch.float32), _ptr(mod_joint, torch.float32),
                               _ptr(mod_final, torch.float32))


def dit_fwd(dims, args: DitArgs, tokens: torch.Tensor, n_img: int, n_ref: int, n_txt: int, pos: torch.Tensor,
            velocity: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    oc = args.w.out_channels
    velocity = velocity if velocity is not None else torch.empty(n_img, oc, dtype=torch.float32, device=tokens.device)
    ws = ws if ws is not None else workspace(dit_workspace_size(dims, n_img, n_ref, n_txt), tokens.device)
    d = make_dims(dims)
    _check("flux3_dit_fwd", lib.flux3_dit_fwd(ctypes.byref(d), ctypes.byref(args.w), ctypes.byref(args.m),
                                              _ptr(tokens, torch.bfloat16), n_img, n_ref, n_txt, _ptr(pos, torch.int32),
                                              _ptr(velocity, torch.float32), _ptr(ws), ws.numel(), _stream(stream)))
    return velocity


def euler_step(latent: torch.Tensor, velocity: torch.Tensor, sigma: float, sigma_next: float, stream=None) -> None:
    _check("flux3_euler_step", lib.flux3_euler_step(_ptr(latent, torch.float32), _ptr(velocity, torch.float32),
                                                    latent.numel(), sigma, sigma_next, _stream(stream)))


def sigma_schedule(n_steps: int, alpha: float) -> List[float]:
    """Noise levels of an n_steps run (host only, no GPU needed)."""
    out = (c_f32 * (n_steps + 1))()
    _check("flux3_sigma_schedule", lib.flux3_sigma_schedule(n_steps, alpha, out))
    return list(out)


def linear_fwd(dims, x: torch.Tensor, w: torch.Tensor, b: Optional[torch.Tensor] = None,
               out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out[r, :D] = x[r] W^T + b in bf16 (a token embedder); out may be a row slice of a
    wider token buffer (its row stride is passed)."""
    rows, k = x.shape
    out = out if out is not None else torch.empty(rows, dims.width, dtype=torch.bfloat16, device=x.device)
    assert out.dtype == torch.bfloat16 and out.stride(1) == 1 and out.shape[0] == rows
    d = make_dims(dims)
    if not out.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    _check("flux3_linear_fwd", lib.flux3_linear_fwd(ctypes.byref(d), _ptr(x, torch.bfloat16), rows, k,
                                                    _ptr(w, torch.bfloat16), _ptr(b, torch.float32), out.data_ptr(),
                                                    out.stride(0), _stream(stream)))
    return out


def cfg_euler_step(latent: torch.Tensor, v_pos: torch.Tensor, v_neg: Optional[torch.Tensor], cfg_scale: float,
                   sigma: float, sigma_next: float, latent_bf16: Optional[torch.Tensor] = None, stream=None) -> None:
    _check("flux3_cfg_euler_step", lib.flux3_cfg_euler_step(
        _ptr(latent, torch.float32), _ptr(v_pos, torch.float32), _ptr(v_neg, torch.float32), latent.numel(),
        cfg_scale, sigma, sigma_next, _ptr(latent_bf16, torch.bfloat16), _stream(stream)))


class SampleArgs:
    """Host struct of the sampling loop; keeps the tensors and the per-step modulation
    structs alive."""

    def __init__(self, n_img: int, n_ref: int, n_txt: int, w_img: torch.Tensor, b_img: Optional[torch.Tensor],
                 w_txt: torch.Tensor, b_txt: Optional[torch.Tensor], text_pos: torch.Tensor,
                 text_neg: Optional[torch.Tensor], pos: torch.Tensor, step_mods: Sequence, n_steps: int,
                 alpha: float, cfg_scale: float, ref_latent: Optional[torch.Tensor] = None,
                 cache_context: bool = False):
        # step_mods: one (mod_stage1, mod_joint, mod_final) device tuple per step
        self._keep = [w_img, b_img, w_txt, b_txt, text_pos, text_neg, pos, step_mods, ref_latent]
        self.mods = (flux3_dit_mod * n_steps)(*[flux3_dit_mod(_ptr(m[0], torch.float32), _ptr(m[1], torch.float32),
                                                             _ptr(m[2], torch.float32)) for m in step_mods])
        self.a = flux3_sample_args(n_img, n_ref, n_txt, w_img.shape[1], w_txt.shape[1], _ptr(w_img, torch.bfloat16),
                                   _ptr(b_img, torch.float32), _ptr(w_txt, torch.bfloat16), _ptr(b_txt, torch.float32),
                                   _ptr(ref_latent, torch.bfloat16), _ptr(text_pos, torch.bfloat16),
                                   _ptr(text_neg, torch.bfloat16), _ptr(pos, torch.int32),
                                   ctypes.cast(self.mods, ctypes.POINTER(flux3_dit_mod)), n_steps, alpha, cfg_scale,
                                   int(bool(cache_context)))


def sample_workspace_size(dims, args: SampleArgs) -> int:
    d = make_dims(dims)
    return int(lib.flux3_sample_workspace_size(ctypes.byref(d), ctypes.byref(args.a)))


def sample_fwd(dims, dit: "DitArgs", args: SampleArgs, latent: torch.Tensor, ws: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    """Runs the sampling loop in place on latent (fp32 [n_img, latent_channels])."""
    ws = ws if ws is not None else workspace(sample_workspace_size(dims, args), latent.device)
    d = make_dims(dims)
    _check("flux3_sample_fwd", lib.flux3_sample_fwd(ctypes.byref(d), ctypes.byref(dit.w), ctypes.byref(args.a),
                                                    _ptr(latent, torch.float32), _ptr(ws), ws.numel(),
                                                    _stream(stream)))
    return latent


def quantize_rows_fp8(x: torch.Tensor, stream=None):
    """Row-wise e4m3 codes (uint8 [rows, k]) and fp32 scales [rows] of a bf16 matrix."""
    rows, k = x.shape
    q = torch.empty(rows, k, dtype=torch.uint8, device=x.device)
    sc = torch.empty(rows, dtype=torch.float32, device=x.device)
    _check("flux3_quantize_rows_fp8", lib.flux3_quantize_rows_fp8(_ptr(x, torch.bfloat16), rows, k, _ptr(q), _ptr(sc),
                                                                  _stream(stream)))
    return q, sc


class Fp8Weights:
    """A block's weights with the input projection (and with quantize_out the output
    projection too) quantized row-wise to e4m3 on the device (flux3_quantize_rows_fp8);
    norms and biases as given."""

    def __init__(self, w, stream=None, quantize_out: bool = False):
        self.w_in, self.s_in = quantize_rows_fp8(w.w_in, stream)
        self.b_in, self.q_norm, self.k_norm = w.b_in, w.q_norm, w.k_norm
        self.w_out, self.b_out = w.w_out, w.b_out
        self.w_out_q, self.s_out = quantize_rows_fp8(w.w_out, stream) if quantize_out else (None, None)


def _fp8_struct(w: Fp8Weights) -> flux3_block_weights_fp8:
    return flux3_block_weights_fp8(_ptr(w.w_in, torch.uint8), _ptr(w.s_in, torch.float32), _ptr(w.b_in, torch.float32),
                                   _ptr(w.q_norm, torch.float32), _ptr(w.k_norm, torch.float32),
                                   _ptr(w.w_out, torch.bfloat16), _ptr(w.b_out, torch.float32),
                                   _ptr(w.w_out_q, torch.uint8), _ptr(w.s_out, torch.float32))


def in_proj_fp8_fwd(dims, weights: Sequence[Fp8Weights], seg_off: Sequence[int], a8: torch.Tensor, sa: torch.Tensor,
                    rope: torch.Tensor, stream=None):
    """in_proj_fwd on e4m3 codes a8 (uint8 [N, D]) with per-token scales sa (fp32 [N])."""
    n = a8.shape[0]
    D, H, F = dims.width, dims.heads, dims.ffn_hidden
    dev = a8.device
    q = torch.empty(H, n, 128, dtype=torch.bfloat16, device=dev)
    k = torch.empty_like(q)
    ldv = ld_vt(n)
    vt = torch.zeros(H, 128, ldv, dtype=torch.bfloat16, device=dev)
    y = torch.zeros(n, D + F, dtype=torch.bfloat16, device=dev)
    d, s = make_dims(dims), Segments(seg_off, None)
    wa = (flux3_block_weights_fp8 * len(weights))(*[_fp8_struct(w) for w in weights])
    _check("flux3_in_proj_fp8_fwd", lib.flux3_in_proj_fp8_fwd(
        ctypes.byref(d), wa, len(weights), ctypes.byref(s.s), _ptr(a8, torch.uint8), _ptr(sa, torch.float32), n,
        _ptr(rope, torch.float32), _ptr(q), _ptr(k), _ptr(vt), ldv, _ptr(y), _stream(stream)))
    return q, k, vt, y


def block_fp8_workspace_size(dims, n: int) -> int:
    d = make_dims(dims)
    return int(lib.flux3_block_fp8_workspace_size(ctypes.byref(d), n))


def block_fp8_fwd(dims, weights: Fp8Weights, seg_off: Sequence[int], mod: torch.Tensor, x: torch.Tensor,
                  rope: torch.Tensor, x_out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                  stream=None) -> torch.Tensor:
    """The joint block with the e4m3 input projection."""
    n = x.shape[0]
    x_out = x_out if x_out is not None else torch.empty_like(x)
    ws = ws if ws is not None else workspace(block_fp8_workspace_size(dims, n), x.device)
    d, s = make_dims(dims), Segments(seg_off, mod)
    w = _fp8_struct(weights)
    _check("flux3_block_fp8_fwd", lib.flux3_block_fp8_fwd(ctypes.byref(d), ctypes.byref(w), ctypes.byref(s.s),
                                                          _ptr(x, torch.bfloat16), _ptr(x_out, torch.bfloat16), n,
                                                          _ptr(rope, torch.float32), _ptr(ws), ws.numel(),
                                                          _stream(stream)))
    return x_out


def block_bwd_workspace_size(dims, n: int) -> int:
    d = make_dims(dims)
    return int(lib.flux3_block_bwd_workspace_size(ctypes.byref(d), n))


def block_bwd(dims, weights, seg_off: Sequence[int], mod: torch.Tensor, x: torch.Tensor, rope: torch.Tensor,
              dxo: torch.Tensor, ws: Optional[torch.Tensor] = None, out: Optional[dict] = None, stream=None) -> dict:
    """Gradients of the joint block (flux3_block_bwd) for the output gradient dxo (fp32
    [N, D]): a dict of dx, dw_in, db_in, dq_norm, dk_norm, dw_out, db_out, dmod (fp32)."""
    n, D = x.shape
    F = dims.ffn_hidden
    dev = x.device
    if out is None:
        out = {"dx": torch.empty(n, D, device=dev), "dw_in": torch.empty(3 * D + 2 * F, D, device=dev),
               "db_in": torch.empty(3 * D + 2 * F, device=dev), "dq_norm": torch.empty(128, device=dev),
               "dk_norm": torch.empty(128, device=dev), "dw_out": torch.empty(D, D + F, device=dev),
               "db_out": torch.empty(D, device=dev), "dmod": torch.empty(len(seg_off) - 1, 3, D, device=dev)}
    ws = ws if ws is not None else workspace(block_bwd_workspace_size(dims, n), dev)
    d, s = make_dims(dims), Segments(seg_off, mod)
    w = block_weights(weights)
    f = lambda k: _ptr(out[k], torch.float32)
    _check("flux3_block_bwd", lib.flux3_block_bwd(ctypes.byref(d), ctypes.byref(w), ctypes.byref(s.s),
                                                  _ptr(x, torch.bfloat16), _ptr(rope, torch.float32),
                                                  _ptr(dxo, torch.float32), n, f("dx"), f("dw_in"), f("db_in"),
                                                  f("dq_norm"), f("dk_norm"), f("dw_out"), f("db_out"), f("dmod"),
                                                  _ptr(ws), ws.numel(), _stream(stream)))
    return out


def stream_block_bwd(dims, weights: Sequence, seg_off: Sequence[int], mod: torch.Tensor, x: torch.Tensor,
                     rope: torch.Tensor, dxo: torch.Tensor, stream=None) -> dict:
    """Gradients of the stage-1 block (flux3_stream_block_bwd): dx [N, D] and, per stream,
    dw_in, db_in, dq_norm, dk_norm, dw_out, db_out, dmod stacked along a leading axis."""
    n, D = x.shape
    F = dims.ffn_hidden
    g = len(seg_off) - 1
    dev = x.device
    out = {"dx": torch.empty(n, D, device=dev), "dw_in": torch.empty(g, 3 * D + 2 * F, D, device=dev),
           "db_in": torch.empty(g, 3 * D + 2 * F, device=dev), "dq_norm": torch.empty(g, 128, device=dev),
           "dk_norm": torch.empty(g, 128, device=dev), "dw_out": torch.empty(g, D, D + F, device=dev),
           "db_out": torch.empty(g, D, device=dev), "dmod": torch.empty(g, 3, D, device=dev)}
    d, s = make_dims(dims), Segments(seg_off, mod)
    ws = workspace(int(lib.flux3_stream_block_bwd_workspace_size(ctypes.byref(d), ctypes.byref(s.s))), dev)
    wa = _weights_array(weights)
    f = lambda k: _ptr(out[k], torch.float32)
    _check("flux3_stream_block_bwd", lib.flux3_stream_block_bwd(
        ctypes.byref(d), wa, ctypes.byref(s.s), _ptr(x, torch.bfloat16), _ptr(rope, torch.float32),
        _ptr(dxo, torch.float32), n, f("dx"), f("dw_in"), f("db_in"), f("dq_norm"), f("dk_norm"), f("dw_out"),
        f("db_out"), f("dmod"), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def nvfp4_scale_bytes(rows: int, k: int) -> int:
    return int(lib.flux3_nvfp4_scale_bytes(rows, k))


def quantize_rows_nvfp4(x: torch.Tensor, stream=None):
    """NVFP4 codes (uint8 [rows, k / 2], two per byte), tiled block scales (uint8) and fp32
    row scales [rows] of a bf16 matrix."""
    rows, k = x.shape
    q = torch.empty(rows, k // 2, dtype=torch.uint8, device=x.device)
    sf = torch.empty(max(1, nvfp4_scale_bytes(rows, k)), dtype=torch.uint8, device=x.device)
    sc = torch.empty(rows, dtype=torch.float32, device=x.device)
    _check("flux3_quantize_rows_nvfp4", lib.flux3_quantize_rows_nvfp4(_ptr(x, torch.bfloat16), rows, k, _ptr(q), _ptr(sf),
                                                                      _ptr(sc), _stream(stream)))
    return q, sf, sc


class Nvfp4Weights:
    """A block's weights with the input projection (and with quantize_out the output
    projection too) quantized to NVFP4 on the device (flux3_quantize_rows_nvfp4); norms
    and biases as given."""

    def __init__(self, w, stream=None, quantize_out: bool = False):
        self.w_in, self.w_sf, self.s_in = quantize_rows_nvfp4(w.w_in, stream)
        self.b_in, self.q_norm, self.k_norm = w.b_in, w.q_norm, w.k_norm
        self.w_out, self.b_out = w.w_out, w.b_out
        self.w_out_q, self.w_out_sf, self.s_out = (quantize_rows_nvfp4(w.w_out, stream) if quantize_out
                                                   else (None, None, None))


def _nvfp4_struct(w: Nvfp4Weights) -> flux3_block_weights_nvfp4:
    return flux3_block_weights_nvfp4(_ptr(w.w_in, torch.uint8), _ptr(w.w_sf, torch.uint8), _ptr(w.s_in, torch.float32),
                                     _ptr(w.b_in, torch.float32), _ptr(w.q_norm, torch.float32),
                                     _ptr(w.k_norm, torch.float32), _ptr(w.w_out, torch.bfloat16),
                                     _ptr(w.b_out, torch.float32), _ptr(w.w_out_q, torch.uint8),
                                     _ptr(w.w_out_sf, torch.uint8), _ptr(w.s_out, torch.float32))


def in_proj_nvfp4_fwd(dims, weights: Nvfp4Weights, a4: torch.Tensor, a_sf: torch.Tensor, sa: torch.Tensor,
                      rope: torch.Tensor, stream=None):
    """in_proj_fwd (one weight set) on NVFP4 codes a4 (uint8 [N, D / 2]) with tiled block
    scales a_sf and per-token scales sa (fp32 [N])."""
    n = a4.shape[0]
    D, H, F = dims.width, dims.heads, dims.ffn_hidden
    dev = a4.device
    q = torch.empty(H, n, 128, dtype=torch.bfloat16, device=dev)
    k = torch.empty_like(q)
    ldv = ld_vt(n)
    vt = torch.zeros(H, 128, ldv, dtype=torch.bfloat16, device=dev)
    y = torch.zeros(n, D + F, dtype=torch.bfloat16, device=dev)
    d = make_dims(dims)
    w = _nvfp4_struct(weights)
    _check("flux3_in_proj_nvfp4_fwd", lib.flux3_in_proj_nvfp4_fwd(
        ctypes.byref(d), ctypes.byref(w), _ptr(a4, torch.uint8), _ptr(a_sf, torch.uint8), _ptr(sa, torch.float32), n,
        _ptr(rope, torch.float32), _ptr(q), _ptr(k), _ptr(vt), ldv, _ptr(y), _stream(stream)))
    return q, k, vt, y


def block_nvfp4_workspace_size(dims, n: int) -> int:
    d = make_dims(dims)
    return int(lib.flux3_block_nvfp4_workspace_size(ctypes.byref(d), n))


def block_nvfp4_fwd(dims, weights: Nvfp4Weights, seg_off: Sequence[int], mod: torch.Tensor, x: torch.Tensor,
                    rope: torch.Tensor, x_out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    """The joint block with the NVFP4 input projection."""
    n = x.shape[0]
    x_out = x_out if x_out is not None else torch.empty_like(x)
    ws = ws if ws is not None else workspace(block_nvfp4_workspace_size(dims, n), x.device)
    d, s = make_dims(dims), Segments(seg_off, mod)
    w = _nvfp4_struct(weights)
    _check("flux3_block_nvfp4_fwd", lib.flux3_block_nvfp4_fwd(ctypes.byref(d), ctypes.byref(w), ctypes.byref(s.s),
                                                              _ptr(x, torch.bfloat16), _ptr(x_out, torch.bfloat16), n,
                                                              _ptr(rope, torch.float32), _ptr(ws), ws.numel(),
                                                              _stream(stream)))
    return x_out


def selftest_timeout(timeout_us: int) -> None:
    """Runs the bounded-wait diagnostic (a device wait that is never satisfied)."""
    _check("flux3_selftest_timeout", lib.flux3_selftest_timeout(timeout_us))


def device_error(reset: bool = True) -> int:
    flags = ctypes.c_uint32(0)
    st = lib.flux3_device_error(ctypes.byref(flags), 1 if reset else 0)
    if st not in (OK, ERR_TIMEOUT):
        raise Flux3Error("flux3_device_error", st)
    return int(flags.value)


class Profile:
    """Per-launch kernel durations (CUDA events around each launch, on its stream)."""

    def __init__(self, capacity: int = 4096):
        self.capacity = capacity
        self.records: List[tuple] = []

    def __enter__(self):
        _check("flux3_profile_begin", lib.flux3_profile_begin(self.capacity))
        return self

    def __exit__(self, *exc):
        ms = (c_f32 * self.capacity)()
        kinds = (c_i32 * self.capacity)()
        n = c_i32(0)
        _check("flux3_profile_end", lib.flux3_profile_end(ms, kinds, self.capacity, ctypes.byref(n)))
        self.records = [(KERNEL_NAMES.get(kinds[i], str(kinds[i])), float(ms[i])) for i in range(n.value)]
        return False
