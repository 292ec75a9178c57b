"""Host-side checks of libflux3.so: it loads without a GPU, exports every function that
include/flux3.h declares, and rejects bad arguments before launching anything."""
import ctypes
import os
import re

import pytest

from flow_matching_image_flux3_b300 import build as fbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    fbuild.build()
    from flow_matching_image_flux3_b300 import binding
    return binding


def header_functions():
    src = open(os.path.join(ROOT, "include", "flux3.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(flux3_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(B):
    names = header_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(B.lib, n), n
    assert set(names) == set(B.EXPORTED)


def test_status_strings_and_version(B):
    for s in range(6):
        assert B.lib.flux3_status_string(s)
    assert b"sm_103a" in B.lib.flux3_version()


def _dims(B, **kw):
    d = dict(width=256, heads=2, head_dim=128, ffn_hidden=768, ln_eps=1e-6, rms_eps=1e-6, rope_theta=1e4)
    d.update(kw)
    return B.flux3_dims(**d)


FAKE = 0x7f0000000000  # a 256-byte aligned address; nothing is launched in these tests


def _weights(B, **kw):
    w = dict(w_in=FAKE, b_in=None, q_norm=FAKE, k_norm=FAKE, w_out=FAKE, b_out=None)
    w.update(kw)
    return B.flux3_block_weights(**w)


def _segs(B, off, mod=FAKE):
    arr = (ctypes.c_int32 * len(off))(*off)
    return B.flux3_segments(len(off) - 1, ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32)), mod), arr


def _block(B, d, w, segs, n, ws_bytes=None, x=FAKE, x_out=FAKE, rope=FAKE, ws=FAKE):
    if ws_bytes is None:
        ws_bytes = B.lib.flux3_block_workspace_size(ctypes.byref(d), n)
    return B.lib.flux3_block_fwd(ctypes.byref(d), ctypes.byref(w) if w is not None else None,
                                 ctypes.byref(segs) if segs is not None else None, x, x_out, n, rope, ws, ws_bytes, None)


def test_dims_validation(B):
    w = _weights(B)
    s, _keep = _segs(B, [0, 64, 144])
    assert _block(B, _dims(B, head_dim=64, width=128), w, s, 144, ws_bytes=1 << 40) == B.ERR_UNSUPPORTED
    assert _block(B, _dims(B, heads=3, width=384), w, s, 144, ws_bytes=1 << 40) == B.ERR_UNSUPPORTED
    assert _block(B, _dims(B, ffn_hidden=100), w, s, 144, ws_bytes=1 << 40) == B.ERR_UNSUPPORTED
    assert _block(B, _dims(B, width=300), w, s, 144, ws_bytes=1 << 40) == B.ERR_INVALID_ARG
    assert _block(B, _dims(B, ln_eps=0.0), w, s, 144, ws_bytes=1 << 40) == B.ERR_INVALID_ARG
    assert _block(B, _dims(B, rope_theta=-1.0), w, s, 144, ws_bytes=1 << 40) == B.ERR_INVALID_ARG
    assert B.lib.flux3_block_fwd(None, ctypes.byref(w), ctypes.byref(s), FAKE, FAKE, 144, FAKE, FAKE, 1 << 40, None) \
        == B.ERR_INVALID_ARG


def test_segment_validation(B):
    d, w = _dims(B), _weights(B)
    for off in ([0, 64, 143], [1, 64, 144], [0, 100, 64, 144], [0] + list(range(1, 18)) + [144]):
        s, _keep = _segs(B, off)
        assert _block(B, d, w, s, 144, ws_bytes=1 << 40) == B.ERR_INVALID_ARG, off
    s, _keep = _segs(B, [0, 64, 144], mod=None)
    assert _block(B, d, w, s, 144, ws_bytes=1 << 40) == B.ERR_INVALID_ARG
    assert _block(B, d, w, None, 144, ws_bytes=1 << 40) == B.ERR_INVALID_ARG


def test_pointer_validation(B):
    d = _dims(B)
    s, _keep = _segs(B, [0, 64, 144])
    assert _block(B, d, _weights(B, w_in=None), s, 144) == B.ERR_INVALID_ARG
    assert _block(B, d, _weights(B, w_out=FAKE + 8), s, 144) == B.ERR_INVALID_ARG
    assert _block(B, d, _weights(B, q_norm=None), s, 144) == B.ERR_INVALID_ARG
    assert _block(B, d, _weights(B), s, 144, x=FAKE + 2) == B.ERR_INVALID_ARG
    assert _block(B, d, _weights(B), s, 144, x_out=None) == B.ERR_INVALID_ARG
    assert _block(B, d, _weights(B), s, 144, rope=None) == B.ERR_INVALID_ARG


def test_workspace_validation(B):
    d, w = _dims(B), _weights(B)
    s, _keep = _segs(B, [0, 64, 144])
    need = B.lib.flux3_block_workspace_size(ctypes.byref(d), 144)
    # a (144x256) + q + k + vt (2x128x144) + y (144x1024), bf16, each rounded up to 256 B
    assert need == sum((b + 255) // 256 * 256 for b in (144 * 256 * 2, 2 * 144 * 128 * 2, 2 * 144 * 128 * 2,
                                                          2 * 128 * 144 * 2, 144 * 1024 * 2))
    assert _block(B, d, w, s, 144, ws_bytes=need - 1) == B.ERR_WORKSPACE
    assert _block(B, d, w, s, 144, ws=None) == B.ERR_WORKSPACE
    assert _block(B, d, w, s, 144, ws=FAKE + 16) == B.ERR_WORKSPACE
    assert B.lib.flux3_block_workspace_size(ctypes.byref(_dims(B, head_dim=64, width=128)), 144) == 0


def test_empty_sequence_is_a_noop(B):
    d, w = _dims(B), _weights(B)
    s, _keep = _segs(B, [0, 0])
    assert _block(B, d, w, s, 0, ws_bytes=0, ws=None) == B.OK
    assert B.lib.flux3_rope_build(ctypes.byref(d), None, 0, None, None) == B.OK
    assert B.lib.flux3_attn_fwd(ctypes.byref(d), None, None, None, 8, 0, None, 1, None, 256, 0, None) == B.OK


def test_attention_argument_checks(B):
    d = _dims(B)
    bad_ld = B.lib.flux3_attn_fwd(ctypes.byref(d), FAKE, FAKE, FAKE, 100, 100, None, 1, FAKE, 256, 0, None)
    assert bad_ld == B.ERR_INVALID_ARG                       # ld_vt % 8 != 0
    short = B.lib.flux3_attn_fwd(ctypes.byref(d), FAKE, FAKE, FAKE, 96, 100, None, 1, FAKE, 256, 0, None)
    assert short == B.ERR_INVALID_ARG                        # ld_vt < N
    narrow = B.lib.flux3_attn_fwd(ctypes.byref(d), FAKE, FAKE, FAKE, 104, 100, None, 1, FAKE, 128, 0, None)
    assert narrow == B.ERR_INVALID_ARG                       # ld_out < width
    off = (ctypes.c_int32 * 3)(0, 50, 99)
    assert B.lib.flux3_attn_fwd(ctypes.byref(d), FAKE, FAKE, FAKE, 104, 100, off, 2, FAKE, 256, 0, None) \
        == B.ERR_INVALID_ARG                                 # offsets do not end at N


def test_dit_argument_checks(B):
    d = _dims(B)
    w = B.flux3_dit_weights(2, 0, 0, None, None, FAKE, None, 128)
    m = B.flux3_dit_mod(None, None, FAKE)
    args = (ctypes.byref(d), ctypes.byref(w), ctypes.byref(m), FAKE, 64, 8, 80, FAKE, FAKE, FAKE, 1 << 40, None)
    assert B.lib.flux3_dit_fwd(*args) == B.ERR_INVALID_ARG   # n_ref > 0 needs three streams
    w.out_channels = 100
    args = (ctypes.byref(d), ctypes.byref(w), ctypes.byref(m), FAKE, 64, 0, 80, FAKE, FAKE, FAKE, 1 << 40, None)
    assert B.lib.flux3_dit_fwd(*args) == B.ERR_UNSUPPORTED
    w.out_channels = 128
    args = (ctypes.byref(d), ctypes.byref(w), ctypes.byref(m), FAKE, 64, 0, 80, FAKE, FAKE, FAKE, 1024, None)
    assert B.lib.flux3_dit_fwd(*args) == B.ERR_WORKSPACE


def test_final_and_euler_argument_checks(B):
    d = _dims(B)
    assert B.lib.flux3_final_fwd(ctypes.byref(d), FAKE, None, 64, FAKE, FAKE, 10, FAKE, FAKE, 1 << 20, None) \
        == B.ERR_UNSUPPORTED
    assert B.lib.flux3_final_fwd(ctypes.byref(d), FAKE, None, 128, FAKE, FAKE, 10, FAKE, FAKE, 100, None) \
        == B.ERR_WORKSPACE
    assert B.lib.flux3_euler_step(None, None, 10, 1.0, 0.5, None) == B.ERR_INVALID_ARG
    assert B.lib.flux3_euler_step(None, None, 0, 1.0, 0.5, None) == B.OK


def test_nvfp4_argument_checks(B):
    FAKE16 = 1 << 20
    assert B.lib.flux3_nvfp4_scale_bytes(300, 3072) == 512 * 192      # rows padded to 256
    assert B.lib.flux3_nvfp4_scale_bytes(256, 3072) == 256 * 192
    assert B.lib.flux3_nvfp4_scale_bytes(1, 100) == 0                 # k % 64 != 0
    assert B.lib.flux3_quantize_rows_nvfp4(FAKE16, 4, 320, FAKE16, FAKE16, FAKE16, None) == B.ERR_UNSUPPORTED
    assert B.lib.flux3_quantize_rows_nvfp4(FAKE16 + 8, 4, 256, FAKE16, FAKE16, FAKE16, None) == B.ERR_INVALID_ARG
    assert B.lib.flux3_quantize_rows_nvfp4(None, 0, 256, None, None, None, None) == B.OK
    d = _dims(B)
    assert B.lib.flux3_in_proj_nvfp4_fwd(ctypes.byref(d), None, None, None, None, 4, None, None, None, None, 8, None,
                                         None) == B.ERR_INVALID_ARG     # no weights
    w = B.flux3_block_weights_nvfp4(FAKE16, FAKE16, FAKE16, None, FAKE16, FAKE16, FAKE16, None)
    assert B.lib.flux3_in_proj_nvfp4_fwd(ctypes.byref(d), ctypes.byref(w), FAKE16, FAKE16, FAKE16, 100, FAKE16,
                                         FAKE16, FAKE16, FAKE16, 96, FAKE16, None) == B.ERR_INVALID_ARG   # ld_vt < N
    assert B.lib.flux3_block_nvfp4_workspace_size(ctypes.byref(d), 144) > B.lib.flux3_block_workspace_size(
        ctypes.byref(d), 144)


def test_backward_argument_checks(B):
    d = _dims(B)
    off = (ctypes.c_int32 * 3)(0, 64, 144)
    segs = B.flux3_segments(2, ctypes.cast(off, ctypes.POINTER(ctypes.c_int32)), FAKE)
    w = B.flux3_block_weights(FAKE, None, FAKE, FAKE, FAKE, None)
    outs = [FAKE] * 8
    assert B.lib.flux3_block_bwd_workspace_size(ctypes.byref(d), 144) > B.lib.flux3_block_workspace_size(
        ctypes.byref(d), 144)
    # no workspace
    assert B.lib.flux3_block_bwd(ctypes.byref(d), ctypes.byref(w), ctypes.byref(segs), FAKE, FAKE, FAKE, 144, *outs,
                                 None, 0, None) == B.ERR_WORKSPACE
    # a missing output
    assert B.lib.flux3_block_bwd(ctypes.byref(d), ctypes.byref(w), ctypes.byref(segs), FAKE, FAKE, FAKE, 144,
                                 *([None] + outs[1:]), FAKE, 1 << 40, None) == B.ERR_INVALID_ARG
    # segments that do not end at N
    assert B.lib.flux3_block_bwd(ctypes.byref(d), ctypes.byref(w), ctypes.byref(segs), FAKE, FAKE, FAKE, 150, *outs,
                                 FAKE, 1 << 40, None) == B.ERR_INVALID_ARG
    # nothing to do
    e = (ctypes.c_int32 * 2)(0, 0)
    s0 = B.flux3_segments(1, ctypes.cast(e, ctypes.POINTER(ctypes.c_int32)), FAKE)
    assert B.lib.flux3_block_bwd(ctypes.byref(d), ctypes.byref(w), ctypes.byref(s0), None, None, None, 0,
                                 *([None] * 8), None, 0, None) == B.OK
    # the per-stream form needs a weight set per stream and the longest stream's workspace
    assert B.lib.flux3_stream_block_bwd_workspace_size(ctypes.byref(d), ctypes.byref(segs)) == \
        B.lib.flux3_block_bwd_workspace_size(ctypes.byref(d), 80)
    ws2 = (B.flux3_block_weights * 2)(w, B.flux3_block_weights(None, None, FAKE, FAKE, FAKE, None))
    assert B.lib.flux3_stream_block_bwd(ctypes.byref(d), ws2, ctypes.byref(segs), FAKE, FAKE, FAKE, 144, *outs, FAKE,
                                        1 << 40, None) == B.ERR_INVALID_ARG
