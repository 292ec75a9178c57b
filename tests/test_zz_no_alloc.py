"""flux3_block_fwd_static: the joint block for callers that cannot allocate device memory
(a host that gives all device memory to its own pool, a loop that cannot afford the
device synchronisation of cudaMalloc, a small C host with no allocator of its own).  Its
scratch is the library's static device array instead of a caller workspace.

Checked through the C-ABI against flux3_block_fwd (the workspace entry point) on two
calls in a row of different sizes, so the second call runs over the first one's leftover
scratch.  This file is collected last, and passes alone or after the other tests."""
import ctypes

import numpy as np
import pytest
import torch

from flow_matching_image_flux3_b300 import synth
from tests.common import REL_L2, MAX_ABS, assert_close, f64, DevWeights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from flow_matching_image_flux3_b300 import build
    build.build()
    from flow_matching_image_flux3_b300 import binding
    return binding


def _full_width_case(n_img_grid, n_txt, seed):
    return synth.make_case(synth.FULL, [synth.Stream("image", n_img_grid[0] * n_img_grid[1], n_img_grid),
                                        synth.text_stream(n_txt)], seed=seed, stage=2, bias=True)


def _both(B, case):
    w = DevWeights(case.weights[0])
    x, mod = case.x.cuda(), case.mod.cuda()
    rope = B.rope_build(case.dims, case.pos.cuda())
    ref = B.block_fwd(case.dims, w, case.seg_off, mod, x, rope)
    got = B.block_fwd_static(case.dims, w, case.seg_off, mod, x, rope)
    torch.cuda.synchronize()
    return got, ref


def test_static_scratch_block_matches_workspace_block(B):
    # call 1: full width, 20x30 image + 160 text = 760 tokens (about 36 MB of scratch)
    c1 = _full_width_case((20, 30), 160, seed=81)
    assert B.block_workspace_size(c1.dims, c1.n) <= B.STATIC_SCRATCH_BYTES
    got1, ref1 = _both(B, c1)
    assert_close("static scratch, call 1", f64(got1), f64(ref1), rl2=REL_L2, ma=MAX_ABS)
    # call 2, right after: a smaller, differently shaped block over the stale scratch
    c2 = synth.config(0, bias=True)
    got2, ref2 = _both(B, c2)
    assert_close("static scratch, call 2", f64(got2), f64(ref2), rl2=REL_L2, ma=MAX_ABS)
    assert B.device_error() == 0


def test_static_scratch_rejects_oversize(B):
    c = _full_width_case((40, 40), 160, seed=82)   # 1,760 tokens need more than 64 MiB
    assert B.block_workspace_size(c.dims, c.n) > B.STATIC_SCRATCH_BYTES
    w = DevWeights(c.weights[0])
    with pytest.raises(B.Flux3Error) as e:
        B.block_fwd_static(c.dims, w, c.seg_off, c.mod.cuda(), c.x.cuda(),
                           torch.empty(c.n, 64, 2, device="cuda"))
    assert e.value.status == B.ERR_WORKSPACE
