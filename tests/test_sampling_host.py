"""The sampling loop's host-side pieces through the C-ABI, on CPU (no GPU needed): the
noise-level schedule against the oracle and the pages' 44-of-50 statement."""
import json
import os

import numpy as np
import pytest

from oracle import sampling as S


@pytest.fixture(scope="module")
def B():
    from flow_matching_image_flux3_b300 import build
    build.build()
    from flow_matching_image_flux3_b300 import binding
    return binding


def test_sigma_schedule_matches_oracle(B):
    for n, alpha in ((50, 6.93), (16, 6.93), (3, 2.0), (1, 1.0)):
        got = np.array(B.sigma_schedule(n, alpha), dtype=np.float64)
        # the library takes alpha as fp32; the oracle gets the same value
        ref = S.sigma_schedule(n, float(np.float32(alpha)))
        np.testing.assert_allclose(got, ref, rtol=2e-7, atol=1e-9)
        assert got[0] == 1.0 and got[-1] == 0.0


def test_sigma_schedule_has_44_of_50_above_half(B):
    facts = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))
    s = B.sigma_schedule(facts["steps_base"]["value"], facts["time_shift"]["value"])
    assert sum(1 for x in s[:-1] if x > 0.5) == facts["steps_above_half_sigma"]["value"]


def test_sigma_schedule_argument_checks(B):
    for n, alpha in ((0, 6.93), (-1, 6.93), (50, 0.0), (50, -1.0), (50, float("inf"))):
        with pytest.raises(B.Flux3Error):
            B.sigma_schedule(n, alpha)
