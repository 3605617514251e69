"""The gemm kernel's results do not depend on its pipeline depths.

The library runs the kernel with two K-tile stages and four tile-record slots;
a second instance built with one stage and two slots (selected by the
test-only environment variable IBWD_TEST_SHALLOW_PIPELINE=1) makes every
producer wait for its consumers far more often, so an ordering mistake (a
slot released or rewritten too early, a missed wait) changes its results.
Both instances do the same arithmetic in the same order, so dq and dw agree
bit for bit in both dK modes and dk in the deterministic mode; in the atomic
mode dk agrees within the parity tolerance (its additions race).
"""
import os

import numpy as np
import pytest

import synth
import sparse_attention_indexer_bwd_gb300 as ibwd
from gpu_util import TOL_DK, assert_close, case_inputs, gemm_path, gpu_gemm, oracle_all, rms_rel

pytestmark = pytest.mark.gpu

W = synth.Workload
CASES = [
    W("multi_tile_ragged", 2, 64, 128, 300, 700, 300, "causal", 11),
    W("window_small", 1, 64, 128, 384, 512, 256, "window", 12),
    W("dense_small", 1, 64, 128, 200, 200, 0, "dense", 14),
]


def shallow(fn, *a, **kw):
    os.environ["IBWD_TEST_SHALLOW_PIPELINE"] = "1"
    try:
        return fn(*a, **kw)
    finally:
        del os.environ["IBWD_TEST_SHALLOW_PIPELINE"]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("mode", [ibwd.IBWD_DK_ATOMIC, ibwd.IBWD_DK_DETERMINISTIC])
def test_shallow_pipeline_is_bitwise_the_production_one(wl, mode):
    x = case_inputs(wl)
    ref = oracle_all(wl, x)
    dI = ref[0].astype(np.float32)
    with gemm_path("blocked"):
        deep = gpu_gemm(wl, x, dI, dk_mode=mode)
        flat = shallow(gpu_gemm, wl, x, dI, dk_mode=mode)
    np.testing.assert_array_equal(flat[0].view(np.int32), deep[0].view(np.int32))
    np.testing.assert_array_equal(flat[1].view(np.int32), deep[1].view(np.int32))
    if mode == ibwd.IBWD_DK_DETERMINISTIC:
        np.testing.assert_array_equal(flat[2].view(np.int32), deep[2].view(np.int32))
    else:
        assert rms_rel(flat[2], deep[2]) <= TOL_DK
    assert_close(*flat, ref[1:], tag=f"shallow {wl.name}")  # and against the oracle
