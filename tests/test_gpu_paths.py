"""The two gemm kernels behind one call.

Atomic sparse calls without options are served either by the blocked kernel
(four query rows against the union of their keys) or by the per-row kernel,
chosen on the device from a sample of the call's blocks (select_kernel's
cost model).  The test-only environment variable IBWD_TEST_GEMM_PATH imposes
either one: both must match the oracle, and the call left to choose must
give, bit for bit, the dq and dw of one of them (both kernels' dq and dw are
reproducible run to run).
"""
import numpy as np
import pytest

import synth
import sparse_attention_indexer_bwd_gb300 as ibwd
from gpu_util import TOL_DK, assert_close, case_inputs, gemm_path, gpu_all, oracle_all, rms_rel

pytestmark = pytest.mark.gpu

W = synth.Workload
CASES = [
    synth.WORKLOADS["tiny"],
    W("multi_tile_ragged", 2, 64, 128, 300, 700, 300, "causal", 11),
    W("window_small", 1, 64, 128, 384, 512, 256, "window", 12),
    W("odd_shapes", 1, 7, 40, 131, 97, 53, "causal", 13),
    W("uniform_small", 1, 16, 64, 130, 512, 256, "uniform", 17),
    W("uniform_sparse", 1, 32, 128, 256, 4096, 128, "uniform", 18),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_both_gemm_kernels_match_the_oracle_and_the_choice_is_one_of_them(wl):
    x = case_inputs(wl)
    ref = oracle_all(wl, x)
    got = {}
    for path in ("rows", "blocked"):
        with gemm_path(path):
            dI, dq, dw, dk = gpu_all(wl, x, dk_mode=ibwd.IBWD_DK_ATOMIC)
        assert_close(dq, dw, dk, ref[1:], tag=f"{wl.name} {path}")
        got[path] = (dq, dw, dk)
    # the two kernels sum in different orders: close, not bitwise
    assert rms_rel(got["rows"][2], got["blocked"][2]) <= TOL_DK
    _, dq, dw, dk = gpu_all(wl, x, dk_mode=ibwd.IBWD_DK_ATOMIC)
    chosen = [p for p in got if np.array_equal(got[p][0], dq) and np.array_equal(got[p][1], dw)]
    assert len(chosen) == 1, "the call's dq and dw are those of exactly one kernel"


def test_the_choice_follows_the_key_overlap():
    # uniform top-384 of 4096 keys: four rows share few keys, the per-row
    # kernel is cheaper; every causal key selected (top-k above S_k): four
    # rows share nearly all theirs, the blocked kernel is
    picks = {}
    for wl in (W("low_overlap", 1, 16, 64, 512, 4096, 384, "uniform", 19),
               W("high_overlap", 1, 16, 64, 512, 512, 512, "causal", 20)):
        x = case_inputs(wl)
        outs = {}
        for path in ("rows", "blocked"):
            with gemm_path(path):
                outs[path] = gpu_all(wl, x, dk_mode=ibwd.IBWD_DK_ATOMIC)[1]
        dq = gpu_all(wl, x, dk_mode=ibwd.IBWD_DK_ATOMIC)[1]
        picks[wl.name] = [p for p in outs if np.array_equal(outs[p], dq)]
    assert picks["low_overlap"] == ["rows"]
    assert picks["high_overlap"] == ["blocked"]
