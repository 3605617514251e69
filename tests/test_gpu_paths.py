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
    W("short_rows_b2", 2, 64, 128, 200, 300, 96, "causal", 19),  # rows of one tile, two batches
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


def test_alternating_choices_on_one_workspace():
    # Consecutive calls on one workspace whose ids pick different kernels:
    # every kernel that reads the choice must read this call's, not the one
    # an earlier call left in the workspace.
    import torch
    from gpu_util import dev, gpu_gemm, t_bf16, t_f32, t_i32
    import oracle
    wl = W("alternating", 1, 16, 64, 256, 4096, 384, "uniform", 22)
    x = case_inputs(wl)
    t = np.arange(wl.S_q)[:, None]
    window = ((t + np.arange(wl.topk)[None, :]) % wl.S_k).astype(np.int32)[None]  # neighbours share keys
    cases = {}
    for name, ids in (("uniform", x["idx"]), ("window", window)):
        I = oracle.forward_sparse(x["q"], x["k"], x["w"], ids, wl.S_k)
        dI = oracle.score_grad_sparse(I, x["attn"], ids, wl.S_k)
        cases[name] = (ids, dI.astype(np.float32), oracle.gemm_sparse(x["q"], x["k"], x["w"], dI, ids, wl.S_k))
    ws = torch.empty(ibwd.indexer_bwd_gemm_workspace_size(1, wl.S_q, wl.S_k, wl.H, wl.D, wl.topk, 0),
                     dtype=torch.uint8, device=dev())
    q, k, w = t_bf16(x["q"]), t_bf16(x["k"]), t_f32(x["w"])
    for name in ("uniform", "window", "uniform", "window", "window", "uniform"):
        ids, dI, ref = cases[name]
        dq = torch.full((1, wl.S_q, wl.H, wl.D), float("nan"), device=dev())
        dw = torch.full((1, wl.S_q, wl.H), float("nan"), device=dev())
        dk = torch.zeros((1, wl.S_k, wl.D), device=dev())
        ibwd.indexer_bwd_gemm(q, k, w, t_f32(dI), t_i32(ids), dq, dw, dk, ibwd.IBWD_DK_ATOMIC, ws)
        assert ibwd.indexer_bwd_last_device_status() == ibwd.IBWD_OK
        assert_close(dq.cpu().numpy(), dw.cpu().numpy(), dk.cpu().numpy(), ref, tag=name)
    # the two id sets do take different kernels
    picks = {}
    for name in ("uniform", "window"):
        ids, dI, _ = cases[name]
        outs = {}
        for path in ("rows", "blocked"):
            with gemm_path(path):
                outs[path] = gpu_gemm(wl, x, dI, idx=ids)[0]
        dq = gpu_gemm(wl, x, dI, idx=ids)[0]
        picks[name] = [p for p in outs if np.array_equal(outs[p], dq)]
    assert picks == {"uniform": ["rows"], "window": ["blocked"]}
