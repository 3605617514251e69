"""The allocation-free gemm entry point (indexer_bwd_gemm_noalloc).

Callers that cannot allocate device memory where they run the backward (code
inside an allocator or pool callback, runtimes that own all device memory up
front, launch paths that must not synchronize) use this entry point: it keeps
its scratch in a fixed array inside the library instead of a workspace.  This
file runs last in the suite; it checks two calls in a row against the regular
entry point (indexer_bwd_gemm) and the oracle, a shape at the exact scratch
limit, the entry point's own status word, and that shapes beyond the fixed
scratch (including ones whose size would wrap around) are refused.  It passes
alone in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
import sparse_attention_indexer_bwd_gb300 as ibwd
from gpu_util import TOL_DK, TOL_DQ, TOL_DW, max_rel, rms_rel, t_bf16, t_f32, t_i32

pytestmark = pytest.mark.gpu


def lib_fns():
    lib = ibwd.load()
    fn = lib.indexer_bwd_gemm_noalloc
    p, i = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i, i, i, p]
    fn.restype = i
    st = lib.indexer_bwd_gemm_noalloc_status
    st.argtypes = [p]
    st.restype = i
    setup = lib.indexer_bwd_gemm_noalloc_setup
    setup.argtypes = []
    setup.restype = i
    return fn, st, setup


def run_case(wl, idx=None):
    fn, status, setup = lib_fns()
    assert setup() == ibwd.IBWD_OK
    x = synth.make_inputs(wl)
    if idx is not None:
        x["idx"] = idx
    I = oracle.forward_sparse(x["q"], x["k"], x["w"], x["idx"], wl.S_k).astype(np.float32)
    dI = oracle.score_grad_sparse(I, x["attn"], x["idx"], wl.S_k).astype(np.float32)
    ref = oracle.gemm_sparse(x["q"], x["k"], x["w"], dI.astype(np.float64), x["idx"], wl.S_k)
    q, k, w, ids, dIt = t_bf16(x["q"]), t_bf16(x["k"]), t_f32(x["w"]), t_i32(x["idx"]), t_f32(dI)
    B, S_q, H, D = x["q"].shape

    def outs():
        dq = torch.full((B, S_q, H, D), float("nan"), device="cuda")
        dw = torch.full((B, S_q, H), float("nan"), device="cuda")
        dk = torch.zeros((B, wl.S_k, D), device="cuda")
        return dq, dw, dk

    reg = outs()
    ibwd.indexer_bwd_gemm(q, k, w, dIt, ids, *reg, dk_mode=ibwd.IBWD_DK_ATOMIC)
    assert ibwd.indexer_bwd_last_device_status() == ibwd.IBWD_OK
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):  # two calls in a row share the library's scratch
        got = outs()
        rc = fn(q.data_ptr(), k.data_ptr(), w.data_ptr(), dIt.data_ptr(), ids.data_ptr(), got[0].data_ptr(),
                got[1].data_ptr(), got[2].data_ptr(), B, S_q, wl.S_k, H, D, wl.topk, stream)
        assert rc == ibwd.IBWD_OK, ibwd.status_string(rc)
        assert status(stream) == ibwd.IBWD_OK  # its own status word: no wait timed out
        g = [t.cpu().numpy() for t in got]
        r = [t.cpu().numpy() for t in reg]
        # against the regular entry point (another kernel: equal within the tolerance)
        assert max_rel(g[0], r[0]) <= TOL_DQ and max_rel(g[1], r[1]) <= TOL_DW
        assert rms_rel(g[2], r[2]) <= TOL_DK
        # and against the oracle directly
        assert max_rel(g[0], ref[0]) <= TOL_DQ and max_rel(g[1], ref[1]) <= TOL_DW
        assert rms_rel(g[2], ref[2]) <= TOL_DK


def test_noalloc_matches_workspace_entry_twice():
    run_case(synth.Workload("noalloc", 2, 64, 128, 300, 700, 300, "causal", 31))


def test_noalloc_at_the_exact_scratch_limit():
    # B * (S_k + 1) = 32768 key rows fill the scratch; the ids reach the last key
    wl = synth.Workload("noalloc_limit", 1, 8, 64, 8, 32767, 16, "uniform", 32)
    idx = synth.make_inputs(wl)["idx"].copy()
    idx[0, :, 0] = wl.S_k - 1
    idx[0, 3, 5] = -1
    run_case(wl, idx)


def test_noalloc_refuses_shapes_beyond_its_scratch():
    fn, status, _ = lib_fns()
    d = torch.zeros(1024, device="cuda")
    p = d.data_ptr()
    # B * (S_k + 1) = 32769 > 32768 key rows: refused before any launch
    assert fn(p, p, p, p, p, p, p, p, 1, 1, 32768, 4, 32, 4, None) == ibwd.IBWD_ERR_UNSUPPORTED
    assert fn(p, p, p, p, p, p, p, p, 2, 1, 20000, 4, 32, 4, None) == ibwd.IBWD_ERR_UNSUPPORTED
    # a row count whose byte size would wrap around in 64-bit arithmetic
    assert fn(p, p, p, p, p, p, p, p, 1 << 28, 1, (1 << 28) - 1, 4, 32, 1, None) == ibwd.IBWD_ERR_UNSUPPORTED
    assert fn(p, p, p, p, p, p, p, p, 1, 1, 2147483647, 4, 32, 4, None) == ibwd.IBWD_ERR_UNSUPPORTED
    assert fn(p, p, p, p, p, p, p, p, 1, 1, 1, 65, 32, 4, None) == ibwd.IBWD_ERR_UNSUPPORTED
    assert fn(p + 4, p, p, p, p, p, p, p, 1, 1, 8, 4, 32, 4, None) == ibwd.IBWD_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.count_nonzero(d) == 0
    assert status(None) == ibwd.IBWD_OK
