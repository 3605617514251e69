"""The allocation-free gemm entry point (indexer_bwd_gemm_noalloc).

Callers that cannot allocate device memory where they run the backward (code
inside an allocator or pool callback, runtimes that own all device memory up
front, launch paths that must not synchronize) use this entry point: it keeps
its scratch in a fixed array inside the library instead of a workspace.  This
file runs last in the suite; it checks that two calls in a row give the same
results as indexer_bwd_gemm, and that shapes beyond the fixed scratch are
refused.  It passes alone in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
import sparse_attention_indexer_bwd_gb300 as ibwd
from gpu_util import TOL_DK, rms_rel, t_bf16, t_f32, t_i32

pytestmark = pytest.mark.gpu


def noalloc_fn():
    lib = ibwd.load()
    fn = lib.indexer_bwd_gemm_noalloc
    p, i = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i, i, i, p]
    fn.restype = i
    return fn


def test_noalloc_matches_workspace_entry_twice():
    fn = noalloc_fn()
    wl = synth.Workload("noalloc", 2, 64, 128, 300, 700, 300, "causal", 31)
    x = synth.make_inputs(wl)
    I = oracle.forward_sparse(x["q"], x["k"], x["w"], x["idx"], wl.S_k).astype(np.float32)
    dI = oracle.score_grad_sparse(I, x["attn"], x["idx"], wl.S_k).astype(np.float32)
    q, k, w, idx, dIt = t_bf16(x["q"]), t_bf16(x["k"]), t_f32(x["w"]), t_i32(x["idx"]), t_f32(dI)
    B, S_q, H, D = x["q"].shape

    def outs():
        dq = torch.full((B, S_q, H, D), float("nan"), device="cuda")
        dw = torch.full((B, S_q, H), float("nan"), device="cuda")
        dk = torch.zeros((B, wl.S_k, D), device="cuda")
        return dq, dw, dk

    ref = outs()
    ibwd.indexer_bwd_gemm(q, k, w, dIt, idx, *ref, dk_mode=ibwd.IBWD_DK_ATOMIC)
    assert ibwd.indexer_bwd_last_device_status() == ibwd.IBWD_OK
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):  # two calls in a row share the library's scratch
        got = outs()
        rc = fn(q.data_ptr(), k.data_ptr(), w.data_ptr(), dIt.data_ptr(), idx.data_ptr(), got[0].data_ptr(),
                got[1].data_ptr(), got[2].data_ptr(), B, S_q, wl.S_k, H, D, wl.topk, stream)
        assert rc == ibwd.IBWD_OK, ibwd.status_string(rc)
        torch.cuda.synchronize()
        # dq and dw come from the same kernel with a single writer: identical;
        # dk is an fp32 atomic sum: equal up to summation order
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
        assert rms_rel(got[2].cpu().numpy(), ref[2].cpu().numpy()) <= TOL_DK * 1e-2


def test_noalloc_refuses_shapes_beyond_its_scratch():
    fn = noalloc_fn()
    d = torch.zeros(1024, device="cuda")
    p = d.data_ptr()
    # B * (S_k + 1) = 2 * 20000 > 32768 key rows: refused before any launch
    assert fn(p, p, p, p, p, p, p, p, 2, 1, 20000, 4, 32, 4, None) == ibwd.IBWD_ERR_UNSUPPORTED
    assert fn(p, p, p, p, p, p, p, p, 1, 1, 1, 65, 32, 4, None) == ibwd.IBWD_ERR_UNSUPPORTED
    assert fn(p + 4, p, p, p, p, p, p, p, 1, 1, 8, 4, 32, 4, None) == ibwd.IBWD_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.count_nonzero(d) == 0
