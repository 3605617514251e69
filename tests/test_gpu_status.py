"""The device status words: a bounded wait that runs out and an operand
outside the fp16 range are reported after the call, and the library stays
usable afterwards.

The test-only environment variable IBWD_TEST_TIMEOUT_NS makes the gemm
kernel's record producer publish nothing, so every other role waits on a
pipeline barrier phase that nothing completes, and shortens the roles' wait
limit to the given ns (1 ms here): the waits run out without any fault, and
the drains of copies and MMAs already issued keep their full limit, so the
kernel exits cleanly.
"""
import os

import numpy as np
import pytest
import torch

import synth
import sparse_attention_indexer_bwd_gb300 as ibwd
import oracle
from gpu_util import assert_close, case_inputs, gemm_path, gpu_gemm, t_bf16, t_f32, t_i32

pytestmark = pytest.mark.gpu

W = synth.Workload
DET = ibwd.IBWD_DK_DETERMINISTIC
ATOM = ibwd.IBWD_DK_ATOMIC


def inputs(wl):
    """Host inputs, the fp32 dI of the oracle and the oracle's gemm on it."""
    x = case_inputs(wl)
    dI = oracle.score_grad_sparse(x["I"], x["attn"], x["idx"], wl.S_k).astype(np.float32)
    ref = oracle.gemm_sparse(x["q"], x["k"], x["w"], dI.astype(np.float64), x["idx"], wl.S_k)
    return x, dI, ref


def raw_gemm(wl, x, dI, mode, q=None, k=None):
    """One gemm call; returns the device status read after it."""
    qt = t_bf16(x["q"]) if q is None else q
    kt = t_bf16(x["k"]) if k is None else k
    B, S_q, H, D = x["q"].shape
    dq = torch.zeros((B, S_q, H, D), device="cuda")
    dw = torch.zeros((B, S_q, H), device="cuda")
    dk = torch.zeros((B, wl.S_k, D), device="cuda")
    ibwd.indexer_bwd_gemm(qt, kt, t_f32(x["w"]), t_f32(dI), t_i32(x["idx"]), dq, dw, dk, mode)
    return ibwd.indexer_bwd_last_device_status()


@pytest.mark.parametrize("mode", [ATOM, DET])
def test_role_wait_timeout_is_reported_and_the_next_call_is_correct(mode):
    wl = W("timeout", 2, 64, 64, 300, 700, 300, "causal", 41)
    x, dI, ref = inputs(wl)
    os.environ["IBWD_TEST_TIMEOUT_NS"] = "1000000"
    try:
        with gemm_path("blocked"):  # the switch stalls the blocked kernel's record producer
            st = raw_gemm(wl, x, dI, mode)
    finally:
        del os.environ["IBWD_TEST_TIMEOUT_NS"]
    assert st == ibwd.IBWD_ERR_TIMEOUT, ibwd.status_string(st)
    # the reader cleared the word; the context is usable and the results right
    assert ibwd.indexer_bwd_last_device_status() == ibwd.IBWD_OK
    dq, dw, dk = gpu_gemm(wl, x, dI, dk_mode=mode)
    assert_close(dq, dw, dk, ref, "after timeout")


def bf16_tensor_with(a, pos, value):
    t = t_bf16(a)
    t.view(-1)[pos] = torch.tensor(value, dtype=torch.bfloat16)
    return t


@pytest.mark.parametrize("which", ["q", "k"])
def test_operand_beyond_fp16_range_is_reported(which):
    wl = W("range", 1, 16, 64, 130, 200, 64, "causal", 42)
    x, dI, _ = inputs(wl)
    if which == "q":
        q = bf16_tensor_with(x["q"], 5 * 64 * 64 + 3, 1.0e5)  # bf16 99840 > 65504
        st = raw_gemm(wl, x, dI, ATOM, q=q)
    else:
        k = bf16_tensor_with(x["k"], 77 * 64 + 10, -7.0e4)
        st = raw_gemm(wl, x, dI, ATOM, k=k)
    assert st == ibwd.IBWD_ERR_RANGE, ibwd.status_string(st)
    assert ibwd.indexer_bwd_last_device_status() == ibwd.IBWD_OK
    # the largest bf16 below the fp16 limit passes
    q = bf16_tensor_with(x["q"], 3, 65280.0)
    assert raw_gemm(wl, x, dI, ATOM, q=q) == ibwd.IBWD_OK


def test_noalloc_status_reports_the_range_bit():
    import ctypes
    lib = ibwd.load()
    fn = lib.indexer_bwd_gemm_noalloc
    p, i = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i, i, i, p]
    fn.restype = i
    st = lib.indexer_bwd_gemm_noalloc_status
    st.argtypes = [p]
    st.restype = i
    wl = W("range_na", 1, 16, 64, 130, 200, 64, "causal", 43)
    x, dI, _ = inputs(wl)
    q = bf16_tensor_with(x["q"], 100, float("inf"))
    k, w, ids, dIt = t_bf16(x["k"]), t_f32(x["w"]), t_i32(x["idx"]), t_f32(dI)
    B, S_q, H, D = x["q"].shape
    dq = torch.zeros((B, S_q, H, D), device="cuda")
    dw = torch.zeros((B, S_q, H), device="cuda")
    dk = torch.zeros((B, wl.S_k, D), device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert st(stream) == ibwd.IBWD_OK  # nothing pending from earlier calls
    rc = fn(q.data_ptr(), k.data_ptr(), w.data_ptr(), dIt.data_ptr(), ids.data_ptr(), dq.data_ptr(),
            dw.data_ptr(), dk.data_ptr(), B, S_q, wl.S_k, H, D, wl.topk, stream)
    assert rc == ibwd.IBWD_OK
    assert st(stream) == ibwd.IBWD_ERR_RANGE
    assert st(stream) == ibwd.IBWD_OK  # cleared by the read
