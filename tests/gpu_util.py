"""Shared helpers of the GPU tests: seeded inputs on both sides, the CUDA path
through the C ABI, the oracle side, and the acceptance metrics."""
from __future__ import annotations

import contextlib
import os

import numpy as np
import torch

import oracle
import synth
import sparse_attention_indexer_bwd_gb300 as ibwd

# acceptance: dQ and dW max|err| / max|ref| <= 2e-3, dK rms_rel <= 1e-3,
# dI (the score-grad output) max|err| / max|ref| <= 1e-5
TOL_DQ = 2e-3
TOL_DW = 2e-3
TOL_DK = 1e-3
TOL_DI = 1e-5


def max_rel(got, ref):
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref).max()
    return float(np.abs(np.asarray(got, np.float64) - ref).max() / den) if den > 0 else float(np.abs(got).max())


def rms_rel(got, ref):
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(np.asarray(got, np.float64) - ref) / den) if den > 0 else float(np.linalg.norm(got))


def dev():
    return torch.device("cuda:0")


@contextlib.contextmanager
def gemm_path(path):
    """Imposes the gemm kernel on calls the device-side choice covers (atomic,
    sparse, no options): "rows" (the per-row kernel) or "blocked"."""
    old = os.environ.get("IBWD_TEST_GEMM_PATH")
    os.environ["IBWD_TEST_GEMM_PATH"] = path
    try:
        yield
    finally:
        if old is None:
            del os.environ["IBWD_TEST_GEMM_PATH"]
        else:
            os.environ["IBWD_TEST_GEMM_PATH"] = old


def t_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev()).view(torch.bfloat16)


def t_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev())


def t_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev())


def case_inputs(wl: synth.Workload):
    """Host inputs (numpy) for a workload, index_score from the oracle forward."""
    x = synth.make_inputs(wl)
    if wl.dense:
        x["I"] = oracle.forward_dense(x["q"], x["k"], x["w"]).astype(np.float32)
    else:
        x["I"] = oracle.forward_sparse(x["q"], x["k"], x["w"], x["idx"], wl.S_k).astype(np.float32)
    return x


def oracle_all(wl, x, grad_scale=1.0):
    if wl.dense:
        dI = oracle.score_grad_dense(x["I"], x["attn"], grad_scale)
        dq, dw, dk = oracle.gemm_dense(x["q"], x["k"], x["w"], dI)
    else:
        dI = oracle.score_grad_sparse(x["I"], x["attn"], x["idx"], wl.S_k, grad_scale)
        dq, dw, dk = oracle.gemm_sparse(x["q"], x["k"], x["w"], dI, x["idx"], wl.S_k)
    return dI, dq, dw, dk


def gpu_all(wl, x, dk_mode=ibwd.IBWD_DK_ATOMIC, grad_scale=1.0, path="whole"):
    """The backward through the C ABI; returns numpy (dI, dq, dw, dk).

    path "whole": one indexer_bwd / indexer_bwd_dense call; "pair": the
    score-grad call, then the gemm call."""
    q, k, w = t_bf16(x["q"]), t_bf16(x["k"]), t_f32(x["w"])
    I, attn = t_f32(x["I"]), t_f32(x["attn"])
    idx = None if wl.dense else t_i32(x["idx"])
    if path == "whole":
        dq, dw, dk = ibwd.indexer_backward(q, k, w, I, attn, idx, grad_scale=grad_scale, dk_mode=dk_mode)
    else:
        assert path == "pair"
        B, S_q, H, D = x["q"].shape
        S_k = x["k"].shape[1]
        dq = torch.full((B, S_q, H, D), float("nan"), device=dev())
        dw = torch.full((B, S_q, H), float("nan"), device=dev())
        dk = torch.full((B, S_k, D), float("nan"), device=dev())
        zero = dk if dk_mode == ibwd.IBWD_DK_ATOMIC else None
        if wl.dense:
            ibwd.indexer_bwd_dense_score_grad(I, attn, grad_scale, zero)
            ibwd.indexer_bwd_dense_gemm(q, k, w, attn, dq, dw, dk, dk_mode)
        else:
            ibwd.indexer_bwd_score_grad(I, attn, idx, S_k, grad_scale, zero)
            ibwd.indexer_bwd_gemm(q, k, w, attn, idx, dq, dw, dk, dk_mode)
    st = ibwd.indexer_bwd_last_device_status()
    assert st == ibwd.IBWD_OK, ibwd.status_string(st)
    # index_score is read only (bitwise: it may hold NaN on padded slots)
    assert torch.equal(I.view(torch.int32), t_f32(x["I"]).view(torch.int32))
    return attn.cpu().numpy(), dq.cpu().numpy(), dw.cpu().numpy(), dk.cpu().numpy()


def gpu_gemm(wl, x, dI, dk_mode=ibwd.IBWD_DK_ATOMIC, idx=None):
    """Kernel 2 alone on a given fp32 dI; returns numpy (dq, dw, dk)."""
    q, k, w = t_bf16(x["q"]), t_bf16(x["k"]), t_f32(x["w"])
    dIt = t_f32(dI)
    B, S_q, H, D = x["q"].shape
    S_k = x["k"].shape[1]
    dq = torch.full((B, S_q, H, D), float("nan"), device=dev())
    dw = torch.full((B, S_q, H), float("nan"), device=dev())
    dk = torch.zeros((B, S_k, D), device=dev()) if dk_mode == ibwd.IBWD_DK_ATOMIC else \
        torch.full((B, S_k, D), float("nan"), device=dev())
    if wl.dense:
        ibwd.indexer_bwd_dense_gemm(q, k, w, dIt, dq, dw, dk, dk_mode)
    else:
        ids = t_i32(x["idx"] if idx is None else idx)
        ibwd.indexer_bwd_gemm(q, k, w, dIt, ids, dq, dw, dk, dk_mode)
    st = ibwd.indexer_bwd_last_device_status()
    assert st == ibwd.IBWD_OK, ibwd.status_string(st)
    return dq.cpu().numpy(), dw.cpu().numpy(), dk.cpu().numpy()


def assert_close(dq, dw, dk, ref, tag=""):
    rq, rw, rk = max_rel(dq, ref[0]), max_rel(dw, ref[1]), rms_rel(dk, ref[2])
    assert np.isfinite(dq).all() and np.isfinite(dw).all() and np.isfinite(dk).all(), tag
    assert rq <= TOL_DQ, f"{tag} dq max_rel {rq:.3e}"
    assert rw <= TOL_DW, f"{tag} dw max_rel {rw:.3e}"
    assert rk <= TOL_DK, f"{tag} dk rms_rel {rk:.3e}"
    return rq, rw, rk
