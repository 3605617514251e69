"""fp64 CPU oracle for the indexer backward -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  It shares no code with the CUDA library and neither
imports the other.  The arithmetic lives in oracle.c (plain loops, double
precision, OpenMP over query rows); this module only marshals numpy arrays.

Every function's definition and its source passage is stated in oracle.c.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Compiles liboracle.so with gcc (strict IEEE: no fast-math)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


_lib = None


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i, d, p = ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.oracle_set_threads.argtypes = [i]
        lib.oracle_forward_sparse.argtypes = [p, p, p, p, i, i, i, i, i, i, d, p]
        lib.oracle_score_grad_sparse.argtypes = [p, p, p, i, i, i, i, d, p]
        lib.oracle_score_grad_dense.argtypes = [p, p, i, i, d, p]
        lib.oracle_gemm_sparse.argtypes = [p, p, p, p, p, i, i, i, i, i, i, d, p, p, p]
        lib.oracle_gemm_sparse_rows.argtypes = [p, p, p, p, p, i, i, i, i, i, i, d, p, i, p, p]
        lib.oracle_forward_dense.argtypes = [p, p, p, i, i, i, i, d, p]
        lib.oracle_gemm_dense.argtypes = [p, p, p, p, i, i, i, i, d, p, p, p]
        lib.oracle_gemm_dense_rows.argtypes = [p, p, p, p, i, i, i, i, d, p, i, p, p]
        _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, name):
    if rc:
        raise MemoryError(f"oracle: {name} failed to allocate")


def set_threads(n: int = 0) -> int:
    """Sets the OpenMP thread count (0 = leave it); returns the count in use."""
    return int(_L().oracle_set_threads(n))


def forward_sparse(q, k, w, idx, S_k: int, sm_scale: float = 1.0) -> np.ndarray:
    """I[b,t,j] = sum_h w relu(sm_scale q[b,t,h].k[b,idx]) (0 on padding), float64."""
    B, S_q, H, D = q.shape
    topk = idx.shape[-1]
    q, qp = _c(q, np.uint16); k, kp = _c(k, np.uint16)
    w, wp = _c(w, np.float32); idx, ip = _c(idx, np.int32)
    out = np.empty((B, S_q, topk), np.float64)
    _check(_L().oracle_forward_sparse(qp, kp, wp, ip, B, S_q, S_k, H, D, topk, float(sm_scale),
                                      out.ctypes.data_as(ctypes.c_void_p)), "forward_sparse")
    return out


def score_grad_sparse(index_score, attn_score, idx, S_k: int, grad_scale: float = 1.0) -> np.ndarray:
    B, S_q, topk = idx.shape
    I, Ip = _c(index_score, np.float32); a, ap = _c(attn_score, np.float32)
    idx, ip = _c(idx, np.int32)
    out = np.empty((B, S_q, topk), np.float64)
    _check(_L().oracle_score_grad_sparse(Ip, ap, ip, B, S_q, S_k, topk, grad_scale,
                                         out.ctypes.data_as(ctypes.c_void_p)), "score_grad_sparse")
    return out


def score_grad_dense(index_score, attn_score, grad_scale: float = 1.0) -> np.ndarray:
    B, S, S2 = index_score.shape
    assert S == S2
    I, Ip = _c(index_score, np.float32); a, ap = _c(attn_score, np.float32)
    out = np.empty((B, S, S), np.float64)
    _check(_L().oracle_score_grad_dense(Ip, ap, B, S, grad_scale,
                                        out.ctypes.data_as(ctypes.c_void_p)), "score_grad_dense")
    return out


def gemm_sparse(q, k, w, dI, idx, S_k: int, sm_scale: float = 1.0):
    """(dq [B,S_q,H,D], dw [B,S_q,H], dk [B,S_k,D]) in float64."""
    B, S_q, H, D = q.shape
    topk = idx.shape[-1]
    q, qp = _c(q, np.uint16); k, kp = _c(k, np.uint16)
    w, wp = _c(w, np.float32); idx, ip = _c(idx, np.int32)
    dI, dp = _c(dI, np.float64)
    dq = np.empty((B, S_q, H, D), np.float64)
    dw = np.empty((B, S_q, H), np.float64)
    dk = np.empty((B, S_k, D), np.float64)
    vp = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    _check(_L().oracle_gemm_sparse(qp, kp, wp, dp, ip, B, S_q, S_k, H, D, topk, float(sm_scale),
                                   vp(dq), vp(dw), vp(dk)), "gemm_sparse")
    return dq, dw, dk


def gemm_sparse_rows(q, k, w, dI_rows, idx, S_k: int, rows, sm_scale: float = 1.0):
    """dQ/dW of the listed global rows (b*S_q + t); dI_rows is [len(rows), topk]."""
    B, S_q, H, D = q.shape
    topk = idx.shape[-1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    q, qp = _c(q, np.uint16); k, kp = _c(k, np.uint16)
    w, wp = _c(w, np.float32); idx, ip = _c(idx, np.int32)
    dI_rows, dp = _c(dI_rows, np.float64)
    n = rows.size
    dq = np.empty((n, H, D), np.float64)
    dw = np.empty((n, H), np.float64)
    vp = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    _check(_L().oracle_gemm_sparse_rows(qp, kp, wp, dp, ip, B, S_q, S_k, H, D, topk, float(sm_scale),
                                        vp(rows), n, vp(dq), vp(dw)), "gemm_sparse_rows")
    return dq, dw


def forward_dense(q, k, w, sm_scale: float = 1.0) -> np.ndarray:
    B, S, H, D = q.shape
    q, qp = _c(q, np.uint16); k, kp = _c(k, np.uint16); w, wp = _c(w, np.float32)
    out = np.empty((B, S, S), np.float64)
    _check(_L().oracle_forward_dense(qp, kp, wp, B, S, H, D, float(sm_scale),
                                     out.ctypes.data_as(ctypes.c_void_p)), "forward_dense")
    return out


def gemm_dense(q, k, w, dI, sm_scale: float = 1.0):
    B, S, H, D = q.shape
    q, qp = _c(q, np.uint16); k, kp = _c(k, np.uint16); w, wp = _c(w, np.float32)
    dI, dp = _c(dI, np.float64)
    dq = np.empty((B, S, H, D), np.float64)
    dw = np.empty((B, S, H), np.float64)
    dk = np.empty((B, S, D), np.float64)
    vp = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    _check(_L().oracle_gemm_dense(qp, kp, wp, dp, B, S, H, D, float(sm_scale), vp(dq), vp(dw), vp(dk)),
           "gemm_dense")
    return dq, dw, dk


def gemm_dense_rows(q, k, w, dI_rows, rows, sm_scale: float = 1.0):
    B, S, H, D = q.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    q, qp = _c(q, np.uint16); k, kp = _c(k, np.uint16); w, wp = _c(w, np.float32)
    dI_rows, dp = _c(dI_rows, np.float64)
    n = rows.size
    dq = np.empty((n, H, D), np.float64)
    dw = np.empty((n, H), np.float64)
    vp = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    _check(_L().oracle_gemm_dense_rows(qp, kp, wp, dp, B, S, H, D, float(sm_scale), vp(rows), n, vp(dq), vp(dw)),
           "gemm_dense_rows")
    return dq, dw
