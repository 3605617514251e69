"""Python binding of libindexer_bwd.so (backward of the DeepSeek-sparse-attention
lightning indexer on GB300 / sm_103a).

Argument marshalling only: every step runs in the CUDA library through its C
ABI (declared in include/indexer_bwd.h).  torch supplies device memory and
streams.  The functions keep the C names; tensors replace pointers and the
shapes are read from them.  A nonzero status raises IndexerBwdError.

There is no CPU fallback: importing the library fails loudly when
libindexer_bwd.so has not been built (``python -m
sparse_attention_indexer_bwd_gb300._build`` or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB as _LIB_PATH

IBWD_OK = 0
IBWD_ERR_INVALID_ARG = 1
IBWD_ERR_UNSUPPORTED = 2
IBWD_ERR_WORKSPACE = 3
IBWD_ERR_CUDA = 4
IBWD_ERR_TIMEOUT = 5
IBWD_ERR_RANGE = 6
IBWD_DK_ATOMIC = 0
IBWD_DK_DETERMINISTIC = 1

EXPORTS = (
    "indexer_bwd_score_grad",
    "indexer_bwd_gemm_workspace_size",
    "indexer_bwd_gemm",
    "indexer_bwd_dense_score_grad",
    "indexer_bwd_dense_gemm_workspace_size",
    "indexer_bwd_dense_gemm",
    "indexer_bwd_last_device_status",
    "indexer_bwd_status_string",
    "indexer_bwd_gemm_noalloc",
    "indexer_bwd_gemm_noalloc_setup",
    "indexer_bwd_gemm_noalloc_status",
    "indexer_fwd",
    "indexer_fwd_dense",
    "indexer_bwd",
    "indexer_bwd_dense",
    "indexer_bwd_ex",
    "indexer_bwd_dense_ex",
)


class Options(ctypes.Structure):
    """ibwd_options of the C header (ids_global, dq_bf16, dw_bf16, dk_bf16, sm_scale)."""
    _fields_ = [("ids_global", ctypes.c_int), ("dq_bf16", ctypes.c_int), ("dw_bf16", ctypes.c_int),
                ("dk_bf16", ctypes.c_void_p), ("sm_scale", ctypes.c_float)]


class IndexerBwdError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: status {status} ({status_string(status)})")
        self.status = status


_lib = None


def library_path() -> str:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Loads libindexer_bwd.so (raises if it is missing: no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"{_LIB_PATH} is missing; build it with "
                          "`python -m sparse_attention_indexer_bwd_gb300._build`")
    lib = ctypes.CDLL(_LIB_PATH)
    p, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.indexer_bwd_score_grad.argtypes = [p, p, p, i, i, i, i, f, p, i, p]
    lib.indexer_bwd_score_grad.restype = i
    lib.indexer_bwd_gemm_workspace_size.argtypes = [i, i, i, i, i, i, i]
    lib.indexer_bwd_gemm_workspace_size.restype = sz
    lib.indexer_bwd_gemm.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i, i, i, i, p, sz, p]
    lib.indexer_bwd_gemm.restype = i
    lib.indexer_bwd_dense_score_grad.argtypes = [p, p, i, i, f, p, i, p]
    lib.indexer_bwd_dense_score_grad.restype = i
    lib.indexer_bwd_dense_gemm_workspace_size.argtypes = [i, i, i, i, i]
    lib.indexer_bwd_dense_gemm_workspace_size.restype = sz
    lib.indexer_bwd_dense_gemm.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, p, sz, p]
    lib.indexer_bwd_dense_gemm.restype = i
    lib.indexer_bwd.argtypes = [p, p, p, p, p, p, p, p, p, i, i, i, i, i, i, f, i, p, sz, p]
    lib.indexer_bwd.restype = i
    lib.indexer_bwd_dense.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i, f, i, p, sz, p]
    lib.indexer_bwd_dense.restype = i
    po = ctypes.POINTER(Options)
    lib.indexer_bwd_ex.argtypes = [p, p, p, p, p, p, p, p, p, i, i, i, i, i, i, f, i, po, p, sz, p]
    lib.indexer_bwd_ex.restype = i
    lib.indexer_bwd_dense_ex.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i, f, i, po, p, sz, p]
    lib.indexer_bwd_dense_ex.restype = i
    lib.indexer_fwd.argtypes = [p, p, p, p, p, i, i, i, i, i, i, p]
    lib.indexer_fwd.restype = i
    lib.indexer_fwd_dense.argtypes = [p, p, p, p, i, i, i, i, p]
    lib.indexer_fwd_dense.restype = i
    lib.indexer_bwd_last_device_status.argtypes = [p]
    lib.indexer_bwd_last_device_status.restype = i
    lib.indexer_bwd_status_string.argtypes = [i]
    lib.indexer_bwd_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().indexer_bwd_status_string(int(status)).decode()


# ----------------------------------------------------------- marshalling ---

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t, dtype, ndim, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype or t.dim() != ndim or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor of {ndim} dims, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device}")


def _check(rc, where):
    if rc != IBWD_OK:
        raise IndexerBwdError(rc, where)


# ------------------------------------------------------------- entry points ---

def indexer_bwd_score_grad(index_score, attn_score, topk_idx, S_k: int, grad_scale: float = 1.0,
                           dk_to_zero=None, stream=None):
    """Kernel 1: dI over attn_score in place; zeroes dk_to_zero [B,S_k,D] if given."""
    _need(index_score, torch.float32, 3, "index_score")
    _need(attn_score, torch.float32, 3, "attn_score")
    _need(topk_idx, torch.int32, 3, "topk_idx")
    B, S_q, topk = attn_score.shape
    D = 0
    if dk_to_zero is not None:
        _need(dk_to_zero, torch.float32, 3, "dk_to_zero")
        D = dk_to_zero.shape[-1]
    rc = load().indexer_bwd_score_grad(_ptr(index_score), _ptr(attn_score), _ptr(topk_idx), B, S_q, S_k, topk,
                                       float(grad_scale), _ptr(dk_to_zero), D, _stream(stream))
    _check(rc, "indexer_bwd_score_grad")


def indexer_bwd_gemm_workspace_size(B, S_q, S_k, H, D, topk, dk_mode=IBWD_DK_ATOMIC) -> int:
    return int(load().indexer_bwd_gemm_workspace_size(B, S_q, S_k, H, D, topk, dk_mode))


def indexer_bwd_gemm(q, k, w, dI, topk_idx, dq, dw, dk, dk_mode=IBWD_DK_ATOMIC, workspace=None, stream=None):
    """Kernel 2: dq, dw (written) and dk (accumulated, or overwritten in deterministic mode)."""
    _need(q, torch.bfloat16, 4, "q")
    _need(k, torch.bfloat16, 3, "k")
    _need(w, torch.float32, 3, "w")
    _need(dI, torch.float32, 3, "dI")
    _need(topk_idx, torch.int32, 3, "topk_idx")
    _need(dq, torch.float32, 4, "dq")
    _need(dw, torch.float32, 3, "dw")
    _need(dk, torch.float32, 3, "dk")
    B, S_q, H, D = q.shape
    S_k = k.shape[1]
    topk = topk_idx.shape[-1]
    if workspace is None:
        workspace = torch.empty(indexer_bwd_gemm_workspace_size(B, S_q, S_k, H, D, topk, dk_mode),
                                dtype=torch.uint8, device=q.device)
    rc = load().indexer_bwd_gemm(_ptr(q), _ptr(k), _ptr(w), _ptr(dI), _ptr(topk_idx), _ptr(dq), _ptr(dw),
                                 _ptr(dk), B, S_q, S_k, H, D, topk, int(dk_mode), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "indexer_bwd_gemm")


def indexer_bwd_dense_score_grad(index_score, attn_score, grad_scale: float = 1.0, dk_to_zero=None,
                                 stream=None):
    _need(index_score, torch.float32, 3, "index_score")
    _need(attn_score, torch.float32, 3, "attn_score")
    B, S, S2 = attn_score.shape
    if S != S2:
        raise ValueError("dense scores must be [B, S, S]")
    D = 0
    if dk_to_zero is not None:
        _need(dk_to_zero, torch.float32, 3, "dk_to_zero")
        D = dk_to_zero.shape[-1]
    rc = load().indexer_bwd_dense_score_grad(_ptr(index_score), _ptr(attn_score), B, S, float(grad_scale),
                                             _ptr(dk_to_zero), D, _stream(stream))
    _check(rc, "indexer_bwd_dense_score_grad")


def indexer_bwd_dense_gemm_workspace_size(B, S, H, D, dk_mode=IBWD_DK_ATOMIC) -> int:
    return int(load().indexer_bwd_dense_gemm_workspace_size(B, S, H, D, dk_mode))


def indexer_bwd_dense_gemm(q, k, w, dI, dq, dw, dk, dk_mode=IBWD_DK_ATOMIC, workspace=None, stream=None):
    _need(q, torch.bfloat16, 4, "q")
    _need(k, torch.bfloat16, 3, "k")
    _need(w, torch.float32, 3, "w")
    _need(dI, torch.float32, 3, "dI")
    _need(dq, torch.float32, 4, "dq")
    _need(dw, torch.float32, 3, "dw")
    _need(dk, torch.float32, 3, "dk")
    B, S, H, D = q.shape
    if workspace is None:
        workspace = torch.empty(indexer_bwd_dense_gemm_workspace_size(B, S, H, D, dk_mode),
                                dtype=torch.uint8, device=q.device)
    rc = load().indexer_bwd_dense_gemm(_ptr(q), _ptr(k), _ptr(w), _ptr(dI), _ptr(dq), _ptr(dw), _ptr(dk),
                                       B, S, H, D, int(dk_mode), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "indexer_bwd_dense_gemm")


def indexer_bwd_last_device_status(stream=None) -> int:
    return int(load().indexer_bwd_last_device_status(_stream(stream)))


def indexer_bwd_status_string(status: int) -> str:
    return status_string(status)


# --------------------------------------------------------------- pipeline ---

def indexer_fwd(q, k, w, topk_idx, out=None, stream=None):
    """Forward logits index_score[t,j] = sum_h w relu(q[t,h].k[topk_idx[t,j]]) (0 on padding)."""
    _need(q, torch.bfloat16, 4, "q")
    _need(k, torch.bfloat16, 3, "k")
    _need(w, torch.float32, 3, "w")
    _need(topk_idx, torch.int32, 3, "topk_idx")
    B, S_q, H, D = q.shape
    S_k = k.shape[1]
    topk = topk_idx.shape[-1]
    if out is None:
        out = torch.empty((B, S_q, topk), dtype=torch.float32, device=q.device)
    rc = load().indexer_fwd(_ptr(q), _ptr(k), _ptr(w), _ptr(topk_idx), _ptr(out), B, S_q, S_k, H, D, topk,
                            _stream(stream))
    _check(rc, "indexer_fwd")
    return out


def indexer_fwd_dense(q, k, w, out=None, stream=None):
    """Dense forward: index_score[t,s] for every key s <= t, 0 above the diagonal ([B,S,S])."""
    _need(q, torch.bfloat16, 4, "q")
    _need(k, torch.bfloat16, 3, "k")
    _need(w, torch.float32, 3, "w")
    B, S, H, D = q.shape
    if out is None:
        out = torch.empty((B, S, S), dtype=torch.float32, device=q.device)
    rc = load().indexer_fwd_dense(_ptr(q), _ptr(k), _ptr(w), _ptr(out), B, S, H, D, _stream(stream))
    _check(rc, "indexer_fwd_dense")
    return out


def indexer_bwd(q, k, w, index_score, attn_score, topk_idx, dq, dw, dk, grad_scale: float = 1.0,
                dk_mode=IBWD_DK_ATOMIC, workspace=None, stream=None):
    """The whole backward in one call (the score-grad kernel, then the gemm
    stage): dI over attn_score; dq, dw and dk all written."""
    _need(q, torch.bfloat16, 4, "q")
    _need(k, torch.bfloat16, 3, "k")
    _need(w, torch.float32, 3, "w")
    _need(index_score, torch.float32, 3, "index_score")
    _need(attn_score, torch.float32, 3, "attn_score")
    _need(topk_idx, torch.int32, 3, "topk_idx")
    _need(dq, torch.float32, 4, "dq")
    _need(dw, torch.float32, 3, "dw")
    _need(dk, torch.float32, 3, "dk")
    B, S_q, H, D = q.shape
    S_k = k.shape[1]
    topk = topk_idx.shape[-1]
    if workspace is None:
        workspace = torch.empty(indexer_bwd_gemm_workspace_size(B, S_q, S_k, H, D, topk, dk_mode),
                                dtype=torch.uint8, device=q.device)
    rc = load().indexer_bwd(_ptr(q), _ptr(k), _ptr(w), _ptr(index_score), _ptr(attn_score), _ptr(topk_idx),
                            _ptr(dq), _ptr(dw), _ptr(dk), B, S_q, S_k, H, D, topk, float(grad_scale),
                            int(dk_mode), _ptr(workspace), workspace.numel() * workspace.element_size(),
                            _stream(stream))
    _check(rc, "indexer_bwd")


def indexer_bwd_dense(q, k, w, index_score, attn_score, dq, dw, dk, grad_scale: float = 1.0,
                      dk_mode=IBWD_DK_ATOMIC, workspace=None, stream=None):
    """Dense variant of indexer_bwd ([B,S,S] scores, every key s <= t)."""
    _need(q, torch.bfloat16, 4, "q")
    _need(k, torch.bfloat16, 3, "k")
    _need(w, torch.float32, 3, "w")
    _need(index_score, torch.float32, 3, "index_score")
    _need(attn_score, torch.float32, 3, "attn_score")
    _need(dq, torch.float32, 4, "dq")
    _need(dw, torch.float32, 3, "dw")
    _need(dk, torch.float32, 3, "dk")
    B, S, H, D = q.shape
    if workspace is None:
        workspace = torch.empty(indexer_bwd_dense_gemm_workspace_size(B, S, H, D, dk_mode),
                                dtype=torch.uint8, device=q.device)
    rc = load().indexer_bwd_dense(_ptr(q), _ptr(k), _ptr(w), _ptr(index_score), _ptr(attn_score), _ptr(dq),
                                  _ptr(dw), _ptr(dk), B, S, H, D, float(grad_scale), int(dk_mode),
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream))
    _check(rc, "indexer_bwd_dense")


def _out_flag(t, name):
    if t.dtype == torch.float32:
        return 0
    if t.dtype == torch.bfloat16:
        return 1
    raise TypeError(f"{name} must be float32 or bfloat16, got {t.dtype}")


def indexer_bwd_ex(q, k, w, index_score, attn_score, topk_idx, dq, dw, dk, grad_scale: float = 1.0,
                   dk_mode=IBWD_DK_ATOMIC, ids_global: bool = False, dk_bf16=None, workspace=None, stream=None,
                   sm_scale: float = 1.0):
    """indexer_bwd with options: dq / dw may be bfloat16 tensors (rounded to
    nearest even from the fp32 results), dk_bf16 an optional bfloat16
    [B,S_k,D] copy of dk, ids_global=True takes ids into the flattened
    [B*S_k] keys, and sm_scale is the forward's logit scale
    (I = sum_h w relu(sm_scale q.k); the gradients scale by it).
    topk_idx=None selects the dense variant."""
    _need(q, torch.bfloat16, 4, "q")
    _need(k, torch.bfloat16, 3, "k")
    _need(w, torch.float32, 3, "w")
    _need(index_score, torch.float32, 3, "index_score")
    _need(attn_score, torch.float32, 3, "attn_score")
    _need(dq, dq.dtype, 4, "dq")
    _need(dw, dw.dtype, 3, "dw")
    _need(dk, torch.float32, 3, "dk")
    if dk_bf16 is not None:
        _need(dk_bf16, torch.bfloat16, 3, "dk_bf16")
    opts = Options(int(bool(ids_global)), _out_flag(dq, "dq"), _out_flag(dw, "dw"),
                   None if dk_bf16 is None else dk_bf16.data_ptr(), float(sm_scale))
    B, S_q, H, D = q.shape
    S_k = k.shape[1]
    lib = load()
    if topk_idx is None:
        if workspace is None:
            workspace = torch.empty(indexer_bwd_dense_gemm_workspace_size(B, S_q, H, D, dk_mode),
                                    dtype=torch.uint8, device=q.device)
        rc = lib.indexer_bwd_dense_ex(_ptr(q), _ptr(k), _ptr(w), _ptr(index_score), _ptr(attn_score), _ptr(dq),
                                      _ptr(dw), _ptr(dk), B, S_q, H, D, float(grad_scale), int(dk_mode),
                                      ctypes.byref(opts), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream))
        _check(rc, "indexer_bwd_dense_ex")
        return
    _need(topk_idx, torch.int32, 3, "topk_idx")
    topk = topk_idx.shape[-1]
    if workspace is None:
        workspace = torch.empty(indexer_bwd_gemm_workspace_size(B, S_q, S_k, H, D, topk, dk_mode),
                                dtype=torch.uint8, device=q.device)
    rc = lib.indexer_bwd_ex(_ptr(q), _ptr(k), _ptr(w), _ptr(index_score), _ptr(attn_score), _ptr(topk_idx),
                            _ptr(dq), _ptr(dw), _ptr(dk), B, S_q, S_k, H, D, topk, float(grad_scale),
                            int(dk_mode), ctypes.byref(opts), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "indexer_bwd_ex")


def indexer_backward(q, k, w, index_score, attn_score, topk_idx=None, grad_scale: float = 1.0,
                     dk_mode=IBWD_DK_ATOMIC, workspace=None, out=None, stream=None, ids_global: bool = False,
                     out_dtype=torch.float32, dk_bf16=None, sm_scale: float = 1.0):
    """The whole backward (indexer_bwd / indexer_bwd_dense, or their _ex forms
    when an option is given): dI over attn_score (index_score is kept), then
    dq, dw, dk.

    topk_idx=None selects the dense-causal variant ([B,S,S] scores).
    `out` may supply preallocated (dq, dw, dk) tensors; out_dtype
    (torch.float32 or torch.bfloat16) is the dtype of dq and dw when they are
    allocated here; dk is always fp32, and dk_bf16 may receive a bf16 copy.
    ids_global=True takes ids into the flattened [B*S_k] keys.  sm_scale is
    the forward's logit scale, I = sum_h w relu(sm_scale q.k): index_score
    must come from that forward, and dq, dw, dk scale by it.
    Returns (dq, dw, dk).
    """
    B, S_q, H, D = q.shape
    S_k = k.shape[1]
    if out is None:
        dq = torch.empty((B, S_q, H, D), dtype=out_dtype, device=q.device)
        dw = torch.empty((B, S_q, H), dtype=out_dtype, device=q.device)
        dk = torch.empty((B, S_k, D), dtype=torch.float32, device=q.device)
    else:
        dq, dw, dk = out
    if (ids_global or dk_bf16 is not None or dq.dtype != torch.float32 or dw.dtype != torch.float32
            or sm_scale != 1.0):
        indexer_bwd_ex(q, k, w, index_score, attn_score, topk_idx, dq, dw, dk, grad_scale, dk_mode, ids_global,
                       dk_bf16, workspace, stream, sm_scale)
    elif topk_idx is None:
        indexer_bwd_dense(q, k, w, index_score, attn_score, dq, dw, dk, grad_scale, dk_mode, workspace, stream)
    else:
        indexer_bwd(q, k, w, index_score, attn_score, topk_idx, dq, dw, dk, grad_scale, dk_mode, workspace,
                    stream)
    return dq, dw, dk
