"""Seeded synthetic inputs for the indexer backward (tests and benchmark).

Holds none of the method's arithmetic: only random draws, causal id sampling
and target-distribution rows.  `index_score` (the forward logits) is not made
here; callers obtain it from the forward of their own side.

The C source (synth.c) is built with gcc into libsynth.so next to it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "libsynth.so")

# one stream per array, so each value depends only on (seed, stream, position)
STREAM_Q, STREAM_K, STREAM_W, STREAM_IDX, STREAM_ATTN = 1, 2, 3, 4, 5


def build(force: bool = False) -> str:
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


_lib = None


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i32, i64, dbl, p = ctypes.c_uint64, ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.synth_u64.argtypes = [u64, u64, u64]
        lib.synth_u64.restype = u64
        lib.synth_normal_f32.argtypes = [u64, u64, i64, dbl, dbl, p]
        lib.synth_normal_bf16.argtypes = [u64, u64, i64, dbl, dbl, p]
        lib.synth_topk_causal.argtypes = [u64, u64, i32, i32, i32, i32, p]
        lib.synth_topk_window.argtypes = [u64, u64, i32, i32, i32, i32, i32, p]
        lib.synth_topk_uniform.argtypes = [u64, u64, i32, i32, i32, i32, p]
        lib.synth_target_sparse.argtypes = [u64, u64, p, i32, i32, i32, i32, dbl, p]
        lib.synth_target_dense.argtypes = [u64, u64, i32, i32, dbl, p]
        for f in ("synth_topk_causal", "synth_topk_window", "synth_topk_uniform", "synth_target_sparse",
                  "synth_target_dense"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def u64(seed: int, stream: int, ctr: int) -> int:
    return int(_L().synth_u64(seed, stream, ctr))


def normal_f32(seed, stream, shape, mean=0.0, std=1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _L().synth_normal_f32(seed, stream, out.size, mean, std, _ptr(out))
    return out


def normal_bf16(seed, stream, shape, mean=0.0, std=1.0) -> np.ndarray:
    """bf16 bit patterns (uint16), rounded to nearest even from fp32."""
    out = np.empty(shape, dtype=np.uint16)
    _L().synth_normal_bf16(seed, stream, out.size, mean, std, _ptr(out))
    return out


def topk_causal(seed, stream, B, S_q, S_k, topk) -> np.ndarray:
    out = np.empty((B, S_q, topk), dtype=np.int32)
    if _L().synth_topk_causal(seed, stream, B, S_q, S_k, topk, _ptr(out)):
        raise MemoryError("synth_topk_causal")
    return out


def topk_uniform(seed, stream, B, S_q, S_k, topk) -> np.ndarray:
    out = np.empty((B, S_q, topk), dtype=np.int32)
    if _L().synth_topk_uniform(seed, stream, B, S_q, S_k, topk, _ptr(out)):
        raise MemoryError("synth_topk_uniform")
    return out


def topk_window(seed, stream, B, S_q, S_k, topk, window=256) -> np.ndarray:
    out = np.empty((B, S_q, topk), dtype=np.int32)
    if _L().synth_topk_window(seed, stream, B, S_q, S_k, topk, window, _ptr(out)):
        raise MemoryError("synth_topk_window")
    return out


def target_sparse(seed, stream, idx: np.ndarray, S_k: int, var=2.0) -> np.ndarray:
    B, S_q, topk = idx.shape
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    out = np.empty((B, S_q, topk), dtype=np.float32)
    if _L().synth_target_sparse(seed, stream, _ptr(idx), B, S_q, S_k, topk, var, _ptr(out)):
        raise MemoryError("synth_target_sparse")
    return out


def target_dense(seed, stream, B, S, var=2.0) -> np.ndarray:
    out = np.empty((B, S, S), dtype=np.float32)
    if _L().synth_target_dense(seed, stream, B, S, var, _ptr(out)):
        raise MemoryError("synth_target_dense")
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, id structure and seed."""
    name: str
    B: int
    H: int
    D: int
    S_q: int
    S_k: int
    topk: int          # 0 for the dense variant
    ids: str           # "causal" | "window" | "uniform" | "dense"
    seed: int

    @property
    def dense(self) -> bool:
        return self.ids == "dense"

    def flops(self) -> float:
        """Nominal gemm-stage FLOP: 6 * rows * selected slots * H * D."""
        if self.dense:
            return 6.0 * self.B * self.H * self.D * self.S_q * (self.S_q + 1) / 2.0
        return 6.0 * self.B * self.S_q * self.topk * self.H * self.D


# The five workloads: a tiny oracle check, two causal top-k shapes (the larger
# is the anchor shape of the pages' timings), a local-window contention shape
# and the dense-causal variant.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 4, 32, 64, 64, 16, "causal", 0),
    "sq4096_topk512": Workload("sq4096_topk512", 1, 64, 128, 4096, 4096, 512, "causal", 1),
    "anchor": Workload("anchor", 1, 64, 128, 8192, 4096, 1024, "causal", 2),
    "window_topk2048": Workload("window_topk2048", 1, 64, 128, 8192, 4096, 2048, "window", 3),
    "dense_s4096": Workload("dense_s4096", 1, 64, 128, 4096, 4096, 0, "dense", 4),
}
# The top-k sweep of the pages' benchmark harness at the anchor shape with
# uniform lengths: every row selects topk distinct keys out of all S_k (the
# causal workloads above are its ragged, monotone-ramp form).
for _i, _k in enumerate((128, 256, 384, 512, 640, 1024, 1536, 2048)):
    WORKLOADS[f"uniform_topk{_k}"] = Workload(f"uniform_topk{_k}", 1, 64, 128, 8192, 4096, _k, "uniform", 10 + _i)


def make_inputs(wl: Workload) -> dict:
    """q, k (bf16 bits), w (fp32), idx (int32, absent for dense), attn (fp32).

    q, k ~ N(0,1) rounded to bf16; w ~ N(0,1)/sqrt(H); attn rows are the
    normalised exp of N(0, 2) logits over the valid slots.
    """
    s = wl.seed
    out = {
        "q": normal_bf16(s, STREAM_Q, (wl.B, wl.S_q, wl.H, wl.D)),
        "k": normal_bf16(s, STREAM_K, (wl.B, wl.S_k, wl.D)),
        "w": normal_f32(s, STREAM_W, (wl.B, wl.S_q, wl.H), 0.0, 1.0 / np.sqrt(wl.H)),
    }
    if wl.dense:
        out["attn"] = target_dense(s, STREAM_ATTN, wl.B, wl.S_q)
    else:
        if wl.ids == "window":
            idx = topk_window(s, STREAM_IDX, wl.B, wl.S_q, wl.S_k, wl.topk)
        elif wl.ids == "uniform":
            idx = topk_uniform(s, STREAM_IDX, wl.B, wl.S_q, wl.S_k, wl.topk)
        else:
            idx = topk_causal(s, STREAM_IDX, wl.B, wl.S_q, wl.S_k, wl.topk)
        out["idx"] = idx
        out["attn"] = target_sparse(s, STREAM_ATTN, idx, wl.S_k)
    return out
