"""Host-only checks of the C ABI (no GPU compute): the library builds, loads
and exports every function include/*.h declares; host-side helpers answer."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

import sparse_attention_indexer_bwd_gb300 as ibwd
from sparse_attention_indexer_bwd_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return ibwd.load()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names += re.findall(r"IBWD_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 8
    assert sorted(names) == sorted(ibwd.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)


def test_status_strings(lib):
    for code in range(7):
        s = ibwd.status_string(code)
        assert isinstance(s, str) and s
    assert ibwd.status_string(99) == "unknown status"


def test_workspace_sizes(lib):
    a = ibwd.indexer_bwd_gemm_workspace_size(1, 8192, 4096, 64, 128, 1024, ibwd.IBWD_DK_ATOMIC)
    nb, tcap = 8192 // 4, 4096 // 128       # blocks of four query rows; records per block (min(S_k, 4*topk) keys)
    # counters + fp16 copy of k (+ a zero row) + per-block info and order + the tile records
    assert a == 256 + 4097 * 128 * 2 + nb * 16 + nb * 4 + nb * tcap * 2560
    d = ibwd.indexer_bwd_gemm_workspace_size(1, 8192, 4096, 64, 128, 1024, ibwd.IBWD_DK_DETERMINISTIC)
    ent = nb * 4096                          # (block, key) entries at most
    u = ent * (128 * 2 + 32)                 # per entry a scaled fp16 dK row and a sector with its factor
    keyoff = ((4096 + 1) * 4 + 255) // 256 * 256
    # key counts per two blocks
    sort = ((nb // 2) * 4096 * 4 + 255) // 256 * 256
    assert d == a + nb * tcap * 512 + u + sort + keyoff
    dnb = 4096 // 4
    dense = 256 + 4097 * 128 * 2 + dnb * 16
    assert ibwd.indexer_bwd_dense_gemm_workspace_size(1, 4096, 64, 128, 0) == dense
    # dense deterministic: block j holds keys [0, 4j + 4): sum over j of 4(j + 1) dK rows
    dd = ibwd.indexer_bwd_dense_gemm_workspace_size(1, 4096, 64, 128, 1)
    dent = 4 * (1024 * 1025 // 2)
    assert dd == dense + dent * (128 * 2 + 32) + keyoff
    # unsupported shapes report 0
    assert ibwd.indexer_bwd_gemm_workspace_size(1, 8, 8, 65, 128, 4, 0) == 0
    assert ibwd.indexer_bwd_gemm_workspace_size(1, 8, 8, 4, 12, 4, 0) == 0
    assert ibwd.indexer_bwd_gemm_workspace_size(1, 8, 8, 4, 32, 4, 5) == 0


def test_shape_errors_need_no_device(lib):
    # invalid shapes are rejected before any CUDA call
    assert lib.indexer_bwd_score_grad(None, None, None, 0, 1, 1, 1, 1.0, None, 0, None) == ibwd.IBWD_ERR_INVALID_ARG
    assert lib.indexer_bwd_score_grad(None, None, None, 1, 1, 1, 1, 1.0, None, 0, None) == ibwd.IBWD_ERR_INVALID_ARG
    assert lib.indexer_bwd_gemm(None, None, None, None, None, None, None, None, 1, 4, 4, 4, 32, 4, 3, None, 0,
                                None) == ibwd.IBWD_ERR_INVALID_ARG
    assert lib.indexer_bwd_gemm(None, None, None, None, None, None, None, None, 1, 4, 4, 100, 32, 4, 0, None, 0,
                                None) == ibwd.IBWD_ERR_UNSUPPORTED
    assert lib.indexer_bwd_dense_gemm(None, None, None, None, None, None, None, 1, 4, 4, 136, 0, None, 0,
                                      None) == ibwd.IBWD_ERR_UNSUPPORTED
    assert lib.indexer_bwd(None, None, None, None, None, None, None, None, None, 1, 4, 4, 4, 32, 4, 1.0, 3, None, 0,
                           None) == ibwd.IBWD_ERR_INVALID_ARG
    # options: flags other than 0/1 are rejected before any device call
    import ctypes
    p = ctypes.c_void_p(16)  # never dereferenced: the option check comes first
    for bad in (ibwd.Options(2, 0, 0, None), ibwd.Options(0, 3, 0, None), ibwd.Options(0, 0, -1, None),
                ibwd.Options(0, 0, 0, None, -1.0), ibwd.Options(0, 0, 0, None, float("nan")),
                ibwd.Options(0, 0, 0, None, float("inf")), ibwd.Options(0, 0, 0, None, -0.0 - 1e-30)):
        assert lib.indexer_bwd_ex(p, p, p, p, p, p, p, p, p, 1, 4, 4, 4, 32, 4, 1.0, 0, ctypes.byref(bad), p,
                                  1 << 20, None) == ibwd.IBWD_ERR_INVALID_ARG
        assert lib.indexer_bwd_dense_ex(p, p, p, p, p, p, p, p, 1, 4, 4, 32, 1.0, 0, ctypes.byref(bad), p,
                                        1 << 20, None) == ibwd.IBWD_ERR_INVALID_ARG
    # matches the C struct: 3 ints, padding, a pointer, a float, padding
    assert ctypes.sizeof(ibwd.Options) == 32 and ibwd.Options.sm_scale.offset == 24
    assert lib.indexer_bwd(None, None, None, None, None, None, None, None, None, 1, 4, 4, 100, 32, 4, 1.0, 0, None,
                           0, None) == ibwd.IBWD_ERR_INVALID_ARG


def test_binding_refuses_to_run_without_library(tmp_path, monkeypatch):
    # the product path has no fallback: a missing library raises on load
    monkeypatch.setattr(ibwd, "_lib", None)
    monkeypatch.setattr(ibwd, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        ibwd.load()
