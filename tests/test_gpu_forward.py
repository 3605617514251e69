"""The forward (index_score from q, k, w and the selected keys) through the C
ABI, against the fp64 oracle's forward: every element on small workloads
(several tiles, ragged tails, B > 1, dense), sampled rows at the anchor
size, padding slots exactly zero, and bitwise determinism."""
import numpy as np
import pytest
import torch

import oracle
import synth
import sparse_attention_indexer_bwd_gb300 as ibwd
from gpu_util import max_rel, t_bf16, t_f32, t_i32

pytestmark = pytest.mark.gpu

TOL_FWD = 1e-5  # fp32 sums of exact bf16 products against fp64

W = synth.Workload
CASES = [
    synth.WORKLOADS["tiny"],
    W("multi_tile_ragged", 2, 64, 128, 300, 700, 300, "causal", 11),
    W("window_small", 1, 64, 128, 384, 512, 256, "window", 12),
    W("odd_shapes", 1, 7, 40, 131, 97, 53, "causal", 13),
    W("dense_small", 1, 64, 128, 200, 200, 0, "dense", 14),
    W("dense_odd", 2, 5, 24, 77, 77, 0, "dense", 15),
]


def run_fwd(wl, x, idx=None):
    q, k, w = t_bf16(x["q"]), t_bf16(x["k"]), t_f32(x["w"])
    if wl.dense:
        out = ibwd.indexer_fwd_dense(q, k, w)
    else:
        out = ibwd.indexer_fwd(q, k, w, t_i32(x["idx"] if idx is None else idx))
    st = ibwd.indexer_bwd_last_device_status()
    assert st == ibwd.IBWD_OK, ibwd.status_string(st)
    return out.cpu().numpy()


def ref_fwd(wl, x, idx=None):
    if wl.dense:
        return oracle.forward_dense(x["q"], x["k"], x["w"])
    return oracle.forward_sparse(x["q"], x["k"], x["w"], x["idx"] if idx is None else idx, wl.S_k)


@pytest.mark.parametrize("wl", CASES, ids=[c.name for c in CASES])
def test_forward_matches_oracle(wl):
    x = synth.make_inputs(wl)
    got = run_fwd(wl, x)
    ref = ref_fwd(wl, x)
    assert max_rel(got, ref) <= TOL_FWD, wl.name
    # padding slots (and the dense upper triangle) are exactly zero
    if wl.dense:
        t = np.arange(wl.S_q)[:, None]
        s = np.arange(wl.S_q)[None, :]
        assert np.all(got[:, s.repeat(wl.S_q, 0) > t.repeat(wl.S_q, 1)] == 0.0)
    else:
        pad = (x["idx"] < 0) | (x["idx"] >= wl.S_k)
        assert np.all(got[pad] == 0.0)
    # bitwise reproducible
    again = run_fwd(wl, x)
    assert np.array_equal(got.view(np.int32), again.view(np.int32))


def test_forward_padding_ids_anywhere():
    wl = CASES[1]
    x = synth.make_inputs(wl)
    rng = np.random.default_rng(5)
    idx = x["idx"].copy()
    bad = rng.random(idx.shape) < 0.2
    idx[bad] = np.where(rng.random(idx.shape) < 0.5, -1, wl.S_k + 3)[bad]
    got = run_fwd(wl, x, idx)
    ref = ref_fwd(wl, x, idx)
    assert max_rel(got, ref) <= TOL_FWD
    assert np.all(got[bad] == 0.0)


def test_forward_anchor_sampled_rows():
    wl = synth.WORKLOADS["anchor"]
    x = synth.make_inputs(wl)
    got = run_fwd(wl, x)
    rows = np.sort(np.random.default_rng(3).permutation(wl.S_q)[:96])
    ref = oracle.forward_sparse(x["q"][:, rows], x["k"], x["w"][:, rows], x["idx"][:, rows], wl.S_k)
    assert max_rel(got[:, rows], ref) <= TOL_FWD


@pytest.mark.parametrize("name", ["multi_tile_ragged", "dense_small"])
def test_forward_then_backward_against_the_oracle_pipeline(name):
    # this library's forward feeding its own backward, against the oracle's
    # forward and backward on the same inputs (tolerances of the backward)
    from gpu_util import TOL_DI, assert_close, oracle_all
    wl = next(c for c in CASES if c.name == name)
    x = synth.make_inputs(wl)
    q, k, w = t_bf16(x["q"]), t_bf16(x["k"]), t_f32(x["w"])
    attn = t_f32(x["attn"])
    if wl.dense:
        I = ibwd.indexer_fwd_dense(q, k, w)
        dq, dw, dk = ibwd.indexer_backward(q, k, w, I, attn, None)
    else:
        idx = t_i32(x["idx"])
        I = ibwd.indexer_fwd(q, k, w, idx)
        dq, dw, dk = ibwd.indexer_backward(q, k, w, I, attn, idx)
    assert ibwd.indexer_bwd_last_device_status() == ibwd.IBWD_OK
    x["I"] = ref_fwd(wl, x).astype(np.float32)
    ref = oracle_all(wl, x)
    assert max_rel(attn.cpu().numpy(), ref[0]) <= TOL_DI
    assert_close(dq.cpu().numpy(), dw.cpu().numpy(), dk.cpu().numpy(), ref[1:], tag=f"pipeline/{name}")
