"""The options of the one-call backward (indexer_bwd_ex / indexer_bwd_dense_ex):
bf16 dq / dw outputs and a bf16 copy of dk are the fp32 results rounded to
nearest even, bit for bit; global top-k ids give the local-id results bit for
bit, and an id of another batch is padding."""
import numpy as np
import pytest
import torch

import synth
import oracle
import sparse_attention_indexer_bwd_gb300 as ibwd
from gpu_util import assert_close, case_inputs, gemm_path, oracle_all, t_bf16, t_f32, t_i32

pytestmark = pytest.mark.gpu

W = synth.Workload
DET = ibwd.IBWD_DK_DETERMINISTIC


def run(wl, x, idx=None, mode=DET, **kw):
    q, k, w = t_bf16(x["q"]), t_bf16(x["k"]), t_f32(x["w"])
    I, attn = t_f32(x["I"]), t_f32(x["attn"])
    ids = None if wl.dense else t_i32(x["idx"] if idx is None else idx)
    dq, dw, dk = ibwd.indexer_backward(q, k, w, I, attn, ids, dk_mode=mode, **kw)
    st = ibwd.indexer_bwd_last_device_status()
    assert st == ibwd.IBWD_OK, ibwd.status_string(st)
    return attn, dq, dw, dk


@pytest.mark.parametrize("wl", [W("opt_sparse", 2, 16, 64, 200, 300, 136, "causal", 31),
                                W("opt_dense", 1, 8, 32, 160, 160, 0, "dense", 32)], ids=lambda w: w.name)
@pytest.mark.parametrize("mode", [ibwd.IBWD_DK_ATOMIC, DET])
def test_bf16_outputs_are_the_rounded_fp32_results(wl, mode):
    x = case_inputs(wl)
    _, dq, dw, dk = run(wl, x, mode=DET)
    dk16 = torch.empty(dk.shape, dtype=torch.bfloat16, device=dk.device)
    a2, dq2, dw2, dk2 = run(wl, x, mode=mode, out_dtype=torch.bfloat16, dk_bf16=dk16)
    assert dq2.dtype == torch.bfloat16 and dw2.dtype == torch.bfloat16
    # dq and dw do not depend on the dK mode: bitwise the rounded fp32 values
    assert torch.equal(dq2.view(torch.int16), dq.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(dw2.view(torch.int16), dw.to(torch.bfloat16).view(torch.int16))
    # the bf16 copy of dk rounds the call's own fp32 dk
    assert torch.equal(dk16.view(torch.int16), dk2.to(torch.bfloat16).view(torch.int16))
    if mode == DET:
        assert torch.equal(dk2.view(torch.int32), dk.view(torch.int32))


@pytest.mark.parametrize("mode", [ibwd.IBWD_DK_ATOMIC, DET])
def test_global_ids_match_local_ids_and_never_alias(mode):
    wl = W("global_ids", 3, 16, 64, 96, 128, 40, "causal", 33)
    x = case_inputs(wl)
    idx = x["idx"].copy()
    B, S_q, L = idx.shape
    # a few slots that point into another batch's key range (globally valid
    # ids) and a positive id past the last batch: all padding for their row
    rng = np.random.default_rng(5)
    pad = idx < 0
    cross = (~pad) & (rng.random(idx.shape) < 0.1)
    local = np.where(cross, -1, idx)              # the same rows with those slots as padding
    off = (np.arange(B) * wl.S_k)[:, None, None]
    glob = np.where(local >= 0, local + off, -1).astype(np.int32)
    other = (np.arange(B)[:, None, None] + 1) % B  # the next batch (the first for the last)
    glob = np.where(cross, (rng.integers(0, wl.S_k, idx.shape) + other * wl.S_k).astype(np.int32), glob)
    glob[0, -1, -1] = np.int32(B * wl.S_k + 7)
    local[0, -1, -1] = -1
    # index_score and attn_score stay as generated: padded slots' values never matter
    with gemm_path("blocked"):  # the kernel global ids run on (the per-row kernel takes local ids only)
        ref_local = run(wl, x, idx=local, mode=mode)
    got = run(wl, x, idx=glob, mode=mode, ids_global=True)
    for a, b in zip(got[:3], ref_local[:3]):           # dI, dq, dw bitwise
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    if mode == DET:
        assert torch.equal(got[3].view(torch.int32), ref_local[3].view(torch.int32))
    # and against the oracle on the local form
    xl = dict(x)
    xl["idx"] = local
    ref = oracle_all(wl, xl)
    assert_close(got[1].cpu().numpy(), got[2].cpu().numpy(), got[3].cpu().numpy(), ref[1:], tag="global ids")


@pytest.mark.parametrize("sm_scale", [0.5, 0.0884])
@pytest.mark.parametrize("wl", [W("scale_sparse", 2, 40, 64, 300, 260, 150, "causal", 34),
                                W("scale_dense", 1, 8, 64, 200, 200, 0, "dense", 35)], ids=lambda w: w.name)
@pytest.mark.parametrize("mode", [ibwd.IBWD_DK_ATOMIC, DET])
def test_logit_scale_matches_the_scaled_oracle(wl, mode, sm_scale):
    """index_score from the forward with the logit scale inside the ReLU; the
    backward with that scale against the oracle's scaled definitions."""
    x = synth.make_inputs(wl)
    if wl.dense:
        x["I"] = oracle.forward_dense(x["q"], x["k"], x["w"], sm_scale).astype(np.float32)
        dI = oracle.score_grad_dense(x["I"], x["attn"])
        ref = oracle.gemm_dense(x["q"], x["k"], x["w"], dI, sm_scale)
    else:
        x["I"] = oracle.forward_sparse(x["q"], x["k"], x["w"], x["idx"], wl.S_k, sm_scale).astype(np.float32)
        dI = oracle.score_grad_sparse(x["I"], x["attn"], x["idx"], wl.S_k)
        ref = oracle.gemm_sparse(x["q"], x["k"], x["w"], dI, x["idx"], wl.S_k, sm_scale)
    attn, dq, dw, dk = run(wl, x, mode=mode, sm_scale=sm_scale)
    assert_close(dq.cpu().numpy(), dw.cpu().numpy(), dk.cpu().numpy(), ref, tag=f"sm_scale {sm_scale}")
    # and the unscaled call on the same I differs by exactly the factor's effect
    if sm_scale == 0.5 and mode == DET:
        _, dq1, dw1, dk1 = run(wl, x, mode=mode)
        assert torch.equal(dq.view(torch.int32), (0.5 * dq1).view(torch.int32))
        assert torch.equal(dk.view(torch.int32), (0.5 * dk1).view(torch.int32))
        assert torch.equal(dw.view(torch.int32), (0.5 * dw1).view(torch.int32))
