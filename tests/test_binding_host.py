"""The Python binding refuses host tensors and wrong dtypes before anything
reaches the library (no GPU needed): it marshals arguments, it never falls
back to computing on the CPU."""
import pytest
import torch

import sparse_attention_indexer_bwd_gb300 as ibwd


def host_inputs(B=1, S_q=8, S_k=8, H=4, D=32, topk=4):
    q = torch.zeros((B, S_q, H, D), dtype=torch.bfloat16)
    k = torch.zeros((B, S_k, D), dtype=torch.bfloat16)
    w = torch.zeros((B, S_q, H))
    I = torch.zeros((B, S_q, topk))
    attn = torch.zeros((B, S_q, topk))
    idx = torch.zeros((B, S_q, topk), dtype=torch.int32)
    dq = torch.zeros((B, S_q, H, D))
    dw = torch.zeros((B, S_q, H))
    dk = torch.zeros((B, S_k, D))
    return q, k, w, I, attn, idx, dq, dw, dk


def test_host_tensors_are_refused_by_every_backward_form():
    q, k, w, I, attn, idx, dq, dw, dk = host_inputs()
    with pytest.raises(ValueError):
        ibwd.indexer_bwd(q, k, w, I, attn, idx, dq, dw, dk)
    with pytest.raises(ValueError):
        ibwd.indexer_bwd_ex(q, k, w, I, attn, idx, dq, dw, dk)
    with pytest.raises(ValueError):
        ibwd.indexer_bwd_gemm(q, k, w, attn, idx, dq, dw, dk)
    with pytest.raises(ValueError):
        ibwd.indexer_bwd_score_grad(I, attn, idx, 8)
    with pytest.raises(ValueError):
        ibwd.indexer_fwd(q, k, w, idx)


def test_wrong_dtypes_and_ranks_are_refused():
    q, k, w, I, attn, idx, dq, dw, dk = host_inputs()
    with pytest.raises(ValueError):
        ibwd.indexer_bwd_gemm(q.float(), k, w, attn, idx, dq, dw, dk)      # q must be bf16
    with pytest.raises(ValueError):
        ibwd.indexer_bwd_gemm(q, k, w, attn, idx.long(), dq, dw, dk)       # ids must be int32
    with pytest.raises(ValueError):
        ibwd.indexer_bwd_score_grad(I[0], attn, idx, 8)                    # [B,S_q,topk]
    with pytest.raises(TypeError):
        ibwd.indexer_bwd_gemm(None, k, w, attn, idx, dq, dw, dk)           # not a tensor


def test_option_output_dtypes():
    assert ibwd._out_flag(torch.zeros(1), "dq") == 0
    assert ibwd._out_flag(torch.zeros(1, dtype=torch.bfloat16), "dq") == 1
    with pytest.raises(TypeError):
        ibwd._out_flag(torch.zeros(1, dtype=torch.float16), "dq")
