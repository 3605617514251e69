"""CUDA path vs the fp64 oracle, element by element, on sizes the oracle
finishes in seconds (several 128-key tiles, ragged tails, B > 1), plus the
determinism, padding and edge-case properties of the path."""
import numpy as np
import pytest
import torch

import oracle
import synth
import sparse_attention_indexer_bwd_gb300 as ibwd
from gpu_util import (TOL_DI, assert_close, case_inputs, gemm_path, gpu_all, gpu_gemm, max_rel, oracle_all, rms_rel)

pytestmark = pytest.mark.gpu

W = synth.Workload
SMALL = [
    synth.WORKLOADS["tiny"],
    W("multi_tile_ragged", 2, 64, 128, 300, 700, 300, "causal", 11),   # 3 tiles, ragged tail, B=2
    W("window_small", 1, 64, 128, 384, 512, 256, "window", 12),        # duplicates, local window
    W("odd_shapes", 1, 7, 40, 131, 97, 53, "causal", 13),              # H, D, topk not tile multiples
    W("dense_small", 1, 64, 128, 200, 200, 0, "dense", 14),
    W("dense_odd", 2, 5, 24, 77, 77, 0, "dense", 15),
    W("dense_256", 1, 8, 64, 256, 256, 0, "dense", 16),                # staged dense score-grad rows
    W("uniform_small", 1, 16, 64, 130, 512, 256, "uniform", 17),       # uniform lengths, 2 full tiles per row
    W("rows128_b2", 2, 16, 64, 90, 300, 128, "causal", 20),            # 128-slot rows: packed score-grad rows
]


@pytest.fixture(scope="module")
def cases():
    out = {}
    for wl in SMALL:
        x = case_inputs(wl)
        out[wl.name] = (wl, x, oracle_all(wl, x))
    return out


@pytest.mark.parametrize("name", [w.name for w in SMALL])
@pytest.mark.parametrize("mode", [ibwd.IBWD_DK_ATOMIC, ibwd.IBWD_DK_DETERMINISTIC])
@pytest.mark.parametrize("path", ["whole", "pair"])
def test_full_path_matches_oracle(cases, name, mode, path):
    wl, x, ref = cases[name]
    dI, dq, dw, dk = gpu_all(wl, x, dk_mode=mode, path=path)
    assert max_rel(dI, ref[0]) <= TOL_DI
    assert_close(dq, dw, dk, ref[1:], tag=f"{name}/mode{mode}/{path}")


@pytest.mark.parametrize("name", [w.name for w in SMALL])
def test_score_grad_exact_zeros_and_rows(cases, name):
    wl, x, ref = cases[name]
    dI, _, _, _ = gpu_all(wl, x)
    if wl.dense:
        pad = np.triu(np.ones((wl.S_q, wl.S_q), bool), 1)[None].repeat(wl.B, 0)
    else:
        pad = (x["idx"] < 0) | (x["idx"] >= wl.S_k)
    assert np.all(dI[pad] == 0.0)
    # rows sum to ~0 (p and ahat are both probability rows)
    assert np.abs(dI.astype(np.float64).sum(-1)).max() <= 1e-5 * np.abs(ref[0]).max() * 8


@pytest.mark.parametrize("name", ["multi_tile_ragged", "dense_small"])
def test_gemm_only_matches_oracle_on_same_dI(cases, name):
    wl, x, _ = cases[name]
    dI = (oracle.score_grad_dense(x["I"], x["attn"]) if wl.dense else
          oracle.score_grad_sparse(x["I"], x["attn"], x["idx"], wl.S_k)).astype(np.float32)
    ref = (oracle.gemm_dense(x["q"], x["k"], x["w"], dI.astype(np.float64)) if wl.dense else
           oracle.gemm_sparse(x["q"], x["k"], x["w"], dI.astype(np.float64), x["idx"], wl.S_k))
    for mode in (ibwd.IBWD_DK_ATOMIC, ibwd.IBWD_DK_DETERMINISTIC):
        dq, dw, dk = gpu_gemm(wl, x, dI, mode)
        assert_close(dq, dw, dk, ref, tag=f"{name} gemm-only mode{mode}")


@pytest.mark.parametrize("name", ["multi_tile_ragged", "window_small", "dense_small", "dense_256"])
def test_whole_call_equals_the_pair_of_calls(cases, name):
    # indexer_bwd runs the same two kernels: dI, dq, dw and the
    # deterministic dK are bitwise those of the two calls
    wl, x, _ = cases[name]
    a = gpu_all(wl, x, dk_mode=ibwd.IBWD_DK_DETERMINISTIC, path="whole")
    b = gpu_all(wl, x, dk_mode=ibwd.IBWD_DK_DETERMINISTIC, path="pair")
    for u, v in zip(a, b):
        assert np.array_equal(u.view(np.int32), v.view(np.int32))


@pytest.mark.parametrize("shape", [(24, 70000, 512, "uniform", 0), (12, 40960, 4200, "uniform", 1),
                                   (40, 3000, 700, "window", 1)])
def test_union_pass_windows_and_wide_rows(shape):
    # The gemm stage takes four query rows at a time against the union of
    # their keys, built per window of at most 32768 keys (4096 when a row has
    # more than 4096 slots): S_k = 70000 needs three windows, topk = 4200 ten;
    # the local-window rows repeat keys within a row (summed per key).  Both
    # against the oracle; the deterministic ones bitwise run to run.
    S_q, S_k, topk, ids, mode = shape
    wl = W(f"union_{S_k}_{topk}", 1, 4, 32, S_q, S_k, topk, ids, 23)
    x = case_inputs(wl)
    ref = oracle_all(wl, x)
    runs = [gpu_all(wl, x, dk_mode=mode) for _ in range(2)]
    assert_close(*runs[0][1:], ref[1:], tag=f"union {shape}")
    assert np.array_equal(runs[0][1], runs[1][1]) and np.array_equal(runs[0][2], runs[1][2])
    if mode == ibwd.IBWD_DK_DETERMINISTIC:
        assert np.array_equal(runs[0][3].view(np.int32), runs[1][3].view(np.int32))


@pytest.mark.parametrize("name", ["multi_tile_ragged", "window_small", "dense_small", "dense_256"])
def test_whole_call_equals_the_pair_of_calls(cases, name):
    # indexer_bwd runs the same two kernels: dI, dq, dw and the
    # deterministic dK are bitwise those of the two calls
    wl, x, _ = cases[name]
    a = gpu_all(wl, x, dk_mode=ibwd.IBWD_DK_DETERMINISTIC, path="whole")
    b = gpu_all(wl, x, dk_mode=ibwd.IBWD_DK_DETERMINISTIC, path="pair")
    for u, v in zip(a, b):
        assert np.array_equal(u.view(np.int32), v.view(np.int32))


@pytest.mark.parametrize("mode", [ibwd.IBWD_DK_ATOMIC, ibwd.IBWD_DK_DETERMINISTIC])
def test_dk_across_a_wide_dynamic_range(mode):
    # Rows 0..191 select keys below 160 only and carry dI at 2^-24 of the
    # other rows', which select keys from 256 up; the dz scale is per block,
    # so the small rows' keys keep their own relative accuracy, element by
    # element, in both dK modes.
    wl = W("fixed_range", 1, 8, 64, 512, 512, 64, "causal", 29)
    x = case_inputs(wl)
    rng = np.random.default_rng(29)
    small = np.arange(wl.S_q) < 192
    idx = np.where(small[:, None], rng.integers(0, 160, (wl.S_q, wl.topk)),
                   rng.integers(256, wl.S_k, (wl.S_q, wl.topk))).astype(np.int32)[None]
    x["idx"] = idx
    x["I"] = oracle.forward_sparse(x["q"], x["k"], x["w"], idx, wl.S_k).astype(np.float32)
    dI = oracle.score_grad_sparse(x["I"], x["attn"], idx, wl.S_k).astype(np.float32)
    dI[0, small] *= np.float32(2.0 ** -24)
    ref = oracle.gemm_sparse(x["q"], x["k"], x["w"], dI.astype(np.float64), idx, wl.S_k)
    dq, dw, dk = gpu_gemm(wl, x, dI, mode, idx=idx)
    keys = np.unique(idx[0, small])
    assert keys.max() < 160 and keys.size > 100
    ks, rk = dk[0, keys], ref[2][0, keys]
    assert np.abs(ks - rk).max() <= 1e-3 * np.abs(rk).max()
    assert_close(dq, dw, dk, ref, tag="wide range")


@pytest.mark.parametrize("mode", [ibwd.IBWD_DK_ATOMIC, ibwd.IBWD_DK_DETERMINISTIC])
def test_dk_with_large_q_and_dI(mode):
    # q entries near the fp16 limit and a large dI: the fp16 operands and the
    # dz scale keep every value in range, the results within the tolerance
    wl = W("fixed_large", 1, 16, 64, 200, 300, 96, "causal", 30)
    x = case_inputs(wl)
    q = synth.bf16_to_f32(x["q"]).astype(np.float32)
    q[0, 7, 3, :8] = 60000.0
    x["q"] = f32_to_bf16_bits(q)
    dI = (oracle.score_grad_sparse(x["I"], x["attn"], x["idx"], wl.S_k) * 1e6).astype(np.float32)
    ref = oracle.gemm_sparse(x["q"], x["k"], x["w"], dI.astype(np.float64), x["idx"], wl.S_k)
    dq, dw, dk = gpu_gemm(wl, x, dI, mode)
    assert_close(dq, dw, dk, ref, tag="large q and dI")


def f32_to_bf16_bits(x):
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


@pytest.mark.parametrize("name", ["multi_tile_ragged", "window_small", "odd_shapes", "dense_small", "dense_odd",
                                  "dense_256"])
def test_determinism(cases, name):
    wl, x, _ = cases[name]
    # the whole backward, and the pair of calls
    pr = [gpu_all(wl, x, dk_mode=ibwd.IBWD_DK_DETERMINISTIC, path="pair") for _ in range(2)]
    for a, b in zip(pr[0], pr[1]):
        assert np.array_equal(a, b)
    runs = [gpu_all(wl, x, dk_mode=ibwd.IBWD_DK_DETERMINISTIC) for _ in range(3)]
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert np.array_equal(a, b)          # dI, dq, dw, dk all bitwise
    at = [gpu_all(wl, x, dk_mode=ibwd.IBWD_DK_ATOMIC) for _ in range(2)]
    assert np.array_equal(at[0][1], at[1][1]) and np.array_equal(at[0][2], at[1][2])
    assert rms_rel(at[0][3], at[1][3]) < 1e-5   # atomic dK: fp32 jitter only
    # on the blocked kernel, dq and dw do not depend on the dK mode
    with gemm_path("blocked"):
        ab = gpu_all(wl, x, dk_mode=ibwd.IBWD_DK_ATOMIC)
    assert np.array_equal(ab[1], runs[0][1]) and np.array_equal(ab[2], runs[0][2])


def test_padding_equivalence_oob_and_garbage(cases):
    wl, x, _ = cases["multi_tile_ragged"]
    dI = oracle.score_grad_sparse(x["I"], x["attn"], x["idx"], wl.S_k).astype(np.float32)
    base = gpu_gemm(wl, x, dI, ibwd.IBWD_DK_DETERMINISTIC)
    pad = x["idx"] < 0
    assert pad.any()
    idx2 = x["idx"].copy()
    idx2[pad] = wl.S_k + (np.arange(pad.sum()) % 9999)       # positive out-of-range ids
    dI2 = dI.copy()
    dI2[pad] = np.float32(0.123)                              # nonzero grad on padded slots
    got = gpu_gemm(wl, x, dI2, ibwd.IBWD_DK_DETERMINISTIC, idx=idx2)
    for a, b in zip(base, got):
        assert np.array_equal(a, b)
    # score-grad: NaN logits and garbage targets on padded slots are ignored
    x2 = dict(x)
    x2["idx"] = idx2
    x2["I"] = x["I"].copy()
    x2["I"][pad] = np.nan
    x2["attn"] = x["attn"].copy()
    x2["attn"][pad] = 7.0
    a1 = gpu_all(wl, x)
    a2 = gpu_all(wl, x2)
    assert np.array_equal(a1[0], a2[0]) and np.array_equal(a1[1], a2[1]) and np.array_equal(a1[2], a2[2])


def test_padding_anywhere_in_row(cases):
    # padding slots shuffled into the middle of rows (not only at the tail)
    wl, x, _ = cases["multi_tile_ragged"]
    rng = np.random.default_rng(3)
    idx = x["idx"].copy()
    for b in range(wl.B):
        for t in range(wl.S_q):
            rng.shuffle(idx[b, t])
    x2 = dict(x)
    x2["idx"] = idx
    x2["I"] = oracle.forward_sparse(x["q"], x["k"], x["w"], idx, wl.S_k).astype(np.float32)
    x2["attn"] = synth.target_sparse(5, 5, idx, wl.S_k)
    ref = oracle_all(wl, x2)
    dI, dq, dw, dk = gpu_all(wl, x2)
    assert max_rel(dI, ref[0]) <= TOL_DI
    assert_close(dq, dw, dk, ref[1:], tag="shuffled padding")


def test_linearity_power_of_two(cases):
    wl, x, _ = cases["multi_tile_ragged"]
    dI = oracle.score_grad_sparse(x["I"], x["attn"], x["idx"], wl.S_k).astype(np.float32)
    a = gpu_gemm(wl, x, dI, ibwd.IBWD_DK_DETERMINISTIC)
    b = gpu_gemm(wl, x, 2.0 * dI, ibwd.IBWD_DK_DETERMINISTIC)
    for u, v in zip(a, b):
        assert np.array_equal(2.0 * u, v)


@pytest.mark.parametrize("grad_scale", [0.5, 1.5])
def test_grad_scale(cases, grad_scale):
    wl, x, _ = cases["odd_shapes"]
    ref = oracle_all(wl, x, grad_scale)
    dI, dq, dw, dk = gpu_all(wl, x, grad_scale=grad_scale)
    assert max_rel(dI, ref[0]) <= TOL_DI
    assert_close(dq, dw, dk, ref[1:], tag=f"grad_scale {grad_scale}")


def test_edge_rows_empty_single_and_all_negative():
    # rows with no valid slot, one valid slot, and all-negative logits
    wl = W("edges", 1, 16, 64, 40, 50, 20, "causal", 21)
    x = synth.make_inputs(wl)
    idx = x["idx"].copy()
    idx[0, 5] = -1                     # empty row
    idx[0, 6] = -1
    idx[0, 6, 3] = 17                  # single valid slot
    idx[0, 7] = 10**6                  # only positive out-of-range ids: empty
    q = synth.bf16_to_f32(x["q"]).copy()
    k = synth.bf16_to_f32(x["k"]).copy()
    k[:] = np.abs(k) + 0.0625          # k > 0
    q[0, 9] = -np.abs(q[0, 9]) - 0.0625  # every z of row 9 is negative
    from test_oracle_pins import f32_to_bf16_bits
    x["q"] = f32_to_bf16_bits(q)
    x["k"] = f32_to_bf16_bits(k)
    x["idx"] = idx
    x["attn"] = synth.target_sparse(9, 5, idx, wl.S_k)
    x["I"] = oracle.forward_sparse(x["q"], x["k"], x["w"], idx, wl.S_k).astype(np.float32)
    ref = oracle_all(wl, x)
    dI, dq, dw, dk = gpu_all(wl, x)
    for r in (5, 6, 7):
        assert np.all(dI[0, r] == 0.0) and np.all(dq[0, r] == 0.0) and np.all(dw[0, r] == 0.0)
    assert np.all(dq[0, 9] == 0.0) and np.all(dw[0, 9] == 0.0)
    assert_close(dq, dw, dk, ref[1:], tag="edges")


def test_topk_one_and_tiny_heads():
    wl = W("topk1", 2, 1, 8, 33, 9, 1, "causal", 22)
    x = case_inputs(wl)
    ref = oracle_all(wl, x)
    dI, dq, dw, dk = gpu_all(wl, x)
    # one slot per row: dI is exactly zero, so every gradient is exactly zero
    assert np.all(dI == 0.0) and np.all(dq == 0.0) and np.all(dw == 0.0) and np.all(dk == 0.0)
    assert np.all(ref[0] == 0.0)


def test_abi_rejects_bad_arguments_before_launch():
    lib = ibwd.load()
    d = torch.zeros(64, device="cuda")
    p = d.data_ptr()
    # misaligned pointer, host pointer, bad shapes, short workspace
    assert lib.indexer_bwd_score_grad(p + 4, p, p, 1, 1, 1, 4, 1.0, None, 0, None) == ibwd.IBWD_ERR_INVALID_ARG
    host = torch.zeros(64)
    assert lib.indexer_bwd_score_grad(host.data_ptr(), p, p, 1, 1, 1, 4, 1.0, None, 0, None) == \
        ibwd.IBWD_ERR_INVALID_ARG
    assert lib.indexer_bwd_score_grad(p, p + 256, p, 0, 1, 1, 4, 1.0, None, 0, None) == ibwd.IBWD_ERR_INVALID_ARG
    assert lib.indexer_bwd_gemm(p, p, p, p, p, p, p, p, 1, 1, 1, 65, 128, 4, 0, p, 10**6, None) == \
        ibwd.IBWD_ERR_UNSUPPORTED
    assert lib.indexer_bwd_gemm(p, p, p, p, p, p, p, p, 1, 1, 1, 4, 12, 4, 0, p, 10**6, None) == \
        ibwd.IBWD_ERR_UNSUPPORTED
    assert lib.indexer_bwd_gemm(p, p, p, p, p, p, p, p, 1, 1, 1, 4, 32, 4, 0, p, 16, None) == \
        ibwd.IBWD_ERR_WORKSPACE
    assert lib.indexer_bwd_gemm(p, p, p, p, p, p, p, p, 1, 1, 1, 4, 32, 4, 7, p, 10**6, None) == \
        ibwd.IBWD_ERR_INVALID_ARG
    before = d.clone()
    torch.cuda.synchronize()
    assert torch.equal(d, before)
    assert ibwd.indexer_bwd_last_device_status() == ibwd.IBWD_OK


def test_two_host_threads_two_streams(cases):
    # concurrent calls from two host threads, each on its own stream with its
    # own workspace and outputs, give the single-call results (dq, dw and the
    # deterministic dK bitwise)
    import threading
    wl, x, _ = cases["multi_tile_ragged"]
    ref = gpu_all(wl, x, dk_mode=ibwd.IBWD_DK_DETERMINISTIC)
    results = [None, None]

    def work(slot):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            results[slot] = gpu_all(wl, x, dk_mode=ibwd.IBWD_DK_DETERMINISTIC)
        s.synchronize()

    ts = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    for got in results:
        assert got is not None
        for a, b in zip(got, ref):
            assert np.array_equal(a.view(np.int32), b.view(np.int32))
