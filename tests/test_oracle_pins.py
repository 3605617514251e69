"""Pins for the fp64 oracle, independent of the oracle itself.

Each check comes from the mathematics or a hand-derived closed form, chosen
so that a plausible slip in the oracle (a dropped term, a wrong sign, a
transposed operand, a wrong index or padding rule) fails at least one:

* hand-derived closed-form case (tests/golden/hand_case.json);
* central finite differences of the KL loss (score-grad) and of the linear
  functional L = sum dI * I(q, k, w) (gemm stage, at logit scales 1, 0.37 and
  0.0884), with loss functions written here, never calling the oracle's
  gradient code;
* homogeneity: <dW,w> = <dQ,q> = <dK,k> = sum dI*I (I is positively
  1-homogeneous in each of q, k, w);
* row invariants of dI (sums to zero; padding is exactly zero; one valid slot
  or uniform rows give exactly zero);
* special cases: all z < 0, w = 0, 2*dI, dense == sparse with every causal
  key selected, -1 vs positive out-of-range padding.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_case.json")


def f32_to_bf16_bits(x):
    x = np.asarray(x, np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16(bits):
    return synth.bf16_to_f32(bits).astype(np.float64)


def small_case(seed=11, B=1, S_q=24, S_k=20, H=3, D=8, topk=7):
    q = synth.normal_bf16(seed, 1, (B, S_q, H, D))
    k = synth.normal_bf16(seed, 2, (B, S_k, D))
    w = synth.normal_f32(seed, 3, (B, S_q, H), 0.0, 0.7)
    idx = synth.topk_causal(seed, 4, B, S_q, S_k, topk)
    attn = synth.target_sparse(seed, 5, idx, S_k)
    return q, k, w, idx, attn


# ---------------------------------------------------------------- golden ---

def test_golden_gemm_hand_case():
    g = json.load(open(GOLDEN))["gemm"]
    q = f32_to_bf16_bits(np.array(g["q"], np.float32)[None])
    k = f32_to_bf16_bits(np.array(g["k"], np.float32)[None])
    w = np.array(g["w"], np.float32)[None]
    idx = np.array(g["idx"], np.int32)[None]
    dI = np.array(g["dI"], np.float64)[None]
    I = oracle.forward_sparse(q, k, w, idx, g["S_k"])
    np.testing.assert_array_equal(I[0], np.array(g["I"]))
    dq, dw, dk = oracle.gemm_sparse(q, k, w, dI, idx, g["S_k"])
    np.testing.assert_array_equal(dw[0], np.array(g["dW"]))
    np.testing.assert_array_equal(dq[0], np.array(g["dQ"]))
    np.testing.assert_array_equal(dk[0], np.array(g["dK"]))


def test_golden_score_grad_hand_case():
    g = json.load(open(GOLDEN))["score_grad"]
    conv = lambda v: [[float("nan") if x == "nan" else x for x in r] for r in v]
    I = np.array(conv(g["index_score"]), np.float32)[None]
    a = np.array(g["attn_score"], np.float32)[None]
    idx = np.array(g["idx"], np.int32)[None]
    dI = oracle.score_grad_sparse(I, a, idx, g["S_k"], g["grad_scale"])
    exp = np.array(g["dI"])
    assert np.all(dI[0, 0] == 0.0)
    assert dI[0, 1, 2] == 0.0
    np.testing.assert_allclose(dI[0, 1, :2], exp[1, :2], rtol=1e-14, atol=0)


# ------------------------------------------------------------ score-grad ---

def kl_loss(I, a, valid, S_q, grad_scale):
    """-(g/S_q) sum_t sum_valid ahat log softmax_valid(I) -- the KL loss up to
    a term constant in I; written independently of the oracle."""
    L = 0.0
    for t in range(I.shape[0]):
        v = valid[t]
        if not v.any():
            continue
        x = I[t][v]
        m = x.max()
        lse = m + math.log(np.exp(x - m).sum())
        A = a[t][v].sum()
        ah = a[t][v] / A
        L -= (grad_scale / S_q) * float((ah * (x - lse)).sum())
    return L


@pytest.mark.parametrize("grad_scale", [1.0, 0.5, 1.5])
def test_score_grad_matches_finite_differences(grad_scale):
    q, k, w, idx, attn = small_case(seed=3)
    S_k = 20
    I32 = synth.normal_f32(7, 9, idx.shape, 0.0, 1.5)
    dI = oracle.score_grad_sparse(I32, attn, idx, S_k, grad_scale)[0]
    I = I32[0].astype(np.float64)
    a = attn[0].astype(np.float64)
    valid = (idx[0] >= 0) & (idx[0] < S_k)
    S_q = I.shape[0]
    rng = np.random.default_rng(0)
    h = 1e-6
    picks = [(t, j) for t in range(S_q) for j in range(idx.shape[-1]) if valid[t, j]]
    for n in rng.choice(len(picks), 40, replace=False):
        t, j = picks[n]
        # only row t depends on I[t, j]; evaluating that row keeps the
        # finite-difference rounding noise small
        Ip = I[t:t + 1].copy(); Ip[0, j] += h
        Im = I[t:t + 1].copy(); Im[0, j] -= h
        lp = kl_loss(Ip, a[t:t + 1], valid[t:t + 1], S_q, grad_scale)
        lm = kl_loss(Im, a[t:t + 1], valid[t:t + 1], S_q, grad_scale)
        fd = (lp - lm) / (2 * h)
        assert abs(fd - dI[t, j]) <= 1e-7 * abs(dI[t, j]) + 1e-10, (t, j, fd, dI[t, j])


def test_score_grad_row_invariants():
    q, k, w, idx, attn = small_case(seed=5, S_q=40, S_k=40, topk=9)
    S_k = 40
    I32 = synth.normal_f32(1, 9, idx.shape, 0.0, 2.0)
    dI = oracle.score_grad_sparse(I32, attn, idx, S_k)
    valid = (idx >= 0) & (idx < S_k)
    # rows sum to zero (sum p = sum ahat = 1)
    assert np.abs(dI.sum(-1)).max() <= 1e-15 * np.abs(dI).max() * idx.shape[-1]
    # padded slots are exactly zero
    assert np.all(dI[~valid] == 0.0)
    # a row with exactly one valid slot is exactly zero
    one = valid.sum(-1) == 1
    assert one.any() and np.all(dI[one] == 0.0)


def test_score_grad_uniform_rows_are_zero():
    S_q, topk, S_k = 5, 8, 100
    idx = np.tile(np.arange(topk, dtype=np.int32), (1, S_q, 1))
    idx[0, 2, 3] = -1
    idx[0, 4, 0] = 500  # positive out-of-range id: padding
    I = np.full((1, S_q, topk), 0.75, np.float32)
    a = np.ones((1, S_q, topk), np.float32)
    dI = oracle.score_grad_sparse(I, a, idx, S_k)
    assert np.all(dI == 0.0)


def test_score_grad_padding_ignores_garbage_and_oob():
    q, k, w, idx, attn = small_case(seed=8, S_q=30, S_k=30, topk=10)
    S_k = 30
    I32 = synth.normal_f32(2, 9, idx.shape)
    base = oracle.score_grad_sparse(I32, attn, idx, S_k)
    pad = idx < 0
    assert pad.any()
    idx2 = idx.copy()
    idx2[pad] = S_k + np.arange(pad.sum(), dtype=np.int32) % 9999
    I2 = I32.copy(); I2[pad] = np.nan
    a2 = attn.copy(); a2[pad] = 0.123
    got = oracle.score_grad_sparse(I2, a2, idx2, S_k)
    np.testing.assert_array_equal(got, base)


# ------------------------------------------------------------ gemm stage ---

def np_forward(q, k, w, idx, S_k, sm_scale=1.0):
    """The forward written with numpy for the finite-difference loss."""
    B, S_q, H, D = q.shape
    I = np.zeros(idx.shape)
    for b in range(B):
        for t in range(S_q):
            for j in range(idx.shape[-1]):
                s = idx[b, t, j]
                if 0 <= s < S_k:
                    z = sm_scale * (q[b, t] @ k[b, s])
                    I[b, t, j] = float(np.sum(w[b, t] * np.maximum(z, 0.0)))
    return I


@pytest.mark.parametrize("sm_scale", [1.0, 0.37, 0.0884])
def test_forward_and_gemm_match_finite_differences(sm_scale):
    q16, k16, w, idx, attn = small_case(seed=13, S_q=10, S_k=9, H=3, D=5, topk=6)
    S_k = 9
    dI = synth.normal_f32(4, 9, idx.shape).astype(np.float64)
    dI[(idx < 0)] = 0.0
    q, k, w64 = bf16(q16), bf16(k16), w.astype(np.float64)
    # the oracle's forward agrees with the numpy forward
    np.testing.assert_allclose(oracle.forward_sparse(q16, k16, w, idx, S_k, sm_scale),
                               np_forward(q, k, w64, idx, S_k, sm_scale), rtol=1e-13, atol=1e-13)
    dq, dw, dk = oracle.gemm_sparse(q16, k16, w, dI, idx, S_k, sm_scale)
    L = lambda q_, k_, w_: float(np.sum(dI * np_forward(q_, k_, w_, idx, S_k, sm_scale)))
    h = 1e-6
    rng = np.random.default_rng(1)

    def kink_free(qq, kk):
        z = np.einsum("btd,bsd->bts", qq.reshape(1, -1, qq.shape[-1]), kk)
        return np.abs(z).min() > 1e-4

    checked = 0
    for which, arr, grad in (("q", q, dq), ("k", k, dk), ("w", w64, dw)):
        for flat in rng.choice(arr.size, 25, replace=False):
            pos = np.unravel_index(flat, arr.shape)
            ap = arr.copy(); ap[pos] += h
            am = arr.copy(); am[pos] -= h
            args_p = {"q": q, "k": k, "w": w64}; args_p[which] = ap
            args_m = {"q": q, "k": k, "w": w64}; args_m[which] = am
            if which in ("q", "k") and not (kink_free(args_p["q"], args_p["k"]) and
                                             kink_free(args_m["q"], args_m["k"])):
                continue
            fd = (L(args_p["q"], args_p["k"], args_p["w"]) - L(args_m["q"], args_m["k"], args_m["w"])) / (2 * h)
            g = grad[pos]
            assert abs(fd - g) <= 1e-6 * max(1.0, abs(g)), (which, pos, fd, g)
            checked += 1
    assert checked >= 50


def test_homogeneity_invariant():
    q16, k16, w, idx, attn = small_case(seed=21, S_q=48, S_k=40, H=4, D=16, topk=12)
    S_k = 40
    I = oracle.forward_sparse(q16, k16, w, idx, S_k)
    dI = oracle.score_grad_sparse(I.astype(np.float32), attn, idx, S_k)
    dq, dw, dk = oracle.gemm_sparse(q16, k16, w, dI, idx, S_k)
    L = float(np.sum(dI * I))
    for v in (np.sum(dw * w), np.sum(dq * bf16(q16)), np.sum(dk * bf16(k16))):
        assert abs(v - L) <= 1e-12 * max(abs(L), np.abs(dI).sum() * np.abs(I).max())


def test_all_negative_logits_give_zero_row():
    q16, k16, w, idx, attn = small_case(seed=2, S_q=16, S_k=16, H=2, D=8, topk=5)
    S_k = 16
    q = bf16(q16); k = bf16(k16)
    k = np.abs(k) + 0.0625                 # k > 0 entrywise
    q[0, 7] = -np.abs(q[0, 7]) - 0.0625    # q[7] < 0 entrywise, so every z of row 7 < 0
    q16 = f32_to_bf16_bits(q.astype(np.float32)); k16 = f32_to_bf16_bits(k.astype(np.float32))
    dI = synth.normal_f32(3, 9, idx.shape).astype(np.float64)
    dq, dw, dk = oracle.gemm_sparse(q16, k16, w, dI, idx, S_k)
    assert np.all(dq[0, 7] == 0.0) and np.all(dw[0, 7] == 0.0)
    # and row 7 contributes nothing to dK: zero its dI and dK is unchanged
    dI2 = dI.copy(); dI2[0, 7] = 0.0
    np.testing.assert_array_equal(oracle.gemm_sparse(q16, k16, w, dI2, idx, S_k)[2], dk)


def test_zero_weights_and_linearity():
    q16, k16, w, idx, attn = small_case(seed=4, S_q=20, S_k=18, H=3, D=8, topk=6)
    S_k = 18
    dI = synth.normal_f32(3, 9, idx.shape).astype(np.float64)
    dq, dw, dk = oracle.gemm_sparse(q16, k16, np.zeros_like(w), dI, idx, S_k)
    assert np.all(dq == 0.0) and np.all(dk == 0.0) and np.abs(dw).max() > 0
    a = oracle.gemm_sparse(q16, k16, w, dI, idx, S_k)
    b = oracle.gemm_sparse(q16, k16, w, 2.0 * dI, idx, S_k)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(2.0 * x, y)


def test_gemm_padding_equivalence():
    q16, k16, w, idx, attn = small_case(seed=9, S_q=26, S_k=26, H=3, D=8, topk=8)
    S_k = 26
    dI = synth.normal_f32(5, 9, idx.shape).astype(np.float64)
    pad = idx < 0
    dI0 = dI.copy(); dI0[pad] = 0.0
    base = oracle.gemm_sparse(q16, k16, w, dI0, idx, S_k)
    idx2 = idx.copy(); idx2[pad] = S_k + 3
    dI2 = dI.copy(); dI2[pad] = 0.123      # nonzero grad on padded slots is ignored
    got = oracle.gemm_sparse(q16, k16, w, dI2, idx2, S_k)
    for x, y in zip(base, got):
        np.testing.assert_array_equal(x, y)


def test_rows_variant_matches_full():
    q16, k16, w, idx, attn = small_case(seed=6, B=2, S_q=20, S_k=18, H=3, D=8, topk=6)
    S_k = 18
    dI = synth.normal_f32(3, 9, idx.shape).astype(np.float64)
    dq, dw, dk = oracle.gemm_sparse(q16, k16, w, dI, idx, S_k)
    rows = np.array([0, 5, 19, 20, 33, 39])
    dqr, dwr = oracle.gemm_sparse_rows(q16, k16, w, dI.reshape(-1, 6)[rows], idx, S_k, rows)
    np.testing.assert_array_equal(dqr, dq.reshape(-1, 3, 8)[rows])
    np.testing.assert_array_equal(dwr, dw.reshape(-1, 3)[rows])


@pytest.mark.parametrize("sm_scale", [1.0, 0.5])
def test_dense_equals_sparse_with_every_causal_key(sm_scale):
    S, H, D = 24, 3, 8
    sc = dict(sm_scale=sm_scale)
    q16 = synth.normal_bf16(1, 1, (1, S, H, D)); k16 = synth.normal_bf16(1, 2, (1, S, D))
    w = synth.normal_f32(1, 3, (1, S, H))
    idx = np.where(np.arange(S)[None, :] <= np.arange(S)[:, None], np.arange(S)[None, :], -1)
    idx = idx.astype(np.int32)[None]
    I_s = oracle.forward_sparse(q16, k16, w, idx, S, **sc)
    I_d = oracle.forward_dense(q16, k16, w, **sc)
    np.testing.assert_array_equal(I_s, I_d)
    a = synth.target_dense(1, 5, 1, S)
    dI_s = oracle.score_grad_sparse(I_s.astype(np.float32), a, idx, S)
    dI_d = oracle.score_grad_dense(I_d.astype(np.float32), a)
    np.testing.assert_array_equal(dI_s, dI_d)
    for x, y in zip(oracle.gemm_sparse(q16, k16, w, dI_s, idx, S, **sc), oracle.gemm_dense(q16, k16, w, dI_d, **sc)):
        np.testing.assert_array_equal(x, y)
    rows = np.array([0, 7, 23])
    dqr, dwr = oracle.gemm_dense_rows(q16, k16, w, dI_d.reshape(S, S)[rows], rows, **sc)
    dq, dw, _ = oracle.gemm_dense(q16, k16, w, dI_d, **sc)
    np.testing.assert_array_equal(dqr, dq[0, rows])
    np.testing.assert_array_equal(dwr, dw[0, rows])


def test_logit_scale_is_a_power_of_two_factor_on_every_output():
    # relu(s x) = s relu(x) for s > 0: with s = 2^-3 every output of the
    # scaled definitions is the unscaled one times s, exactly
    q16, k16, w, idx, attn = small_case(seed=17, S_q=30, S_k=25, H=3, D=8, topk=9)
    S_k = 25
    s = 0.125
    np.testing.assert_array_equal(oracle.forward_sparse(q16, k16, w, idx, S_k, s),
                                  s * oracle.forward_sparse(q16, k16, w, idx, S_k))
    dI = synth.normal_f32(3, 9, idx.shape).astype(np.float64)
    for x, y in zip(oracle.gemm_sparse(q16, k16, w, dI, idx, S_k, s), oracle.gemm_sparse(q16, k16, w, dI, idx, S_k)):
        np.testing.assert_allclose(x, s * y, rtol=1e-14, atol=1e-300)


def test_duplicate_ids_count_as_separate_slots():
    # a key selected twice in a row counts twice: same as two rows selecting it once
    S_k, H, D = 6, 2, 4
    q16 = synth.normal_bf16(2, 1, (1, 1, H, D)); k16 = synth.normal_bf16(2, 2, (1, S_k, D))
    w = synth.normal_f32(2, 3, (1, 1, H))
    idx = np.array([[[3, 3, 1]]], np.int32)
    dI = np.array([[[0.25, 0.5, -0.75]]])
    dq, dw, dk = oracle.gemm_sparse(q16, k16, w, dI, idx, S_k)
    idx1 = np.array([[[3, 1]]], np.int32)
    dq1, dw1, dk1 = oracle.gemm_sparse(q16, k16, w, np.array([[[0.75, -0.75]]]), idx1, S_k)
    np.testing.assert_allclose(dq, dq1, rtol=1e-15, atol=1e-17)
    np.testing.assert_allclose(dw, dw1, rtol=1e-15, atol=1e-17)
    np.testing.assert_allclose(dk, dk1, rtol=1e-15, atol=1e-17)
