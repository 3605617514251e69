"""The seeded input generators hold the structure the input recipe states:
distinct causal ids with tail padding, uniform-length rows over all keys,
local-window rows, normalised targets, and reproducibility per seed."""
import numpy as np

import synth


def test_causal_ids_are_distinct_causal_and_tail_padded():
    B, S_q, S_k, topk = 2, 96, 48, 20
    idx = synth.topk_causal(3, 4, B, S_q, S_k, topk)
    for b in range(B):
        for t in range(S_q):
            row = idx[b, t]
            n = min(t * S_k // S_q, S_k - 1) + 1        # keys [0, floor(t*S_k/S_q)]
            m = min(n, topk)
            assert np.all(row[m:] == -1) and np.all(row[:m] >= 0) and np.all(row[:m] < n)
            assert len(set(row[:m].tolist())) == m


def test_uniform_ids_fill_every_slot_from_all_keys():
    B, S_q, S_k, topk = 1, 64, 100, 40
    idx = synth.topk_uniform(5, 4, B, S_q, S_k, topk)
    assert idx.min() >= 0 and idx.max() < S_k
    for row in idx[0]:
        assert len(set(row.tolist())) == topk
    # the rows use the whole key range, not a causal prefix
    assert idx[0, 0].max() > S_k // 2


def test_window_ids_concentrate_in_the_local_window():
    B, S_q, S_k, topk = 1, 256, 1024, 64
    idx = synth.topk_window(7, 4, B, S_q, S_k, topk, window=32)
    t = S_q - 1
    c = t * S_k // S_q
    row = idx[0, t]
    assert np.all(row >= 0) and np.all(row <= c)
    assert np.sum(row > c - 32) >= topk // 2          # half the slots from the window


def test_targets_are_distributions_over_the_valid_slots():
    idx = synth.topk_causal(1, 4, 1, 40, 30, 12)
    attn = synth.target_sparse(1, 5, idx, 30)
    valid = idx >= 0
    assert np.all(attn[valid] > 0)
    np.testing.assert_allclose(np.where(valid, attn, 0).sum(-1), 1.0, rtol=1e-5)


def test_generators_are_reproducible_per_seed():
    wl = synth.WORKLOADS["tiny"]
    a, b = synth.make_inputs(wl), synth.make_inputs(wl)
    for key in a:
        assert np.array_equal(a[key], b[key])
    u1 = synth.topk_uniform(11, 4, 1, 8, 50, 10)
    u2 = synth.topk_uniform(12, 4, 1, 8, 50, 10)
    assert not np.array_equal(u1, u2)


def test_sweep_workloads_are_registered():
    for k in (128, 256, 384, 512, 640, 1024, 1536, 2048):
        wl = synth.WORKLOADS[f"uniform_topk{k}"]
        assert (wl.S_q, wl.S_k, wl.H, wl.D, wl.topk, wl.ids) == (8192, 4096, 64, 128, k, "uniform")
