"""The seeded workload generator: shapes, determinism and the recipes'
structural promises (tables, ragged lengths, needle placement)."""
import numpy as np
import torch

from decode_sparse_attention_gb300 import synth


def test_deterministic():
    w = synth.WORKLOADS["tiny_fp32"]
    a, b = synth.make(w, seed=3), synth.make(w, seed=3)
    for k in ("q", "k_cache", "v_cache", "block_tables", "meta_block_tables"):
        assert torch.equal(a[k], b[k])
    c = synth.make(w, seed=4)
    assert not torch.equal(a["k_cache"], c["k_cache"])


def test_tables_are_permutations():
    w = synth.WORKLOADS["bf16_paged"].replace(B=3)
    x = synth.make(w, seed=0)
    bt = x["block_tables"].numpy()
    assert sorted(bt.ravel().tolist()) == list(range(x["P"]))
    assert x["k_cache"].shape == (3 * 128, 128, 8, 128) and x["k_cache"].dtype == torch.bfloat16


def test_ragged_lengths_and_pool():
    w = synth.WORKLOADS["ragged"].replace(B=16)
    L = synth.draw_seq_lens(w, np.random.default_rng(1))
    assert np.all(L % 128 == 0) and np.all(L >= w.k * w.BS) and np.all(L <= 131072)


def test_ragged_small_pool_unused_slots():
    w = synth.WORKLOADS["ragged"].replace(B=4, ragged=(200, 3000, 1), MMBPR=None, k=2)
    x = synth.make(w, seed=2)
    bt = x["block_tables"].numpy()
    for b, nb in enumerate(x["nb"]):
        assert np.all(bt[b, :nb] >= 0) and np.all(bt[b, nb:] == -1)
    used = sorted(bt[bt >= 0].tolist())
    assert used == list(range(x["P"]))


def test_needle_not_in_forced_window():
    w = synth.WORKLOADS["tiny_fp32"]
    for seed in range(20):
        x = synth.make(w, seed=seed)
        _, j, tok = x["needle"]
        assert 1 <= j <= x["nb"][0] - 2
        p = int(x["block_tables"][0, j])
        assert torch.equal(x["k_cache"][p, tok, 0], 3.0 * x["q"][0, 0])


def test_probe_needle_at_probe_offset_and_importance():
    w = synth.WORKLOADS["probe_importance"]
    x = synth.make(w, seed=0)
    _, j, tok = x["needle"]
    assert j == 64 and tok % (w.BS // w.n_probe) == 0
    imp = x["importance"].numpy()
    assert abs(imp.sum() - 1.0) < 1e-4 and np.all(imp >= 0)


def test_window_metadata_lengths():
    w = synth.WORKLOADS["long_context"].replace(B=1)
    x = synth.make(w, seed=5)
    t = x["t"]
    assert 0 <= t < 128
    assert int(x["meta_seq_lens"][0]) == 128 * ((65536 - t) // 128)
