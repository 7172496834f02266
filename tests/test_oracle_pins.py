"""Pins of the oracle to facts fixed by the pages and by the mathematics:
hand-worked examples (tests/golden), closed forms, invariants, brute force and
library routines (torch.amax/amin, sorting, torch SDPA in fp64).

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong tie rule) fails it.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from _common import from_bits, odt, to_np
from decode_sparse_attention_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def ragged_case(dtype, seed=0, B=3, N=2, D=5, BS=4, seq_lens=(0, 5, 13), MKBPR=4, MMBPR=2):
    g = torch.Generator().manual_seed(seed)
    P = B * MKBPR + 3
    k = torch.randn((P, BS, N, D), generator=g).to(dtype)
    bt = torch.randperm(P, generator=g)[:B * MKBPR].reshape(B, MKBPR).to(torch.int32)
    M = B * MMBPR + 2
    mbt = torch.randperm(M, generator=g)[:B * MMBPR].reshape(B, MMBPR).to(torch.int32)
    sl = torch.tensor(seq_lens, dtype=torch.int32)
    return k, bt, mbt, sl, M


# --------------------------------------------------------------------------
# a1 metadata
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_metadata_equals_torch_amax_amin(dtype):
    BS = 4
    k, bt, mbt, sl, M = ragged_case(dtype, BS=BS, seq_lens=(0, 5, 13), MKBPR=4, MMBPR=2)
    N, D = k.shape[2], k.shape[3]
    sentinel = torch.full((M, BS, N, D), 7.0, dtype=dtype)
    mx, mn = to_np(sentinel).copy(), to_np(sentinel).copy()
    oracle.prefill_metadata(to_np(k), odt(k), to_np(sl), to_np(bt), to_np(mbt), mx, mn)
    mx_t, mn_t = from_bits(mx, dtype), from_bits(mn, dtype)
    touched = torch.zeros(M, BS, dtype=torch.bool)
    for b, L in enumerate(sl.tolist()):
        nb = (L + BS - 1) // BS
        for ms in range((nb + BS - 1) // BS):
            m = int(mbt[b, ms])
            for r in range(BS):
                j = ms * BS + r
                touched[m, r] = True
                if j >= nb:   # absent block: zero metadata
                    assert torch.all(mx_t[m, r] == 0) and torch.all(mn_t[m, r] == 0)
                    continue
                valid = min(BS, L - j * BS)
                toks = k[int(bt[b, j]), :valid].float()          # [valid, N, D]
                assert torch.equal(mx_t[m, r].float(), torch.amax(toks, dim=0))
                assert torch.equal(mn_t[m, r].float(), torch.amin(toks, dim=0))
    # rows of meta blocks no request uses are left alone
    assert torch.all(mx_t[~touched] == 7.0) and torch.all(mn_t[~touched] == 7.0)
    assert touched.sum() == BS * 2   # request 1: 1 meta block, request 2: 1, request 0: none


def test_metadata_signed_zero_reading():
    """-0 sorts below +0: max of {-0,+0} is +0, min is -0 (bits checked)."""
    k = torch.tensor([-0.0, 0.0, -0.0], dtype=torch.float32).reshape(1, 3, 1, 1)
    mx = np.full((1, 3, 1, 1), 5, np.float32)
    mn = mx.copy()
    oracle.prefill_metadata(k.numpy(), oracle.F32, np.array([3], np.int32),
                            np.array([[0]], np.int32), np.array([[0]], np.int32), mx, mn)
    assert mx[0, 0, 0, 0] == 0 and not np.signbit(mx[0, 0, 0, 0])
    assert mn[0, 0, 0, 0] == 0 and np.signbit(mn[0, 0, 0, 0])
    assert np.all(mx[0, 1:] == 0) and np.all(mn[0, 1:] == 0)   # absent blocks 1, 2


def test_metadata_rejects_bad_table_entry():
    k, bt, mbt, sl, M = ragged_case(torch.float32)
    bt = bt.clone()
    bt[1, 0] = 10 ** 6
    mx = np.zeros((M, 4, 2, 5), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.prefill_metadata(to_np(k), oracle.F32, to_np(sl), to_np(bt), to_np(mbt), mx, mx.copy())


# --------------------------------------------------------------------------
# f1 incremental metadata update
# --------------------------------------------------------------------------

UPD_PREV, UPD_NEW = (0, 3, 13, 8), (0, 9, 21, 8)   # BS=4: empty, in-block, new meta block, no growth


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_metadata_update_rows_against_torch(dtype):
    """Rows of blocks [prev // BS, ceil(L / BS)) hold the amax/amin of the
    blocks' valid tokens at the new lengths, rows past the block count inside
    the meta blocks begun since prev are zero, and every other row keeps what
    it held (planted values: neither recomputed nor re-zeroed)."""
    BS = 4
    k, bt, mbt, sl, M = ragged_case(dtype, B=4, BS=BS, seq_lens=UPD_NEW, MKBPR=6, MMBPR=2)
    N, D = k.shape[2], k.shape[3]
    prev = torch.tensor(UPD_PREV, dtype=torch.int32)
    planted = torch.full((M, BS, N, D), 3.0, dtype=dtype)
    mx, mn = to_np(planted).copy(), to_np(planted).copy()
    oracle.update_metadata(to_np(k), odt(k), to_np(prev), to_np(sl), to_np(bt), to_np(mbt), mx, mn)
    mx_t, mn_t = from_bits(mx, dtype), from_bits(mn, dtype)
    for b, (P0, L) in enumerate(zip(UPD_PREV, UPD_NEW)):
        nb = (L + BS - 1) // BS
        zero_from = (((P0 + BS - 1) // BS + BS - 1) // BS) * BS   # end of meta blocks in use
        for j in range(((nb + BS - 1) // BS) * BS):
            m, r = int(mbt[b, j // BS]), j % BS
            if j < P0 // BS or (nb <= j < zero_from):
                assert torch.all(mx_t[m, r] == 3.0) and torch.all(mn_t[m, r] == 3.0), (b, j)
            elif j >= nb:
                assert torch.all(mx_t[m, r] == 0) and torch.all(mn_t[m, r] == 0), (b, j)
            else:
                toks = k[int(bt[b, j]), :min(BS, L - j * BS)].float()
                assert torch.equal(mx_t[m, r].float(), torch.amax(toks, dim=0)), (b, j)
                assert torch.equal(mn_t[m, r].float(), torch.amin(toks, dim=0)), (b, j)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_metadata_update_after_prefill_equals_prefill_at_new_lengths(dtype):
    BS = 4
    k, bt, mbt, sl, M = ragged_case(dtype, seed=3, B=4, BS=BS, seq_lens=UPD_NEW, MKBPR=6, MMBPR=2)
    N, D = k.shape[2], k.shape[3]
    prev = np.array(UPD_PREV, np.int32)
    sent = to_np(torch.full((M, BS, N, D), 7.0, dtype=dtype))
    mx, mn = sent.copy(), sent.copy()
    oracle.prefill_metadata(to_np(k), odt(k), prev, to_np(bt), to_np(mbt), mx, mn)
    oracle.update_metadata(to_np(k), odt(k), prev, to_np(sl), to_np(bt), to_np(mbt), mx, mn)
    fx, fn = sent.copy(), sent.copy()
    oracle.prefill_metadata(to_np(k), odt(k), to_np(sl), to_np(bt), to_np(mbt), fx, fn)
    assert np.array_equal(mx, fx) and np.array_equal(mn, fn)
    # idempotent: an update with no new token rebuilds the partial last block only
    oracle.update_metadata(to_np(k), odt(k), to_np(sl), to_np(sl), to_np(bt), to_np(mbt), mx, mn)
    assert np.array_equal(mx, fx) and np.array_equal(mn, fn)


def test_metadata_update_rejects_shrinking_lengths():
    k, bt, mbt, sl, M = ragged_case(torch.float32, B=4, seq_lens=UPD_NEW, MKBPR=6, MMBPR=2)
    mx = np.zeros((M, 4, 2, 5), np.float32)
    prev = np.array([0, 10, 13, 8], np.int32)          # 10 > 9
    with pytest.raises(oracle.OracleError):
        oracle.update_metadata(to_np(k), oracle.F32, prev, to_np(sl), to_np(bt), to_np(mbt), mx,
                               mx.copy())


# --------------------------------------------------------------------------
# a2, a3: group mean and Quest score
# --------------------------------------------------------------------------

def test_quest_score_hand_example():
    gd = golden("quest_score_hand.json")
    q = np.array([gd["q_heads"]], np.float32)                    # [1, H=2, D=2]
    qg = oracle.group_mean_query(q, oracle.F32, N=1)
    assert np.array_equal(qg[0, 0], gd["expected_qg"])
    mx = np.array(gd["max_row"], np.float32).reshape(1, 1, 1, 2)
    mn = np.array(gd["min_row"], np.float32).reshape(1, 1, 1, 2)
    sc, ab = oracle.quest_scores(qg, mx, mn, oracle.F32, np.array([[0]], np.int32),
                                 np.array([1], np.int32))
    assert sc[0, 0, 0] == gd["expected_score"]
    assert ab[0, 0, 0] == 11.0


def test_group_mean_is_contiguous_grouping():
    """q-head h belongs to KV head h // (H/N): a library mean over contiguous
    groups, and a swapped grouping would give different numbers."""
    g = torch.Generator().manual_seed(3)
    q = torch.rand((2, 8, 6), generator=g) * 2 - 1
    qg = oracle.group_mean_query(q.numpy(), oracle.F32, N=2)
    ref = q.double().reshape(2, 2, 4, 6).mean(dim=2).numpy()
    assert np.allclose(qg, ref, rtol=0, atol=1e-15)
    wrong = q.double().reshape(2, 4, 2, 6).permute(0, 2, 1, 3).mean(dim=2).numpy()
    assert not np.allclose(qg, wrong)


def _meta_and_scores(seed, dtype=torch.float32, q=None, B=2, H=4, N=2, D=8, BS=4, L=(13, 16)):
    k, bt, mbt, sl, M = ragged_case(dtype, seed=seed, B=B, N=N, D=D, BS=BS, seq_lens=L,
                                    MKBPR=4, MMBPR=1)
    mx = np.zeros((M, BS, N, D), to_np(k).dtype)
    mn = mx.copy()
    oracle.prefill_metadata(to_np(k), odt(k), to_np(sl), to_np(bt), to_np(mbt), mx, mn)
    if q is None:
        g = torch.Generator().manual_seed(seed + 100)
        q = torch.rand((B, H, D), generator=g) * 2 - 1
    qg = oracle.group_mean_query(q.numpy(), oracle.F32, N)
    sc, ab = oracle.quest_scores(qg, mx, mn, odt(k), to_np(mbt), to_np(sl))
    return k, bt, sl, qg, sc, mx, mn, mbt


@pytest.mark.parametrize("seed", range(5))
def test_quest_score_is_upper_bound(seed):
    """Every valid token's qg.k is at most its block's score."""
    k, bt, sl, qg, sc, *_ = _meta_and_scores(seed)
    BS, N = k.shape[1], k.shape[2]
    for b, L in enumerate(sl.tolist()):
        for j in range((L + BS - 1) // BS):
            valid = min(BS, L - j * BS)
            for n in range(N):
                toks = k[int(bt[b, j]), :valid, n].double().numpy()
                dots = toks @ qg[b, n]
                assert dots.max() <= sc[b, n, j] + 1e-12
                if valid == 1:   # a one-token block: the bound is the exact dot
                    assert np.isclose(sc[b, n, j], dots[0], rtol=0, atol=1e-12)


def test_quest_score_closed_forms():
    """qg >= 0: s = qg.M;  qg <= 0: s = qg.m;  zero metadata: s = 0."""
    B, H, N, D = 2, 4, 2, 8
    g = torch.Generator().manual_seed(11)
    qpos = torch.rand((B, H, D), generator=g)
    k, bt, sl, qg, sc, mx, mn, mbt = _meta_and_scores(4, q=qpos, B=B, H=H, N=N, D=D)
    BS = k.shape[1]
    for sign, table in ((1, mx), (-1, mn)):
        qg_s = sign * qg
        sc_s, _ = oracle.quest_scores(qg_s, mx, mn, oracle.F32, to_np(mbt), to_np(sl))
        for b, L in enumerate(sl.tolist()):
            for j in range((L + BS - 1) // BS):
                row = table[int(mbt[b, j // BS]), j % BS]             # [N, D]
                for n in range(N):
                    assert np.isclose(sc_s[b, n, j], float(qg_s[b, n] @ row[n].astype(np.float64)),
                                      rtol=0, atol=1e-12)
    zero = np.zeros_like(mx)
    sc0, _ = oracle.quest_scores(qg, zero, zero, oracle.F32, to_np(mbt), to_np(sl))
    for b, L in enumerate(sl.tolist()):
        assert np.all(sc0[b, :, :(L + BS - 1) // BS] == 0)


# --------------------------------------------------------------------------
# a4, a5: forced window and deterministic top-k
# --------------------------------------------------------------------------

def test_forced_window_hand_cases():
    for c in golden("forced_window.json")["cases"]:
        nb = (c["seq_len"] + c["BS"] - 1) // c["BS"]
        f = oracle.forced_set(c["seq_len"], c["BS"], c["t"], nb)
        assert np.flatnonzero(f).tolist() == c["forced"], c


def _select_from_scores(scores, k, t=-1, L=None, BS=1):
    """Drive the oracle's Quest select with prescribed block scores: D=1,
    q=1, max=min=score, one request, one KV head, BS rows per meta block."""
    nb = len(scores)
    L = nb * BS if L is None else L
    MMBPR = (nb + BS - 1) // BS
    mx = np.zeros((MMBPR, BS, 1, 1), np.float32)
    for j, s in enumerate(scores):
        mx[j // BS, j % BS, 0, 0] = s
    q = np.ones((1, 1, 1), np.float32)
    sel, sf = oracle.quest_select(q, oracle.F32, mx, mx.copy(), oracle.F32,
                                  np.arange(MMBPR, dtype=np.int32)[None], np.array([L], np.int32),
                                  N=1, k=k, t=t)
    return sel[0, 0], sf[0, 0, :nb]


@pytest.mark.parametrize("seed", range(20))
def test_topk_matches_full_sort(seed):
    rng = np.random.default_rng(seed)
    nb = int(rng.integers(1, 40))
    k = int(rng.integers(1, 12))
    scores = rng.integers(-5, 6, size=nb).astype(np.float32) * 0.5     # many exact ties
    sel, _ = _select_from_scores(scores, k)
    order = sorted(range(nb), key=lambda j: (-scores[j], j))[:k]        # library sort
    expect = sorted(order) + [-1] * (k - min(k, nb))
    assert sel.tolist() == expect


def test_topk_ties_go_to_lower_index():
    sel, _ = _select_from_scores(np.array([1, 3, 3, 3, 2], np.float32), 2)
    assert sel.tolist() == [1, 2]


def test_k_above_block_count_pads():
    sel, _ = _select_from_scores(np.array([0.5, -1.0, 2.0], np.float32), 5)
    assert sel.tolist() == [0, 1, 2, -1, -1]


def test_window_blocks_forced_even_with_lowest_scores():
    scores = np.array([-100, 5, 4, 3, 2, 1, -100, -100], np.float32)
    # BS=2, L=16 (8 blocks), t=3: w0 = min(floor(13/2), 7) = 6 -> window {6,7}, sink {0}
    sel, _ = _select_from_scores(scores, 5, t=3, L=16, BS=2)
    assert sel.tolist() == [0, 1, 2, 6, 7]
    with pytest.raises(oracle.OracleError):
        _select_from_scores(scores, 2, t=3, L=16, BS=2)     # |F| = 3 > k


@pytest.mark.parametrize("seed", range(10))
def test_planted_needle_always_selected(seed):
    w = synth.WORKLOADS["tiny_fp32"]
    x = synth.make(w, seed=seed)
    mx, mn = to_np(x["maxblocks"]).copy(), to_np(x["minblocks"]).copy()
    oracle.prefill_metadata(to_np(x["k_cache"]), oracle.F32, to_np(x["meta_seq_lens"]),
                            to_np(x["block_tables"]), to_np(x["meta_block_tables"]), mx, mn)
    sel, _ = oracle.quest_select(to_np(x["q"]), oracle.F32, mx, mn, oracle.F32,
                                 to_np(x["meta_block_tables"]), to_np(x["seq_lens"]),
                                 N=w.N, k=w.k, t=x["t"])
    _, j, _ = x["needle"]
    for n in range(w.N):
        assert j in sel[0, n].tolist()
        assert 0 in sel[0, n].tolist() and (x["nb"][0] - 1) in sel[0, n].tolist()


def test_quest_select_deterministic():
    w = synth.WORKLOADS["tiny_fp32"]
    x = synth.make(w, seed=1)
    mx, mn = to_np(x["maxblocks"]).copy(), to_np(x["minblocks"]).copy()
    oracle.prefill_metadata(to_np(x["k_cache"]), oracle.F32, to_np(x["meta_seq_lens"]),
                            to_np(x["block_tables"]), to_np(x["meta_block_tables"]), mx, mn)
    a = oracle.quest_select(to_np(x["q"]), oracle.F32, mx, mn, oracle.F32,
                            to_np(x["meta_block_tables"]), to_np(x["seq_lens"]), w.N, w.k, 0)
    b = oracle.quest_select(to_np(x["q"]), oracle.F32, mx, mn, oracle.F32,
                            to_np(x["meta_block_tables"]), to_np(x["seq_lens"]), w.N, w.k, 0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1], equal_nan=True)


# --------------------------------------------------------------------------
# a6..a8 probe / importance selector
# --------------------------------------------------------------------------

def _probe_case(q, ktok, BS, n_probe, k, importance=None):
    """One request, one KV head, D=len(q); K tokens laid out block by block."""
    D = len(q)
    ktok = np.asarray(ktok, np.float32).reshape(-1, D)
    L = ktok.shape[0]
    nb = (L + BS - 1) // BS
    kc = np.zeros((nb, BS, 1, D), np.float32)
    for t in range(L):
        kc[t // BS, t % BS, 0] = ktok[t]
    imp = None if importance is None else np.asarray(importance, np.float32)[None]
    return oracle.probe_select(np.asarray(q, np.float32).reshape(1, 1, D), oracle.F32, kc,
                               oracle.F32, np.arange(nb, dtype=np.int32)[None],
                               np.array([L], np.int32), N=1, k=k, n_probe=n_probe,
                               importance=imp)


def test_probe_select_hand_example():
    gd = golden("probe_select_hand.json")
    for c in gd["cases"]:
        sel, probe, imps, nimp = _probe_case(gd["q"], gd["k_tokens"], gd["BS"], gd["n_probe"],
                                             c["k"], gd["importance"] if c["importance"] else None)
        assert sel[0, 0].tolist() == c["selected"], c
        assert int(nimp[0, 0]) == c["n_imp"], c
        assert np.array_equal(probe[0, 0], np.float32(gd["expected_probe"]))
        if c["importance"]:
            assert np.array_equal(imps[0], np.float32(gd["expected_imp_sum"]))


def test_probe_select_tie_readings():
    gd = golden("probe_select_ties.json")
    for c in gd["cases"]:
        sel, *_ = _probe_case(gd["q"], gd["k_tokens"], gd["BS"], gd["n_probe"], c["k"])
        assert sel[0, 0].tolist() == c["selected"], c


def test_probe_offsets_hand_cases():
    gd = golden("probe_offsets.json")
    BS = gd["BS"]
    for c in gd["cases"]:
        v = c["valid"]
        # block 0 full and dull (all zero), block 1 holds v tokens with K[t] = t + 1
        toks = [[0.0, 0.0]] * BS + [[t + 1.0, 0.0] for t in range(v)]
        _, probe, _, _ = _probe_case([1.0, 0.0], toks, BS, gd["n_probe"], 1)
        assert probe[0, 0, 1] == c["probe"], c
        assert probe[0, 0, 0] == 0.0


def test_probe_needle_at_offset_found_and_between_offsets_missed():
    BS, n_probe = 32, 8
    base = np.zeros((3 * BS, 4), np.float32)
    found = base.copy(); found[BS + 8, 0] = 50.0        # offset 8 is probed
    missed = base.copy(); missed[BS + 9, 0] = 50.0      # offset 9 is not
    _, p1, _, _ = _probe_case([1, 0, 0, 0], found, BS, n_probe, 1)
    _, p2, _, _ = _probe_case([1, 0, 0, 0], missed, BS, n_probe, 1)
    assert p1[0, 0, 1] == 50.0 and p2[0, 0, 1] == 0.0


def test_importance_budget_k1_and_k32():
    """Budget (k+1)/2: k=1 -> 1 importance block and no probe block;
    k=32 -> 16 + 16."""
    rng = np.random.default_rng(5)
    BS, nb = 4, 40
    toks = rng.uniform(-1, 1, size=(nb * BS, 8)).astype(np.float32)
    imp = rng.gamma(0.1, size=nb * BS).astype(np.float32)
    q = rng.uniform(-1, 1, size=8).astype(np.float32)
    sel, probe, imps, nimp = _probe_case(q, toks, BS, 2, 1, imp)
    assert int(nimp[0, 0]) == 1
    assert sel[0, 0].tolist() == [int(np.argmax(imps[0]))]          # no probe pick, no recency
    sel, probe, imps, nimp = _probe_case(q, toks, BS, 2, 32, imp)
    assert int(nimp[0, 0]) == 16
    s = sel[0, 0]
    assert len(set(s.tolist())) == 32 and np.all(s >= 0)
    imp_top16 = sorted(range(nb), key=lambda j: (-imps[0, j], j))[:16]
    assert set(imp_top16) <= set(s.tolist())


@pytest.mark.parametrize("seed", range(12))
def test_recency_kept_and_importance_never_evicted(seed):
    rng = np.random.default_rng(seed)
    BS = int(rng.integers(1, 6))
    L = int(rng.integers(1, 60))
    nb = (L + BS - 1) // BS
    k = int(rng.integers(1, 12))
    D = 4
    toks = rng.uniform(-1, 1, size=(L, D)).astype(np.float32)
    imp = rng.gamma(0.1, size=L).astype(np.float32)
    q = rng.uniform(-1, 1, size=D).astype(np.float32)
    sel, probe, imps, nimp = _probe_case(q, toks, BS, 3, k, imp)
    s = [x for x in sel[0, 0].tolist() if x >= 0]
    n_imp = int(nimp[0, 0])
    assert len(s) == min(k, nb) and len(set(s)) == len(s)
    imp_picks = sorted(range(nb), key=lambda j: (-imps[0, j], j))[:n_imp]
    assert set(imp_picks) <= set(s)
    if len(s) > n_imp:                       # at least one probe pick
        assert nb - 1 in s


# --------------------------------------------------------------------------
# a9 attention over the selected blocks
# --------------------------------------------------------------------------

def _sdpa_over(q, kc, vc, bt, L, sel_row, n, BS, scale):
    """torch SDPA (fp64, CPU) over the tokens of the listed blocks."""
    ks, vs = [], []
    for j in sel_row:
        if j < 0:
            continue
        valid = min(BS, L - j * BS)
        ks.append(kc[bt[j], :valid, n])
        vs.append(vc[bt[j], :valid, n])
    K = torch.cat(ks).double()[None, None]
    V = torch.cat(vs).double()[None, None]
    return torch.nn.functional.scaled_dot_product_attention(
        q.double()[None, None, None], K, V, scale=scale)[0, 0, 0]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_attention_all_blocks_equals_dense_sdpa(dtype):
    g = torch.Generator().manual_seed(2)
    B, H, N, D, BS = 2, 4, 2, 16, 8
    L = [37, 16]
    MKBPR = 5
    P = B * MKBPR
    kc = torch.randn((P, BS, N, D), generator=g).to(dtype)
    vc = torch.randn((P, BS, N, D), generator=g).to(dtype)
    q = (torch.rand((B, H, D), generator=g) * 2 - 1).to(dtype)
    bt = torch.randperm(P, generator=g).reshape(B, MKBPR).to(torch.int32)
    k = 5
    sel = np.full((B, N, k), -1, np.int32)
    for b in range(B):
        nb = (L[b] + BS - 1) // BS
        sel[b, :, :nb] = np.arange(nb)[::-1]          # order of the list does not matter
    out, lse = oracle.sparse_attention(to_np(q), odt(q), to_np(kc), to_np(vc), odt(kc),
                                       to_np(bt), np.array(L, np.int32), sel, N)
    scale = 1 / np.sqrt(D)
    for b in range(B):
        for h in range(H):
            ref = _sdpa_over(q[b, h], kc, vc, bt[b].tolist(), L[b], sel[b, h // 2], h // 2, BS, scale)
            assert np.allclose(out[b, h], ref.numpy(), rtol=0, atol=1e-12)
            # lse: log of the softmax normaliser over all tokens
            nb = (L[b] + BS - 1) // BS
            K = torch.cat([kc[bt[b, j], :min(BS, L[b] - j * BS), h // 2] for j in range(nb)]).double()
            logits = (K @ q[b, h].double()) * scale
            assert np.isclose(lse[b, h], torch.logsumexp(logits, 0).item(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_attention_sparse_subset_convex_hull_and_sdpa(seed):
    g = torch.Generator().manual_seed(seed)
    B, H, N, D, BS, MKBPR = 1, 4, 4, 8, 4, 6
    P = MKBPR + 2
    kc = torch.randn((P, BS, N, D), generator=g)
    vc = torch.randn((P, BS, N, D), generator=g)
    q = torch.randn((B, H, D), generator=g)
    bt = torch.randperm(P, generator=g)[:MKBPR].reshape(1, MKBPR).to(torch.int32)
    L = 22
    sel = np.array([[[5, 1, -1], [0, 2, 3], [4, -1, -1], [1, 3, 5]]], np.int32)   # per query head
    out, _ = oracle.sparse_attention(q.numpy(), oracle.F32, kc.numpy(), vc.numpy(), oracle.F32,
                                     bt.numpy(), np.array([L], np.int32), sel, N)
    for h in range(H):
        ref = _sdpa_over(q[0, h], kc, vc, bt[0].tolist(), L, sel[0, h], h, BS, 1 / np.sqrt(D))
        assert np.allclose(out[0, h], ref.numpy(), rtol=0, atol=1e-12)
        rows = torch.cat([vc[bt[0, j], :min(BS, L - j * BS), h] for j in sel[0, h] if j >= 0])
        assert np.all(out[0, h] <= rows.max(0).values.numpy() + 1e-12)
        assert np.all(out[0, h] >= rows.min(0).values.numpy() - 1e-12)


def test_attention_invariant_under_page_permutation():
    g = torch.Generator().manual_seed(9)
    B, H, N, D, BS, MKBPR = 1, 2, 1, 8, 4, 5
    kc = torch.randn((MKBPR, BS, N, D), generator=g)
    vc = torch.randn((MKBPR, BS, N, D), generator=g)
    q = torch.randn((B, H, D), generator=g)
    sel = np.array([[[4, 0, 2]]], np.int32)
    L = np.array([19], np.int32)
    bt = np.arange(MKBPR, dtype=np.int32)[None]
    out1, lse1 = oracle.sparse_attention(q.numpy(), 0, kc.numpy(), vc.numpy(), 0, bt, L, sel, N)
    perm = torch.randperm(MKBPR, generator=g)
    kc2, vc2 = torch.empty_like(kc), torch.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    out2, lse2 = oracle.sparse_attention(q.numpy(), 0, kc2.numpy(), vc2.numpy(), 0,
                                         perm.numpy().astype(np.int32)[None], L, sel, N)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def test_attention_empty_selection_and_errors():
    kc = np.zeros((2, 4, 1, 4), np.float32)
    q = np.ones((1, 1, 4), np.float32)
    bt = np.array([[0, 1]], np.int32)
    L = np.array([8], np.int32)
    out, lse = oracle.sparse_attention(q, 0, kc, kc, 0, bt, L, np.full((1, 1, 2), -1, np.int32), 1)
    assert np.all(out == 0) and lse[0, 0] == -np.inf
    with pytest.raises(oracle.OracleError):   # duplicate block in one row
        oracle.sparse_attention(q, 0, kc, kc, 0, bt, L, np.array([[[1, 1]]], np.int32), 1)
    with pytest.raises(oracle.OracleError):   # block beyond the sequence
        oracle.sparse_attention(q, 0, kc, kc, 0, bt, L, np.array([[[2, -1]]], np.int32), 1)


def test_quantize_query_half_even():
    gd = golden("quantize_query.json")
    q8, s = oracle.quantize_query(np.array(gd["q"], np.float32))
    assert s == gd["s_q"] and q8.tolist() == gd["q8"]
    q8, s = oracle.quantize_query(np.zeros(4, np.float32))
    assert s == 0.0 and q8.tolist() == [0, 0, 0, 0]


def test_attention_int8_equals_dequantised_sdpa():
    """The int8 path is the fp path on dequantised values: q8*s_q, k8*s_k,
    v8*s_v (the integer dot is exact)."""
    g = torch.Generator().manual_seed(4)
    B, H, N, D, BS, MKBPR = 1, 4, 2, 16, 8, 3
    k8 = torch.randint(-127, 128, (MKBPR, BS, N, D), generator=g).to(torch.int8)
    v8 = torch.randint(-127, 128, (MKBPR, BS, N, D), generator=g).to(torch.int8)
    ks = torch.rand((MKBPR, BS, N), generator=g) / 127 + 0.001
    vs = torch.rand((MKBPR, BS, N), generator=g) / 127 + 0.001
    q = torch.rand((B, H, D), generator=g) * 2 - 1
    bt = np.arange(MKBPR, dtype=np.int32)[None]
    L = 20
    sel = np.array([[[2, 0, -1], [1, 2, 0]]], np.int32)
    out, _ = oracle.sparse_attention(q.numpy(), 0, k8.numpy(), v8.numpy(), oracle.I8, bt,
                                     np.array([L], np.int32), sel, N, k_scale=ks.numpy(),
                                     v_scale=vs.numpy())
    kd = k8.double() * ks.double()[..., None]
    vd = v8.double() * vs.double()[..., None]
    for h in range(H):
        q8, s_q = oracle.quantize_query(q[0, h].numpy())
        qd = torch.from_numpy(q8.astype(np.float64)) * s_q
        ref = _sdpa_over(qd, kd, vd, bt[0].tolist(), L, sel[0, h // 2], h // 2, BS, 1 / np.sqrt(D))
        assert np.allclose(out[0, h], ref.numpy(), rtol=0, atol=1e-12)


def test_probe_int8_score_is_scaled_integer_dot():
    """int8 probe score = (s_q*s_k) * sum(q8*k8), each product rounded to fp32."""
    rng = np.random.default_rng(1)
    D, BS = 16, 4
    k8 = rng.integers(-127, 128, size=(2, BS, 1, D)).astype(np.int8)
    ks = rng.uniform(0.001, 0.01, size=(2, BS, 1)).astype(np.float32)
    q = rng.uniform(-1, 1, size=(1, 1, D)).astype(np.float32)
    sel, probe, _, _ = oracle.probe_select(q, oracle.F32, k8, oracle.I8,
                                           np.array([[0, 1]], np.int32), np.array([8], np.int32),
                                           N=1, k=1, n_probe=4, k_scale=ks)
    q8, s_q = oracle.quantize_query(q[0, 0])
    for j in range(2):
        dots = [np.float32(np.float32(s_q) * ks[j, t, 0]) *
                np.float32(int(np.dot(q8.astype(np.int64), k8[j, t, 0].astype(np.int64))))
                for t in range(BS)]
        assert probe[0, 0, j] == max(dots)


# --------------------------------------------------------------------------
# f3 prefill importance
# --------------------------------------------------------------------------

def prefill_case(dtype, seed=0, B=2, H=4, N=2, D=16, BS=8, lens=(29, 0), S_max=32, zero_q=False):
    """Paged prefill: K in a shuffled page pool, queries [B, S_max, H, D]."""
    g = torch.Generator().manual_seed(seed)
    MKBPR = (S_max + BS - 1) // BS
    P = B * MKBPR + 2
    if dtype == torch.int8:
        kc = torch.randint(-127, 128, (P, BS, N, D), generator=g).to(torch.int8)
        ks = torch.rand((P, BS, N), generator=g) / 127 + 0.001
        q = torch.rand((B, S_max, H, D), generator=g) * 4 - 2
    else:
        kc = torch.randn((P, BS, N, D), generator=g).to(dtype)
        ks = None
        q = (torch.rand((B, S_max, H, D), generator=g) * 4 - 2).to(dtype)
    if zero_q:
        q = torch.zeros_like(q)
    bt = torch.randperm(P, generator=g)[:B * MKBPR].reshape(B, MKBPR).to(torch.int32)
    return q, kc, ks, bt, np.array(lens, np.int32)


def gathered_keys(kc, ks, bt, b, S, n, BS):
    """K of KV head n, positions 0..S-1, in position order (fp64; int8 keys
    dequantised with their scales)."""
    rows = [kc[int(bt[b, s // BS]), s % BS, n].double() for s in range(S)]
    K = torch.stack(rows) if rows else torch.zeros((0, kc.shape[-1]), dtype=torch.float64)
    if ks is not None and S:
        K = K * torch.stack([ks[int(bt[b, s // BS]), s % BS, n].double() for s in range(S)])[:, None]
    return K


def sdpa_importance(qd, Kh, scale):
    """Column sums of the causal attention matrix through torch SDPA: with the
    values one-hot (V = I), output row i is row i of the probability matrix,
    so summing the outputs over positions and heads gives the mass each key
    received.  qd [H, S, D], Kh [H, S, D] fp64."""
    H, S, _ = qd.shape
    V = torch.eye(S, dtype=torch.float64).expand(H, S, S)
    P = torch.nn.functional.scaled_dot_product_attention(qd[None], Kh[None], V[None],
                                                         is_causal=True, scale=scale)[0]
    return P.sum(dim=(0, 1))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_prefill_importance_equals_sdpa_column_sums(dtype):
    BS, H, N, D = 8, 4, 2, 16
    q, kc, _, bt, lens = prefill_case(dtype, seed=3, H=H, N=N, D=D, BS=BS, lens=(29, 17))
    scale = 1 / np.sqrt(D)
    imp, lse = oracle.prefill_importance(to_np(q), odt(q), to_np(kc), odt(kc), to_np(bt), lens, N)
    G = H // N
    for b, S in enumerate(lens.tolist()):
        qd = q[b, :S].double().permute(1, 0, 2)                       # [H, S, D]
        Kh = torch.stack([gathered_keys(kc, None, bt, b, S, h // G, BS) for h in range(H)])
        ref = sdpa_importance(qd, Kh, scale)
        assert np.allclose(imp[b, :S], ref.numpy(), rtol=1e-12, atol=1e-12)
        assert np.all(imp[b, S:] == 0)
        # lse of each row: log-sum-exp of its causal logits (library routine)
        logits = torch.einsum("hid,hsd->his", qd, Kh) * scale
        mask = torch.ones(S, S, dtype=torch.bool).tril()
        ref_lse = torch.logsumexp(logits.masked_fill(~mask, -np.inf), dim=-1)
        assert np.allclose(lse[b, :, :S], ref_lse.numpy(), rtol=0, atol=1e-12)


def test_prefill_importance_uniform_closed_form():
    """q = 0: every row is uniform over its i+1 keys, so lse = log(i+1) and
    importance[s] = H * sum_{i=s}^{S-1} 1/(i+1)."""
    BS, H, N = 8, 6, 3
    q, kc, _, bt, lens = prefill_case(torch.float32, seed=1, H=H, N=N, BS=BS, lens=(31, 5),
                                      zero_q=True)
    imp, lse = oracle.prefill_importance(to_np(q), odt(q), to_np(kc), odt(kc), to_np(bt), lens, N)
    for b, S in enumerate(lens.tolist()):
        harm = np.array([sum(1.0 / (i + 1) for i in range(s, S)) for s in range(S)])
        assert np.allclose(imp[b, :S], H * harm, rtol=1e-13, atol=0)
        assert np.allclose(lse[b, :, :S], np.log(np.arange(1, S + 1))[None], rtol=0, atol=1e-13)


@pytest.mark.parametrize("seed", range(3))
def test_prefill_importance_mass_conservation(seed):
    """Every query row sums to one: sum_s importance = H * S; importance >= 0;
    the last token is seen only by the last query."""
    BS, H, N, D = 4, 8, 2, 8
    q, kc, _, bt, lens = prefill_case(torch.float32, seed=seed, H=H, N=N, D=D, BS=BS,
                                      lens=(23, 1), S_max=24)
    imp, lse = oracle.prefill_importance(to_np(q), odt(q), to_np(kc), odt(kc), to_np(bt), lens, N)
    for b, S in enumerate(lens.tolist()):
        assert np.isclose(imp[b].sum(), H * S, rtol=1e-13)
        assert np.all(imp[b, :S] > 0)
    # row 0 of every head attends only to key 0: lse = its own logit
    G = H // N
    K0 = kc[int(bt[0, 0]), 0].double()
    for h in range(H):
        l00 = float(q[0, 0, h].double() @ K0[h // G]) / np.sqrt(D)
        assert np.isclose(lse[0, h, 0], l00, rtol=0, atol=1e-13)


def test_prefill_importance_int8_equals_dequantised_sdpa():
    """int8 keys: the query row quantised as for decode, logits from the exact
    integer dot times s_q * s_k; equal to SDPA on the dequantised operands."""
    BS, H, N, D = 8, 4, 2, 16
    q, kc, ks, bt, lens = prefill_case(torch.int8, seed=5, H=H, N=N, D=D, BS=BS, lens=(21, 30))
    imp, _ = oracle.prefill_importance(q.numpy(), oracle.F32, kc.numpy(), oracle.I8, to_np(bt),
                                       lens, N, k_scale=ks.numpy())
    G = H // N
    for b, S in enumerate(lens.tolist()):
        qd = torch.zeros((H, S, D), dtype=torch.float64)
        for h in range(H):
            for i in range(S):
                q8, s_q = oracle.quantize_query(q[b, i, h].numpy())
                qd[h, i] = torch.from_numpy(q8.astype(np.float64)) * s_q
        Kh = torch.stack([gathered_keys(kc, ks, bt, b, S, h // G, BS) for h in range(H)])
        ref = sdpa_importance(qd, Kh, 1 / np.sqrt(D))
        assert np.allclose(imp[b, :S], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_prefill_importance_first_query_and_errors():
    """Summing only the queries from position f on leaves importance[s >= f]
    unchanged (a key is seen only by later queries); bad lengths and table
    entries are rejected."""
    BS, H, N, D = 8, 4, 2, 16
    q, kc, _, bt, lens = prefill_case(torch.float32, seed=7, H=H, N=N, D=D, BS=BS, lens=(30, 19))
    full, lse_full = oracle.prefill_importance(to_np(q), odt(q), to_np(kc), odt(kc), to_np(bt),
                                               lens, N)
    f = 12
    part, lse_part = oracle.prefill_importance(to_np(q), odt(q), to_np(kc), odt(kc), to_np(bt),
                                               lens, N, first_query=f)
    assert np.array_equal(part[:, f:], full[:, f:])
    assert np.array_equal(lse_part[:, :, f:], lse_full[:, :, f:], equal_nan=True)
    assert np.all(np.isnan(lse_part[:, :, :f]))
    with pytest.raises(oracle.OracleError):
        oracle.prefill_importance(to_np(q), odt(q), to_np(kc), odt(kc), to_np(bt),
                                  np.array([33, 0], np.int32), N)
    bad = to_np(bt).copy()
    bad[0, 1] = kc.shape[0]
    with pytest.raises(oracle.OracleError):
        oracle.prefill_importance(to_np(q), odt(q), to_np(kc), odt(kc), bad, lens, N)
