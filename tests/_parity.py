"""Comparison rules shared by the GPU parity tests.

Selection: where floating point decides the set, the oracle's fp32 scores
decide what is unique.  Index sets must be identical wherever the oracle's gap
between the last taken and the first left-out candidate exceeds 1e-4
relative; inside that band any GPU pick is accepted if its oracle score is
within the band of the boundary score (several answers are correct there).
Scores: |gpu - ref| <= 1e-5 * max(|ref|, sum_d |max-term_d|).
"""
import numpy as np
import torch

import oracle
from _common import to_np

SEL_GAP = 1e-4
SCORE_TOL = 1e-5


def rel_gap(a, b):
    return abs(a - b) / max(abs(a), abs(b), 1e-30)


def check_one_selection(g_row, o_row, scores, nb, k, fixed, what="", band=SEL_GAP):
    """g_row/o_row: [k] selections (ascending, -1 pad); scores: oracle fp32
    scores [nb]; fixed: bool [nb] of blocks chosen regardless of score."""
    g_row = np.asarray(g_row)
    o_row = np.asarray(o_row)
    g_set = [int(j) for j in g_row if j >= 0]
    # shape: ascending, distinct, -1 padded, count min(k, nb)
    assert len(g_set) == min(k, nb), (what, g_row, o_row)
    assert g_set == sorted(set(g_set)), (what, g_row)
    assert np.all(g_row[len(g_set):] == -1), (what, g_row)
    assert all(0 <= j < nb for j in g_set), (what, g_row)
    if np.array_equal(g_row, o_row):
        return True
    fixed_idx = set(np.flatnonzero(fixed).tolist())
    assert fixed_idx <= set(g_set), (what, "fixed blocks missing", g_row, fixed_idx)
    cand = [j for j in range(nb) if j not in fixed_idx]
    order = sorted(cand, key=lambda j: (-scores[j], j))
    want = min(k - len(fixed_idx), len(cand))
    if want == len(cand) or want == 0:
        raise AssertionError((what, "sets must match", g_row, o_row))
    s_in, s_out = float(scores[order[want - 1]]), float(scores[order[want]])
    assert rel_gap(s_in, s_out) <= band, (what, "clear gap but different sets", g_row, o_row,
                                           s_in, s_out)
    width = 2 * band * max(abs(s_in), abs(s_out), 1e-30)
    for j in set(g_set) - fixed_idx:
        assert scores[j] >= s_in - width, (what, "pick below the tie band", j, scores[j], s_in)
    for j in cand:
        if scores[j] > s_in + width:
            assert j in g_set, (what, "clearly better block left out", j, scores[j], s_in)
    return False


def check_scores(g_scores, o_scores, o_abs, what=""):
    g = np.asarray(g_scores, np.float64)
    tol = SCORE_TOL * np.maximum(np.abs(o_scores), o_abs)
    err = np.abs(g - o_scores)
    bad = err > tol + 1e-30
    assert not bad.any(), (what, float(err[bad].max()), float(tol[bad].min()))
    return float((err / np.maximum(tol, 1e-30)).max()) if err.size else 0.0


def quest_reference(x, w, q_dt=None):
    """Oracle chain a1..a5 on the host copies of a workload: returns
    (maxblocks, minblocks, selected, fp32 scores, double scores, abs sums)."""
    kv_dt = {torch.float32: oracle.F32, torch.bfloat16: oracle.BF16, torch.float16: oracle.F16}[x["k_cache"].dtype]
    q_dt = q_dt if q_dt is not None else {torch.float32: oracle.F32, torch.bfloat16: oracle.BF16,
                                          torch.float16: oracle.F16}[x["q"].dtype]
    mx = to_np(x["maxblocks"]).copy()
    mn = to_np(x["minblocks"]).copy()
    oracle.prefill_metadata(to_np(x["k_cache"]), kv_dt, to_np(x["meta_seq_lens"]),
                            to_np(x["block_tables"]), to_np(x["meta_block_tables"]), mx, mn)
    sel, sf = oracle.quest_select(to_np(x["q"]), q_dt, mx, mn, kv_dt, to_np(x["meta_block_tables"]),
                                  to_np(x["seq_lens"]), w.N, w.k, x["t"])
    qg = oracle.group_mean_query(to_np(x["q"]), q_dt, w.N)
    sd, sa = oracle.quest_scores(qg, mx, mn, kv_dt, to_np(x["meta_block_tables"]), to_np(x["seq_lens"]))
    return mx, mn, sel, sf, sd, sa


def forced_flags(L, BS, t, nb):
    return oracle.forced_set(int(L), BS, t, nb)


def check_quest_rows(w, x, gsel, osel, osf, what=""):
    """The gap rule on every (request, KV head) row of a Quest selection;
    returns how many rows equal the oracle's exactly."""
    L = to_np(x["seq_lens"])
    exact = 0
    for b in range(gsel.shape[0]):
        nb = x["nb"][b]
        fixed = forced_flags(L[b], w.BS, x["t"], nb)
        for n in range(w.N):
            exact += check_one_selection(gsel[b, n], osel[b, n], osf[b, n, :nb], nb, w.k, fixed,
                                         (what, b, n))
    return exact


def probe_fixed(w, nb, oimp_row, n_imp):
    """Blocks a probe selection holds regardless of the probe scores: the
    importance picks (bit-exact fp32 sums) and, once a probe pick exists,
    the most recent block."""
    imp_picks = sorted(range(nb), key=lambda j: (-oimp_row[j], j))[:n_imp] if n_imp else []
    fixed = np.zeros(nb, bool)
    fixed[imp_picks] = True
    if w.k > n_imp and nb > n_imp:
        fixed[nb - 1] = True
    return fixed


def check_probe_rows(w, x, gsel, osel, oprobe, oimp, onimp, what=""):
    """The gap rule on every (request, query head) row of a probe selection
    (bit-exact for int8 caches, whose probe scores are exact integer dots)."""
    exact = 0
    for b in range(gsel.shape[0]):
        nb = x["nb"][b]
        for h in range(w.H):
            if w.kv_dtype == "i8":
                assert np.array_equal(gsel[b, h], osel[b, h]), (what, b, h)
                exact += 1
                continue
            fixed = probe_fixed(w, nb, oimp[b], int(onimp[b, h]))
            exact += check_one_selection(gsel[b, h], osel[b, h], oprobe[b, h, :nb], nb, w.k,
                                         fixed, (what, b, h))
    return exact


def oracle_attention(x, w, sel):
    """The oracle's attention over a given selection ([B, N or H, k])."""
    return oracle.sparse_attention(to_np(x["q"]), DT_OF[x["q"].dtype], to_np(x["k_cache"]),
                                   to_np(x["v_cache"]), DT_OF[x["k_cache"].dtype],
                                   to_np(x["block_tables"]), to_np(x["seq_lens"]),
                                   np.ascontiguousarray(sel, np.int32), w.N,
                                   k_scale=to_np(x["k_scale"]) if "k_scale" in x else None,
                                   v_scale=to_np(x["v_scale"]) if "v_scale" in x else None)


DT_OF = {torch.float32: oracle.F32, torch.bfloat16: oracle.BF16, torch.float16: oracle.F16,
         torch.int8: oracle.I8}
