"""GPU parity: every kernel through the C ABI against the oracle, element by
element, on seeded inputs that span several tiles and ragged tails.

Tolerances: metadata bit-exact; Quest scores 1e-5 relative (to
max(|s|, sum|max-term|)); selections exact outside a 1e-4 relative score gap
(see _parity.py); attention max-abs 2e-3 for 16-bit KV caches (fp32
accumulation) and 1e-5 for fp32 and int8 caches (all arithmetic in fp32).
"""
import numpy as np
import pytest
import torch

import oracle
from _common import odt, to_np
from _parity import (check_one_selection, check_probe_rows, check_quest_rows, check_scores,
                     forced_flags, oracle_attention, quest_reference)
from decode_sparse_attention_gb300 import questsparse as qs
from decode_sparse_attention_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def attn_tol(dtype):
    return 2e-3 if dtype in (torch.bfloat16, torch.float16) else 1e-5


def to_dev(x):
    return {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in x.items()}


def sync_ok():
    torch.cuda.synchronize()
    code = qs.read_status(DEV)
    assert code == 0, qs.device_error_string(code)


# ---------------------------------------------------------------------------
# workloads: the five configurations at test sizes, plus edge variants
# ---------------------------------------------------------------------------

W = synth.WORKLOADS
QUEST_CASES = {
    "tiny_fp32": W["tiny_fp32"],
    "bf16_paged_b3": W["bf16_paged"].replace(B=3),
    "bf16_paged_b3_window": W["bf16_paged"].replace(B=3, t=0),
    "long_context_b1": W["long_context"].replace(B=1),
    "ragged_tails": W["ragged"].replace(B=5, ragged=(300, 9000, 1), MMBPR=None, k=6),
    "ragged_t77": W["ragged"].replace(B=4, ragged=(1000, 6000, 1), MMBPR=None, k=8, t=77),
    "k_above_blocks": W["bf16_paged"].replace(B=2, seq_len=700, MMBPR=None, k=9),
    "fp16_d64_bs32": W["bf16_paged"].replace(B=2, H=8, N=2, D=64, BS=32, seq_len=3000, MMBPR=None,
                                             k=12, kv_dtype="f16", q_dtype="f16"),
    "g1_fp32q": W["bf16_paged"].replace(B=2, H=8, N=8, seq_len=5000, MMBPR=None, k=5,
                                        q_dtype="f32", t=3),
    "g2_bs16": W["tiny_fp32"].replace(B=3, seq_len=777, k=7, kv_dtype="bf16", q_dtype="bf16"),
    # units of 1..3 scoring chunks: the persistent chunk-queue selector
    "ragged_multi_chunk": W["ragged"].replace(B=6, ragged=(100, 40000, 1), MMBPR=None, k=8),
    "ragged_multi_chunk_window": W["ragged"].replace(B=5, ragged=(5000, 40000, 1), MMBPR=None,
                                                     k=10, t=50),
    "fp32_d64_multi_chunk": W["tiny_fp32"].replace(B=3, seq_len=9000, k=6),
}


def make(w, seed=0, seq_lens=None):
    x = synth.make(w, seed=seed, device="cpu", seq_lens=seq_lens)
    return x, to_dev(x)


# ---------------------------------------------------------------------------
# a1 metadata
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", list(QUEST_CASES))
def test_metadata_bit_exact(name):
    w = QUEST_CASES[name]
    x, g = make(w, seed=1)
    # sentinel-filled pools: rows the kernel must not touch keep their bits
    sent = torch.full_like(x["maxblocks"], 3.0)
    x["maxblocks"], x["minblocks"] = sent.clone(), sent.clone()
    g["maxblocks"], g["minblocks"] = sent.to(DEV), sent.clone().to(DEV)
    qs.quest_prefill_metadata(g["k_cache"], g["meta_seq_lens"], g["block_tables"],
                              g["meta_block_tables"], g["maxblocks"], g["minblocks"])
    sync_ok()
    mx, mn = to_np(x["maxblocks"]).copy(), to_np(x["minblocks"]).copy()
    oracle.prefill_metadata(to_np(x["k_cache"]), odt(x["k_cache"]), to_np(x["meta_seq_lens"]),
                            to_np(x["block_tables"]), to_np(x["meta_block_tables"]), mx, mn)
    assert np.array_equal(to_np(g["maxblocks"]), mx)
    assert np.array_equal(to_np(g["minblocks"]), mn)


def test_metadata_full_size_bf16_paged():
    w = W["bf16_paged"]
    x, g = make(w, seed=0)
    qs.quest_prefill_metadata(g["k_cache"], g["meta_seq_lens"], g["block_tables"],
                              g["meta_block_tables"], g["maxblocks"], g["minblocks"])
    sync_ok()
    mx, mn = to_np(x["maxblocks"]).copy(), to_np(x["minblocks"]).copy()
    oracle.prefill_metadata(to_np(x["k_cache"]), oracle.BF16, to_np(x["meta_seq_lens"]),
                            to_np(x["block_tables"]), to_np(x["meta_block_tables"]), mx, mn)
    assert np.array_equal(to_np(g["maxblocks"]), mx) and np.array_equal(to_np(g["minblocks"]), mn)


# ---------------------------------------------------------------------------
# a2..a5 Quest select
# ---------------------------------------------------------------------------

def run_quest(w, x, g):
    qs.quest_prefill_metadata(g["k_cache"], g["meta_seq_lens"], g["block_tables"],
                              g["meta_block_tables"], g["maxblocks"], g["minblocks"])
    MMBPR = g["meta_block_tables"].shape[1]
    sel = torch.full((w.B, w.N, w.k), -5, dtype=torch.int32, device=DEV)
    scores = torch.full((w.B, w.N, MMBPR * w.BS), float("nan"), device=DEV)
    qs.quest_block_select_paged_in_out_w(g["q"], g["maxblocks"], g["minblocks"],
                                         g["meta_block_tables"], g["seq_lens"], x["t"], sel,
                                         scores=scores)
    sync_ok()
    return sel.cpu().numpy(), scores.cpu().numpy()


def compare_quest(w, x, gsel, gscores, what):
    mx, mn, osel, osf, osd, osa = quest_reference(x, w)
    L = to_np(x["seq_lens"])
    exact = 0
    for b in range(w.B):
        nb = x["nb"][b]
        fixed = forced_flags(L[b], w.BS, x["t"], nb)
        for n in range(w.N):
            check_scores(gscores[b, n, :nb], osd[b, n, :nb], osa[b, n, :nb], (what, b, n))
            exact += check_one_selection(gsel[b, n], osel[b, n], osf[b, n, :nb], nb, w.k, fixed,
                                         (what, b, n))
    return osel, exact


@pytest.mark.parametrize("name", list(QUEST_CASES))
def test_quest_select_parity(name):
    w = QUEST_CASES[name]
    for seed in range(2):
        x, g = make(w, seed=seed)
        gsel, gsc = run_quest(w, x, g)
        _, exact = compare_quest(w, x, gsel, gsc, (name, seed))
        assert exact >= 0.9 * w.B * w.N, (name, seed, exact)


@pytest.mark.parametrize("seed", range(5))
def test_quest_needle_selected(seed):
    w = W["tiny_fp32"]
    x, g = make(w, seed=seed)
    gsel, gsc = run_quest(w, x, g)
    compare_quest(w, x, gsel, gsc, ("needle", seed))
    _, j, _ = x["needle"]
    for n in range(w.N):
        assert j in gsel[0, n].tolist()


def test_quest_select_queue_empty_and_long_requests():
    """Chunk-queue selector: an empty request and a one-block request among
    multi-chunk ones; every unit is emitted once, padded with -1."""
    w = W["ragged"].replace(B=4, seq_len=None, ragged=(1, 2, 1), MMBPR=None, k=6)
    x, g = make(w, seed=3, seq_lens=[0, 30000, 77, 41000])
    gsel, gsc = run_quest(w, x, g)
    assert np.all(gsel[0] == -1) and np.all(gsel[2, :, 1:] == -1) and np.all(gsel[2, :, 0] == 0)
    _, exact = compare_quest(w, x, gsel, gsc, "queue-empty-long")
    assert exact >= 0.9 * w.B * w.N


def test_quest_select_queue_bad_length_is_reported():
    w = W["ragged"].replace(B=3, seq_len=None, ragged=(1, 2, 1), MMBPR=None, k=6)
    x, g = make(w, seed=1, seq_lens=[20000, 30000, 500])
    sl = g["seq_lens"].clone()
    sl[1] = 10 ** 8                      # more blocks than the metadata table holds
    qs.quest_prefill_metadata(g["k_cache"], g["meta_seq_lens"], g["block_tables"],
                              g["meta_block_tables"], g["maxblocks"], g["minblocks"])
    sel = torch.full((w.B, w.N, w.k), -5, dtype=torch.int32, device=DEV)
    for _ in range(2):                   # the queue counters rearm after an error too
        qs.quest_block_select_paged_in_out_w(g["q"], g["maxblocks"], g["minblocks"],
                                             g["meta_block_tables"], sl, x["t"], sel)
        torch.cuda.synchronize()
        assert qs.read_status(DEV) == 3  # QS_DEV_ESEQ_LEN
        assert torch.all(sel[1] == -1)
    gsel, gsc = run_quest(w, x, g)       # and a clean call still matches the oracle
    compare_quest(w, x, gsel, gsc, "queue-after-error")


def test_quest_select_deterministic():
    w = W["bf16_paged"].replace(B=4)
    x, g = make(w, seed=3)
    a = run_quest(w, x, g)
    b = run_quest(w, x, g)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1], equal_nan=True)


def test_quest_select_ties_lower_index():
    """Identical metadata rows everywhere: every score ties, the lowest k
    indices win."""
    w = W["bf16_paged"].replace(B=2, seq_len=128 * 40, MMBPR=None, k=8)
    x, g = make(w, seed=0)
    g["maxblocks"].fill_(0.5)
    g["minblocks"].fill_(-0.25)
    sel = torch.empty((w.B, w.N, w.k), dtype=torch.int32, device=DEV)
    qs.quest_block_select_paged_in_out(g["q"], g["maxblocks"], g["minblocks"],
                                       g["meta_block_tables"], g["seq_lens"], sel)
    sync_ok()
    assert np.all(sel.cpu().numpy() == np.arange(8, dtype=np.int32))


# ---------------------------------------------------------------------------
# a6..a8 probe / importance select
# ---------------------------------------------------------------------------

PROBE_CASES = {
    "probe_fp32": W["probe_importance"],
    "probe_i8": W["probe_importance_i8"],
    "probe_fp32_noimp_tail": W["probe_importance"].replace(importance=False, seq_len=4001, k=9),
    "probe_i8_k1": W["probe_importance_i8"].replace(k=1, seq_len=2050, needle=False,
                                                    needle_block=None),
    "probe_bf16_d64": W["probe_importance"].replace(B=3, H=8, N=4, D=64, kv_dtype="bf16",
                                                    q_dtype="bf16", seq_len=1500, k=10, n_probe=5,
                                                    needle=False, needle_block=None),
    "probe_g4": W["probe_importance"].replace(B=2, H=16, N=4, seq_len=3000, k=20, n_probe=3,
                                              needle=False, needle_block=None),
}


def run_probe(w, x, g):
    sel = torch.full((w.B, w.H, w.k), -5, dtype=torch.int32, device=DEV)
    qs.probe_select(g["q"], g["k_cache"], g["block_tables"], g["seq_lens"], w.k, w.n_probe,
                    importance=g.get("importance"), k_scale=g.get("k_scale"), selected=sel)
    sync_ok()
    return sel.cpu().numpy()


def probe_reference(w, x):
    return oracle.probe_select(to_np(x["q"]), odt(x["q"]), to_np(x["k_cache"]), odt(x["k_cache"]),
                               to_np(x["block_tables"]), to_np(x["seq_lens"]), w.N, w.k, w.n_probe,
                               importance=to_np(x["importance"]) if "importance" in x else None,
                               k_scale=to_np(x["k_scale"]) if "k_scale" in x else None)


@pytest.mark.parametrize("name", list(PROBE_CASES))
def test_probe_select_parity(name):
    w = PROBE_CASES[name]
    for seed in range(3):
        x, g = make(w, seed=seed)
        gsel = run_probe(w, x, g)
        osel, oprobe, oimp, onimp = probe_reference(w, x)
        check_probe_rows(w, x, gsel, osel, oprobe, oimp, onimp, (name, seed))
        if w.needle:
            _, j, _ = x["needle"]
            for n in range(w.N):
                assert j in gsel[0, n * w.G].tolist(), (name, seed, n)


# ---------------------------------------------------------------------------
# a9 sparse attention (selection taken from the oracle)
# ---------------------------------------------------------------------------

ATTN_CASES = dict(QUEST_CASES)
ATTN_CASES.update({k: v for k, v in PROBE_CASES.items()})


def attention_case(name, seed, per_query_head=None):
    w = ATTN_CASES[name]
    x, g = make(w, seed=seed)
    if w.mode == "quest" and not per_query_head:
        _, _, osel, *_ = quest_reference(x, w)
    else:
        osel, *_ = probe_reference(w, x) if w.mode == "probe" else (None,)
        if osel is None:
            rng = np.random.default_rng(seed)
            osel = np.full((w.B, w.H, w.k), -1, np.int32)
            for b in range(w.B):
                for h in range(w.H):
                    c = np.sort(rng.permutation(x["nb"][b])[:w.k])
                    osel[b, h, :len(c)] = c
    sel = torch.from_numpy(osel).to(DEV)
    lse = torch.full((w.B, w.H), float("nan"), device=DEV)
    out = qs.sparse_decode_attn(g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                                g["seq_lens"], sel, k_scale=g.get("k_scale"),
                                v_scale=g.get("v_scale"), lse=lse)
    sync_ok()
    oout, olse = oracle.sparse_attention(to_np(x["q"]), odt(x["q"]), to_np(x["k_cache"]),
                                         to_np(x["v_cache"]), odt(x["k_cache"]),
                                         to_np(x["block_tables"]), to_np(x["seq_lens"]), osel, w.N,
                                         k_scale=to_np(x["k_scale"]) if "k_scale" in x else None,
                                         v_scale=to_np(x["v_scale"]) if "v_scale" in x else None)
    return w, x, out.cpu().numpy(), lse.cpu().numpy(), oout, olse


@pytest.mark.parametrize("name", list(ATTN_CASES))
def test_attention_parity(name):
    for seed in range(2):
        w, x, gout, glse, oout, olse = attention_case(name, seed)
        tol = attn_tol(x["k_cache"].dtype)
        err = np.abs(gout - oout).max()
        assert err <= tol, (name, seed, err)
        fin = np.isfinite(olse)
        assert np.array_equal(fin, np.isfinite(glse))
        assert np.abs(glse[fin] - olse[fin]).max() <= max(tol, 1e-5) * 10, (name, seed)


@pytest.mark.parametrize("name", ["bf16_paged_b3", "ragged_tails", "tiny_fp32"])
def test_attention_per_query_head_selection(name):
    w, x, gout, glse, oout, olse = attention_case(name, 7, per_query_head=True)
    assert np.abs(gout - oout).max() <= attn_tol(x["k_cache"].dtype)


def test_attention_empty_and_padded_rows():
    w = W["bf16_paged"].replace(B=3, seq_len=None, ragged=(1, 2, 1), MMBPR=None, k=4)
    x, g = make(w, seed=0, seq_lens=[0, 130, 517])
    osel = np.full((3, w.N, 4), -1, np.int32)
    osel[1, :, :2] = [0, 1]
    osel[2, ::2, :1] = 4          # one partial block (5 valid tokens) for even heads
    sel = torch.from_numpy(osel).to(DEV)
    lse = torch.zeros((3, w.H), device=DEV)
    out = qs.sparse_decode_attn(g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                                g["seq_lens"], sel, lse=lse)
    sync_ok()
    oout, olse = oracle.sparse_attention(to_np(x["q"]), oracle.BF16, to_np(x["k_cache"]),
                                         to_np(x["v_cache"]), oracle.BF16,
                                         to_np(x["block_tables"]), to_np(x["seq_lens"]), osel, w.N)
    assert np.abs(out.cpu().numpy() - oout).max() <= 2e-3
    assert np.all(out.cpu().numpy()[0] == 0) and np.all(np.isneginf(lse.cpu().numpy()[0]))
    assert np.array_equal(np.isneginf(lse.cpu().numpy()), np.isneginf(olse))


def test_attention_all_blocks_equals_dense():
    """k = nb: the sparse path is dense softmax attention (checked against
    torch SDPA on the GPU in fp32 as a second, independent reference)."""
    w = W["bf16_paged"].replace(B=2, seq_len=1000, MMBPR=None, k=8)
    x, g = make(w, seed=4)
    sel = torch.arange(8, dtype=torch.int32, device=DEV).expand(w.B, w.N, 8).contiguous()
    out = qs.sparse_decode_attn(g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                                g["seq_lens"], sel)
    sync_ok()
    for b in range(w.B):
        pages = g["block_tables"][b, :8].long()
        K = g["k_cache"][pages].reshape(-1, w.N, w.D)[:1000].float()
        V = g["v_cache"][pages].reshape(-1, w.N, w.D)[:1000].float()
        K = K.repeat_interleave(w.G, dim=1).permute(1, 0, 2)
        V = V.repeat_interleave(w.G, dim=1).permute(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(
            g["q"][b].float()[:, None], K, V, scale=w.D ** -0.5)[:, 0]
        assert (out[b] - ref).abs().max().item() < 2e-3


# ---------------------------------------------------------------------------
# fused decode step
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny_fp32", "bf16_paged_b3_window", "ragged_t77", "probe_fp32",
                                  "probe_i8"])
def test_decode_step_parity(name):
    w = ATTN_CASES[name]
    x, g = make(w, seed=2)
    mode = 0 if w.mode == "quest" else 1
    if mode == 0:
        qs.quest_prefill_metadata(g["k_cache"], g["meta_seq_lens"], g["block_tables"],
                                  g["meta_block_tables"], g["maxblocks"], g["minblocks"])
    rows = w.N if mode == 0 else w.H
    sel = torch.full((w.B, rows, w.k), -5, dtype=torch.int32, device=DEV)
    out = torch.empty((w.B, w.H, w.D), dtype=torch.float32, device=DEV)
    nbytes = qs.step_workspace_bytes(mode, w.B, w.H, w.N, w.D, w.BS, w.k,
                                     MMBPR=g["meta_block_tables"].shape[1], MKBPR=x["MKBPR"])
    ws = qs.workspace(nbytes, DEV, ("step", name))
    p = qs.make_step_params(mode, g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                            g["seq_lens"], w.k, sel, out, ws, maxblocks=g.get("maxblocks"),
                            minblocks=g.get("minblocks"),
                            metadata_block_tables=g["meta_block_tables"],
                            tokens_since_metadata_update=x["t"], importance=g.get("importance"),
                            n_probe=w.n_probe, k_scale=g.get("k_scale"), v_scale=g.get("v_scale"))
    if mode == 0:
        _, _, osel, osf, *_ = quest_reference(x, w)
    else:
        osel, oprobe, oimp, onimp = probe_reference(w, x)
    for _ in range(2):   # twice: the workspace counters must rearm
        qs.sparse_decode_step(p, DEV)
        sync_ok()
        gsel = sel.cpu().numpy()
        # every row: the selection follows the gap rule, and the attention
        # equals the oracle's attention over the selection the GPU made
        if mode == 0:
            check_quest_rows(w, x, gsel, osel, osf, name)
        else:
            check_probe_rows(w, x, gsel, osel, oprobe, oimp, onimp, name)
        oout, _ = oracle_attention(x, w, gsel)
        err = np.abs(out.cpu().numpy() - oout).max()
        assert err <= attn_tol(x["k_cache"].dtype), (name, err)


# ---------------------------------------------------------------------------
# argument checks and device-side error reporting (no faults)
# ---------------------------------------------------------------------------

def test_host_validation_errors():
    w = W["bf16_paged"].replace(B=2, seq_len=1000, MMBPR=None, k=4)
    x, g = make(w, seed=0)
    sel = torch.empty((w.B, w.N, w.k), dtype=torch.int32, device=DEV)
    with pytest.raises(qs.QuestSparseError, match="invalid"):
        qs.quest_block_select_paged_in_out_w(g["q"], g["maxblocks"], g["minblocks"],
                                             g["meta_block_tables"], g["seq_lens"], 400, sel)
    bad = torch.empty((w.B, w.H, 96), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(qs.QuestSparseError):
        qs.sparse_decode_attn(bad, g["k_cache"], g["v_cache"], g["block_tables"], g["seq_lens"], sel)
    with pytest.raises(qs.QuestSparseError):
        qs.quest_prefill_metadata(g["k_cache"].cpu(), g["meta_seq_lens"], g["block_tables"],
                                  g["meta_block_tables"], g["maxblocks"], g["minblocks"])


def test_device_errors_are_reported_and_recoverable():
    w = W["bf16_paged"].replace(B=2, seq_len=1000, MMBPR=None, k=4)
    x, g = make(w, seed=0)
    bt = g["block_tables"].clone()
    bt[1, 3] = 10 ** 6                       # physical page out of range
    sel = torch.tensor([[[0, 3, -1, -1]] * w.N] * w.B, dtype=torch.int32, device=DEV)
    qs.sparse_decode_attn(g["q"], g["k_cache"], g["v_cache"], bt, g["seq_lens"], sel)
    torch.cuda.synchronize()
    assert qs.read_status(DEV) == 1          # QS_DEV_EBLOCK_TABLE, then reset
    sl = g["seq_lens"].clone()
    sl[0] = 10 ** 7                          # seq_len beyond the table
    qs.quest_prefill_metadata(g["k_cache"], sl, g["block_tables"], g["meta_block_tables"],
                              g["maxblocks"], g["minblocks"])
    torch.cuda.synchronize()
    assert qs.read_status(DEV) == 3          # QS_DEV_ESEQ_LEN
    sel2 = torch.tensor([[[0, 100, -1, -1]] * w.N] * w.B, dtype=torch.int32, device=DEV)
    qs.sparse_decode_attn(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["seq_lens"], sel2)
    torch.cuda.synchronize()
    assert qs.read_status(DEV) == 4          # QS_DEV_ESELECTED
    # the context is intact: a clean call still matches the oracle
    test_quest_select_parity("k_above_blocks")
