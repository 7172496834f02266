"""GPU checks shared by the full-size parity tests: the Quest chain through
the C ABI (metadata, selection with scores, attention), the decode step
against the separate kernels, and the complete comparison with the oracle.
No arithmetic of the method lives here."""
import numpy as np
import torch

from _common import to_np
from _parity import check_quest_rows, check_scores, oracle_attention, quest_reference
from decode_sparse_attention_gb300 import questsparse as qs

DEV = torch.device("cuda:0")
ATTN_TOL = 2e-3
SCAN_ROWS_BF16_D128 = 128      # metadata rows one scan chunk scores (bf16, D = 128)


def sync_ok():
    torch.cuda.synchronize()
    code = qs.read_status(DEV)
    assert code == 0, qs.device_error_string(code)


def scan_chunks(x, w):
    return sum(-(-nb // SCAN_ROWS_BF16_D128) * w.N for nb in x["nb"])


def gpu_chain(w, x):
    """Metadata, selection (with scores) and attention through the C ABI."""
    qs.quest_prefill_metadata(x["k_cache"], x["meta_seq_lens"], x["block_tables"],
                              x["meta_block_tables"], x["maxblocks"], x["minblocks"])
    MMBPR = x["meta_block_tables"].shape[1]
    sel = torch.full((w.B, w.N, w.k), -5, dtype=torch.int32, device=DEV)
    scores = torch.full((w.B, w.N, MMBPR * w.BS), float("nan"), device=DEV)
    qs.quest_block_select_paged_in_out_w(x["q"], x["maxblocks"], x["minblocks"],
                                         x["meta_block_tables"], x["seq_lens"], x["t"], sel,
                                         scores=scores)
    lse = torch.full((w.B, w.H), float("nan"), device=DEV)
    out = qs.sparse_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["block_tables"],
                                x["seq_lens"], sel, lse=lse)
    sync_ok()
    return sel, scores, out, lse


def step_matches_kernels(w, x, sel, out, lse):
    """The decode step (two kernels, and the fused kernel where it is taken)
    gives the separate kernels' selection and output bit for bit."""
    MMBPR = x["meta_block_tables"].shape[1]
    nbytes = qs.step_workspace_bytes(0, w.B, w.H, w.N, w.D, w.BS, w.k, MMBPR=MMBPR,
                                     MKBPR=x["MKBPR"])
    for fused in (0, 1):
        s2 = torch.full_like(sel, -5)
        o2 = torch.full_like(out, float("nan"))
        l2 = torch.full_like(lse, float("nan"))
        ws = qs.workspace(nbytes, DEV, ("full-size-step", w.name, fused))
        p = qs.make_step_params(0, x["q"], x["k_cache"], x["v_cache"], x["block_tables"],
                                x["seq_lens"], w.k, s2, o2, ws, maxblocks=x["maxblocks"],
                                minblocks=x["minblocks"],
                                metadata_block_tables=x["meta_block_tables"],
                                tokens_since_metadata_update=x["t"], lse=l2, fused_select=fused)
        if fused and qs.step_kernels(p) != 1:
            continue
        for _ in range(2):   # twice: the workspace counters rearm
            qs.sparse_decode_step(p, DEV)
        sync_ok()
        assert torch.equal(s2, sel), fused
        assert torch.equal(o2.view(torch.int32), out.view(torch.int32)), fused
        assert torch.equal(l2.view(torch.int32), lse.view(torch.int32)), fused


def full_oracle_check(w, x, what):
    sel, scores, out, lse = gpu_chain(w, x)
    xo = dict(x)        # the oracle builds its metadata into zeroed pools
    xo["maxblocks"] = torch.zeros_like(x["maxblocks"])
    xo["minblocks"] = torch.zeros_like(x["minblocks"])
    mx, mn, osel, osf, osd, osa = quest_reference(xo, w)
    assert np.array_equal(to_np(x["maxblocks"]), mx), what
    assert np.array_equal(to_np(x["minblocks"]), mn), what
    gsc = scores.cpu().numpy()
    for b in range(w.B):
        nb = x["nb"][b]
        for n in range(w.N):
            check_scores(gsc[b, n, :nb], osd[b, n, :nb], osa[b, n, :nb], (what, b, n))
    gsel = sel.cpu().numpy()
    exact = check_quest_rows(w, x, gsel, osel, osf, what)
    assert exact >= 0.9 * w.B * w.N, (what, exact)
    oout, olse = oracle_attention(x, w, gsel)
    err = np.abs(out.cpu().numpy() - oout).max()
    assert err <= ATTN_TOL, (what, err)
    assert np.abs(lse.cpu().numpy() - olse).max() <= 1e-3, what
    step_matches_kernels(w, x, sel, out, lse)
