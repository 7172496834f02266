"""GPU parity of the fused Quest decode step (one kernel: selection + attention).

The fused kernel scores, selects and attends with the same arithmetic as the
selector and the attention kernels, so against the two-kernel step it must
agree bit for bit (selected indices and attention output); against the
oracle, every row's selection follows the gap rule and the attention matches
the oracle's attention over the selection the kernel made.  Cases cover
one-unit and many-unit CTAs, ragged tails, k above the block count, empty
requests, the sink + window forcing, G = 1/2/4, fp32 and 16-bit caches,
D = 64 and 128, and device-side error reporting.
"""
import numpy as np
import pytest
import torch

import oracle
from _common import odt, to_np
from _parity import check_quest_rows, oracle_attention, quest_reference
from decode_sparse_attention_gb300 import questsparse as qs
from decode_sparse_attention_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
W = synth.WORKLOADS

CASES = {
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
    # 1600 units of 3 blocks: CTAs hold up to 7 units each
    "many_units_per_cta": W["bf16_paged"].replace(B=200, H=8, N=8, seq_len=300, MMBPR=None, k=2),
}


def sync_ok():
    torch.cuda.synchronize()
    code = qs.read_status(DEV)
    assert code == 0, qs.device_error_string(code)


def to_dev(x):
    return {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in x.items()}


def run_step(w, x, g, fused, t=None, reps=2, meta_tables=None):
    """Runs the Quest step `reps` times with fused_select = fused; returns the
    selection, output and lse of the last run."""
    mbt = g["meta_block_tables"] if meta_tables is None else meta_tables
    sel = torch.full((w.B, w.N, w.k), -5, dtype=torch.int32, device=DEV)
    out = torch.full((w.B, w.H, w.D), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((w.B, w.H), float("nan"), dtype=torch.float32, device=DEV)
    nbytes = qs.step_workspace_bytes(0, w.B, w.H, w.N, w.D, w.BS, w.k, MMBPR=mbt.shape[1],
                                     MKBPR=x["MKBPR"])
    ws = qs.workspace(nbytes, DEV, ("fused-step", w.name, fused, w.B, w.k))
    p = qs.make_step_params(0, g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                            g["seq_lens"], w.k, sel, out, ws, maxblocks=g["maxblocks"],
                            minblocks=g["minblocks"], metadata_block_tables=mbt,
                            tokens_since_metadata_update=x["t"] if t is None else t, lse=lse,
                            fused_select=fused)
    for _ in range(reps):   # repeated: the workspace counters must rearm
        qs.sparse_decode_step(p, DEV)
    return sel, out, lse


def prepare(w, seed, seq_lens=None):
    x = synth.make(w, seed=seed, device="cpu", seq_lens=seq_lens)
    g = to_dev(x)
    qs.quest_prefill_metadata(g["k_cache"], g["meta_seq_lens"], g["block_tables"],
                              g["meta_block_tables"], g["maxblocks"], g["minblocks"])
    return x, g


@pytest.mark.parametrize("name", list(CASES))
def test_fused_step_equals_two_kernel_step_and_oracle(name):
    w = CASES[name]
    for seed in range(2):
        x, g = prepare(w, seed)
        s1, o1, l1 = run_step(w, x, g, fused=1)
        sync_ok()
        s0, o0, l0 = run_step(w, x, g, fused=0)
        sync_ok()
        # bit for bit against the selector + attention pair
        assert torch.equal(s1, s0), (name, seed)
        assert torch.equal(o1.view(torch.int32), o0.view(torch.int32)), (name, seed)
        assert torch.equal(l1.view(torch.int32), l0.view(torch.int32)), (name, seed)
        # and against the oracle: the gap rule on every row, the attention
        # against the oracle's attention over the selection made
        _, _, osel, osf, *_ = quest_reference(x, w)
        gsel = s1.cpu().numpy()
        check_quest_rows(w, x, gsel, osel, osf, (name, seed))
        oout, olse = oracle_attention(x, w, gsel)
        tol = 2e-3 if x["k_cache"].dtype in (torch.bfloat16, torch.float16) else 1e-5
        err = np.abs(o1.cpu().numpy() - oout).max()
        assert err <= tol, (name, seed, err)


def test_fused_step_empty_requests():
    w = W["bf16_paged"].replace(B=3, seq_len=None, ragged=(1, 2, 1), MMBPR=None, k=4)
    x, g = prepare(w, 0, seq_lens=[0, 130, 517])
    s1, o1, l1 = run_step(w, x, g, fused=1)
    sync_ok()
    s0, o0, l0 = run_step(w, x, g, fused=0)
    sync_ok()
    assert torch.equal(s1, s0)
    assert torch.equal(o1.view(torch.int32), o0.view(torch.int32))
    assert torch.all(s1[0] == -1) and torch.all(o1[0] == 0) and torch.all(torch.isneginf(l1[0]))
    assert torch.all(s1[1, :, 2:] == -1)      # two blocks only


def test_fused_step_full_size_bf16_paged():
    """At the bf16_paged size (B=20, 128 blocks, k=8), the library's choice,
    the forced fused kernel and the two-kernel step agree bit for bit, and
    match the oracle."""
    w = W["bf16_paged"]
    x, g = prepare(w, 0)
    sa, oa, la = run_step(w, x, g, fused=-1)
    s1, o1, l1 = run_step(w, x, g, fused=1)
    s0, o0, l0 = run_step(w, x, g, fused=0)
    sync_ok()
    assert torch.equal(sa, s1) and torch.equal(s1, s0)
    assert torch.equal(oa.view(torch.int32), o0.view(torch.int32))
    assert torch.equal(o1.view(torch.int32), o0.view(torch.int32))
    _, _, osel, osf, *_ = quest_reference(x, w)
    gsel = s1.cpu().numpy()
    check_quest_rows(w, x, gsel, osel, osf, "full")
    oout, _ = oracle_attention(x, w, gsel)
    err = np.abs(o1.cpu().numpy() - oout).max()
    assert err <= 2e-3, err


@pytest.mark.parametrize("fused", [1, 0])
def test_fused_step_reports_bad_metadata_table(fused):
    """A metadata table entry out of range: both forms report
    QS_DEV_EMETA_TABLE and treat that block's rows as unscored."""
    w = W["bf16_paged"].replace(B=2, seq_len=1000, MMBPR=None, k=4)
    x, g = prepare(w, 0)
    mbt = g["meta_block_tables"].clone()
    mbt[1, 0] = 10 ** 6
    run_step(w, x, g, fused=fused, meta_tables=mbt, reps=1)
    torch.cuda.synchronize()
    assert qs.read_status(DEV) == 2
    s, o, _ = run_step(w, x, g, fused=fused, reps=1)
    sync_ok()


@pytest.mark.parametrize("fused", [1, 0])
def test_fused_step_reports_bad_seq_len(fused):
    w = W["bf16_paged"].replace(B=2, seq_len=1000, MMBPR=None, k=4)
    x, g = prepare(w, 0)
    g = dict(g)
    g["seq_lens"] = g["seq_lens"].clone()
    g["seq_lens"][0] = 10 ** 7
    sel, out, _ = run_step(w, x, g, fused=fused, reps=1)
    torch.cuda.synchronize()
    assert qs.read_status(DEV) == 3
    assert torch.all(sel[0] == -1)


@pytest.mark.parametrize("fused", [1, 0])
def test_step_all_scores_tie(fused):
    """Identical metadata rows everywhere: every block scores the same, so
    both forms of the step take the lowest k indices (ties to the lower
    index) and agree bit for bit."""
    w = W["bf16_paged"].replace(B=2, seq_len=128 * 40, MMBPR=None, k=8)
    x, g = prepare(w, 0)
    g["maxblocks"].fill_(0.5)
    g["minblocks"].fill_(-0.25)
    sel, out, _ = run_step(w, x, g, fused=fused)
    sync_ok()
    assert np.all(sel.cpu().numpy() == np.arange(8, dtype=np.int32))
