"""GPU parity of the incremental metadata update (qs_update_metadata).

After a GPU prefill at prev_lens, the update to seq_lens must leave exactly
what a prefill at seq_lens leaves: compared bit for bit with the oracle's
prefill at seq_lens (and the oracle's own update), and with the GPU prefill.
Cases: fp32 / bf16 / fp16, D = 64 and 128, BS = 16 .. 128, empty requests,
no growth, growth inside the partial block, growth into a new metadata block;
a bad prev_len is reported and its request left untouched; at the full ragged
batch size a one-block update equals a full prefill.
"""
import numpy as np
import pytest
import torch

import oracle
from _common import odt, to_np
from decode_sparse_attention_gb300 import questsparse as qs
from decode_sparse_attention_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
W = synth.WORKLOADS

CASES = {
    "tiny_fp32": W["tiny_fp32"].replace(B=4, seq_len=None, ragged=(1, 2, 1), t=-1, needle=False),
    "bf16_bs128": W["bf16_paged"].replace(B=5, seq_len=None, ragged=(1, 2, 1), MMBPR=None),
    "fp16_d64_bs32": W["bf16_paged"].replace(B=5, H=8, N=2, D=64, BS=32, seq_len=None,
                                             ragged=(1, 2, 1), MMBPR=None, kv_dtype="f16",
                                             q_dtype="f16"),
    "bf16_bs16": W["tiny_fp32"].replace(B=5, seq_len=None, ragged=(1, 2, 1), kv_dtype="bf16",
                                        q_dtype="bf16", t=-1, needle=False),
}


def lengths(w):
    """(prev, new) per request: empty, no growth, growth inside the partial
    block, a whole block, and growth that enters a new metadata block."""
    BS = w.BS
    new = [0, 3 * BS + 5, 5 * BS - 1, 7 * BS, BS * BS + 3][:w.B]
    prev = [0, 3 * BS + 5, 4 * BS + 2, 6 * BS, BS * BS - 2][:w.B]
    return prev, new


def sync_ok():
    torch.cuda.synchronize()
    code = qs.read_status(DEV)
    assert code == 0, qs.device_error_string(code)


@pytest.mark.parametrize("name", list(CASES))
def test_update_equals_prefill_at_new_lengths(name):
    w = CASES[name]
    prev, new = lengths(w)
    x = synth.make(w, seed=5, device="cpu", seq_lens=new)
    g = {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in x.items()}
    prev_t = torch.tensor(prev, dtype=torch.int32, device=DEV)
    new_t = g["seq_lens"]
    # GPU: prefill at prev, then update to new (pools start from a sentinel)
    sentinel = torch.full_like(g["maxblocks"], 5.0)
    mx, mn = sentinel.clone(), sentinel.clone()
    qs.quest_prefill_metadata(g["k_cache"], prev_t, g["block_tables"], g["meta_block_tables"],
                              mx, mn)
    qs.quest_update_metadata(g["k_cache"], prev_t, new_t, g["block_tables"],
                             g["meta_block_tables"], mx, mn)
    # GPU prefill at new
    fx, fn = sentinel.clone(), sentinel.clone()
    qs.quest_prefill_metadata(g["k_cache"], new_t, g["block_tables"], g["meta_block_tables"],
                              fx, fn)
    sync_ok()
    assert torch.equal(mx.view(torch.int16 if mx.element_size() == 2 else torch.int32),
                       fx.view(torch.int16 if fx.element_size() == 2 else torch.int32))
    assert torch.equal(mn.view(torch.int16 if mn.element_size() == 2 else torch.int32),
                       fn.view(torch.int16 if fn.element_size() == 2 else torch.int32))
    # oracle: prefill at new, and prefill at prev + update
    ox, on = to_np(sentinel).copy(), to_np(sentinel).copy()
    oracle.prefill_metadata(to_np(x["k_cache"]), odt(x["k_cache"]), np.array(new, np.int32),
                            to_np(x["block_tables"]), to_np(x["meta_block_tables"]), ox, on)
    ux, un = to_np(sentinel).copy(), to_np(sentinel).copy()
    oracle.prefill_metadata(to_np(x["k_cache"]), odt(x["k_cache"]), np.array(prev, np.int32),
                            to_np(x["block_tables"]), to_np(x["meta_block_tables"]), ux, un)
    oracle.update_metadata(to_np(x["k_cache"]), odt(x["k_cache"]), np.array(prev, np.int32),
                           np.array(new, np.int32), to_np(x["block_tables"]),
                           to_np(x["meta_block_tables"]), ux, un)
    assert np.array_equal(to_np(mx), ox) and np.array_equal(to_np(mn), on)
    assert np.array_equal(to_np(mx), ux) and np.array_equal(to_np(mn), un)


def test_update_reports_bad_prev_len_and_leaves_the_request():
    w = CASES["bf16_bs128"]
    prev, new = lengths(w)
    x = synth.make(w, seed=1, device="cpu", seq_lens=new)
    g = {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in x.items()}
    prev_t = torch.tensor(prev, dtype=torch.int32, device=DEV)
    qs.quest_prefill_metadata(g["k_cache"], prev_t, g["block_tables"], g["meta_block_tables"],
                              g["maxblocks"], g["minblocks"])
    sync_ok()
    before = g["maxblocks"].clone()
    bad = prev_t.clone()
    bad[2] = new[2] + 1                      # longer than the request now is
    qs.quest_update_metadata(g["k_cache"], bad, g["seq_lens"], g["block_tables"],
                             g["meta_block_tables"], g["maxblocks"], g["minblocks"])
    torch.cuda.synchronize()
    assert qs.read_status(DEV) == 3          # QS_DEV_ESEQ_LEN
    m = int(g["meta_block_tables"][2, 0])
    assert torch.equal(g["maxblocks"][m].view(torch.int16), before[m].view(torch.int16))
    with pytest.raises(qs.QuestSparseError):
        qs.quest_update_metadata(g["k_cache"], bad[:2], g["seq_lens"], g["block_tables"],
                                 g["meta_block_tables"], g["maxblocks"], g["minblocks"])


def test_update_full_size_ragged_one_block():
    """Ragged batch (64 requests, ~33K blocks): metadata built one block
    short of each request, then updated, equals a full prefill bit for bit."""
    w = W["ragged"]
    x = synth.make(w, seed=0, device=DEV)
    L = x["seq_lens"]
    prev = torch.clamp(L - w.BS, min=0).to(torch.int32)
    mx, mn = torch.zeros_like(x["maxblocks"]), torch.zeros_like(x["minblocks"])
    qs.quest_prefill_metadata(x["k_cache"], prev, x["block_tables"], x["meta_block_tables"],
                              mx, mn)
    qs.quest_update_metadata(x["k_cache"], prev, L, x["block_tables"], x["meta_block_tables"],
                             mx, mn)
    fx, fn = torch.zeros_like(mx), torch.zeros_like(mn)
    qs.quest_prefill_metadata(x["k_cache"], L, x["block_tables"], x["meta_block_tables"], fx, fn)
    sync_ok()
    assert torch.equal(mx.view(torch.int16), fx.view(torch.int16))
    assert torch.equal(mn.view(torch.int16), fn.view(torch.int16))
