"""fp16 Quest path at the shapes of the CANN page's usage example (its
primary dtype): metadata built from fp16 K with B=4, N=8, BLOCK_SIZE=128,
D=128 and 200 KV blocks per request, and selection + sparse attention at
B=20, H=32, N=8, k=8 over 16384-token requests.  Metadata bit-exact against
the oracle, Quest scores within 1e-5 relative, selections by the gap rule on
every row, attention within 2e-3 of the oracle's attention over the selection
the GPU made, and the decode step bit for bit against the separate kernels.
"""
import numpy as np
import pytest
import torch

import oracle
from _common import to_np
from _gpu_checks import DEV, full_oracle_check, sync_ok
from decode_sparse_attention_gb300 import questsparse as qs
from decode_sparse_attention_gb300 import synth

pytestmark = pytest.mark.gpu
W = synth.WORKLOADS
FP16 = dict(kv_dtype="f16", q_dtype="f16")


@pytest.mark.parametrize("seed", [0, 1])
def test_fp16_metadata_usage_example(seed):
    """B=4, N=8, BLOCK_SIZE=128, D=128, 200 KV blocks per request (ragged
    lengths up to 25600 tokens, partial last blocks), fp16 K."""
    w = W["bf16_paged"].replace(B=4, seq_len=None, ragged=(3000, 25600, 1), MKBPR=200,
                                MMBPR=2, **FP16)
    x = synth.make(w, seed=seed, device=DEV)
    assert x["block_tables"].shape[1] == 200
    sent = torch.full_like(x["maxblocks"], 3.0)      # rows the kernel must not touch
    x["maxblocks"], x["minblocks"] = sent.clone(), sent.clone()
    qs.quest_prefill_metadata(x["k_cache"], x["meta_seq_lens"], x["block_tables"],
                              x["meta_block_tables"], x["maxblocks"], x["minblocks"])
    sync_ok()
    mx, mn = to_np(sent).copy(), to_np(sent).copy()
    oracle.prefill_metadata(to_np(x["k_cache"]), oracle.F16, to_np(x["meta_seq_lens"]),
                            to_np(x["block_tables"]), to_np(x["meta_block_tables"]), mx, mn)
    assert np.array_equal(to_np(x["maxblocks"]), mx)
    assert np.array_equal(to_np(x["minblocks"]), mn)


@pytest.mark.parametrize("seed", [0, 1])
def test_fp16_select_attention_step_usage_example(seed):
    w = W["bf16_paged"].replace(**FP16)          # B=20 H=32 N=8 D=128 BS=128 k=8
    x = synth.make(w, seed=seed, device=DEV)
    full_oracle_check(w, x, ("fp16", seed))


def test_fp16_window_multi_metadata_blocks():
    """fp16 with the sink + window forcing and 4 metadata blocks per
    request (the long-context shape at B=2)."""
    w = W["long_context"].replace(B=2, **FP16)
    x = synth.make(w, seed=5, device=DEV)
    full_oracle_check(w, x, "fp16-long")
