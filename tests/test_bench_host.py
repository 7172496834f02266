"""Host-side logic of bench.py: algorithmic byte counting and the
max-over-ranks reduction of the replicas path (world size 2, gloo, CPU)."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from decode_sparse_attention_gb300 import synth


def test_selected_kv_bytes_counts_valid_tokens_once_per_kv_head():
    w = synth.WORKLOADS["bf16_paged"].replace(B=1, H=4, N=2, BS=4, D=8)
    sel = np.array([[[0, 2, -1], [1, 2, 3]]], np.int32)           # per KV head
    L = np.array([14])                                              # block 3 holds 2 tokens
    kv = bench.selected_kv_bytes(sel, L, w, 2, False)
    assert kv == (4 + 4 + 4 + 4 + 2) * 8 * 2 * 2
    selq = np.array([[[0, 1, -1], [1, 3, -1], [2, -1, -1], [2, -1, -1]]], np.int32)  # per query head
    kvq = bench.selected_kv_bytes(selq, L, w, 2, False)
    assert kvq == (4 + 4 + 2 + 4) * 8 * 2 * 2                      # {0,1,3} and {2}


def test_step_bytes_bf16_paged_matches_hand_count():
    w = synth.WORKLOADS["bf16_paged"]
    x = {"seq_lens": torch.full((20,), 16384, dtype=torch.int32),
         "k_cache": torch.empty(0, dtype=torch.bfloat16)}
    sel = np.tile(np.arange(8, dtype=np.int32), (20, 8, 1))
    nb = bench.step_bytes(w, x, sel, 2)
    assert nb["kv"] == 160 * 8 * 128 * 128 * 2 * 2
    assert nb["select"] == 20 * 128 * 8 * 128 * 2 * 2
    assert abs(nb["step"] / 1e6 - 94.9) < 0.2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2")
    dist.init_process_group("gloo", rank=rank, world_size=2)
    v = bench.max_over_ranks(10.0 + 5.0 * rank)
    bench.barrier()
    out[rank] = v
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == 15.0 and out[1] == 15.0


def test_max_over_ranks_single_process_identity():
    assert bench.max_over_ranks(3.5) == 3.5


def test_importance_tile_ops_counts_causal_tile_pairs():
    """The executed-flop count of the prefill importance producer: both of its
    passes multiply every (128-row query tile, 128-key tile) pair that holds
    at least one causal (row, key) pair, per KV head (a tile pair does when
    its first key is at or before the position of its last row).  Checked by
    enumerating the tile pairs, ragged and tile-unaligned lengths included."""
    import itertools
    for lens, H, N in (([4096], 16, 8), ([300, 0, 129, 64], 16, 8), ([1500, 1037], 4, 2),
                       ([150, 33], 32, 4), ([200, 77], 4, 4)):
        G = H // N
        S_max = max(lens) + 37
        want = 0
        for S in lens:
            for qt, kt in itertools.product(range((S * G + 127) // 128), range((S + 127) // 128)):
                rows = range(128 * qt, min(128 * qt + 128, S * G))
                keys = range(128 * kt, min(128 * kt + 128, S))
                if any(s <= r // G for r in (rows[-1],) for s in (keys[0],)):
                    want += 1
        assert bench.importance_tile_ops(lens, S_max, H, N) == 2 * N * want
    assert bench.importance_tile_ops([4096], 4096, 16, 8) == 16896
