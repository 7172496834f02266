"""Seeded synthetic workloads shaped like the pages' decode configurations.

This module draws inputs only: random tensors, page permutations, sequence
lengths and a planted needle.  It holds none of the method's arithmetic, so the
kernels and the oracle can both read its output without sharing any step of
the computation.  Everything is drawn with a seeded ``torch.Generator`` on the
requested device (CPU for test-sized cases, CUDA for the benchmark's large
pools) plus a seeded numpy generator for the prefill-importance draws.

Workload recipes (sizes per the pages' examples and the decode settings the
pages report):
  tiny_fp32        fp32, B=1 H=4 N=2 D=64 BLOCK_SIZE=16, seq_len 512, k=4,
                   sink+window on (t=0); q,K ~U(-1,1), V ~N(0,1); one needle
                   block whose key at one token is 3x the query of the first
                   query head of each KV head's group.
  bf16_paged       bf16, B=20 H=32 N=8 D=128 BLOCK_SIZE=128 MMBPR=1, seq_len
                   16384, k=8; q ~U(-1,1); K ~N(0,1) with 4 outlier channels
                   per KV head scaled x8; V ~N(0,1); block tables a seeded
                   permutation of 2560 pages (the Ascend usage example's shape).
  probe_importance B=1 H=16 N=8 D=128 BLOCK_SIZE=32, S=4096, k=32, n_probe=8,
                   per-token prefill importance ~Dirichlet(0.1); needle in
                   block 64 at a probe offset; fp32 KV or int8 KV + per
                   (token, head) fp32 scales (the small engine's 2B shape).
  long_context     bf16, B=8 seq_len 65536 (512 blocks, 4 metadata blocks per
                   request), k=64, window on with t ~U{0..127}.
  ragged           bf16, B=64, seq_len ~U[2048,131072] rounded to 128 and
                   clamped to >= k*BLOCK_SIZE, shuffled shared page pool,
                   MMBPR=8, k=32, sink+window on (t=0).
  fp16_paged       the bf16_paged shape with fp16 K, V and queries.
Prefill queries for the importance producer (``prefill_queries``): one row
per (position, query head) drawn like the decode query, over the same pages.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

F32, BF16, F16, I8 = "f32", "bf16", "f16", "i8"
TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16, F16: torch.float16, I8: torch.int8}


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    H: int
    N: int
    D: int
    BS: int
    k: int
    seq_len: Optional[int] = None          # uniform length; None -> ragged draw
    ragged: Optional[tuple] = None         # (lo, hi, multiple) for ragged lengths
    t: int = -1                            # tokens since metadata update (-1: no window)
    t_random: bool = False                 # draw t ~U{0..BS-1} per seed
    kv_dtype: str = BF16
    q_dtype: str = BF16
    mode: str = "quest"                    # "quest" or "probe"
    n_probe: int = 8
    importance: bool = False
    needle: bool = False
    needle_block: Optional[int] = None     # fixed needle block (probe config)
    outlier_channels: int = 0
    q_dist: str = "uniform"
    k_dist: str = "uniform"
    MMBPR: Optional[int] = None            # metadata blocks per request slot count
    MKBPR: Optional[int] = None            # KV blocks per request slot count

    @property
    def G(self):
        return self.H // self.N

    def replace(self, **kw):
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", B=1, H=4, N=2, D=64, BS=16, k=4, seq_len=512, t=0,
                          kv_dtype=F32, q_dtype=F32, needle=True),
    "bf16_paged": Workload("bf16_paged", B=20, H=32, N=8, D=128, BS=128, k=8, seq_len=16384,
                           t=-1, outlier_channels=4, k_dist="normal", MMBPR=1),
    "probe_importance": Workload("probe_importance", B=1, H=16, N=8, D=128, BS=32, k=32,
                                 seq_len=4096, kv_dtype=F32, q_dtype=F32, mode="probe",
                                 n_probe=8, importance=True, needle=True, needle_block=64),
    "probe_importance_i8": Workload("probe_importance_i8", B=1, H=16, N=8, D=128, BS=32, k=32,
                                    seq_len=4096, kv_dtype=I8, q_dtype=F32, mode="probe",
                                    n_probe=8, importance=True, needle=True, needle_block=64),
    "long_context": Workload("long_context", B=8, H=32, N=8, D=128, BS=128, k=64,
                             seq_len=65536, t_random=True, outlier_channels=4,
                             k_dist="normal", MMBPR=4),
    "ragged": Workload("ragged", B=64, H=32, N=8, D=128, BS=128, k=32,
                       ragged=(2048, 131072, 128), t=0, outlier_channels=4, k_dist="normal",
                       MMBPR=8),
    # the bf16_paged shape in fp16 (the Ascend kernels' primary dtype)
    "fp16_paged": Workload("fp16_paged", B=20, H=32, N=8, D=128, BS=128, k=8, seq_len=16384,
                           t=-1, outlier_channels=4, k_dist="normal", MMBPR=1, kv_dtype=F16,
                           q_dtype=F16),
}


def ceil_div(a, b):
    return (a + b - 1) // b


def _uniform(shape, gen, device, lo=-1.0, hi=1.0):
    x = torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
    return x.mul_(hi - lo).add_(lo)


def _normal(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def _randperm(n, gen, device):
    return torch.randperm(n, generator=gen, device=device).to(torch.int32)


def draw_seq_lens(w: Workload, rng: np.random.Generator):
    if w.seq_len is not None:
        return np.full(w.B, w.seq_len, np.int64)
    lo, hi, mult = w.ragged
    s = rng.integers(lo, hi + 1, size=w.B)
    s = np.rint(s / mult).astype(np.int64) * mult
    # "k <= blocks enforced": every request holds at least k blocks
    return np.maximum(s, w.k * w.BS)


def make(w: Workload, seed: int = 0, device="cpu", seq_lens=None):
    """Returns a dict of tensors on ``device`` plus a few host-side facts.

    Keys: q, k_cache, v_cache, (k_scale, v_scale for int8), block_tables,
    seq_lens, meta_seq_lens, meta_block_tables, maxblocks, minblocks (zeroed
    pools), importance (probe mode), t, needle (block, token) or None.
    Unused table slots hold -1.
    """
    device = torch.device(device)
    rng = np.random.default_rng(seed)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    B, H, N, D, BS, G = w.B, w.H, w.N, w.D, w.BS, w.G
    L = np.asarray(draw_seq_lens(w, rng) if seq_lens is None else seq_lens, np.int64)
    nb = [ceil_div(int(x), BS) for x in L]
    MKBPR = w.MKBPR or max(max(nb), 1)
    assert max(nb) <= MKBPR
    P = int(sum(nb)) if w.ragged is not None else B * MKBPR
    P = max(P, 1)

    t = w.t
    if w.t_random:
        t = int(rng.integers(0, BS))
    # metadata is built at the last update, t tokens ago, at a multiple of BS
    if t >= 0:
        meta_L = np.array([BS * (max(int(x) - t, 0) // BS) for x in L], np.int64)
    else:
        meta_L = L.copy()

    # page tables: one shuffled pool, each request takes its pages in order
    perm = _randperm(P, gen, device).cpu().numpy()
    bt = np.full((B, MKBPR), -1, np.int32)
    off = 0
    for b in range(B):
        if w.ragged is None:
            bt[b, :] = perm[b * MKBPR:(b + 1) * MKBPR]
            off += MKBPR
        else:
            bt[b, :nb[b]] = perm[off:off + nb[b]]
            off += nb[b]

    n_meta = [ceil_div(x, BS) for x in nb]
    MMBPR = w.MMBPR or max(max(n_meta), 1)
    assert max(n_meta) <= MMBPR
    M = int(sum(n_meta)) if w.ragged is not None else B * MMBPR
    M = max(M, 1)
    mperm = _randperm(M, gen, device).cpu().numpy()
    mbt = np.full((B, MMBPR), -1, np.int32)
    off = 0
    for b in range(B):
        if w.ragged is None:
            mbt[b, :] = mperm[b * MMBPR:(b + 1) * MMBPR]
        else:
            mbt[b, :n_meta[b]] = mperm[off:off + n_meta[b]]
            off += n_meta[b]

    # query
    qf = _uniform((B, H, D), gen, device) if w.q_dist == "uniform" else _normal((B, H, D), gen, device)

    out = {}
    if w.kv_dtype == I8:
        k8 = torch.randint(-127, 128, (P, BS, N, D), generator=gen, device=device,
                           dtype=torch.int32).to(torch.int8)
        v8 = torch.randint(-127, 128, (P, BS, N, D), generator=gen, device=device,
                           dtype=torch.int32).to(torch.int8)
        ks = _uniform((P, BS, N), gen, device, 0.5 / 127, 1.5 / 127)
        vs = _uniform((P, BS, N), gen, device, 0.5 / 127, 1.5 / 127)
        out.update(k_scale=ks, v_scale=vs)
        kc, vc = k8, v8
    else:
        kf = _uniform((P, BS, N, D), gen, device) if w.k_dist == "uniform" else _normal((P, BS, N, D), gen, device)
        if w.outlier_channels:
            ch = torch.stack([_randperm(D, gen, device)[:w.outlier_channels] for _ in range(N)])
            for n in range(N):
                kf[:, :, n, ch[n].long()] *= 8.0
        vf = _normal((P, BS, N, D), gen, device)
        kc, vc = kf, vf

    needle = None
    if w.needle:
        b0 = 0
        if w.needle_block is not None:
            j = w.needle_block
            tok = (BS // max(w.n_probe, 1)) * 2 if w.mode == "probe" else int(rng.integers(0, BS))
        else:
            # any block the window does not force in
            j = int(rng.integers(1, max(nb[b0] - 1, 2)))
            tok = int(rng.integers(0, min(BS, int(L[b0]) - j * BS)))
        p = int(bt[b0, j])
        for n in range(N):
            if w.kv_dtype == I8:
                # full-scale int8 row with the sign pattern of the query and a
                # large scale: a dominant key for the group's first head
                kc[p, tok, n, :] = torch.where(qf[b0, n * G] >= 0, 127, -127).to(torch.int8)
                out["k_scale"][p, tok, n] = 3.0 / 127
            else:
                kc[p, tok, n, :] = 3.0 * qf[b0, n * G, :]
        needle = (b0, j, tok)

    td = TORCH_DTYPE[w.kv_dtype]
    out["q"] = qf.to(TORCH_DTYPE[w.q_dtype])
    out["k_cache"] = kc if w.kv_dtype == I8 else kc.to(td)
    out["v_cache"] = vc if w.kv_dtype == I8 else vc.to(td)
    del kc, vc
    out["block_tables"] = torch.from_numpy(bt).to(device)
    out["seq_lens"] = torch.from_numpy(L.astype(np.int32)).to(device)
    out["meta_seq_lens"] = torch.from_numpy(meta_L.astype(np.int32)).to(device)
    out["meta_block_tables"] = torch.from_numpy(mbt).to(device)
    if w.mode == "quest":
        mdt = TORCH_DTYPE[w.kv_dtype]
        out["maxblocks"] = torch.zeros((M, BS, N, D), dtype=mdt, device=device)
        out["minblocks"] = torch.zeros((M, BS, N, D), dtype=mdt, device=device)
    if w.importance:
        S_max = MKBPR * BS
        imp = np.zeros((B, S_max), np.float32)
        for b in range(B):
            g = rng.gamma(0.1, size=int(L[b]))
            imp[b, :L[b]] = (g / g.sum()).astype(np.float32)
        out["importance"] = torch.from_numpy(imp).to(device)
    out["t"] = t
    out["needle"] = needle
    out["nb"] = nb
    out["MKBPR"] = MKBPR
    out["MMBPR"] = MMBPR
    out["P"] = P
    out["M"] = M
    return out


def prefill_queries(w: Workload, S_max: int, seed: int = 0, device="cpu"):
    """Query rows of a prefill of up to S_max tokens, [B, S_max, H, D], drawn
    like the decode queries (U(-1,1) or N(0,1) per the workload) in the query
    dtype; positions past a request's prefill length hold draws too and are
    never read."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 7919)
    shape = (w.B, S_max, w.H, w.D)
    qf = _uniform(shape, gen, device) if w.q_dist == "uniform" else _normal(shape, gen, device)
    return qf.to(TORCH_DTYPE[w.q_dtype])


def softmax_scale(D):
    return 1.0 / math.sqrt(D)
