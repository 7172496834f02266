"""GPU parity at the full sizes of the long-context and ragged workloads.

long_context (B=8, 65536 tokens = 512 blocks of 128, 4 metadata blocks per
request, k=64, window on with a random t): every output against the oracle
-- metadata bit-exact, Quest scores within 1e-5 relative, selections by the
gap rule on every row, attention within 2e-3 of the oracle's attention over
the selection the GPU made -- and the decode step (both forms) bit for bit
against the separate kernels.  Its 256 scoring chunks exceed the SM count,
so scan CTAs score more than one chunk each.

ragged_multi_chunk (24 requests of 20K..60K tokens, ~580 scoring chunks: every
scan CTA scores two or more): the same checks on every request.

ragged (B=64, 2048..131072 tokens, the whole 17 GB paged pool): the oracle
runs on a seeded sample of whole requests (metadata included); every
request is checked through properties that hold at any size -- selections
well formed, the forced blocks present, the picks the top of the GPU's own
scores, and the attention equal to a dense fp32 softmax over the selected
tokens computed with torch on the device.
"""
import numpy as np
import pytest
import torch

from _common import to_np
from _gpu_checks import (ATTN_TOL, DEV, full_oracle_check, gpu_chain, scan_chunks,
                         step_matches_kernels)
from _parity import check_quest_rows, check_scores, forced_flags, oracle_attention, quest_reference  # noqa: F401
from decode_sparse_attention_gb300 import synth

pytestmark = pytest.mark.gpu
W = synth.WORKLOADS


@pytest.mark.parametrize("seed", [0, 1])
def test_long_context_full_size(seed):
    w = W["long_context"]
    x = synth.make(w, seed=seed, device=DEV)
    assert scan_chunks(x, w) > torch.cuda.get_device_properties(DEV).multi_processor_count
    full_oracle_check(w, x, ("long_context", seed, x["t"]))


def test_ragged_multi_chunk_per_scan_cta():
    w = W["ragged"].replace(B=24, ragged=(20000, 60000, 128), MMBPR=None)
    x = synth.make(w, seed=3, device=DEV)
    assert scan_chunks(x, w) >= 2 * torch.cuda.get_device_properties(DEV).multi_processor_count
    full_oracle_check(w, x, "ragged_multi_chunk")


# ---------------------------------------------------------------------------
# the ragged batch at full size: oracle on a sample, properties everywhere
# ---------------------------------------------------------------------------

def sample_inputs(x, reqs):
    """Host copies of whole requests with their KV pages and metadata blocks
    renumbered densely (the oracle builds its own metadata for them)."""
    bt = to_np(x["block_tables"])[reqs]
    pages = sorted(set(int(p) for p in bt.ravel() if p >= 0))
    remap = {p: i for i, p in enumerate(pages)}
    bt2 = np.vectorize(lambda p: remap.get(int(p), -1))(bt).astype(np.int32)
    idx = torch.tensor(pages, dtype=torch.long, device=DEV)
    mbt = to_np(x["meta_block_tables"])[reqs]
    metas = [int(m) for m in mbt.ravel() if m >= 0]
    mremap = {m: i for i, m in enumerate(metas)}
    mbt2 = np.vectorize(lambda m: mremap.get(int(m), -1))(mbt).astype(np.int32)
    midx = torch.tensor(metas, dtype=torch.long, device=DEV)
    sub = {"q": x["q"][reqs].cpu(), "k_cache": x["k_cache"][idx].cpu(),
           "v_cache": x["v_cache"][idx].cpu(), "block_tables": torch.from_numpy(bt2),
           "seq_lens": x["seq_lens"][reqs].cpu(), "meta_seq_lens": x["meta_seq_lens"][reqs].cpu(),
           "meta_block_tables": torch.from_numpy(mbt2),
           "maxblocks": torch.zeros_like(x["maxblocks"][midx]).cpu(),
           "minblocks": torch.zeros_like(x["minblocks"][midx]).cpu(),
           "t": x["t"], "nb": [x["nb"][b] for b in reqs]}
    return sub, midx


def dense_attention_torch(w, x, sel):
    """fp32 softmax attention over the selected blocks' valid tokens, with
    torch on the device (an independent library computation)."""
    out = torch.empty((w.B, w.H, w.D), device=DEV)
    G = w.G
    scale = w.D ** -0.5
    for b in range(w.B):
        L = int(x["seq_lens"][b])
        for n in range(w.N):
            js = [int(j) for j in sel[b, n] if j >= 0]
            pages = x["block_tables"][b, js].long()
            K = x["k_cache"][pages, :, n, :].float()          # [k, BS, D]
            V = x["v_cache"][pages, :, n, :].float()
            valid = torch.tensor([min(w.BS, L - j * w.BS) for j in js], device=DEV)
            mask = torch.arange(w.BS, device=DEV)[None, :] < valid[:, None]
            K, V = K[mask], V[mask]                            # [T, D]
            q = x["q"][b, n * G:(n + 1) * G].float()          # [G, D]
            p = torch.softmax((q @ K.T) * scale, dim=-1)
            out[b, n * G:(n + 1) * G] = p @ V
    return out


def check_selection_properties(w, x, gsel, gsc):
    """At any size: count min(k, nb), ascending and distinct, the forced
    blocks present, and every other pick ranked above every block left out
    by the GPU's own scores (score descending, ties to the lower index)."""
    L = to_np(x["seq_lens"])
    for b in range(w.B):
        nb = x["nb"][b]
        fixed = forced_flags(L[b], w.BS, x["t"], nb)
        for n in range(w.N):
            row = gsel[b, n]
            picks = [int(j) for j in row if j >= 0]
            assert len(picks) == min(w.k, nb) and picks == sorted(set(picks)), (b, n, row)
            assert np.all(row[len(picks):] == -1)
            assert set(np.flatnonzero(fixed).tolist()) <= set(picks), (b, n)
            chosen = set(picks) - set(np.flatnonzero(fixed).tolist())
            rest = [j for j in range(nb) if not fixed[j] and j not in chosen]
            if chosen and rest:
                s = gsc[b, n]
                worst = min(chosen, key=lambda j: (s[j], -j))
                best_left = max(rest, key=lambda j: (s[j], -j))
                assert (s[worst], -worst) > (s[best_left], -best_left), (b, n, worst, best_left)


def test_ragged_full_size_sampled_oracle():
    w = W["ragged"]
    x = synth.make(w, seed=0, device=DEV)
    sel, scores, out, lse = gpu_chain(w, x)
    gsel = sel.cpu().numpy()
    gsc = scores.cpu().numpy()

    # every request: properties and the torch attention
    check_selection_properties(w, x, gsel, gsc)
    ref = dense_attention_torch(w, x, gsel)
    assert (out - ref).abs().max().item() <= ATTN_TOL

    # a seeded sample of whole requests against the oracle: the shortest, the
    # longest and two drawn at random
    L = to_np(x["seq_lens"])
    rng = np.random.default_rng(7)
    reqs = sorted({int(np.argmin(L)), int(np.argmax(L)), *rng.choice(w.B, 2, replace=False).tolist()})
    sub, midx = sample_inputs(x, reqs)
    ws = w.replace(B=len(reqs))
    mx, mn, osel, osf, osd, osa = quest_reference(sub, ws)
    assert np.array_equal(to_np(x["maxblocks"][midx]), mx)
    assert np.array_equal(to_np(x["minblocks"][midx]), mn)
    for i, b in enumerate(reqs):
        nb = x["nb"][b]
        for n in range(w.N):
            check_scores(gsc[b, n, :nb], osd[i, n, :nb], osa[i, n, :nb], ("ragged", b, n))
    check_quest_rows(ws, sub, gsel[reqs], osel, osf, "ragged-sample")
    oout, _ = oracle_attention(sub, ws, gsel[reqs])
    assert np.abs(out.cpu().numpy()[reqs] - oout).max() <= ATTN_TOL
    step_matches_kernels(w, x, sel, out, lse)
