"""GPU parity of the prefill importance producer (qs_prefill_importance).

Small cases (several row, key and query-part tiles, ragged lengths, empty
requests) are compared element by element with the oracle in double:
importance within rtol 1e-4 / atol 1e-6 and the row log-sum-exp within
1e-5 (relative + absolute).  The bound: each logit is a dot of D products
accumulated in fp32.  bf16/fp16/int8 products are exact; fp32 operands reach
the tensor cores as bf16 high and low parts (x = hi + lo + r, |r| <= 2^-17
|x|) and each product keeps hi.hi + hi.lo + lo.hi, so a product is off by at
most 2^-15 of |q_d k_d| and typically by about 2^-19 (these bounds are
checked on the host in test_split_bf16_bound.py); with the scale 1/sqrt(D)
and operands of magnitude <= 1 the logit error is about 1e-6 (the errors of
the D terms have random signs), and the accumulation adds ~D * 2^-24
relative to sum |q_d k_d|.  The base-2 exponential is the SFU approximation (~2 ulp),
and a token's importance is an fp32 sum of up to G * S probabilities, so the
relative error stays near 1e-5; 1e-4 leaves a margin of ten.

At the full probe_importance size (B=1, S=4096, H=16, N=8, D=128, fp32 and
int8) the checks are what holds at any size plus what the oracle computes
exactly on a slice: total mass H*S, the log-sum-exp of the first 512 rows
(causal rows depend only on the prefix), and importance[s] for the last 128
positions (the oracle summing only the queries from S-128 on).
"""
import time

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
RTOL, ATOL = 1e-4, 1e-6
LSE_TOL = 1e-5

PI = W["probe_importance"]
CASES = {
    # name: (workload, prefill lengths)
    "f32_d128_g2_bs32": (PI.replace(B=4, seq_len=None, ragged=(1, 2, 1), needle=False),
                         [300, 0, 129, 64]),
    "f32_parts_d64": (PI.replace(B=2, H=4, N=2, D=64, seq_len=None, ragged=(1, 2, 1),
                                 needle=False), [1500, 1037]),
    "bf16_d64_g4_bs16": (PI.replace(B=3, H=8, N=2, D=64, BS=16, seq_len=None, ragged=(1, 2, 1),
                                    kv_dtype="bf16", q_dtype="bf16", needle=False),
                         [257, 31, 190]),
    "f16_d128_g1_bs64": (PI.replace(B=2, H=4, N=4, BS=64, seq_len=None, ragged=(1, 2, 1),
                                    kv_dtype="f16", q_dtype="f16", needle=False), [200, 77]),
    "f32_d64_g8": (PI.replace(B=2, H=32, N=4, D=64, BS=32, seq_len=None, ragged=(1, 2, 1),
                              needle=False), [150, 33]),
    "i8_d128_g2": (PI.replace(B=2, seq_len=None, ragged=(1, 2, 1), kv_dtype="i8",
                              needle=False), [261, 96]),
    "i8_bf16q_d64": (PI.replace(B=2, H=4, N=2, D=64, seq_len=None, ragged=(1, 2, 1),
                                kv_dtype="i8", q_dtype="bf16", needle=False), [130, 5]),
}


def inputs(w, lens, seed, device):
    x = synth.make(w, seed=seed, device="cpu", seq_lens=lens)
    S_max = x["MKBPR"] * w.BS
    q = synth.prefill_queries(w, S_max, seed=seed, device="cpu")
    g = {k: (v.to(device) if torch.is_tensor(v) else v) for k, v in x.items()}
    return x, g, q, S_max


def sync_ok():
    torch.cuda.synchronize()
    code = qs.read_status(DEV)
    assert code == 0, qs.device_error_string(code)


def oracle_run(w, x, q, lens, first_query=0):
    return oracle.prefill_importance(to_np(q), odt(q), to_np(x["k_cache"]), odt(x["k_cache"]),
                                     to_np(x["block_tables"]), np.array(lens, np.int32), w.N,
                                     k_scale=None if "k_scale" not in x else to_np(x["k_scale"]),
                                     first_query=first_query)


def gpu_run(w, g, q, lens):
    lens_t = torch.tensor(lens, dtype=torch.int32, device=DEV)
    B, S_max = q.shape[0], q.shape[1]
    lse = torch.full((B, w.H, S_max), float("nan"), dtype=torch.float32, device=DEV)
    imp = qs.prefill_importance(q.to(DEV), g["k_cache"], g["block_tables"], lens_t,
                                k_scale=g.get("k_scale"), lse=lse)
    return imp, lse


@pytest.mark.parametrize("name", list(CASES))
def test_importance_matches_oracle(name):
    w, lens = CASES[name]
    x, g, q, S_max = inputs(w, lens, 11, DEV)
    imp, lse = gpu_run(w, g, q, lens)
    sync_ok()
    ref, ref_lse = oracle_run(w, x, q, lens)
    got, got_lse = imp.cpu().double().numpy(), lse.cpu().double().numpy()
    for b, S in enumerate(lens):
        assert np.all(got[b, S:] == 0)
        np.testing.assert_allclose(got[b, :S], ref[b, :S], rtol=RTOL, atol=ATOL)
        np.testing.assert_allclose(got_lse[b, :, :S], ref_lse[b, :, :S], rtol=LSE_TOL,
                                   atol=LSE_TOL)
        assert np.isclose(got[b].sum(), w.H * S, rtol=1e-5)


def test_importance_block_size_one_long_table():
    """BLOCK_SIZE 1 and 2100 tokens: the key packing follows one table entry
    per key, 2100 entries, and the last key tile is partial."""
    w = PI.replace(B=1, H=2, N=1, D=64, BS=1, seq_len=None, ragged=(1, 2, 1), needle=False)
    lens = [2100]
    x, g, q, _ = inputs(w, lens, 3, DEV)
    imp, lse = gpu_run(w, g, q, lens)
    sync_ok()
    ref, ref_lse = oracle_run(w, x, q, lens)
    np.testing.assert_allclose(imp.cpu().double().numpy()[0], ref[0], rtol=RTOL, atol=ATOL)
    np.testing.assert_allclose(lse.cpu().double().numpy()[0], ref_lse[0], rtol=LSE_TOL,
                               atol=LSE_TOL)


@pytest.mark.parametrize("kv", ["f32", "i8"])
def test_importance_full_size(kv):
    w = PI.replace(kv_dtype=kv)
    lens = [w.seq_len]
    x, g, q, S_max = inputs(w, lens, 0, DEV)
    imp, lse = gpu_run(w, g, q, lens)
    imp2, _ = gpu_run(w, g, q, lens)
    sync_ok()
    assert torch.equal(imp, imp2)                          # deterministic
    got, got_lse = imp.cpu().double().numpy(), lse.cpu().double().numpy()
    S = lens[0]
    assert np.all(got[0] > 0) and np.isclose(got[0].sum(), w.H * S, rtol=1e-5)
    # the first 512 rows' lse: a prefill of 512 tokens has the same rows
    _, pre_lse = oracle_run(w, x, q, [512])
    np.testing.assert_allclose(got_lse[0, :, :512], pre_lse[0, :, :512], rtol=LSE_TOL,
                               atol=LSE_TOL)
    # the last 128 tokens are seen only by the last 128 queries
    f = S - 128
    tail, tail_lse = oracle_run(w, x, q, lens, first_query=f)
    np.testing.assert_allclose(got[0, f:], tail[0, f:], rtol=RTOL, atol=ATOL)
    np.testing.assert_allclose(got_lse[0, :, f:], tail_lse[0, :, f:], rtol=LSE_TOL, atol=LSE_TOL)


def test_importance_feeds_probe_selector():
    """Producer -> selector on the probe_importance shape: the GPU selection
    from the produced importance equals the oracle's from the same values."""
    w = PI
    lens = [w.seq_len]
    x, g, q, S_max = inputs(w, lens, 2, DEV)
    imp, _ = gpu_run(w, g, q, lens)
    qd = g["q"]
    sel = qs.probe_select(qd, g["k_cache"], g["block_tables"], g["seq_lens"], w.k,
                          n_probe=w.n_probe, importance=imp)
    sync_ok()
    ref_sel, _, _, n_imp = oracle.probe_select(to_np(x["q"]), odt(x["q"]), to_np(x["k_cache"]),
                                               odt(x["k_cache"]), to_np(x["block_tables"]),
                                               to_np(x["seq_lens"]), w.N, w.k, w.n_probe,
                                               importance=imp.cpu().numpy())
    assert np.array_equal(np.sort(sel.cpu().numpy(), -1), np.sort(ref_sel, -1))
    assert np.all(n_imp == (w.k + 1) // 2)


def test_importance_errors_and_empty():
    w, lens = CASES["f32_d128_g2_bs32"]
    x, g, q, S_max = inputs(w, lens, 5, DEV)
    # every request empty: zeros, no error
    imp, _ = gpu_run(w, g, q, [0, 0, 0, 0])
    sync_ok()
    assert torch.count_nonzero(imp) == 0
    # a length past S_max: reported, that request left zero, the others right
    bad = [lens[0], S_max + 1, lens[2], lens[3]]
    imp, _ = gpu_run(w, g, q, bad)
    torch.cuda.synchronize()
    assert qs.read_status(DEV) == 3                        # QS_DEV_ESEQ_LEN
    assert torch.count_nonzero(imp[1]) == 0
    ref, _ = oracle_run(w, x, q, [lens[0], 0, lens[2], lens[3]])
    np.testing.assert_allclose(imp.cpu().double().numpy()[0], ref[0], rtol=RTOL, atol=ATOL)
    # a table entry outside the pool
    bt = g["block_tables"].clone()
    bt[0, 1] = g["k_cache"].shape[0]
    qs.prefill_importance(q.to(DEV), g["k_cache"], bt,
                          torch.tensor(lens, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert qs.read_status(DEV) == 1                        # QS_DEV_EBLOCK_TABLE
    # host-side checks
    with pytest.raises(qs.QuestSparseError):
        qs.prefill_importance(q.to(DEV).to(torch.bfloat16), g["k_cache"], g["block_tables"],
                              torch.tensor(lens, dtype=torch.int32, device=DEV))


def test_bounded_wait_runs_out_and_reports_timeout():
    """Every wait of the tensor-core passes is bounded.  The library's
    self-check runs that same wait on an mbarrier nothing arrives on: it must
    return within seconds with QS_DEV_ETIMEOUT (6) in the status word, and
    the context must stay usable (a producer call afterwards still matches
    the oracle)."""
    t0 = time.time()
    assert qs.check_bounded_wait(DEV) == 6
    assert time.time() - t0 < 30.0
    w, lens = CASES["f32_d128_g2_bs32"]
    x, g, q, S_max = inputs(w, lens, 9, DEV)
    imp, _ = gpu_run(w, g, q, lens)
    sync_ok()
    ref, _ = oracle_run(w, x, q, lens)
    for b, S in enumerate(lens):
        np.testing.assert_allclose(imp.cpu().double().numpy()[b, :S], ref[b, :S], rtol=RTOL, atol=ATOL)

