"""The workspace-free attention entry point (qs_sparse_decode_attn_noalloc).

It serves callers that cannot allocate device memory: it takes its scratch
from a fixed array inside the library.  This file is collected last on
purpose.  The test calls the entry point through the C ABI twice in a row --
with different sizes, so the second call must clear what the first left in
the shared array -- and checks each result against the regular entry point
(qs_sparse_decode_attn with a caller workspace) within the attention
tolerance of the other GPU tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from decode_sparse_attention_gb300 import questsparse as qs
from decode_sparse_attention_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _noalloc(lib, x, w, sel, out, lse):
    P, I32, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    fn = lib.qs_sparse_decode_attn_noalloc
    fn.argtypes = [P, I32, P, P, P, P, I32, I32, P, I32, P, P, I32, I32, F, I32, I32, I32, I32,
                   I32, P, P, P, P]
    fn.restype = I32
    dt = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2, torch.int8: 3}
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = fn(ptr(x["q"]), dt[x["q"].dtype], ptr(x["k_cache"]), ptr(x["v_cache"]),
            ptr(x.get("k_scale")), ptr(x.get("v_scale")), dt[x["k_cache"].dtype],
            x["k_cache"].shape[0], ptr(x["block_tables"]), x["block_tables"].shape[1],
            ptr(x["seq_lens"]), ptr(sel), sel.shape[1], sel.shape[2], w.D ** -0.5, w.B, w.H,
            w.N, w.D, w.BS, ptr(out), ptr(lse), ptr(qs.status_word(DEV)),
            ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream))
    assert rc == 0, lib.qs_status_string(rc)


def _case(w, seed):
    x = synth.make(w, seed=seed, device=DEV)
    rng = np.random.default_rng(seed)
    sel = np.full((w.B, w.N, w.k), -1, np.int32)
    for b in range(w.B):
        c = np.sort(rng.permutation(x["nb"][b])[:w.k])
        sel[b, :, :len(c)] = c
    return x, torch.from_numpy(sel).to(DEV)


def test_noalloc_matches_workspace_entry_point_twice():
    lib = qs.lib()
    lib.qs_status_string.restype = ctypes.c_char_p
    cases = [synth.WORKLOADS["bf16_paged"].replace(B=6, k=8),                      # 48 units
             synth.WORKLOADS["ragged"].replace(B=3, ragged=(900, 5000, 1), MMBPR=None, k=5)]
    for i, w in enumerate(cases):       # two calls in a row, different sizes
        x, sel = _case(w, seed=11 + i)
        ref_lse = torch.empty((w.B, w.H), device=DEV)
        ref = qs.sparse_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["block_tables"],
                                    x["seq_lens"], sel, lse=ref_lse)
        out = torch.full((w.B, w.H, w.D), float("nan"), device=DEV)
        lse = torch.full((w.B, w.H), float("nan"), device=DEV)
        _noalloc(lib, x, w, sel, out, lse)
        torch.cuda.synchronize()
        assert qs.read_status(DEV) == 0
        assert torch.isfinite(out).all()
        assert (out - ref).abs().max().item() <= 2e-3
        assert (lse - ref_lse).abs().max().item() <= 2e-3


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = qs.lib()
    fn = lib.qs_sparse_decode_attn_noalloc
    fn.restype = ctypes.c_int32
    P, I32, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    fn.argtypes = [P, I32, P, P, P, P, I32, I32, P, I32, P, P, I32, I32, F, I32, I32, I32, I32,
                   I32, P, P, P, P]
    dummy = ctypes.c_void_p(16)
    # 4096 requests x 8 KV heads needs far more than the fixed scratch; the
    # size check comes before any pointer is touched
    rc = fn(dummy, 1, dummy, dummy, None, None, 1, 1, dummy, 1, dummy, dummy, 8, 8, 0.1, 4096,
            32, 8, 128, 128, dummy, None, dummy, None)
    assert rc == 5   # QS_EWORKSPACE
