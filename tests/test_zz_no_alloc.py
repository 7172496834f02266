"""The workspace-free attention entry point (qs_sparse_decode_attn_noalloc).

It serves callers that cannot allocate device memory (a decode loop that
forbids allocations once it runs, a plugin handed only input and output
pointers): it takes its scratch from a fixed 4 MiB array inside the library.
This file is collected last on purpose, so that a run stopping at its first
failure has run every other test before it.

Both entry points launch the same kernel with the same launch plan, and its
split-K merge combines the partials in a fixed order, so the workspace-free
result must equal qs_sparse_decode_attn's bit for bit.  The tests call it
through the C ABI twice in a row with different sizes, once after planting
stale non-zero arrival counters in the shared array (the call must clear
them), and at the size limit: 495 (request, KV head) units at H/N = 4,
D = 128 are served, 496 are refused.
"""
import ctypes

import numpy as np
import pytest
import torch

from decode_sparse_attention_gb300 import questsparse as qs
from decode_sparse_attention_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
P, I32, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
QS_EWORKSPACE = 5


def _fn(lib):
    fn = lib.qs_sparse_decode_attn_noalloc
    fn.argtypes = [P, I32, P, P, P, P, I32, I32, P, I32, P, P, I32, I32, F, I32, I32, I32, I32,
                   I32, P, P, P, P]
    fn.restype = I32
    lib.qs_status_string.restype = ctypes.c_char_p
    lib.qs_status_string.argtypes = [I32]
    return fn


def _noalloc(lib, x, w, sel, out, lse):
    dt = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2, torch.int8: 3}
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return _fn(lib)(ptr(x["q"]), dt[x["q"].dtype], ptr(x["k_cache"]), ptr(x["v_cache"]),
                    ptr(x.get("k_scale")), ptr(x.get("v_scale")), dt[x["k_cache"].dtype],
                    x["k_cache"].shape[0], ptr(x["block_tables"]), x["block_tables"].shape[1],
                    ptr(x["seq_lens"]), ptr(sel), sel.shape[1], sel.shape[2], w.D ** -0.5, w.B,
                    w.H, w.N, w.D, w.BS, ptr(out), ptr(lse), ptr(qs.status_word(DEV)),
                    ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream))


class _DeviceWords:
    """A view of device memory the library owns, for torch.as_tensor."""

    def __init__(self, addr, n):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "<i4", "data": (addr, False),
                                         "strides": None, "version": 3}


def _scratch_words(lib):
    fn = lib.qs_sparse_decode_attn_noalloc_scratch
    fn.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_size_t)]
    fn.restype = I32
    addr, nbytes = ctypes.c_void_p(), ctypes.c_size_t()
    assert fn(ctypes.byref(addr), ctypes.byref(nbytes)) == 0
    assert nbytes.value == 4 << 20
    return torch.as_tensor(_DeviceWords(addr.value, nbytes.value // 4), device=DEV)


def _case(w, seed):
    x = synth.make(w, seed=seed, device=DEV)
    rng = np.random.default_rng(seed)
    sel = np.full((w.B, w.N, w.k), -1, np.int32)
    for b in range(w.B):
        c = np.sort(rng.permutation(x["nb"][b])[:w.k])
        sel[b, :, :len(c)] = c
    return x, torch.from_numpy(sel).to(DEV)


def _check_equal(lib, w, x, sel):
    ref_lse = torch.empty((w.B, w.H), device=DEV)
    ref = qs.sparse_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["block_tables"],
                                x["seq_lens"], sel, lse=ref_lse)
    out = torch.full((w.B, w.H, w.D), float("nan"), device=DEV)
    lse = torch.full((w.B, w.H), float("nan"), device=DEV)
    rc = _noalloc(lib, x, w, sel, out, lse)
    assert rc == 0, lib.qs_status_string(rc)
    torch.cuda.synchronize()
    assert qs.read_status(DEV) == 0
    assert torch.isfinite(out).all()
    assert torch.equal(out, ref), (out - ref).abs().max().item()
    assert torch.equal(lse, ref_lse)


def test_noalloc_matches_workspace_entry_point_twice():
    lib = qs.lib()
    cases = [synth.WORKLOADS["bf16_paged"].replace(B=6, k=8),                      # 48 units
             synth.WORKLOADS["ragged"].replace(B=3, ragged=(900, 5000, 1), MMBPR=None, k=5)]
    for i, w in enumerate(cases):       # two calls in a row, different sizes
        x, sel = _case(w, seed=11 + i)
        _check_equal(lib, w, x, sel)


def test_noalloc_clears_stale_counters():
    """Non-zero words planted where the arrival counters live (the first
    words of the array) would make a split unit's merge run early or never;
    the call must clear them before its kernel runs."""
    lib = qs.lib()
    w = synth.WORKLOADS["bf16_paged"].replace(B=5, k=8)   # 40 units, split between CTAs
    x, sel = _case(w, seed=21)
    words = _scratch_words(lib)
    for _ in range(2):
        words[:4096].fill_(0x7)
        torch.cuda.synchronize()
        _check_equal(lib, w, x, sel)


def test_noalloc_size_limit():
    """495 units at H/N = 4, D = 128 fit the 4 MiB scratch and match the
    workspace entry point; 496 units are refused before anything is
    enqueued."""
    lib = qs.lib()
    w = synth.WORKLOADS["bf16_paged"].replace(B=99, H=20, N=5, seq_len=600, MMBPR=None, k=3)
    assert w.B * w.N == 495
    x, sel = _case(w, seed=5)
    _check_equal(lib, w, x, sel)
    assert qs.workspace_size(qs.OP_SPARSE_ATTN, 62, 32, 8, 128, 128, 3, 8, 8) > 4 << 20
    words = _scratch_words(lib)
    words[:8].fill_(0x5)
    torch.cuda.synchronize()
    dummy = ctypes.c_void_p(16)
    # 62 requests x 8 KV heads = 496 units: refused from the size alone, and
    # the rejected call enqueues nothing (the planted words stay)
    rc = _fn(lib)(dummy, 1, dummy, dummy, None, None, 1, 1, dummy, 1, dummy, dummy, 8, 3, 0.1,
                  62, 32, 8, 128, 128, dummy, None, dummy, None)
    assert rc == QS_EWORKSPACE
    torch.cuda.synchronize()
    assert torch.all(words[:8] == 0x5)


def test_noalloc_rejected_call_leaves_the_array_alone():
    """A call that fails an argument check (here: an unsupported head dim)
    writes nothing to the shared array."""
    lib = qs.lib()
    w = synth.WORKLOADS["bf16_paged"].replace(B=2, seq_len=600, MMBPR=None, k=3)
    x, sel = _case(w, seed=6)
    words = _scratch_words(lib)
    words[:16].fill_(0x9)
    torch.cuda.synchronize()
    out = torch.empty((w.B, w.H, w.D), device=DEV)
    bad = w.replace(D=96)
    rc = _noalloc(lib, x, bad, sel, out, None)
    assert rc != 0
    torch.cuda.synchronize()
    assert torch.all(words[:16] == 0x9)
    _check_equal(lib, w, x, sel)       # and the next good call still matches
