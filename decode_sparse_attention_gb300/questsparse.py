"""Python binding of the questsparse C ABI (argument marshalling only).

Every step of the computation runs in the CUDA kernels of libquestsparse.so;
this module passes torch tensors' device pointers, sizes and the current CUDA
stream through ctypes.  It never computes a result itself and raises if the
library is missing.

Names follow the pages' Python interface (CANN select_attention_operators:
quest_prefill_metadata, quest_block_select_paged[_in_out[_w]]) plus the probe
selector and the sparse decode attention.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libquestsparse.so")

F32, BF16, F16, I8 = 0, 1, 2, 3
_DT = {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16, torch.int8: I8}
OP_BLOCK_SELECT, OP_PROBE_SELECT, OP_SPARSE_ATTN, OP_STEP_QUEST, OP_STEP_PROBE = range(5)

_lib = None
_lock = threading.Lock()


class QuestSparseError(RuntimeError):
    pass


P, I32, SZ, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float


class StepParams(ctypes.Structure):
    """Mirror of qs_step_params (include/questsparse.h)."""
    _fields_ = [
        ("mode", I32), ("q", P), ("q_dtype", I32),
        ("k_cache", P), ("v_cache", P), ("k_scale", P), ("v_scale", P), ("kv_dtype", I32),
        ("num_kv_blocks", I32), ("block_tables", P), ("MKBPR", I32), ("seq_lens", P),
        ("maxblocks", P), ("minblocks", P), ("meta_block_tables", P), ("MMBPR", I32),
        ("num_meta_blocks", I32), ("tokens_since_metadata_update", I32),
        ("importance", P), ("importance_stride", I32), ("n_probe", I32),
        ("B", I32), ("H", I32), ("N", I32), ("D", I32), ("BS", I32), ("k", I32),
        ("softmax_scale", F),
        ("selected", P), ("out", P), ("lse_opt", P),
        ("workspace", P), ("workspace_bytes", SZ), ("dev_status", P),
        ("fused_select", I32),
    ]


def lib():
    """The loaded CUDA library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise QuestSparseError(
                    "libquestsparse.so is not built; run decode_sparse_attention_gb300.build.build()")
            L = ctypes.CDLL(LIB_PATH)
            L.qs_version.restype = I32
            L.qs_status_string.argtypes = [I32]
            L.qs_status_string.restype = ctypes.c_char_p
            L.qs_read_status.argtypes = [P, P, I32, P]
            L.qs_workspace_size.argtypes = [I32, I32, I32, I32, I32, I32, I32, I32, I32,
                                            ctypes.POINTER(SZ)]
            L.qs_prefill_metadata.argtypes = [P, I32, I32, I32, I32, I32, P, I32, P, I32, P, I32,
                                              I32, P, P, P, P]
            L.qs_update_metadata.argtypes = [P, I32, I32, I32, I32, I32, P, P, I32, P, I32, P,
                                             I32, I32, P, P, P, P]
            L.qs_block_select_paged.argtypes = [P, I32, P, P, I32, P, I32, I32, P, I32, I32, I32,
                                                I32, I32, I32, I32, P, P, P, SZ, P, P]
            L.qs_probe_select.argtypes = [P, I32, P, P, I32, I32, P, I32, P, P, I32, I32, I32,
                                          I32, I32, I32, I32, I32, P, P, SZ, P, P]
            L.qs_sparse_decode_attn.argtypes = [P, I32, P, P, P, P, I32, I32, P, I32, P, P, I32,
                                                I32, F, I32, I32, I32, I32, I32, P, P, P, SZ, P,
                                                P]
            L.qs_prefill_importance_workspace_size.argtypes = [I32, I32, I32, I32, I32, I32,
                                                               ctypes.POINTER(SZ)]
            L.qs_prefill_importance.argtypes = [P, I32, P, P, I32, I32, P, I32, P, I32, I32, I32,
                                                I32, I32, I32, F, P, P, P, SZ, P, P]
            L.qs_sparse_decode_step.argtypes = [ctypes.POINTER(StepParams), P]
            L.qs_step_kernels.argtypes = [ctypes.POINTER(StepParams), P]
            L.qs_check_bounded_wait.argtypes = [P, P]
            for f in ("qs_read_status", "qs_workspace_size", "qs_prefill_metadata", "qs_check_bounded_wait",
                      "qs_block_select_paged", "qs_probe_select", "qs_sparse_decode_attn",
                      "qs_sparse_decode_step", "qs_update_metadata", "qs_step_kernels",
                      "qs_prefill_importance_workspace_size", "qs_prefill_importance"):
                getattr(L, f).restype = I32
            _lib = L
    return _lib


def _check(rc, what):
    if rc != 0:
        raise QuestSparseError("%s: %s" % (what, lib().qs_status_string(rc).decode()))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dt(t):
    try:
        return _DT[t.dtype]
    except KeyError:
        raise QuestSparseError("unsupported dtype %s" % t.dtype) from None


def _req(t, name, dtype=None, dim=None):
    if not t.is_cuda:
        raise QuestSparseError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise QuestSparseError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise QuestSparseError("%s must be %s" % (name, dtype))
    if dim is not None and t.dim() != dim:
        raise QuestSparseError("%s must have %d dims" % (name, dim))
    return t


def _rows(t, name, B):
    """t holds one row (or entry) per request: at least B of them."""
    if t.shape[0] < B:
        raise QuestSparseError("%s must have a row per request (%d < %d)" % (name, t.shape[0], B))


def _shape(t, name, shape):
    if tuple(t.shape) != tuple(shape):
        raise QuestSparseError("%s must be %s, got %s" % (name, list(shape), list(t.shape)))


# ---------------------------------------------------------------------------
# per-device scratch: the device status word and zero-initialised workspaces
# ---------------------------------------------------------------------------

_status = {}
_workspaces = {}


def status_word(device) -> torch.Tensor:
    device = torch.device(device)
    key = device.index if device.index is not None else torch.cuda.current_device()
    if key not in _status:
        _status[key] = torch.zeros(1, dtype=torch.int32, device=device)
    return _status[key]


def workspace_size(op, B, H, N, D, BS, k, max_blocks_per_req, sel_heads):
    n = SZ(0)
    _check(lib().qs_workspace_size(op, B, H, N, D, BS, k, max_blocks_per_req, sel_heads,
                                   ctypes.byref(n)), "qs_workspace_size")
    return n.value


def workspace(nbytes, device, key="default") -> torch.Tensor:
    """A zero-filled byte buffer of at least nbytes, cached per (device, key).

    A workspace belongs to one set of call sizes: the kernels rearm their
    arrival counters after every call, but the rest is scratch, so a buffer
    is only reused by calls whose key (op and sizes) is the same."""
    device = torch.device(device)
    k = (device.index if device.index is not None else torch.cuda.current_device(), key, nbytes)
    buf = _workspaces.get(k)
    if buf is None:
        buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[k] = buf
    return buf


def reset_workspace(buf: torch.Tensor):
    """Zero a workspace again (needed after a call reported a device error)."""
    buf.zero_()


def read_status(device=None, reset=True) -> int:
    """Device-side error code of the calls so far on this device (0 = none)."""
    device = torch.device(device or "cuda")
    st = status_word(device)
    code = ctypes.c_int32(0)
    _check(lib().qs_read_status(_ptr(st), ctypes.byref(code), 1 if reset else 0,
                                _stream(device)), "qs_read_status")
    return code.value


def check_bounded_wait(device=None) -> int:
    """Runs the device-side bounded-wait self-check on `device` and returns
    the device code it left (QS_DEV_ETIMEOUT, 6, when the wait ran out as it
    should)."""
    device = torch.device(device or "cuda")
    read_status(device)   # start from a clear status word
    st = status_word(device)
    _check(lib().qs_check_bounded_wait(_ptr(st), _stream(device)), "qs_check_bounded_wait")
    return read_status(device)


def device_error_string(code: int) -> str:
    return lib().qs_status_string(100 + code).decode()


# ---------------------------------------------------------------------------
# operations
# ---------------------------------------------------------------------------

def quest_prefill_metadata(k_cache, seq_lens, block_tables, metadata_block_tables, maxblocks,
                           minblocks):
    """Fills maxblocks/minblocks [num_meta, BS, N, D] with per-block channel
    max/min of K (zero rows for absent blocks).  Argument order as in the
    CANN page's usage example."""
    _req(k_cache, "k_cache", dim=4)
    P_, BS, N, D = k_cache.shape
    _req(seq_lens, "seq_lens", torch.int32, 1)
    _req(block_tables, "block_tables", torch.int32, 2)
    _req(metadata_block_tables, "metadata_block_tables", torch.int32, 2)
    for t, nm in ((maxblocks, "maxblocks"), (minblocks, "minblocks")):
        _req(t, nm, k_cache.dtype, 4)
        if tuple(t.shape[1:]) != (BS, N, D):
            raise QuestSparseError("%s must be [num_meta, BS, N, D]" % nm)
    B = seq_lens.shape[0]
    _rows(block_tables, "block_tables", B)
    _rows(metadata_block_tables, "metadata_block_tables", B)
    rc = lib().qs_prefill_metadata(_ptr(k_cache), _dt(k_cache), P_, BS, N, D, _ptr(seq_lens), B,
                                   _ptr(block_tables), block_tables.shape[1],
                                   _ptr(metadata_block_tables), metadata_block_tables.shape[1],
                                   maxblocks.shape[0], _ptr(maxblocks), _ptr(minblocks),
                                   _ptr(status_word(k_cache.device)), _stream(k_cache.device))
    _check(rc, "qs_prefill_metadata")


def quest_update_metadata(k_cache, prev_lens, seq_lens, block_tables, metadata_block_tables,
                          maxblocks, minblocks):
    """Refreshes maxblocks/minblocks after decoding: rebuilds the rows of the
    blocks touched since the requests held prev_lens tokens (the block that
    held the last tokens and every block begun since) and zeroes the tail rows
    of metadata blocks begun since, leaving the rest."""
    _req(k_cache, "k_cache", dim=4)
    P_, BS, N, D = k_cache.shape
    _req(prev_lens, "prev_lens", torch.int32, 1)
    _req(seq_lens, "seq_lens", torch.int32, 1)
    _req(block_tables, "block_tables", torch.int32, 2)
    _req(metadata_block_tables, "metadata_block_tables", torch.int32, 2)
    for t, nm in ((maxblocks, "maxblocks"), (minblocks, "minblocks")):
        _req(t, nm, k_cache.dtype, 4)
        if tuple(t.shape[1:]) != (BS, N, D):
            raise QuestSparseError("%s must be [num_meta, BS, N, D]" % nm)
    B = seq_lens.shape[0]
    if prev_lens.shape[0] != B:
        raise QuestSparseError("prev_lens and seq_lens must have one entry per request")
    _rows(block_tables, "block_tables", B)
    _rows(metadata_block_tables, "metadata_block_tables", B)
    rc = lib().qs_update_metadata(_ptr(k_cache), _dt(k_cache), P_, BS, N, D, _ptr(prev_lens),
                                  _ptr(seq_lens), B, _ptr(block_tables), block_tables.shape[1],
                                  _ptr(metadata_block_tables), metadata_block_tables.shape[1],
                                  maxblocks.shape[0], _ptr(maxblocks), _ptr(minblocks),
                                  _ptr(status_word(k_cache.device)), _stream(k_cache.device))
    _check(rc, "qs_update_metadata")


def quest_block_select_paged_in_out_w(query, maxblocks, minblocks, metadata_block_tables,
                                      seq_lens, tokens_since_metadata_update, selected_indices,
                                      scores=None):
    """Quest select with sink + window forcing; writes selected_indices
    [B, N, k] (in-sequence block indices, ascending, -1 padded)."""
    _req(query, "query", dim=3)
    B, H, D = query.shape
    _req(maxblocks, "maxblocks", dim=4)
    _req(minblocks, "minblocks", maxblocks.dtype, 4)
    M, BS, N, D2 = maxblocks.shape
    if D2 != D:
        raise QuestSparseError("head dim mismatch")
    _req(metadata_block_tables, "metadata_block_tables", torch.int32, 2)
    _req(seq_lens, "seq_lens", torch.int32, 1)
    _rows(metadata_block_tables, "metadata_block_tables", B)
    _rows(seq_lens, "seq_lens", B)
    _req(selected_indices, "selected_indices", torch.int32, 3)
    k = selected_indices.shape[2]
    if tuple(selected_indices.shape) != (B, N, k):
        raise QuestSparseError("selected_indices must be [B, N, k]")
    MMBPR = metadata_block_tables.shape[1]
    if scores is not None:
        _req(scores, "scores", torch.float32)
        if scores.numel() < B * N * MMBPR * BS:
            raise QuestSparseError("scores must hold [B, N, MMBPR*BS] floats")
    nbytes = workspace_size(OP_BLOCK_SELECT, B, H, N, D, BS, k, MMBPR * BS, N)
    ws = workspace(nbytes, query.device, ("select", B, H, N, D, BS, k, MMBPR))
    rc = lib().qs_block_select_paged(_ptr(query), _dt(query), _ptr(maxblocks), _ptr(minblocks),
                                     _dt(maxblocks), _ptr(metadata_block_tables), MMBPR, M,
                                     _ptr(seq_lens), B, H, N, D, BS, k,
                                     int(tokens_since_metadata_update), _ptr(selected_indices),
                                     _ptr(scores), _ptr(ws), ws.numel(),
                                     _ptr(status_word(query.device)), _stream(query.device))
    _check(rc, "qs_block_select_paged")
    return selected_indices


def quest_block_select_paged_in_out(query, maxblocks, minblocks, metadata_block_tables, seq_lens,
                                    selected_indices):
    """Quest select without the window (tokens_since_metadata_update = -1)."""
    return quest_block_select_paged_in_out_w(query, maxblocks, minblocks, metadata_block_tables,
                                             seq_lens, -1, selected_indices)


def quest_block_select_paged(query, maxblocks, minblocks, metadata_block_tables, seq_lens, k):
    """Quest select into a new [B, N, k] int32 tensor (window off)."""
    B = query.shape[0]
    N = maxblocks.shape[2]
    out = torch.empty((B, N, k), dtype=torch.int32, device=query.device)
    return quest_block_select_paged_in_out(query, maxblocks, minblocks, metadata_block_tables,
                                           seq_lens, out)


def probe_select(q, k_cache, block_tables, seq_lens, k, n_probe=8, importance=None,
                 k_scale=None, selected=None):
    """Probe / prefill-importance selection per query head: [B, H, k]."""
    _req(q, "q", dim=3)
    B, H, D = q.shape
    _req(k_cache, "k_cache", dim=4)
    P_, BS, N, D2 = k_cache.shape
    if D2 != D:
        raise QuestSparseError("head dim mismatch")
    _req(block_tables, "block_tables", torch.int32, 2)
    _req(seq_lens, "seq_lens", torch.int32, 1)
    _rows(block_tables, "block_tables", B)
    _rows(seq_lens, "seq_lens", B)
    if importance is not None:
        _req(importance, "importance", torch.float32, 2)
        _rows(importance, "importance", B)
    if k_scale is not None:
        _req(k_scale, "k_scale", torch.float32, 3)
        _shape(k_scale, "k_scale", (P_, BS, N))
    if selected is None:
        selected = torch.empty((B, H, k), dtype=torch.int32, device=q.device)
    _req(selected, "selected", torch.int32, 3)
    _shape(selected, "selected", (B, H, k))
    MKBPR = block_tables.shape[1]
    nbytes = workspace_size(OP_PROBE_SELECT, B, H, N, D, BS, k, MKBPR, H)
    ws = workspace(nbytes, q.device, ("probe", B, H, N, D, BS, k, MKBPR))
    rc = lib().qs_probe_select(_ptr(q), _dt(q), _ptr(k_cache), _ptr(k_scale), _dt(k_cache), P_,
                               _ptr(block_tables), MKBPR, _ptr(seq_lens), _ptr(importance),
                               0 if importance is None else importance.shape[1], B, H, N, D, BS,
                               k, n_probe, _ptr(selected), _ptr(ws), ws.numel(),
                               _ptr(status_word(q.device)), _stream(q.device))
    _check(rc, "qs_probe_select")
    return selected


def prefill_importance_workspace_size(B, H, N, D, S_max, kv_dtype):
    n = SZ(0)
    _check(lib().qs_prefill_importance_workspace_size(B, H, N, D, S_max, kv_dtype,
                                                      ctypes.byref(n)),
           "qs_prefill_importance_workspace_size")
    return n.value


def prefill_importance(q, k_cache, block_tables, prefill_lens, softmax_scale=None, k_scale=None,
                       importance=None, lse=None):
    """Prefill importance: the attention each prefill token received, summed
    over query heads and later query positions (causal, exact).

    q: [B, S_max, H, D] prefill query rows; K through block_tables into
    k_cache [P, BS, N, D].  Returns importance [B, S_max] fp32 (the layout
    probe_select takes); fills lse [B, H, S_max] when given."""
    _req(q, "q", dim=4)
    B, S_max, H, D = q.shape
    _req(k_cache, "k_cache", dim=4)
    P_, BS, N, D2 = k_cache.shape
    if D2 != D:
        raise QuestSparseError("head dim mismatch")
    _req(block_tables, "block_tables", torch.int32, 2)
    _req(prefill_lens, "prefill_lens", torch.int32, 1)
    _rows(block_tables, "block_tables", B)
    _rows(prefill_lens, "prefill_lens", B)
    if k_scale is not None:
        _req(k_scale, "k_scale", torch.float32, 3)
        _shape(k_scale, "k_scale", (P_, BS, N))
    if importance is None:
        importance = torch.empty((B, S_max), dtype=torch.float32, device=q.device)
    _req(importance, "importance", torch.float32, 2)
    _shape(importance, "importance", (B, S_max))
    if lse is not None:
        _req(lse, "lse", torch.float32, 3)
        _shape(lse, "lse", (B, H, S_max))
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    nbytes = prefill_importance_workspace_size(B, H, N, D, S_max, _dt(k_cache))
    ws = workspace(nbytes, q.device, ("importance", B, H, N, D, S_max))
    rc = lib().qs_prefill_importance(_ptr(q), _dt(q), _ptr(k_cache), _ptr(k_scale), _dt(k_cache),
                                     P_, _ptr(block_tables), block_tables.shape[1],
                                     _ptr(prefill_lens), S_max, B, H, N, D, BS,
                                     float(softmax_scale), _ptr(importance), _ptr(lse), _ptr(ws),
                                     ws.numel(), _ptr(status_word(q.device)), _stream(q.device))
    _check(rc, "qs_prefill_importance")
    return importance


def sparse_decode_attn(q, k_cache, v_cache, block_tables, seq_lens, selected, softmax_scale=None,
                       k_scale=None, v_scale=None, out=None, lse=None):
    """Exact attention over the selected blocks: returns out [B, H, D] fp32
    (and fills lse [B, H] when given)."""
    _req(q, "q", dim=3)
    B, H, D = q.shape
    _req(k_cache, "k_cache", dim=4)
    _req(v_cache, "v_cache", k_cache.dtype, 4)
    P_, BS, N, D2 = k_cache.shape
    if D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise QuestSparseError("cache shape mismatch")
    _req(block_tables, "block_tables", torch.int32, 2)
    _req(seq_lens, "seq_lens", torch.int32, 1)
    _rows(block_tables, "block_tables", B)
    _rows(seq_lens, "seq_lens", B)
    _req(selected, "selected", torch.int32, 3)
    sel_heads, k = selected.shape[1], selected.shape[2]
    if selected.shape[0] != B or sel_heads not in (N, H):
        raise QuestSparseError("selected must be [B, N, k] or [B, H, k]")
    for t, nm in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        if t is not None:
            _req(t, nm, torch.float32, 3)
            _shape(t, nm, (P_, BS, N))
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.float32, device=q.device)
    _req(out, "out", torch.float32, 3)
    _shape(out, "out", (B, H, D))
    if lse is not None:
        _req(lse, "lse", torch.float32)
        if lse.numel() != B * H:
            raise QuestSparseError("lse must hold [B, H] floats")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    nbytes = workspace_size(OP_SPARSE_ATTN, B, H, N, D, BS, k, block_tables.shape[1], sel_heads)
    ws = workspace(nbytes, q.device, ("attn", B, H, N, D, BS, k, sel_heads))
    rc = lib().qs_sparse_decode_attn(_ptr(q), _dt(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                     _ptr(v_scale), _dt(k_cache), P_, _ptr(block_tables),
                                     block_tables.shape[1], _ptr(seq_lens), _ptr(selected),
                                     sel_heads, k, float(softmax_scale), B, H, N, D, BS, _ptr(out),
                                     _ptr(lse), _ptr(ws), ws.numel(),
                                     _ptr(status_word(q.device)), _stream(q.device))
    _check(rc, "qs_sparse_decode_attn")
    return out


def make_step_params(mode, q, k_cache, v_cache, block_tables, seq_lens, k, selected, out,
                     ws, softmax_scale=None, maxblocks=None, minblocks=None,
                     metadata_block_tables=None, tokens_since_metadata_update=-1,
                     importance=None, n_probe=8, k_scale=None, v_scale=None, lse=None,
                     fused_select=-1):
    """Fills a qs_step_params for qs_sparse_decode_step (pointers are captured;
    keep the tensors alive while the params are in use).  fused_select (Quest
    mode): -1 lets the library choose between the fused one-kernel step and
    the selector + attention pair, 0 forces the pair, 1 the fused kernel
    whenever the sizes fit it."""
    B, H, D = q.shape
    P_, BS, N, _ = k_cache.shape
    p = StepParams()
    p.mode = mode
    p.q, p.q_dtype = q.data_ptr(), _dt(q)
    p.k_cache, p.v_cache = k_cache.data_ptr(), v_cache.data_ptr()
    p.k_scale = k_scale.data_ptr() if k_scale is not None else None
    p.v_scale = v_scale.data_ptr() if v_scale is not None else None
    p.kv_dtype = _dt(k_cache)
    p.num_kv_blocks = P_
    p.block_tables, p.MKBPR = block_tables.data_ptr(), block_tables.shape[1]
    p.seq_lens = seq_lens.data_ptr()
    if mode == 0:
        p.maxblocks, p.minblocks = maxblocks.data_ptr(), minblocks.data_ptr()
        p.meta_block_tables = metadata_block_tables.data_ptr()
        p.MMBPR = metadata_block_tables.shape[1]
        p.num_meta_blocks = maxblocks.shape[0]
        p.tokens_since_metadata_update = int(tokens_since_metadata_update)
    else:
        p.importance = importance.data_ptr() if importance is not None else None
        p.importance_stride = importance.shape[1] if importance is not None else 0
        p.n_probe = n_probe
    p.B, p.H, p.N, p.D, p.BS, p.k = B, H, N, D, BS, k
    p.softmax_scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    p.selected, p.out = selected.data_ptr(), out.data_ptr()
    p.lse_opt = lse.data_ptr() if lse is not None else None
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    p.dev_status = status_word(q.device).data_ptr()
    p.fused_select = int(fused_select)
    return p


def step_workspace_bytes(mode, B, H, N, D, BS, k, MMBPR=0, MKBPR=0):
    if mode == 0:
        return workspace_size(OP_STEP_QUEST, B, H, N, D, BS, k, MMBPR * BS, N)
    return workspace_size(OP_STEP_PROBE, B, H, N, D, BS, k, MKBPR, H)


def step_kernels(params: StepParams) -> int:
    """Number of kernels one qs_sparse_decode_step(params) launches (1: the
    fused Quest kernel, 2: selector + attention)."""
    n = I32(0)
    _check(lib().qs_step_kernels(ctypes.byref(params), ctypes.byref(n)), "qs_step_kernels")
    return int(n.value)


def sparse_decode_step(params: StepParams, device=None):
    """Enqueues one decode step (selector + attention) on the current stream."""
    device = torch.device(device or "cuda")
    _check(lib().qs_sparse_decode_step(ctypes.byref(params), _stream(device)),
           "qs_sparse_decode_step")
