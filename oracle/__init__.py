"""ctypes front end of the reference oracle -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It takes numpy arrays (bf16/fp16 as raw
``uint16`` bits) and returns numpy arrays.  See ``oracle.h`` for the page
citations and the layouts.
"""
import ctypes

import numpy as np

from . import build as _build

F32, BF16, F16, I8 = 0, 1, 2, 3
_ERRORS = {-1: "EINVAL", -2: "ERANGE", -3: "EFORCED", -4: "EDUP"}

_lib = None


class OracleError(RuntimeError):
    pass


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        _lib = ctypes.CDLL(path)
        P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        _lib.orc_prefill_metadata.argtypes = [P, I, I, I, I, I, P, I, P, I, P, I, I, P, P]
        _lib.orc_update_metadata.argtypes = [P, I, I, I, I, I, P, P, I, P, I, P, I, I, P, P]
        _lib.orc_group_mean_query.argtypes = [P, I, I, I, I, I, P]
        _lib.orc_quest_scores.argtypes = [P, P, P, I, P, I, I, P, I, I, I, I, P, P]
        _lib.orc_quest_select.argtypes = [P, I, P, P, I, P, I, I, P, I, I, I, I, I, I, I, P, P]
        _lib.orc_forced_set.argtypes = [I, I, I, I, P]
        _lib.orc_probe_select.argtypes = [P, I, P, P, I, I, P, I, P, P, I, I, I, I, I, I, I, I,
                                          P, P, P, P]
        _lib.orc_sparse_attention.argtypes = [P, I, P, P, P, P, I, I, P, I, P, P, I, I, D, I, I,
                                              I, I, I, P, P]
        _lib.orc_quantize_query.argtypes = [P, I, I, P, P]
        _lib.orc_prefill_importance.argtypes = [P, I, P, P, I, I, P, I, P, I, I, I, I, I, I, D,
                                                I, P, P]
        for f in ("orc_prefill_metadata", "orc_update_metadata", "orc_group_mean_query",
                  "orc_quest_scores",
                  "orc_quest_select", "orc_forced_set", "orc_probe_select",
                  "orc_sparse_attention", "orc_quantize_query", "orc_prefill_importance"):
            getattr(_lib, f).restype = ctypes.c_int
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc < 0:
        raise OracleError("%s: %s" % (what, _ERRORS.get(rc, rc)))
    return rc


def _elem_np(dt):
    return {F32: np.float32, BF16: np.uint16, F16: np.uint16, I8: np.int8}[dt]


def prefill_metadata(k_cache, kv_dt, seq_lens, block_tables, meta_block_tables,
                     maxblocks, minblocks):
    """a1.  k_cache [P,BS,N,D]; maxblocks/minblocks [M,BS,N,D] are updated in
    place (same element dtype as k_cache) and returned."""
    P, BS, N, D = k_cache.shape
    k_cache = _c(k_cache, _elem_np(kv_dt))
    seq_lens = _c(seq_lens, np.int32)
    bt = _c(block_tables, np.int32)
    mbt = _c(meta_block_tables, np.int32)
    assert maxblocks.flags.c_contiguous and minblocks.flags.c_contiguous
    rc = lib().orc_prefill_metadata(_p(k_cache), kv_dt, P, BS, N, D, _p(seq_lens),
                                    len(seq_lens), _p(bt), bt.shape[1], _p(mbt), mbt.shape[1],
                                    maxblocks.shape[0], _p(maxblocks), _p(minblocks))
    _check(rc, "prefill_metadata")
    return maxblocks, minblocks


def update_metadata(k_cache, kv_dt, prev_lens, seq_lens, block_tables, meta_block_tables,
                    maxblocks, minblocks):
    """f1.  Rebuilds, in place, the metadata rows of the blocks touched since
    the requests held prev_lens tokens (see oracle.h); returns the arrays."""
    P, BS, N, D = k_cache.shape
    k_cache = _c(k_cache, _elem_np(kv_dt))
    prev = _c(prev_lens, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    bt = _c(block_tables, np.int32)
    mbt = _c(meta_block_tables, np.int32)
    assert maxblocks.flags.c_contiguous and minblocks.flags.c_contiguous
    rc = lib().orc_update_metadata(_p(k_cache), kv_dt, P, BS, N, D, _p(prev), _p(seq_lens),
                                   len(seq_lens), _p(bt), bt.shape[1], _p(mbt), mbt.shape[1],
                                   maxblocks.shape[0], _p(maxblocks), _p(minblocks))
    _check(rc, "update_metadata")
    return maxblocks, minblocks


def group_mean_query(q, q_dt, N):
    B, H, D = q.shape
    q = _c(q, _elem_np(q_dt))
    qg = np.zeros((B, N, D), np.float64)
    _check(lib().orc_group_mean_query(_p(q), q_dt, B, H, N, D, _p(qg)), "group_mean_query")
    return qg


def quest_scores(qg, maxblocks, minblocks, meta_dt, meta_block_tables, seq_lens):
    """a3 in double: returns (scores, abs_sums), both [B, N, MMBPR*BS] with NaN
    where j >= nb_b."""
    B, N, D = qg.shape
    M, BS, _, _ = maxblocks.shape
    mbt = _c(meta_block_tables, np.int32)
    MMBPR = mbt.shape[1]
    qg = _c(qg, np.float64)
    mx = _c(maxblocks, _elem_np(meta_dt))
    mn = _c(minblocks, _elem_np(meta_dt))
    sl = _c(seq_lens, np.int32)
    sc = np.full((B, N, MMBPR * BS), np.nan)
    ab = np.full((B, N, MMBPR * BS), np.nan)
    rc = lib().orc_quest_scores(_p(qg), _p(mx), _p(mn), meta_dt, _p(mbt), MMBPR, M, _p(sl),
                                B, N, D, BS, _p(sc), _p(ab))
    _check(rc, "quest_scores")
    return sc, ab


def quest_select(q, q_dt, maxblocks, minblocks, meta_dt, meta_block_tables, seq_lens,
                 N, k, t):
    """a2..a5: returns (selected [B,N,k] int32, fp32 scores [B,N,MMBPR*BS])."""
    B, H, D = q.shape
    M, BS, _, _ = maxblocks.shape
    mbt = _c(meta_block_tables, np.int32)
    MMBPR = mbt.shape[1]
    q = _c(q, _elem_np(q_dt))
    mx = _c(maxblocks, _elem_np(meta_dt))
    mn = _c(minblocks, _elem_np(meta_dt))
    sl = _c(seq_lens, np.int32)
    sel = np.full((B, N, k), -7, np.int32)
    sf = np.full((B, N, MMBPR * BS), np.nan, np.float32)
    rc = lib().orc_quest_select(_p(q), q_dt, _p(mx), _p(mn), meta_dt, _p(mbt), MMBPR, M,
                                _p(sl), B, H, N, D, BS, k, t, _p(sel), _p(sf))
    _check(rc, "quest_select")
    return sel, sf


def forced_set(seq_len, BS, t, nb):
    f = np.zeros(max(nb, 1), np.uint8)
    rc = lib().orc_forced_set(seq_len, BS, t, nb, _p(f))
    _check(rc, "forced_set")
    return f[:nb].astype(bool)


def quantize_query(qvec):
    qvec = _c(qvec, np.float32)
    q8 = np.zeros(qvec.shape[0], np.int8)
    s = np.zeros(1, np.float32)
    _check(lib().orc_quantize_query(_p(qvec), F32, qvec.shape[0], _p(q8), _p(s)), "quantize")
    return q8, float(s[0])


def probe_select(q, q_dt, k_cache, kv_dt, block_tables, seq_lens, N, k, n_probe,
                 importance=None, k_scale=None):
    """a6..a8: returns (selected [B,H,k], probe [B,H,MKBPR], imp_sum [B,MKBPR],
    n_imp [B,H])."""
    B, H, D = q.shape
    P, BS, _, _ = k_cache.shape
    bt = _c(block_tables, np.int32)
    MKBPR = bt.shape[1]
    q = _c(q, _elem_np(q_dt))
    kc = _c(k_cache, _elem_np(kv_dt))
    ks = None if k_scale is None else _c(k_scale, np.float32)
    sl = _c(seq_lens, np.int32)
    imp = None if importance is None else _c(importance, np.float32)
    S_max = 0 if imp is None else imp.shape[1]
    sel = np.full((B, H, k), -7, np.int32)
    probe = np.full((B, H, MKBPR), np.nan, np.float32)
    imps = np.full((B, MKBPR), np.nan, np.float32)
    nimp = np.zeros((B, H), np.int32)
    rc = lib().orc_probe_select(_p(q), q_dt, _p(kc), _p(ks), kv_dt, P, _p(bt), MKBPR, _p(sl),
                                _p(imp), S_max, B, H, N, D, BS, k, n_probe, _p(sel),
                                _p(probe), _p(imps), _p(nimp))
    _check(rc, "probe_select")
    return sel, probe, imps, nimp


def sparse_attention(q, q_dt, k_cache, v_cache, kv_dt, block_tables, seq_lens, selected,
                     N, softmax_scale=None, k_scale=None, v_scale=None):
    """a9 in double: returns (out [B,H,D] float64, lse [B,H] float64)."""
    B, H, D = q.shape
    P, BS, _, _ = k_cache.shape
    sel = _c(selected, np.int32)
    _, sel_heads, k = sel.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / np.sqrt(D)
    bt = _c(block_tables, np.int32)
    q = _c(q, _elem_np(q_dt))
    kc = _c(k_cache, _elem_np(kv_dt))
    vc = _c(v_cache, _elem_np(kv_dt))
    ks = None if k_scale is None else _c(k_scale, np.float32)
    vs = None if v_scale is None else _c(v_scale, np.float32)
    sl = _c(seq_lens, np.int32)
    out = np.zeros((B, H, D), np.float64)
    lse = np.zeros((B, H), np.float64)
    rc = lib().orc_sparse_attention(_p(q), q_dt, _p(kc), _p(vc), _p(ks), _p(vs), kv_dt, P,
                                    _p(bt), bt.shape[1], _p(sl), _p(sel), sel_heads, k,
                                    float(softmax_scale), B, H, N, D, BS, _p(out), _p(lse))
    _check(rc, "sparse_attention")
    return out, lse


def prefill_importance(q, q_dt, k_cache, kv_dt, block_tables, prefill_lens, N,
                       softmax_scale=None, k_scale=None, first_query=0):
    """f3 in double: q [B, S_max, H, D] (prefill queries), K through the
    paged cache.  Returns (importance [B, S_max] float64, lse [B, H, S_max]
    float64, NaN where not computed)."""
    B, S_max, H, D = q.shape
    P, BS, _, _ = k_cache.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / np.sqrt(D)
    bt = _c(block_tables, np.int32)
    q = _c(q, _elem_np(q_dt))
    kc = _c(k_cache, _elem_np(kv_dt))
    ks = None if k_scale is None else _c(k_scale, np.float32)
    pl = _c(prefill_lens, np.int32)
    imp = np.zeros((B, S_max), np.float64)
    lse = np.full((B, H, S_max), np.nan)
    rc = lib().orc_prefill_importance(_p(q), q_dt, _p(kc), _p(ks), kv_dt, P, _p(bt),
                                      bt.shape[1], _p(pl), S_max, B, H, N, D, BS,
                                      float(softmax_scale), int(first_query), _p(imp), _p(lse))
    _check(rc, "prefill_importance")
    return imp, lse


__all__ = ["F32", "BF16", "F16", "I8", "OracleError", "prefill_metadata", "update_metadata",
           "group_mean_query", "quest_scores", "quest_select", "forced_set", "quantize_query",
           "probe_select", "sparse_attention", "prefill_importance", "lib"]
