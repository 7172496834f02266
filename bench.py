"""Decode-step benchmark: select + sparse decode attention on one GB300.

One step = the whole hot path over one batch: block selection (Quest, or the
probe/importance selector) followed by the split-K sparse attention, enqueued
through the C ABI (qs_sparse_decode_step) and replayed as a CUDA graph.  The
metadata prefill is set-up, timed separately and reported on its own.

The headline workload (default: the ragged batch, B=64 requests of 2K-128K
tokens, the largest configuration) gives the contract keys (value, roofline,
e2e, cpu_baseline, clocks, gpu_launches); every workload of --configs is then
measured the same way and reported as its own record under "configs".

Timing: the step runs once for each of R input sets (same shapes and
lengths, other seeds), R chosen so that one rotation moves more than 3x the
129 MB L2, and the R steps are captured back to back in one CUDA graph, as
consecutive layers of one forward graph would run them; W warm-up steps,
then K steps (whole rotations, then single-step graphs for the remainder)
replayed back to back, each set's inputs evicted from L2 by the others'
traffic before its next turn.  value = the span of the K steps on the
launching stream's CUDA events / K.  The same loop with one graph per step
(which adds the graph-to-graph launch gap to every step) is reported beside
it.  Workloads too small for a rotation of at most
--max-sets sets are timed one step at a time with a 256 MiB L2 flush before
each.  The dominant kernel (the attention) and the selector are timed alone
the same way; a flushed one-step time is reported beside the value.  Under
torchrun every rank runs an independent replica (the path needs no
collective) and the slowest rank's time is reported.

JSON line keys: metric, value (us per step, lower is better), unit, roofline
(attention kernel vs the measured HBM copy bandwidth), selector (its own
bytes and rate), cpu_baseline (the reference oracle on the host, bounded
sample, with the CPU model and core count), e2e (the same step through the C
ABI from pinned host buffers, copies included), clocks, gpu_launches, configs,
prefill_importance and prefill_importance_i8 (the tensor-core importance
producer on the fp32 and int8 probe prefills, against the measured bf16
tensor rate).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from decode_sparse_attention_gb300 import synth  # noqa: E402

METRIC = "select+sparse decode-attn µs/step and achieved HBM GB/s (% of peak), 1×GB300"
UNIT = "us/step"
FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# distributed helpers (replicas; CPU-testable with gloo)
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, device=None) -> float:
    """Max of a per-rank float over the process group (identity without one)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# algorithmic bytes (per step) -- the counting rule of the design notes
# ---------------------------------------------------------------------------

def elem_bytes(dtype):
    return {torch.float32: 4, torch.bfloat16: 2, torch.float16: 2, torch.int8: 1}[dtype]


def selected_kv_bytes(sel: np.ndarray, seq_lens: np.ndarray, w, kv_es: int, int8: bool) -> int:
    """K and V bytes of the valid tokens of the selected blocks, each block
    counted once per KV head (the union over the group's query heads)."""
    total_tok = 0
    rows = sel.shape[1]
    for b in range(sel.shape[0]):
        L = int(seq_lens[b])
        if rows == w.N:
            groups = [[n] for n in range(w.N)]
        else:
            groups = [list(range(n * w.G, (n + 1) * w.G)) for n in range(w.N)]
        for grp in groups:
            blocks = set()
            for r in grp:
                blocks.update(int(j) for j in sel[b, r] if j >= 0)
            for j in blocks:
                total_tok += max(0, min(w.BS, L - j * w.BS))
    per_tok = w.D * kv_es * 2 + (8 if int8 else 0)
    return total_tok * per_tok


def step_bytes(w, x, sel, q_es):
    L = x["seq_lens"].cpu().numpy()
    kv_es = elem_bytes(x["k_cache"].dtype)
    int8 = x["k_cache"].dtype == torch.int8
    q = w.B * w.H * w.D * q_es
    kv = selected_kv_bytes(sel, L, w, kv_es, int8)
    idx = sel.size * 4
    out = w.B * w.H * w.D * 4
    if w.mode == "quest":
        rows = sum((int(l) + w.BS - 1) // w.BS for l in L)
        select = rows * w.N * w.D * kv_es * 2
    else:
        # probed K rows + the importance of every token
        select = 0
        for l in L:
            nb = (int(l) + w.BS - 1) // w.BS
            for j in range(nb):
                valid = min(w.BS, int(l) - j * w.BS)
                step = max(1, valid // max(w.n_probe, 1))
                select += len(range(0, valid, step)) * w.N * (w.D * kv_es + (4 if int8 else 0))
        if w.importance:
            select += int(L.sum()) * 4
    return {"q": q, "select": select, "kv": kv, "indices": idx, "out": out,
            "step": q + select + kv + idx + out, "attention": q + kv + idx + out}


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.proc = None
        # raw samples: QS_CLOCKS_DIR if set (to keep them), else a temporary folder
        out_dir = os.environ.get("QS_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, "clocks_rank%d.csv" % gpu_index)
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + CLOCK_QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() in ("active", "0x1", "1"):
                        reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# peaks and committed ncu traffic
# ---------------------------------------------------------------------------

def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 tensor rate for a kernel timed alone: the measured burst
    figure (MEASURED_PEAKS.json), else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            v = float(json.load(f)["bf16_tflops"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("qs_attention.cu", "qs_attention_kernel.cuh", "qs_common.cuh"):
        with open(os.path.join(ROOT, "decode_sparse_attention_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(workload: str):
    """dram read+write bytes per attention launch from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "sparse_attn_%s.md" % workload)
    try:
        txt = open(p).read()
    except OSError:
        return None
    m_hash = re.search(r"source_sha256_16:\s*([0-9a-f]+)", txt)
    m_val = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", txt)
    if not m_hash or not m_val or m_hash.group(1) != kernel_source_hash():
        return None
    return int(m_val.group(1))


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------

def setup(w, seed, dev, fused_select=-1, seq_lens=None):
    from decode_sparse_attention_gb300 import questsparse as qs
    x = synth.make(w, seed=seed, device=dev, seq_lens=seq_lens)
    mode = 0 if w.mode == "quest" else 1
    meta_ms = None
    if mode == 0:
        # metadata prefill: set-up of the step, timed on its own
        for _ in range(2):
            qs.quest_prefill_metadata(x["k_cache"], x["meta_seq_lens"], x["block_tables"],
                                      x["meta_block_tables"], x["maxblocks"], x["minblocks"])
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        qs.quest_prefill_metadata(x["k_cache"], x["meta_seq_lens"], x["block_tables"],
                                  x["meta_block_tables"], x["maxblocks"], x["minblocks"])
        e1.record()
        torch.cuda.synchronize()
        meta_ms = e0.elapsed_time(e1)
    rows = w.N if mode == 0 else w.H
    sel = torch.full((w.B, rows, w.k), -1, dtype=torch.int32, device=dev)
    out = torch.empty((w.B, w.H, w.D), dtype=torch.float32, device=dev)
    nbytes = qs.step_workspace_bytes(mode, w.B, w.H, w.N, w.D, w.BS, w.k,
                                     MMBPR=x["meta_block_tables"].shape[1], MKBPR=x["MKBPR"])
    ws = qs.workspace(nbytes, dev, "bench-step")
    params = qs.make_step_params(mode, x["q"], x["k_cache"], x["v_cache"], x["block_tables"],
                                 x["seq_lens"], w.k, sel, out, ws, maxblocks=x.get("maxblocks"),
                                 minblocks=x.get("minblocks"),
                                 metadata_block_tables=x["meta_block_tables"],
                                 tokens_since_metadata_update=x["t"],
                                 importance=x.get("importance"), n_probe=w.n_probe,
                                 k_scale=x.get("k_scale"), v_scale=x.get("v_scale"),
                                 fused_select=fused_select)
    return x, mode, sel, out, params, meta_ms


def metadata_update(w, x, dev, flush, sink, reps=5):
    """Times the incremental metadata update for one decoded block per request
    (the metadata is refreshed every BS tokens): rows rebuilt since
    prev = meta_len - BS, one update after an L2 flush per sample.  Returns
    (median us, bytes: K read for the touched blocks + rows written)."""
    from decode_sparse_attention_gb300 import questsparse as qs
    L = x["meta_seq_lens"]
    prev = torch.clamp(L - w.BS, min=0).to(torch.int32)
    args = (x["k_cache"], prev, L, x["block_tables"], x["meta_block_tables"], x["maxblocks"],
            x["minblocks"])
    for _ in range(2):
        qs.quest_update_metadata(*args)
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        flush_l2(flush, sink)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        qs.quest_update_metadata(*args)
        e1.record()
        torch.cuda.synchronize()
        times.append(1000.0 * e0.elapsed_time(e1))
    es = elem_bytes(x["k_cache"].dtype)
    row = w.N * w.D * es
    nbytes = 0
    for p0, l in zip(prev.cpu().tolist(), L.cpu().tolist()):
        nb = (l + w.BS - 1) // w.BS
        rows = (nb + w.BS - 1) // w.BS * w.BS
        zero_from = max(nb, ((p0 + w.BS - 1) // w.BS + w.BS - 1) // w.BS * w.BS)
        for j in range(p0 // w.BS, rows):
            if j < nb:
                nbytes += min(w.BS, l - j * w.BS) * row + 2 * row
            elif j >= zero_from:
                nbytes += 2 * row
    return statistics.median(times), nbytes


def importance_tile_ops(lens, S_max, H, N):
    """128 x 128 tensor-core tiles the two passes of the prefill importance
    producer multiply, for prefill lengths `lens` (the loops of its kernels:
    rows pass, query tile qt against key tiles 0 .. last position / 128;
    column pass, key tile kt against query tiles kt*G .. (S*G - 1) / 128)."""
    G = H // N
    ntq = (S_max * G + 127) // 128
    ops = 0
    for S in lens:
        if S <= 0:
            continue
        for qt in range(ntq):
            if qt * 128 >= S * G:
                break
            last_pos = min(qt * 128 + 127, S * G - 1) // G
            ops += last_pos // 128 + 1
        for kt in range((S + 127) // 128):
            ops += max(0, (S * G + 127) // 128 - kt * G)
    return ops * N


def prefill_importance_timing(dev, workload="probe_importance", reps=5):
    """The prefill importance producer on the prefill of a probe workload
    (B=1, S=4096, H=16, N=8, D=128; fp32 cache for probe_importance, int8
    for probe_importance_i8): median of `reps` calls timed with CUDA events
    after two warm-up calls.  The passes run on the tensor cores (fp32
    operands split into bf16 high and low parts, three MMAs per product;
    int8 operands are exact in bf16, one MMA), so the roofline is the
    measured dense bf16 rate; executed flops count every 128 x 128 x D tile
    product the kernels issue (masked parts of diagonal tiles included),
    algorithmic flops one logit (2*D) per causal (query row, key) pair."""
    from decode_sparse_attention_gb300 import questsparse as qs
    from decode_sparse_attention_gb300 import synth
    w = synth.WORKLOADS[workload]
    x = synth.make(w, seed=0, device=dev)
    S_max = x["MKBPR"] * w.BS
    q = synth.prefill_queries(w, S_max, seed=0, device=dev)
    int8 = x["k_cache"].dtype == torch.int8
    args = (q, x["k_cache"], x["block_tables"], x["seq_lens"])
    kw = {"k_scale": x["k_scale"]} if int8 else {}
    for _ in range(2):
        qs.prefill_importance(*args, **kw)
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        qs.prefill_importance(*args, **kw)
        e1.record()
        torch.cuda.synchronize()
        times.append(1000.0 * e0.elapsed_time(e1))
    us = statistics.median(times)
    lens = x["seq_lens"].cpu().tolist()
    pairs = sum(int(S) * (int(S) + 1) // 2 for S in lens)
    alg = 2.0 * w.D * w.H * pairs
    products = 3 if x["k_cache"].dtype == torch.float32 else 1
    executed = importance_tile_ops(lens, S_max, w.H, w.N) * 2.0 * 128 * 128 * w.D * products
    peak, peak_kind = tensor_peak()
    cache = {torch.float32: "fp32", torch.int8: "int8", torch.bfloat16: "bf16",
             torch.float16: "fp16"}[x["k_cache"].dtype]
    packing = "pack_kernel (queries, keys)"
    if int8:
        packing = "quantize_rows_kernel (queries) + " + packing
    return {
        "kernels": packing + " + importance_tc_kernel (rows, columns) + importance_sum_kernel",
        "workload": "%s prefill: B=%d S=%d H=%d N=%d D=%d BLOCK_SIZE=%d %s cache, %s queries" % (
            workload, w.B, S_max, w.H, w.N, w.D, w.BS, cache, str(q.dtype).replace("torch.", "")),
        "us": round(us, 1),
        "bound": "tensor",
        "algorithmic_tflops": round(alg / (us * 1e-6) / 1e12, 2),
        "executed_tflops": round(executed / (us * 1e-6) / 1e12, 2),
        "peak_tflops": peak,
        "peak_kind": peak_kind,
        "frac_executed": round(executed / (us * 1e-6) / 1e12 / peak, 4),
        "products_per_logit": products,
        "status": qs.read_status(dev),
    }


def flush_l2(flush, sink):
    """Evict the L2: write a buffer twice the L2 size, then read it back, so
    the next kernel starts with none of its inputs cached and no dirty lines
    left to write back on its time."""
    flush.add_(1)
    torch.sum(flush.view(torch.int32), dim=0, out=sink)


def timed_graph(graph, flush, sink, steps, stream):
    """Per-step CUDA-event durations (ms) of replays of one graph with an L2
    flush between steps (each replay bracketed by its own events)."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    with torch.cuda.stream(stream):     # flush, replay and both events on one stream
        for s, e in evs:
            flush_l2(flush, sink)
            s.record(stream)
            graph.replay()
            e.record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in evs]


def timed_rotation(graphs, steps, stream):
    """Back-to-back replays cycling through the graphs of R input sets (the
    other R-1 sets' traffic evicts a set's inputs from L2 before its next
    turn).  Returns the per-step intervals between consecutive events (ms)
    and the whole span (ms) from the first event to the last."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for i in range(steps):
            graphs[i % len(graphs)].replay()
            evs[i + 1].record(stream)
    torch.cuda.synchronize()
    iv = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
    return iv, evs[0].elapsed_time(evs[-1])


def capture_rotation(fns, stream):
    """One CUDA graph holding one call of each fn, back to back on one stream
    (each fn was already run once eagerly by capture())."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for fn in fns:
            fn()
    return g


def timed_rotation_graph(g_rot, singles, steps, stream):
    """Exactly `steps` steps: the rotation graph (one step per input set)
    replayed back to back, then single-step graphs for the remainder.
    Returns per-step times (ms) of each rotation (its interval / R) and the
    whole span (ms) from the first event to the last."""
    R = len(singles)
    full, rest = divmod(steps, R)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(full + 2)]
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for i in range(full):
            g_rot.replay()
            evs[i + 1].record(stream)
        for i in range(rest):
            singles[i].replay()
        evs[-1].record(stream)
    torch.cuda.synchronize()
    iv = [evs[i].elapsed_time(evs[i + 1]) / R for i in range(full)]
    return iv, evs[0].elapsed_time(evs[-1])


def l2_bytes(dev):
    try:
        return int(torch.cuda.get_device_properties(dev).L2_cache_size)
    except (AttributeError, RuntimeError):
        return 126 << 20


def capture(fn, stream):
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def host_cpu():
    """CPU model and logical core count of this host (for the CPU baseline)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"cpu_model": model or "unknown", "nproc": os.cpu_count()}


def committed_selector_traffic(workload: str):
    """dram read+write bytes of the selector kernels of one step from the
    committed ncu summary, if taken on the current selector source."""
    p = os.path.join(ROOT, "profiles", "sparse_attn_%s.md" % workload)
    try:
        txt = open(p).read()
    except OSError:
        return None
    m_hash = re.search(r"selector_source_sha256_16:\s*([0-9a-f]+)", txt)
    m_val = re.search(r"selector_dram_bytes_per_step:\s*([0-9]+)", txt)
    if not m_hash or not m_val or m_hash.group(1) != selector_source_hash():
        return None
    return int(m_val.group(1))


def selector_source_hash():
    h = hashlib.sha256()
    for f in ("qs_select.cu", "qs_probe.cu", "qs_topk.cuh", "qs_quest_score.cuh", "qs_common.cuh"):
        with open(os.path.join(ROOT, "decode_sparse_attention_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measure(args, w, dev, stream, flush, sink, rank, cpu_seconds, headline):
    """Times one workload's decode step (and its selector and attention
    alone); returns its record.  headline: also the metadata update and the
    prefill importance producer."""
    from decode_sparse_attention_gb300 import questsparse as qs

    # input set 0, its step bytes, then as many more sets (same lengths, other
    # seeds) as it takes for the rotation to exceed 3x the L2
    sets = [setup(w, args.seed + rank, dev, args.fused_select)]
    x0, mode, sel0, out0, params0, meta_ms = sets[0]
    with torch.cuda.stream(stream):
        for _ in range(3):
            qs.sparse_decode_step(params0, dev)
    torch.cuda.synchronize()
    assert qs.read_status(dev) == 0
    q_es = elem_bytes(x0["q"].dtype)
    nbytes = step_bytes(w, x0, sel0.cpu().numpy(), q_es)
    n_sets = max(2, math.ceil(3 * l2_bytes(dev) / max(nbytes["step"], 1)) + 1)
    rotate = n_sets <= args.max_sets
    if rotate:
        seq = x0["seq_lens"].cpu().tolist()
        for i in range(1, n_sets):
            sets.append(setup(w, args.seed + rank + 1000 * i, dev, args.fused_select,
                              seq_lens=seq))

    # graphs: the step, the selector alone and the attention alone per set
    g_step, g_sel, g_attn = [], [], []
    f_step, f_sel, f_attn = [], [], []
    keep = []   # buffers the captured graphs write into must outlive them
    for (x, _, sel, out, params, _) in sets:
        f_step.append(lambda params=params: qs.sparse_decode_step(params, dev))
        g_step.append(capture(f_step[-1], stream))
        sel2 = torch.empty_like(sel)

        def run_selector(x=x, sel2=sel2):
            if mode == 0:
                qs.quest_block_select_paged_in_out_w(x["q"], x["maxblocks"], x["minblocks"],
                                                     x["meta_block_tables"], x["seq_lens"],
                                                     x["t"], sel2)
            else:
                qs.probe_select(x["q"], x["k_cache"], x["block_tables"], x["seq_lens"], w.k,
                                w.n_probe, importance=x.get("importance"),
                                k_scale=x.get("k_scale"), selected=sel2)
        f_sel.append(run_selector)
        g_sel.append(capture(run_selector, stream))
        attn_out = torch.empty_like(out)

        def run_attn(x=x, sel=sel, attn_out=attn_out):
            qs.sparse_decode_attn(x["q"], x["k_cache"], x["v_cache"], x["block_tables"],
                                  x["seq_lens"], sel, k_scale=x.get("k_scale"),
                                  v_scale=x.get("v_scale"), out=attn_out)
        f_attn.append(run_attn)
        g_attn.append(capture(run_attn, stream))
        keep.append((sel2, attn_out))
    # the R steps (and the kernels alone) of one rotation back to back in one
    # graph, as consecutive layers of one forward graph would run them
    r_step = r_sel = r_attn = None
    if rotate:
        r_step = capture_rotation(f_step, stream)
        r_sel = capture_rotation(f_sel, stream)
        r_attn = capture_rotation(f_attn, stream)
    torch.cuda.synchronize()
    # algorithmic bytes: the mean over the sets (selections differ per set)
    per_set = [step_bytes(w, s[0], s[2].cpu().numpy(), q_es) for s in sets]
    nbytes = {k: int(round(sum(d[k] for d in per_set) / len(per_set))) for k in per_set[0]}

    sampler = ClockSampler(dev.index or 0)
    t_end = time.time() + args.preroll_s
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            if not rotate:
                flush_l2(flush, sink)
            g_step[i % len(g_step)].replay()
        while time.time() < t_end:  # keep the clocks under load for the sampler
            for g in g_step:
                g.replay()
    torch.cuda.synchronize()
    barrier()
    if rotate:
        durs, span = timed_rotation_graph(r_step, g_step, args.steps, stream)
        step_us = 1000.0 * span / args.steps
        _, span1 = timed_rotation(g_step, args.steps, stream)
        step_us_graph_per_step = 1000.0 * span1 / args.steps
    else:
        durs = timed_graph(g_step[0], flush, sink, args.steps, stream)
        step_us = 1000.0 * sum(durs) / len(durs)
        step_us_graph_per_step = step_us
    barrier()
    n_side = max(args.steps // 2, 3)
    if rotate:
        _, attn_span = timed_rotation_graph(r_attn, g_attn, n_side, stream)
        _, sel_span = timed_rotation_graph(r_sel, g_sel, n_side, stream)
        attn_us = 1000.0 * attn_span / n_side
        sel_us = 1000.0 * sel_span / n_side
    else:
        attn_us = 1000.0 * statistics.mean(timed_graph(g_attn[0], flush, sink, n_side, stream))
        sel_us = 1000.0 * statistics.median(timed_graph(g_sel[0], flush, sink, n_side, stream))
    # the same step, one at a time after an L2 flush (each bracketed by its
    # own events: includes the graph launch latency a lone step pays)
    flushed = timed_graph(g_step[0], flush, sink, max(args.steps // 4, 3), stream)
    clocks = sampler.stop()
    assert qs.read_status(dev) == 0

    step_us_max = max_over_ranks(step_us, dev)

    # end to end through the C ABI from pinned host buffers
    x, _, _, out, params, _ = sets[0]
    host = {k: x[k].cpu().pin_memory() for k in ("q", "seq_lens", "block_tables",
                                                 "meta_block_tables")}
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = host_out.numel() * host_out.element_size()
    e2e_ms = []
    for i in range(max(args.steps // 4, 3) + 3):
        flush_l2(flush, sink)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for k_, v in host.items():
                x[k_].copy_(v, non_blocking=True)
            qs.sparse_decode_step(params, dev)
            host_out.copy_(out, non_blocking=True)
        stream.synchronize()
        if i >= 3:
            e2e_ms.append(1000.0 * (time.perf_counter() - t0))
    e2e_us = max_over_ranks(1000.0 * statistics.median(e2e_ms), dev)

    peak, peak_kind = hbm_peak()
    achieved = nbytes["attention"] / (attn_us * 1e-6) / 1e9
    sel_gbs = nbytes["select"] / (sel_us * 1e-6) / 1e9
    kernels = qs.step_kernels(params0)
    rec = {
        "workload": w.name,
        "config": {
            "workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "block_size": w.BS,
            "seq_len": w.seq_len if w.seq_len else "ragged", "k": w.k,
            "tokens_since_metadata_update": x0["t"], "selector": w.mode,
            "n_probe": w.n_probe if w.mode == "probe" else None,
            "kv_dtype": w.kv_dtype, "q_dtype": w.q_dtype,
            "l2": ("inputs larger than L2: %d input sets (same lengths, other seeds) replayed in "
                   "rotation, %.0f MB of step traffic per rotation vs %d MB of L2"
                   % (len(sets), len(sets) * nbytes["step"] / 1e6, l2_bytes(dev) >> 20))
                  if rotate else "256 MiB written then read back between timed steps",
            "step": ("qs_sparse_decode_step once per input set, the R steps of a rotation "
                     "captured back to back in one CUDA graph (as consecutive layers of one "
                     "forward graph run); the graph replayed back to back, value = span / "
                     "steps; step_us_graph_per_step: one graph per step instead"
                     if rotate else
                     "qs_sparse_decode_step captured as one CUDA graph; value = mean of "
                     "per-step event pairs"),
            "fused_select": args.fused_select,
            "kernels_per_step": kernels,
        },
        "dtype": {torch.bfloat16: "bf16", torch.float32: "f32", torch.float16: "f16",
                  torch.int8: "i8"}[x0["k_cache"].dtype],
        "us_per_step": round(step_us_max, 3),
        "step_gbs": round(nbytes["step"] / (step_us_max * 1e-6) / 1e9, 1),
        "step_frac_of_peak": round(nbytes["step"] / (step_us_max * 1e-6) / 1e9 / peak, 4),
        "step_frac_of_8tbs": round(nbytes["step"] / (step_us_max * 1e-6) / 1e9 / 8000.0, 4),
        "algorithmic_bytes": nbytes,
        "step_us_p10_p50_p90": [round(1000 * float(np.percentile(durs, p)), 3) for p in (10, 50, 90)],
        "step_us_graph_per_step": round(step_us_graph_per_step, 3),
        "step_us_flushed_single": round(1000.0 * statistics.median(flushed), 3),
        "roofline": {
            "kernel": "sparse_attn_kernel",
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": committed_traffic(w.name),
            "launch_us": round(attn_us, 3),
            "bytes_per_launch": nbytes["attention"],
        },
        "selector": {
            "kernels": ("quest_select_unit_kernel" if w.mode == "quest" and
                        x0["meta_block_tables"].shape[1] * w.BS <= 128
                        else "quest_scan_kernel + quest_unit_topk_kernel" if w.mode == "quest"
                        else "probe_select_kernel"),
            "us": round(sel_us, 3),
            "bytes": nbytes["select"],
            "achieved_gbs": round(sel_gbs, 1),
            "frac": round(sel_gbs / peak, 4),
            "traffic": committed_selector_traffic(w.name),
        },
        "metadata_prefill_us": None if meta_ms is None else round(meta_ms * 1000, 2),
        "e2e": {"value": round(e2e_us, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "clocks": clocks,
        "gpu_launches": kernels * args.steps,
    }
    if meta_ms is not None:
        L = x0["meta_seq_lens"].cpu().numpy()
        kbytes = int(sum(int(l) for l in L)) * w.N * w.D * elem_bytes(x0["k_cache"].dtype)
        mrows = sum(((int(l) + w.BS - 1) // w.BS + w.BS - 1) // w.BS * w.BS
                    for l in x0["seq_lens"].cpu().numpy())
        mbytes = mrows * w.N * w.D * elem_bytes(x0["k_cache"].dtype) * 2
        rec["metadata_prefill_gbs"] = round((kbytes + mbytes) / (meta_ms * 1e-3) / 1e9, 1)
        if headline:
            upd_us, upd_bytes = metadata_update(w, x0, dev, flush, sink)
            rec["metadata_update_us"] = round(upd_us, 2)
            rec["metadata_update_gbs"] = round(upd_bytes / (upd_us * 1e-6) / 1e9, 1)
            rec["metadata_update"] = ("one decoded block per request: rows rebuilt since "
                                      "meta_len - BS, one update after an L2 flush, %d bytes"
                                      % upd_bytes)
    if rank == 0 and cpu_seconds > 0:
        rec["cpu_baseline"] = cpu_baseline(w, x0, cpu_seconds)
    del sets, keep, g_step, g_sel, g_attn, r_step, r_sel, r_attn, f_step, f_sel, f_attn
    return rec


SUB_CONFIGS = "bf16_paged,fp16_paged,probe_importance,probe_importance_i8,long_context"


def run_ours(args, w):
    from decode_sparse_attention_gb300 import questsparse as qs
    ws_, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws_ > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    qs.lib()
    stream = torch.cuda.Stream(dev)
    flush = torch.zeros(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    sink = torch.zeros((), dtype=torch.int64, device=dev)

    cpu = 0 if args.no_cpu_baseline else args.cpu_seconds
    head = measure(args, w, dev, stream, flush, sink, rank, cpu, headline=True)
    torch.cuda.empty_cache()
    subs = {}
    names = [n for n in (args.configs.split(",") if args.configs else []) if n and n != w.name]
    for name in names:
        sub_cpu = 0 if args.no_cpu_baseline else args.sub_cpu_seconds
        subs[name] = measure(args, synth.WORKLOADS[name], dev, stream, flush, sink, rank, sub_cpu,
                             headline=False)
        torch.cuda.empty_cache()

    res = {
        "metric": METRIC,
        "value": head["us_per_step"],
        "unit": UNIT,
        "n_gpus": ws_,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(head["us_per_step"] / 1000.0, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": head["dtype"],
        "data": "synthetic",
        "config": dict(head["config"], parallelism="replicas" if ws_ > 1 else "single GPU"),
    }
    for k_ in ("step_gbs", "step_frac_of_peak", "step_frac_of_8tbs", "algorithmic_bytes",
               "step_us_p10_p50_p90", "step_us_graph_per_step", "step_us_flushed_single", "roofline",
               "selector",
               "metadata_prefill_us", "metadata_prefill_gbs", "metadata_update_us",
               "metadata_update_gbs", "metadata_update", "e2e", "clocks", "gpu_launches",
               "cpu_baseline"):
        if k_ in head:
            res[k_] = head[k_]
    if rank == 0 and not args.no_importance:
        which = [v for v in args.importance.split(",") if v]
        if "fp32" in which:
            res["prefill_importance"] = prefill_importance_timing(dev, "probe_importance")
        if "int8" in which:
            res["prefill_importance_i8"] = prefill_importance_timing(dev, "probe_importance_i8")
    res["configs"] = subs
    if ws_ > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return res if rank == 0 else None



# ---------------------------------------------------------------------------
# oracle on the host (CPU baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def _np_bits(t):
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def oracle_inputs(w, x, reqs):
    """Host copies of the sampled requests (their pages renumbered), with the
    oracle's own metadata for the Quest selector (built untimed: it is set-up)."""
    import oracle
    bt = x["block_tables"].cpu().numpy()[reqs]
    pages = sorted(set(int(p) for p in bt.ravel() if p >= 0))
    remap = {p: i for i, p in enumerate(pages)}
    bt2 = np.vectorize(lambda p: remap.get(int(p), -1))(bt).astype(np.int32)
    idx = torch.tensor(pages, dtype=torch.long, device=x["k_cache"].device)
    sub = {"q": _np_bits(x["q"][reqs]), "seq_lens": x["seq_lens"].cpu().numpy()[reqs],
           "k": _np_bits(x["k_cache"][idx]), "v": _np_bits(x["v_cache"][idx]), "bt": bt2}
    dt = {torch.float32: oracle.F32, torch.bfloat16: oracle.BF16, torch.float16: oracle.F16,
          torch.int8: oracle.I8}
    sub["q_dt"], sub["kv_dt"] = dt[x["q"].dtype], dt[x["k_cache"].dtype]
    if "k_scale" in x:
        sub["ks"], sub["vs"] = x["k_scale"][idx].cpu().numpy(), x["v_scale"][idx].cpu().numpy()
    if "importance" in x:
        sub["imp"] = x["importance"][reqs].cpu().numpy()
    if w.mode == "quest":
        mbt = x["meta_block_tables"].cpu().numpy()[reqs]
        n_meta = int((mbt >= 0).sum())
        mbt2 = np.full_like(mbt, -1)
        c = 0
        for r in range(mbt.shape[0]):
            for s in range(mbt.shape[1]):
                if mbt[r, s] >= 0:
                    mbt2[r, s] = c
                    c += 1
        shape = (max(n_meta, 1), w.BS, w.N, w.D)
        mx = np.zeros(shape, sub["k"].dtype)
        mn = np.zeros(shape, sub["k"].dtype)
        oracle.prefill_metadata(sub["k"], sub["kv_dt"], x["meta_seq_lens"].cpu().numpy()[reqs],
                                bt2, mbt2, mx, mn)
        sub.update(mx=mx, mn=mn, mbt=mbt2)
    return sub


def oracle_step(w, t, sub):
    import oracle
    if w.mode == "quest":
        sel, _ = oracle.quest_select(sub["q"], sub["q_dt"], sub["mx"], sub["mn"], sub["kv_dt"],
                                     sub["mbt"], sub["seq_lens"], w.N, w.k, t)
    else:
        sel, *_ = oracle.probe_select(sub["q"], sub["q_dt"], sub["k"], sub["kv_dt"], sub["bt"],
                                      sub["seq_lens"], w.N, w.k, w.n_probe,
                                      importance=sub.get("imp"), k_scale=sub.get("ks"))
    oracle.sparse_attention(sub["q"], sub["q_dt"], sub["k"], sub["v"], sub["kv_dt"], sub["bt"],
                            sub["seq_lens"], sel, w.N, k_scale=sub.get("ks"), v_scale=sub.get("vs"))


def oracle_sample_reqs(w, x, budget_s):
    """Requests to run per oracle step: grows until one step takes ~1/8 of the
    budget (at least one request)."""
    n = 1
    while True:
        reqs = list(range(min(n, w.B)))
        sub = oracle_inputs(w, x, reqs)
        t0 = time.perf_counter()
        oracle_step(w, x["t"], sub)
        dt = time.perf_counter() - t0
        if dt > budget_s / 8 or n >= w.B:
            return reqs, sub, dt
        n = min(w.B, max(n + 1, int(n * budget_s / 8 / max(dt, 1e-4))))


def cpu_baseline(w, x, budget_s):
    reqs, sub, _ = oracle_sample_reqs(w, x, budget_s)
    times = []
    t_stop = time.perf_counter() + budget_s
    while time.perf_counter() < t_stop or len(times) < 2:
        t0 = time.perf_counter()
        oracle_step(w, x["t"], sub)
        times.append(time.perf_counter() - t0)
    per_step_us = statistics.median(times) * 1e6 * w.B / len(reqs)
    return dict({"value": round(per_step_us, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
                 "sample": "%d of %d requests per step, %d runs, scaled by %d/%d to a full step"
                           % (len(reqs), w.B, len(times), w.B, len(reqs))}, **host_cpu())


def run_reference(args, w):
    ws_, rank, _ = dist_env()
    if rank != 0:
        return None
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    x = synth.make(w, seed=args.seed, device=dev)
    reqs, sub, dt = oracle_sample_reqs(w, x, min(args.cpu_seconds, 8.0))
    for _ in range(args.warmup):
        oracle_step(w, x["t"], sub)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(w, x["t"], sub)
        times.append(time.perf_counter() - t0)
    us = statistics.mean(times) * 1e6 * w.B / len(reqs)
    sample = ("oracle (single-threaded C, double) on %d of %d requests per step, scaled by %d/%d"
              % (len(reqs), w.B, w.B, len(reqs)))
    return {"impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT,
            "n_gpus": ws_, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(us / 1000, 4), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D,
                       "block_size": w.BS, "k": w.k, "selector": w.mode},
            "cpu_baseline": dict({"value": round(us, 1), "unit": UNIT, "cores": 1,
                                  "kind": "oracle", "sample": sample}, **host_cpu()),
            "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="ragged", choices=sorted(synth.WORKLOADS),
                    help="the headline workload (value, roofline, e2e)")
    ap.add_argument("--configs", default=SUB_CONFIGS,
                    help="comma-separated workloads measured after the headline, each reported "
                         "as its own record under 'configs' ('' for none)")
    ap.add_argument("--sub-cpu-seconds", type=float, default=4.0,
                    help="oracle seconds per record under 'configs'")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-importance", action="store_true",
                    help="skip timing the prefill importance producer")
    ap.add_argument("--importance", default="fp32,int8",
                    help="comma list of the importance producer timings to run: fp32 "
                         "(probe_importance prefill), int8 (probe_importance_i8 prefill)")
    ap.add_argument("--max-sets", type=int, default=128,
                    help="most input sets to rotate through; workloads needing more (tiny "
                         "steps) are timed with an L2 flush between steps instead")
    ap.add_argument("--fused-select", type=int, default=-1, choices=[-1, 0, 1],
                    help="Quest step: -1 library's choice, 0 selector + attention kernels, "
                         "1 the fused one-kernel step")
    ap.add_argument("--preroll-s", type=float, default=1.5,
                    help="seconds of back-to-back steps before the timed loop (clock sampling)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    w = synth.WORKLOADS[args.workload]
    res = run_reference(args, w) if args.impl == "reference" else run_ours(args, w)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
