"""Host-only checks: the C-ABI library builds, loads without a GPU and exports
every function include/questsparse.h declares; the Python binding rejects
bad arguments before any CUDA call; host-side helpers behave."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(qs_[a-z_0-9]+)\s*\(", txt))
    return names


@pytest.fixture(scope="module")
def built_lib():
    from decode_sparse_attention_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    for f in ("qs_prefill_metadata", "qs_update_metadata", "qs_block_select_paged",
              "qs_probe_select", "qs_sparse_decode_attn", "qs_sparse_decode_step",
              "qs_step_kernels", "qs_workspace_size", "qs_read_status", "qs_status_string",
              "qs_version", "qs_prefill_importance", "qs_prefill_importance_workspace_size"):
        assert f in names


def test_library_exports_every_declared_symbol(built_lib):
    for name in declared_functions():
        assert hasattr(built_lib, name), name


def test_status_strings_and_version(built_lib):
    built_lib.qs_status_string.restype = ctypes.c_char_p
    built_lib.qs_status_string.argtypes = [ctypes.c_int32]
    assert built_lib.qs_status_string(0) == b"ok"
    assert b"workspace" in built_lib.qs_status_string(5)
    assert b"block_tables" in built_lib.qs_status_string(101)
    assert built_lib.qs_version() >= 10000


def test_workspace_size_without_gpu(built_lib):
    from decode_sparse_attention_gb300 import questsparse as qs
    n = qs.workspace_size(qs.OP_BLOCK_SELECT, 20, 32, 8, 128, 128, 8, 128, 8)
    assert n >= 20 * 8 * 128 * 4                      # one fp32 score per block and KV head
    a = qs.workspace_size(qs.OP_SPARSE_ATTN, 20, 32, 8, 128, 128, 8, 128, 8)
    assert a >= 160 * 4 + 160 * 4 * 130 * 4
    s = qs.workspace_size(qs.OP_STEP_QUEST, 20, 32, 8, 128, 128, 8, 128, 8)
    assert s >= n + a
    with pytest.raises(qs.QuestSparseError):
        qs.workspace_size(qs.OP_SPARSE_ATTN, 2, 32, 8, 128, 128, 8, 128, 5)   # sel_heads


def test_prefill_importance_workspace_without_gpu(built_lib):
    """Row log-sum-exps (B*H*S_max fp32) plus per-part column sums; fp32,
    bf16 and fp16 caches add the packed bf16/fp16 operand tiles of the
    tensor-core passes (queries B*S_max*H*D and keys B*S_max*N*D elements,
    two parts for fp32), int8 caches the quantised query rows and their
    scales."""
    from decode_sparse_attention_gb300 import questsparse as qs
    base = 16 * 4096 * 4 + 8 * 4096 * 4
    packed = 4096 * 16 * 128 * 2 + 4096 * 8 * 128 * 2
    f = qs.prefill_importance_workspace_size(1, 16, 8, 128, 4096, qs.F32)
    assert f >= base + 2 * packed
    h = qs.prefill_importance_workspace_size(1, 16, 8, 128, 4096, qs.BF16)
    assert base + packed <= h < f
    i8 = qs.prefill_importance_workspace_size(1, 16, 8, 128, 4096, qs.I8)
    assert i8 >= base + 4096 * 16 * 128 + 4096 * 16 * 4
    with pytest.raises(qs.QuestSparseError):
        qs.prefill_importance_workspace_size(1, 24, 8, 128, 4096, qs.F32)   # H/N = 3
    with pytest.raises(qs.QuestSparseError):
        qs.prefill_importance_workspace_size(1, 16, 8, 96, 4096, qs.F32)   # D


def test_binding_rejects_host_tensors(built_lib):
    from decode_sparse_attention_gb300 import questsparse as qs
    q = torch.zeros(1, 4, 64)
    kc = torch.zeros(2, 16, 2, 64)
    with pytest.raises(qs.QuestSparseError, match="CUDA"):
        qs.sparse_decode_attn(q, kc, kc, torch.zeros(1, 2, dtype=torch.int32),
                              torch.zeros(1, dtype=torch.int32),
                              torch.zeros(1, 2, 4, dtype=torch.int32))


def test_prefill_importance_binding_rejects_host_tensors(built_lib):
    from decode_sparse_attention_gb300 import questsparse as qs
    q = torch.zeros(1, 64, 4, 64)
    kc = torch.zeros(4, 16, 2, 64)
    with pytest.raises(qs.QuestSparseError, match="CUDA"):
        qs.prefill_importance(q, kc, torch.zeros(1, 4, dtype=torch.int32),
                              torch.zeros(1, dtype=torch.int32))


def test_step_params_layout_matches_header():
    """The ctypes mirror of qs_step_params has the C struct's field order."""
    from decode_sparse_attention_gb300 import questsparse as qs
    txt = open(os.path.join(ROOT, "include", "questsparse.h")).read()
    body = txt[txt.index("typedef struct {\n    int32_t mode;"):txt.index("} qs_step_params;")]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    c_fields = []
    for decl in body.replace("typedef struct {", "").split(";"):
        decl = decl.strip()
        if not decl:
            continue
        # "const int32_t* block_tables" / "int32_t B, H, N" ...
        parts = decl.split()
        names = " ".join(parts[1:]) if parts[0] != "const" else " ".join(parts[2:])
        for nm in names.split(","):
            c_fields.append(nm.strip().lstrip("*").strip())
    py_fields = [f[0] for f in qs.StepParams._fields_]
    assert py_fields == c_fields


def test_step_kernels_query_without_gpu(built_lib):
    """qs_step_kernels decides without touching the device: probe mode and
    fused_select = 0 always run two kernels; a NULL argument is rejected."""
    from decode_sparse_attention_gb300 import questsparse as qs
    p = qs.StepParams()
    p.mode, p.B, p.H, p.N, p.D, p.BS, p.k = 1, 1, 16, 8, 128, 32, 32
    assert qs.step_kernels(p) == 2
    ws = (ctypes.c_uint8 * 1024)()
    p.mode, p.MMBPR, p.fused_select = 0, 1, 0
    p.workspace, p.workspace_bytes = ctypes.addressof(ws), 1 << 40
    assert qs.step_kernels(p) == 2
    n = ctypes.c_int32(0)
    assert built_lib.qs_step_kernels(None, ctypes.byref(n)) == 1       # QS_EINVAL


def test_step_kernels_counts_the_scan_path(built_lib):
    """A Quest step whose units have more metadata rows than the one-CTA
    selector scores in one load step runs scan + per-unit top-k + attention:
    three kernels (the ragged and long-context workloads), else two."""
    from decode_sparse_attention_gb300 import questsparse as qs
    ws = (ctypes.c_uint8 * 1024)()
    cases = [
        # kv dtype, D, MMBPR, BS -> kernels
        (qs.BF16, 128, 1, 128, 2),     # bf16_paged: 128 rows, one chunk
        (qs.F16, 128, 1, 128, 2),
        (qs.BF16, 128, 4, 128, 3),     # long_context: 512 rows
        (qs.BF16, 128, 8, 128, 3),     # ragged: up to 1024 rows
        (qs.F32, 128, 1, 64, 2),       # fp32 rows are twice as wide: 64 rows per step
        (qs.F32, 128, 1, 128, 3),
        (qs.BF16, 64, 2, 128, 2),      # D = 64: 256 rows
        (qs.BF16, 64, 3, 128, 3),
        (qs.F32, 64, 1, 128, 2),
    ]
    for dt, D, MMBPR, BS, want in cases:
        p = qs.StepParams()
        p.mode, p.kv_dtype, p.q_dtype = 0, dt, dt
        p.B, p.H, p.N, p.D, p.BS, p.k, p.MMBPR, p.fused_select = 4, 32, 8, D, BS, 8, MMBPR, 0
        p.workspace, p.workspace_bytes = ctypes.addressof(ws), 1 << 40
        assert qs.step_kernels(p) == want, (dt, D, MMBPR, BS)


def header_enum_values():
    """name -> value of every enumerator the header declares."""
    txt = open(os.path.join(ROOT, "include", "questsparse.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    vals = {}
    for body in re.findall(r"enum\s*\w*\s*\{(.*?)\}", txt, flags=re.S):
        for name, v in re.findall(r"\b(QS_[A-Z0-9_]+)\s*=\s*(-?\d+)", body):
            vals[name] = int(v)
    return vals


def test_binding_constants_match_the_header():
    from decode_sparse_attention_gb300 import questsparse as qs
    v = header_enum_values()
    assert (qs.F32, qs.BF16, qs.F16, qs.I8) == (v["QS_F32"], v["QS_BF16"], v["QS_F16"], v["QS_I8"])
    assert (qs.OP_BLOCK_SELECT, qs.OP_PROBE_SELECT, qs.OP_SPARSE_ATTN, qs.OP_STEP_QUEST,
            qs.OP_STEP_PROBE) == (v["QS_OP_BLOCK_SELECT"], v["QS_OP_PROBE_SELECT"],
                                  v["QS_OP_SPARSE_ATTN"], v["QS_OP_DECODE_STEP_QUEST"],
                                  v["QS_OP_DECODE_STEP_PROBE"])
    assert v["QS_OK"] == 0 and v["QS_DEV_OK"] == 0 and v["QS_DEV_ETIMEOUT"] == 6


def test_device_status_strings_cover_every_code(built_lib):
    """Every device-side code the header declares has its own message."""
    built_lib.qs_status_string.restype = ctypes.c_char_p
    built_lib.qs_status_string.argtypes = [ctypes.c_int32]
    v = header_enum_values()
    dev = sorted(val for name, val in v.items() if name.startswith("QS_DEV_E"))
    msgs = [built_lib.qs_status_string(100 + c) for c in dev]
    assert all(m and m != built_lib.qs_status_string(999) for m in msgs)
    assert len(set(msgs)) == len(msgs)


def test_binding_checks_sizes_before_any_call(built_lib, monkeypatch):
    """Outputs and per-request inputs of the wrong size are refused by the
    binding before the library is called (the C ABI trusts its sizes).  The
    device placement check is switched off so host tensors reach them."""
    from decode_sparse_attention_gb300 import questsparse as qs

    def req_no_device(t, name, dtype=None, dim=None):
        if dtype is not None and t.dtype != dtype:
            raise qs.QuestSparseError("%s must be %s" % (name, dtype))
        if dim is not None and t.dim() != dim:
            raise qs.QuestSparseError("%s must have %d dims" % (name, dim))
        return t

    def no_call(*a, **k):
        raise AssertionError("the library was called")

    monkeypatch.setattr(qs, "_req", req_no_device)
    monkeypatch.setattr(qs, "lib", no_call)
    monkeypatch.setattr(qs, "workspace_size", no_call)
    monkeypatch.setattr(qs, "prefill_importance_workspace_size", no_call)
    i32 = torch.int32
    B, H, N, D, BS, k = 3, 8, 2, 64, 16, 4
    q = torch.zeros(B, H, D, dtype=torch.bfloat16)
    kc = torch.zeros(10, BS, N, D, dtype=torch.bfloat16)
    bt = torch.zeros(B, 5, dtype=i32)
    sl = torch.zeros(B, dtype=i32)
    sel = torch.zeros(B, N, k, dtype=i32)
    E = qs.QuestSparseError
    with pytest.raises(E, match="row per request"):
        qs.sparse_decode_attn(q, kc, kc, bt[:2], sl, sel)
    with pytest.raises(E, match="row per request"):
        qs.sparse_decode_attn(q, kc, kc, bt, sl[:2], sel)
    with pytest.raises(E, match="selected"):
        qs.sparse_decode_attn(q, kc, kc, bt, sl, torch.zeros(B, 3, k, dtype=i32))
    with pytest.raises(E, match="out must be"):
        qs.sparse_decode_attn(q, kc, kc, bt, sl, sel, out=torch.zeros(B, H, D // 2))
    with pytest.raises(E, match="lse"):
        qs.sparse_decode_attn(q, kc, kc, bt, sl, sel, lse=torch.zeros(B, H - 1))
    with pytest.raises(E, match="v_scale must be"):
        qs.sparse_decode_attn(q, kc, kc, bt, sl, sel, v_scale=torch.zeros(10, BS, N + 1))
    with pytest.raises(E, match="selected must be"):
        qs.probe_select(q, kc, bt, sl, k, selected=torch.zeros(B, N, k, dtype=i32))
    with pytest.raises(E, match="row per request"):
        qs.probe_select(q, kc, bt, sl, k, importance=torch.zeros(B - 1, 80))
    with pytest.raises(E, match="k_scale must be"):
        qs.probe_select(q, kc, bt, sl, k, k_scale=torch.zeros(10, BS, 1))
    qp = torch.zeros(B, 80, H, D, dtype=torch.bfloat16)
    with pytest.raises(E, match="lse must be"):
        qs.prefill_importance(qp, kc, bt, sl, lse=torch.zeros(B, H, 79))
    with pytest.raises(E, match="importance must be"):
        qs.prefill_importance(qp, kc, bt, sl, importance=torch.zeros(B, 81))
    with pytest.raises(E, match="row per request"):
        qs.prefill_importance(qp, kc, bt, sl[:1])
    mx = torch.zeros(6, BS, N, D, dtype=torch.bfloat16)
    with pytest.raises(E, match="row per request"):
        qs.quest_prefill_metadata(kc, sl, bt, torch.zeros(B - 1, 2, dtype=i32), mx, mx)
    with pytest.raises(E, match="row per request"):
        qs.quest_update_metadata(kc, sl, sl, bt[:1], torch.zeros(B, 2, dtype=i32), mx, mx)
    with pytest.raises(E, match="row per request"):
        qs.quest_block_select_paged_in_out_w(q, mx, mx, torch.zeros(B, 2, dtype=i32), sl[:2], 0,
                                             sel)


def test_step_kernel_rule_follows_the_selector_constants():
    """qs_step_kernels restates the unit selector's one-step row count; its
    constants must stay those of the selector's launch rule."""
    csrc = os.path.join(ROOT, "decode_sparse_attention_gb300", "csrc")
    sel = open(os.path.join(csrc, "qs_select.cu")).read()
    api = open(os.path.join(csrc, "qs_api.cu")).read()
    threads = int(re.search(r"constexpr int kThreads = (\d+);", sel).group(1))
    unroll = int(re.search(r"constexpr int kUnroll = (\d+);", sel).group(1))
    assert "(kThreads / 32) * (32 / (D * DtInfo<MT>::bytes / 16)) * kUnroll" in sel
    assert "if (maxnb <= kRows)" in sel
    warps = int(re.search(r"constexpr int kUnitSelectWarps = (\d+);", api).group(1))
    in_flight = int(re.search(r"constexpr int kUnitSelectRowsInFlight = (\d+);", api).group(1))
    assert (warps, in_flight) == (threads // 32, unroll)
