// Host side of the C ABI: device queries, status strings, workspace sizing
// and the decode step.
#include <map>
#include <mutex>
#include <utility>

#include "qs_internal.cuh"

namespace qs {

namespace {
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];
}  // namespace

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
    if (dev < kMaxDevices && g_sms[dev] > 0) return g_sms[dev];
    int n = 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    if (dev < kMaxDevices) g_sms[dev] = n;
    return n;
}

cudaError_t last_launch_error() { return cudaGetLastError(); }

bool ensure_smem(const void* func, size_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, size_t> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lk(mu);
    auto key = std::make_pair(func, dev);
    auto it = done.find(key);
    if (it != done.end() && it->second >= bytes) return true;
    const size_t want = bytes < 48 * 1024 ? 48 * 1024 : align_up(bytes, 1024);
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(want)) != cudaSuccess)
        return false;
    done[key] = want;
    return true;
}

}  // namespace qs

extern "C" int32_t qs_version(void) { return 1 * 10000 + 0 * 100 + 0; }

extern "C" const char* qs_status_string(int32_t code) {
    if (code >= 100) {
        switch (code - 100) {
            case QS_DEV_OK: return "device: ok";
            case QS_DEV_EBLOCK_TABLE: return "device: block_tables entry out of range";
            case QS_DEV_EMETA_TABLE: return "device: meta_block_tables entry out of range";
            case QS_DEV_ESEQ_LEN: return "device: seq_len out of range";
            case QS_DEV_ESELECTED: return "device: selected block index beyond the sequence";
            case QS_DEV_EFORCED: return "device: forced window larger than k";
            case QS_DEV_ETIMEOUT: return "device: bounded wait timed out";
            default: return "device: unknown code";
        }
    }
    switch (code) {
        case QS_OK: return "ok";
        case QS_EINVAL: return "invalid argument";
        case QS_EDTYPE: return "unsupported dtype";
        case QS_EUNSUPPORTED: return "unsupported size (no kernel instantiation)";
        case QS_ECUDA: return "CUDA error";
        case QS_EWORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

extern "C" qs_status qs_read_status(const int32_t* dev_status, int32_t* host_code, int32_t reset,
                                    qs_stream_t stream) {
    if (!dev_status || !host_code) return QS_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(host_code, dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return QS_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return QS_ECUDA;
    if (reset && cudaMemsetAsync(const_cast<int32_t*>(dev_status), 0, sizeof(int32_t), s) != cudaSuccess)
        return QS_ECUDA;
    return QS_OK;
}

extern "C" qs_status qs_workspace_size(qs_op op, int32_t B, int32_t H, int32_t N, int32_t D,
                                       int32_t BS, int32_t k, int32_t max_blocks_per_req,
                                       int32_t sel_heads, size_t* bytes) {
    if (!bytes || B < 0 || H <= 0 || N <= 0 || H % N || D <= 0 || BS <= 0 || k <= 0 ||
        max_blocks_per_req < 0)
        return QS_EINVAL;
    using namespace qs;
    switch (op) {
        case QS_OP_BLOCK_SELECT: *bytes = select_workspace_bytes(B, N, max_blocks_per_req); break;
        case QS_OP_PROBE_SELECT: *bytes = probe_workspace_bytes(B, H, N, max_blocks_per_req); break;
        case QS_OP_SPARSE_ATTN:
            if (sel_heads != N && sel_heads != H) return QS_EINVAL;
            *bytes = attn_workspace_bytes(B, H, N, D, sel_heads);
            break;
        case QS_OP_DECODE_STEP_QUEST:
            *bytes = align_up(select_workspace_bytes(B, N, max_blocks_per_req), 256) +
                     attn_workspace_bytes(B, H, N, D, N);
            break;
        case QS_OP_DECODE_STEP_PROBE:
            *bytes = align_up(probe_workspace_bytes(B, H, N, max_blocks_per_req), 256) +
                     attn_workspace_bytes(B, H, N, D, H);
            break;
        default: return QS_EINVAL;
    }
    return QS_OK;
}

extern "C" qs_status qs_sparse_decode_step(const qs_step_params* p, qs_stream_t stream) {
    using namespace qs;
    if (!p) return QS_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(p->workspace);
    size_t sel_ws;
    int sel_heads;
    qs_status st;
    if (p->mode == 0) {
        if (p->MMBPR < 0 || p->BS <= 0) return QS_EINVAL;
        sel_ws = align_up(select_workspace_bytes(p->B, p->N, p->MMBPR * p->BS), 256);
        sel_heads = p->N;
        if (!ws || p->workspace_bytes < sel_ws) return QS_EWORKSPACE;
        bool fused = false;
        st = quest_step_fused(p, ws + sel_ws, p->workspace_bytes - sel_ws, s, &fused, true);
        if (fused) return st;
        st = block_select_impl(p->q, p->q_dtype, p->maxblocks, p->minblocks, p->kv_dtype,
                               p->meta_block_tables, p->MMBPR, p->num_meta_blocks, p->seq_lens,
                               p->B, p->H, p->N, p->D, p->BS, p->k,
                               p->tokens_since_metadata_update, p->selected, nullptr, ws, sel_ws,
                               p->dev_status, s);
    } else if (p->mode == 1) {
        sel_ws = align_up(probe_workspace_bytes(p->B, p->H, p->N, p->MKBPR), 256);
        sel_heads = p->H;
        if (!ws || p->workspace_bytes < sel_ws) return QS_EWORKSPACE;
        st = probe_select_impl(p->q, p->q_dtype, p->k_cache, p->k_scale, p->kv_dtype,
                               p->num_kv_blocks, p->block_tables, p->MKBPR, p->seq_lens,
                               p->importance, p->importance_stride, p->B, p->H, p->N, p->D, p->BS,
                               p->k, p->n_probe, p->selected, ws, sel_ws, p->dev_status, s);
    } else {
        return QS_EINVAL;
    }
    if (st != QS_OK) return st;
    return sparse_attn_impl(p->q, p->q_dtype, p->k_cache, p->v_cache, p->k_scale, p->v_scale,
                            p->kv_dtype, p->num_kv_blocks, p->block_tables, p->MKBPR, p->seq_lens,
                            p->selected, sel_heads, p->k, p->softmax_scale, p->B, p->H, p->N, p->D,
                            p->BS, p->out, p->lse_opt, ws + sel_ws, p->workspace_bytes - sel_ws,
                            p->dev_status, s, /*pdl=*/true);
}

namespace {

// Metadata rows of one unit that the one-CTA-per-unit Quest selector scores
// in a single load step: 8 warps, a row per lane group of D*e/16 lanes, 8
// rows in flight per group.  Units with more rows take the scan and then a
// per-unit top-k kernel (the selector's launch rule).  0: no such kernel.
constexpr int kUnitSelectWarps = 8;        // 256 threads per unit CTA
constexpr int kUnitSelectRowsInFlight = 8;  // rows in flight per lane group

int quest_unit_rows(qs_dtype meta_dtype, int32_t D) {
    const int e = meta_dtype == QS_F32 ? 4 : 2;
    const int lanes_per_row = D * e / 16;
    if (D <= 0 || lanes_per_row <= 0 || lanes_per_row > 32 || 32 % lanes_per_row != 0) return 0;
    return kUnitSelectWarps * (32 / lanes_per_row) * kUnitSelectRowsInFlight;
}

}  // namespace

extern "C" qs_status qs_step_kernels(const qs_step_params* p, int32_t* kernels) {
    using namespace qs;
    if (!p || !kernels) return QS_EINVAL;
    *kernels = 2;
    if (p->mode != 0) return QS_OK;
    if (p->MMBPR < 0 || p->BS <= 0) return QS_EINVAL;
    const size_t sel_ws = align_up(select_workspace_bytes(p->B, p->N, p->MMBPR * p->BS), 256);
    if (!p->workspace || p->workspace_bytes < sel_ws) return QS_EWORKSPACE;
    bool fused = false;
    quest_step_fused(p, static_cast<uint8_t*>(p->workspace) + sel_ws, p->workspace_bytes - sel_ws,
                     nullptr, &fused, false);
    if (fused) {
        *kernels = 1;
    } else if (static_cast<long long>(p->MMBPR) * p->BS > quest_unit_rows(p->kv_dtype, p->D)) {
        *kernels = 3;   // scan + per-unit top-k + attention
    }
    return QS_OK;
}
