// Exact decode attention over the selected KV blocks only (Kestrel-LLM
// article 10-2, section 2: token scores over the selected blocks, softmax
// renormalised over that set, weighted sum of V), with the in-sequence ->
// physical mapping through block_tables (CANN select_attention_operators page,
// top-k section: the returned indices are in-sequence).
//
// GB300 design (HBM-bound, ~2 flop/byte, so CUDA cores, no tensor cores):
//  * Work = (unit, selected block, sub-tile) tiles; a unit is (request, KV
//    head) when the selection is per KV head -- all H/N query heads of the
//    group share each K/V tile, read once -- or (request, query head).
//  * Persistent grid of about one CTA per SM; CTA c owns a contiguous range of
//    tiles (stream-K split), so every SM streams the same number of tiles.
//  * A prologue stages the CTA's tile list (selected block -> physical rows,
//    valid rows, unit) and the queries of its units in shared memory.
//  * Every warp owns a fixed slice of rows of each tile and streams exactly
//    those rows with 16-byte cp.async copies into its own multi-stage ring,
//    several tiles ahead, so the warps never wait on one another between
//    tiles.  (A head slice of a paged block is rows of D elements 2 KB apart;
//    gathered with 2-D TMA boxes or per-row bulk copies, the copy engine's
//    request rate capped a whole SM near 32 GB/s on GB300, so the gather
//    uses the load/store path, which all 256 threads feed in parallel.)
//  * Each warp keeps its own online-softmax state (running max, sum,
//    accumulator) over its rows; warps are merged at the end of a unit.  Q.K
//    uses 8 lanes per token and packed fp32x2 FMAs with a transposing shuffle
//    reduction; P.V gives each lane D/32 output channels.
//  * A unit split across CTAs is merged on the device: each CTA writes a
//    (max, sum, acc) partial; the last to arrive (atomic counter, no spin)
//    combines them and rearms the counter.
//  * Inside the fused decode step it is launched as a programmatic dependent
//    of the selector: ring zeroing, query staging and block-table prefetches
//    (none of which the selector writes) overlap the selector's tail.
#include "qs_attention_kernel.cuh"

namespace qs {

size_t attn_workspace_bytes(int B, int H, int N, int D, int sel_heads) {
    // counters per unit + one (max, sum, acc) partial slot per (CTA, unit)
    // pair of the stream-K split: a slot index is CTA + unit, at most
    // grid + units - 2, and the planner keeps the grid within units + 1024.
    const long long units = static_cast<long long>(B) * sel_heads;
    const int G = sel_heads == N ? H / N : 1;
    const long long slots = 2 * units + 1024;
    return align_up(static_cast<size_t>(units) * 4, 256) +
           align_up(static_cast<size_t>(slots) * G * (D + 2) * 4, 256);
}

qs_status sparse_attn_impl(const void* q, qs_dtype q_dtype, const void* k_cache, const void* v_cache,
                           const float* k_scale, const float* v_scale, qs_dtype kv_dtype,
                           int32_t num_kv_blocks, const int32_t* block_tables, int32_t MKBPR,
                           const int32_t* seq_lens, const int32_t* selected, int32_t sel_heads,
                           int32_t k, float softmax_scale, int32_t B, int32_t H, int32_t N,
                           int32_t D, int32_t BS, float* out, float* lse_opt, void* workspace,
                           size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream,
                           bool pdl, bool clear_counters) {
    if (B < 0 || H <= 0 || N <= 0 || H % N != 0 || BS <= 0 || k <= 0 || MKBPR < 0 ||
        num_kv_blocks <= 0)
        return QS_EINVAL;
    if (sel_heads != N && sel_heads != H) return QS_EINVAL;
    if (B == 0) return QS_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !selected || !out || !dev_status)
        return QS_EINVAL;
    if (q_dtype != QS_F32 && q_dtype != QS_BF16 && q_dtype != QS_F16) return QS_EDTYPE;
    int es;
    switch (kv_dtype) {
        case QS_F32: es = 4; break;
        case QS_BF16: case QS_F16: es = 2; break;
        case QS_I8: es = 1; break;
        default: return QS_EDTYPE;
    }
    const bool int8 = kv_dtype == QS_I8;
    if (int8 && (!k_scale || !v_scale)) return QS_EINVAL;
    if (D != 64 && D != 128) return QS_EUNSUPPORTED;
    if (D * es < 128) return QS_EUNSUPPORTED;              // a K row spans 8 lanes x 16 B
    if (BS % 16 || BS > 4096) return QS_EUNSUPPORTED;
    if (static_cast<long long>(num_kv_blocks) * BS > (1LL << 31) - 1) return QS_EUNSUPPORTED;
    const int G = sel_heads == N ? H / N : 1;
    if (G != 1 && G != 2 && G != 4) return QS_EUNSUPPORTED;
    const int q_es = q_dtype == QS_F32 ? 4 : 2;
    const uintptr_t al = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
                         reinterpret_cast<uintptr_t>(v_cache);
    if (al % 16) return QS_EINVAL;
    if (int8 && ((reinterpret_cast<uintptr_t>(k_scale) | reinterpret_cast<uintptr_t>(v_scale)) % 4))
        return QS_EINVAL;
    const long long units = static_cast<long long>(B) * sel_heads;
    AttnArgs a = {};
    AttnPlan pl = {};
    if (!plan_attention(BS, D, G, es, q_es, int8, units, k, MKBPR, &a, &pl)) return QS_EUNSUPPORTED;
    if (pl.grid > units + 1024) return QS_EUNSUPPORTED;   // partial slots: grid + units
    const size_t need = attn_workspace_bytes(B, H, N, D, sel_heads);
    if (!workspace || workspace_bytes < need) return QS_EWORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.q = static_cast<const uint8_t*>(q);
    a.q_dt = q_dtype;
    a.q_es = q_es;
    a.kc = static_cast<const uint8_t*>(k_cache);
    a.vc = static_cast<const uint8_t*>(v_cache);
    a.ks = k_scale;
    a.vs = v_scale;
    a.bt = block_tables;
    a.MKBPR = MKBPR;
    a.seq_lens = seq_lens;
    a.sel = selected;
    a.sel_heads = sel_heads;
    a.k = k;
    a.num_kv_blocks = num_kv_blocks;
    a.B = B; a.H = H; a.N = N; a.BS = BS;
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    a.out = out;
    a.lse = lse_opt;
    a.counters = reinterpret_cast<uint32_t*>(ws);
    a.partial = reinterpret_cast<float*>(ws + align_up(static_cast<size_t>(units) * 4, 256));
    a.dev_status = dev_status;
    // every check has passed: only now may the call touch the workspace
    if (clear_counters &&
        cudaMemsetAsync(a.counters, 0, static_cast<size_t>(units) * sizeof(uint32_t), stream) !=
            cudaSuccess)
        return QS_ECUDA;
    switch (kv_dtype) {
        case QS_F32: return D == 128 ? dispatch_g<Dt::F32, 128>(G, a, pl, pdl, stream)
                                     : dispatch_g<Dt::F32, 64>(G, a, pl, pdl, stream);
        case QS_BF16: return D == 128 ? dispatch_g<Dt::BF16, 128>(G, a, pl, pdl, stream)
                                      : dispatch_g<Dt::BF16, 64>(G, a, pl, pdl, stream);
        case QS_F16: return D == 128 ? dispatch_g<Dt::F16, 128>(G, a, pl, pdl, stream)
                                     : dispatch_g<Dt::F16, 64>(G, a, pl, pdl, stream);
        default: return dispatch_g<Dt::I8, 128>(G, a, pl, pdl, stream);
    }
}

}  // namespace qs

extern "C" qs_status qs_sparse_decode_attn(const void* q, qs_dtype q_dtype, const void* k_cache,
                                           const void* v_cache, const float* k_scale,
                                           const float* v_scale, qs_dtype kv_dtype,
                                           int32_t num_kv_blocks, const int32_t* block_tables,
                                           int32_t MKBPR, const int32_t* seq_lens,
                                           const int32_t* selected, int32_t sel_heads, int32_t k,
                                           float softmax_scale, int32_t B, int32_t H, int32_t N,
                                           int32_t D, int32_t BS, float* out, float* lse_opt,
                                           void* workspace, size_t workspace_bytes,
                                           int32_t* dev_status, qs_stream_t stream) {
    return qs::sparse_attn_impl(q, q_dtype, k_cache, v_cache, k_scale, v_scale, kv_dtype,
                                num_kv_blocks, block_tables, MKBPR, seq_lens, selected, sel_heads,
                                k, softmax_scale, B, H, N, D, BS, out, lse_opt, workspace,
                                workspace_bytes, dev_status, reinterpret_cast<cudaStream_t>(stream),
                                false, false);
}
