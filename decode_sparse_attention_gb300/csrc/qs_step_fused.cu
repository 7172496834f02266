// Fused Quest decode step: block selection and sparse attention in one
// persistent kernel (the selection of the CANN select_attention_operators
// page, quest_block_select_paged steps 1-2.3 with sink + window forcing,
// followed by the exact attention over the selected blocks of the Kestrel-LLM
// article 10-2, section 2).
//
// Each CTA selects the units its stream-K tile range touches and streams
// their K/V straight away; nothing is handed between CTAs, so there is no
// wait, and the step costs one launch instead of two.  The price is that a
// unit split between CTAs has its metadata scanned by each of them (the
// second scan mostly hits L2) and that every CTA's K/V stream starts only
// after its own selection.
#include "qs_attention_kernel.cuh"

#ifndef QS_FUSED_SELECT_RATIO
// largest (metadata rows a CTA may scan) / (K/V rows it streams) for which
// the automatic choice takes the fused kernel.  Measured on GB300 the fused
// kernel did not beat the two-kernel step at any of the benchmark shapes
// (bf16_paged: 53.5 vs 51.2 us; long_context: 97.2 vs 81.9 us): its CTAs
// scan their units' metadata (twice where a unit is split), select, and only
// then start the K/V stream, while the two-kernel step scans each unit once.
// So by default the automatic choice never fuses; callers can still ask for
// the fused kernel with fused_select = 1.
#define QS_FUSED_SELECT_RATIO 0.0
#endif

namespace qs {

namespace {

// Selection scratch inside the ring region, after the prologue staging
// (which must hold the block-table rows); false if it does not fit.
bool plan_fused_select(int D, int k, int MMBPR, int BS, long long tpu, AttnArgs* a) {
    const long long upc = plan_units_per_cta(a->tpc, tpu);
    const long long rows = upc * MMBPR * BS;
    if (!a->bt_staged) return false;
    size_t off = a->sel_end;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, 16);
        return static_cast<uint32_t>(at);
    };
    a->sel_off_mbt = take(static_cast<size_t>(upc) * MMBPR * 4);
    a->sel_off_qg = take(static_cast<size_t>(upc) * D * 4);
    a->sel_off_keys = take(static_cast<size_t>(rows) * 4);
    a->sel_off_flags = take(static_cast<size_t>(rows));
    a->sel_off_sel = take(static_cast<size_t>(upc) * k * 4);
    a->sel_off_wtk = take(static_cast<size_t>(upc) * sizeof(WarpTopkScratch));
    a->sel_end = static_cast<uint32_t>(off);
    const size_t ring = static_cast<size_t>(a->NW) * a->S * a->stage_bytes;
    return upc <= kQSlots && off <= ring;
}

}  // namespace

qs_status quest_step_fused(const qs_step_params* p, void* attn_ws, size_t attn_ws_bytes,
                           cudaStream_t stream, bool* taken, bool launch) {
    *taken = false;
    if (p->fused_select == 0) return QS_OK;
    const int B = p->B, H = p->H, N = p->N, D = p->D, BS = p->BS, k = p->k;
    if (p->mode != 0 || B <= 0 || H <= 0 || N <= 0 || H % N || k <= 0 || BS <= 0 ||
        p->MMBPR < 0 || p->MKBPR < 0 || p->num_kv_blocks <= 0 || p->num_meta_blocks < 0)
        return QS_OK;
    const int G = H / N;
    if (G != 1 && G != 2 && G != 4) return QS_OK;
    if (D != 64 && D != 128) return QS_OK;
    if (BS % 16 || BS > 4096) return QS_OK;
    if (p->q_dtype != QS_F32 && p->q_dtype != QS_BF16 && p->q_dtype != QS_F16) return QS_OK;
    int es;
    switch (p->kv_dtype) {
        case QS_F32: es = 4; break;
        case QS_BF16: case QS_F16: es = 2; break;
        default: return QS_OK;
    }
    if (D * es < 128) return QS_OK;
    if (!p->q || !p->k_cache || !p->v_cache || !p->block_tables || !p->seq_lens ||
        !p->maxblocks || !p->minblocks || !p->meta_block_tables || !p->selected || !p->out ||
        !p->dev_status)
        return QS_OK;
    if ((reinterpret_cast<uintptr_t>(p->q) | reinterpret_cast<uintptr_t>(p->k_cache) |
         reinterpret_cast<uintptr_t>(p->v_cache) | reinterpret_cast<uintptr_t>(p->maxblocks) |
         reinterpret_cast<uintptr_t>(p->minblocks)) % 16)
        return QS_OK;
    const int t = p->tokens_since_metadata_update;
    if (t >= 0 && static_cast<long long>(k) < 2 + (static_cast<long long>(t) + BS - 1) / BS)
        return QS_OK;
    const long long maxnb = static_cast<long long>(p->MMBPR) * BS;
    if (maxnb > (1 << 24)) return QS_OK;
    if (static_cast<long long>(p->num_kv_blocks) * BS > (1LL << 31) - 1) return QS_OK;
    const long long units = static_cast<long long>(B) * N;
    AttnArgs a = {};
    AttnPlan pl = {};
    const int q_es = p->q_dtype == QS_F32 ? 4 : 2;
    if (!plan_attention(BS, D, G, es, q_es, false, units, k, p->MKBPR, &a, &pl)) return QS_OK;
    if (pl.grid > units + 1024) return QS_OK;
    const long long tpu = static_cast<long long>(k) * a.split;
    if (!plan_fused_select(D, k, p->MMBPR, BS, tpu, &a)) return QS_OK;
    const long long n_units_max = plan_units_per_cta(a.tpc, tpu);
    if (p->fused_select < 0) {
        // the fused kernel pays for the per-CTA selection before its first
        // K/V tile: take it only where that scan is small next to the tile
        // stream and the two-kernel step would be bound by its launch
        // latencies rather than by the stream
        if (static_cast<double>(n_units_max * maxnb) >
            QS_FUSED_SELECT_RATIO * static_cast<double>(a.tpc) * a.TR)
            return QS_OK;
    }
    if (!attn_ws || attn_ws_bytes < attn_workspace_bytes(B, H, N, D, N)) return QS_OK;

    *taken = true;
    if (!launch) return QS_OK;
    uint8_t* ws = static_cast<uint8_t*>(attn_ws);
    a.q = static_cast<const uint8_t*>(p->q);
    a.q_dt = p->q_dtype;
    a.q_es = q_es;
    a.kc = static_cast<const uint8_t*>(p->k_cache);
    a.vc = static_cast<const uint8_t*>(p->v_cache);
    a.bt = p->block_tables;
    a.MKBPR = p->MKBPR;
    a.seq_lens = p->seq_lens;
    a.sel = nullptr;
    a.sel_heads = N;
    a.k = k;
    a.num_kv_blocks = p->num_kv_blocks;
    a.B = B; a.H = H; a.N = N; a.BS = BS;
    a.scale_log2 = p->softmax_scale * 1.4426950408889634f;
    a.out = p->out;
    a.lse = p->lse_opt;
    a.counters = reinterpret_cast<uint32_t*>(ws);
    a.partial = reinterpret_cast<float*>(ws + align_up(static_cast<size_t>(units) * 4, 256));
    a.dev_status = p->dev_status;
    a.maxb = static_cast<const uint8_t*>(p->maxblocks);
    a.minb = static_cast<const uint8_t*>(p->minblocks);
    a.mbt = p->meta_block_tables;
    a.MMBPR = p->MMBPR;
    a.num_meta = p->num_meta_blocks;
    a.t = t;
    a.sel_out = p->selected;
    switch (p->kv_dtype) {
        case QS_F32: return D == 128 ? dispatch_g<Dt::F32, 128, true>(G, a, pl, false, stream)
                                     : dispatch_g<Dt::F32, 64, true>(G, a, pl, false, stream);
        case QS_BF16: return D == 128 ? dispatch_g<Dt::BF16, 128, true>(G, a, pl, false, stream)
                                      : dispatch_g<Dt::BF16, 64, true>(G, a, pl, false, stream);
        default: return D == 128 ? dispatch_g<Dt::F16, 128, true>(G, a, pl, false, stream)
                                 : dispatch_g<Dt::F16, 64, true>(G, a, pl, false, stream);
    }
}

}  // namespace qs
