// Kernel of the exact decode attention over the selected KV blocks only (Kestrel-LLM
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
//  * A prologue stages, with cp.async copies issued before the wait for the
//    selector, the raw query rows of the CTA's units and the block-table rows
//    and lengths of their requests; after the wait it builds the tile list
//    (selected block -> byte offset of its rows, valid rows, unit) from the
//    selection and those staged rows in one round trip.
//  * Every warp owns a fixed slice of rows of each tile and streams exactly
//    those rows with 16-byte cp.async copies into its own multi-stage ring,
//    several tiles ahead, so the warps never wait on one another between
//    tiles.  (A head slice of a paged block is rows of D elements 2 KB apart;
//    gathered with 2-D TMA boxes or per-row bulk copies, the copy engine's
//    request rate capped a whole SM near 32 GB/s on GB300, so the gather
//    uses the load/store path, which all 256 threads feed in parallel.)
//  * Each warp keeps its own online-softmax state (running max, sum,
//    accumulator) over its rows; warps are merged at the end of a unit (one
//    warp per head reduces the warps' maxima and sums, every thread then
//    combines its output channels).  Q.K uses 8 lanes per token and packed
//    fp32x2 FMAs with a transposing shuffle reduction; P.V gives each lane
//    D/32 output channels and runs over all of a warp's rows (p = 0 past the
//    valid ones: when a warp loads fewer than its rows of a tile it zeroes
//    the V rows, and int8 scales, it leaves out, so those bytes are finite);
//    the accumulators are rescaled only when a head's max grew.
//  * A unit split across CTAs is merged on the device: each CTA writes a
//    (max, sum, acc) partial; the last to arrive (atomic counter, no spin)
//    combines them and rearms the counter.
//  * Inside the decode step it is launched as a programmatic dependent of the
//    selector: the staging copies (none of which read what the selector
//    writes) are issued before the grid-dependency wait.
#pragma once

#include <cmath>

#include "qs_internal.cuh"
#include "qs_quest_score.cuh"
#include "qs_topk.cuh"

namespace qs {
namespace {

constexpr int kMaxWarps = 16;
constexpr int kRPW = 8;                  // rows of a tile each warp owns
constexpr int kQSlots = 8;               // units a CTA's tile range may touch
constexpr int kMaxTilesPerCta = 512;
constexpr int kMaxStages = 6;
constexpr int kSmemBudget = 225 * 1024;
constexpr size_t kStageTablesMax = 64 * 1024;   // block-table rows staged in shared memory
constexpr int kMergeFast = 8;            // split partials merged in one round trip

struct AttnArgs {
    const uint8_t* q;
    int q_dt, q_es;
    const uint8_t* kc;
    const uint8_t* vc;
    const float* ks;
    const float* vs;
    const int32_t* bt;
    int MKBPR;
    const int32_t* seq_lens;
    const int32_t* sel;
    int sel_heads, k, num_kv_blocks, B, H, N, BS, TR, split, S, NW, rpw;
    float scale_log2;
    float* out;
    float* lse;
    float* partial;
    uint32_t* counters;
    int T;                   // tiles of the whole launch (< 2^31)
    int tpc;
    int32_t* dev_status;
    int bt_staged;           // block-table rows of the CTA's requests staged in shared memory
    // dynamic shared memory layout (bytes)
    uint32_t off_q, off_stage, off_p, off_ml, off_f;
    uint32_t stage_bytes;    // one warp's slot of one stage
    uint32_t rows_bytes;     // rpw rows of one head: rpw * D * elem bytes
    // fused Quest selection (decode step)
    const uint8_t* maxb;
    const uint8_t* minb;
    const int32_t* mbt;
    int MMBPR, num_meta, t;
    int32_t* sel_out;        // selected [B, N, k]
    // byte offsets inside the ring region, used before the first tile is
    // issued: raw query rows (per unit), block-table rows and lengths (per
    // request); for the fused selection also metadata-table rows, group-mean
    // queries, keys, flags, selections and per-warp top-k scratch
    uint32_t sel_off_qraw, sel_off_mbt, sel_off_bt, sel_off_len, sel_off_qg, sel_off_keys,
        sel_off_flags, sel_off_sel, sel_off_wtk, sel_end;
};

struct TileInfo {
    long long off;   // byte offset of the tile's first row, head nkv, in the K/V pools
    int rows;        // valid rows in the tile (0: nothing to do)
    int meta;        // unit (relative to the CTA's first unit) | kFirst | kLast
};
constexpr int kFirst = 1 << 8, kLast = 1 << 9;

template <Dt KT> struct KvTraits {
    static constexpr int es = DtInfo<KT>::bytes;
    static constexpr int epc = 16 / es;  // elements per 16-byte chunk
};

QS_DEVINL void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
QS_DEVINL void cp_async16_s(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
QS_DEVINL void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
QS_DEVINL void cp_async4_s(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
QS_DEVINL void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most n of this thread's copy groups are still pending.
QS_DEVINL void cp_async_wait(int n) {
    switch (n) {
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
        case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
    }
}

// ---- Q.K partial over one 16-byte chunk of a K row, G heads ---------------

template <Dt KT, int G, int EPC>
QS_DEVINL void qk_chunk(const unsigned long long (&qp)[G][EPC / 2], uint4 kv,
                        unsigned long long (&acc)[G]) {
    if constexpr (KT == Dt::F32) {
        const unsigned long long k01 = (static_cast<unsigned long long>(kv.y) << 32) | kv.x;
        const unsigned long long k23 = (static_cast<unsigned long long>(kv.w) << 32) | kv.z;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            acc[h] = fma2(qp[h][0], k01, acc[h]);
            acc[h] = fma2(qp[h][1], k23, acc[h]);
        }
    } else {
        const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = pair_to_float2<KT>(w[i]);
            const unsigned long long k2 = pack2(f.x, f.y);
#pragma unroll
            for (int h = 0; h < G; ++h) acc[h] = fma2(qp[h][i], k2, acc[h]);
        }
    }
}

// Transposing reduction of G per-lane values over the 8 lanes of a token.
// Afterwards lane g (bits 0..2 of the lane id) holds the full sum of head
// head_of_lane<G>(g).
template <int G, typename V>
QS_DEVINL V reduce8(const V (&v)[G], int g) {
    if constexpr (G == 4) {
        const bool up = g & 4;
        V s0 = up ? v[0] : v[2], s1 = up ? v[1] : v[3];
        V k0 = up ? v[2] : v[0], k1 = up ? v[3] : v[1];
        k0 += __shfl_xor_sync(0xffffffffu, s0, 4);
        k1 += __shfl_xor_sync(0xffffffffu, s1, 4);
        const bool up2 = g & 2;
        V s = up2 ? k0 : k1;
        V k = up2 ? k1 : k0;
        k += __shfl_xor_sync(0xffffffffu, s, 2);
        k += __shfl_xor_sync(0xffffffffu, k, 1);
        return k;
    } else if constexpr (G == 2) {
        const bool up = g & 4;
        V s = up ? v[0] : v[1];
        V k = up ? v[1] : v[0];
        k += __shfl_xor_sync(0xffffffffu, s, 4);
        k += __shfl_xor_sync(0xffffffffu, k, 2);
        k += __shfl_xor_sync(0xffffffffu, k, 1);
        return k;
    } else {
        V k = v[0];
        k += __shfl_xor_sync(0xffffffffu, k, 4);
        k += __shfl_xor_sync(0xffffffffu, k, 2);
        k += __shfl_xor_sync(0xffffffffu, k, 1);
        return k;
    }
}
template <int G> QS_DEVINL int head_of_lane(int g) {
    return G == 4 ? (g >> 1) : G == 2 ? (g >> 2) : 0;
}
template <int G> QS_DEVINL bool rep_lane(int g) {
    return G == 4 ? !(g & 1) : G == 2 ? !(g & 3) : g == 0;
}
// A lane of the first token group that holds head h after reduce8.
template <int G> QS_DEVINL int lane_of_head(int h) { return h * (8 / G); }

QS_DEVINL float sext8(uint32_t w, int i) {
    return static_cast<float>(static_cast<int32_t>(w << (24 - 8 * i)) >> 24);
}

// ---- prologue staging -------------------------------------------------------
//
// With one batch of cp.async copies, stages what the tile list and the query
// set-up of units u_first .. u_first + n_units - 1 read and the preceding
// kernel does not write: the units' raw query rows and, when they fit, the
// block-table rows and lengths of their requests.
template <int D, int G>
QS_DEVINL void stage_unit_inputs(const AttnArgs& a, int u_first, int n_units, int b_first,
                                 int n_req, uint8_t* scratch) {
    const int tid = threadIdx.x, nthreads = blockDim.x;
    const int qrow = G * D * a.q_es;              // bytes of one unit's query rows
    const int qchunks = qrow / 16;
    uint8_t* qraw = scratch + a.sel_off_qraw;
    for (int e = tid; e < n_units * qchunks; e += nthreads) {
        const int us = e / qchunks, c = e - us * qchunks;
        const int u = u_first + us;
        const int b = u / a.sel_heads, s = u - b * a.sel_heads;
        cp_async16(qraw + static_cast<size_t>(us) * qrow + c * 16,
                   a.q + (static_cast<size_t>(b) * a.H + static_cast<size_t>(s) * G) * D * a.q_es +
                       c * 16);
    }
    int32_t* len_s = reinterpret_cast<int32_t*>(scratch + a.sel_off_len);
    if (tid < n_req) cp_async4(len_s + tid, a.seq_lens + b_first + tid);
    if (a.bt_staged) {
        int32_t* bt_s = reinterpret_cast<int32_t*>(scratch + a.sel_off_bt);
        const int32_t* src = a.bt + static_cast<size_t>(b_first) * a.MKBPR;
        const int total = n_req * a.MKBPR;
        if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
            const int vec = total / 4;
            for (int e = tid; e < vec; e += nthreads) cp_async16(bt_s + 4 * e, src + 4 * e);
            for (int e = 4 * vec + tid; e < total; e += nthreads) cp_async4(bt_s + e, src + e);
        } else {
            for (int e = tid; e < total; e += nthreads) cp_async4(bt_s + e, src + e);
        }
    }
}

// The fused selection also stages each unit's metadata-table row.
QS_DEVINL void stage_meta_tables(const AttnArgs& a, int u_first, int n_units,
                                 uint8_t* scratch) {
    int32_t* mbt_s = reinterpret_cast<int32_t*>(scratch + a.sel_off_mbt);
    for (int e = threadIdx.x; e < n_units * a.MMBPR; e += blockDim.x) {
        const int us = e / a.MMBPR, i = e - us * a.MMBPR;
        const size_t b = static_cast<size_t>((u_first + us) / a.N);
        cp_async4(mbt_s + e, a.mbt + b * a.MMBPR + i);
    }
}

// ---- fused Quest selection (decode step) ----------------------------------
//
// Selects the blocks of the units into sel_s[unit - u_first][0..k) in shared
// memory with the standalone selector's arithmetic: group-mean query (heads
// summed in order, then / G), RowChunk scores of every metadata row, sink +
// window forcing, top-k (key descending, ties to the lower index), ascending
// emission padded with -1.  One warp selects each unit; the CTA holding a
// unit's first tile writes the selection out.  Called by all threads after
// the staged inputs landed and qf (fp32 query rows) was written.
template <Dt KT, int D, int G>
QS_DEVINL void quest_select_units(const AttnArgs& a, int u_first, int n_units, int t0, int tpu,
                                  const float* qf,
                                  uint8_t* scratch) {
    constexpr int MES = DtInfo<KT>::bytes;        // metadata element bytes
    constexpr int kLPR = D * MES / 16;            // lanes per metadata row
    constexpr int kRPWL = 32 / kLPR;              // rows per warp and load
    constexpr int kEl = RowChunk<KT>::kElems;     // channels per 16-byte slice
    constexpr int kU = 8;                         // rows in flight per lane
    static_assert(kLPR >= 1 && kLPR <= 32 && 32 % kLPR == 0, "metadata row must tile a warp");
    __shared__ int s_nb[kQSlots], s_roff[kQSlots + 1];

    const int tid = threadIdx.x, nthreads = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5, nw = nthreads >> 5;
    const int32_t* mbt_s = reinterpret_cast<const int32_t*>(scratch + a.sel_off_mbt);
    const int32_t* len_s = reinterpret_cast<const int32_t*>(scratch + a.sel_off_len);
    float* qg_s = reinterpret_cast<float*>(scratch + a.sel_off_qg);
    uint32_t* keys = reinterpret_cast<uint32_t*>(scratch + a.sel_off_keys);
    uint8_t* flags = scratch + a.sel_off_flags;
    int32_t* sel_s = reinterpret_cast<int32_t*>(scratch + a.sel_off_sel);
    WarpTopkScratch* wtk = reinterpret_cast<WarpTopkScratch*>(scratch + a.sel_off_wtk);
    const int BS = a.BS, maxnb = a.MMBPR * BS;
    const int b_first = u_first / a.N;   // lengths are staged per request
    __syncthreads();

    // group-mean query of each unit (step 1)
    for (int e = tid; e < n_units * D; e += nthreads) {
        const int us = e / D, d = e - us * D;
        float acc = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g) acc += qf[(us * G + g) * D + d];
        qg_s[e] = group_mean(acc, G);
    }
    // rows of the units, concatenated
    if (tid == 0) {
        int off = 0;
        for (int us = 0; us < n_units; ++us) {
            const int L = len_s[(u_first + us) / a.N - b_first];
            int nb = L < 0 ? -1 : (L + BS - 1) / BS;
            if (nb > maxnb) nb = -1;
            s_nb[us] = nb;
            s_roff[us] = off;
            off += max(nb, 0);
        }
        s_roff[n_units] = off;
    }
    __syncthreads();
    const int R = s_roff[n_units];

    // scores of every row (steps 2.1, 2.2): kLPR lanes per row, kU rows in
    // flight per lane, 128-bit streaming loads
    const int sub = lane / kLPR, cl = lane % kLPR;
    const size_t row_stride = static_cast<size_t>(a.N) * D * MES;
    const int rows_step = nw * kRPWL * kU;
    for (int base = 0; base < R; base += rows_step) {
        uint4 vmx[kU], vmn[kU];
        int rus[kU];
        bool live[kU];
#pragma unroll
        for (int r = 0; r < kU; ++r) {
            const int row = base + (r * nw + warp) * kRPWL + sub;
            vmx[r] = vmn[r] = make_uint4(0, 0, 0, 0);
            live[r] = false;
            rus[r] = 0;
            if (row < R) {
                int us = 0;
                while (s_roff[us + 1] <= row) ++us;
                rus[r] = us;
                const int j = row - s_roff[us];
                const int m = mbt_s[us * a.MMBPR + j / BS];
                if (m < 0 || m >= a.num_meta) {
                    set_status(a.dev_status, QS_DEV_EMETA_TABLE);
                } else {
                    live[r] = true;
                    const int nkv = static_cast<int>((u_first + us) % a.N);
                    const size_t off = (static_cast<size_t>(m) * BS + j % BS) * row_stride +
                                       static_cast<size_t>(nkv) * D * MES + cl * 16;
                    vmx[r] = ldg_stream(a.maxb + off);
                    vmn[r] = ldg_stream(a.minb + off);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kU; ++r) {
            const int row = base + (r * nw + warp) * kRPWL + sub;
            float qreg[kEl];
            const float* qs = qg_s + rus[r] * D + cl * kEl;
#pragma unroll
            for (int e = 0; e < kEl; e += 4) {
                const float4 v = *reinterpret_cast<const float4*>(qs + e);
                qreg[e] = v.x; qreg[e + 1] = v.y; qreg[e + 2] = v.z; qreg[e + 3] = v.w;
            }
            RowChunk<KT> rc;
            rc.prepare(qreg);
            const float sc = row_score_reduce<kLPR>(rc.dot(vmx[r], vmn[r]));
            if (cl == 0 && row < R) keys[row] = float_key(live[r] ? sc : __int_as_float(0xff800000));
        }
    }
    __syncthreads();

    // forced set and top-k (step 2.3 + window), one warp per unit
    for (int us = warp; us < n_units; us += nw) {
        const int u = u_first + us;
        int32_t* sel_us = sel_s + us * a.k;
        const int nb = s_nb[us];
        const int w0 = forced_window_start(len_s[(u_first + us) / a.N - b_first], BS, nb, a.t);
        const int n_forced = forced_count(nb, w0, a.t);
        if (nb < 0 || n_forced > a.k) {
            if (lane == 0) set_status(a.dev_status, nb < 0 ? QS_DEV_ESEQ_LEN : QS_DEV_EFORCED);
            for (int i = lane; i < a.k; i += 32) sel_us[i] = -1;
        } else {
            const uint32_t* ku = keys + s_roff[us];
            uint8_t* fu = flags + s_roff[us];
            for (int j = lane; j < nb; j += 32)
                fu[j] = (a.t >= 0 && (j == 0 || j >= w0)) ? kFixed : kCand;
            __syncwarp();
            const int want = min(a.k - n_forced, nb - n_forced);
            warp_topk_smem(ku, fu, nb, want, wtk[us]);
            warp_emit_flags(fu, kFixed | kPick, nb, a.k, sel_us);
        }
        __syncwarp();
        if (u * tpu >= t0) {
            int32_t* out_g = a.sel_out + static_cast<size_t>(u) * a.k;
            for (int i = lane; i < a.k; i += 32) out_g[i] = sel_us[i];
        }
    }
    __syncthreads();
}

// kSel = false: the selection is an input (a.sel, written by a selector
//   kernel that precedes this one on the stream).
// kSel = true: fused decode step.  Before streaming, every CTA computes the
//   Quest selection of each unit its tile range touches (a unit split between
//   two CTAs is selected by both, with identical arithmetic and therefore an
//   identical result); the CTA holding a unit's first tile writes it out.  No
//   CTA waits on another.
template <Dt KT, int D, int G, bool kSel>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) sparse_attn_kernel(const AttnArgs a) {
    constexpr bool kInt8 = KT == Dt::I8;
    constexpr int ES = KvTraits<KT>::es;
    constexpr int EPC = KvTraits<KT>::epc;
    constexpr int ROWB = D * ES;          // bytes of one head row of K or V
    constexpr int CR = ROWB / 16;         // 16-byte chunks per row
    constexpr int CPL = CR / 8;           // chunks per lane in Q.K (8 lanes per token)
    constexpr int EPL = D / 32;           // output channels per lane in P.V
    constexpr int qpw = kRPW / 4;         // token quads per warp and tile
    static_assert(CR % 8 == 0 && CPL >= 1, "K row must split over 8 lanes");
    static_assert(EPL % 2 == 0, "P.V uses fp32 pairs");
    static_assert((kRPW * CR) % 32 == 0, "a warp's rows split evenly over its lanes");

    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_lastv[2];   // this CTA arrived last for s_split[i]
    __shared__ int s_split[2];   // units of this CTA shared with other CTAs
    __shared__ int s_nsplit;
    TileInfo* info = reinterpret_cast<TileInfo*>(smem);
    float* qf = reinterpret_cast<float*>(smem + a.off_q);   // the units' query rows, fp32
    uint8_t* stages = smem + a.off_stage;
    unsigned long long* pbuf = reinterpret_cast<unsigned long long*>(smem + a.off_p);
    float* ml = reinterpret_cast<float*>(smem + a.off_ml);   // [NW][2G]: max, sum
    float* fbuf = reinterpret_cast<float*>(smem + a.off_f);  // [NW][G] factors, [G] max, [G] sum

    const int tid = threadIdx.x, nthreads = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int S = a.S;
    // 32-bit index arithmetic throughout: the planner keeps T below 2^31
    const int tpu = a.k * a.split;  // tiles per unit
    const int t0 = static_cast<int>(blockIdx.x) * a.tpc;
    const int t1 = min(a.T, t0 + a.tpc);
    const int n = static_cast<int>(t1 - t0);
    const int u_first = t0 / tpu;
    const int n_units = static_cast<int>((t1 - 1) / tpu - u_first + 1);
    const int b_first = u_first / a.sel_heads;
    const int n_req = static_cast<int>((u_first + n_units - 1) / a.sel_heads - b_first + 1);
    const int G_per_kv = a.H / a.N;
    if (tid == 0) s_nsplit = 0;
    constexpr int kQSlotFloats = G * D;

    // ---- prologue: stage what the preceding kernel does not write (query
    // rows, block-table rows, lengths; fused: metadata-table rows), then wait
    // for it (the selection), then convert the queries and build the tile list
    stage_unit_inputs<D, G>(a, u_first, n_units, b_first, n_req, stages);
    if constexpr (kSel) stage_meta_tables(a, u_first, n_units, stages);
    cp_async_commit();
    if constexpr (!kSel) pdl_wait();   // the selection is written by the preceding kernel
    cp_async_wait(0);
    __syncthreads();
    {
        const uint8_t* qraw = stages + a.sel_off_qraw;
        for (int e = tid; e < n_units * kQSlotFloats; e += nthreads) {
            if (a.q_dt == QS_F32) qf[e] = reinterpret_cast<const float*>(qraw)[e];
            else if (a.q_dt == QS_BF16) qf[e] = load_elem<Dt::BF16>(qraw, e);
            else qf[e] = load_elem<Dt::F16>(qraw, e);
        }
    }
    const int32_t* len_s = reinterpret_cast<const int32_t*>(stages + a.sel_off_len);
    const int32_t* bt_s = reinterpret_cast<const int32_t*>(stages + a.sel_off_bt);
    const int32_t* sel_src = a.sel;      // selection rows, indexed by unit - sel_u0
    int sel_u0 = 0;
    if constexpr (kSel) {
        quest_select_units<KT, D, G>(a, u_first, n_units, t0, tpu, qf, stages);
        sel_src = reinterpret_cast<const int32_t*>(stages + a.sel_off_sel);
        sel_u0 = u_first;
    } else {
        __syncthreads();
    }

    // tile list
    const size_t pool_row = static_cast<size_t>(a.N) * ROWB;   // bytes between tokens
    for (int i = tid; i < n; i += nthreads) {
        const int t = t0 + i;
        const int u = t / tpu;
        const int i2 = static_cast<int>(t - u * tpu);
        const int sidx = i2 / a.split, sp = i2 - sidx * a.split;
        const int b = u / a.sel_heads;
        const int s_row = static_cast<int>(u - b * a.sel_heads);
        const int nkv = a.sel_heads == a.N ? s_row : s_row / G_per_kv;
        const int j = sel_src[(u - sel_u0) * a.k + sidx];
        const int L = len_s[b - b_first];
        const int meta = static_cast<int>(u - u_first) | ((i == 0 || i2 == 0) ? kFirst : 0) |
                         ((i == n - 1 || i2 == tpu - 1) ? kLast : 0);
        TileInfo ti{0, 0, meta};
        if (j >= 0) {
            if (L < 0 || L > a.MKBPR * a.BS) {
                set_status(a.dev_status, QS_DEV_ESEQ_LEN);
            } else if (j >= (L + a.BS - 1) / a.BS) {
                set_status(a.dev_status, QS_DEV_ESELECTED);
            } else {
                const int p = a.bt_staged ? bt_s[(b - b_first) * a.MKBPR + j]
                                          : a.bt[static_cast<size_t>(b) * a.MKBPR + j];
                if (p < 0 || p >= a.num_kv_blocks) {
                    set_status(a.dev_status, QS_DEV_EBLOCK_TABLE);
                } else {
                    ti.rows = min(a.TR, max(0, L - j * a.BS - sp * a.TR));
                    ti.off = (static_cast<long long>(p) * a.BS + sp * a.TR) *
                                 static_cast<long long>(pool_row) + nkv * ROWB;
                }
            }
        }
        info[i] = ti;
    }
    __syncthreads();   // the staging area is free from here on: the ring takes it

    // ---- per-warp row streams: lane -> (row within a copy step, 16-byte
    // chunk) of the warp's kRPW rows, offsets fixed for the whole loop
    const int r0 = warp * kRPW;
    constexpr int kRowsPerCopy = CR >= 32 ? 1 : 32 / CR;          // rows one warp copy covers
    constexpr int kCopies = kRPW * CR / 32;                         // copy steps per array
    const int c_row = CR >= 32 ? 0 : lane / CR;
    const int c_chunk = CR >= 32 ? lane : lane % CR;
    const long long src_lane = static_cast<long long>(r0 + c_row) * static_cast<long long>(pool_row) +
                               c_chunk * 16;
    const long long jstep = static_cast<long long>(kRowsPerCopy) * static_cast<long long>(pool_row);
    const uint32_t ring = smem_addr(stages) + static_cast<uint32_t>(warp * S) * a.stage_bytes +
                          c_row * ROWB + c_chunk * 16;
    constexpr uint32_t dstep = kRowsPerCopy * ROWB;
    const uint32_t vpart = a.rows_bytes;
    const uint8_t* kc = a.kc;
    const uint8_t* vc = a.vc;
    auto issue = [&](int i, int st) {
        if (i < n) {
            const TileInfo ti = info[i];
            const int rw = ti.rows - r0;
            if (rw > 0) {
                const uint8_t* ks = kc + ti.off + src_lane;
                const uint8_t* vs = vc + ti.off + src_lane;
                const uint32_t d = ring + static_cast<uint32_t>(st) * a.stage_bytes;
                if (rw >= kRPW) {
#pragma unroll
                    for (int j = 0; j < kCopies; ++j) {
                        cp_async16_s(d + j * dstep, ks + j * jstep);
                        cp_async16_s(d + vpart + j * dstep, vs + j * jstep);
                    }
                } else {
                    // rows past rw: P.V reads them with p = 0, so their V
                    // bytes are zeroed (the slot may never have been loaded)
#pragma unroll
                    for (int j = 0; j < kCopies; ++j)
                        if (c_row + j * kRowsPerCopy < rw) {
                            cp_async16_s(d + j * dstep, ks + j * jstep);
                            cp_async16_s(d + vpart + j * dstep, vs + j * jstep);
                        } else {
                            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(d + vpart + j * dstep),
                                         "r"(0u)
                                         : "memory");
                        }
                }
                if constexpr (kInt8) {
                    // one fp32 scale per (token, KV head): index off / ROWB;
                    // zero past rw (P.V multiplies p = 0 by the V scale)
                    if (lane < kRPW) {
                        const uint32_t sd = smem_addr(stages) +
                                            static_cast<uint32_t>(warp * S + st) * a.stage_bytes +
                                            2 * a.rows_bytes + lane * 4;
                        if (lane < rw) {
                            const size_t si = static_cast<size_t>(ti.off / ROWB) +
                                              static_cast<size_t>(r0 + lane) * a.N;
                            cp_async4_s(sd, a.ks + si);
                            cp_async4_s(sd + kRPW * 4, a.vs + si);
                        } else {
                            asm volatile("st.shared.u32 [%0], %1;" ::"r"(sd), "r"(0u) : "memory");
                            asm volatile("st.shared.u32 [%0], %1;" ::"r"(sd + kRPW * 4), "r"(0u) : "memory");
                        }
                    }
                }
            }
        }
        cp_async_commit();
    };

    const int tq = lane >> 3, g = lane & 7;
    const int hl = head_of_lane<G>(g);
    const bool rep = rep_lane<G>(g);

    unsigned long long qp[CPL][G][EPC / 2];   // fp32 query pairs (float caches)
    int32_t q8w[CPL][G][4];                   // packed int8 query (int8 caches)
    float sq_hl = 0.f;                        // int8 query scale of head hl
    float m_run = -INFINITY, l_run = 0.f;     // for head hl
    unsigned long long acc[G][EPL / 2];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < EPL / 2; ++e) acc[h][e] = 0ull;
    unsigned long long* pw = pbuf + static_cast<size_t>(warp) * kRPW * G;
    uint8_t* mine = stages + static_cast<size_t>(warp) * S * a.stage_bytes;

    for (int i = 0; i < S - 1; ++i) issue(i, i);
    int st_cur = 0, st_next = S - 1;            // ring slots of tiles i and i+S-1
    for (int i = 0; i < n; ++i) {
        issue(i + S - 1, st_next);
        st_next = st_next + 1 == S ? 0 : st_next + 1;
        cp_async_wait(S - 1);
        __syncwarp();
        const TileInfo ti = info[i];
        const int st = st_cur;
        st_cur = st_cur + 1 == S ? 0 : st_cur + 1;
        uint8_t* cur = mine + static_cast<size_t>(st) * a.stage_bytes;
        if (ti.meta & kFirst) {
            // query rows of the unit, fp32 (and int8 quantised for int8 caches)
            const float* qs = qf + static_cast<size_t>(ti.meta & 0xff) * kQSlotFloats;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float s_q = 0.f;
                if constexpr (kInt8) {
                    float amax = 0.f;
#pragma unroll
                    for (int d = lane; d < D; d += 32) amax = fmaxf(amax, fabsf(qs[h * D + d]));
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                    s_q = amax == 0.f ? 0.f : __fdiv_rn(amax, 127.f);
                    if (h == hl) sq_hl = s_q;
                }
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    const int d0 = (g + 8 * c) * EPC;
                    float qv[EPC];
#pragma unroll
                    for (int e = 0; e < EPC; e += 4) {
                        const float4 v4 = *reinterpret_cast<const float4*>(qs + h * D + d0 + e);
                        qv[e] = v4.x; qv[e + 1] = v4.y; qv[e + 2] = v4.z; qv[e + 3] = v4.w;
                    }
                    if constexpr (kInt8) {
#pragma unroll
                        for (int w4 = 0; w4 < 4; ++w4) {
                            uint32_t word = 0;
#pragma unroll
                            for (int bb = 0; bb < 4; ++bb) {
                                int v = 0;
                                if (s_q != 0.f)
                                    v = min(127, max(-127, __float2int_rn(__fdiv_rn(qv[4 * w4 + bb], s_q))));
                                word |= (static_cast<uint32_t>(v) & 0xffu) << (8 * bb);
                            }
                            q8w[c][h][w4] = static_cast<int32_t>(word);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < EPC / 2; ++e) qp[c][h][e] = pack2(qv[2 * e], qv[2 * e + 1]);
                    }
                }
            }
        }
        const int rw = min(kRPW, ti.rows - r0);   // warp-uniform
        if (rw > 0) {
            const uint8_t* ktile = cur;
            const uint8_t* vtile = cur + a.rows_bytes;
            const float* kst = reinterpret_cast<const float*>(cur + 2 * a.rows_bytes);
            const float* vst = kst + kRPW;
            // ---- Q.K for the warp's rows (the logits of rows past rw are
            // replaced by -inf)
            float x[qpw];
#pragma unroll
            for (int qi = 0; qi < qpw; ++qi) {
                const int row = 4 * qi + tq;
                const uint8_t* krow = ktile + row * ROWB;
                float s;
                if constexpr (kInt8) {
                    int iacc[G];
#pragma unroll
                    for (int h = 0; h < G; ++h) iacc[h] = 0;
#pragma unroll
                    for (int c = 0; c < CPL; ++c) {
                        const uint4 kv = *reinterpret_cast<const uint4*>(krow + (g + 8 * c) * 16);
                        const int w[4] = {static_cast<int>(kv.x), static_cast<int>(kv.y),
                                          static_cast<int>(kv.z), static_cast<int>(kv.w)};
#pragma unroll
                        for (int h = 0; h < G; ++h)
#pragma unroll
                            for (int e = 0; e < 4; ++e) iacc[h] = __dp4a(q8w[c][h][e], w[e], iacc[h]);
                    }
                    const int tot = reduce8<G, int>(iacc, g);
                    const float sk = row < rw ? kst[row] : 0.f;
                    s = __fmul_rn(__fmul_rn(sq_hl, sk), static_cast<float>(tot)) * a.scale_log2;
                } else {
                    unsigned long long pacc[G];
#pragma unroll
                    for (int h = 0; h < G; ++h) pacc[h] = 0ull;
#pragma unroll
                    for (int c = 0; c < CPL; ++c) {
                        const uint4 kv = *reinterpret_cast<const uint4*>(krow + (g + 8 * c) * 16);
                        qk_chunk<KT, G, EPC>(qp[c], kv, pacc);
                    }
                    float hs[G];
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float2 f = unpack2(pacc[h]);
                        hs[h] = f.x + f.y;
                    }
                    s = reduce8<G, float>(hs, g) * a.scale_log2;
                }
                x[qi] = row < rw ? s : -INFINITY;
            }
            // ---- online softmax update (per warp, per head)
            float mx = x[0];
#pragma unroll
            for (int qi = 1; qi < qpw; ++qi) mx = fmaxf(mx, x[qi]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float m_new = fmaxf(m_run, mx);
            const bool grew = m_new != m_run;
            float lsum = 0.f;
#pragma unroll
            for (int qi = 0; qi < qpw; ++qi) {
                const float p = m_new == -INFINITY ? 0.f : exp2_approx(x[qi] - m_new);
                lsum += p;
                if (rep) pw[(4 * qi + tq) * G + hl] = pack2(p, p);
            }
            lsum += __shfl_xor_sync(0xffffffffu, lsum, 8);
            lsum += __shfl_xor_sync(0xffffffffu, lsum, 16);
            const float alpha = grew ? exp2_approx(m_run - m_new) : 1.f;
            l_run = l_run * alpha + lsum;
            m_run = m_new;
            if (__any_sync(0xffffffffu, grew)) {
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float al = __shfl_sync(0xffffffffu, alpha, lane_of_head<G>(h));
                    const unsigned long long a2 = pack2(al, al);
#pragma unroll
                    for (int e = 0; e < EPL / 2; ++e) acc[h][e] = mul2(acc[h][e], a2);
                }
            }
            __syncwarp();
            // ---- P.V over every row of the warp's slice: rows past rw have
            // p = 0 and finite (zeroed or earlier) data in the ring
#pragma unroll
            for (int r = 0; r < kRPW; ++r) {
                {
                    float v[EPL];
                    if constexpr (KT == Dt::F32) {
                        const float* vr = reinterpret_cast<const float*>(vtile + r * ROWB) + lane * EPL;
                        if constexpr (EPL == 4) {
                            const float4 v4 = *reinterpret_cast<const float4*>(vr);
                            v[0] = v4.x; v[1] = v4.y; v[2] = v4.z; v[3] = v4.w;
                        } else {
                            const float2 v2 = *reinterpret_cast<const float2*>(vr);
                            v[0] = v2.x; v[1] = v2.y;
                        }
                    } else if constexpr (kInt8) {
                        const uint32_t w = *reinterpret_cast<const uint32_t*>(vtile + r * ROWB + lane * EPL);
#pragma unroll
                        for (int e = 0; e < EPL; ++e) v[e] = sext8(w, e);
                    } else {
                        const uint32_t* vr = reinterpret_cast<const uint32_t*>(vtile + r * ROWB + lane * EPL * 2);
                        uint32_t vw[EPL / 2];
                        if constexpr (EPL == 4) {
                            const uint2 t2 = *reinterpret_cast<const uint2*>(vr);
                            vw[0] = t2.x; vw[1] = t2.y;
                        } else {
                            vw[0] = vr[0];
                        }
#pragma unroll
                        for (int e = 0; e < EPL / 2; ++e) {
                            const float2 f = pair_to_float2<KT>(vw[e]);
                            v[2 * e] = f.x;
                            v[2 * e + 1] = f.y;
                        }
                    }
                    unsigned long long p2[G];
                    const unsigned long long* prow = pw + r * G;
                    if constexpr (G == 4) {
                        const ulonglong2 a01 = *reinterpret_cast<const ulonglong2*>(prow);
                        const ulonglong2 a23 = *reinterpret_cast<const ulonglong2*>(prow + 2);
                        p2[0] = a01.x; p2[1] = a01.y; p2[2] = a23.x; p2[3] = a23.y;
                    } else if constexpr (G == 2) {
                        const ulonglong2 a01 = *reinterpret_cast<const ulonglong2*>(prow);
                        p2[0] = a01.x; p2[1] = a01.y;
                    } else {
                        p2[0] = prow[0];
                    }
                    if constexpr (kInt8) {
                        const float vsc = vst[r];
                        const unsigned long long s2 = pack2(vsc, vsc);
#pragma unroll
                        for (int h = 0; h < G; ++h) p2[h] = mul2(p2[h], s2);
                    }
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int e = 0; e < EPL / 2; ++e)
                            acc[h][e] = fma2(p2[h], pack2(v[2 * e], v[2 * e + 1]), acc[h][e]);
                }
            }
        }
        __syncwarp();

        // ---- end of a unit within this CTA: merge warps, write output/partial
        if (ti.meta & kLast) {
            const int u = static_cast<int>(u_first + (ti.meta & 0xff));
            float* accw = reinterpret_cast<float*>(cur);     // this warp's consumed stage slot
            const int NW = a.NW;
            if (rep && tq == 0) {
                ml[warp * 2 * G + hl] = m_run;
                ml[warp * 2 * G + G + hl] = l_run;
            }
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < EPL / 2; ++e)
                    *reinterpret_cast<unsigned long long*>(&accw[h * D + lane * EPL + 2 * e]) = acc[h][e];
            __syncthreads();
            // per head: the largest warp max, each warp's factor, the total sum
            for (int h = warp; h < G; h += NW) {
                const float mw = lane < NW ? ml[lane * 2 * G + h] : -INFINITY;
                const float lw = lane < NW ? ml[lane * 2 * G + G + h] : 0.f;
                float M = mw;
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
                const float f = (M == -INFINITY || mw == -INFINITY) ? 0.f : exp2_approx(mw - M);
                float Ls = lw * f;
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
                if (lane < NW) fbuf[lane * G + h] = f;
                if (lane == 0) {
                    fbuf[NW * G + h] = M;
                    fbuf[NW * G + G + h] = Ls;
                }
            }
            __syncthreads();
            const int ut0 = u * tpu, ut1 = ut0 + tpu;
            const bool owned = ut0 >= t0 && ut1 <= t1;
            const int b = u / a.sel_heads, s = u % a.sel_heads;
            const int h0 = a.sel_heads == a.N ? s * G_per_kv : s;
            const int c = blockIdx.x;
            float* slot = a.partial + static_cast<size_t>(c + u) * G * (D + 2);
            for (int idx = tid; idx < G * D; idx += nthreads) {
                const int h = idx / D, d = idx - h * D;
                float A = 0.f;
                for (int w = 0; w < NW; ++w) {
                    const float* aw2 = reinterpret_cast<const float*>(
                        stages + (static_cast<size_t>(w) * S + st) * a.stage_bytes);
                    A = fmaf(aw2[h * D + d], fbuf[w * G + h], A);
                }
                const float M = fbuf[NW * G + h], Ls = fbuf[NW * G + G + h];
                if (owned) {
                    a.out[(static_cast<size_t>(b) * a.H + h0 + h) * D + d] = Ls > 0.f ? A / Ls : 0.f;
                    if (d == 0 && a.lse)
                        a.lse[static_cast<size_t>(b) * a.H + h0 + h] =
                            Ls > 0.f ? (M + log2f(Ls)) * 0.69314718055994531f : -INFINITY;
                } else {
                    slot[2 * G + h * D + d] = A;
                    if (d == 0) {
                        slot[h] = M;
                        slot[G + h] = Ls;
                    }
                }
            }
            if (!owned) {
                // shared with other CTAs: merged after the tile loop
                if (tid == 0) s_split[s_nsplit++] = u;
            }
            // reset the warp state for the next unit
            m_run = -INFINITY;
            l_run = 0.f;
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < EPL / 2; ++e) acc[h][e] = 0ull;
            __syncthreads();
        }
    }
    cp_async_wait(0);

    // ---- units this CTA shares with others: the last CTA to arrive merges
    // the (max, sum, acc) partials of all of them.  One fence for all of this
    // CTA's partials, then every shared unit's arrival in the same round trip.
    __syncthreads();
    const int nsplit = s_nsplit;
    if (nsplit > 0) {
        __threadfence();
        __syncthreads();
        if (tid < nsplit) {
            const int u = s_split[tid];
            const int ut0 = u * tpu, ut1 = ut0 + tpu;
            const int c_first = static_cast<int>(ut0 / a.tpc);
            const int c_last = static_cast<int>((ut1 - 1) / a.tpc);
            const uint32_t prev = atomicAdd(&a.counters[u], 1u);
            const bool last = prev == static_cast<uint32_t>(c_last - c_first);
            if (last) a.counters[u] = 0;  // rearm for the next call
            s_lastv[tid] = last;
        }
        __syncthreads();
        for (int k2 = 0; k2 < nsplit; ++k2) {
            if (!s_lastv[k2]) continue;   // uniform: shared memory
            __threadfence();
            const int u = s_split[k2];
            const int ut0 = u * tpu, ut1 = ut0 + tpu;
            const int c_first = static_cast<int>(ut0 / a.tpc);
            const int c_last = static_cast<int>((ut1 - 1) / a.tpc);
            const int b = u / a.sel_heads, s = u % a.sel_heads;
            const int h0 = a.sel_heads == a.N ? s * G_per_kv : s;
            const int ncta = c_last - c_first + 1;
            for (int idx = tid; idx < G * D; idx += nthreads) {
                const int h = idx / D, d = idx % D;
                float M = -INFINITY, Ls = 0.f, A = 0.f;
                if (ncta <= kMergeFast) {
                    // the usual case: every partial requested in one round trip
                    float mv[kMergeFast], lv[kMergeFast], av[kMergeFast];
#pragma unroll
                    for (int q = 0; q < kMergeFast; ++q) {
                        mv[q] = -INFINITY;
                        lv[q] = av[q] = 0.f;
                        if (q < ncta) {
                            const float* sl = a.partial + static_cast<size_t>(c_first + q + u) * G * (D + 2);
                            mv[q] = ldcg_f32(sl + h);
                            lv[q] = ldcg_f32(sl + G + h);
                            av[q] = ldcg_f32(sl + 2 * G + h * D + d);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < kMergeFast; ++q) M = fmaxf(M, mv[q]);
                    if (M != -INFINITY) {
#pragma unroll
                        for (int q = 0; q < kMergeFast; ++q) {
                            const float f = q < ncta ? exp2_approx(mv[q] - M) : 0.f;
                            Ls += lv[q] * f;
                            A += av[q] * f;
                        }
                    }
                } else {
                    for (int cc = c_first; cc <= c_last; ++cc)
                        M = fmaxf(M, ldcg_f32(a.partial + static_cast<size_t>(cc + u) * G * (D + 2) + h));
                    if (M != -INFINITY) {
                        for (int cc = c_first; cc <= c_last; ++cc) {
                            const float* sl = a.partial + static_cast<size_t>(cc + u) * G * (D + 2);
                            const float f = exp2_approx(ldcg_f32(sl + h) - M);
                            Ls += ldcg_f32(sl + G + h) * f;
                            A += ldcg_f32(sl + 2 * G + h * D + d) * f;
                        }
                    }
                }
                a.out[(static_cast<size_t>(b) * a.H + h0 + h) * D + d] = Ls > 0.f ? A / Ls : 0.f;
                if (d == 0 && a.lse)
                    a.lse[static_cast<size_t>(b) * a.H + h0 + h] =
                        Ls > 0.f ? (M + log2f(Ls)) * 0.69314718055994531f : -INFINITY;
            }
        }
    }
}

struct AttnPlan {
    int grid, threads;
    size_t smem;
};

// Launch shape of the attention: tile rows TR (= BS / split), warps
// (TR / 8), tiles per CTA and ring depth.  One CTA per SM and a balanced
// stream-K split (every CTA the same number of tiles), because the tile loop
// needs all 16 warps of an SM to keep up with HBM: measured on GB300, an SM
// with 8 warps streams at about half the rate, so layouts with fewer CTAs or
// fewer warps per SM lose more than they save in split-unit merges.  Among
// the sub-tilings the per-CTA critical path (tiles x (rows + a per-tile
// overhead of about 24 rows)) is minimised.
// Shared-memory layout for one candidate; false if it does not fit.
inline bool plan_layout(int TR, int D, int G, int es, bool int8, int tpc, int q_slots,
                        size_t budget, AttnArgs* a, AttnPlan* pl) {
    const int NW = TR / kRPW;
    const int rpw = kRPW;
    if (NW < 1 || NW > kMaxWarps || TR % kRPW) return false;
    const uint32_t rows_bytes = static_cast<uint32_t>(rpw) * D * es;
    size_t stage = 2 * static_cast<size_t>(rows_bytes) + (int8 ? 2 * rpw * 4 : 0);
    const size_t merge_need = static_cast<size_t>(G) * D * 4;
    if (stage < merge_need) stage = merge_need;
    stage = align_up(stage, 128);
    size_t off = align_up(static_cast<size_t>(tpc) * sizeof(TileInfo), 128);
    a->off_q = static_cast<uint32_t>(off);
    off = align_up(off + static_cast<size_t>(q_slots) * G * D * 4, 128);
    a->off_p = static_cast<uint32_t>(off);
    off = align_up(off + static_cast<size_t>(NW) * rpw * G * 8, 128);
    a->off_ml = static_cast<uint32_t>(off);
    off = align_up(off + static_cast<size_t>(NW) * 2 * G * 4, 16);
    a->off_f = static_cast<uint32_t>(off);
    off = align_up(off + static_cast<size_t>(NW + 2) * G * 4, 128);
    a->off_stage = static_cast<uint32_t>(off);
    long long S = (static_cast<long long>(budget) - static_cast<long long>(off)) /
                  static_cast<long long>(NW * stage);
    if (S > kMaxStages) S = kMaxStages;
    if (S < 2) return false;
    pl->smem = off + static_cast<size_t>(S) * NW * stage;
    pl->threads = NW * 32;
    a->stage_bytes = static_cast<uint32_t>(stage);
    a->rows_bytes = rows_bytes;
    a->S = static_cast<int>(S);
    a->NW = NW;
    a->rpw = rpw;
    return pl->smem <= budget;
}

// Units a range of tpc tiles can touch: exactly tpc / tpu for unit-aligned
// ranges, else up to (tpc - 1) / tpu + 2.
inline long long plan_units_per_cta(long long tpc, long long tpu) {
    return tpc % tpu == 0 ? tpc / tpu : (tpc - 1) / tpu + 2;
}

// Prologue staging inside the ring region (raw query rows per unit, lengths
// and, when they fit, block-table rows per request); returns the first free
// byte after it.
inline size_t plan_staging(int G, int D, int q_es, int MKBPR, long long upc, AttnArgs* a) {
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, 16);
        return static_cast<uint32_t>(at);
    };
    const size_t ring = static_cast<size_t>(a->NW) * a->S * a->stage_bytes;
    a->sel_off_qraw = take(static_cast<size_t>(upc) * G * D * q_es);
    a->sel_off_len = take(static_cast<size_t>(upc) * 4);
    const size_t bt_bytes = static_cast<size_t>(upc) * MKBPR * 4;
    a->bt_staged = bt_bytes <= kStageTablesMax && off + bt_bytes <= ring;
    a->sel_off_bt = take(a->bt_staged ? bt_bytes : 0);
    return off;
}

bool plan_attention(int BS, int D, int G, int es, int q_es, bool int8, long long units, int k,
                    int MKBPR, AttnArgs* a, AttnPlan* pl) {
    const int nsm = num_sms();
    long long best_cost = -1;
    int best_split = 0;
    for (int split = 1; split <= 16; split *= 2) {
        if (BS % split) break;
        const int TR = BS / split;
        if (TR < 16 || TR % 16 || TR > kMaxWarps * kRPW) continue;
        const long long T = units * k * split;
        const long long tpc = (T + nsm - 1) / nsm;
        const long long cost = tpc * (TR + 24);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best_split = split;
        }
    }
    if (best_cost < 0) return false;
    const int split = best_split, TR = BS / split;
    const long long tpu = static_cast<long long>(k) * split;
    const long long T = units * tpu;
    long long tpc = (T + nsm - 1) / nsm;
    if (tpc > (kQSlots - 1) * tpu) tpc = (kQSlots - 1) * tpu;  // at most kQSlots units per CTA
    if (tpc > kMaxTilesPerCta) tpc = kMaxTilesPerCta;
    if (tpc < 1) tpc = 1;
    const long long q_slots = plan_units_per_cta(tpc, tpu);
    if (!plan_layout(TR, D, G, es, int8, static_cast<int>(tpc),
                     static_cast<int>(q_slots < kQSlots ? q_slots : kQSlots), kSmemBudget, a, pl))
        return false;
    const size_t ring = static_cast<size_t>(a->NW) * a->S * a->stage_bytes;
    a->sel_end = static_cast<uint32_t>(plan_staging(G, D, q_es, MKBPR, q_slots, a));
    if (a->sel_end > ring) return false;
    if (T + tpc > 0x7fffffffLL) return false;   // the kernel indexes tiles in 32 bits
    pl->grid = static_cast<int>((T + tpc - 1) / tpc);
    a->T = static_cast<int>(T);
    a->tpc = static_cast<int>(tpc);
    a->TR = TR;
    a->split = split;
    return true;
}

template <Dt KT, int D, int G, bool kSel>
qs_status launch_attn(const AttnArgs& a, const AttnPlan& pl, bool pdl, cudaStream_t s) {
    auto kern = sparse_attn_kernel<KT, D, G, kSel>;
    if (!ensure_smem(reinterpret_cast<const void*>(kern), pl.smem)) return QS_ECUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.grid);
    cfg.blockDim = dim3(pl.threads);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return QS_ECUDA;
    QS_CHECK_LAUNCH();
    return QS_OK;
}

template <Dt KT, int D, bool kSel = false>
qs_status dispatch_g(int G, const AttnArgs& a, const AttnPlan& pl, bool pdl, cudaStream_t s) {
    switch (G) {
        case 1: return launch_attn<KT, D, 1, kSel>(a, pl, pdl, s);
        case 2: return launch_attn<KT, D, 2, kSel>(a, pl, pdl, s);
        case 4: return launch_attn<KT, D, 4, kSel>(a, pl, pdl, s);
        default: return QS_EUNSUPPORTED;
    }
}

}  // namespace
}  // namespace qs
