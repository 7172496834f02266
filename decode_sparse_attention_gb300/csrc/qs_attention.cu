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
//  * Persistent grid of one CTA per SM; CTA c owns a contiguous range of
//    tiles (stream-K split), so every SM streams the same number of tiles.
//  * One producer warp gathers the tiles with 2-D TMA loads (tensor maps over
//    the whole paged pool; box = one head's [rows x D] slice of one block)
//    into a multi-stage shared-memory ring guarded by mbarriers; the unit's
//    query rows come in with a 1-D bulk copy.  Eight consumer warps compute.
//  * Each consumer warp keeps its own online-softmax state (running max, sum,
//    accumulator) over its rows of every tile, so tiles need no CTA-wide
//    barrier; warps are merged at the end of a unit.  Q.K uses 8 lanes per
//    token and packed fp32x2 FMAs with a transposing shuffle reduction; P.V
//    gives each lane D/32 output channels.
//  * A unit split across CTAs is merged on the device: each CTA writes a
//    (max, sum, acc) partial; the last to arrive (atomic counter, no spin)
//    combines them and rearms the counter.
//  * Launched as a programmatic dependent of the selector: barrier set-up and
//    tensor-map prefetch overlap the selector's tail.
#include <cmath>

#include "qs_common.cuh"

namespace qs {
namespace {

constexpr int kNW = 8;                      // consumer warps
constexpr int kThreadsAttn = (kNW + 1) * 32;
constexpr int kSmemBudget = 225 * 1024;

struct AttnArgs {
    const uint8_t* q;
    int q_dt, q_es;
    const int32_t* bt;
    int MKBPR;
    const int32_t* seq_lens;
    const int32_t* sel;
    int sel_heads, k, num_kv_blocks, B, H, N, BS, TR, split, S;
    float scale_log2;
    float* out;
    float* lse;
    float* partial;
    uint32_t* counters;
    long long T;
    int tpc;
    int32_t* dev_status;
    // dynamic shared memory layout (bytes from the 1024-aligned base)
    uint32_t off_v, off_q, off_sc, off_info, off_bar, off_p, off_alpha, off_merge;
    uint32_t tile_bytes, q_slot, sc_tile, sc_bytes;
};

struct TileInfo {
    int unit;
    int rows;
    int new_unit;
    int pad;
};

template <Dt KT> struct KvTraits {
    static constexpr int es = DtInfo<KT>::bytes;
    static constexpr int epc = 16 / es;  // elements per 16-byte chunk
};

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

QS_DEVINL void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

QS_DEVINL float sext8(uint32_t w, int i) {
    return static_cast<float>(static_cast<int32_t>(w << (24 - 8 * i)) >> 24);
}

template <Dt KT, int D, int G>
__global__ void __launch_bounds__(kThreadsAttn, 1)
sparse_attn_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const __grid_constant__ CUtensorMap ksmap,
                   const __grid_constant__ CUtensorMap vsmap, const AttnArgs a) {
    constexpr bool kInt8 = KT == Dt::I8;
    constexpr int ES = KvTraits<KT>::es;
    constexpr int EPC = KvTraits<KT>::epc;
    constexpr int CR = D * ES / 16;       // 16-byte chunks per K row
    constexpr int CPL = CR / 8;           // chunks per lane in Q.K (8 lanes per token)
    constexpr int EPL = D / 32;           // output channels per lane in P.V
    static_assert(CR % 8 == 0 && CPL >= 1, "K row must split over 8 lanes");
    static_assert(EPL % 2 == 0, "P.V uses fp32 pairs");

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ int s_last;

    const int S = a.S;
    uint8_t* kt = smem;
    uint8_t* vt = smem + a.off_v;
    uint8_t* qsl = smem + a.off_q;
    uint8_t* sct = smem + a.off_sc;
    TileInfo* info = reinterpret_cast<TileInfo*>(smem + a.off_info);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.off_bar);
    uint64_t* empty = full + S;
    unsigned long long* pbuf = reinterpret_cast<unsigned long long*>(smem + a.off_p);
    float* alpha_s = reinterpret_cast<float*>(smem + a.off_alpha);
    float* merge = reinterpret_cast<float*>(smem + a.off_merge);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long tpu = static_cast<long long>(a.k) * a.split;  // tiles per unit
    const long long t0 = static_cast<long long>(blockIdx.x) * a.tpc;
    const long long t1 = min(a.T, t0 + a.tpc);
    const int G_per_kv = a.H / a.N;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kNW);
        }
        fence_mbar_init();
    }
    if (warp == kNW && lane == 0) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
        if constexpr (kInt8) {
            prefetch_tensormap(&ksmap);
            prefetch_tensormap(&vsmap);
        }
    }
    __syncthreads();
    pdl_wait();  // the selection is written by the preceding kernel

    if (warp == kNW) {
        // ------------------------------------------------------------ producer
        bool timed_out = false;
        for (long long tb = t0; tb < t1 && !timed_out; tb += 32) {
            const long long t = tb + lane;
            int u = 0, rows = 0, p = 0, nu = 0, x = 0, y = 0;
            size_t qoff = 0;
            if (t < t1) {
                u = static_cast<int>(t / tpu);
                const int i2 = static_cast<int>(t % tpu);
                const int sidx = i2 / a.split, sp = i2 % a.split;
                const int b = u / a.sel_heads, s = u % a.sel_heads;
                const int n = a.sel_heads == a.N ? s : s / G_per_kv;
                const int h0 = a.sel_heads == a.N ? s * G_per_kv : s;
                nu = (t == t0) || (i2 == 0);
                qoff = (static_cast<size_t>(b) * a.H + h0) * D * a.q_es;
                const int j = a.sel[static_cast<size_t>(u) * a.k + sidx];
                const int L = a.seq_lens[b];
                if (j >= 0) {
                    if (L < 0 || L > a.MKBPR * a.BS) {
                        set_status(a.dev_status, QS_DEV_ESEQ_LEN);
                    } else if (j >= (L + a.BS - 1) / a.BS) {
                        set_status(a.dev_status, QS_DEV_ESELECTED);
                    } else {
                        p = a.bt[static_cast<size_t>(b) * a.MKBPR + j];
                        if (p < 0 || p >= a.num_kv_blocks) {
                            set_status(a.dev_status, QS_DEV_EBLOCK_TABLE);
                        } else {
                            rows = min(a.TR, max(0, L - j * a.BS - sp * a.TR));
                            x = n * D;
                            y = p * a.BS + sp * a.TR;
                        }
                    }
                }
            }
            const int cnt = static_cast<int>(min(32LL, t1 - tb));
            bool stop = false;
            for (int ii = 0; ii < cnt && !stop; ++ii) {
                const int rows_i = __shfl_sync(0xffffffffu, rows, ii);
                const int u_i = __shfl_sync(0xffffffffu, u, ii);
                const int nu_i = __shfl_sync(0xffffffffu, nu, ii);
                const int x_i = __shfl_sync(0xffffffffu, x, ii);
                const int y_i = __shfl_sync(0xffffffffu, y, ii);
                const unsigned long long qo_i = __shfl_sync(0xffffffffu, static_cast<unsigned long long>(qoff), ii);
                const long long i = tb + ii - t0;
                const int st = static_cast<int>(i % S);
                int ok = 1;
                if (lane == 0) {
                    const uint32_t par = static_cast<uint32_t>((i / S) & 1) ^ 1u;
                    ok = mbar_wait(&empty[st], par) ? 1 : 0;
                    if (!ok) set_status(a.dev_status, QS_DEV_ETIMEOUT);
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) {        // warp-uniform exit
                    stop = true;
                    break;
                }
                if (lane == 0) {
                    info[st] = TileInfo{u_i, rows_i, nu_i, 0};
                    uint32_t bytes = 0;
                    if (rows_i > 0) bytes += 2 * a.tile_bytes + (kInt8 ? 2 * a.sc_bytes : 0);
                    const uint32_t qbytes = static_cast<uint32_t>(G * D * a.q_es);
                    if (nu_i) bytes += qbytes;
                    mbar_arrive_expect_tx(&full[st], bytes);
                    if (rows_i > 0) {
                        tma_load_2d(kt + static_cast<size_t>(st) * a.tile_bytes, &kmap, x_i, y_i, &full[st]);
                        tma_load_2d(vt + static_cast<size_t>(st) * a.tile_bytes, &vmap, x_i, y_i, &full[st]);
                        if constexpr (kInt8) {
                            tma_load_2d(sct + static_cast<size_t>(st) * 2 * a.sc_tile, &ksmap, 0, y_i, &full[st]);
                            tma_load_2d(sct + static_cast<size_t>(st) * 2 * a.sc_tile + a.sc_tile, &vsmap, 0, y_i,
                                        &full[st]);
                        }
                    }
                    if (nu_i) bulk_copy_g2s(qsl + static_cast<size_t>(st) * a.q_slot, a.q + qo_i, qbytes, &full[st]);
                }
                __syncwarp();
            }
            timed_out = stop;
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int tq = lane >> 3, g = lane & 7;
    const int TR = a.TR;
    const int nwa = min(kNW, TR / 4);         // warps with rows in a tile
    const int rpw = TR / nwa;                 // rows per active warp
    const int qpw = rpw / 4;                  // quads per warp
    const bool wact = warp < nwa;
    const int r0 = warp * rpw;
    const int hl = head_of_lane<G>(g);
    const bool rep = rep_lane<G>(g);

    unsigned long long qp[CPL][G][EPC / 2];   // fp32 query pairs (float caches)
    int32_t q8w[CPL][G][4];                   // packed int8 query (int8 caches)
    float sq[G];                              // int8 query scales
    float m_run = -INFINITY, l_run = 0.f;     // for head hl
    unsigned long long acc[G][EPL / 2];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        sq[h] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL / 2; ++e) acc[h][e] = 0ull;
    }
    unsigned long long* pw = pbuf + static_cast<size_t>(warp) * rpw * G;
    float* aw = alpha_s + warp * G;
    const int ct = threadIdx.x;               // consumer thread id, < kNW*32

    bool failed = false;
    for (long long t = t0; t < t1; ++t) {
        const long long i = t - t0;
        const int st = static_cast<int>(i % S);
        const uint32_t par = static_cast<uint32_t>((i / S) & 1);
        if (!mbar_wait(&full[st], par)) {
            set_status(a.dev_status, QS_DEV_ETIMEOUT);
            failed = true;
            break;
        }
        const TileInfo ti = info[st];
        if (ti.new_unit) {
            // query rows of the unit, fp32 (and int8 quantised for int8 caches)
            const uint8_t* qs = qsl + static_cast<size_t>(st) * a.q_slot;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float s_q = 0.f;
                if constexpr (kInt8) {
                    float amax = 0.f;
                    for (int d = lane; d < D; d += 32)
                        amax = fmaxf(amax, fabsf(load_q(qs, a.q_dt, static_cast<size_t>(h) * D + d)));
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                    s_q = amax == 0.f ? 0.f : __fdiv_rn(amax, 127.f);
                    sq[h] = s_q;
                }
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    const int d0 = (g + 8 * c) * EPC;
                    float qv[EPC];
#pragma unroll
                    for (int e = 0; e < EPC; ++e) qv[e] = load_q(qs, a.q_dt, static_cast<size_t>(h) * D + d0 + e);
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
        if (wact && ti.rows > 0) {
            const int rows = ti.rows;
            const uint8_t* ktile = kt + static_cast<size_t>(st) * a.tile_bytes;
            const uint8_t* vtile = vt + static_cast<size_t>(st) * a.tile_bytes;
            const float* kst = reinterpret_cast<const float*>(sct + static_cast<size_t>(st) * 2 * a.sc_tile);
            const float* vst = reinterpret_cast<const float*>(sct + static_cast<size_t>(st) * 2 * a.sc_tile + a.sc_tile);
            const int n_kv = (ti.unit % a.sel_heads) / (a.sel_heads == a.N ? 1 : G_per_kv);
            // ---- Q.K for the warp's rows
            float x[8];
#pragma unroll
            for (int qi = 0; qi < 8; ++qi) {
                x[qi] = -INFINITY;
                if (qi < qpw) {
                    const int row = r0 + 4 * qi + tq;
                    const uint8_t* krow = ktile + static_cast<size_t>(row) * D * ES;
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
                        const float sk = kst[row * a.N + n_kv];
                        s = __fmul_rn(__fmul_rn(sq[hl], sk), static_cast<float>(tot)) * a.scale_log2;
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
                    x[qi] = row < rows ? s : -INFINITY;
                }
            }
            // ---- online softmax update (per warp, per head)
            float mx = x[0];
#pragma unroll
            for (int qi = 1; qi < 8; ++qi) mx = fmaxf(mx, x[qi]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float m_new = fmaxf(m_run, mx);
            const float alpha = m_new == -INFINITY ? 1.f : exp2_approx(m_run - m_new);
            float lsum = 0.f;
#pragma unroll
            for (int qi = 0; qi < 8; ++qi) {
                if (qi < qpw) {
                    const float p = m_new == -INFINITY ? 0.f : exp2_approx(x[qi] - m_new);
                    lsum += p;
                    if (rep) pw[(4 * qi + tq) * G + hl] = pack2(p, p);
                }
            }
            lsum += __shfl_xor_sync(0xffffffffu, lsum, 8);
            lsum += __shfl_xor_sync(0xffffffffu, lsum, 16);
            l_run = l_run * alpha + lsum;
            m_run = m_new;
            if (rep && tq == 0) aw[hl] = alpha;
            __syncwarp();
            // ---- P.V for the warp's rows
            float al[G];
#pragma unroll
            for (int h = 0; h < G; ++h) al[h] = aw[h];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const unsigned long long a2 = pack2(al[h], al[h]);
#pragma unroll
                for (int e = 0; e < EPL / 2; ++e) acc[h][e] = mul2(acc[h][e], a2);
            }
            const int rmax = min(rpw, rows - r0);
            for (int r = 0; r < rmax; ++r) {
                const int row = r0 + r;
                float v[EPL];
                if constexpr (KT == Dt::F32) {
                    const float* vr = reinterpret_cast<const float*>(vtile + static_cast<size_t>(row) * D * 4) + lane * EPL;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) v[e] = vr[e];
                } else if constexpr (kInt8) {
                    const uint32_t w = *reinterpret_cast<const uint32_t*>(vtile + static_cast<size_t>(row) * D + lane * EPL);
#pragma unroll
                    for (int e = 0; e < EPL; ++e) v[e] = sext8(w, e);
                } else {
                    const uint32_t* vr = reinterpret_cast<const uint32_t*>(vtile + static_cast<size_t>(row) * D * 2 + lane * EPL * 2);
#pragma unroll
                    for (int e = 0; e < EPL / 2; ++e) {
                        const float2 f = pair_to_float2<KT>(vr[e]);
                        v[2 * e] = f.x;
                        v[2 * e + 1] = f.y;
                    }
                }
                const unsigned long long* prow = pw + r * G;
                float vs = 1.f;
                if constexpr (kInt8) vs = vst[row * a.N + n_kv];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    unsigned long long p2 = prow[h];
                    if constexpr (kInt8) {
                        const float2 pf = unpack2(p2);
                        p2 = pack2(pf.x * vs, pf.y * vs);
                    }
#pragma unroll
                    for (int e = 0; e < EPL / 2; ++e) acc[h][e] = fma2(p2, pack2(v[2 * e], v[2 * e + 1]), acc[h][e]);
                }
            }
            __syncwarp();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);

        // ---- end of a unit within this CTA: merge warps, write output/partial
        if (t + 1 == t1 || (t + 1) % tpu == 0) {
            const int u = static_cast<int>(t / tpu);
            float* mw = merge;                                   // [kNW][G] max
            float* lw = merge + kNW * G;                         // [kNW][G] sum
            float* accw = merge + 2 * kNW * G;                   // [kNW][G][D]
            if (rep && tq == 0) {
                mw[warp * G + hl] = m_run;
                lw[warp * G + hl] = l_run;
            }
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < EPL / 2; ++e) {
                    const float2 f = unpack2(acc[h][e]);
                    accw[(warp * G + h) * D + lane * EPL + 2 * e] = f.x;
                    accw[(warp * G + h) * D + lane * EPL + 2 * e + 1] = f.y;
                }
            named_bar_sync(1, kNW * 32);
            const long long ut0 = static_cast<long long>(u) * tpu, ut1 = ut0 + tpu;
            const bool owned = ut0 >= t0 && ut1 <= t1;
            const int b = u / a.sel_heads, s = u % a.sel_heads;
            const int h0 = a.sel_heads == a.N ? s * G_per_kv : s;
            const int c = blockIdx.x;
            float* slot = a.partial + static_cast<size_t>(c + u) * G * (D + 2);
            for (int idx = ct; idx < G * D; idx += kNW * 32) {
                const int h = idx / D, d = idx % D;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kNW; ++w) M = fmaxf(M, mw[w * G + h]);
                float Ls = 0.f, A = 0.f;
                if (M != -INFINITY) {
#pragma unroll
                    for (int w = 0; w < kNW; ++w) {
                        const float f = exp2_approx(mw[w * G + h] - M);
                        Ls += lw[w * G + h] * f;
                        A += accw[(w * G + h) * D + d] * f;
                    }
                }
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
                __threadfence();
                named_bar_sync(1, kNW * 32);
                const int c_first = static_cast<int>(ut0 / a.tpc);
                const int c_last = static_cast<int>((ut1 - 1) / a.tpc);
                if (ct == 0) {
                    const uint32_t prev = atomicAdd(&a.counters[u], 1u);
                    const bool last = prev == static_cast<uint32_t>(c_last - c_first);
                    if (last) a.counters[u] = 0;
                    s_last = last;
                }
                named_bar_sync(1, kNW * 32);
                if (s_last) {
                    __threadfence();
                    for (int idx = ct; idx < G * D; idx += kNW * 32) {
                        const int h = idx / D, d = idx % D;
                        float M = -INFINITY;
                        for (int cc = c_first; cc <= c_last; ++cc)
                            M = fmaxf(M, ldcg_f32(a.partial + static_cast<size_t>(cc + u) * G * (D + 2) + h));
                        float Ls = 0.f, A = 0.f;
                        if (M != -INFINITY) {
                            for (int cc = c_first; cc <= c_last; ++cc) {
                                const float* sl = a.partial + static_cast<size_t>(cc + u) * G * (D + 2);
                                const float f = exp2_approx(ldcg_f32(sl + h) - M);
                                Ls += ldcg_f32(sl + G + h) * f;
                                A += ldcg_f32(sl + 2 * G + h * D + d) * f;
                            }
                        }
                        a.out[(static_cast<size_t>(b) * a.H + h0 + h) * D + d] = Ls > 0.f ? A / Ls : 0.f;
                        if (d == 0 && a.lse)
                            a.lse[static_cast<size_t>(b) * a.H + h0 + h] =
                                Ls > 0.f ? (M + log2f(Ls)) * 0.69314718055994531f : -INFINITY;
                    }
                }
            }
            // reset the warp state for the next unit
            m_run = -INFINITY;
            l_run = 0.f;
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < EPL / 2; ++e) acc[h][e] = 0ull;
            named_bar_sync(1, kNW * 32);
        }
    }
    (void)failed;
}

}  // namespace
}  // namespace qs

namespace qs {
namespace {

constexpr int kMaxGrid = 1024;

bool tmap_dtype(int es, CUtensorMapDataType* dt) {
    switch (es) {
        case 1: *dt = CU_TENSOR_MAP_DATA_TYPE_UINT8; return true;
        case 2: *dt = CU_TENSOR_MAP_DATA_TYPE_UINT16; return true;
        case 4: *dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT32; return true;
        default: return false;
    }
}

struct AttnPlan {
    int TR, split, S, grid;
    size_t smem;
};

// Tile rows, split and ring depth: the smallest per-CTA critical path
// (tiles x rows, plus a per-tile overhead) over the admissible sub-tilings.
bool plan_attention(int BS, int D, int G, int es, int q_es, int N, bool int8, long long units,
                    int k, AttnArgs* a, AttnPlan* pl) {
    const int nsm = num_sms();
    long long best_cost = -1;
    for (int split = 1; split <= 8; split *= 2) {
        if (BS % split) break;
        const int TR = BS / split;
        if (TR < 16 || TR % 16 || TR > 256) continue;
        const long long T = units * k * split;
        const long long tpc = (T + nsm - 1) / nsm;
        const long long cost = tpc * (TR + 24);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            pl->TR = TR;
            pl->split = split;
        }
    }
    if (best_cost < 0) return false;
    const int TR = pl->TR;
    const int nwa = TR / 4 < kNW ? TR / 4 : kNW;
    const int rpw = TR / nwa;
    const uint32_t tile_bytes = static_cast<uint32_t>(TR) * D * es;
    const uint32_t q_slot = static_cast<uint32_t>(align_up(static_cast<size_t>(G) * D * q_es, 128));
    const uint32_t sc_tile = int8 ? static_cast<uint32_t>(align_up(static_cast<size_t>(TR) * N * 4, 128)) : 0;
    const size_t per_stage = 2 * static_cast<size_t>(tile_bytes) + q_slot + 2 * sc_tile + 16 + 16;
    const size_t fixed = 1024 /* alignment slack */ + static_cast<size_t>(kNW) * rpw * G * 8 +
                         kNW * G * 4 + (2 * kNW * G + static_cast<size_t>(kNW) * G * D) * 4 + 256;
    long long S = (static_cast<long long>(kSmemBudget) - static_cast<long long>(fixed)) /
                  static_cast<long long>(per_stage);
    if (S > 8) S = 8;
    if (S < 2) return false;
    pl->S = static_cast<int>(S);
    size_t off = 0;
    off += S * tile_bytes;
    a->off_v = static_cast<uint32_t>(off);
    off += S * tile_bytes;
    a->off_q = static_cast<uint32_t>(off);
    off += S * q_slot;
    a->off_sc = static_cast<uint32_t>(off);
    off += S * 2 * sc_tile;
    a->off_info = static_cast<uint32_t>(off);
    off += S * 16;
    a->off_bar = static_cast<uint32_t>(align_up(off, 8));
    off = a->off_bar + S * 16;
    a->off_p = static_cast<uint32_t>(align_up(off, 16));
    off = a->off_p + static_cast<size_t>(kNW) * rpw * G * 8;
    a->off_alpha = static_cast<uint32_t>(align_up(off, 16));
    off = a->off_alpha + kNW * G * 4;
    a->off_merge = static_cast<uint32_t>(align_up(off, 16));
    off = a->off_merge + (2 * kNW * G + static_cast<size_t>(kNW) * G * D) * 4;
    pl->smem = off + 1024;
    a->tile_bytes = tile_bytes;
    a->q_slot = q_slot;
    a->sc_tile = sc_tile;
    a->sc_bytes = int8 ? static_cast<uint32_t>(TR) * N * 4 : 0;
    const long long T = units * k * pl->split;
    long long target = nsm < kMaxGrid ? nsm : kMaxGrid;
    if (target > T) target = T;
    if (target < 1) target = 1;
    const long long tpc = (T + target - 1) / target;
    pl->grid = static_cast<int>((T + tpc - 1) / tpc);
    a->T = T;
    a->tpc = static_cast<int>(tpc);
    a->TR = TR;
    a->split = pl->split;
    a->S = pl->S;
    return pl->smem <= static_cast<size_t>(kSmemBudget) + 1024;
}

template <Dt KT, int D, int G>
qs_status launch_attn(const AttnArgs& a, const CUtensorMap& km, const CUtensorMap& vm,
                      const CUtensorMap& ksm, const CUtensorMap& vsm, const AttnPlan& pl,
                      cudaStream_t s) {
    auto kern = sparse_attn_kernel<KT, D, G>;
    if (!ensure_smem(reinterpret_cast<const void*>(kern), pl.smem))
        return QS_ECUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.grid);
    cfg.blockDim = dim3(kThreadsAttn);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, km, vm, ksm, vsm, a) != cudaSuccess) return QS_ECUDA;
    QS_CHECK_LAUNCH();
    return QS_OK;
}

template <Dt KT, int D>
qs_status dispatch_g(int G, const AttnArgs& a, const CUtensorMap& km, const CUtensorMap& vm,
                     const CUtensorMap& ksm, const CUtensorMap& vsm, const AttnPlan& pl,
                     cudaStream_t s) {
    switch (G) {
        case 1: return launch_attn<KT, D, 1>(a, km, vm, ksm, vsm, pl, s);
        case 2: return launch_attn<KT, D, 2>(a, km, vm, ksm, vsm, pl, s);
        case 4: return launch_attn<KT, D, 4>(a, km, vm, ksm, vsm, pl, s);
        default: return QS_EUNSUPPORTED;
    }
}

}  // namespace

size_t attn_workspace_bytes(int B, int H, int N, int D, int sel_heads) {
    // counters per unit + one (max, sum, acc) partial slot per (CTA, unit)
    // pair a stream-K range can produce: at most units + grid slots.
    const long long units = static_cast<long long>(B) * sel_heads;
    const int G = sel_heads == N ? H / N : 1;
    const long long slots = units + kMaxGrid;
    return align_up(static_cast<size_t>(units) * 4, 256) +
           align_up(static_cast<size_t>(slots) * G * (D + 2) * 4, 256);
}

qs_status sparse_attn_impl(const void* q, qs_dtype q_dtype, const void* k_cache, const void* v_cache,
                           const float* k_scale, const float* v_scale, qs_dtype kv_dtype,
                           int32_t num_kv_blocks, const int32_t* block_tables, int32_t MKBPR,
                           const int32_t* seq_lens, const int32_t* selected, int32_t sel_heads,
                           int32_t k, float softmax_scale, int32_t B, int32_t H, int32_t N,
                           int32_t D, int32_t BS, float* out, float* lse_opt, void* workspace,
                           size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream) {
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
    if (BS % 16 || BS > 256 * 8) return QS_EUNSUPPORTED;
    if (int8 && N % 4) return QS_EUNSUPPORTED;              // scale rows: multiples of 16 B
    const int G = sel_heads == N ? H / N : 1;
    if (G != 1 && G != 2 && G != 4) return QS_EUNSUPPORTED;
    const int q_es = q_dtype == QS_F32 ? 4 : 2;
    const uintptr_t al = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
                         reinterpret_cast<uintptr_t>(v_cache) |
                         (int8 ? reinterpret_cast<uintptr_t>(k_scale) | reinterpret_cast<uintptr_t>(v_scale) : 0);
    if (al % 16) return QS_EINVAL;
    const long long units = static_cast<long long>(B) * sel_heads;
    AttnArgs a = {};
    AttnPlan pl = {};
    if (!plan_attention(BS, D, G, es, q_es, N, int8, units, k, &a, &pl)) return QS_EUNSUPPORTED;
    const size_t need = attn_workspace_bytes(B, H, N, D, sel_heads);
    if (!workspace || workspace_bytes < need) return QS_EWORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.q = static_cast<const uint8_t*>(q);
    a.q_dt = q_dtype;
    a.q_es = q_es;
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

    CUtensorMap km, vm, ksm, vsm;
    const uint64_t rows = static_cast<uint64_t>(num_kv_blocks) * BS;
    const uint64_t cols = static_cast<uint64_t>(N) * D;
    if (!encode_2d(&km, k_cache, es, cols, rows, cols * es, D, a.TR) ||
        !encode_2d(&vm, v_cache, es, cols, rows, cols * es, D, a.TR))
        return QS_ECUDA;
    if (int8) {
        if (!encode_2d(&ksm, k_scale, 4, N, rows, static_cast<uint64_t>(N) * 4, N, a.TR) ||
            !encode_2d(&vsm, v_scale, 4, N, rows, static_cast<uint64_t>(N) * 4, N, a.TR))
            return QS_ECUDA;
    } else {
        ksm = km;
        vsm = vm;
    }
    switch (kv_dtype) {
        case QS_F32: return D == 128 ? dispatch_g<Dt::F32, 128>(G, a, km, vm, ksm, vsm, pl, stream)
                                     : dispatch_g<Dt::F32, 64>(G, a, km, vm, ksm, vsm, pl, stream);
        case QS_BF16: return D == 128 ? dispatch_g<Dt::BF16, 128>(G, a, km, vm, ksm, vsm, pl, stream)
                                      : dispatch_g<Dt::BF16, 64>(G, a, km, vm, ksm, vsm, pl, stream);
        case QS_F16: return D == 128 ? dispatch_g<Dt::F16, 128>(G, a, km, vm, ksm, vsm, pl, stream)
                                     : dispatch_g<Dt::F16, 64>(G, a, km, vm, ksm, vsm, pl, stream);
        default: return dispatch_g<Dt::I8, 128>(G, a, km, vm, ksm, vsm, pl, stream);
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
                                workspace_bytes, dev_status, reinterpret_cast<cudaStream_t>(stream));
}
