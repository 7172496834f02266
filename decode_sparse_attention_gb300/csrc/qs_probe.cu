// Probe / prefill-importance block selection (Kestrel-LLM article 10-2
// 'sparse top-k block selection'):
//   section 2 probe loop     n_probe evenly strided tokens per block, block
//                            score = the largest probe dot product
//   importance pre-selection (k+1)/2 blocks with the largest summed prefill
//                            importance, ties to the lower index
//   top-k fill               the rest by probe score, ties to the lower index,
//                            never padded
//   recency insurance        the last block replaces the lowest-scoring probe
//                            pick; importance picks are never evicted
// One selection per query head.
//
// GB300 design: grid = (block chunks, B*N).  A CTA scores a chunk of blocks
// for all H/N query heads of one KV head, so each probed K row is read once
// for the whole group.  The request's length, the chunk's block-table
// entries, the queries and the chunk's prefill importance (into L2) are all
// requested in one round trip; every lane group then has all probe rows of
// its two blocks in flight at once, and while they are, one thread per block
// sums the block's importance in token order.  A unit of 2..8 chunks runs as
// a thread-block cluster whose CTAs write their probe scores and importance
// sums into the leader CTA's shared memory (larger units use global buffers
// and an arrival counter).  The leader then selects: the importance picks,
// then every query head at once (up to 256 blocks: counting top-k over all
// heads with every thread; more blocks: histogram top-k passes over the CTA,
// one head at a time), a min-reduction for the recency eviction, and the
// indices written in ascending order.
#include <cooperative_groups.h>

#include "qs_internal.cuh"
#include "qs_topk.cuh"

namespace qs {

struct ProbeArgs {
    const void* q;
    int q_dt;
    const uint8_t* k_cache;
    const float* k_scale;
    int num_kv_blocks;
    const int32_t* bt;
    int MKBPR;
    const int32_t* seq_lens;
    const float* importance;
    int imp_stride;
    int B, H, N, BS, k, n_probe;
    int32_t* selected;     // [B, H, k]
    float* probe;          // [B*H, MKBPR]
    float* isum;           // [B*N, MKBPR] block importance sums (global mode)
    uint32_t* counters;    // [B*N]
    int32_t* dev_status;
    uint32_t imp_smem_off;   // byte offset of the staged importance values in dynamic smem
    int imp_staged;          // the chunk's importance values fit the staging area
};

// Launches the selector for one KV dtype and head size; G = H/N in {1,2,4,8}.
template <Dt KT, int D> qs_status probe_launch(const ProbeArgs& a, int G, cudaStream_t s);

#if defined(QS_PROBE_KT)
namespace {

constexpr int kThreads = 256;

// q . K-row partial over one 16-byte chunk, for G heads.
template <Dt T, int G> struct ProbeChunk;

template <int G> struct ProbeChunk<Dt::F32, G> {
    static constexpr int kEl = 4;
    static QS_DEVINL void dot(const float (&q)[G][16], uint4 v, float (&acc)[G]) {
        const float e[4] = {__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                            __uint_as_float(v.w)};
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[h] = fmaf(q[h][i], e[i], acc[h]);
    }
};

template <Dt T, int G> struct ProbeChunk16 {
    static constexpr int kEl = 8;
    static QS_DEVINL void dot(const float (&q)[G][16], uint4 v, float (&acc)[G]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = pair_to_float2<T>(w[i]);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                acc[h] = fmaf(q[h][2 * i], f.x, acc[h]);
                acc[h] = fmaf(q[h][2 * i + 1], f.y, acc[h]);
            }
        }
    }
};
template <int G> struct ProbeChunk<Dt::BF16, G> : ProbeChunk16<Dt::BF16, G> {};
template <int G> struct ProbeChunk<Dt::F16, G> : ProbeChunk16<Dt::F16, G> {};

enum Mode : int { kSingle = 0, kCluster = 1, kGlobal = 2 };

// Blocks one CTA scores: every lane group (one K row per group) takes two
// blocks and has all their probe rows in flight at once.
template <Dt KT, int D> constexpr int blocks_per_chunk() {
    return 2 * (kThreads / (D * DtInfo<KT>::bytes / 16));
}
constexpr int kProbeBatch = 8;     // probe rows of one block loaded together

template <Dt KT, int D, int G, int MODE>
__global__ void __launch_bounds__(kThreads, 1) probe_select_kernel(ProbeArgs a) {
    constexpr bool kInt8 = KT == Dt::I8;
    constexpr int kElemBytes = DtInfo<KT>::bytes;
    constexpr int kLanesPerRow = D * kElemBytes / 16;
    constexpr int kEl = 16 / kElemBytes;  // elements per 16-byte chunk
    constexpr int kGroups = kThreads / kLanesPerRow;
    constexpr int kBlocksPerChunk = blocks_per_chunk<KT, D>();
    static_assert(kLanesPerRow >= 1 && kLanesPerRow <= 32, "row must span 1..32 lanes");

    // dynamic: probe keys [G][kstr] u32, importance keys [kstr] u32 (kstr =
    // MKBPR rounded up to 4 words), flags [G][MKBPR] u8, importance flags
    // [MKBPR] u8
    extern __shared__ __align__(16) uint8_t dyn[];
    __shared__ __align__(16) float s_q[G][D];
    __shared__ __align__(16) int8_t s_q8[G][D];
    __shared__ float s_sq[G];
    __shared__ TopkFastScratch s_fast;
    __shared__ TopkScratch<kThreads> s_topk;
    __shared__ unsigned long long s_wmin[kThreads / 32];   // recency: lowest (probe key, index) pick per warp
    __shared__ int s_last;

    pdl_launch_dependents();

    const int u = blockIdx.y;
    const int b = u / a.N, n = u % a.N;
    const int BS = a.BS;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int grp = threadIdx.x / kLanesPerRow;
    const int cl = threadIdx.x % kLanesPerRow;
    const int j_base = blockIdx.x * kBlocksPerChunk + grp;
    const int kstr = (a.MKBPR + 3) & ~3;
    // one round trip for everything that depends on no other load: the
    // length, the lane group's block-table entries, the queries and (into
    // L2) the importance of the chunk's tokens
    const int L = ldg_now_s32(a.seq_lens + b);
    int p_raw[2];
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
        const int j = j_base + jj * kGroups;
        p_raw[jj] = j < a.MKBPR ? ldg_now_s32(a.bt + static_cast<size_t>(b) * a.MKBPR + j) : -1;
    }
    constexpr int kQPerThread = (G * D + kThreads - 1) / kThreads;
    uint32_t qbits[kQPerThread];
#pragma unroll
    for (int r = 0; r < kQPerThread; ++r) {
        const int i = threadIdx.x + r * kThreads;
        qbits[r] = i < G * D ? ldg_now_q_bits(a.q, a.q_dt, (static_cast<size_t>(b) * a.H + n * G) * D + i) : 0u;
    }
    // the chunk's importance values go to shared memory (4-byte cp.async)
    const float* imp_row = a.importance ? a.importance + static_cast<size_t>(b) * a.imp_stride : nullptr;
    const long long imp_t0 = static_cast<long long>(blockIdx.x) * kBlocksPerChunk * BS;
    float* s_imp = reinterpret_cast<float*>(dyn + a.imp_smem_off);
    if (imp_row && a.imp_staged) {
        const long long t1 = min(static_cast<long long>(a.imp_stride),
                                 imp_t0 + static_cast<long long>(kBlocksPerChunk) * BS);
        for (long long t = imp_t0 + threadIdx.x; t < t1; t += kThreads)
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(s_imp + (t - imp_t0))),
                         "l"(imp_row + t)
                         : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    const bool bad_len = L < 0 || L > a.MKBPR * BS ||
                         (a.importance != nullptr && L > a.imp_stride);
    if (bad_len) {   // uniform over the unit's CTAs
        if (blockIdx.x == 0) {
            if (threadIdx.x == 0) set_status(a.dev_status, QS_DEV_ESEQ_LEN);
            for (int i = threadIdx.x; i < G * a.k; i += kThreads)
                a.selected[(static_cast<size_t>(b) * a.H + n * G) * a.k + i] = -1;
        }
        return;
    }
    const int nb = (L + BS - 1) / BS;
    const int n_chunks = max(1, (nb + kBlocksPerChunk - 1) / kBlocksPerChunk);
    if (MODE != kCluster && static_cast<int>(blockIdx.x) >= n_chunks) return;
    const int n_probe = max(1, a.n_probe);
    uint32_t* pkeys = reinterpret_cast<uint32_t*>(dyn);
    uint32_t* ikeys = pkeys + static_cast<size_t>(G) * kstr;
    uint8_t* flags = reinterpret_cast<uint8_t*>(ikeys + kstr);   // [G][MKBPR]
    uint8_t* imp_flags = flags + static_cast<size_t>(G) * a.MKBPR;
    uint32_t* dst_pkeys = pkeys;
    uint32_t* dst_ikeys = ikeys;
    if constexpr (MODE == kCluster) {
        dst_pkeys = cooperative_groups::this_cluster().map_shared_rank(pkeys, 0);
        dst_ikeys = cooperative_groups::this_cluster().map_shared_rank(ikeys, 0);
    }
    topk_fast_clear<kThreads>(s_fast, nb);

    // queries of the group (fp32), plus the int8 quantisation for int8 caches
#pragma unroll
    for (int r = 0; r < kQPerThread; ++r) {
        const int i = threadIdx.x + r * kThreads;
        if (i < G * D) s_q[i / D][i % D] = q_bits_value(qbits[r], a.q_dt);
    }
    __syncthreads();
    if constexpr (kInt8) {
        for (int h = warp; h < G; h += kThreads / 32) {
            float amax = 0.f;
            for (int d = lane; d < D; d += 32) amax = fmaxf(amax, fabsf(s_q[h][d]));
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const float sq = amax == 0.f ? 0.f : __fdiv_rn(amax, 127.f);
            for (int d = lane; d < D; d += 32) {
                int v = 0;
                if (sq != 0.f) v = min(127, max(-127, __float2int_rn(__fdiv_rn(s_q[h][d], sq))));
                s_q8[h][d] = static_cast<int8_t>(v);
            }
            if (lane == 0) s_sq[h] = sq;
        }
        __syncthreads();
    }

    // ---- probe scores of this chunk's blocks (two blocks per lane group)
    const unsigned gmask = kLanesPerRow == 32
                               ? 0xffffffffu
                               : (((1u << kLanesPerRow) - 1u) << (lane / kLanesPerRow * kLanesPerRow));
    float qr[G][16];
    int32_t q8r[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        if constexpr (kInt8) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                q8r[h][i] = *reinterpret_cast<const int32_t*>(&s_q8[h][cl * 16 + 4 * i]);
        } else {
#pragma unroll
            for (int i = 0; i < kEl; ++i) qr[h][i] = s_q[h][cl * kEl + i];
        }
    }
    const size_t row_bytes = static_cast<size_t>(a.N) * D * kElemBytes;
    int p_blk[2], p0s[2], steps[2], nps[2];
    uint4 v[2][kProbeBatch];
    float sk[2][kProbeBatch];
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
        const int j = j_base + jj * kGroups;
        nps[jj] = 0;
        p_blk[jj] = -1;
        if (j < nb) {
            const int p = p_raw[jj];
            if (p < 0 || p >= a.num_kv_blocks) {
                if (cl == 0) set_status(a.dev_status, QS_DEV_EBLOCK_TABLE);
            } else {
                const int p0 = j * BS, p_end = min(p0 + BS, L);
                steps[jj] = max(1, (p_end - p0) / n_probe);
                nps[jj] = (p_end - p0 + steps[jj] - 1) / steps[jj];
                p_blk[jj] = p;
                p0s[jj] = p0;
            }
        }
    }
    // first batch of both blocks in flight together
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
        const uint8_t* base = a.k_cache + static_cast<size_t>(max(p_blk[jj], 0)) * BS * row_bytes +
                              static_cast<size_t>(n) * D * kElemBytes + cl * 16;
#pragma unroll
        for (int i = 0; i < kProbeBatch; ++i) {
            v[jj][i] = make_uint4(0, 0, 0, 0);
            sk[jj][i] = 0.f;
            if (i < nps[jj]) {
                const int t = i * steps[jj];
                v[jj][i] = ldg_stream(base + static_cast<size_t>(t) * row_bytes);
                if constexpr (kInt8) sk[jj][i] = a.k_scale[(static_cast<size_t>(p_blk[jj]) * BS + t) * a.N + n];
            }
        }
    }
    // importance of this chunk's blocks while the probe rows are in flight:
    // one thread per block, the sum taken in token order (fp32, sequential,
    // as the importance picks require) from the values staged in shared memory
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    if (imp_row) {
        for (int jj = threadIdx.x; jj < kBlocksPerChunk; jj += kThreads) {
            const int j = blockIdx.x * kBlocksPerChunk + jj;
            if (j >= nb) break;
            const int p0 = j * BS, p_end = min(p0 + BS, L);
            const float* src = a.imp_staged ? s_imp + (p0 - imp_t0) : imp_row + p0;
            float sacc = 0.f;
#pragma unroll 8
            for (int t = 0; t < p_end - p0; ++t) sacc = __fadd_rn(sacc, src[t]);
            if (MODE != kGlobal) dst_ikeys[j] = float_key(sacc);
            else a.isum[static_cast<size_t>(u) * a.MKBPR + j] = sacc;
        }
    }
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
        const int j = j_base + jj * kGroups;
        float best[G];
#pragma unroll
        for (int h = 0; h < G; ++h) best[h] = -1e30f;
        for (int i0 = 0; i0 < nps[jj]; i0 += kProbeBatch) {
            if (i0 > 0) {   // more probes than one batch (short final block)
                const uint8_t* base = a.k_cache + static_cast<size_t>(p_blk[jj]) * BS * row_bytes +
                                      static_cast<size_t>(n) * D * kElemBytes + cl * 16;
#pragma unroll
                for (int i = 0; i < kProbeBatch; ++i)
                    if (i0 + i < nps[jj]) {
                        const int t = (i0 + i) * steps[jj];
                        v[jj][i] = ldg_stream(base + static_cast<size_t>(t) * row_bytes);
                        if constexpr (kInt8)
                            sk[jj][i] = a.k_scale[(static_cast<size_t>(p_blk[jj]) * BS + t) * a.N + n];
                    }
            }
#pragma unroll
            for (int i = 0; i < kProbeBatch; ++i) {
                if (i0 + i >= nps[jj]) break;
                if constexpr (kInt8) {
                    const int w[4] = {static_cast<int>(v[jj][i].x), static_cast<int>(v[jj][i].y),
                                      static_cast<int>(v[jj][i].z), static_cast<int>(v[jj][i].w)};
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        int acc = 0;
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc = __dp4a(q8r[h][e], w[e], acc);
#pragma unroll
                        for (int o = kLanesPerRow / 2; o >= 1; o >>= 1) acc += __shfl_xor_sync(gmask, acc, o);
                        const float dot = __fmul_rn(__fmul_rn(s_sq[h], sk[jj][i]), static_cast<float>(acc));
                        best[h] = fmaxf(best[h], dot);
                    }
                } else {
                    float acc[G];
#pragma unroll
                    for (int h = 0; h < G; ++h) acc[h] = 0.f;
                    ProbeChunk<KT, G>::dot(qr, v[jj][i], acc);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
#pragma unroll
                        for (int o = kLanesPerRow / 2; o >= 1; o >>= 1) acc[h] += __shfl_xor_sync(gmask, acc[h], o);
                        best[h] = fmaxf(best[h], acc[h]);
                    }
                }
            }
        }
        if (cl == 0 && j < nb) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                if (MODE != kGlobal) dst_pkeys[h * kstr + j] = float_key(best[h]);
                else a.probe[(static_cast<size_t>(b) * a.H + n * G + h) * a.MKBPR + j] = best[h];
            }
        }
    }

    // ---- all probe scores of the unit in the leader's shared memory
    if constexpr (MODE == kCluster) {
        cooperative_groups::this_cluster().sync();
        if (blockIdx.x != 0) return;
    } else if constexpr (MODE == kGlobal) {
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const uint32_t prev = atomicAdd(&a.counters[u], 1u);
            s_last = prev == static_cast<uint32_t>(n_chunks - 1);
            if (s_last) a.counters[u] = 0;
        }
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        for (int e = threadIdx.x; e < G * nb; e += kThreads) {
            const int h = e / nb, j = e % nb;
            pkeys[h * kstr + j] =
                float_key(ldcg_f32(a.probe + (static_cast<size_t>(b) * a.H + n * G + h) * a.MKBPR + j));
        }
        if (a.importance)
            for (int j = threadIdx.x; j < nb; j += kThreads)
                ikeys[j] = float_key(ldcg_f32(a.isum + static_cast<size_t>(u) * a.MKBPR + j));
    } else {
        __syncthreads();
    }

    // ---- importance pre-selection (same for every head of the request)
    const int n_imp = a.importance ? min((a.k + 1) / 2, nb) : 0;
    const bool small = nb <= kProbeRankMax && G * nb <= kThreads * kRankMaxPerThread &&
                       G <= kThreads / 32;
    for (int j = threadIdx.x; j < nb; j += kThreads) imp_flags[j] = kCand;
    if (small) {   // the counting top-k reads whole groups of 4 keys: zero padding
        const int pad = ((nb + 3) & ~3) - nb;
        for (int e = threadIdx.x; e < (G + 1) * pad; e += kThreads)
            (e < G * pad ? pkeys + static_cast<size_t>(e / pad) * kstr : ikeys)[nb + e % pad] = 0u;
    }
    __syncthreads();
    if (n_imp > 0) {
        if (small) {
            block_rank_topk<kThreads>(ikeys, 0, imp_flags, 0, nb, 1, n_imp);
            __syncthreads();
        } else {
            topk_fast<kThreads>(ikeys, imp_flags, nb, n_imp, s_fast, s_topk);
        }
    }
    for (int j = threadIdx.x; j < nb; j += kThreads)
        imp_flags[j] = (imp_flags[j] & kPick) ? kFixed : 0;
    const int want = min(a.k - n_imp, nb - n_imp);
    if (small) {
        // every query head at once: the importance picks leave the candidates
        // (their keys zeroed), counting top-k over all heads, then one warp
        // per head for recency and the ordered output
        __syncthreads();
        for (int e = threadIdx.x; e < G * nb; e += kThreads) {
            const int h = e / nb, j = e - h * nb;
            const bool fixed = imp_flags[j] != 0;
            flags[static_cast<size_t>(h) * a.MKBPR + j] = fixed ? kFixed : kCand;
            if (fixed) pkeys[static_cast<size_t>(h) * kstr + j] = 0u;
        }
        __syncthreads();
        block_rank_topk<kThreads>(pkeys, kstr, flags, a.MKBPR, nb, G, want);
        __syncthreads();
        if (warp < G) {
            const int h = warp;
            const size_t row = static_cast<size_t>(b) * a.H + n * G + h;
            const uint32_t* keys = pkeys + static_cast<size_t>(h) * kstr;
            uint8_t* fl = flags + static_cast<size_t>(h) * a.MKBPR;
            if (want > 0 && !(fl[nb - 1] & (kFixed | kPick))) {
                // the last block replaces the probe pick with the lowest probe
                // score (ties: the larger index); importance picks stay
                unsigned long long mine = ~0ull;
                for (int j = lane; j < nb; j += 32)
                    if (fl[j] & kPick) {
                        const unsigned long long c = (static_cast<unsigned long long>(keys[j]) << 32) |
                                                     (0xffffffffu - static_cast<uint32_t>(j));
                        mine = c < mine ? c : mine;
                    }
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) {
                    const unsigned long long other = __shfl_xor_sync(0xffffffffu, mine, o);
                    mine = other < mine ? other : mine;
                }
                if (lane == 0) {
                    const int victim = static_cast<int>(0xffffffffu - static_cast<uint32_t>(mine & 0xffffffffu));
                    fl[victim] &= static_cast<uint8_t>(~kPick);
                    fl[nb - 1] |= kPick;
                }
                __syncwarp();
            }
            warp_emit_flags(fl, kFixed | kPick, nb, a.k, a.selected + row * a.k);
        }
        return;
    }

    // ---- per query head: probe fill, recency insurance, ordered output
    for (int h = 0; h < G; ++h) {
        const size_t row = static_cast<size_t>(b) * a.H + n * G + h;
        const uint32_t* keys = pkeys + static_cast<size_t>(h) * kstr;
        topk_fast_clear<kThreads>(s_fast, nb);
        for (int j = threadIdx.x; j < nb; j += kThreads) flags[j] = imp_flags[j] ? kFixed : kCand;
        __syncthreads();
        topk_fast<kThreads>(keys, flags, nb, want, s_fast, s_topk);
        if (want > 0 && !(flags[nb - 1] & (kFixed | kPick))) {
            // the last block replaces the probe pick with the lowest probe
            // score (ties: the larger index); importance picks stay
            unsigned long long mine = ~0ull;
            for (int j = threadIdx.x; j < nb; j += kThreads)
                if (flags[j] & kPick) {
                    const unsigned long long c =
                        (static_cast<unsigned long long>(keys[j]) << 32) | (0xffffffffu - static_cast<uint32_t>(j));
                    mine = c < mine ? c : mine;
                }
            // minimum over the block: warp shuffles, then one thread over the warps
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const unsigned long long other = __shfl_xor_sync(0xffffffffu, mine, o);
                mine = other < mine ? other : mine;
            }
            if (lane == 0) s_wmin[warp] = mine;
            __syncthreads();
            if (threadIdx.x == 0) {
                unsigned long long best = ~0ull;
                for (int w = 0; w < kThreads / 32; ++w) best = s_wmin[w] < best ? s_wmin[w] : best;
                const int victim = static_cast<int>(0xffffffffu - static_cast<uint32_t>(best & 0xffffffffu));
                flags[victim] &= static_cast<uint8_t>(~kPick);
                flags[nb - 1] |= kPick;
            }
            __syncthreads();
        }
        block_emit_flags<kThreads>(flags, kFixed | kPick, nb, a.k, a.selected + row * a.k, s_topk);
        __syncthreads();
    }
}

template <Dt KT, int D, int G, int MODE>
qs_status launch_mode(const ProbeArgs& a, int chunks, size_t smem, cudaStream_t s) {
    auto kern = probe_select_kernel<KT, D, G, MODE>;
    if (!ensure_smem(reinterpret_cast<const void*>(kern), smem)) return QS_ECUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(chunks, a.B * a.N);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = chunks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = MODE == kCluster ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return QS_ECUDA;
    QS_CHECK_LAUNCH();
    return QS_OK;
}

template <Dt KT, int D, int G>
qs_status launch(const ProbeArgs& a, cudaStream_t s) {
    constexpr int kBlocksPerChunk = blocks_per_chunk<KT, D>();
    const size_t kstr = (static_cast<size_t>(a.MKBPR) + 3) & ~static_cast<size_t>(3);
    const size_t keys_smem = align_up(kstr * (4 * G + 4) + static_cast<size_t>(a.MKBPR) * (G + 1), 16);
    // the chunk's importance values are staged in shared memory up to 64 KB
    // (block sizes beyond that read them from global memory)
    const size_t imp_bytes = static_cast<size_t>(kBlocksPerChunk) * a.BS * 4;
    const bool staged = a.importance != nullptr && imp_bytes <= 64 * 1024;
    const size_t smem = keys_smem + (staged ? imp_bytes : 0);
    if (smem > 160 * 1024) return QS_EUNSUPPORTED;
    ProbeArgs a2 = a;
    a2.imp_smem_off = static_cast<uint32_t>(keys_smem);
    a2.imp_staged = staged ? 1 : 0;
    const int chunks = max(1, (a.MKBPR + kBlocksPerChunk - 1) / kBlocksPerChunk);
    if (chunks == 1) return launch_mode<KT, D, G, kSingle>(a2, chunks, smem, s);
    if (chunks <= 8) return launch_mode<KT, D, G, kCluster>(a2, chunks, smem, s);
    return launch_mode<KT, D, G, kGlobal>(a2, chunks, smem, s);
}

}  // namespace

template <Dt KT, int D>
qs_status probe_launch(const ProbeArgs& a, int G, cudaStream_t s) {
    switch (G) {
        case 1: return launch<KT, D, 1>(a, s);
        case 2: return launch<KT, D, 2>(a, s);
        case 4: return launch<KT, D, 4>(a, s);
        case 8: return launch<KT, D, 8>(a, s);
        default: return QS_EUNSUPPORTED;
    }
}

// One (KV dtype, D) pair per object file: the build compiles this file once
// per pair so that the kernel variants compile in parallel.
template qs_status probe_launch<Dt::QS_PROBE_KT, QS_PROBE_D>(const ProbeArgs&, int, cudaStream_t);

}  // namespace qs
#endif  // QS_PROBE_KT

#if !defined(QS_PROBE_KT)
extern template qs_status probe_launch<Dt::F32, 128>(const ProbeArgs&, int, cudaStream_t);
extern template qs_status probe_launch<Dt::F32, 64>(const ProbeArgs&, int, cudaStream_t);
extern template qs_status probe_launch<Dt::BF16, 128>(const ProbeArgs&, int, cudaStream_t);
extern template qs_status probe_launch<Dt::BF16, 64>(const ProbeArgs&, int, cudaStream_t);
extern template qs_status probe_launch<Dt::F16, 128>(const ProbeArgs&, int, cudaStream_t);
extern template qs_status probe_launch<Dt::F16, 64>(const ProbeArgs&, int, cudaStream_t);
extern template qs_status probe_launch<Dt::I8, 128>(const ProbeArgs&, int, cudaStream_t);

namespace {
constexpr int kMaxG = 8;
}  // namespace

size_t probe_workspace_bytes(int B, int H, int N, int MKBPR) {
    // probe scores [B*H, MKBPR], importance sums [B*N, MKBPR], counters [B*N]
    return align_up(static_cast<size_t>(B) * H * MKBPR * 4, 256) +
           align_up(static_cast<size_t>(B) * N * MKBPR * 4, 256) +
           align_up(static_cast<size_t>(B) * N * 4, 256);
}

qs_status probe_select_impl(const void* q, qs_dtype q_dtype, const void* k_cache,
                            const float* k_scale, qs_dtype kv_dtype, int32_t num_kv_blocks,
                            const int32_t* block_tables, int32_t MKBPR, const int32_t* seq_lens,
                            const float* importance, int32_t importance_stride, int32_t B,
                            int32_t H, int32_t N, int32_t D, int32_t BS, int32_t k,
                            int32_t n_probe, int32_t* selected, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream) {
    if (B < 0 || H <= 0 || N <= 0 || H % N != 0 || BS <= 0 || k <= 0 || MKBPR < 0 ||
        num_kv_blocks < 0)
        return QS_EINVAL;
    if (B == 0) return QS_OK;
    if (!q || !k_cache || !block_tables || !seq_lens || !selected || !dev_status) return QS_EINVAL;
    if (importance && importance_stride <= 0) return QS_EINVAL;
    if (q_dtype != QS_F32 && q_dtype != QS_BF16 && q_dtype != QS_F16) return QS_EDTYPE;
    if (kv_dtype == QS_I8 && !k_scale) return QS_EINVAL;
    if (D != 64 && D != 128) return QS_EUNSUPPORTED;
    if (kv_dtype == QS_I8 && D != 128) return QS_EUNSUPPORTED;
    const int G = H / N;
    if (G > kMaxG) return QS_EUNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(k_cache) % 16) return QS_EINVAL;
    const size_t need = probe_workspace_bytes(B, H, N, MKBPR);
    if (!workspace || workspace_bytes < need) return QS_EWORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    ProbeArgs a;
    a.q = q;
    a.q_dt = q_dtype;
    a.k_cache = static_cast<const uint8_t*>(k_cache);
    a.k_scale = k_scale;
    a.num_kv_blocks = num_kv_blocks;
    a.bt = block_tables;
    a.MKBPR = MKBPR;
    a.seq_lens = seq_lens;
    a.importance = importance;
    a.imp_stride = importance_stride;
    a.B = B; a.H = H; a.N = N; a.BS = BS; a.k = k; a.n_probe = n_probe;
    a.selected = selected;
    a.probe = reinterpret_cast<float*>(ws);
    a.isum = reinterpret_cast<float*>(ws + align_up(static_cast<size_t>(B) * H * MKBPR * 4, 256));
    a.counters = reinterpret_cast<uint32_t*>(ws + align_up(static_cast<size_t>(B) * H * MKBPR * 4, 256) +
                                             align_up(static_cast<size_t>(B) * N * MKBPR * 4, 256));
    a.dev_status = dev_status;
    switch (kv_dtype) {
        case QS_F32: return D == 128 ? probe_launch<Dt::F32, 128>(a, G, stream) : probe_launch<Dt::F32, 64>(a, G, stream);
        case QS_BF16: return D == 128 ? probe_launch<Dt::BF16, 128>(a, G, stream) : probe_launch<Dt::BF16, 64>(a, G, stream);
        case QS_F16: return D == 128 ? probe_launch<Dt::F16, 128>(a, G, stream) : probe_launch<Dt::F16, 64>(a, G, stream);
        case QS_I8: return probe_launch<Dt::I8, 128>(a, G, stream);
        default: return QS_EDTYPE;
    }
}

}  // namespace qs

extern "C" qs_status qs_probe_select(const void* q, qs_dtype q_dtype, const void* k_cache,
                                     const float* k_scale, qs_dtype kv_dtype,
                                     int32_t num_kv_blocks, const int32_t* block_tables,
                                     int32_t MKBPR, const int32_t* seq_lens,
                                     const float* importance, int32_t importance_stride,
                                     int32_t B, int32_t H, int32_t N, int32_t D, int32_t BS,
                                     int32_t k, int32_t n_probe, int32_t* selected,
                                     void* workspace, size_t workspace_bytes,
                                     int32_t* dev_status, qs_stream_t stream) {
    return qs::probe_select_impl(q, q_dtype, k_cache, k_scale, kv_dtype, num_kv_blocks,
                                 block_tables, MKBPR, seq_lens, importance, importance_stride, B,
                                 H, N, D, BS, k, n_probe, selected, workspace, workspace_bytes,
                                 dev_status, reinterpret_cast<cudaStream_t>(stream));
}
#endif  // !QS_PROBE_KT
