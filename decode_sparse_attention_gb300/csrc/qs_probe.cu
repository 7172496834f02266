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
// for the whole group.  The last CTA of a (request, KV head) runs the
// selection for its query heads: two CTA-wide radix top-k passes (importance,
// then probe) and a min-reduction for the recency eviction.
#include "qs_common.cuh"
#include "qs_topk.cuh"

namespace qs {
namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerChunk = 8;
constexpr int kMaxG = 8;

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
    uint32_t* counters;    // [B*N]
    int32_t* dev_status;
};

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

template <Dt KT, int D, int G>
__global__ void __launch_bounds__(kThreads) probe_select_kernel(ProbeArgs a) {
    constexpr bool kInt8 = KT == Dt::I8;
    constexpr int kElemBytes = DtInfo<KT>::bytes;
    constexpr int kLanesPerRow = D * kElemBytes / 16;
    constexpr int kEl = 16 / kElemBytes;  // elements per 16-byte chunk
    constexpr int kGroups = kThreads / kLanesPerRow;
    static_assert(kLanesPerRow >= 1 && kLanesPerRow <= 32, "row must span 1..32 lanes");

    extern __shared__ __align__(16) uint8_t dyn[];
    __shared__ __align__(16) float s_q[G][D];
    __shared__ __align__(16) int8_t s_q8[G][D];
    __shared__ float s_sq[G];
    __shared__ TopkScratch<kThreads> s_topk;
    __shared__ int s_last;

    pdl_launch_dependents();

    const int u = blockIdx.y;
    const int b = u / a.N, n = u % a.N;
    const int BS = a.BS;
    const int L = a.seq_lens[b];
    const bool bad_len = L < 0 || L > a.MKBPR * BS ||
                         (a.importance != nullptr && L > a.imp_stride);
    if (bad_len) {
        if (blockIdx.x == 0) {
            if (threadIdx.x == 0) set_status(a.dev_status, QS_DEV_ESEQ_LEN);
            for (int i = threadIdx.x; i < G * a.k; i += kThreads)
                a.selected[(static_cast<size_t>(b) * a.H + n * G) * a.k + i] = -1;
        }
        return;
    }
    const int nb = (L + BS - 1) / BS;
    const int n_chunks = max(1, (nb + kBlocksPerChunk - 1) / kBlocksPerChunk);
    if (static_cast<int>(blockIdx.x) >= n_chunks) return;
    const int n_probe = max(1, a.n_probe);

    // queries of the group (fp32), plus the int8 quantisation for int8 caches
    for (int i = threadIdx.x; i < G * D; i += kThreads) {
        const int h = i / D, d = i % D;
        s_q[h][d] = load_q(a.q, a.q_dt, (static_cast<size_t>(b) * a.H + n * G + h) * D + d);
    }
    __syncthreads();
    if constexpr (kInt8) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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

    // probe scores of this chunk's blocks
    const int lane = threadIdx.x & 31;
    const int grp = threadIdx.x / kLanesPerRow;
    const int cl = threadIdx.x % kLanesPerRow;
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
    const int j_begin = blockIdx.x * kBlocksPerChunk;
    const int j_end = min(nb, j_begin + kBlocksPerChunk);
    for (int j = j_begin + grp; j < j_end; j += kGroups) {
        const int p = a.bt[static_cast<size_t>(b) * a.MKBPR + j];
        float best[G];
#pragma unroll
        for (int h = 0; h < G; ++h) best[h] = -1e30f;
        if (p < 0 || p >= a.num_kv_blocks) {
            if (cl == 0) set_status(a.dev_status, QS_DEV_EBLOCK_TABLE);
        } else {
            const int p0 = j * BS;
            const int p_end = min(p0 + BS, L);
            const int step = max(1, (p_end - p0) / n_probe);
            const uint8_t* base = a.k_cache + static_cast<size_t>(p) * BS * row_bytes +
                                  static_cast<size_t>(n) * D * kElemBytes + cl * 16;
            for (int ps = p0; ps < p_end; ps += step) {
                const int t = ps - p0;
                const uint4 v = ldg_stream(base + static_cast<size_t>(t) * row_bytes);
                if constexpr (kInt8) {
                    int acc[G];
                    const int w[4] = {static_cast<int>(v.x), static_cast<int>(v.y),
                                      static_cast<int>(v.z), static_cast<int>(v.w)};
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        acc[h] = 0;
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[h] = __dp4a(q8r[h][i], w[i], acc[h]);
#pragma unroll
                        for (int o = kLanesPerRow / 2; o >= 1; o >>= 1)
                            acc[h] += __shfl_xor_sync(gmask, acc[h], o);
                    }
                    const float sk = a.k_scale[(static_cast<size_t>(p) * BS + t) * a.N + n];
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float dot = __fmul_rn(__fmul_rn(s_sq[h], sk), static_cast<float>(acc[h]));
                        best[h] = fmaxf(best[h], dot);
                    }
                } else {
                    float acc[G];
#pragma unroll
                    for (int h = 0; h < G; ++h) acc[h] = 0.f;
                    ProbeChunk<KT, G>::dot(qr, v, acc);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
#pragma unroll
                        for (int o = kLanesPerRow / 2; o >= 1; o >>= 1)
                            acc[h] += __shfl_xor_sync(gmask, acc[h], o);
                        best[h] = fmaxf(best[h], acc[h]);
                    }
                }
            }
        }
        if (cl == 0)
#pragma unroll
            for (int h = 0; h < G; ++h)
                a.probe[(static_cast<size_t>(b) * a.H + n * G + h) * a.MKBPR + j] = best[h];
    }

    if (n_chunks > 1) {
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
    } else {
        __syncthreads();
    }

    // selection for the G query heads of this KV head
    uint32_t* keys = reinterpret_cast<uint32_t*>(dyn);
    uint8_t* imp_flags = dyn + static_cast<size_t>(a.MKBPR) * 4;
    uint8_t* flags = imp_flags + a.MKBPR;
    int n_imp = 0;
    if (a.importance) {
        // summed prefill importance per block, fp32 in token order
        for (int j = threadIdx.x; j < nb; j += kThreads) {
            const int p0 = j * BS, p_end = min(p0 + BS, L);
            float s = 0.f;
            const float* imp = a.importance + static_cast<size_t>(b) * a.imp_stride;
            for (int ps = p0; ps < p_end; ++ps) s = __fadd_rn(s, imp[ps]);
            keys[j] = float_key(s);
            imp_flags[j] = kCand;
        }
        __syncthreads();
        n_imp = min((a.k + 1) / 2, nb);
        topk_flags<kThreads>(keys, imp_flags, nb, n_imp, s_topk);
        for (int j = threadIdx.x; j < nb; j += kThreads)
            imp_flags[j] = (imp_flags[j] & kPick) ? kFixed : 0;
    } else {
        for (int j = threadIdx.x; j < nb; j += kThreads) imp_flags[j] = 0;
    }
    __syncthreads();
    for (int h = 0; h < G; ++h) {
        const size_t row = static_cast<size_t>(b) * a.H + n * G + h;
        for (int j = threadIdx.x; j < nb; j += kThreads) {
            keys[j] = float_key(ldcg_f32(a.probe + row * a.MKBPR + j));
            flags[j] = imp_flags[j] ? kFixed : kCand;
        }
        __syncthreads();
        const int want = min(a.k - n_imp, nb - n_imp);
        topk_flags<kThreads>(keys, flags, nb, want, s_topk);
        // recency insurance
        if (want > 0 && !(flags[nb - 1] & (kFixed | kPick))) {
            if (threadIdx.x == 0) s_topk.best = ~0ull;
            __syncthreads();
            unsigned long long mine = ~0ull;
            for (int j = threadIdx.x; j < nb; j += kThreads)
                if (flags[j] & kPick) {
                    // smallest probe score first, then the larger index
                    const unsigned long long c =
                        (static_cast<unsigned long long>(keys[j]) << 32) | (0xffffffffu - static_cast<uint32_t>(j));
                    mine = c < mine ? c : mine;
                }
            atomicMin(&s_topk.best, mine);
            __syncthreads();
            if (threadIdx.x == 0) {
                const int victim = static_cast<int>(0xffffffffu - static_cast<uint32_t>(s_topk.best & 0xffffffffu));
                flags[victim] &= static_cast<uint8_t>(~kPick);
                flags[nb - 1] |= kPick;
            }
            __syncthreads();
        }
        emit_sorted<kThreads>(flags, kFixed | kPick, nb, a.k, a.selected + row * a.k, s_topk);
    }
}

template <Dt KT, int D, int G>
qs_status launch(const ProbeArgs& a, cudaStream_t s) {
    const size_t smem = align_up(static_cast<size_t>(a.MKBPR) * 6, 16);
    if (smem > 160 * 1024) return QS_EUNSUPPORTED;
    auto kern = probe_select_kernel<KT, D, G>;
    if (!ensure_smem(reinterpret_cast<const void*>(kern), smem))
        return QS_ECUDA;
    const int chunks = max(1, (a.MKBPR + kBlocksPerChunk - 1) / kBlocksPerChunk);
    dim3 grid(chunks, a.B * a.N);
    kern<<<grid, kThreads, smem, s>>>(a);
    QS_CHECK_LAUNCH();
    return QS_OK;
}

template <Dt KT, int D>
qs_status launch_g(const ProbeArgs& a, int G, cudaStream_t s) {
    switch (G) {
        case 1: return launch<KT, D, 1>(a, s);
        case 2: return launch<KT, D, 2>(a, s);
        case 4: return launch<KT, D, 4>(a, s);
        case 8: return launch<KT, D, 8>(a, s);
        default: return QS_EUNSUPPORTED;
    }
}

}  // namespace

size_t probe_workspace_bytes(int B, int H, int N, int MKBPR) {
    return align_up(static_cast<size_t>(B) * H * MKBPR * 4, 256) +
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
    a.counters = reinterpret_cast<uint32_t*>(ws + align_up(static_cast<size_t>(B) * H * MKBPR * 4, 256));
    a.dev_status = dev_status;
    switch (kv_dtype) {
        case QS_F32: return D == 128 ? launch_g<Dt::F32, 128>(a, G, stream) : launch_g<Dt::F32, 64>(a, G, stream);
        case QS_BF16: return D == 128 ? launch_g<Dt::BF16, 128>(a, G, stream) : launch_g<Dt::BF16, 64>(a, G, stream);
        case QS_F16: return D == 128 ? launch_g<Dt::F16, 128>(a, G, stream) : launch_g<Dt::F16, 64>(a, G, stream);
        case QS_I8: return launch_g<Dt::I8, 128>(a, G, stream);
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
