// Quest block selection (CANN ops-transformer select_attention_operators page,
// section 'quest_block_select_paged: decode-time top-k prediction'):
//   step 1    group-mean query qg[b][n] over the H/N heads of group n
//   step 2.1  walk the request's metadata blocks through meta_block_tables
//   step 2.2  score s_j = sum_d max(qg_d*max_jd, qg_d*min_jd)
//   step 2.3  top-k over all blocks of the request
// plus the '_in_out_w' sink + window forcing driven by
// tokens_since_metadata_update.
//
// GB300 design: the scan of the metadata rows is the whole cost, so each
// (request, KV head) is split into row chunks of one load step each: every
// lane keeps 8 rows of max/min in flight with 128-bit streaming loads and
// computes the group-mean query of its own 16-byte slice of D.  A unit of
// one chunk scores into shared memory; a unit of 2..8 chunks runs as one
// thread-block cluster whose CTAs write their scores straight into the
// leader CTA's shared memory (distributed shared memory) before a cluster
// barrier; larger units fall back to a global score buffer and an arrival
// counter.  The leader then selects with a histogram top-k (one 1024-bin
// pass, exact ranking inside the boundary bin) and one warp writes the
// indices in ascending order.
#include <cooperative_groups.h>

#include "qs_internal.cuh"
#include "qs_quest_score.cuh"
#include "qs_topk.cuh"

namespace qs {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;     // rows in flight per lane: a chunk loads in one step
constexpr int kMaxG = 8;       // query heads per KV head

// Rows of one chunk: every lane group keeps kUnroll rows in flight.
template <Dt MT, int D> constexpr int rows_per_chunk() {
    return (kThreads / 32) * (32 / (D * DtInfo<MT>::bytes / 16)) * kUnroll;
}

struct SelectArgs {
    const void* q;
    int q_dt;
    const uint8_t* maxb;
    const uint8_t* minb;
    const int32_t* mbt;
    int MMBPR, num_meta;
    const int32_t* seq_lens;
    int B, H, N, BS, k, t;
    int32_t* selected;
    float* scores;        // [B*N, maxnb]
    bool scores_out;      // the caller asked for the scores
    uint32_t* counters;   // [B*N]
    int32_t* dev_status;
};

enum Mode : int { kSingle = 0, kCluster = 1, kGlobal = 2 };

template <Dt MT, int D, int MODE>
__global__ void __launch_bounds__(kThreads, 2) quest_select_kernel(SelectArgs a) {
    constexpr int kElemBytes = DtInfo<MT>::bytes;
    constexpr int kLanesPerRow = D * kElemBytes / 16;   // 8, 16 or 32
    constexpr int kRowsPerWarp = 32 / kLanesPerRow;
    constexpr int kEl = RowChunk<MT>::kElems;
    constexpr int kRowsPerChunk = rows_per_chunk<MT, D>();
    static_assert(kLanesPerRow >= 1 && kLanesPerRow <= 32, "row must span 1..32 lanes");

    extern __shared__ __align__(16) uint8_t dyn[];   // keys [maxnb] u32, flags [maxnb] u8
    __shared__ TopkFastScratch s_fast;
    __shared__ TopkScratch<kThreads> s_topk;
    __shared__ int s_last;

    pdl_launch_dependents();

    const int u = blockIdx.y;
    const int b = u / a.N, n = u % a.N;
    const int BS = a.BS;
    const int maxnb = a.MMBPR * BS;
    const int L = a.seq_lens[b];
    int32_t* sel_out = a.selected + static_cast<size_t>(u) * a.k;
    if (L < 0 || (L + BS - 1) / BS > maxnb) {   // uniform over the unit's CTAs
        if (blockIdx.x == 0) {
            if (threadIdx.x == 0) set_status(a.dev_status, QS_DEV_ESEQ_LEN);
            for (int i = threadIdx.x; i < a.k; i += kThreads) sel_out[i] = -1;
        }
        return;
    }
    const int nb = (L + BS - 1) / BS;
    const int n_chunks = max(1, (nb + kRowsPerChunk - 1) / kRowsPerChunk);
    if (MODE != kCluster && static_cast<int>(blockIdx.x) >= n_chunks) return;
    uint32_t* keys = reinterpret_cast<uint32_t*>(dyn);
    uint8_t* flags = dyn + static_cast<size_t>(maxnb) * 4;
    topk_fast_clear<kThreads>(s_fast);

    // steps 1, 2.1, 2.2
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane / kLanesPerRow;          // row slot within the warp
    const int cl = lane % kLanesPerRow;           // 16-byte chunk within the row
    const int G = a.H / a.N;
    const size_t head_off = static_cast<size_t>(n) * D * kElemBytes + static_cast<size_t>(cl) * 16;
    const size_t row_stride = static_cast<size_t>(a.N) * D * kElemBytes;
    const int j_begin = blockIdx.x * kRowsPerChunk;
    const int j_end = min(nb, j_begin + kRowsPerChunk);
    float* scores_u = a.scores + static_cast<size_t>(u) * maxnb;
    uint32_t* dst_keys = keys;
    if constexpr (MODE == kCluster)
        dst_keys = cooperative_groups::this_cluster().map_shared_rank(keys, 0);
    // Table entries and the G heads' query slices are all requested before
    // either is used (in-order issue would otherwise serialise the round
    // trips); the metadata rows follow once the table entries are back.
    int mrow[kUnroll];
#pragma unroll
    for (int r = 0; r < kUnroll; ++r) {
        const int j = j_begin + (r * (kThreads / 32) + warp) * kRowsPerWarp + sub;
        mrow[r] = j < j_end ? a.mbt[static_cast<size_t>(b) * a.MMBPR + j / BS] : -1;
    }
    constexpr int kQBytes = kEl * 4;                 // fp32 query slice; 16-bit uses half
    constexpr int kQVec = (kQBytes + 15) / 16;       // 16-byte loads per head slice
    uint4 qraw[kMaxG][kQVec];
    const int q_es = a.q_dt == QS_F32 ? 4 : 2;
    const uint8_t* qbase = static_cast<const uint8_t*>(a.q) +
                           ((static_cast<size_t>(b) * a.H + static_cast<size_t>(n) * G) * D + cl * kEl) * q_es;
#pragma unroll
    for (int g = 0; g < kMaxG; ++g)
#pragma unroll
        for (int v = 0; v < kQVec; ++v) {
            qraw[g][v] = make_uint4(0, 0, 0, 0);
            if (g < G && v * 16 < kEl * q_es) {
                const uint8_t* p = qbase + static_cast<size_t>(g) * D * q_es + v * 16;
                if (kEl * q_es >= 16) qraw[g][v] = *reinterpret_cast<const uint4*>(p);
                else {
                    const uint2 h = *reinterpret_cast<const uint2*>(p);
                    qraw[g][v] = make_uint4(h.x, h.y, 0, 0);
                }
            }
        }
    // group-mean query of this lane's slice
    float qreg[kEl];
    {
        float acc[kEl];
#pragma unroll
        for (int e = 0; e < kEl; ++e) acc[e] = 0.f;
#pragma unroll
        for (int g = 0; g < kMaxG; ++g) {
            if (g >= G) break;
            const uint32_t* w = reinterpret_cast<const uint32_t*>(&qraw[g][0]);
            if (a.q_dt == QS_F32) {
#pragma unroll
                for (int e = 0; e < kEl; ++e) acc[e] += __uint_as_float(w[e]);
            } else {
#pragma unroll
                for (int e = 0; e < kEl / 2; ++e) {
                    const float2 f = a.q_dt == QS_BF16 ? pair_to_float2<Dt::BF16>(w[e])
                                                       : pair_to_float2<Dt::F16>(w[e]);
                    acc[2 * e] += f.x;
                    acc[2 * e + 1] += f.y;
                }
            }
        }
#pragma unroll
        for (int e = 0; e < kEl; ++e) qreg[e] = acc[e] / static_cast<float>(G);
    }
    uint4 vmx[kUnroll], vmn[kUnroll];
    bool live[kUnroll];
#pragma unroll
    for (int r = 0; r < kUnroll; ++r) {
        const int j = j_begin + (r * (kThreads / 32) + warp) * kRowsPerWarp + sub;
        const int m = mrow[r];
        live[r] = j < j_end;
        vmx[r] = vmn[r] = make_uint4(0, 0, 0, 0);
        if (live[r]) {
            if (m < 0 || m >= a.num_meta) {
                set_status(a.dev_status, QS_DEV_EMETA_TABLE);
                live[r] = false;
            } else {
                const size_t off = (static_cast<size_t>(m) * BS + j % BS) * row_stride + head_off;
                vmx[r] = ldg_stream(a.maxb + off);
                vmn[r] = ldg_stream(a.minb + off);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kUnroll; ++r) {
        const int j = j_begin + (r * (kThreads / 32) + warp) * kRowsPerWarp + sub;
        const float s = row_score_reduce<kLanesPerRow>(RowChunk<MT>::dot(qreg, vmx[r], vmn[r]));
        if (cl == 0 && j < j_end) {
            const float v = live[r] ? s : __int_as_float(0xff800000);
            if (MODE != kGlobal) dst_keys[j] = float_key(v);
            if (MODE == kGlobal || a.scores_out) scores_u[j] = v;
        }
    }

    // all scores of the unit in the leader's shared memory
    if constexpr (MODE == kCluster) {
        cooperative_groups::this_cluster().sync();
        if (blockIdx.x != 0) return;
    } else if constexpr (MODE == kGlobal) {
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const uint32_t prev = atomicAdd(&a.counters[u], 1u);
            s_last = prev == static_cast<uint32_t>(n_chunks - 1);
            if (s_last) a.counters[u] = 0;  // every chunk has arrived: rearm
        }
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        for (int j = threadIdx.x; j < nb; j += kThreads) keys[j] = float_key(ldcg_f32(scores_u + j));
    }

    // step 2.3 + window
    const int w0 = forced_window_start(L, BS, nb, a.t);   // nb: no window
    const int n_forced = forced_count(nb, w0, a.t);
    if (n_forced > a.k) {
        if (threadIdx.x == 0) set_status(a.dev_status, QS_DEV_EFORCED);
        for (int i = threadIdx.x; i < a.k; i += kThreads) sel_out[i] = -1;
        return;
    }
    for (int j = threadIdx.x; j < nb; j += kThreads)
        flags[j] = (a.t >= 0 && (j == 0 || j >= w0)) ? kFixed : kCand;
    __syncthreads();
    const int want = min(a.k - n_forced, nb - n_forced);
    topk_fast<kThreads>(keys, flags, nb, want, s_fast, s_topk);
    if (warp == 0) warp_emit_flags(flags, kFixed | kPick, nb, a.k, sel_out);
}

template <Dt MT, int D, int MODE>
qs_status launch_mode(const SelectArgs& a, int chunks, size_t smem, cudaStream_t s) {
    auto kern = quest_select_kernel<MT, D, MODE>;
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

template <Dt MT, int D>
qs_status launch(const SelectArgs& a, cudaStream_t s) {
    const int maxnb = a.MMBPR * a.BS;
    const size_t smem = align_up(static_cast<size_t>(maxnb) * 5, 16);
    if (smem > 160 * 1024) return QS_EUNSUPPORTED;
    constexpr int kRowsPerChunk = rows_per_chunk<MT, D>();
    const int chunks = max(1, (maxnb + kRowsPerChunk - 1) / kRowsPerChunk);
    if (chunks == 1) return launch_mode<MT, D, kSingle>(a, chunks, smem, s);
    if (chunks <= 8) return launch_mode<MT, D, kCluster>(a, chunks, smem, s);
    return launch_mode<MT, D, kGlobal>(a, chunks, smem, s);
}

}  // namespace

size_t select_workspace_bytes(int B, int N, int maxnb) {
    return align_up(static_cast<size_t>(B) * N * maxnb * 4, 256) +
           align_up(static_cast<size_t>(B) * N * 4, 256);
}

qs_status block_select_impl(const void* q, qs_dtype q_dtype, const void* maxblocks,
                            const void* minblocks, qs_dtype meta_dtype,
                            const int32_t* meta_block_tables, int32_t MMBPR,
                            int32_t num_meta_blocks, const int32_t* seq_lens, int32_t B,
                            int32_t H, int32_t N, int32_t D, int32_t BS, int32_t k, int32_t t,
                            int32_t* selected, float* scores_opt, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream) {
    if (B < 0 || H <= 0 || N <= 0 || H % N != 0 || BS <= 0 || k <= 0 || MMBPR < 0 ||
        num_meta_blocks < 0)
        return QS_EINVAL;
    if (B == 0) return QS_OK;
    if (!q || !maxblocks || !minblocks || !meta_block_tables || !seq_lens || !selected ||
        !dev_status)
        return QS_EINVAL;
    if (q_dtype != QS_F32 && q_dtype != QS_BF16 && q_dtype != QS_F16) return QS_EDTYPE;
    if (meta_dtype != QS_F32 && meta_dtype != QS_BF16 && meta_dtype != QS_F16) return QS_EDTYPE;
    if (D != 64 && D != 128) return QS_EUNSUPPORTED;
    if (H / N > kMaxG) return QS_EUNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(maxblocks) | reinterpret_cast<uintptr_t>(minblocks) |
         reinterpret_cast<uintptr_t>(q)) % 16)
        return QS_EINVAL;
    if (t >= 0 && static_cast<long long>(k) < 2 + (static_cast<long long>(t) + BS - 1) / BS)
        return QS_EINVAL;  // the forced set may not fit
    const long long maxnb_ll = static_cast<long long>(MMBPR) * BS;
    if (maxnb_ll > (1 << 24)) return QS_EUNSUPPORTED;
    const int maxnb = static_cast<int>(maxnb_ll);
    const size_t need = select_workspace_bytes(B, N, maxnb);
    if (!workspace || workspace_bytes < need) return QS_EWORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    SelectArgs a;
    a.q = q;
    a.q_dt = q_dtype;
    a.maxb = static_cast<const uint8_t*>(maxblocks);
    a.minb = static_cast<const uint8_t*>(minblocks);
    a.mbt = meta_block_tables;
    a.MMBPR = MMBPR;
    a.num_meta = num_meta_blocks;
    a.seq_lens = seq_lens;
    a.B = B; a.H = H; a.N = N; a.BS = BS; a.k = k; a.t = t;
    a.selected = selected;
    a.scores = scores_opt ? scores_opt : reinterpret_cast<float*>(ws);
    a.scores_out = scores_opt != nullptr;
    a.counters = reinterpret_cast<uint32_t*>(ws + align_up(static_cast<size_t>(B) * N * maxnb * 4, 256));
    a.dev_status = dev_status;
    if (D == 128) {
        switch (meta_dtype) {
            case QS_F32: return launch<Dt::F32, 128>(a, stream);
            case QS_BF16: return launch<Dt::BF16, 128>(a, stream);
            default: return launch<Dt::F16, 128>(a, stream);
        }
    }
    switch (meta_dtype) {
        case QS_F32: return launch<Dt::F32, 64>(a, stream);
        case QS_BF16: return launch<Dt::BF16, 64>(a, stream);
        default: return launch<Dt::F16, 64>(a, stream);
    }
}

}  // namespace qs

extern "C" qs_status qs_block_select_paged(const void* q, qs_dtype q_dtype, const void* maxblocks,
                                           const void* minblocks, qs_dtype meta_dtype,
                                           const int32_t* meta_block_tables, int32_t MMBPR,
                                           int32_t num_meta_blocks, const int32_t* seq_lens,
                                           int32_t B, int32_t H, int32_t N, int32_t D,
                                           int32_t BS, int32_t k,
                                           int32_t tokens_since_metadata_update,
                                           int32_t* selected, float* scores_opt, void* workspace,
                                           size_t workspace_bytes, int32_t* dev_status,
                                           qs_stream_t stream) {
    return qs::block_select_impl(q, q_dtype, maxblocks, minblocks, meta_dtype, meta_block_tables,
                                 MMBPR, num_meta_blocks, seq_lens, B, H, N, D, BS, k,
                                 tokens_since_metadata_update, selected, scores_opt, workspace,
                                 workspace_bytes, dev_status,
                                 reinterpret_cast<cudaStream_t>(stream));
}
