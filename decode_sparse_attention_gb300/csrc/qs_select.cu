// Quest block selection (CANN ops-transformer select_attention_operators page,
// section 'quest_block_select_paged: decode-time top-k prediction'):
//   step 1    group-mean query qg[b][n] over the H/N heads of group n
//   step 2.1  walk the request's metadata blocks through meta_block_tables
//   step 2.2  score s_j = sum_d max(qg_d*max_jd, qg_d*min_jd)
//   step 2.3  top-k over all blocks of the request
// plus the '_in_out_w' sink + window forcing driven by
// tokens_since_metadata_update.
//
// GB300 design: the scan of the metadata rows is the whole cost, so it is
// spread over many CTAs: grid = (row chunks, B*N units).  Each CTA scores one
// chunk of rows of one (request, KV head) with 128-bit streaming loads (a row
// of one head is D*elem bytes, read by D*elem/16 lanes; several rows in flight
// per lane) and writes fp32 scores to a buffer.  The last CTA of a unit to
// finish (atomic arrival counter, no spinning) runs the CTA-wide radix top-k
// and writes the selection.  The counter is reset by that CTA, so the
// workspace stays zeroed between calls.
#include "qs_common.cuh"
#include "qs_topk.cuh"

namespace qs {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerChunk = 64;
constexpr int kUnroll = 4;

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
    uint32_t* counters;   // [B*N]
    int32_t* dev_status;
};

// Partial score of one 16-byte chunk of a max row and a min row against the
// matching fp32 query channels.
template <Dt T> struct RowChunk;

template <> struct RowChunk<Dt::F32> {
    static constexpr int kElems = 4;
    static QS_DEVINL float dot(const float* qg, uint4 mx, uint4 mn) {
        const uint32_t a[4] = {mx.x, mx.y, mx.z, mx.w};
        const uint32_t c[4] = {mn.x, mn.y, mn.z, mn.w};
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float p1 = qg[i] * __uint_as_float(a[i]);
            const float p2 = qg[i] * __uint_as_float(c[i]);
            s += fmaxf(p1, p2);
        }
        return s;
    }
};

template <Dt T> struct RowChunk16 {
    static constexpr int kElems = 8;
    static QS_DEVINL float dot(const float* qg, uint4 mx, uint4 mn) {
        const uint32_t a[4] = {mx.x, mx.y, mx.z, mx.w};
        const uint32_t c[4] = {mn.x, mn.y, mn.z, mn.w};
        unsigned long long acc = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 fa = pair_to_float2<T>(a[i]);
            const float2 fc = pair_to_float2<T>(c[i]);
            const unsigned long long q2 = pack2(qg[2 * i], qg[2 * i + 1]);
            const float2 p1 = unpack2(mul2(q2, pack2(fa.x, fa.y)));
            const float2 p2 = unpack2(mul2(q2, pack2(fc.x, fc.y)));
            const float2 m = make_float2(fmaxf(p1.x, p2.x), fmaxf(p1.y, p2.y));
            acc = fma2(pack2(1.f, 1.f), pack2(m.x, m.y), acc);
        }
        const float2 r = unpack2(acc);
        return r.x + r.y;
    }
};
template <> struct RowChunk<Dt::BF16> : RowChunk16<Dt::BF16> {};
template <> struct RowChunk<Dt::F16> : RowChunk16<Dt::F16> {};

template <Dt MT, int D>
__global__ void __launch_bounds__(kThreads) quest_select_kernel(SelectArgs a) {
    constexpr int kElemBytes = DtInfo<MT>::bytes;
    constexpr int kLanesPerRow = D * kElemBytes / 16;   // 8, 16 or 32
    constexpr int kRowsPerWarp = 32 / kLanesPerRow;
    constexpr int kEl = RowChunk<MT>::kElems;
    static_assert(kLanesPerRow >= 1 && kLanesPerRow <= 32, "row must span 1..32 lanes");

    extern __shared__ __align__(16) uint8_t dyn[];
    __shared__ float s_qg[D];
    __shared__ TopkScratch<kThreads> s_topk;
    __shared__ int s_last;

    pdl_launch_dependents();

    const int u = blockIdx.y;
    const int b = u / a.N, n = u % a.N;
    const int BS = a.BS;
    const int maxnb = a.MMBPR * BS;
    const int L = a.seq_lens[b];
    int32_t* sel_out = a.selected + static_cast<size_t>(u) * a.k;
    if (L < 0 || (L + BS - 1) / BS > maxnb) {
        if (blockIdx.x == 0) {
            if (threadIdx.x == 0) set_status(a.dev_status, QS_DEV_ESEQ_LEN);
            for (int i = threadIdx.x; i < a.k; i += kThreads) sel_out[i] = -1;
        }
        return;
    }
    const int nb = (L + BS - 1) / BS;
    const int n_chunks = max(1, (nb + kRowsPerChunk - 1) / kRowsPerChunk);
    if (static_cast<int>(blockIdx.x) >= n_chunks) return;

    // step 1: group-mean query of KV head n
    const int G = a.H / a.N;
    for (int d = threadIdx.x; d < D; d += kThreads) {
        float s = 0.f;
        for (int g = 0; g < G; ++g)
            s += load_q(a.q, a.q_dt, (static_cast<size_t>(b) * a.H + n * G + g) * D + d);
        s_qg[d] = s / static_cast<float>(G);
    }
    __syncthreads();

    // steps 2.1-2.2: score this chunk's rows
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane / kLanesPerRow;          // row slot within the warp
    const int cl = lane % kLanesPerRow;           // 16-byte chunk within the row
    float qreg[kEl];
#pragma unroll
    for (int i = 0; i < kEl; ++i) qreg[i] = s_qg[cl * kEl + i];
    const size_t head_off = static_cast<size_t>(n) * D * kElemBytes + static_cast<size_t>(cl) * 16;
    const size_t row_stride = static_cast<size_t>(a.N) * D * kElemBytes;
    const int j_begin = blockIdx.x * kRowsPerChunk;
    const int j_end = min(nb, j_begin + kRowsPerChunk);
    constexpr int kRowsPerStep = (kThreads / 32) * kRowsPerWarp * kUnroll;
    float* scores_u = a.scores + static_cast<size_t>(u) * maxnb;
    for (int j0 = j_begin; j0 < j_end; j0 += kRowsPerStep) {
        uint4 vmx[kUnroll], vmn[kUnroll];
        bool live[kUnroll];
#pragma unroll
        for (int r = 0; r < kUnroll; ++r) {
            const int j = j0 + (r * (kThreads / 32) + warp) * kRowsPerWarp + sub;
            live[r] = j < j_end;
            vmx[r] = vmn[r] = make_uint4(0, 0, 0, 0);
            if (live[r]) {
                const int m = a.mbt[static_cast<size_t>(b) * a.MMBPR + j / BS];
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
            const int j = j0 + (r * (kThreads / 32) + warp) * kRowsPerWarp + sub;
            float s = RowChunk<MT>::dot(qreg, vmx[r], vmn[r]);
#pragma unroll
            for (int o = kLanesPerRow / 2; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (cl == 0 && j < j_end) scores_u[j] = live[r] ? s : __int_as_float(0xff800000);
        }
    }

    // arrival: the last chunk of the unit selects
    if (n_chunks > 1) {
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
    } else {
        __syncthreads();
    }

    // step 2.3 + window: keys and flags in shared memory
    uint32_t* keys = reinterpret_cast<uint32_t*>(dyn);
    uint8_t* flags = dyn + static_cast<size_t>(maxnb) * 4;
    int w0 = nb;  // first window block (nb: none)
    if (a.t >= 0 && nb > 0) {
        w0 = L - a.t >= 0 ? (L - a.t) / BS : 0;
        w0 = min(w0, nb - 1);
    }
    for (int j = threadIdx.x; j < nb; j += kThreads) {
        keys[j] = float_key(ldcg_f32(scores_u + j));
        const bool forced = a.t >= 0 && (j == 0 || j >= w0);
        flags[j] = forced ? kFixed : kCand;
    }
    __syncthreads();
    const int n_forced = a.t >= 0 && nb > 0 ? (nb - w0) + (w0 > 0 ? 1 : 0) : 0;
    if (n_forced > a.k) {
        if (threadIdx.x == 0) set_status(a.dev_status, QS_DEV_EFORCED);
        for (int i = threadIdx.x; i < a.k; i += kThreads) sel_out[i] = -1;
        return;
    }
    const int want = min(a.k - n_forced, nb - n_forced);
    topk_flags<kThreads>(keys, flags, nb, want, s_topk);
    emit_sorted<kThreads>(flags, kFixed | kPick, nb, a.k, sel_out, s_topk);
}

template <Dt MT, int D>
qs_status launch(const SelectArgs& a, cudaStream_t s) {
    const int maxnb = a.MMBPR * a.BS;
    const size_t smem = align_up(static_cast<size_t>(maxnb) * 5, 16);
    if (smem > 200 * 1024) return QS_EUNSUPPORTED;
    auto kern = quest_select_kernel<MT, D>;
    if (!ensure_smem(reinterpret_cast<const void*>(kern), smem))
        return QS_ECUDA;
    const int chunks = max(1, (maxnb + kRowsPerChunk - 1) / kRowsPerChunk);
    dim3 grid(chunks, a.B * a.N);
    kern<<<grid, kThreads, smem, s>>>(a);
    QS_CHECK_LAUNCH();
    return QS_OK;
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
    if ((reinterpret_cast<uintptr_t>(maxblocks) | reinterpret_cast<uintptr_t>(minblocks)) % 16)
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
