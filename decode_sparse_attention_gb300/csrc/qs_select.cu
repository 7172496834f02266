// Quest block selection (CANN ops-transformer select_attention_operators page,
// section 'quest_block_select_paged: decode-time top-k prediction'):
//   step 1    group-mean query qg[b][n] over the H/N heads of group n
//   step 2.1  walk the request's metadata blocks through meta_block_tables
//   step 2.2  score s_j = sum_d max(qg_d*max_jd, qg_d*min_jd)
//   step 2.3  top-k over all blocks of the request
// plus the '_in_out_w' sink + window forcing driven by
// tokens_since_metadata_update.
//
// GB300 design: the scan of the metadata rows is the whole cost.
//  * Units of one chunk (short requests: all rows fit one load step, every
//    lane keeping 8 rows of max/min in flight with 128-bit streaming loads):
//    one CTA per unit scores into shared memory and selects.
//  * Longer units: a persistent scan kernel, one CTA per SM, walks a static
//    stride of 64 KB chunks (32 KB of max rows + 32 KB of min rows of one
//    (request, KV head)), with the requests' lengths and the metadata table
//    staged in shared memory up front so that a chunk's cp.async copies are
//    issued without a global round trip, and a three-stage ring keeping two
//    chunks in flight while one is scored.  Scores go to a global buffer.
//    A second kernel, a programmatic dependent of the scan, selects one unit
//    per CTA from those scores.
// Selection: histogram top-k (key descending, ties to the lower index), then
// the block writes the indices in ascending order.
#include <algorithm>

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

// Metadata block of row j, and j's row inside it.
#define QS_META_BLOCK(a, j) ((a).bs_shift >= 0 ? (j) >> (a).bs_shift : (j) / (a).BS)
#define QS_META_ROW(a, j) ((a).bs_shift >= 0 ? (j) & ((a).BS - 1) : (j) % (a).BS)

struct SelectArgs {
    const void* q;
    int q_dt;
    const uint8_t* maxb;
    const uint8_t* minb;
    const int32_t* mbt;
    int MMBPR, num_meta;
    const int32_t* seq_lens;
    int B, H, N, BS, k, t;
    int bs_shift;         // log2(BS) when BS is a power of two, else -1
    int32_t* selected;
    float* scores;        // [B*N, maxnb]
    bool scores_out;      // the caller asked for the scores
    int32_t* dev_status;
};

// Scores every row of unit (b, n), whose rows fit one chunk (steps 1, 2.1,
// 2.2).  Keys go to keys_s (shared, indexed by row); scores to scores_u
// (global, indexed by row) when given.  The request's length, the table
// entries of every row the unit may have and the query slices are requested
// together, in one round trip, before the length is used; returns false
// (uniformly) for a length out of range, else the block count in *nb_out and
// the length in *L_out.
template <Dt MT, int D>
QS_DEVINL bool score_unit(const SelectArgs& a, int b, int n, uint32_t* keys_s, float* scores_u,
                          int* nb_out, int* L_out) {
    constexpr int kElemBytes = DtInfo<MT>::bytes;
    constexpr int kLanesPerRow = D * kElemBytes / 16;   // 8, 16 or 32
    constexpr int kRowsPerWarp = 32 / kLanesPerRow;
    constexpr int kEl = RowChunk<MT>::kElems;
    static_assert(kLanesPerRow >= 1 && kLanesPerRow <= 32, "row must span 1..32 lanes");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane / kLanesPerRow;          // row slot within the warp
    const int cl = lane % kLanesPerRow;           // 16-byte chunk within the row
    const int G = a.H / a.N;
    const int BS = a.BS;
    const size_t head_off = static_cast<size_t>(n) * D * kElemBytes + static_cast<size_t>(cl) * 16;
    const size_t row_stride = static_cast<size_t>(a.N) * D * kElemBytes;
    const int maxnb = a.MMBPR * BS;
    const int L = ldg_now_s32(a.seq_lens + b);
    int mrow[kUnroll];
#pragma unroll
    for (int r = 0; r < kUnroll; ++r) {
        const int j = (r * (kThreads / 32) + warp) * kRowsPerWarp + sub;
        mrow[r] = j < maxnb ? ldg_now_s32(a.mbt + static_cast<size_t>(b) * a.MMBPR + QS_META_BLOCK(a, j)) : -1;
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
                if (kEl * q_es >= 16) qraw[g][v] = ldg_now_v4(p);
                else {
                    const uint2 h = ldg_now_v2(p);
                    qraw[g][v] = make_uint4(h.x, h.y, 0, 0);
                }
            }
        }
    if (L < 0 || (L + BS - 1) / BS > maxnb) return false;
    const int nb = (L + BS - 1) / BS;
    *nb_out = nb;
    *L_out = L;
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
        for (int e = 0; e < kEl; ++e) qreg[e] = group_mean(acc[e], G);
    }
    RowChunk<MT> rc;
    rc.prepare(qreg);
    uint4 vmx[kUnroll], vmn[kUnroll];
    bool live[kUnroll];
#pragma unroll
    for (int r = 0; r < kUnroll; ++r) {
        const int j = (r * (kThreads / 32) + warp) * kRowsPerWarp + sub;
        const int m = mrow[r];
        live[r] = j < nb;
        vmx[r] = vmn[r] = make_uint4(0, 0, 0, 0);
        if (live[r]) {
            if (m < 0 || m >= a.num_meta) {
                set_status(a.dev_status, QS_DEV_EMETA_TABLE);
                live[r] = false;
            } else {
                const size_t off = (static_cast<size_t>(m) * BS + QS_META_ROW(a, j)) * row_stride + head_off;
                vmx[r] = ldg_stream(a.maxb + off);
                vmn[r] = ldg_stream(a.minb + off);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kUnroll; ++r) {
        const int j = (r * (kThreads / 32) + warp) * kRowsPerWarp + sub;
        const float s = row_score_reduce<kLanesPerRow>(rc.dot(vmx[r], vmn[r]));
        if (cl == 0 && j < nb) {
            const float v = live[r] ? s : __int_as_float(0xff800000);
            keys_s[j] = float_key(v);
            if (scores_u) scores_u[j] = v;
        }
    }
    return true;
}

// Forced set, top-k and emission of one unit whose nb keys are in keys_s
// (step 2.3 + window).  All threads; ends with a barrier.
// kRankPath: units of up to kRankMaxPerThread keys per thread select with the
// counting top-k over all threads (the forced blocks' keys, and the padding
// up to a multiple of 4 entries, are zeroed so that they leave the
// candidates); larger units, and the top-k kernel after the scan, use the
// histogram levels.  keys_s holds round_up(nb, 4) writable words.
template <bool kRankPath>
QS_DEVINL void select_unit(const SelectArgs& a, int L, int nb, uint32_t* keys_s,
                           uint8_t* flags, int32_t* sel_out, TopkFastScratch& s_fast,
                           TopkScratch<kThreads>& s_topk) {
    const int w0 = forced_window_start(L, a.BS, nb, a.t);   // nb: no window
    const int n_forced = forced_count(nb, w0, a.t);
    if (n_forced > a.k) {
        if (threadIdx.x == 0) set_status(a.dev_status, QS_DEV_EFORCED);
        for (int i = threadIdx.x; i < a.k; i += kThreads) sel_out[i] = -1;
        __syncthreads();
        return;
    }
    const bool small = kRankPath && nb <= kThreads * kRankMaxPerThread;
    if (!small) topk_fast_clear<kThreads>(s_fast, nb);
    for (int j = threadIdx.x; j < nb; j += kThreads) {
        const bool forced = a.t >= 0 && (j == 0 || j >= w0);
        flags[j] = forced ? kFixed : kCand;
        if (small && forced) keys_s[j] = 0u;
    }
    if (small && static_cast<int>(threadIdx.x) < ((nb + 3) & ~3) - nb) keys_s[nb + threadIdx.x] = 0u;
    __syncthreads();
    const int want = min(a.k - n_forced, nb - n_forced);
    if (small) {
        block_rank_topk<kThreads>(keys_s, 0, flags, 0, nb, 1, want);
        __syncthreads();
        if (threadIdx.x < 32) warp_emit_flags(flags, kFixed | kPick, nb, a.k, sel_out);
    } else {
        topk_fast<kThreads>(keys_s, flags, nb, want, s_fast, s_topk);
        block_emit_flags<kThreads>(flags, kFixed | kPick, nb, a.k, sel_out, s_topk);
    }
    __syncthreads();
}

// One CTA per unit; the unit's rows fit one chunk.
template <Dt MT, int D>
__global__ void __launch_bounds__(kThreads, 2) quest_select_unit_kernel(SelectArgs a) {
    extern __shared__ __align__(16) uint8_t dyn[];   // keys [maxnb] u32, flags [maxnb] u8
    __shared__ TopkFastScratch s_fast;
    __shared__ TopkScratch<kThreads> s_topk;
    pdl_launch_dependents();
    const int u = blockIdx.x;
    const int b = u / a.N, n = u % a.N;
    const int maxnb = a.MMBPR * a.BS;
    int32_t* sel_out = a.selected + static_cast<size_t>(u) * a.k;
    uint32_t* keys = reinterpret_cast<uint32_t*>(dyn);
    uint8_t* flags = dyn + ((static_cast<size_t>(maxnb) + 3) & ~static_cast<size_t>(3)) * 4;
    int nb = 0, L = 0;
    if (!score_unit<MT, D>(a, b, n, keys, a.scores_out ? a.scores + static_cast<size_t>(u) * maxnb : nullptr,
                           &nb, &L)) {
        if (threadIdx.x == 0) set_status(a.dev_status, QS_DEV_ESEQ_LEN);
        for (int i = threadIdx.x; i < a.k; i += kThreads) sel_out[i] = -1;
        return;
    }
    __syncthreads();
    select_unit<true>(a, L, nb, keys, flags, sel_out, s_fast, s_topk);
}

// ---- units longer than one chunk: a streaming scan, then one top-k per unit

constexpr int kScanThreads = 512;
constexpr int kRowsPerLane = 4;    // consecutive rows a lane group scores per chunk

// Rows of one scan chunk: every lane group of kLPR lanes scores kRowsPerLane
// consecutive rows (32 KB of max rows and 32 KB of min rows at 16-bit D=128).
template <Dt MT, int D> constexpr int scan_rows() {
    return kScanThreads / (D * DtInfo<MT>::bytes / 16) * kRowsPerLane;
}

// Transposing sum over the kLPR lanes of a row group of four per-lane row
// partials: afterwards the lowest lane of each kLPR/4-lane quarter holds the
// total of row (bit kLPR/2 of the lane ? 2 : 0) + (bit kLPR/4 ? 1 : 0).
template <int kLPR>
QS_DEVINL float reduce_rows4(const float (&v)[4], int cl) {
    static_assert(kLPR >= 8, "four rows need at least 8 lanes per row");
    const bool h1 = cl & (kLPR / 2);
    float a0 = h1 ? v[2] : v[0], a1 = h1 ? v[3] : v[1];
    const float s0 = h1 ? v[0] : v[2], s1 = h1 ? v[1] : v[3];
    a0 += __shfl_xor_sync(0xffffffffu, s0, kLPR / 2);
    a1 += __shfl_xor_sync(0xffffffffu, s1, kLPR / 2);
    const bool h2 = cl & (kLPR / 4);
    float k = h2 ? a1 : a0;
    k += __shfl_xor_sync(0xffffffffu, h2 ? a0 : a1, kLPR / 4);
#pragma unroll
    for (int o = kLPR / 8; o >= 1; o >>= 1) k += __shfl_xor_sync(0xffffffffu, k, o);
    return k;
}

struct ScanLayout {
    uint32_t off_cpre, off_lens, off_mbt, off_q, qslot_bytes;
    bool mbt_in_smem;
};

QS_DEVINL void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
QS_DEVINL void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// All of this thread's copy groups but the most recent one have landed.
QS_DEVINL void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Persistent scan: CTA c scores chunks c, c + grid, c + 2 grid, ...  The
// requests' lengths, the chunk prefix over requests and (when it fits) the
// whole metadata table are staged in shared memory first.  Each lane group
// of kLPR lanes loads kRowsPerLane consecutive rows of max and min (one
// metadata block: BS is a multiple of 16) straight into registers, one chunk
// ahead of the one it scores, together with the query slices of the next
// chunk; every row's score goes to the global score buffer.
template <Dt MT, int D>
__global__ void __launch_bounds__(kScanThreads, 1) quest_scan_kernel(SelectArgs a, ScanLayout l) {
    constexpr int kElemBytes = DtInfo<MT>::bytes;
    constexpr int kLPR = D * kElemBytes / 16;          // 16-byte slices per row
    constexpr int kGroups = 32 / kLPR;                 // lane groups per warp
    constexpr int kRows = scan_rows<MT, D>();
    constexpr int kEl = RowChunk<MT>::kElems;
    static_assert(kLPR >= 8 && kLPR <= 32 && 32 % kLPR == 0, "row must tile a warp");
    extern __shared__ __align__(16) uint8_t dyn[];
    __shared__ TopkScratch<kScanThreads> s_scan;
    pdl_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = a.B, N = a.N, BS = a.BS, G = a.H / a.N;
    const int maxnb = a.MMBPR * BS;
    int* cpre = reinterpret_cast<int*>(dyn + l.off_cpre);
    int* lens = reinterpret_cast<int*>(dyn + l.off_lens);
    int* mbt_s = reinterpret_cast<int*>(dyn + l.off_mbt);

    // lengths and chunks per unit of each request (0 for an empty request or
    // one out of range: the top-k kernel handles those without scores)
    {
        const int per = (B + kScanThreads - 1) / kScanThreads;
        const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
        int sum = 0;
        for (int b = b0; b < b1; ++b) {
            const int L = a.seq_lens[b];
            lens[b] = L;
            const int nb = L < 0 ? -1 : (L + BS - 1) / BS;
            sum += (nb <= 0 || nb > maxnb) ? 0 : (nb + kRows - 1) / kRows * N;
        }
        if (l.mbt_in_smem)
            for (int e = tid; e < B * a.MMBPR; e += kScanThreads) mbt_s[e] = a.mbt[e];
        int total;
        int before = block_exclusive_scan<kScanThreads>(sum, s_scan, &total);
        for (int b = b0; b < b1; ++b) {
            cpre[b] = before;
            const int L = lens[b];
            const int nb = L < 0 ? -1 : (L + BS - 1) / BS;
            before += (nb <= 0 || nb > maxnb) ? 0 : (nb + kRows - 1) / kRows * N;
        }
        if (tid == 0) cpre[B] = total;
    }
    __syncthreads();
    const int total = cpre[B];
    const int n_mine = total > static_cast<int>(blockIdx.x)
                           ? (total - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                           : 0;
    const int cl = lane % kLPR;                        // 16-byte slice of a row
    const int r0 = (warp * kGroups + lane / kLPR) * kRowsPerLane;   // first row in the chunk
    const size_t row_stride = static_cast<size_t>(N) * D * kElemBytes;
    const int q_es = a.q_dt == QS_F32 ? 4 : 2;

    // query rows of a chunk's unit (G heads) go through a 3-slot ring in
    // shared memory (cp.async), the metadata rows straight into registers
    const int qrow_bytes = G * D * q_es;
    uint8_t* qslots = dyn + l.off_q;
    struct Loads {
        uint4 mx[kRowsPerLane], mn[kRowsPerLane];
        int b, n, j;          // request, KV head, first row (of this lane)
        int nrows;            // rows of this lane inside the unit (0..4)
        bool bad_meta;
    };
    auto load = [&](int i, Loads& x) {
        x.nrows = 0;
        x.bad_meta = false;
        if (i < n_mine) {
            const int c = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
            int lo = 0, hi = B;                        // cpre[lo] <= c < cpre[hi]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (cpre[mid] <= c) lo = mid;
                else hi = mid;
            }
            const int L = lens[lo];
            const int nb = (L + BS - 1) / BS;
            const int nch = (nb + kRows - 1) / kRows;
            const int r = c - cpre[lo];
            const int n = r / nch, ci = r - n * nch;
            x.b = lo;
            x.n = n;
            x.j = ci * kRows + r0;
            x.nrows = max(0, min(kRowsPerLane, nb - x.j));
            const uint8_t* qsrc = static_cast<const uint8_t*>(a.q) +
                                  (static_cast<size_t>(lo) * a.H + static_cast<size_t>(n) * G) * D * q_es;
            uint8_t* qdst = qslots + static_cast<size_t>(i % 3) * l.qslot_bytes;
            for (int o = tid * 16; o < qrow_bytes; o += kScanThreads * 16) cp_async16(qdst + o, qsrc + o);
            if (x.nrows > 0) {
                const int blk = QS_META_BLOCK(a, x.j);
                const int m = l.mbt_in_smem ? mbt_s[lo * a.MMBPR + blk]
                                            : a.mbt[static_cast<size_t>(lo) * a.MMBPR + blk];
                if (m < 0 || m >= a.num_meta) {
                    x.bad_meta = true;
                } else {
                    const size_t off = (static_cast<size_t>(m) * BS + QS_META_ROW(a, x.j)) * row_stride +
                                       static_cast<size_t>(n) * D * kElemBytes + cl * 16;
#pragma unroll
                    for (int k = 0; k < kRowsPerLane; ++k)
                        if (k < x.nrows) {
                            x.mx[k] = ldg_stream(a.maxb + off + k * row_stride);
                            x.mn[k] = ldg_stream(a.minb + off + k * row_stride);
                        }
                }
            }
        }
        cp_async_commit();
    };
    auto score = [&](int i, const Loads& x) {
        // the chunk's query rows have landed (this thread's copies, then
        // everyone's after the barrier); a slot is rewritten two chunks later
        cp_async_wait1();
        __syncthreads();
        // group-mean query of this lane's slice (step 1)
        const uint8_t* qs = qslots + static_cast<size_t>(i % 3) * l.qslot_bytes;
        float acc[kEl];
#pragma unroll
        for (int e = 0; e < kEl; ++e) acc[e] = 0.f;
        for (int g = 0; g < G; ++g) {
            if (a.q_dt == QS_F32) {
                const float* qp = reinterpret_cast<const float*>(qs) + g * D + cl * kEl;
#pragma unroll
                for (int e = 0; e < kEl; ++e) acc[e] += qp[e];
            } else {
                const uint32_t* qp = reinterpret_cast<const uint32_t*>(qs + (static_cast<size_t>(g) * D + cl * kEl) * 2);
#pragma unroll
                for (int e = 0; e < kEl / 2; ++e) {
                    const float2 f = a.q_dt == QS_BF16 ? pair_to_float2<Dt::BF16>(qp[e])
                                                       : pair_to_float2<Dt::F16>(qp[e]);
                    acc[2 * e] += f.x;
                    acc[2 * e + 1] += f.y;
                }
            }
        }
        float qreg[kEl];
#pragma unroll
        for (int e = 0; e < kEl; ++e) qreg[e] = group_mean(acc[e], G);
        RowChunk<MT> rc;
        rc.prepare(qreg);
        // rows (step 2.2)
        float v[kRowsPerLane];
#pragma unroll
        for (int k = 0; k < kRowsPerLane; ++k)
            v[k] = k < x.nrows && !x.bad_meta ? rc.dot(x.mx[k], x.mn[k]) : 0.f;
        const float tot = reduce_rows4<kLPR>(v, cl);
        const int rr = ((cl & (kLPR / 2)) ? 2 : 0) + ((cl & (kLPR / 4)) ? 1 : 0);
        if ((cl & (kLPR / 4 - 1)) == 0 && rr < x.nrows) {
            if (x.bad_meta && rr == 0) set_status(a.dev_status, QS_DEV_EMETA_TABLE);
            a.scores[static_cast<size_t>(x.b * N + x.n) * maxnb + x.j + rr] =
                x.bad_meta ? __int_as_float(0xff800000) : tot;
        }
    };

    Loads cur, nxt;
#pragma unroll
    for (int k = 0; k < kRowsPerLane; ++k) cur.mx[k] = cur.mn[k] = nxt.mx[k] = nxt.mn[k] = make_uint4(0, 0, 0, 0);
    load(0, cur);
    for (int i = 0; i < n_mine; i += 2) {
        load(i + 1, nxt);
        score(i, cur);
        if (i + 1 >= n_mine) break;
        load(i + 2, cur);
        score(i + 1, nxt);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// The units' scores (written by the scan) -> forced set, top-k, emission.
// Launched as a programmatic dependent of the scan, so its CTAs start while
// scan CTAs still hold the SMs: left to itself the block scheduler then packs
// several of them onto the first SMs that free up (measured on GB300: the 64
// CTAs of the long-context batch on 16 SMs, each running at a quarter of the
// SM).  So when the units fit on the SMs, each gets a CTA held alone on its
// SM by a padded shared-memory request; with more units than SMs (where
// packing costs less than running units one after another: ragged batch,
// 512 units, 47 vs 58 us) one CTA per unit, unpadded.  Each CTA loops over
// units all the same.
constexpr size_t kTopkOnePerSmSmem = 120 * 1024;
__global__ void __launch_bounds__(kThreads) quest_unit_topk_kernel(SelectArgs a) {
    extern __shared__ __align__(16) uint8_t dyn[];   // keys [maxnb] u32, flags [maxnb] u8
    __shared__ TopkFastScratch s_fast;
    __shared__ TopkScratch<kThreads> s_topk;
    pdl_launch_dependents();
    const int maxnb = a.MMBPR * a.BS;
    uint32_t* keys = reinterpret_cast<uint32_t*>(dyn);
    uint8_t* flags = dyn + static_cast<size_t>(maxnb) * 4;
    pdl_wait();   // the scores are written by the scan
    for (int u = blockIdx.x; u < a.B * a.N; u += gridDim.x) {
        const int b = u / a.N;
        const int L = a.seq_lens[b];
        int32_t* sel_out = a.selected + static_cast<size_t>(u) * a.k;
        if (L < 0 || (L + a.BS - 1) / a.BS > maxnb) {   // uniform over the CTA
            if (threadIdx.x == 0) set_status(a.dev_status, QS_DEV_ESEQ_LEN);
            for (int i = threadIdx.x; i < a.k; i += kThreads) sel_out[i] = -1;
            continue;
        }
        const int nb = (L + a.BS - 1) / a.BS;
        const float* scores_u = a.scores + static_cast<size_t>(u) * maxnb;
        for (int j = threadIdx.x; j < nb; j += kThreads) keys[j] = float_key(ldcg_f32(scores_u + j));
        __syncthreads();
        select_unit<false>(a, L, nb, keys, flags, sel_out, s_fast, s_topk);   // ends with a barrier
    }
}

template <Dt MT, int D>
qs_status launch(const SelectArgs& a, cudaStream_t s) {
    const int maxnb = a.MMBPR * a.BS;
    constexpr int kRows = rows_per_chunk<MT, D>();
    const size_t key_smem = align_up(align_up(static_cast<size_t>(maxnb), 4) * 4 + maxnb, 16);
    if (key_smem > 100 * 1024) return QS_EUNSUPPORTED;
    if (maxnb <= kRows) {
        auto kern = quest_select_unit_kernel<MT, D>;
        if (!ensure_smem(reinterpret_cast<const void*>(kern), key_smem)) return QS_ECUDA;
        kern<<<a.B * a.N, kThreads, key_smem, s>>>(a);
        QS_CHECK_LAUNCH();
        return QS_OK;
    }
    // scan: lengths, chunk prefix and the metadata table (if it fits)
    constexpr int kSRows = scan_rows<MT, D>();
    ScanLayout l = {};
    size_t off = 0;
    l.off_cpre = static_cast<uint32_t>(off);
    off = align_up(off + static_cast<size_t>(a.B + 1) * 4, 16);
    l.off_lens = static_cast<uint32_t>(off);
    off = align_up(off + static_cast<size_t>(a.B) * 4, 16);
    l.off_mbt = static_cast<uint32_t>(off);
    const size_t mbt_bytes = static_cast<size_t>(a.B) * a.MMBPR * 4;
    l.mbt_in_smem = off + mbt_bytes <= 160 * 1024;
    if (l.mbt_in_smem) off += mbt_bytes;
    off = align_up(off, 16);
    l.off_q = static_cast<uint32_t>(off);
    l.qslot_bytes = static_cast<uint32_t>(align_up(static_cast<size_t>(a.H / a.N) * D *
                                                   (a.q_dt == QS_F32 ? 4 : 2), 16));
    off += 3 * static_cast<size_t>(l.qslot_bytes);
    const size_t smem = align_up(off, 16);
    if (smem > 200 * 1024) return QS_EUNSUPPORTED;
    auto scan = quest_scan_kernel<MT, D>;
    if (!ensure_smem(reinterpret_cast<const void*>(scan), smem)) return QS_ECUDA;
    const long long chunks = static_cast<long long>(a.B) * a.N * ((maxnb + kSRows - 1) / kSRows);
    const int grid = static_cast<int>(std::min<long long>(num_sms(), std::max<long long>(chunks, 1)));
    scan<<<grid, kScanThreads, smem, s>>>(a, l);
    QS_CHECK_LAUNCH();
    // top-k per unit, a programmatic dependent of the scan: one CTA per unit,
    // alone on its SM when the units fit (see quest_unit_topk_kernel)
    auto topk = quest_unit_topk_kernel;
    const bool spread = a.B * a.N <= num_sms();
    const size_t topk_smem = spread ? std::max(key_smem, kTopkOnePerSmSmem) : key_smem;
    if (!ensure_smem(reinterpret_cast<const void*>(topk), topk_smem)) return QS_ECUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.B * a.N));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = topk_smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, topk, a) != cudaSuccess) return QS_ECUDA;
    QS_CHECK_LAUNCH();
    return QS_OK;
}

}  // namespace

size_t select_workspace_bytes(int B, int N, int maxnb) {
    // scores [B*N, maxnb] f32 (written by the scan, read by the top-k)
    return align_up(static_cast<size_t>(B) * N * maxnb * 4, 256);
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
    a.bs_shift = (BS & (BS - 1)) == 0 ? __builtin_ctz(static_cast<unsigned>(BS)) : -1;
    a.selected = selected;
    a.scores = scores_opt ? scores_opt : reinterpret_cast<float*>(ws);
    a.scores_out = scores_opt != nullptr;
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
