// Prefill importance producer on the tensor cores (tcgen05, sm_103a): the
// attention mass each prefill token received, per head, summed over the heads
// (Kestrel-LLM 10-2, section 1, signal 2; section 2, the decode call site
// that reads prefill_importance), for every cache dtype, in two passes:
//   rows:    lse2[i,g] = log2 sum_{s<=i} 2^(l2[i,g,s])
//   columns: mass[s]   = sum_{i>=s, g} 2^(l2[i,g,s] - lse2[i,g])
// with l2 = softmax_scale * log2(e) * (q . k).
//
// GB300 design:
//  * A pack kernel writes, per (request, KV head), the query rows (position
//    i, head g -> row i*G + g) and the key rows as 128-row bf16 tiles in the
//    tensor cores' canonical K-major layout (8-row x 16-byte core matrices,
//    no swizzle), so that a pass loads a tile with bulk copies.  fp32 inputs
//    are split into a high part bf16(x) and a low part bf16(x - high); a dot
//    product is then hi.hi + hi.lo + lo.hi (three MMAs), which leaves a
//    relative error of at most 2^-15 per product against fp32's 2^-24 (the
//    dropped lo.lo term, <= 2^-16, and the split residuals, <= 2^-17 each;
//    the median is near 2^-19).  bf16 and fp16 inputs need
//    one MMA each and are exact up to the fp32 accumulation.  int8 caches
//    (with the queries quantised per row as the decode calls do) enter as
//    bf16, which holds every int8 value exactly; a dot of D <= 128 products
//    of magnitude <= 127^2 stays below 2^24, so the fp32 accumulation is
//    exact too, and the epilogue applies the query and key scales (packed
//    next to the tiles) as the logit = scale * (s_q * s_k) * int_dot.
//  * Each pass is one CTA per 128-row resident tile: warp 8 loads the
//    resident tile once and streams the other operand's tiles through two
//    shared-memory slots (cp.async.bulk, mbarrier transaction counts) and one
//    of its threads issues the MMAs (M = N = 128, K = 16) into one of two
//    TMEM accumulators; warps 0-7 read the accumulator rows of their TMEM lane
//    quarter (warp w: quarter w % 4, columns 64 * (w / 4) .. +63; tcgen05.ld),
//    apply the causal mask and the softmax arithmetic, and hand the
//    accumulator back; the two halves of a row are combined at the end.
//    Loads, MMAs and the epilogue of consecutive tiles overlap.
//  * Rows pass: resident = 128 query rows, streamed = key tiles 0 .. last
//    position; column pass: resident = 128 keys, streamed = the query tiles
//    that can see them (split into parts of the query range); the rows'
//    lse2 values, written by the rows pass (and, for int8, the streamed
//    rows' scales), reach each epilogue warp's shared buffer one tile ahead
//    through cp.async.
//  * Every wait is bounded: on running out it records QS_DEV_ETIMEOUT and the
//    CTA leaves its work, freeing its TMEM.
#include <cuda_bf16.h>

#include <cmath>

#include "qs_common.cuh"

namespace qs {
namespace imptc {

constexpr int kRows = 128;                 // tile rows (MMA M and N)
constexpr int kEpiWarps = 8;               // warps 0-7: two per TMEM lane quarter
constexpr int kThreads = (kEpiWarps + 1) * 32;
constexpr int kTmemCols = 256;             // two 128-column fp32 accumulators
constexpr uint32_t kSpinMax = 1u << 20;    // bounded mbarrier waits: tries of
constexpr uint32_t kSuspendNs = 1000;      // at most ~1 us each (about a second)
constexpr int kCopyPiece = 16 * 1024;      // bytes per bulk copy
constexpr int kHalfCols = 64;              // accumulator columns of one epilogue warp
// per epilogue warp: two tiles x (row values, scales) of its 64 columns
constexpr uint32_t kStageBytes = 2 * 2 * kHalfCols * 4;
constexpr float kLn2 = 0.6931471805599453f;

struct TcArgs {
    const uint8_t* qpack;     // [B*N, ntq, nsplit] tiles of 128 x D bf16
    const uint8_t* kpack;     // [B*N, ntk, nsplit] tiles
    const float* qscale;      // int8: [B*N, ntq*128] query-row scales (packed row order)
    const float* kscale;      // int8: [B*N, ntk*128] key scales
    float* lse2;              // [B*N, ls_stride] base-2 row log-sum-exps, row = i*G + g
    float* part;              // [B*N, parts, S_max] column sums
    float* lse_out;           // optional [B, H, S_max] natural log-sum-exps
    const int32_t* lens;      // [B]
    int32_t* status;
    int B, H, N, G, g_shift, S_max, MKBPR, BS;
    int ntq, ntk, nsplit, ls_stride;
    int parts, part_tiles;    // column pass: query tiles per part
    float scale_log2;
};

QS_DEVINL bool len_ok(const TcArgs& a, int S) {
    return S >= 0 && S <= a.S_max && static_cast<long long>(S) <= static_cast<long long>(a.MKBPR) * a.BS;
}

// ---- packing ----------------------------------------------------------------

struct PackArgs {
    const uint8_t* src;       // queries [B, S_max, H, D] or the paged key cache [P, BS, N, D]
    const float* scale;       // int8: query scales [B, S_max, H] or key scales [P, BS, N]
    float* scale_dst;         // int8: the rows' scales in packed order [B*N, ntiles*128]
    const int32_t* bt;        // [B, MKBPR] (keys)
    const int32_t* lens;
    uint8_t* dst;
    int32_t* status;
    int B, H, N, G, S_max, MKBPR, BS, P, ntiles, nsplit;
};

// Byte offset of bf16 element (r, d) inside a 128 x D tile: core matrix
// (r / 8, d / 8) at ((r/8) * (D/8) + d/8) * 128, row r % 8 at +16 * (r % 8).
// One thread per 16-byte chunk (8 elements of one row): rows of a core matrix
// are consecutive threads, so the stores are contiguous.
template <Dt T, int D, bool kKeys>
__global__ void pack_kernel(const PackArgs a) {
    constexpr int CH = D / 8;                         // 16-byte chunks of a bf16 row
    constexpr int kTile = kRows * D * 2;
    const long long per_tile = static_cast<long long>(kRows) * CH;
    const long long total = static_cast<long long>(a.B) * a.N * a.ntiles * per_tile;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long tile_lin = idx / per_tile;    // (b*N + n) * ntiles + tile
        const int w = static_cast<int>(idx - tile_lin * per_tile);
        const int rr = w & 7, c = (w >> 3) % CH, m = (w >> 3) / CH;
        const int r = m * 8 + rr;                     // row inside the tile
        const int bn = static_cast<int>(tile_lin / a.ntiles);
        const int tile = static_cast<int>(tile_lin - static_cast<long long>(bn) * a.ntiles);
        const int b = bn / a.N, n = bn - b * a.N;
        const int S = a.lens[b];
        const bool ok = S >= 0 && S <= a.S_max &&
                        static_cast<long long>(S) <= static_cast<long long>(a.MKBPR) * a.BS;
        const int pr = tile * kRows + r;              // packed row
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = 0.f;
        const uint8_t* src = nullptr;
        size_t row_idx = 0;                           // the row's scale index (int8)
        if (ok) {
            if constexpr (!kKeys) {
                if (pr < S * a.G) {
                    const int i = pr / a.G, g = pr - i * a.G;
                    row_idx = (static_cast<size_t>(b) * a.S_max + i) * a.H + n * a.G + g;
                    src = a.src + row_idx * static_cast<size_t>(D) * DtInfo<T>::bytes;
                }
            } else if (pr < S) {
                const int e = a.bt[static_cast<size_t>(b) * a.MKBPR + pr / a.BS];
                if (e < 0 || e >= a.P) {
                    if (c == 0) set_status(a.status, QS_DEV_EBLOCK_TABLE);
                } else {
                    row_idx = (static_cast<size_t>(e) * a.BS + pr % a.BS) * a.N + n;
                    src = a.src + row_idx * static_cast<size_t>(D) * DtInfo<T>::bytes;
                }
            }
        }
        if constexpr (T == Dt::I8) {
            if (c == 0) a.scale_dst[static_cast<size_t>(tile_lin) * kRows + r] = src ? a.scale[row_idx] : 0.f;
        }
        if (src) {
            if constexpr (T == Dt::I8) {
                const uint2 u = *reinterpret_cast<const uint2*>(src + c * 8);
                const uint32_t wv[2] = {u.x, u.y};
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    x[e] = static_cast<float>(static_cast<int8_t>((wv[e >> 2] >> (8 * (e & 3))) & 0xffu));
            } else if constexpr (T == Dt::F32) {
                const uint4 u0 = *reinterpret_cast<const uint4*>(src + c * 32);
                const uint4 u1 = *reinterpret_cast<const uint4*>(src + c * 32 + 16);
                const uint32_t wv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(wv[e]);
            } else {
                const uint4 u = *reinterpret_cast<const uint4*>(src + c * 16);
                const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = pair_to_float2<T>(wv[e]);
                    x[2 * e] = f.x;
                    x[2 * e + 1] = f.y;
                }
            }
        }
        // high part (the value itself for bf16; fp16 rows are stored as fp16)
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if constexpr (T == Dt::F16) {
                const __half2 h = __floats2half2_rn(x[2 * e], x[2 * e + 1]);
                hi[e] = *reinterpret_cast<const uint32_t*>(&h);
                lo[e] = 0u;
            } else {
                const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
                hi[e] = *reinterpret_cast<const uint32_t*>(&h);
                const float2 hf = __bfloat1622float2(h);
                const __nv_bfloat162 l = __floats2bfloat162_rn(x[2 * e] - hf.x, x[2 * e + 1] - hf.y);
                lo[e] = *reinterpret_cast<const uint32_t*>(&l);
            }
        }
        uint8_t* out = a.dst + static_cast<size_t>(tile_lin) * a.nsplit * kTile +
                       (static_cast<size_t>(m) * CH + c) * 128 + rr * 16;
        stg_v4(out, make_uint4(hi[0], hi[1], hi[2], hi[3]));
        if (a.nsplit == 2) stg_v4(out + kTile, make_uint4(lo[0], lo[1], lo[2], lo[3]));
    }
}

// ---- tcgen05 / mbarrier / bulk-copy primitives ------------------------------

QS_DEVINL uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    // start >> 4 | leading (K-direction core-matrix step) >> 4 << 16 |
    // stride (8-row group step) >> 4 << 32 | descriptor version 1 << 46;
    // base offset 0, no swizzle
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
           (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B of format
// fmt (0 fp16, 1 bf16), both K-major, N = M = 128.
QS_DEVINL uint32_t umma_idesc(uint32_t fmt) {
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
}

QS_DEVINL void umma(uint32_t d_tmem, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(ad), "l"(bd), "r"(idesc), "r"(accumulate)
        : "memory");
}
QS_DEVINL void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
QS_DEVINL void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
QS_DEVINL void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
QS_DEVINL void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Waits for the completion of the phase with the given parity; false when
// the bound ran out (kSpinMax tries, each suspending the thread for at most
// kSuspendNs unless the phase completes first).
QS_DEVINL bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t it = 0; it < kSpinMax; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
            "selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity), "r"(kSuspendNs)
            : "memory");
        if (ok) return true;
    }
    return false;
}
// Bulk copy of `bytes` (multiple of 16) from global memory into this CTA's
// shared memory, completing on bar's transaction count.
QS_DEVINL void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    for (uint32_t o = 0; o < bytes; o += kCopyPiece) {
        const uint32_t sz = bytes - o < static_cast<uint32_t>(kCopyPiece) ? bytes - o : kCopyPiece;
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                dst + o),
            "l"(static_cast<const uint8_t*>(src) + o), "r"(sz), "r"(bar)
            : "memory");
    }
}
QS_DEVINL void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
QS_DEVINL void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane.
QS_DEVINL void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// 16-byte asynchronous copy global -> shared (L2 only) and its groups.
QS_DEVINL void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
QS_DEVINL void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
QS_DEVINL void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
QS_DEVINL void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Shared-memory layout of a pass: resident tile (nsplit parts), two streamed
// slots, barriers, TMEM address, the second column halves' row states, the
// epilogue warps' staging buffers.
template <int D>
struct Smem {
    static constexpr uint32_t tile = kRows * D * 2;
    uint32_t res, slot0, bars, tmem_ptr, half, stage, bytes;
    QS_DEVINL __host__ Smem(int nsplit) {
        res = 0;
        slot0 = res + nsplit * tile;
        bars = slot0 + 2 * nsplit * tile;
        tmem_ptr = bars + 8 * 8;
        half = tmem_ptr + 16;
        stage = half + 2 * kRows * 4;
        bytes = stage + kEpiWarps * kStageBytes;
    }
};

// One pass.  kCols = false: rows pass (resident query tile qt, streamed key
// tiles); kCols = true: column pass (resident key tile, streamed query tiles
// of this part).
template <int D, bool kCols, bool kI8>
__global__ void __launch_bounds__(kThreads, 1) importance_tc_kernel(const TcArgs a, uint32_t fmt) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const Smem<D> L(a.nsplit);
    constexpr uint32_t kTile = Smem<D>::tile;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = a.G;

    int bn, part = 0, rt;
    if constexpr (!kCols) {
        bn = blockIdx.x;
        rt = static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y);   // longest rows first
    } else {
        part = blockIdx.x % a.parts;
        bn = blockIdx.x / a.parts;
        rt = blockIdx.y;                                                      // longest columns first
    }
    const int b = bn / a.N, n = bn - b * a.N;
    const int S = a.lens[b];
    if (!len_ok(a, S)) {
        if (tid == 0) set_status(a.status, QS_DEV_ESEQ_LEN);
        return;
    }
    // streamed tile range [t_lo, t_hi)
    int t_lo, t_hi;
    if constexpr (!kCols) {
        if (rt * kRows >= S * G) return;
        const int last_pos = min(rt * kRows + kRows - 1, S * G - 1) >> a.g_shift;
        t_lo = 0;
        t_hi = last_pos / kRows + 1;
    } else {
        if (rt * kRows >= S) return;
        const int first_q = (rt * kRows * G) / kRows;          // first query tile seeing these keys
        t_lo = max(first_q, part * a.part_tiles);
        t_hi = min((S * G + kRows - 1) / kRows, (part + 1) * a.part_tiles);
        if (t_lo >= t_hi) {
            if (tid < kRows && rt * kRows + tid < a.S_max)
                a.part[(static_cast<size_t>(bn) * a.parts + part) * a.S_max + rt * kRows + tid] = 0.f;
            return;
        }
    }
    const int nt = t_hi - t_lo;

    const uint32_t sbase = smem_addr(smem);
    const uint32_t bar_res = sbase + L.bars;
    auto bar_full = [&](int s) { return sbase + L.bars + 8 + 8 * s; };
    auto bar_mma = [&](int s) { return sbase + L.bars + 24 + 8 * s; };
    auto bar_empty = [&](int s) { return sbase + L.bars + 40 + 8 * s; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.tmem_ptr);
    __shared__ int s_fail;
    if (tid == 0) {
        s_fail = 0;
        mbar_init(bar_res, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar_full(s), 1);
            mbar_init(bar_mma(s), 1);
            mbar_init(bar_empty(s), kEpiWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const uint8_t* res_src;
    const uint8_t* str_base;
    if constexpr (!kCols) {
        res_src = a.qpack + (static_cast<size_t>(bn) * a.ntq + rt) * a.nsplit * kTile;
        str_base = a.kpack + static_cast<size_t>(bn) * a.ntk * a.nsplit * kTile;
    } else {
        res_src = a.kpack + (static_cast<size_t>(bn) * a.ntk + rt) * a.nsplit * kTile;
        str_base = a.qpack + static_cast<size_t>(bn) * a.ntq * a.nsplit * kTile;
    }
    const float* lse_row = a.lse2 + static_cast<size_t>(bn) * a.ls_stride;
    const uint32_t slot_bytes = a.nsplit * kTile;

    if (warp == kEpiWarps) {
        // ---- loads and MMA issue (one thread)
        if (lane == 0) {
            bool ok = true;
            auto load_slot = [&](int t, int s) {
                mbar_expect_tx(bar_full(s), slot_bytes);
                bulk_load(sbase + L.slot0 + s * slot_bytes, str_base + static_cast<size_t>(t) * slot_bytes,
                          slot_bytes, bar_full(s));
            };
            mbar_expect_tx(bar_res, slot_bytes);
            bulk_load(sbase + L.res, res_src, slot_bytes, bar_res);
            for (int j = 0; j < min(2, nt); ++j) load_slot(t_lo + j, j);
            ok = mbar_wait(bar_res, 0);
            const uint32_t idesc = umma_idesc(fmt);
            constexpr uint32_t kSbo = D * 16;   // 8-row group step: D/8 core matrices of 128 bytes
            for (int j = 0; j < nt && ok; ++j) {
                const int s = j & 1;
                const uint32_t use = static_cast<uint32_t>(j >> 1);
                ok = mbar_wait(bar_full(s), use & 1u);
                if (ok && j >= 2) ok = mbar_wait(bar_empty(s), (use - 1u) & 1u);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(s * kRows);
                const uint32_t ra = sbase + L.res, rb = sbase + L.slot0 + s * slot_bytes;
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t ko = static_cast<uint32_t>(ks) * 256u;
                    const uint64_t ah = umma_desc(ra + ko, 128, kSbo), bh = umma_desc(rb + ko, 128, kSbo);
                    umma(d_tmem, ah, bh, idesc, ks > 0 ? 1u : 0u);
                    if (a.nsplit == 2) {
                        const uint64_t al = umma_desc(ra + kTile + ko, 128, kSbo);
                        const uint64_t bl = umma_desc(rb + kTile + ko, 128, kSbo);
                        umma(d_tmem, ah, bl, idesc, 1u);
                        umma(d_tmem, al, bh, idesc, 1u);
                    }
                }
                umma_commit(bar_mma(s));
                // refill the slot of tile j-1 with tile j+1 once its MMAs are done
                if (j >= 1 && j + 1 < nt) {
                    const int ps = (j + 1) & 1;
                    ok = mbar_wait(bar_mma(ps), static_cast<uint32_t>((j - 1) >> 1) & 1u);
                    if (ok) load_slot(t_lo + j + 1, ps);
                }
            }
            if (!ok) {
                set_status(a.status, QS_DEV_ETIMEOUT);
                atomicExch(&s_fail, 1);
            }
        }
    } else {
        // ---- epilogue: accumulator row r = this thread's TMEM lane, column
        // half hc of every 128-column tile
        const int quarter = warp & 3, hc = warp >> 2;
        const int r = quarter * 32 + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        float qf = a.scale_log2;
        float m_run = -INFINITY, l_run = 0.f, colsum = 0.f;
        // row pass: query row pr = rt*128 + r; column pass: key s = rt*128 + r
        const int pr_res = rt * kRows + r;
        const int i_res = pr_res >> a.g_shift;
        // int8: the resident row's scale (query: folded into qf; key: kf_res)
        float kf_res = 1.f;
        const float* str_scale = nullptr;   // the streamed rows' scales
        if constexpr (kI8) {
            if constexpr (!kCols) {
                qf = __fmul_rn(a.qscale[static_cast<size_t>(bn) * a.ntq * kRows + pr_res], a.scale_log2);
                str_scale = a.kscale + static_cast<size_t>(bn) * a.ntk * kRows;
            } else {
                kf_res = a.kscale[static_cast<size_t>(bn) * a.ntk * kRows + pr_res];
                str_scale = a.qscale + static_cast<size_t>(bn) * a.ntq * kRows;
            }
        }
        // The per-column values of a streamed tile (column pass: the query
        // rows' lse2; int8: the streamed rows' scales) are staged in this
        // warp's shared buffer one tile ahead with cp.async (lanes 0-15:
        // lse2, lanes 16-31: scales; 16 bytes each), so the epilogue reads
        // them from shared memory instead of waiting on L2 every tile.
        constexpr bool kStage = kCols || kI8;
        const uint32_t stg = sbase + L.stage + static_cast<uint32_t>(warp) * kStageBytes;
        const float* stg_f = reinterpret_cast<const float*>(smem + L.stage + warp * kStageBytes);
        auto stage_tile = [&](int t, int buf) {
            const uint32_t d = stg + static_cast<uint32_t>(buf) * (2 * kHalfCols * 4);
            const size_t col = static_cast<size_t>(t) * kRows + hc * kHalfCols;
            if (kCols && lane < 16) cp_async16(d + lane * 16, lse_row + col + lane * 4);
            if (kI8 && lane >= 16) cp_async16(d + kHalfCols * 4 + (lane - 16) * 16, str_scale + col + (lane - 16) * 4);
            cp_async_commit();
        };
        if constexpr (kStage) stage_tile(t_lo, 0);
        for (int j = 0; j < nt; ++j) {
            const int s = j & 1;
            const uint32_t use = static_cast<uint32_t>(j >> 1);
            if constexpr (kStage) {
                if (j + 1 < nt) stage_tile(t_lo + j + 1, (j + 1) & 1);
                else cp_async_commit();
            }
            if (!mbar_wait(bar_mma(s), use & 1u)) {
                if (lane == 0) {
                    set_status(a.status, QS_DEV_ETIMEOUT);
                    atomicExch(&s_fail, 1);
                }
                break;
            }
            tc_fence_after();
            if constexpr (kStage) {
                cp_async_wait1();   // this tile's group (the next tile's may still fly)
                __syncwarp();
            }
            const float* cur = stg_f + (j & 1) * (2 * kHalfCols);
            const int t = t_lo + j;
#pragma unroll 1
            for (int c0 = hc * 64; c0 < hc * 64 + 64; c0 += 32) {
                float v[32];
                float sc[32];   // int8: the streamed rows' scales of these columns
                if constexpr (kI8) {
                    const float4* s4 = reinterpret_cast<const float4*>(cur + kHalfCols + (c0 - hc * 64));
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) {
                        const float4 w4 = s4[q4];
                        sc[4 * q4] = w4.x; sc[4 * q4 + 1] = w4.y; sc[4 * q4 + 2] = w4.z; sc[4 * q4 + 3] = w4.w;
                    }
                }
                tmem_ld32(lane_base + static_cast<uint32_t>(s * kRows + c0), v);
                if constexpr (!kCols) {
                    // keys t*128 + c0 + jj <= i (and the row exists)
                    const int k0 = t * kRows + c0;
                    const bool row_ok = pr_res < S * G;
                    if constexpr (kI8) {
                        // logit (base 2) = (dot * s_q * scale * log2 e) * s_k
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) v[jj] = __fmul_rn(__fmul_rn(v[jj], qf), sc[jj]);
                    }
                    float cmax = -INFINITY;
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj)
                        if (row_ok && k0 + jj <= i_res) cmax = fmaxf(cmax, v[jj]);
                    if (cmax != -INFINITY) {
                        const float mt = kI8 ? cmax : __fmul_rn(cmax, qf);
                        if (mt > m_run) {
                            l_run *= exp2_approx(m_run - mt);
                            m_run = mt;
                        }
                        float add = 0.f;
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) {
                            const float p = kI8 ? exp2_approx(v[jj] - m_run) : exp2_approx(fmaf(v[jj], qf, -m_run));
                            add += (k0 + jj <= i_res) ? p : 0.f;
                        }
                        l_run += add;
                    }
                } else {
                    // query rows pr = t*128 + c0 + jj with position >= key s, < S
                    const float4* lse_s = reinterpret_cast<const float4*>(cur + (c0 - hc * 64));
                    const int pr0 = t * kRows + c0;
                    const int pr_min = pr_res * G;     // first row of a position >= the key
                    const int pr_end = S * G;
                    if (pr_res < S) {
                        float lse[32];
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4) {
                            const float4 l4 = lse_s[q4];
                            lse[4 * q4] = l4.x; lse[4 * q4 + 1] = l4.y;
                            lse[4 * q4 + 2] = l4.z; lse[4 * q4 + 3] = l4.w;
                        }
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) {
                            const int pr = pr0 + jj;
                            float p;
                            if constexpr (kI8)
                                p = exp2_approx(__fmul_rn(__fmul_rn(v[jj], __fmul_rn(sc[jj], qf)), kf_res) - lse[jj]);
                            else
                                p = exp2_approx(fmaf(v[jj], qf, -lse[jj]));
                            colsum += (pr >= pr_min && pr < pr_end) ? p : 0.f;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();   // also: every lane has read this tile's staged values
            if (lane == 0) mbar_arrive(bar_empty(s));
        }
        if constexpr (kStage) cp_async_wait0();
        // combine the two column halves of every row (the second half's
        // state goes through shared memory)
        float* half_m = reinterpret_cast<float*>(smem + L.half);
        float* half_x = half_m + kRows;
        if (hc == 1) {
            half_m[r] = m_run;
            half_x[r] = kCols ? colsum : l_run;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
        if (hc == 1) {
            // nothing more: the first half writes the row
        } else if constexpr (!kCols) {
            const float m1 = half_m[r], l1 = half_x[r];
            const float M = fmaxf(m_run, m1);
            if (M != -INFINITY) {
                l_run = (m_run == -INFINITY ? 0.f : l_run * exp2_approx(m_run - M)) +
                        (m1 == -INFINITY ? 0.f : l1 * exp2_approx(m1 - M));
                m_run = M;
            }
            if (pr_res < S * G && !s_fail) {
                const float l2 = m_run + log2f(l_run);
                a.lse2[static_cast<size_t>(bn) * a.ls_stride + pr_res] = l2;
                if (a.lse_out) {
                    const int g = pr_res & (G - 1);
                    a.lse_out[(static_cast<size_t>(b) * a.H + n * G + g) * a.S_max + i_res] = l2 * kLn2;
                }
            }
        } else if (pr_res < a.S_max) {
            a.part[(static_cast<size_t>(bn) * a.parts + part) * a.S_max + pr_res] = colsum + half_x[r];
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
}

// Self-check of the bounded wait: one thread waits on an mbarrier that
// nothing arrives on, runs out and records QS_DEV_ETIMEOUT.
__global__ void bounded_wait_check_kernel(int32_t* status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!mbar_wait(smem_addr(&bar), 0)) set_status(status, QS_DEV_ETIMEOUT);
    }
}

}  // namespace imptc

// ---- host -----------------------------------------------------------------------

namespace {

using namespace imptc;

template <Dt T, int D>
bool launch_tc_dt(const TcArgs& a, const PackArgs& pq, const PackArgs& pk, cudaStream_t st) {
    const int sms = num_sms();
    auto grid_of = [&](long long total) {
        long long g = (total + 255) / 256;
        if (g > static_cast<long long>(sms) * 16) g = static_cast<long long>(sms) * 16;
        return static_cast<unsigned>(g > 0 ? g : 1);
    };
    const long long per_tile = static_cast<long long>(kRows) * (D / 8);
    pack_kernel<T, D, false><<<grid_of(static_cast<long long>(a.B) * a.N * a.ntq * per_tile), 256, 0, st>>>(pq);
    pack_kernel<T, D, true><<<grid_of(static_cast<long long>(a.B) * a.N * a.ntk * per_tile), 256, 0, st>>>(pk);
    const Smem<D> L(a.nsplit);
    constexpr bool kI8 = T == Dt::I8;
    auto k_rows = importance_tc_kernel<D, false, kI8>;
    auto k_cols = importance_tc_kernel<D, true, kI8>;
    if (!ensure_smem(reinterpret_cast<const void*>(k_rows), L.bytes) ||
        !ensure_smem(reinterpret_cast<const void*>(k_cols), L.bytes))
        return false;
    const uint32_t fmt = T == Dt::F16 ? 0u : 1u;
    k_rows<<<dim3(static_cast<unsigned>(a.B * a.N), static_cast<unsigned>(a.ntq)), kThreads, L.bytes, st>>>(a, fmt);
    k_cols<<<dim3(static_cast<unsigned>(a.B * a.N * a.parts), static_cast<unsigned>(a.ntk)), kThreads, L.bytes,
             st>>>(a, fmt);
    return cudaGetLastError() == cudaSuccess;
}

}  // namespace

size_t importance_tc_workspace(long long B, long long H, long long N, long long D, long long S_max,
                               bool f32, bool int8, size_t* off_q, size_t* off_k, size_t* off_lse,
                               size_t* off_qs, size_t* off_ks) {
    const long long G = H / N;
    const long long ntq = (S_max * G + kRows - 1) / kRows, ntk = (S_max + kRows - 1) / kRows;
    const size_t tile = static_cast<size_t>(kRows) * D * 2 * (f32 ? 2 : 1);
    size_t off = 0;
    *off_q = off;
    off = align_up(off + static_cast<size_t>(B * N * ntq) * tile, 256);
    *off_k = off;
    off = align_up(off + static_cast<size_t>(B * N * ntk) * tile, 256);
    *off_lse = off;
    off = align_up(off + static_cast<size_t>(B * N * ntq) * kRows * 4, 256);
    // int8: the rows' scales in packed order
    *off_qs = off;
    if (int8) off = align_up(off + static_cast<size_t>(B * N * ntq) * kRows * 4, 256);
    *off_ks = off;
    if (int8) off = align_up(off + static_cast<size_t>(B * N * ntk) * kRows * 4, 256);
    return off;
}

bool importance_tc_launch(const void* q, const float* q_scale, Dt dt, const void* k_cache,
                          const float* k_scale, int32_t num_kv_blocks, const int32_t* block_tables,
                          int32_t MKBPR, const int32_t* lens, int32_t S_max, int32_t B, int32_t H,
                          int32_t N, int32_t D, int32_t BS, float scale_log2, float* part, int parts,
                          float* lse_out, uint8_t* ws, int32_t* status, cudaStream_t st) {
    size_t oq, ok_, ol, oqs, oks;
    importance_tc_workspace(B, H, N, D, S_max, dt == Dt::F32, dt == Dt::I8, &oq, &ok_, &ol, &oqs, &oks);
    const int G = H / N;
    TcArgs a{};
    a.ntq = static_cast<int>((static_cast<long long>(S_max) * G + kRows - 1) / kRows);
    a.ntk = static_cast<int>((static_cast<long long>(S_max) + kRows - 1) / kRows);
    a.nsplit = dt == Dt::F32 ? 2 : 1;
    a.ls_stride = a.ntq * kRows;
    a.qpack = ws + oq;
    a.kpack = ws + ok_;
    a.qscale = reinterpret_cast<const float*>(ws + oqs);
    a.kscale = reinterpret_cast<const float*>(ws + oks);
    a.lse2 = reinterpret_cast<float*>(ws + ol);
    a.part = part;
    a.lse_out = lse_out;
    a.lens = lens;
    a.status = status;
    a.B = B; a.H = H; a.N = N; a.G = G;
    a.g_shift = __builtin_ctz(static_cast<unsigned>(G));
    a.S_max = S_max; a.MKBPR = MKBPR; a.BS = BS;
    a.parts = parts;
    a.part_tiles = (a.ntq + parts - 1) / parts;
    a.scale_log2 = scale_log2;

    PackArgs pq{};
    pq.src = static_cast<const uint8_t*>(q);
    pq.scale = q_scale;
    pq.scale_dst = reinterpret_cast<float*>(ws + oqs);
    pq.lens = lens; pq.dst = ws + oq; pq.status = status;
    pq.B = B; pq.H = H; pq.N = N; pq.G = G; pq.S_max = S_max; pq.MKBPR = MKBPR; pq.BS = BS;
    pq.P = num_kv_blocks; pq.ntiles = a.ntq; pq.nsplit = a.nsplit;
    PackArgs pk = pq;
    pk.src = static_cast<const uint8_t*>(k_cache);
    pk.scale = k_scale;
    pk.scale_dst = reinterpret_cast<float*>(ws + oks);
    pk.bt = block_tables;
    pk.dst = ws + ok_;
    pk.ntiles = a.ntk;

    switch (dt) {
        case Dt::F32: return D == 64 ? launch_tc_dt<Dt::F32, 64>(a, pq, pk, st) : launch_tc_dt<Dt::F32, 128>(a, pq, pk, st);
        case Dt::BF16: return D == 64 ? launch_tc_dt<Dt::BF16, 64>(a, pq, pk, st) : launch_tc_dt<Dt::BF16, 128>(a, pq, pk, st);
        case Dt::I8: return D == 64 ? launch_tc_dt<Dt::I8, 64>(a, pq, pk, st) : launch_tc_dt<Dt::I8, 128>(a, pq, pk, st);
        default: return D == 64 ? launch_tc_dt<Dt::F16, 64>(a, pq, pk, st) : launch_tc_dt<Dt::F16, 128>(a, pq, pk, st);
    }
}

}  // namespace qs

extern "C" qs_status qs_check_bounded_wait(int32_t* dev_status, qs_stream_t stream) {
    if (!dev_status) return QS_EINVAL;
    qs::imptc::bounded_wait_check_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        dev_status);
    return cudaGetLastError() == cudaSuccess ? QS_OK : QS_ECUDA;
}
