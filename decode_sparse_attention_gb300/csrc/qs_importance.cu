// Prefill importance producer: the attention mass each prefill token
// received, per head, summed over the heads (Kestrel-LLM 10-2, section 1,
// signal 2; section 2, the decode call site that reads prefill_importance).
//
// For request b, KV head n and its G = H/N query heads, the causal logits of
// query row (i, g) against key s <= i are recomputed twice:
//   pass 1 (rows):    lse2[i,g] = log2 sum_{s<=i} 2^(l2[i,g,s]),
//   pass 2 (columns): mass[s]   = sum_{i>=s, g} 2^(l2[i,g,s] - lse2[i,g]),
// with l2 the logit in base 2 (softmax_scale * log2(e) folded into the query
// factor).  Both passes are the same tiled fp32 contraction over D on the CUDA
// cores: 128 resident rows held in shared memory for the CTA's life times 64
// streamed rows per tile (cp.async into a double-buffered ring), 256 threads,
// each owning an 8 x 4 block of logits accumulated with packed fp32x2 FMAs
// (even and odd channels in the two lanes).  Pass 1 keeps the queries
// resident and streams keys; pass 2 keeps keys resident and streams queries,
// so that every column sum stays in registers.  A last kernel adds the KV
// heads' (and query-range parts') column sums per token.  Both passes form
// each logit with the same operations in the same order, so pass 2's
// probabilities are exactly the ones pass 1 normalised.
//
// This CUDA-core form serves int8 caches; fp32, bf16 and fp16 caches take the
// tensor-core form (qs_importance_tc.cu), whose passes feed the same column
// sums into the same final kernel.
#include <cmath>
#include <type_traits>

#include "qs_internal.cuh"

namespace qs {
namespace imp {

constexpr int kThreads = 256;
constexpr int kRes = 128;       // resident rows per CTA
constexpr int kStr = 64;        // streamed rows per tile
constexpr int kTabMax = 2048;   // block-table entries staged per CTA (pass 1)
constexpr int kMaxParts = 8;    // query-range parts of pass 2
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct Args {
    const uint8_t* q;         // [B, S_max, H, D] QT (int8 mode: quantised rows)
    const float* s_q;         // int8 mode: [B, S_max, H] query scales
    const uint8_t* k;         // [P, BS, N, D] KT
    const float* k_scale;     // int8: [P, BS, N]
    const int32_t* bt;        // [B, MKBPR]
    const int32_t* lens;      // [B]
    float* lse2;              // workspace [B, N, S_max * G]
    float* part;              // workspace [B, N, parts, S_max]
    float* lse_out;           // optional [B, H, S_max]
    float* importance;        // [B, S_max]
    int32_t* status;
    int P, MKBPR, S_max, B, H, N, G, BS;
    int g_shift;              // log2 G
    int bs_shift;             // log2 BS, or -1 when BS is not a power of two
    int parts, part_tiles;    // pass 2 split of the query tiles
    float scale_log2;         // softmax_scale * log2(e)
};

QS_DEVINL void cpa16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
QS_DEVINL void cpa4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
QS_DEVINL void cpa_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
QS_DEVINL void cpa_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

QS_DEVINL uint4 ldg_nc(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 16 bytes of elements of type T -> 16/sizeof(T) floats at dst (16-B aligned).
template <Dt T> QS_DEVINL void store_chunk(float* dst, uint4 w);
template <> QS_DEVINL void store_chunk<Dt::F32>(float* dst, uint4 w) {
    *reinterpret_cast<uint4*>(dst) = w;
}
template <Dt T> QS_DEVINL void store_chunk16(float* dst, uint4 w) {
    const float2 a = pair_to_float2<T>(w.x), b = pair_to_float2<T>(w.y);
    const float2 c = pair_to_float2<T>(w.z), d = pair_to_float2<T>(w.w);
    reinterpret_cast<float4*>(dst)[0] = make_float4(a.x, a.y, b.x, b.y);
    reinterpret_cast<float4*>(dst)[1] = make_float4(c.x, c.y, d.x, d.y);
}
template <> QS_DEVINL void store_chunk<Dt::BF16>(float* dst, uint4 w) {
    store_chunk16<Dt::BF16>(dst, w);
}
template <> QS_DEVINL void store_chunk<Dt::F16>(float* dst, uint4 w) {
    store_chunk16<Dt::F16>(dst, w);
}
template <> QS_DEVINL void store_chunk<Dt::I8>(float* dst, uint4 w) {
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; j++) {
        reinterpret_cast<float4*>(dst)[j] =
            make_float4(static_cast<float>(static_cast<int8_t>(v[j] & 0xffu)),
                        static_cast<float>(static_cast<int8_t>((v[j] >> 8) & 0xffu)),
                        static_cast<float>(static_cast<int8_t>((v[j] >> 16) & 0xffu)),
                        static_cast<float>(static_cast<int8_t>(v[j] >> 24)));
    }
}

// Shared-memory layout of one pass.  Rows are fp32 with a pitch of D + 4
// floats, so 4 consecutive rows (resident reads) or 8 (streamed reads) of a
// 16-byte column fall in distinct banks.
template <Dt QT, Dt KT, int D, bool kCols>
struct Layout {
    static constexpr Dt RT = kCols ? KT : QT;            // resident element type
    static constexpr Dt ST = kCols ? QT : KT;            // streamed element type
    static constexpr int pitch = D + 4;
    static constexpr int raw_row = ST == Dt::F32 ? 0 : D * DtInfo<ST>::bytes;
    static constexpr size_t res = 0;
    static constexpr size_t str = res + size_t(kRes) * pitch * 4;
    static constexpr size_t stg = str + size_t(2) * kStr * pitch * 4;
    static constexpr size_t tab = stg + size_t(2) * kStr * raw_row;
    static constexpr size_t rpos = tab + (kCols ? 0 : size_t(kTabMax) * 4);
    static constexpr size_t rfac = rpos + size_t(kRes) * 4;
    static constexpr size_t spos = rfac + size_t(kRes) * 4;
    static constexpr size_t sfac = spos + size_t(2) * kStr * 4;
    static constexpr size_t slse = sfac + size_t(2) * kStr * 4;
    static constexpr size_t bytes = slse + size_t(2) * kStr * 4;
    static_assert(bytes <= 227 * 1024, "shared memory");
    static_assert(size_t(kRes) * 2 * 16 * 4 <= size_t(2) * kStr * pitch * 4, "reduction scratch");
};

}  // namespace imp
}  // namespace qs

namespace qs {
namespace imp {

// One pass over a (request, KV head) tile.  Pass 1 (kCols = false): CTA
// (b*N + n, row tile) holds the 128 query rows (position base + r/G, head
// n*G + r%G) and streams the keys 0 .. last position in 64-key tiles; it
// writes the rows' base-2 log-sum-exp.  Pass 2 (kCols = true): CTA
// ((b*N + n)*parts + part, key tile) holds keys base .. base+127 and streams
// its part of the query tiles (64 rows = 64/G positions x G heads) that can
// see them; it writes the keys' column sums of this part.
template <Dt QT, Dt KT, int D, bool kCols>
__global__ void __launch_bounds__(kThreads, 1) importance_pass_kernel(const Args a) {
    using L = Layout<QT, KT, D, kCols>;
    constexpr Dt RT = L::RT, ST = L::ST;
    constexpr int pitch = L::pitch;
    constexpr bool kInt8 = KT == Dt::I8;
    constexpr int q_row_bytes = D * DtInfo<QT>::bytes, k_row_bytes = D * DtInfo<KT>::bytes;
    constexpr int RCPR = D * DtInfo<RT>::bytes / 16, SCPR = D * DtInfo<ST>::bytes / 16;
    constexpr int REPC = 16 / DtInfo<RT>::bytes, SEPC = 16 / DtInfo<ST>::bytes;

    extern __shared__ __align__(16) uint8_t smem[];
    float* s_res = reinterpret_cast<float*>(smem + L::res);
    float* s_str = reinterpret_cast<float*>(smem + L::str);
    uint8_t* s_stg = smem + L::stg;
    int32_t* s_tab = reinterpret_cast<int32_t*>(smem + L::tab);
    int32_t* s_rpos = reinterpret_cast<int32_t*>(smem + L::rpos);
    float* s_rfac = reinterpret_cast<float*>(smem + L::rfac);
    int32_t* s_spos = reinterpret_cast<int32_t*>(smem + L::spos);
    float* s_sfac = reinterpret_cast<float*>(smem + L::sfac);
    float* s_slse = reinterpret_cast<float*>(smem + L::slse);

    const int tid = threadIdx.x;
    const int G = a.G;
    const int TQs = kStr / G;   // query positions per streamed tile (pass 2)
    int b, n, part = 0, base;
    if constexpr (!kCols) {
        b = blockIdx.x / a.N;
        n = blockIdx.x - b * a.N;
        base = (gridDim.y - 1 - blockIdx.y) * (kRes / G);   // longest rows first
    } else {
        part = blockIdx.x % a.parts;
        const int bn = blockIdx.x / a.parts;
        b = bn / a.N;
        n = bn - b * a.N;
        base = blockIdx.y * kRes;                           // longest columns first
    }
    const int S = a.lens[b];
    if (S < 0 || S > a.S_max || static_cast<long long>(S) > static_cast<long long>(a.MKBPR) * a.BS) {
        if (tid == 0) set_status(a.status, QS_DEV_ESEQ_LEN);
        return;
    }
    if (base >= S) return;
    const size_t bn_rows = static_cast<size_t>(b) * a.N + n;
    const int h0 = n * G;
    const int32_t* bt_row = a.bt + static_cast<size_t>(b) * a.MKBPR;

    int tile_lo, tile_hi;
    if constexpr (!kCols) {
        tile_lo = 0;
        tile_hi = (min(base + kRes / G, S) - 1) / kStr + 1;
    } else {
        tile_lo = max(base / TQs, part * a.part_tiles);
        tile_hi = min((S - 1) / TQs + 1, (part + 1) * a.part_tiles);
        if (tile_lo >= tile_hi) {   // no query of this part sees these keys
            if (tid < kRes && base + tid < a.S_max)
                a.part[(bn_rows * a.parts + part) * a.S_max + base + tid] = 0.f;
            return;
        }
    }

    // block-table entries of the streamed keys (pass 1), validated once
    bool staged = false;
    if constexpr (!kCols) {
        const int n_ent = (min(tile_hi * kStr, S) + a.BS - 1) / a.BS;
        staged = n_ent <= kTabMax;
        if (staged) {
            for (int j = tid; j < n_ent; j += kThreads) {
                int e = bt_row[j];
                if (e < 0 || e >= a.P) {
                    set_status(a.status, QS_DEV_EBLOCK_TABLE);
                    e = -1;
                }
                s_tab[j] = e;
            }
        }
        __syncthreads();
    }
    auto blk_of = [&](int s) { return a.bs_shift >= 0 ? s >> a.bs_shift : s / a.BS; };
    auto entry = [&](int j) -> int {
        if constexpr (!kCols) {
            if (staged) return s_tab[j];
        }
        int e = __ldg(bt_row + j);
        if (e < 0 || e >= a.P) {
            set_status(a.status, QS_DEV_EBLOCK_TABLE);
            e = -1;
        }
        return e;
    };
    auto q_src = [&](int i, int g) {
        return a.q + ((static_cast<size_t>(b) * a.S_max + i) * a.H + h0 + g) * q_row_bytes;
    };
    auto k_tok = [&](int e, int s) {
        const int row = a.bs_shift >= 0 ? (s & (a.BS - 1)) : s % a.BS;
        return (static_cast<size_t>(e) * a.BS + row) * a.N + n;
    };

    // resident rows (fp32) and their position / factor
    for (int c = tid; c < kRes * RCPR; c += kThreads) {
        const int r = c / RCPR, ch = c - r * RCPR;
        const uint8_t* src = nullptr;
        if constexpr (!kCols) {
            const int i = base + r / G;
            if (i < S) src = q_src(i, r % G);
        } else {
            const int s = base + r;
            if (s < S) {
                const int e = entry(blk_of(s));
                if (e >= 0) src = a.k + k_tok(e, s) * k_row_bytes;
            }
        }
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (src) w = ldg_nc(src + ch * 16);
        store_chunk<RT>(s_res + r * pitch + ch * REPC, w);
    }
    if (tid < kRes) {
        const int r = tid;
        int pos = -1;
        float fac = 1.f;
        if constexpr (!kCols) {
            const int i = base + r / G;
            if (i < S) {
                pos = i;
                fac = a.scale_log2;
                if constexpr (kInt8)
                    fac = __fmul_rn(a.s_q[(static_cast<size_t>(b) * a.S_max + i) * a.H + h0 + r % G],
                                    a.scale_log2);
            }
        } else {
            const int s = base + r;
            if (s < S) {
                const int e = entry(blk_of(s));
                if (e >= 0) {
                    pos = s;
                    if constexpr (kInt8) fac = a.k_scale[k_tok(e, s)];
                }
            }
        }
        s_rpos[r] = pos;
        s_rfac[r] = fac;
    }

    // streamed tile t -> ring slot buf: 4 threads per row, each copying every
    // 4th 16-byte chunk of it (fp32 rows straight into the ring, others raw)
    auto issue = [&](int t, int buf) {
        const int r = tid >> 2, c0 = tid & 3;
        const uint8_t* src = nullptr;
        int pos = -1;
        size_t tok = 0;
        if constexpr (!kCols) {
            const int s = t * kStr + r;
            if (s < S) {
                const int e = entry(blk_of(s));
                if (e >= 0) {
                    tok = k_tok(e, s);
                    src = a.k + tok * k_row_bytes;
                    pos = s;
                }
            }
        } else {
            const int i = t * TQs + (r >> a.g_shift);
            if (i < S) {
                src = q_src(i, r & (G - 1));
                pos = i;
            }
        }
        uint8_t* dst = ST == Dt::F32
                           ? reinterpret_cast<uint8_t*>(s_str + (buf * kStr + r) * pitch)
                           : s_stg + (buf * kStr + r) * L::raw_row;
#pragma unroll
        for (int j = 0; j < SCPR / 4; ++j) {
            const int ch = c0 + 4 * j;
            if (src) cpa16(smem_addr(dst + ch * 16), src + ch * 16);
            else *reinterpret_cast<uint4*>(dst + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        if (c0 == 0) {
            if (pos >= 0) {
                if constexpr (!kCols) {
                    if constexpr (kInt8) cpa4(smem_addr(s_sfac + buf * kStr + r), a.k_scale + tok);
                } else {
                    const int g = r & (G - 1);
                    cpa4(smem_addr(s_slse + buf * kStr + r),
                         a.lse2 + bn_rows * a.S_max * G + static_cast<size_t>(pos) * G + g);
                    if constexpr (kInt8)
                        cpa4(smem_addr(s_sfac + buf * kStr + r),
                             a.s_q + (static_cast<size_t>(b) * a.S_max + pos) * a.H + h0 + g);
                }
            }
            s_spos[buf * kStr + r] = pos;
        }
        cpa_commit();
    };

    const int lane = tid & 31, warp = tid >> 5;
    const int rg = (warp & 3) * 4 + (lane >> 3);   // resident rows rg + 16u
    const int sg = (warp >> 2) * 8 + (lane & 7);   // streamed rows sg + 16v
    float st_a[8], st_b[8];   // pass 1: running max, running sum; pass 2: column sums
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        st_a[u] = kCols ? 0.f : -INFINITY;
        st_b[u] = 0.f;
    }

    issue(tile_lo, 0);
    for (int t = tile_lo; t < tile_hi; ++t) {
        const int buf = (t - tile_lo) & 1;
        cpa_wait_all();
        __syncthreads();   // tile t landed; every thread is done with tile t-1
        if (t + 1 < tile_hi) issue(t + 1, buf ^ 1);
        if constexpr (ST != Dt::F32) {
            const uint8_t* src = s_stg + buf * kStr * L::raw_row;
            float* dst = s_str + buf * kStr * pitch;
            for (int c = tid; c < kStr * SCPR; c += kThreads) {
                const int r = c / SCPR, ch = c - r * SCPR;
                store_chunk<ST>(dst + r * pitch + ch * SEPC,
                                *reinterpret_cast<const uint4*>(src + r * L::raw_row + ch * 16));
            }
            __syncthreads();
        }

        // 8 x 4 dot products: even channels in the low lane, odd in the high
        // lane; all first halves of a 4-channel step before the second halves.
        // The channel loop is unrolled completely (measured 10 % faster than
        // unrolling by 4 at D = 128).
        const float* Sm = s_str + buf * kStr * pitch;
        unsigned long long acc[8][4];
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc[u][v] = 0ull;
#pragma unroll
        for (int d = 0; d < D; d += 4) {
            ulonglong2 rv[8], sv[4];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                rv[u] = *reinterpret_cast<const ulonglong2*>(s_res + (rg + 16 * u) * pitch + d);
#pragma unroll
            for (int v = 0; v < 4; ++v)
                sv[v] = *reinterpret_cast<const ulonglong2*>(Sm + (sg + 16 * v) * pitch + d);
#pragma unroll
            for (int u = 0; u < 8; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] = fma2(rv[u].x, sv[v].x, acc[u][v]);
#pragma unroll
            for (int u = 0; u < 8; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] = fma2(rv[u].y, sv[v].y, acc[u][v]);
        }

        // Logit arithmetic, identical in both passes: a = dot, then
        //   fp caches:   2^(fma(a, qf, -ref))            (qf = scale * log2 e > 0)
        //   int8 caches: 2^((a * qf) * kf - ref)         (qf with s_q, kf = s_k)
        // A tile wholly inside the causal triangle and the lengths skips the masks.
        const int* spos = s_spos + buf * kStr;
        auto epilogue = [&](auto masked_tag) {
            constexpr bool kMasked = decltype(masked_tag)::value;
            if constexpr (!kCols) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int ipos = s_rpos[rg + 16 * u];
                    if (kMasked && ipos < 0) continue;
                    const float qf = s_rfac[rg + 16 * u];
                    float x[4];
                    bool ok[4];
                    float tmax = -INFINITY;
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const int sr = sg + 16 * v;
                        const float2 f = unpack2(acc[u][v]);
                        x[v] = __fadd_rn(f.x, f.y);
                        if constexpr (kInt8) x[v] = __fmul_rn(__fmul_rn(x[v], qf), s_sfac[buf * kStr + sr]);
                        ok[v] = true;
                        if constexpr (kMasked) {
                            const int kp = spos[sr];
                            ok[v] = kp >= 0 && kp <= ipos;
                        }
                        if (ok[v]) tmax = fmaxf(tmax, x[v]);
                    }
                    if (kMasked && tmax == -INFINITY) continue;
                    if constexpr (!kInt8) tmax = __fmul_rn(tmax, qf);
                    if (tmax > st_a[u]) {
                        st_b[u] *= exp2_approx(st_a[u] - tmax);
                        st_a[u] = tmax;
                    }
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        if (!ok[v]) continue;
                        if constexpr (kInt8) st_b[u] += exp2_approx(x[v] - st_a[u]);
                        else st_b[u] += exp2_approx(fmaf(x[v], qf, -st_a[u]));
                    }
                }
            } else {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int sr = sg + 16 * v;
                    const int ipos = spos[sr];
                    if (kMasked && ipos < 0) continue;
                    const float lse = s_slse[buf * kStr + sr];
                    float qf = a.scale_log2;
                    if constexpr (kInt8) qf = __fmul_rn(s_sfac[buf * kStr + sr], a.scale_log2);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        if constexpr (kMasked) {
                            const int kp = s_rpos[rg + 16 * u];
                            if (kp < 0 || kp > ipos) continue;
                        }
                        const float2 f = unpack2(acc[u][v]);
                        const float x = __fadd_rn(f.x, f.y);
                        if constexpr (kInt8)
                            st_a[u] += exp2_approx(__fmul_rn(__fmul_rn(x, qf), s_rfac[rg + 16 * u]) - lse);
                        else
                            st_a[u] += exp2_approx(fmaf(x, qf, -lse));
                    }
                }
            }
        };
        bool interior;
        if constexpr (!kCols) interior = t * kStr + kStr - 1 <= base && base + kRes / G - 1 < S;
        else interior = base + kRes - 1 <= t * TQs && t * TQs + TQs - 1 < S;
        if (interior) epilogue(std::false_type{});
        else epilogue(std::true_type{});
    }

    // combine the 16 streamed groups of every resident row (scratch: ring)
    __syncthreads();
    float* red_a = s_str;
    float* red_b = s_str + 16 * kRes;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        red_a[sg * kRes + rg + 16 * u] = st_a[u];
        if constexpr (!kCols) red_b[sg * kRes + rg + 16 * u] = st_b[u];
    }
    __syncthreads();
    if (tid < kRes) {
        const int r = tid;
        if constexpr (!kCols) {
            const int i = base + r / G, g = r % G;
            if (i < S) {
                float M = -INFINITY;
#pragma unroll
                for (int j = 0; j < 16; ++j) M = fmaxf(M, red_a[j * kRes + r]);
                float Z = 0.f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float mj = red_a[j * kRes + r];
                    if (mj != -INFINITY) Z += red_b[j * kRes + r] * exp2_approx(mj - M);
                }
                const float l2 = M + log2f(Z);
                a.lse2[bn_rows * a.S_max * G + static_cast<size_t>(i) * G + g] = l2;
                if (a.lse_out)
                    a.lse_out[(static_cast<size_t>(b) * a.H + h0 + g) * a.S_max + i] = l2 * kLn2;
            }
        } else if (base + r < a.S_max) {
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) s += red_a[j * kRes + r];
            a.part[(bn_rows * a.parts + part) * a.S_max + base + r] = s;
        }
    }
}

// importance[b][s] = sum over KV heads (ascending) and parts of the column
// sums for s < S, 0 beyond (and for a request with a bad length).
__global__ void importance_sum_kernel(const Args a) {
    const size_t total = static_cast<size_t>(a.B) * a.S_max;
    for (size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int b = static_cast<int>(idx / a.S_max);
        const int s = static_cast<int>(idx - static_cast<size_t>(b) * a.S_max);
        const int S = a.lens[b];
        float v = 0.f;
        if (S >= 0 && S <= a.S_max &&
            static_cast<long long>(S) <= static_cast<long long>(a.MKBPR) * a.BS && s < S) {
            for (int n = 0; n < a.N; ++n)
                for (int p = 0; p < a.parts; ++p)
                    v += a.part[((static_cast<size_t>(b) * a.N + n) * a.parts + p) * a.S_max + s];
        }
        a.importance[idx] = v;
    }
}

// int8 caches: every prefill query row (b, i, h), i < S, quantised as the
// decode calls quantise their query: s_q = max|q| / 127, q8 = rint(q / s_q)
// (fp32, correctly rounded division), one warp per row.
template <int D>
__global__ void quantize_rows_kernel(const void* q, int q_dt, const int32_t* lens, int B,
                                     int S_max, int H, int8_t* q8, float* s_q) {
    constexpr int PER = D / 32;
    const int lane = threadIdx.x & 31;
    const long long rows = static_cast<long long>(B) * S_max * H;
    const long long warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         row < rows; row += warps) {
        const int b = static_cast<int>(row / (static_cast<long long>(S_max) * H));
        const int i = static_cast<int>((row / H) % S_max);
        if (i >= lens[b]) continue;
        float x[PER];
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            x[j] = load_q(q, q_dt, static_cast<size_t>(row) * D + lane * PER + j);
            amax = fmaxf(amax, fabsf(x[j]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float s = amax == 0.f ? 0.f : __fdiv_rn(amax, 127.f);
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            int v = 0;
            if (s != 0.f) v = min(127, max(-127, __float2int_rn(__fdiv_rn(x[j], s))));
            q8[static_cast<size_t>(row) * D + lane * PER + j] = static_cast<int8_t>(v);
        }
        if (lane == 0) s_q[row] = s;
    }
}

}  // namespace imp
}  // namespace qs

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {

using namespace qs;
using namespace qs::imp;

struct WsPlan {
    int parts, part_tiles;
    size_t lse2, part, q8, s_q, tc, bytes;
};

// Pass 2 splits each key tile's query range into up to kMaxParts parts of
// about 16 streamed tiles, so that the keys near the start of a long prefill
// (seen by every query) do not leave one CTA working long after the rest.
WsPlan plan_ws(long long B, long long H, long long N, long long D, long long S_max, bool int8,
               bool f32) {
    WsPlan w{};
    const long long G = H / N;
    const long long tq = kStr / G;
    const long long qtiles = (S_max + tq - 1) / tq;
    long long parts = (qtiles + 15) / 16;
    if (parts < 1) parts = 1;
    if (parts > kMaxParts) parts = kMaxParts;
    w.parts = static_cast<int>(parts);
    w.part_tiles = static_cast<int>(qtiles > 0 ? (qtiles + parts - 1) / parts : 1);
    size_t off = 0;
    w.lse2 = off;
    off = align_up(off + static_cast<size_t>(B * H * S_max) * 4, 256);
    w.part = off;
    off = align_up(off + static_cast<size_t>(B * N * parts * S_max) * 4, 256);
    w.q8 = off;
    if (int8) off = align_up(off + static_cast<size_t>(B * S_max * H * D), 256);
    w.s_q = off;
    if (int8) off = align_up(off + static_cast<size_t>(B * S_max * H) * 4, 256);
    // tensor-core form: packed operand tiles and its own lse2 rows
    w.tc = off;
    if (!int8) {
        size_t oq, ok, ol;
        off = align_up(off + importance_tc_workspace(B, H, N, D, S_max, f32, &oq, &ok, &ol), 256);
    }
    w.bytes = off > 0 ? off : 256;
    return w;
}

qs_status check_dims(int32_t B, int32_t H, int32_t N, int32_t D, int32_t S_max) {
    if (B < 0 || H <= 0 || N <= 0 || S_max < 0 || H % N != 0) return QS_EINVAL;
    const int G = H / N;
    if (G > 64 || (G & (G - 1)) != 0) return QS_EUNSUPPORTED;
    if (D != 64 && D != 128) return QS_EUNSUPPORTED;
    if ((static_cast<long long>(S_max) + kRes / G - 1) / (kRes / G) > 65535 ||
        (static_cast<long long>(S_max) + kRes - 1) / kRes > 65535)
        return QS_EUNSUPPORTED;
    return QS_OK;
}

template <Dt QT, Dt KT, int D>
bool launch_passes(const Args& a, cudaStream_t st) {
    auto k1 = importance_pass_kernel<QT, KT, D, false>;
    auto k2 = importance_pass_kernel<QT, KT, D, true>;
    constexpr size_t b1 = Layout<QT, KT, D, false>::bytes;
    constexpr size_t b2 = Layout<QT, KT, D, true>::bytes;
    if (!ensure_smem(reinterpret_cast<const void*>(k1), b1) ||
        !ensure_smem(reinterpret_cast<const void*>(k2), b2))
        return false;
    const unsigned rows_tiles = static_cast<unsigned>((a.S_max + kRes / a.G - 1) / (kRes / a.G));
    const unsigned key_tiles = static_cast<unsigned>((a.S_max + kRes - 1) / kRes);
    k1<<<dim3(static_cast<unsigned>(a.B * a.N), rows_tiles), kThreads, b1, st>>>(a);
    k2<<<dim3(static_cast<unsigned>(a.B * a.N * a.parts), key_tiles), kThreads, b2, st>>>(a);
    return true;
}

template <Dt QT, Dt KT>
bool launch_d(int D, const Args& a, cudaStream_t st) {
    return D == 64 ? launch_passes<QT, KT, 64>(a, st) : launch_passes<QT, KT, 128>(a, st);
}

}  // namespace

extern "C" qs_status qs_prefill_importance_workspace_size(int32_t B, int32_t H, int32_t N,
                                                          int32_t D, int32_t S_max,
                                                          qs_dtype kv_dtype, size_t* bytes) {
    if (!bytes) return QS_EINVAL;
    const qs_status rc = check_dims(B, H, N, D, S_max);
    if (rc != QS_OK) return rc;
    *bytes = plan_ws(B, H, N, D, S_max, kv_dtype == QS_I8, kv_dtype == QS_F32).bytes;
    return QS_OK;
}

extern "C" qs_status qs_prefill_importance(const void* q, qs_dtype q_dtype, const void* k_cache,
                                           const float* k_scale, qs_dtype kv_dtype,
                                           int32_t num_kv_blocks, const int32_t* block_tables,
                                           int32_t MKBPR, const int32_t* prefill_lens,
                                           int32_t S_max, int32_t B, int32_t H, int32_t N,
                                           int32_t D, int32_t BS, float softmax_scale,
                                           float* importance, float* lse_opt, void* workspace,
                                           size_t workspace_bytes, int32_t* dev_status,
                                           qs_stream_t stream) {
    const qs_status rc = check_dims(B, H, N, D, S_max);
    if (rc != QS_OK) return rc;
    if (BS <= 0 || MKBPR < 0 || num_kv_blocks < 0 || !std::isfinite(softmax_scale) ||
        !(softmax_scale > 0.f))
        return QS_EINVAL;
    if (B == 0 || S_max == 0) return QS_OK;
    const bool int8 = kv_dtype == QS_I8;
    if (int8) {
        if (q_dtype != QS_F32 && q_dtype != QS_BF16 && q_dtype != QS_F16) return QS_EDTYPE;
        if (!k_scale) return QS_EINVAL;
    } else if ((kv_dtype != QS_F32 && kv_dtype != QS_BF16 && kv_dtype != QS_F16) ||
               q_dtype != kv_dtype) {
        return QS_EDTYPE;
    }
    if (!q || !k_cache || !block_tables || !prefill_lens || !importance || !dev_status)
        return QS_EINVAL;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
         reinterpret_cast<uintptr_t>(workspace)) % 16 != 0)
        return QS_EINVAL;
    const WsPlan w = plan_ws(B, H, N, D, S_max, int8, kv_dtype == QS_F32);
    if (!workspace || workspace_bytes < w.bytes) return QS_EWORKSPACE;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    Args a{};
    a.q = static_cast<const uint8_t*>(int8 ? static_cast<const void*>(ws + w.q8) : q);
    a.s_q = int8 ? reinterpret_cast<const float*>(ws + w.s_q) : nullptr;
    a.k = static_cast<const uint8_t*>(k_cache);
    a.k_scale = k_scale;
    a.bt = block_tables;
    a.lens = prefill_lens;
    a.lse2 = reinterpret_cast<float*>(ws + w.lse2);
    a.part = reinterpret_cast<float*>(ws + w.part);
    a.lse_out = lse_opt;
    a.importance = importance;
    a.status = dev_status;
    a.P = num_kv_blocks;
    a.MKBPR = MKBPR;
    a.S_max = S_max;
    a.B = B;
    a.H = H;
    a.N = N;
    a.G = H / N;
    a.g_shift = __builtin_ctz(static_cast<unsigned>(a.G));
    a.BS = BS;
    a.bs_shift = (BS & (BS - 1)) == 0 ? __builtin_ctz(static_cast<unsigned>(BS)) : -1;
    a.parts = w.parts;
    a.part_tiles = w.part_tiles;
    a.scale_log2 = softmax_scale * kLog2e;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int sms = num_sms();
    if (int8) {
        const long long rows = static_cast<long long>(B) * S_max * H;
        long long grid = (rows + 7) / 8;
        if (grid > static_cast<long long>(sms) * 16) grid = static_cast<long long>(sms) * 16;
        if (D == 64)
            quantize_rows_kernel<64><<<static_cast<unsigned>(grid), 256, 0, st>>>(
                q, q_dtype, prefill_lens, B, S_max, H, reinterpret_cast<int8_t*>(ws + w.q8),
                reinterpret_cast<float*>(ws + w.s_q));
        else
            quantize_rows_kernel<128><<<static_cast<unsigned>(grid), 256, 0, st>>>(
                q, q_dtype, prefill_lens, B, S_max, H, reinterpret_cast<int8_t*>(ws + w.q8),
                reinterpret_cast<float*>(ws + w.s_q));
    }
    bool ok;
    if (int8) {
        ok = launch_d<Dt::I8, Dt::I8>(D, a, st);
    } else {
        const Dt dt = kv_dtype == QS_F32 ? Dt::F32 : kv_dtype == QS_BF16 ? Dt::BF16 : Dt::F16;
        ok = importance_tc_launch(q, dt, k_cache, num_kv_blocks, block_tables, MKBPR, prefill_lens,
                                  S_max, B, H, N, D, BS, a.scale_log2, a.part, w.parts, lse_opt,
                                  ws + w.tc, dev_status, st);
    }
    if (!ok) return QS_ECUDA;
    const size_t total = static_cast<size_t>(B) * S_max;
    long long grid = static_cast<long long>((total + 255) / 256);
    if (grid > static_cast<long long>(sms) * 8) grid = static_cast<long long>(sms) * 8;
    importance_sum_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(a);
    QS_CHECK_LAUNCH();
    return QS_OK;
}
