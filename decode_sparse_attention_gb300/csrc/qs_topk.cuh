// Deterministic top-k over keys held in shared memory, block-wide and
// one-warp forms.
//
// Order: larger key first, equal keys by lower index first, no randomness
// (Kestrel-LLM 10-2 section 1: ties are broken by the block index;
// CANN Quest page step 2.3: top-k over all blocks of the request).
//
// The result is a set, returned as flags (kPick), so the cost does not grow
// with k; callers emit the picked indices in ascending order.
//
// Every routine runs on all threads of the block (blockDim.x, a multiple of
// 32, at most NT: the template argument only sizes the scratch).
#pragma once

#include "qs_common.cuh"

namespace qs {

enum : uint8_t { kCand = 1, kPick = 2, kFixed = 4 };

// Scratch of a block-wide exclusive scan (one partial per warp).
template <int NT> struct TopkScratch {
    int warp_sums[NT / 32 + 1];
};

// Exclusive prefix sum of v over the CTA in thread order; total in *total.
template <int NT>
QS_DEVINL int block_exclusive_scan(int v, TopkScratch<NT>& s, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = static_cast<int>(blockDim.x) >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s.warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? s.warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < nw) s.warp_sums[lane] = w;
    }
    __syncthreads();
    const int before = warp ? s.warp_sums[warp - 1] : 0;
    *total = s.warp_sums[nw - 1];
    __syncthreads();
    return before + x - v;
}

QS_DEVINL unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// ---------------------------------------------------------------------------
// Histogram top-k: MSB-first radix selection with 8-bit digits below the
// candidates' common key prefix.  Each level builds a 256-bin histogram of
// the digit over the keys still in play (shared-memory atomics, one copy of
// the bins per warp of a group of eight, summed by the scan), one warp
// finds the digit that holds the want-th key, keys with a larger digit are
// taken, and the boundary digit is refined with the next 8 bits until at
// most kListMax keys remain in it; those are ranked exactly (key descending,
// lower index first) by four threads per key.  If all 32 bits get fixed, the
// remaining keys are equal and the lowest indices are taken.  Four block
// barriers per level; usually one or two levels.
// ---------------------------------------------------------------------------

constexpr int kHistBins = 256;
constexpr int kHistCopies = 8;   // at most; warp w counts into copy w % copies

// Histogram copies for n keys: more warps contending on a few crowded bins
// pay for more copies; few keys do not pay for clearing and summing them.
QS_DEVINL int topk_hist_copies(int n) { return n <= 128 ? 1 : (n <= 512 ? 4 : kHistCopies); }
constexpr int kListMax = 64;

struct TopkFastScratch {
    __align__(16) uint32_t hist[kHistCopies][kHistBins];
    uint32_t list_key[kListMax];
    int list_idx[kListMax];
    uint32_t wmax[32], wmin[32];
    int wcnt[32];
    int nlist, dstar, remaining, inbin;
};

// Clears the histogram copies a top-k over n keys uses; call before
// topk_fast with a barrier in between (the callers' next phase provides it).
template <int NT>
QS_DEVINL void topk_fast_clear(TopkFastScratch& s, int n) {
    const int words = topk_hist_copies(n) * kHistBins;
    for (int i = threadIdx.x; i < words; i += blockDim.x) (&s.hist[0][0])[i] = 0;
    if (threadIdx.x == 0) s.nlist = 0;
}

// Value of an order-preserving key (the inverse of float_key; -0 was folded).
QS_DEVINL float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Candidate count and key range (one barrier).
template <int NT>
QS_DEVINL void topk_range(const uint32_t* keys, const uint8_t* flags, int n, TopkFastScratch& s,
                          uint32_t* kmax_out, uint32_t* kmin_out, int* ncand_out) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NT_ = static_cast<int>(blockDim.x), NW = NT_ >> 5;
    uint32_t lmax = 0, lmin = 0xffffffffu;
    int lc = 0;
    for (int j = tid; j < n; j += NT_)
        if (flags[j] & kCand) {
            const uint32_t k = keys[j];
            lmax = max(lmax, k);
            lmin = min(lmin, k);
            ++lc;
        }
    lmax = __reduce_max_sync(0xffffffffu, lmax);
    lmin = __reduce_min_sync(0xffffffffu, lmin);
    lc = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(lc)));
    if (lane == 0) {
        s.wmax[warp] = lmax;
        s.wmin[warp] = lmin;
        s.wcnt[warp] = lc;
    }
    __syncthreads();
    const uint32_t a = lane < NW ? s.wmax[lane] : 0u;
    const uint32_t b = lane < NW ? s.wmin[lane] : 0xffffffffu;
    const int c = lane < NW ? s.wcnt[lane] : 0;
    *kmax_out = __reduce_max_sync(0xffffffffu, a);
    *kmin_out = __reduce_min_sync(0xffffffffu, b);
    *ncand_out = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(c)));
    // (a second call rewrites the warp partials only after further barriers)
}

// Warp 0: the digit (bin) holding the remaining-th key from the top of the
// histogram copies; stores it, the count still wanted inside it, and its size.
QS_DEVINL void topk_boundary(TopkFastScratch& s, int remaining, int copies) {
    const int lane = threadIdx.x & 31;
    const int d_hi = kHistBins - 1 - 8 * lane;      // lane's bins d_hi .. d_hi-7
    uint4 h0 = make_uint4(0, 0, 0, 0), h1 = make_uint4(0, 0, 0, 0);
    for (int cp = 0; cp < copies; ++cp) {
        const uint4 a0 = *reinterpret_cast<const uint4*>(&s.hist[cp][d_hi - 7]);
        const uint4 a1 = *reinterpret_cast<const uint4*>(&s.hist[cp][d_hi - 3]);
        h0.x += a0.x; h0.y += a0.y; h0.z += a0.z; h0.w += a0.w;
        h1.x += a1.x; h1.y += a1.y; h1.z += a1.z; h1.w += a1.w;
    }
    const int cnt[8] = {static_cast<int>(h1.w), static_cast<int>(h1.z), static_cast<int>(h1.y),
                        static_cast<int>(h1.x), static_cast<int>(h0.w), static_cast<int>(h0.z),
                        static_cast<int>(h0.y), static_cast<int>(h0.x)};   // descending bins
    int c = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) c += cnt[i];
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const int excl = incl - c;
    if (excl < remaining && incl >= remaining) {
        int above = excl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (above + cnt[i] >= remaining) {
                s.dstar = d_hi - i;
                s.remaining = remaining - above;
                s.inbin = cnt[i];
                break;
            }
            above += cnt[i];
        }
    }
}

// Exact ranks (key descending, lower index first) of the listed keys, four
// threads per key; the first `remaining` are picked.  Ends with a barrier.
QS_DEVINL void topk_rank_list(TopkFastScratch& s, uint8_t* flags, int remaining) {
    const int tid = threadIdx.x;
    const int nlist = s.nlist;
    const int e = tid >> 2, part = tid & 3;
    int rank = 0;
    uint32_t ke = 0;
    int ie = 0;
    if (e < nlist) {
        ke = s.list_key[e];
        ie = s.list_idx[e];
        for (int f = part; f < nlist; f += 4) {
            const uint32_t kf = s.list_key[f];
            rank += kf > ke || (kf == ke && s.list_idx[f] < ie);
        }
    }
    rank += __shfl_xor_sync(0xffffffffu, rank, 1);
    rank += __shfl_xor_sync(0xffffffffu, rank, 2);
    if (part == 0 && e < nlist && rank < remaining) flags[ie] |= kPick;
    __syncthreads();
}

// Sets kPick on the top `want` entries among those flagged kCand (keys and
// flags in shared memory).  Requires the histogram cleared beforehand and at
// least 4 * kListMax threads.  May clear kCand on entries it settles.
//
// Level 0 (from kValueLevelMin candidates up) buckets the candidates
// linearly by value over [min, max] (256 buckets; monotonic, so bucket order
// is key order): for typical score distributions the keys spread over the
// bins, where 8-bit digits of the order-preserving keys crowd into a few
// exponent bins and their shared-memory atomics serialise.  If the boundary
// bucket is too crowded, or the values are not finite, the exact bit
// refinement below takes over on the keys still undecided.  Measured on
// GB300 (64 CTAs of 256 threads, with emission): 512 keys 2.3-3.6 us and
// 1024 keys 3.0-4.0 us against 2.6-3.5 and 3.6-5.3 us without it; at 128
// keys the bit levels alone were as fast or faster.
constexpr int kValueLevelMin = 256;
template <int NT>
QS_DEVINL void topk_fast(const uint32_t* keys, uint8_t* flags, int n, int want,
                         TopkFastScratch& s, TopkScratch<NT>& rs) {
    const int tid = threadIdx.x, warp = tid >> 5;
    const int NT_ = static_cast<int>(blockDim.x);   // <= NT
    if (want <= 0) return;
    const int copies = topk_hist_copies(n);
    const int wcopy = warp % copies;
    uint32_t kmax, kmin;
    int ncand;
    topk_range<NT>(keys, flags, n, s, &kmax, &kmin, &ncand);
    if (want >= ncand) {          // everything goes
        for (int j = tid; j < n; j += NT_)
            if (flags[j] & kCand) flags[j] |= kPick;
        __syncthreads();
        return;
    }
    int remaining = want;
    {
        const float vmax = key_value(kmax), vmin = key_value(kmin);
        const float span = __fsub_rn(vmax, vmin);
        const float scale = __fdiv_rn(static_cast<float>(kHistBins), span);
        if (ncand >= kValueLevelMin && span > 0.f && isfinite(span) && isfinite(scale) &&
            scale > 0.f) {
            auto bucket = [&](uint32_t key) {
                const float x = __fmul_rn(__fsub_rn(key_value(key), vmin), scale);
                return min(kHistBins - 1, max(0, static_cast<int>(x)));
            };
            for (int j = tid; j < n; j += NT_)
                if (flags[j] & kCand) atomicAdd(&s.hist[wcopy][bucket(keys[j])], 1u);
            __syncthreads();
            if (warp == 0) topk_boundary(s, remaining, copies);
            __syncthreads();
            const int dstar = s.dstar;
            const int rem = s.remaining;
            const int inbin = s.inbin;
            const bool settled = inbin == rem || inbin <= kListMax;
            for (int j = tid; j < n; j += NT_) {
                const uint8_t f = flags[j];
                if (!(f & kCand)) continue;
                const int bk = bucket(keys[j]);
                if (bk > dstar) {
                    flags[j] = static_cast<uint8_t>((f & ~kCand) | kPick);
                } else if (bk < dstar) {
                    flags[j] = static_cast<uint8_t>(f & ~kCand);
                } else if (inbin == rem) {
                    flags[j] = static_cast<uint8_t>(f | kPick);
                } else if (inbin <= kListMax) {
                    const int pos = atomicAdd(&s.nlist, 1);
                    s.list_key[pos] = keys[j];
                    s.list_idx[pos] = j;
                }
            }
            if (!settled)
                for (int i = tid; i < copies * kHistBins; i += NT_) (&s.hist[0][0])[i] = 0;
            __syncthreads();
            if (settled) {
                if (inbin != rem) topk_rank_list(s, flags, rem);
                return;
            }
            // a crowded boundary bucket: refine its keys exactly by bits
            remaining = rem;
            topk_range<NT>(keys, flags, n, s, &kmax, &kmin, &ncand);
        }
    }
    // keys in play: candidates whose bits under pmask equal prefix
    const uint32_t diff = kmax ^ kmin;
    int hi = diff ? 31 - __clz(diff) : -1;              // highest bit not yet fixed
    uint32_t pmask = hi < 0 ? 0xffffffffu : (hi >= 31 ? 0u : ~((2u << hi) - 1u));
    uint32_t prefix = kmax & pmask;
    while (hi >= 0) {
        const int lo = hi >= 7 ? hi - 7 : 0;
        const uint32_t dmask = (2u << (hi - lo)) - 1u;
        // histogram of the digit over the keys in play (the bins are clear);
        // each warp counts into its own copy (same-address atomics serialise;
        // measured on GB300, warp-aggregating them with match_any was slower)
        for (int j = tid; j < n; j += NT_)
            if ((flags[j] & kCand) && (keys[j] & pmask) == prefix)
                atomicAdd(&s.hist[wcopy][(keys[j] >> lo) & dmask], 1u);
        __syncthreads();
        if (warp == 0) topk_boundary(s, remaining, copies);
        __syncthreads();
        const uint32_t dstar = static_cast<uint32_t>(s.dstar);
        remaining = s.remaining;
        const int inbin = s.inbin;
        // digits above the boundary are taken; the boundary digit is listed
        // when it is small; the bins are cleared for a next level
        const bool last_level = inbin == remaining || inbin <= kListMax;
        for (int j = tid; j < n; j += NT_)
            if ((flags[j] & kCand) && (keys[j] & pmask) == prefix) {
                const uint32_t d = (keys[j] >> lo) & dmask;
                if (d > dstar) {
                    flags[j] |= kPick;
                } else if (d == dstar) {
                    if (inbin == remaining) {
                        flags[j] |= kPick;
                    } else if (inbin <= kListMax) {
                        const int pos = atomicAdd(&s.nlist, 1);
                        s.list_key[pos] = keys[j];
                        s.list_idx[pos] = j;
                    }
                }
            }
        if (!last_level)
            for (int i = tid; i < copies * kHistBins; i += NT_) (&s.hist[0][0])[i] = 0;
        __syncthreads();
        if (last_level) {
            if (inbin != remaining) topk_rank_list(s, flags, remaining);
            return;
        }
        prefix |= dstar << lo;
        pmask |= dmask << lo;
        hi = lo - 1;
    }
    // every bit fixed: the keys in play are equal; take the lowest indices
    const int per = (n + NT_ - 1) / NT_;
    const int j0 = min(n, tid * per), j1 = min(n, j0 + per);
    int eq = 0;
    for (int j = j0; j < j1; ++j) eq += (flags[j] & kCand) && keys[j] == prefix;
    int tot;
    int before = block_exclusive_scan<NT>(eq, rs, &tot);
    for (int j = j0; j < j1; ++j)
        if ((flags[j] & kCand) && keys[j] == prefix) {
            if (before < remaining) flags[j] |= kPick;
            ++before;
        }
    __syncthreads();
}

// Largest unit the probe selector ranks with the counting top-k in one pass
// over its heads (larger units take the histogram levels, one head at a time).
constexpr int kProbeRankMax = 256;

// Counting top-k over `sets` independent key arrays at once, all threads of
// the block: entry i of set s is picked when it is a candidate and fewer than
// `want` candidates of its set precede it (a larger key, or an equal key at
// a lower index).  Set s has its keys at mkeys + s * kstride and its flags at
// flags + s * fstride; mkeys holds 0 for every entry that is not a
// candidate (candidate keys are never 0), so the rank loop reads no flags.
// The key arrays are read with 16-byte loads: kstride and the arrays' start
// are multiples of 4 words, and entries n .. round_up(n, 4) - 1 must hold 0.
// Every entry of a 16-byte group is compared with one threshold: key_i - 1
// for groups before i's group (an equal key at a lower index precedes),
// key_i from i's group on; the entries of i's own group before i that equal
// key_i are added afterwards.  The cost grows with sets * n * n: callers keep
// sets * n within kRankMaxPerThread keys per thread.  Each key is ranked by
// `parts` threads (a power of two, up to 8) that split the comparisons; no
// barrier inside (callers order the key writes before and the flag reads
// after with their own).
constexpr int kRankMaxPerThread = 4;
template <int NT>
QS_DEVINL void block_rank_topk(const uint32_t* mkeys, int kstride, uint8_t* flags, int fstride,
                               int n, int sets, int want) {
    const int NT_ = static_cast<int>(blockDim.x);
    const int pairs = sets * n;
    int parts = 1;
    while (parts < 8 && pairs * parts * 2 <= NT_) parts <<= 1;
    const int nq = (n + 3) >> 2;                      // 16-byte groups of keys
    for (int base = 0; base < pairs * parts; base += NT_) {
        const int t = base + static_cast<int>(threadIdx.x);
        const int e = t / parts, part = t - e * parts;  // parts consecutive lanes per key
        const bool live = e < pairs;
        const int s = live ? e / n : 0, i = live ? e - s * n : 0;
        const uint32_t* ks = mkeys + static_cast<size_t>(s) * kstride;
        const uint32_t ki = live ? ks[i] : 0u;
        int rank = 0;
        if (ki != 0u) {
            const uint32_t lo = ki - 1u;
            const int gi = i >> 2;
            int r0 = 0, r1 = 0;
            int g = part;
            for (; g + parts < nq; g += 2 * parts) {   // two groups per step, two sums
                const uint4 a = *reinterpret_cast<const uint4*>(ks + 4 * g);
                const uint4 b = *reinterpret_cast<const uint4*>(ks + 4 * (g + parts));
                const uint32_t ta = g < gi ? lo : ki, tb = g + parts < gi ? lo : ki;
                r0 += (a.x > ta) + (a.y > ta) + (a.z > ta) + (a.w > ta);
                r1 += (b.x > tb) + (b.y > tb) + (b.z > tb) + (b.w > tb);
            }
            if (g < nq) {
                const uint4 a = *reinterpret_cast<const uint4*>(ks + 4 * g);
                const uint32_t ta = g < gi ? lo : ki;
                r0 += (a.x > ta) + (a.y > ta) + (a.z > ta) + (a.w > ta);
            }
            rank = r0 + r1;
            if (gi % parts == part) {   // i's group: equal keys before i precede too
                const int ri = i & 3;
                const uint32_t* kg = ks + 4 * gi;
                rank += (0 < ri && kg[0] == ki) + (1 < ri && kg[1] == ki) + (2 < ri && kg[2] == ki);
            }
        }
        for (int o = 1; o < parts; o <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
        if (live && part == 0 && ki != 0u && rank < want)
            flags[static_cast<size_t>(s) * fstride + i] |= kPick;
    }
}

// One warp writes the indices j with (flags[j] & bits) in ascending order
// into out[0..k), -1 padded; returns their number (in every lane).
QS_DEVINL int warp_emit_flags(const uint8_t* flags, uint8_t bits, int n, int k, int32_t* out) {
    const int lane = threadIdx.x & 31;
    const unsigned below = lanemask_lt();
    int base = 0;
    for (int j0 = 0; j0 < n; j0 += 32) {
        const int j = j0 + lane;
        const bool e = j < n && (flags[j] & bits);
        const unsigned em = __ballot_sync(0xffffffffu, e);
        const int pos = base + __popc(em & below);
        if (e && pos < k) out[pos] = j;
        base += __popc(em);
    }
    for (int p = base + lane; p < k; p += 32) out[p] = -1;
    return base;
}

// All threads write the indices j with (flags[j] & bits) in ascending order
// into out[0..k), -1 padded: one warp's ballots up to 256 entries, a block
// prefix count over contiguous slices above that.
template <int NT>
QS_DEVINL void block_emit_flags(const uint8_t* flags, uint8_t bits, int n, int k, int32_t* out,
                                TopkScratch<NT>& rs) {
    const int tid = threadIdx.x, NT_ = static_cast<int>(blockDim.x);
    if (n <= 256) {
        if (tid < 32) warp_emit_flags(flags, bits, n, k, out);
        return;
    }
    const int per = (n + NT_ - 1) / NT_;
    const int j0 = min(n, tid * per), j1 = min(n, j0 + per);
    int c = 0;
    for (int j = j0; j < j1; ++j) c += (flags[j] & bits) != 0;
    int tot;
    int pos = block_exclusive_scan<NT>(c, rs, &tot);
    for (int j = j0; j < j1; ++j)
        if (flags[j] & bits) {
            if (pos < k) out[pos] = j;
            ++pos;
        }
    for (int i = tot + tid; i < k; i += NT_) out[i] = -1;
}

}  // namespace qs

namespace qs {

// ---------------------------------------------------------------------------
// One-warp top-k over keys in shared memory (no block barriers, so several
// warps can select for different units at once).  Same order as above: key
// descending, equal keys by lower index.  MSB-first radix selection with
// 8-bit digits below the candidates' common prefix: a warp-private 256-bin
// histogram finds the digit holding the want-th key; digits above it are
// taken; the boundary digit is refined with the next 8 bits until at most
// kWarpListMax keys remain in it, which are then ranked exactly (or, once
// all 32 bits are fixed, the remaining equal keys are taken in index order).
// ---------------------------------------------------------------------------

constexpr int kWarpListMax = 64;

struct WarpTopkScratch {
    __align__(16) uint32_t hist[kHistBins];
    uint32_t list_key[kWarpListMax];
    int list_idx[kWarpListMax];
};

// Sets kPick on the top `want` entries among those flagged kCand; called by
// all 32 lanes of one warp.
QS_DEVINL void warp_topk_smem(const uint32_t* keys, uint8_t* flags, int n, int want,
                              WarpTopkScratch& w) {
    const int lane = threadIdx.x & 31;
    const unsigned below = lanemask_lt();
    if (want <= 0) return;
    uint32_t kmax = 0, kmin = 0xffffffffu;
    int c = 0;
    for (int j = lane; j < n; j += 32)
        if (flags[j] & kCand) {
            const uint32_t k = keys[j];
            kmax = max(kmax, k);
            kmin = min(kmin, k);
            ++c;
        }
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    c = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(c)));
    if (want >= c) {
        for (int j = lane; j < n; j += 32)
            if (flags[j] & kCand) flags[j] |= kPick;
        __syncwarp();
        return;
    }
    // keys still in play: candidates whose bits under pmask equal prefix
    const uint32_t diff = kmax ^ kmin;
    int hi = diff ? 31 - __clz(diff) : -1;            // highest bit not yet fixed
    uint32_t pmask = hi < 0 ? 0xffffffffu : (hi >= 31 ? 0u : ~((2u << hi) - 1u));
    uint32_t prefix = kmax & pmask;
    int remaining = want;
    while (hi >= 0) {
        const int lo = hi >= 7 ? hi - 7 : 0;
        const uint32_t dmask = (2u << (hi - lo)) - 1u;
        for (int i = lane; i < kHistBins; i += 32) w.hist[i] = 0;
        __syncwarp();
        for (int j = lane; j < n; j += 32)
            if ((flags[j] & kCand) && (keys[j] & pmask) == prefix)
                atomicAdd(&w.hist[(keys[j] >> lo) & dmask], 1u);
        __syncwarp();
        // boundary digit: lane l sums digits 255-8l .. 248-8l (descending)
        const int d_hi = kHistBins - 1 - 8 * lane;
        const uint4 h0 = *reinterpret_cast<const uint4*>(&w.hist[d_hi - 7]);
        const uint4 h1 = *reinterpret_cast<const uint4*>(&w.hist[d_hi - 3]);
        const int cnt[8] = {static_cast<int>(h1.w), static_cast<int>(h1.z), static_cast<int>(h1.y),
                            static_cast<int>(h1.x), static_cast<int>(h0.w), static_cast<int>(h0.z),
                            static_cast<int>(h0.y), static_cast<int>(h0.x)};
        int sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) sum += cnt[i];
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int excl = incl - sum;
        int dsel = -1, above = 0, inbin = 0;
        if (excl < remaining && incl >= remaining) {
            int acc = excl;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (dsel < 0 && acc + cnt[i] >= remaining) {
                    dsel = d_hi - i;
                    above = acc;
                    inbin = cnt[i];
                }
                if (dsel < 0) acc += cnt[i];
            }
        }
        const unsigned who = __ballot_sync(0xffffffffu, dsel >= 0);
        const int src = __ffs(who) - 1;
        const uint32_t dstar = static_cast<uint32_t>(__shfl_sync(0xffffffffu, dsel, src));
        above = __shfl_sync(0xffffffffu, above, src);
        inbin = __shfl_sync(0xffffffffu, inbin, src);
        // digits above the boundary are taken
        for (int j = lane; j < n; j += 32)
            if ((flags[j] & kCand) && (keys[j] & pmask) == prefix && ((keys[j] >> lo) & dmask) > dstar)
                flags[j] |= kPick;
        remaining -= above;
        prefix |= dstar << lo;
        pmask |= dmask << lo;
        if (inbin == remaining) {          // the whole boundary digit goes
            for (int j = lane; j < n; j += 32)
                if ((flags[j] & kCand) && (keys[j] & pmask) == prefix) flags[j] |= kPick;
            __syncwarp();
            return;
        }
        if (inbin <= kWarpListMax) {       // rank the few keys left exactly
            int base = 0;
            for (int j0 = 0; j0 < n; j0 += 32) {
                const int j = j0 + lane;
                const bool in = j < n && (flags[j] & kCand) && (keys[j] & pmask) == prefix;
                const unsigned m = __ballot_sync(0xffffffffu, in);
                if (in) {
                    const int pos = base + __popc(m & below);
                    w.list_key[pos] = keys[j];
                    w.list_idx[pos] = j;
                }
                base += __popc(m);
            }
            __syncwarp();
            for (int e = lane; e < inbin; e += 32) {
                const uint32_t ke = w.list_key[e];
                int rank = 0;
                for (int f = 0; f < inbin; ++f) {
                    const uint32_t kf = w.list_key[f];
                    rank += kf > ke || (kf == ke && f < e);   // the list is in index order
                }
                if (rank < remaining) flags[w.list_idx[e]] |= kPick;
            }
            __syncwarp();
            return;
        }
        hi = lo - 1;
    }
    // every bit fixed: the keys in play are equal; take the lowest indices
    int taken = 0;
    for (int j0 = 0; j0 < n && taken < remaining; j0 += 32) {
        const int j = j0 + lane;
        const bool in = j < n && (flags[j] & kCand) && keys[j] == prefix;
        const unsigned m = __ballot_sync(0xffffffffu, in);
        if (in && taken + __popc(m & below) < remaining) flags[j] |= kPick;
        taken += __popc(m);
    }
    __syncwarp();
}

}  // namespace qs
