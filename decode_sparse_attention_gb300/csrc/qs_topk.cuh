// CTA-wide deterministic top-k over keys held in shared memory.
//
// Order: larger key first, equal keys by lower index first, no randomness
// (Kestrel-LLM 10-2 section 1: ties are broken by the block index;
// CANN Quest page step 2.3: top-k over all blocks of the request).
//
// Method: an MSB-first radix select over the 32-bit keys (4 passes of 8-bit
// digits, histograms with warp-aggregated shared-memory atomics) finds the
// k-th largest key T and how many keys equal to T are taken; the picks are
// every candidate key > T plus the first keys == T in index order (a
// CTA-wide prefix count).  The result is a set, returned as flags, so the
// cost is independent of k.
#pragma once

#include "qs_common.cuh"

namespace qs {

enum : uint8_t { kCand = 1, kPick = 2, kFixed = 4 };

template <int NT> struct TopkScratch {
    uint32_t hist[256];
    int warp_sums[NT / 32 + 1];
    uint32_t prefix;
    int remaining;
    int count;
    unsigned long long best;
};

// Exclusive prefix sum of v over the CTA in thread order; total in *total.
template <int NT>
QS_DEVINL int block_exclusive_scan(int v, TopkScratch<NT>& s, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s.warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < NT / 32 ? s.warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < NT / 32) s.warp_sums[lane] = w;
    }
    __syncthreads();
    const int before = warp ? s.warp_sums[warp - 1] : 0;
    *total = s.warp_sums[NT / 32 - 1];
    __syncthreads();
    return before + x - v;
}

// Sets kPick on the top `want` entries among those flagged kCand.
// Requires 0 <= want <= number of candidates.
template <int NT>
QS_DEVINL void topk_flags(const uint32_t* keys, uint8_t* flags, int n, int want,
                          TopkScratch<NT>& s) {
    const int tid = threadIdx.x, lane = tid & 31;
    if (want <= 0) return;
    uint32_t prefix = 0, mask = 0;
    int remaining = want;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = tid; i < 256; i += NT) s.hist[i] = 0;
        __syncthreads();
        for (int base = 0; base < n; base += NT) {
            const int j = base + tid;
            bool ok = false;
            uint32_t digit = 0x100u + lane;
            if (j < n && (flags[j] & kCand)) {
                const uint32_t key = keys[j];
                if ((key & mask) == prefix) {
                    ok = true;
                    digit = (key >> shift) & 0xffu;
                }
            }
            const unsigned peers = __match_any_sync(0xffffffffu, digit);
            if (ok && lane == __ffs(peers) - 1) atomicAdd(&s.hist[digit], __popc(peers));
        }
        __syncthreads();
        if (tid < 32) {
            // lane l owns digits 255-8l ... 248-8l (descending)
            uint32_t c[8];
            uint32_t sum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                c[i] = s.hist[255 - 8 * lane - i];
                sum += c[i];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const uint32_t excl = incl - sum;
            // the lane whose range first reaches `remaining`
            const bool hit = excl < static_cast<uint32_t>(remaining) &&
                             incl >= static_cast<uint32_t>(remaining);
            if (hit) {
                uint32_t above = excl;
                int d = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (above + c[i] >= static_cast<uint32_t>(remaining)) {
                        d = 255 - 8 * lane - i;
                        break;
                    }
                    above += c[i];
                }
                s.prefix = prefix | (static_cast<uint32_t>(d) << shift);
                s.remaining = remaining - static_cast<int>(above);
            }
        }
        __syncthreads();
        prefix = s.prefix;
        remaining = s.remaining;
        mask |= 0xffu << shift;
        __syncthreads();
    }
    // prefix = T (the want-th largest key); take every key > T and the first
    // `remaining` keys == T in index order.
    const int per = (n + NT - 1) / NT;
    const int j0 = min(n, tid * per), j1 = min(n, j0 + per);
    int eq = 0;
    for (int j = j0; j < j1; ++j) eq += (flags[j] & kCand) && keys[j] == prefix;
    int tot;
    int before = block_exclusive_scan<NT>(eq, s, &tot);
    for (int j = j0; j < j1; ++j) {
        if (!(flags[j] & kCand)) continue;
        const uint32_t key = keys[j];
        if (key > prefix) {
            flags[j] |= kPick;
        } else if (key == prefix) {
            if (before < remaining) flags[j] |= kPick;
            ++before;
        }
    }
    __syncthreads();
}

// Writes the indices j with (flags[j] & bits) != 0 in ascending order into
// out[0..k), padding with -1; at most k indices are written.  Returns the
// number of flagged entries (same value in every thread).
template <int NT>
QS_DEVINL int emit_sorted(const uint8_t* flags, uint8_t bits, int n, int k, int32_t* out,
                          TopkScratch<NT>& s) {
    const int tid = threadIdx.x;
    const int per = (n + NT - 1) / NT;
    const int j0 = min(n, tid * per), j1 = min(n, j0 + per);
    int c = 0;
    for (int j = j0; j < j1; ++j) c += (flags[j] & bits) != 0;
    int tot;
    int pos = block_exclusive_scan<NT>(c, s, &tot);
    for (int j = j0; j < j1; ++j)
        if (flags[j] & bits) {
            if (pos < k) out[pos] = j;
            ++pos;
        }
    for (int i = tot + tid; i < k; i += NT) out[i] = -1;
    return tot;
}

// Number of entries with (flags & bits) != 0 (same value in every thread).
template <int NT>
QS_DEVINL int count_flags(const uint8_t* flags, uint8_t bits, int n, TopkScratch<NT>& s) {
    int c = 0;
    for (int j = threadIdx.x; j < n; j += NT) c += (flags[j] & bits) != 0;
    int tot;
    block_exclusive_scan<NT>(c, s, &tot);
    return tot;
}

}  // namespace qs
