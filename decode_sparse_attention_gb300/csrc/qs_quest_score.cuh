// Quest block score of one 16-byte slice of a metadata row pair (CANN
// ops-transformer select_attention_operators page, quest_block_select_paged
// step 2.2): sum over the slice's channels d of max(qg_d * max_d, qg_d * min_d),
// qg being the group-mean query in fp32.  Every selector (one CTA per unit,
// the streaming scan, the fused decode step) scores through these helpers, so
// they compute bit-identical scores and therefore identical selections.
#pragma once

#include "qs_common.cuh"

namespace qs {

// Since max_d >= min_d channel by channel, max(q_d * max_d, q_d * min_d) is
// q_d * max_d where q_d >= 0 and q_d * min_d where q_d < 0 (the two products
// are rounded monotonically, so the fp32 maxima agree; only the sign of a zero
// product can differ, and the selection keys fold -0 into +0).  A lane's
// query slice is fixed while it scores many rows, so it is prepared once: the
// channels in fp32 (pairs for 16-bit metadata) and, per 32-bit word of a
// metadata row, a bit mask that picks the max or the min element.  A row
// slice then costs one bitwise select, the widening to fp32 and one fused
// multiply-add per channel pair.
template <Dt T> struct RowChunk;

template <> struct RowChunk<Dt::F32> {
    static constexpr int kElems = 4;
    float q[4];
    uint32_t take_max[4];
    QS_DEVINL void prepare(const float* qg) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            q[i] = qg[i];
            take_max[i] = qg[i] >= 0.f ? 0xffffffffu : 0u;
        }
    }
    QS_DEVINL float dot(uint4 mx, uint4 mn) const {
        const uint32_t a[4] = {mx.x, mx.y, mx.z, mx.w};
        const uint32_t c[4] = {mn.x, mn.y, mn.z, mn.w};
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            s = __fmaf_rn(q[i], __uint_as_float((a[i] & take_max[i]) | (c[i] & ~take_max[i])), s);
        return s;
    }
};

template <Dt T> struct RowChunk16 {
    static constexpr int kElems = 8;
    unsigned long long q2[4];
    uint32_t take_max[4];   // per word: 0xffff in the half whose channel takes max
    QS_DEVINL void prepare(const float* qg) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            q2[i] = pack2(qg[2 * i], qg[2 * i + 1]);
            take_max[i] = (qg[2 * i] >= 0.f ? 0x0000ffffu : 0u) |
                          (qg[2 * i + 1] >= 0.f ? 0xffff0000u : 0u);
        }
    }
    QS_DEVINL float dot(uint4 mx, uint4 mn) const {
        const uint32_t a[4] = {mx.x, mx.y, mx.z, mx.w};
        const uint32_t c[4] = {mn.x, mn.y, mn.z, mn.w};
        unsigned long long acc = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t w = (a[i] & take_max[i]) | (c[i] & ~take_max[i]);
            const float2 f = pair_to_float2<T>(w);
            acc = fma2(q2[i], pack2(f.x, f.y), acc);
        }
        const float2 r = unpack2(acc);
        return r.x + r.y;
    }
};
template <> struct RowChunk<Dt::BF16> : RowChunk16<Dt::BF16> {};
template <> struct RowChunk<Dt::F16> : RowChunk16<Dt::F16> {};

// Group mean of G query values: their sum (in head order) divided by G.  For
// G a power of two the quotient is an exact scaling, computed as a product
// with 2^-log2(G), which gives the same bits as the division.
QS_DEVINL float group_mean(float sum, int G) {
    if ((G & (G - 1)) == 0) return __fmul_rn(sum, __int_as_float((127 - (__ffs(G) - 1)) << 23));
    return __fdiv_rn(sum, static_cast<float>(G));
}

// Sum of a row's slice scores over the kLanesPerRow lanes that hold it
// (butterfly: every lane of the row ends with the full score).
template <int kLanesPerRow>
QS_DEVINL float row_score_reduce(float s) {
#pragma unroll
    for (int o = kLanesPerRow / 2; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

// First forced window block of a request (sink + window forcing of the
// '_in_out_w' variant): blocks from w0 on are newer than the metadata, which
// was built tokens_since_metadata_update = t tokens ago.  Returns nb when the
// window is off (t < 0) or the request is empty.
QS_DEVINL int forced_window_start(int L, int BS, int nb, int t) {
    if (t < 0 || nb <= 0) return nb;
    int w0 = L - t >= 0 ? (L - t) / BS : 0;
    return min(w0, nb - 1);
}
// Number of forced blocks: {0} and [w0, nb).
QS_DEVINL int forced_count(int nb, int w0, int t) {
    return t >= 0 && nb > 0 ? (nb - w0) + (w0 > 0 ? 1 : 0) : 0;
}

}  // namespace qs
