// Quest block score of one 16-byte slice of a metadata row pair (CANN
// ops-transformer select_attention_operators page, quest_block_select_paged
// step 2.2): sum over the slice's channels d of max(qg_d * max_d, qg_d * min_d),
// qg being the group-mean query in fp32.  The standalone selector and the
// fused decode step both score through this one function, so the two
// compute bit-identical scores and therefore identical selections.
#pragma once

#include "qs_common.cuh"

namespace qs {

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
