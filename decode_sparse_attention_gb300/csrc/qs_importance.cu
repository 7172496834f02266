// Prefill importance producer: the attention mass each prefill token
// received, per head, summed over the heads (Kestrel-LLM 10-2, section 1,
// signal 2; section 2, the decode call site that reads prefill_importance).
//
// For request b, KV head n and its G = H/N query heads, the causal logits of
// query row (i, g) against key s <= i are formed twice:
//   pass 1 (rows):    lse2[i,g] = log2 sum_{s<=i} 2^(l2[i,g,s]),
//   pass 2 (columns): mass[s]   = sum_{i>=s, g} 2^(l2[i,g,s] - lse2[i,g]),
// with l2 the logit in base 2.  The passes run on the tensor cores
// (qs_importance_tc.cu) for every cache dtype.  This file holds the entry
// points, the workspace plan, the quantisation of the query rows for int8
// caches (as the decode calls quantise their query) and the last kernel,
// which adds the KV heads' (and query-range parts') column sums per token.
#include <cmath>

#include "qs_internal.cuh"

namespace qs {
namespace imp {

constexpr int kMaxParts = 8;    // query-range parts of the column pass
constexpr int kPartRows = 64;   // query rows per planning tile of the parts
constexpr float kLog2e = 1.4426950408889634f;

struct Args {
    const int32_t* lens;      // [B]
    float* part;              // workspace [B, N, parts, S_max]
    float* importance;        // [B, S_max]
    int MKBPR, S_max, B, N, BS;
    int parts;
};

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
    int parts;
    size_t part, q8, s_q, tc, bytes;
};

// The column pass splits each key tile's query range into up to kMaxParts
// parts, so that the keys near the start of a long prefill (seen by every
// query) do not leave one CTA working long after the rest.
WsPlan plan_ws(long long B, long long H, long long N, long long D, long long S_max, bool int8,
               bool f32) {
    WsPlan w{};
    const long long G = H / N;
    const long long qtiles = (S_max * G + kPartRows - 1) / kPartRows;
    long long parts = (qtiles + 15) / 16;
    if (parts < 1) parts = 1;
    if (parts > kMaxParts) parts = kMaxParts;
    w.parts = static_cast<int>(parts);
    size_t off = 0;
    w.part = off;
    off = align_up(off + static_cast<size_t>(B * N * parts * S_max) * 4, 256);
    w.q8 = off;
    if (int8) off = align_up(off + static_cast<size_t>(B * S_max * H * D), 256);
    w.s_q = off;
    if (int8) off = align_up(off + static_cast<size_t>(B * S_max * H) * 4, 256);
    // the passes' packed operand tiles, row log-sum-exps (and int8 scales)
    w.tc = off;
    {
        size_t oq, ok, ol, oqs, oks;
        off = align_up(off + importance_tc_workspace(B, H, N, D, S_max, f32, int8, &oq, &ok, &ol, &oqs, &oks),
                       256);
    }
    w.bytes = off > 0 ? off : 256;
    return w;
}

qs_status check_dims(int32_t B, int32_t H, int32_t N, int32_t D, int32_t S_max) {
    if (B < 0 || H <= 0 || N <= 0 || S_max < 0 || H % N != 0) return QS_EINVAL;
    const int G = H / N;
    if (G > 64 || (G & (G - 1)) != 0) return QS_EUNSUPPORTED;
    if (D != 64 && D != 128) return QS_EUNSUPPORTED;
    // grid heights of the passes: 128-row query and key tiles
    if ((static_cast<long long>(S_max) * G + 127) / 128 > 65535 ||
        (static_cast<long long>(S_max) + 127) / 128 > 65535)
        return QS_EUNSUPPORTED;
    return QS_OK;
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
    a.lens = prefill_lens;
    a.part = reinterpret_cast<float*>(ws + w.part);
    a.importance = importance;
    a.MKBPR = MKBPR;
    a.S_max = S_max;
    a.B = B;
    a.N = N;
    a.BS = BS;
    a.parts = w.parts;
    const float scale_log2 = softmax_scale * kLog2e;

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
    const Dt dt = int8 ? Dt::I8 : kv_dtype == QS_F32 ? Dt::F32 : kv_dtype == QS_BF16 ? Dt::BF16 : Dt::F16;
    const bool ok = importance_tc_launch(int8 ? static_cast<const void*>(ws + w.q8) : q,
                                         int8 ? reinterpret_cast<const float*>(ws + w.s_q) : nullptr, dt,
                                         k_cache, k_scale, num_kv_blocks, block_tables, MKBPR,
                                         prefill_lens, S_max, B, H, N, D, BS, scale_log2, a.part, w.parts,
                                         lse_opt, ws + w.tc, dev_status, st);
    if (!ok) return QS_ECUDA;
    const size_t total = static_cast<size_t>(B) * S_max;
    long long grid = static_cast<long long>((total + 255) / 256);
    if (grid > static_cast<long long>(sms) * 8) grid = static_cast<long long>(sms) * 8;
    importance_sum_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(a);
    QS_CHECK_LAUNCH();
    return QS_OK;
}
