// Quest metadata build: per KV block and KV head, the channel-wise max and min
// of K over the block's valid tokens, packed into paged metadata blocks whose
// unused tail rows are zero (CANN ops-transformer select_attention_operators,
// section 'quest_prefill_metadata: metadata construction').
//
// GB300 design: the op is a streaming reduction over the whole K cache.  One
// CTA reduces one in-sequence KV block for ALL heads at once, so every token
// row it reads is one contiguous N*D run (2 KB at N=8, D=128, bf16), read with
// 128-bit streaming loads, 8 in flight per thread.  Max/min run on integer
// keys (sign-magnitude -> two's complement), which is exact, independent of
// the reduction order, and orders -0 below +0.
#include "qs_common.cuh"

namespace qs {
namespace {

constexpr int kUnroll = 8;

// Integer-ordered view of a float element: key(-x) < key(+0) < key(x>0).  The
// map is its own inverse.
template <Dt T> struct KeyOps;

template <> struct KeyOps<Dt::F32> {
    static QS_DEVINL uint32_t to_key(uint32_t u) {
        return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) & 0x7fffffffu);
    }
    static QS_DEVINL uint32_t vmax(uint32_t a, uint32_t b) {
        return static_cast<uint32_t>(max(static_cast<int32_t>(a), static_cast<int32_t>(b)));
    }
    static QS_DEVINL uint32_t vmin(uint32_t a, uint32_t b) {
        return static_cast<uint32_t>(min(static_cast<int32_t>(a), static_cast<int32_t>(b)));
    }
    static constexpr uint32_t kLowest = 0x80000000u;   // INT32_MIN
    static constexpr uint32_t kHighest = 0x7fffffffu;  // INT32_MAX
};

// Two 16-bit (bf16 / fp16) elements per word, compared as signed halves.
struct KeyOps16 {
    static QS_DEVINL uint32_t to_key(uint32_t w) {
        uint32_t s = (w >> 15) & 0x00010001u;
        return w ^ (s * 0x7fffu);
    }
    static QS_DEVINL uint32_t vmax(uint32_t a, uint32_t b) {
        uint32_t d;
        asm("max.s16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    }
    static QS_DEVINL uint32_t vmin(uint32_t a, uint32_t b) {
        uint32_t d;
        asm("min.s16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    }
    static constexpr uint32_t kLowest = 0x80008000u;
    static constexpr uint32_t kHighest = 0x7fff7fffu;
};
template <> struct KeyOps<Dt::BF16> : KeyOps16 {};
template <> struct KeyOps<Dt::F16> : KeyOps16 {};

template <Dt T>
QS_DEVINL void reduce_vec(uint4 v, uint4& mx, uint4& mn) {
    using K = KeyOps<T>;
    uint32_t a[4] = {v.x, v.y, v.z, v.w};
    uint32_t* pmx = &mx.x;
    uint32_t* pmn = &mn.x;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t k = K::to_key(a[i]);
        pmx[i] = K::vmax(pmx[i], k);
        pmn[i] = K::vmin(pmn[i], k);
    }
}

template <Dt T>
QS_DEVINL uint4 from_keys(uint4 k) {
    using K = KeyOps<T>;
    return make_uint4(K::to_key(k.x), K::to_key(k.y), K::to_key(k.z), K::to_key(k.w));
}

// NT threads: 256 for the prefill (many items per launch), 1024 for the
// incremental update (a few rows per request, so each row gets more token
// groups in flight).
template <Dt T, int NT>
__global__ void __launch_bounds__(NT)
prefill_metadata_kernel(const uint8_t* __restrict__ k_cache, int num_kv_blocks, int BS, int vpr,
                        const int32_t* __restrict__ prev_lens, const int32_t* __restrict__ seq_lens,
                        int B,
                        const int32_t* __restrict__ block_tables, int MKBPR,
                        const int32_t* __restrict__ meta_tables, int MMBPR, int num_meta,
                        uint8_t* __restrict__ maxblocks, uint8_t* __restrict__ minblocks,
                        int32_t* dev_status) {
    using K = KeyOps<T>;
    extern __shared__ uint4 smem[];  // [groups][vpr] max, then [groups][vpr] min
    const size_t row_bytes = static_cast<size_t>(vpr) * 16;
    const int groups = vpr >= NT ? 1 : NT / vpr;
    uint4* s_max = smem;
    uint4* s_min = smem + static_cast<size_t>(groups) * min(vpr, NT);
    const int slots = MMBPR * BS;
    const long long items = static_cast<long long>(B) * slots;

    // one (request, in-sequence block slot) item: reduce the block or zero
    // its row; returns early where the item needs nothing
    auto item = [&](int b, int j) {
        const int L = seq_lens[b];
        if (L < 0 || L > MKBPR * BS) {
            if (j == 0 && threadIdx.x == 0) set_status(dev_status, QS_DEV_ESEQ_LEN);
            return;
        }
        const int nb = (L + BS - 1) / BS;
        const int n_meta = (nb + BS - 1) / BS;
        if (j >= n_meta * BS) return;  // metadata slot the request does not use
        const int m = meta_tables[static_cast<size_t>(b) * MMBPR + j / BS];
        if (m < 0 || m >= num_meta) {
            if (threadIdx.x == 0) set_status(dev_status, QS_DEV_EMETA_TABLE);
            return;
        }
        const size_t out_off = (static_cast<size_t>(m) * BS + j % BS) * row_bytes;
        if (j >= nb) {  // block beyond the sequence: zero row (all heads)
            for (int v = threadIdx.x; v < vpr; v += NT) {
                stg_v4(maxblocks + out_off + static_cast<size_t>(v) * 16, make_uint4(0, 0, 0, 0));
                stg_v4(minblocks + out_off + static_cast<size_t>(v) * 16, make_uint4(0, 0, 0, 0));
            }
            return;
        }
        const int p = block_tables[static_cast<size_t>(b) * MKBPR + j];
        if (p < 0 || p >= num_kv_blocks) {
            if (threadIdx.x == 0) set_status(dev_status, QS_DEV_EBLOCK_TABLE);
            return;
        }
        const int valid = min(BS, L - j * BS);
        const uint8_t* blk = k_cache + static_cast<size_t>(p) * BS * row_bytes;

        for (int v0 = 0; v0 < vpr; v0 += NT) {
            // thread -> (token group g, vector v) for this slice of the row
            const int span = min(vpr - v0, NT);
            const int g = groups > 1 ? threadIdx.x / vpr : 0;
            const int v = groups > 1 ? threadIdx.x % vpr : threadIdx.x;
            const bool active = v < span && g < groups;
            uint4 mx = make_uint4(K::kLowest, K::kLowest, K::kLowest, K::kLowest);
            uint4 mn = make_uint4(K::kHighest, K::kHighest, K::kHighest, K::kHighest);
            if (active) {
                const uint8_t* src = blk + static_cast<size_t>(v0 + v) * 16;
                int t = g;
                for (; t + (kUnroll - 1) * groups < valid; t += kUnroll * groups) {
                    uint4 r[kUnroll];
#pragma unroll
                    for (int u = 0; u < kUnroll; ++u)
                        r[u] = ldg_stream(src + static_cast<size_t>(t + u * groups) * row_bytes);
#pragma unroll
                    for (int u = 0; u < kUnroll; ++u) reduce_vec<T>(r[u], mx, mn);
                }
                for (; t < valid; t += groups)
                    reduce_vec<T>(ldg_stream(src + static_cast<size_t>(t) * row_bytes), mx, mn);
            }
            if (groups > 1) {
                if (active) {
                    s_max[g * span + v] = mx;
                    s_min[g * span + v] = mn;
                }
                __syncthreads();
                if (active && g == 0) {
                    for (int gg = 1; gg < groups; ++gg) {
                        uint4 a = s_max[gg * span + v], c = s_min[gg * span + v];
                        mx.x = K::vmax(mx.x, a.x); mx.y = K::vmax(mx.y, a.y);
                        mx.z = K::vmax(mx.z, a.z); mx.w = K::vmax(mx.w, a.w);
                        mn.x = K::vmin(mn.x, c.x); mn.y = K::vmin(mn.y, c.y);
                        mn.z = K::vmin(mn.z, c.z); mn.w = K::vmin(mn.w, c.w);
                    }
                }
                __syncthreads();
            }
            if (active && g == 0) {
                const size_t o = out_off + static_cast<size_t>(v0 + v) * 16;
                stg_v4(maxblocks + o, from_keys<T>(mx));
                stg_v4(minblocks + o, from_keys<T>(mn));
            }
        }
        };
    if (prev_lens) {
        // incremental update: per request, the rows of the blocks touched
        // since prev_lens (the block that held the last tokens and every
        // block begun since) and the zero rows of meta blocks begun since
        // (rows past the block count in meta blocks already in use are zero
        // from the earlier build)
        for (int b = blockIdx.x; b < B; b += gridDim.x) {
            const int L = seq_lens[b], P0 = prev_lens[b];
            if (L < 0 || L > MKBPR * BS || P0 < 0 || P0 > L) {
                if (threadIdx.x == 0) set_status(dev_status, QS_DEV_ESEQ_LEN);
                continue;
            }
            const int nb = (L + BS - 1) / BS;
            const int rows = (nb + BS - 1) / BS * BS;
            const int zero_from = max(nb, ((P0 + BS - 1) / BS + BS - 1) / BS * BS);
            for (int j = P0 / BS; j < rows; ++j)
                if (j < nb || j >= zero_from) item(b, j);
        }
        return;
    }
    for (long long it = blockIdx.x; it < items; it += gridDim.x)
        item(static_cast<int>(it / slots), static_cast<int>(it % slots));
}

}  // namespace
}  // namespace qs

using namespace qs;

static qs_status metadata_impl(const void* k_cache, qs_dtype kv_dtype, int32_t num_kv_blocks,
                               int32_t BS, int32_t N, int32_t D, const int32_t* prev_lens,
                               const int32_t* seq_lens, int32_t B,
                                         const int32_t* block_tables, int32_t MKBPR,
                                         const int32_t* meta_block_tables, int32_t MMBPR,
                                         int32_t num_meta_blocks, void* maxblocks,
                                         void* minblocks, int32_t* dev_status,
                                         qs_stream_t stream) {
    if (B < 0 || BS <= 0 || N <= 0 || D <= 0 || MKBPR < 0 || MMBPR < 0 || num_kv_blocks < 0 ||
        num_meta_blocks < 0)
        return QS_EINVAL;
    if (B == 0) return QS_OK;
    if (!k_cache || !seq_lens || !block_tables || !meta_block_tables || !maxblocks ||
        !minblocks || !dev_status)
        return QS_EINVAL;
    if (static_cast<long long>(MMBPR) * BS < MKBPR) return QS_EINVAL;
    int es;
    switch (kv_dtype) {
        case QS_F32: es = 4; break;
        case QS_BF16: case QS_F16: es = 2; break;
        default: return QS_EDTYPE;
    }
    const long long row_bytes = static_cast<long long>(N) * D * es;
    if (row_bytes % 16 != 0) return QS_EUNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(maxblocks) |
         reinterpret_cast<uintptr_t>(minblocks)) % 16 != 0)
        return QS_EINVAL;
    const int vpr = static_cast<int>(row_bytes / 16);
    const int nt = prev_lens ? 1024 : 256;
    const int groups = vpr >= nt ? 1 : nt / vpr;
    const size_t smem = static_cast<size_t>(groups) * (vpr < nt ? vpr : nt) * 16 * 2;
    const long long items = prev_lens ? B : static_cast<long long>(B) * MMBPR * BS;
    long long grid = static_cast<long long>(num_sms()) * 4;
    if (grid > items) grid = items;
    if (grid < 1) grid = 1;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    auto args = [&](auto kern) {
        if (smem > 48 * 1024 && !ensure_smem(reinterpret_cast<const void*>(kern), smem))
            return false;
        kern<<<static_cast<unsigned>(grid), nt, smem, s>>>(
            static_cast<const uint8_t*>(k_cache), num_kv_blocks, BS, vpr, prev_lens, seq_lens, B,
            block_tables, MKBPR, meta_block_tables, MMBPR, num_meta_blocks,
            static_cast<uint8_t*>(maxblocks), static_cast<uint8_t*>(minblocks), dev_status);
        return true;
    };
    bool ok;
    if (prev_lens) {
        switch (kv_dtype) {
            case QS_F32: ok = args(prefill_metadata_kernel<Dt::F32, 1024>); break;
            case QS_BF16: ok = args(prefill_metadata_kernel<Dt::BF16, 1024>); break;
            default: ok = args(prefill_metadata_kernel<Dt::F16, 1024>); break;
        }
    } else {
        switch (kv_dtype) {
            case QS_F32: ok = args(prefill_metadata_kernel<Dt::F32, 256>); break;
            case QS_BF16: ok = args(prefill_metadata_kernel<Dt::BF16, 256>); break;
            default: ok = args(prefill_metadata_kernel<Dt::F16, 256>); break;
        }
    }
    if (!ok) return QS_ECUDA;
    QS_CHECK_LAUNCH();
    return QS_OK;
}

extern "C" qs_status qs_prefill_metadata(const void* k_cache, qs_dtype kv_dtype,
                                         int32_t num_kv_blocks, int32_t BS, int32_t N,
                                         int32_t D, const int32_t* seq_lens, int32_t B,
                                         const int32_t* block_tables, int32_t MKBPR,
                                         const int32_t* meta_block_tables, int32_t MMBPR,
                                         int32_t num_meta_blocks, void* maxblocks,
                                         void* minblocks, int32_t* dev_status,
                                         qs_stream_t stream) {
    return metadata_impl(k_cache, kv_dtype, num_kv_blocks, BS, N, D, nullptr, seq_lens, B,
                         block_tables, MKBPR, meta_block_tables, MMBPR, num_meta_blocks,
                         maxblocks, minblocks, dev_status, stream);
}

extern "C" qs_status qs_update_metadata(const void* k_cache, qs_dtype kv_dtype,
                                        int32_t num_kv_blocks, int32_t BS, int32_t N, int32_t D,
                                        const int32_t* prev_lens, const int32_t* seq_lens,
                                        int32_t B, const int32_t* block_tables, int32_t MKBPR,
                                        const int32_t* meta_block_tables, int32_t MMBPR,
                                        int32_t num_meta_blocks, void* maxblocks,
                                        void* minblocks, int32_t* dev_status,
                                        qs_stream_t stream) {
    if (!prev_lens) return QS_EINVAL;
    return metadata_impl(k_cache, kv_dtype, num_kv_blocks, BS, N, D, prev_lens, seq_lens, B,
                         block_tables, MKBPR, meta_block_tables, MMBPR, num_meta_blocks,
                         maxblocks, minblocks, dev_status, stream);
}
