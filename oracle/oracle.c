/*
 * Reference oracle (TEST INFRASTRUCTURE ONLY) -- see oracle.h for the page
 * titles, layouts and the contract of every function.  Slow on purpose: one
 * thread, double precision, no blocking, the steps in the pages' order.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* element decoding                                                          */
/* ------------------------------------------------------------------------ */

static size_t esize(int dt) {
    switch (dt) {
    case ORC_F32: return 4;
    case ORC_BF16: return 2;
    case ORC_F16: return 2;
    case ORC_I8: return 1;
    default: return 0;
    }
}

/* IEEE binary16 -> double, written out from the format's definition. */
static double half_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp(1.0 + m / 1024.0, e - 15);
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* value of element i of a floating-point array of dtype dt */
static double dec(const void* base, int dt, size_t i) {
    switch (dt) {
    case ORC_F32: return (double)((const float*)base)[i];
    case ORC_BF16: return bf16_bits_to_double(((const uint16_t*)base)[i]);
    case ORC_F16: return half_bits_to_double(((const uint16_t*)base)[i]);
    default: return NAN;
    }
}

/* the same as fp32 (exact for all three float dtypes) */
static float decf(const void* base, int dt, size_t i) { return (float)dec(base, dt, i); }

static int is_float_dt(int dt) { return dt == ORC_F32 || dt == ORC_BF16 || dt == ORC_F16; }

static int ceil_div(int a, int b) { return (a + b - 1) / b; }

/* ------------------------------------------------------------------------ */
/* a1: metadata (Quest-ops, 'quest_prefill_metadata: metadata construction')  */
/* ------------------------------------------------------------------------ */

/* Total order used for max/min: -0 sorts below +0 (IEEE 754-2019
 * maximum/minimum).  The pages do not discuss signed zero; this reading makes
 * max/min independent of the reduction order. */
static int less_total(double a, double b) {
    if (a < b) return 1;
    if (a == b && signbit(a) && !signbit(b)) return 1;
    return 0;
}

/* One metadata row: for KV block j of request b, the channel-wise max and min
 * over its valid tokens (or a zero row when j >= nb), written at row r of
 * meta block m.  Returns ORC_ERANGE for a bad block-table entry. */
static int meta_row(const void* k_cache, int kv_dt, int num_kv_blocks, int BS, int N, int D,
                    int L, int nb, const int32_t* bt_row, int j, int m, int r,
                    void* maxblocks, void* minblocks) {
    const size_t es = esize(kv_dt);
    const size_t row = (size_t)N * D; /* elements of one token (all heads) */
    const size_t out_row = ((size_t)m * BS + r) * row;
    if (j >= nb) {
        /* absent KV block: zero metadata ('tail zero fill') */
        memset((char*)maxblocks + out_row * es, 0, row * es);
        memset((char*)minblocks + out_row * es, 0, row * es);
        return ORC_OK;
    }
    const int p = bt_row[j];
    if (p < 0 || p >= num_kv_blocks) return ORC_ERANGE;
    int valid = L - j * BS;
    if (valid > BS) valid = BS;
    for (int n = 0; n < N; n++) {
        for (int d = 0; d < D; d++) {
            /* channel-wise reduce over the block's valid tokens */
            size_t imax = ((size_t)p * BS) * row + (size_t)n * D + d;
            size_t imin = imax;
            double vmax = dec(k_cache, kv_dt, imax), vmin = vmax;
            for (int t = 1; t < valid; t++) {
                size_t i = ((size_t)p * BS + t) * row + (size_t)n * D + d;
                double v = dec(k_cache, kv_dt, i);
                if (less_total(vmax, v)) { vmax = v; imax = i; }
                if (less_total(v, vmin)) { vmin = v; imin = i; }
            }
            size_t o = out_row + (size_t)n * D + d;
            memcpy((char*)maxblocks + o * es, (const char*)k_cache + imax * es, es);
            memcpy((char*)minblocks + o * es, (const char*)k_cache + imin * es, es);
        }
    }
    return ORC_OK;
}

/* For every request: blocks [first_block[b], nb) are rebuilt and the zero
 * rows [max(nb, zero_from[b]), n_meta * BS) written (NULL arrays: from 0, i.e.
 * every row of the used meta blocks). */
static int metadata_rows(const void* k_cache, int kv_dt, int num_kv_blocks, int BS, int N, int D,
                         const int32_t* first_block, const int32_t* zero_from,
                         const int32_t* seq_lens, int B,
                         const int32_t* block_tables, int MKBPR,
                         const int32_t* meta_block_tables, int MMBPR, int num_meta_blocks,
                         void* maxblocks, void* minblocks) {
    for (int b = 0; b < B; b++) {
        const int L = seq_lens[b];
        if (L < 0 || L > MKBPR * BS) return ORC_EINVAL;
        const int nb = ceil_div(L, BS);
        const int n_meta = ceil_div(nb, BS);
        if (n_meta > MMBPR) return ORC_EINVAL;
        const int j0 = first_block ? first_block[b] : 0;
        const int z0 = zero_from ? (zero_from[b] > nb ? zero_from[b] : nb) : nb;
        for (int j = j0; j < n_meta * BS; j++) {
            if (j >= nb && j < z0) continue;   /* already zero */
            const int m = meta_block_tables[(size_t)b * MMBPR + j / BS];
            if (m < 0 || m >= num_meta_blocks) return ORC_ERANGE;
            const int rc = meta_row(k_cache, kv_dt, num_kv_blocks, BS, N, D, L, nb,
                                    block_tables + (size_t)b * MKBPR, j, m, j % BS, maxblocks,
                                    minblocks);
            if (rc != ORC_OK) return rc;
        }
    }
    return ORC_OK;
}

int orc_prefill_metadata(const void* k_cache, int kv_dt, int num_kv_blocks, int BS,
                         int N, int D, const int32_t* seq_lens, int B,
                         const int32_t* block_tables, int MKBPR,
                         const int32_t* meta_block_tables, int MMBPR,
                         int num_meta_blocks, void* maxblocks, void* minblocks) {
    if (!is_float_dt(kv_dt) || BS <= 0 || N <= 0 || D <= 0 || B < 0 || MKBPR < 0 ||
        MMBPR < 0)
        return ORC_EINVAL;
    return metadata_rows(k_cache, kv_dt, num_kv_blocks, BS, N, D, NULL, NULL, seq_lens, B,
                         block_tables, MKBPR, meta_block_tables, MMBPR, num_meta_blocks,
                         maxblocks, minblocks);
}

/* f1: incremental update after decoding.  The metadata was last built (or
 * updated) at lengths prev_lens; the requests now hold seq_lens tokens.  The
 * block that held the last tokens then (possibly partial) and every block
 * begun since are rebuilt, and the rows past the new block count inside the
 * meta blocks begun since are zeroed (rows past the block count inside meta
 * blocks already in use were zeroed by the earlier build); every other row is
 * left as it is.  So prefill at prev_lens followed by this update equals
 * prefill at seq_lens. */
int orc_update_metadata(const void* k_cache, int kv_dt, int num_kv_blocks, int BS, int N, int D,
                        const int32_t* prev_lens, const int32_t* seq_lens, int B,
                        const int32_t* block_tables, int MKBPR,
                        const int32_t* meta_block_tables, int MMBPR, int num_meta_blocks,
                        void* maxblocks, void* minblocks) {
    if (!is_float_dt(kv_dt) || BS <= 0 || N <= 0 || D <= 0 || B < 0 || MKBPR < 0 ||
        MMBPR < 0 || !prev_lens)
        return ORC_EINVAL;
    int32_t* first = (int32_t*)malloc(sizeof(int32_t) * 2 * (size_t)(B > 0 ? B : 1));
    if (!first) return ORC_EINVAL;
    int32_t* zfrom = first + (B > 0 ? B : 1);
    for (int b = 0; b < B; b++) {
        if (prev_lens[b] < 0 || prev_lens[b] > seq_lens[b]) {
            free(first);
            return ORC_EINVAL;
        }
        first[b] = prev_lens[b] / BS;
        zfrom[b] = ceil_div(ceil_div(prev_lens[b], BS), BS) * BS;  /* end of meta blocks in use */
    }
    const int rc = metadata_rows(k_cache, kv_dt, num_kv_blocks, BS, N, D, first, zfrom, seq_lens,
                                 B, block_tables, MKBPR, meta_block_tables, MMBPR,
                                 num_meta_blocks, maxblocks, minblocks);
    free(first);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* a2: group-mean query (Quest-ops, decode-time algorithm, step 1)            */
/* ------------------------------------------------------------------------ */

int orc_group_mean_query(const void* q, int q_dt, int B, int H, int N, int D,
                         double* qg) {
    if (!is_float_dt(q_dt) || N <= 0 || H <= 0 || H % N != 0 || D <= 0) return ORC_EINVAL;
    const int G = H / N; /* every group of H/N consecutive query heads */
    for (int b = 0; b < B; b++)
        for (int n = 0; n < N; n++)
            for (int d = 0; d < D; d++) {
                double s = 0.0;
                for (int g = 0; g < G; g++)
                    s += dec(q, q_dt, ((size_t)b * H + (size_t)n * G + g) * D + d);
                qg[((size_t)b * N + n) * D + d] = s / G;
            }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* a3: Quest block score (Quest-ops, decode-time algorithm, steps 2.1-2.2)    */
/* ------------------------------------------------------------------------ */

int orc_quest_scores(const double* qg, const void* maxblocks, const void* minblocks,
                     int meta_dt, const int32_t* meta_block_tables, int MMBPR,
                     int num_meta_blocks, const int32_t* seq_lens, int B, int N,
                     int D, int BS, double* scores, double* abs_out) {
    if (!is_float_dt(meta_dt) || BS <= 0 || N <= 0 || D <= 0) return ORC_EINVAL;
    const int maxnb = MMBPR * BS;
    for (int b = 0; b < B; b++) {
        const int L = seq_lens[b];
        if (L < 0) return ORC_EINVAL;
        const int nb = ceil_div(L, BS);
        if (nb > maxnb) return ORC_EINVAL;
        for (int n = 0; n < N; n++) {
            const double* g = qg + ((size_t)b * N + n) * D;
            for (int j = 0; j < nb; j++) {
                /* 2.1: the metadata block holding row j of this request */
                const int m = meta_block_tables[(size_t)b * MMBPR + j / BS];
                if (m < 0 || m >= num_meta_blocks) return ORC_ERANGE;
                const size_t base = (((size_t)m * BS + j % BS) * N + n) * D;
                double s = 0.0, sa = 0.0;
                for (int d = 0; d < D; d++) {
                    /* 2.2.1 products with the max and min vectors */
                    double pmax = g[d] * dec(maxblocks, meta_dt, base + d);
                    double pmin = g[d] * dec(minblocks, meta_dt, base + d);
                    /* 2.2.2 elementwise max of the two products */
                    double cmp = pmax > pmin ? pmax : pmin;
                    /* 2.2.3 reduce-sum over the channel dimension */
                    s += cmp;
                    sa += fabs(cmp);
                }
                scores[((size_t)b * N + n) * maxnb + j] = s;
                if (abs_out) abs_out[((size_t)b * N + n) * maxnb + j] = sa;
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* a4: forced sink + local-window set (Quest-ops, the '_in_out_w' variant)     */
/* ------------------------------------------------------------------------ */

/* Metadata covers the blocks finished at the last update, which happened
 * t tokens ago at a multiple of BLOCK_SIZE; blocks from w0 on have no (or
 * incomplete) metadata and are forced in together with the sink block 0. */
int orc_forced_set(int seq_len, int BS, int t, int nb, uint8_t* forced) {
    if (BS <= 0 || nb < 0) return ORC_EINVAL;
    memset(forced, 0, (size_t)nb);
    if (t < 0 || nb == 0) return 0;
    int w0 = (seq_len - t) >= 0 ? (seq_len - t) / BS : 0;
    if (w0 > nb - 1) w0 = nb - 1;
    int count = 0;
    forced[0] = 1;
    count = 1;
    for (int j = w0; j < nb; j++)
        if (!forced[j]) { forced[j] = 1; count++; }
    return count;
}

/* ------------------------------------------------------------------------ */
/* a5: deterministic top-k (Quest-ops step 2.3; tie rule from Kestrel 10-2 §1) */
/* ------------------------------------------------------------------------ */

static int cmp_int32(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

int orc_quest_select(const void* q, int q_dt, const void* maxblocks,
                     const void* minblocks, int meta_dt,
                     const int32_t* meta_block_tables, int MMBPR, int num_meta_blocks,
                     const int32_t* seq_lens, int B, int H, int N, int D, int BS,
                     int k, int t, int32_t* selected, float* scores_f32) {
    if (k <= 0 || N <= 0 || H % N != 0) return ORC_EINVAL;
    const int maxnb = MMBPR * BS;
    double* qg = (double*)malloc(sizeof(double) * (size_t)B * N * D + 8);
    double* sc = (double*)malloc(sizeof(double) * ((size_t)B * N * maxnb + 1));
    float* sf = (float*)malloc(sizeof(float) * ((size_t)maxnb + 1));
    uint8_t* used = (uint8_t*)malloc((size_t)maxnb + 1);
    int32_t* res = (int32_t*)malloc(sizeof(int32_t) * ((size_t)k + 1));
    int rc = ORC_OK;
    if (!qg || !sc || !sf || !used || !res) { rc = ORC_EINVAL; goto done; }
    rc = orc_group_mean_query(q, q_dt, B, H, N, D, qg);
    if (rc) goto done;
    rc = orc_quest_scores(qg, maxblocks, minblocks, meta_dt, meta_block_tables, MMBPR,
                          num_meta_blocks, seq_lens, B, N, D, BS, sc, NULL);
    if (rc) goto done;
    for (int b = 0; b < B; b++) {
        const int L = seq_lens[b];
        const int nb = ceil_div(L, BS);
        for (int n = 0; n < N; n++) {
            /* the top-k ranks the fp32 block scores (the kernels score in fp32) */
            for (int j = 0; j < nb; j++) {
                sf[j] = (float)sc[((size_t)b * N + n) * maxnb + j];
                if (scores_f32) scores_f32[((size_t)b * N + n) * maxnb + j] = sf[j];
            }
            int nf = orc_forced_set(L, BS, t, nb, used);
            if (nf < 0) { rc = nf; goto done; }
            if (nf > k) { rc = ORC_EFORCED; goto done; }
            int cnt = 0;
            for (int j = 0; j < nb; j++)
                if (used[j]) res[cnt++] = j;
            /* greedy: repeatedly take the best unused block, ties to the lower
             * block index, no randomness */
            while (cnt < k) {
                int best = -1;
                for (int j = 0; j < nb; j++) {
                    if (used[j]) continue;
                    if (best < 0 || sf[j] > sf[best]) best = j;
                }
                if (best < 0) break; /* fewer blocks than k: stop, no padding */
                used[best] = 1;
                res[cnt++] = best;
            }
            qsort(res, (size_t)cnt, sizeof(int32_t), cmp_int32);
            int32_t* out = selected + ((size_t)b * N + n) * k;
            for (int i = 0; i < k; i++) out[i] = i < cnt ? res[i] : -1;
        }
    }
done:
    free(qg); free(sc); free(sf); free(used); free(res);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* int8 query quantisation (reading of Kestrel 10-2 §2: "q8 KV takes an int8 x  */
/* int8 dot + scale"; the pages leave the query side open)                    */
/* ------------------------------------------------------------------------ */

int orc_quantize_query(const void* q, int q_dt, int D, int8_t* q8, float* s_q) {
    if (!is_float_dt(q_dt) || D <= 0) return ORC_EINVAL;
    float amax = 0.0f;
    for (int d = 0; d < D; d++) {
        float a = fabsf(decf(q, q_dt, (size_t)d));
        if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
        *s_q = 0.0f;
        for (int d = 0; d < D; d++) q8[d] = 0;
        return ORC_OK;
    }
    const float s = amax / 127.0f; /* fp32, round to nearest */
    *s_q = s;
    for (int d = 0; d < D; d++) {
        float r = rintf(decf(q, q_dt, (size_t)d) / s); /* half-even */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q8[d] = (int8_t)r;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* a6..a8: probe / importance selector (Kestrel 10-2, §1 and §2)              */
/* ------------------------------------------------------------------------ */

/* The probe score starts from this floor before the first dot product of a
 * block is taken into account (the engine's starting value; every block has
 * at least one probe, so it never survives). */
static const float PROBE_FLOOR = -1e30f;

/* Positions probed in the token range [first, end) of one block: the block is
 * sampled with a fixed stride, stride = (end - first) / n_probe tokens rounded
 * down, at least 1, starting at the block's first token.  A full 32-token
 * block with 8 probes is sampled at offsets 0, 4, ..., 28; a 5-token tail at
 * every token.  Writes the positions to pos[] and returns how many. */
static int probe_positions(int first, int end, int n_probe, int* pos) {
    int stride = (end - first) / n_probe;
    if (stride < 1) stride = 1;
    int count = 0;
    for (int p = first; p < end; p += stride) pos[count++] = p;
    return count;
}

/* The score of one probe: q_h . K[position] for KV head kh.  Float caches: the
 * dot product in double, rounded once to fp32.  int8 caches: the exact integer
 * dot of the quantised query and the int8 key, scaled by s_q * s_k (two fp32
 * roundings, as the int8 reading states). */
static float probe_dot(const float* qf, const int8_t* q8, float s_q, const void* k_cache,
                       const float* k_scale, int kv_dt, size_t token_row, int N, int kh, int D) {
    const size_t base = (token_row * (size_t)N + (size_t)kh) * (size_t)D;
    if (kv_dt == ORC_I8) {
        long long idot = 0;
        for (int d = 0; d < D; d++) idot += (long long)q8[d] * ((const int8_t*)k_cache)[base + d];
        const float s_k = k_scale[token_row * (size_t)N + (size_t)kh];
        const float s = s_q * s_k;
        return s * (float)idot;
    }
    double sum = 0.0;
    for (int d = 0; d < D; d++) sum += (double)qf[d] * dec(k_cache, kv_dt, base + d);
    return (float)sum;
}

/* Block importance: the prefill importance of the block's tokens added up in
 * fp32, token after token in order (the importance picks depend on these
 * exact fp32 sums). */
static float block_importance(const float* imp_row, int first, int end) {
    float total = 0.0f;
    for (int p = first; p < end; p++) total = total + imp_row[p];
    return total;
}

/* Ranking used by both greedy passes: block a ranks before block b when its
 * value is larger, or equal with the lower block index. */
static int ranks_before(const float* value, int a, int b) {
    if (value[a] != value[b]) return value[a] > value[b];
    return a < b;
}

enum { PICK_IMPORTANCE = 1, PICK_PROBE = 2 };

/* One greedy pass: up to `quota` times, take the best-ranked block not taken
 * yet and append it to the pick list (with its origin tag).  Stops early when
 * every block is taken: the list is never padded.  Returns the new length. */
static int greedy_pass(const float* value, int nb, int quota, uint8_t* taken,
                       int32_t* picks, uint8_t* origin, int n_picks, uint8_t tag) {
    for (int round = 0; round < quota; round++) {
        int choice = -1;
        for (int j = 0; j < nb; j++)
            if (!taken[j] && (choice < 0 || ranks_before(value, j, choice))) choice = j;
        if (choice < 0) break;
        taken[choice] = 1;
        picks[n_picks] = choice;
        origin[n_picks] = tag;
        n_picks++;
    }
    return n_picks;
}

/* Recency insurance: the pick that makes room for the last block is the probe
 * pick with the lowest probe score; among equal scores the larger block
 * index (the one the greedy fill took later).  Importance picks are never
 * candidates.  Returns its position in the pick list, or -1 if there is no
 * probe pick. */
static int recency_victim(const float* probe, const int32_t* picks, const uint8_t* origin,
                          int n_picks) {
    int victim = -1;
    for (int i = 0; i < n_picks; i++) {
        if (origin[i] != PICK_PROBE) continue;
        if (victim < 0) { victim = i; continue; }
        const float a = probe[picks[i]], b = probe[picks[victim]];
        if (a < b || (a == b && picks[i] > picks[victim])) victim = i;
    }
    return victim;
}

int orc_probe_select(const void* q, int q_dt, const void* k_cache,
                     const float* k_scale, int kv_dt, int num_kv_blocks,
                     const int32_t* block_tables, int MKBPR, const int32_t* seq_lens,
                     const float* importance, int S_max, int B, int H, int N, int D,
                     int BS, int k, int n_probe, int32_t* selected, float* probe_out,
                     float* imp_out, int32_t* n_imp_out) {
    if (k <= 0 || N <= 0 || H % N != 0 || D <= 0 || BS <= 0) return ORC_EINVAL;
    if (kv_dt == ORC_I8 && !k_scale) return ORC_EINVAL;
    if (kv_dt != ORC_I8 && !is_float_dt(kv_dt)) return ORC_EINVAL;
    if (n_probe < 1) n_probe = 1;
    const int G = H / N;
    const size_t cap = (size_t)MKBPR + 1;
    float* probe = (float*)malloc(sizeof(float) * cap);
    float* imp = (float*)malloc(sizeof(float) * cap);
    uint8_t* taken = (uint8_t*)malloc(cap);
    int32_t* picks = (int32_t*)malloc(sizeof(int32_t) * ((size_t)k + 1));
    uint8_t* origin = (uint8_t*)malloc((size_t)k + 1);
    int* pos = (int*)malloc(sizeof(int) * ((size_t)BS + 1));
    float* qf = (float*)malloc(sizeof(float) * (size_t)D);
    int8_t* q8 = (int8_t*)malloc((size_t)D);
    int rc = ORC_OK;
    if (!probe || !imp || !taken || !picks || !origin || !pos || !qf || !q8) {
        rc = ORC_EINVAL;
        goto done;
    }
    for (int b = 0; b < B; b++) {
        const int L = seq_lens[b];
        if (L < 0 || L > MKBPR * BS) { rc = ORC_EINVAL; goto done; }
        if (importance && L > S_max) { rc = ORC_EINVAL; goto done; }
        const int nb = ceil_div(L, BS);
        const int32_t* bt_row = block_tables + (size_t)b * MKBPR;
        for (int j = 0; j < nb; j++)
            if (bt_row[j] < 0 || bt_row[j] >= num_kv_blocks) { rc = ORC_ERANGE; goto done; }

        /* signal 2: summed prefill importance per block (shared by the heads) */
        for (int j = 0; j < nb; j++) {
            const int first = j * BS, end = first + BS < L ? first + BS : L;
            imp[j] = importance ? block_importance(importance + (size_t)b * S_max, first, end)
                                : 0.0f;
            if (imp_out) imp_out[(size_t)b * MKBPR + j] = imp[j];
        }

        for (int h = 0; h < H; h++) {
            const int kh = h / G;
            float s_q = 0.0f;
            for (int d = 0; d < D; d++) qf[d] = decf(q, q_dt, ((size_t)b * H + h) * D + d);
            if (kv_dt == ORC_I8) orc_quantize_query(qf, ORC_F32, D, q8, &s_q);

            /* signal 1: the probe score of every block, the largest dot
             * product over its probe positions */
            for (int j = 0; j < nb; j++) {
                const int first = j * BS, end = first + BS < L ? first + BS : L;
                const int np = probe_positions(first, end, n_probe, pos);
                float score = PROBE_FLOOR;
                for (int i = 0; i < np; i++) {
                    const size_t token_row = (size_t)bt_row[j] * BS + (size_t)(pos[i] - first);
                    const float s = probe_dot(qf, q8, s_q, k_cache, k_scale, kv_dt, token_row, N,
                                              kh, D);
                    if (s > score) score = s;
                }
                probe[j] = score;
                if (probe_out) probe_out[((size_t)b * H + h) * MKBPR + j] = score;
            }

            /* half of the budget, rounded up, goes to the most important
             * blocks; the probe score fills the rest */
            memset(taken, 0, (size_t)nb + 1);
            int n_picks = 0;
            if (importance)
                n_picks = greedy_pass(imp, nb, (k + 1) / 2, taken, picks, origin, n_picks,
                                      PICK_IMPORTANCE);
            const int n_imp = n_picks;
            n_picks = greedy_pass(probe, nb, k - n_picks, taken, picks, origin, n_picks,
                                  PICK_PROBE);

            /* insurance: the most recent block is always attended to, unless
             * the budget holds no probe pick it could take the place of */
            if (nb > 0 && !taken[nb - 1]) {
                const int v = recency_victim(probe, picks, origin, n_picks);
                if (v >= 0) {
                    taken[picks[v]] = 0;
                    picks[v] = nb - 1;
                    taken[nb - 1] = 1;
                }
            }

            qsort(picks, (size_t)n_picks, sizeof(int32_t), cmp_int32);
            int32_t* out = selected + ((size_t)b * H + h) * k;
            for (int i = 0; i < k; i++) out[i] = i < n_picks ? picks[i] : -1;
            if (n_imp_out) n_imp_out[(size_t)b * H + h] = n_imp;
        }
    }
done:
    free(probe); free(imp); free(taken); free(picks); free(origin); free(pos); free(qf); free(q8);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* a9: exact attention over the selected blocks (Kestrel 10-2 §1, the cost     */
/* paragraph: softmax renormalised over the selected blocks only; Quest-ops:  */
/* indices are in-sequence and go through block_tables)                      */
/* ------------------------------------------------------------------------ */

int orc_sparse_attention(const void* q, int q_dt, const void* k_cache,
                         const void* v_cache, const float* k_scale,
                         const float* v_scale, int kv_dt, int num_kv_blocks,
                         const int32_t* block_tables, int MKBPR,
                         const int32_t* seq_lens, const int32_t* selected,
                         int sel_heads, int k, double softmax_scale, int B, int H,
                         int N, int D, int BS, double* out, double* lse) {
    if (k <= 0 || N <= 0 || H % N != 0 || D <= 0 || BS <= 0) return ORC_EINVAL;
    if (sel_heads != N && sel_heads != H) return ORC_EINVAL;
    if (kv_dt == ORC_I8 && (!k_scale || !v_scale)) return ORC_EINVAL;
    if (kv_dt != ORC_I8 && !is_float_dt(kv_dt)) return ORC_EINVAL;
    const int G = H / N;
    const size_t max_tok = (size_t)k * BS;
    double* logit = (double*)malloc(sizeof(double) * (max_tok + 1));
    size_t* vrow = (size_t*)malloc(sizeof(size_t) * (max_tok + 1));
    size_t* srow = (size_t*)malloc(sizeof(size_t) * (max_tok + 1));
    double* qd = (double*)malloc(sizeof(double) * (size_t)D);
    float* qf = (float*)malloc(sizeof(float) * (size_t)D);
    int8_t* q8 = (int8_t*)malloc((size_t)D);
    int rc = ORC_OK;
    if (!logit || !vrow || !srow || !qd || !qf || !q8) { rc = ORC_EINVAL; goto done; }
    for (int b = 0; b < B; b++) {
        const int L = seq_lens[b];
        if (L < 0 || L > MKBPR * BS) { rc = ORC_EINVAL; goto done; }
        const int nb = ceil_div(L, BS);
        for (int h = 0; h < H; h++) {
            const int n = h / G;
            const int s = sel_heads == H ? h : n;
            const int32_t* row = selected + ((size_t)b * sel_heads + s) * k;
            const size_t qoff = ((size_t)b * H + h) * D;
            float s_q = 0.0f;
            for (int d = 0; d < D; d++) { qd[d] = dec(q, q_dt, qoff + d); qf[d] = (float)qd[d]; }
            if (kv_dt == ORC_I8) orc_quantize_query(qf, ORC_F32, D, q8, &s_q);
            /* token scores over the selected blocks only */
            size_t T = 0;
            for (int i = 0; i < k; i++) {
                const int j = row[i];
                if (j < 0) continue;
                if (j >= nb) { rc = ORC_ERANGE; goto done; }
                for (int i2 = 0; i2 < i; i2++)
                    if (row[i2] == j) { rc = ORC_EDUP; goto done; }
                const int p = block_tables[(size_t)b * MKBPR + j];
                if (p < 0 || p >= num_kv_blocks) { rc = ORC_ERANGE; goto done; }
                int valid = L - j * BS;
                if (valid > BS) valid = BS;
                for (int t = 0; t < valid; t++) {
                    const size_t tok = ((size_t)p * BS + t) * N + n;
                    const size_t kr = tok * D;
                    double dot = 0.0;
                    if (kv_dt == ORC_I8) {
                        long long acc = 0;
                        for (int d = 0; d < D; d++)
                            acc += (long long)q8[d] * ((const int8_t*)k_cache)[kr + d];
                        dot = (double)s_q * (double)k_scale[tok] * (double)acc;
                    } else {
                        for (int d = 0; d < D; d++) dot += qd[d] * dec(k_cache, kv_dt, kr + d);
                    }
                    logit[T] = softmax_scale * dot;
                    vrow[T] = kr;
                    srow[T] = tok;
                    T++;
                }
            }
            double* o = out + qoff;
            if (T == 0) {
                for (int d = 0; d < D; d++) o[d] = 0.0;
                if (lse) lse[(size_t)b * H + h] = -INFINITY;
                continue;
            }
            /* softmax over the selected set: subtract the max, normalise */
            double m = logit[0];
            for (size_t i = 1; i < T; i++) if (logit[i] > m) m = logit[i];
            double l = 0.0;
            for (size_t i = 0; i < T; i++) { logit[i] = exp(logit[i] - m); l += logit[i]; }
            /* weighted sum of V */
            for (int d = 0; d < D; d++) {
                double acc = 0.0;
                for (size_t i = 0; i < T; i++) {
                    double v = kv_dt == ORC_I8
                                   ? (double)((const int8_t*)v_cache)[vrow[i] + d] * (double)v_scale[srow[i]]
                                   : dec(v_cache, kv_dt, vrow[i] + d);
                    acc += logit[i] * v;
                }
                o[d] = acc / l;
            }
            if (lse) lse[(size_t)b * H + h] = m + log(l);
        }
    }
done:
    free(logit); free(vrow); free(srow); free(qd); free(qf); free(q8);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* f3: prefill importance (Kestrel 10-2 §1, signal 2: the attention each     */
/* token received during an exact prefill, reduced per head and summed over  */
/* the heads into prefill_importance[s]; §2, the decode call site: the sums  */
/* are formed when the prefill ends)                                         */
/* ------------------------------------------------------------------------ */

int orc_prefill_importance(const void* q, int q_dt, const void* k_cache,
                           const float* k_scale, int kv_dt, int num_kv_blocks,
                           const int32_t* block_tables, int MKBPR,
                           const int32_t* prefill_lens, int S_max, int B, int H, int N,
                           int D, int BS, double softmax_scale, int first_query,
                           double* importance, double* lse) {
    if (B < 0 || N <= 0 || H % N != 0 || D <= 0 || BS <= 0 || S_max < 0) return ORC_EINVAL;
    if (!is_float_dt(q_dt)) return ORC_EINVAL;
    if (kv_dt == ORC_I8 ? !k_scale : !is_float_dt(kv_dt)) return ORC_EINVAL;
    if (kv_dt != ORC_I8 && q_dt != kv_dt) return ORC_EINVAL;
    const int G = H / N;
    const size_t SD = (size_t)S_max * D;
    /* keys of one (request, KV head) gathered in position order, the query
     * row in double (or quantised), one row of logits, one head's masses */
    double* kd = (double*)malloc(sizeof(double) * (SD + 1));
    double* ks = (double*)malloc(sizeof(double) * ((size_t)S_max + 1));
    double* logit = (double*)malloc(sizeof(double) * ((size_t)S_max + 1));
    double* imp_head = (double*)malloc(sizeof(double) * ((size_t)S_max + 1));
    double* qd = (double*)malloc(sizeof(double) * (size_t)D);
    float* qf = (float*)malloc(sizeof(float) * (size_t)D);
    int8_t* q8 = (int8_t*)malloc((size_t)D);
    int rc = ORC_OK;
    if (!kd || !ks || !logit || !imp_head || !qd || !qf || !q8) { rc = ORC_EINVAL; goto done; }
    for (int b = 0; b < B; b++) {
        const int S = prefill_lens[b];
        if (S < 0 || S > S_max || S > MKBPR * BS) { rc = ORC_EINVAL; goto done; }
        double* imp = importance + (size_t)b * S_max;
        for (int s = 0; s < S_max; s++) imp[s] = 0.0;
        for (int h = 0; h < H; h++) {
            const int n = h / G;
            /* gather K of KV head n for positions 0..S-1 through the table */
            for (int s = 0; s < S; s++) {
                const int p = block_tables[(size_t)b * MKBPR + s / BS];
                if (p < 0 || p >= num_kv_blocks) { rc = ORC_ERANGE; goto done; }
                const size_t tok = ((size_t)p * BS + s % BS) * N + n;
                for (int d = 0; d < D; d++)
                    kd[(size_t)s * D + d] = kv_dt == ORC_I8
                        ? (double)((const int8_t*)k_cache)[tok * D + d]
                        : dec(k_cache, kv_dt, tok * D + d);
                ks[s] = kv_dt == ORC_I8 ? (double)k_scale[tok] : 1.0;
            }
            for (int s = 0; s < S; s++) imp_head[s] = 0.0;
            for (int i = first_query > 0 ? first_query : 0; i < S; i++) {
                const size_t qoff = (((size_t)b * S_max + i) * H + h) * D;
                double rowscale = 1.0;
                for (int d = 0; d < D; d++) { qd[d] = dec(q, q_dt, qoff + d); qf[d] = (float)qd[d]; }
                if (kv_dt == ORC_I8) {
                    float s_q = 0.0f;
                    orc_quantize_query(qf, ORC_F32, D, q8, &s_q);
                    for (int d = 0; d < D; d++) qd[d] = (double)q8[d];
                    rowscale = (double)s_q;
                }
                /* causal logits l_s, s <= i, then the row's log-sum-exp */
                double m = -INFINITY;
                for (int s = 0; s <= i; s++) {
                    double dot = 0.0;
                    for (int d = 0; d < D; d++) dot += qd[d] * kd[(size_t)s * D + d];
                    logit[s] = softmax_scale * rowscale * ks[s] * dot;
                    if (logit[s] > m) m = logit[s];
                }
                double z = 0.0;
                for (int s = 0; s <= i; s++) z += exp(logit[s] - m);
                const double row_lse = m + log(z);
                if (lse) lse[((size_t)b * H + h) * S_max + i] = row_lse;
                /* the mass this query gave each key */
                for (int s = 0; s <= i; s++) imp_head[s] += exp(logit[s] - row_lse);
            }
            for (int s = 0; s < S; s++) imp[s] += imp_head[s];
        }
    }
done:
    free(kd); free(ks); free(logit); free(imp_head); free(qd); free(qf); free(q8);
    return rc;
}
