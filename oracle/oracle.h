/*
 * Reference oracle for query-aware sparse KV-block selection and sparse decode
 * attention.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * CPU-baseline leg of the benchmark call it; the product path never does.
 *
 * Plain single-threaded C11, double precision, written from the method's
 * description on two pages:
 *   [Quest-ops]  "ops-transformer select_attention_operators: Quest-based sparse
 *                attention block prediction kernels on Ascend 910B"
 *                (sections 'quest_prefill_metadata: metadata construction' and
 *                'quest_block_select_paged: decode-time top-k prediction').
 *   [Kestrel]    "Kestrel-LLM article 10-2: sparse top-k block selection in the
 *                inference engine" (section 1 'three signals + one insurance',
 *                section 2 'code walk-through').
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Layouts (row-major, element offsets):
 *   k_cache/v_cache [P, BS, N, D]      element (p,t,n,d) at ((p*BS+t)*N+n)*D+d
 *   k_scale/v_scale [P, BS, N] (int8)  one fp32 scale per (token, KV head)
 *   maxblocks/minblocks [M, BS, N, D]  row r of meta block m = KV block
 *                                      (table slot)*BS + r of the request
 *   block_tables [B, MKBPR], meta_block_tables [B, MMBPR], seq_lens [B]
 *   q [B, H, D]; query head h belongs to KV head h / (H/N).
 * dtype codes: 0 = fp32, 1 = bf16, 2 = fp16, 3 = int8 (+ fp32 scale).
 * Every function returns 0 on success and a negative code on a bad argument
 * or an out-of-range table entry (it then leaves its outputs partly written).
 */
#ifndef QS_ORACLE_H
#define QS_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F16 = 2, ORC_I8 = 3 };
enum { ORC_OK = 0, ORC_EINVAL = -1, ORC_ERANGE = -2, ORC_EFORCED = -3, ORC_EDUP = -4 };

/* Per-block channel max/min metadata (a1).  Writes only the rows of the meta
 * blocks a request uses; rows of KV blocks beyond the request's block count
 * inside those meta blocks are zeroed.  Output elements are the storage-dtype
 * bits of the selected input element (max/min is exact). */
int orc_prefill_metadata(const void* k_cache, int kv_dt, int num_kv_blocks, int BS,
                         int N, int D, const int32_t* seq_lens, int B,
                         const int32_t* block_tables, int MKBPR,
                         const int32_t* meta_block_tables, int MMBPR,
                         int num_meta_blocks, void* maxblocks, void* minblocks);

/* Incremental metadata update after decoding (f1): with the metadata last
 * built at lengths prev_lens, rebuilds the rows of blocks
 * [prev_lens[b] / BS, ceil(seq_lens[b] / BS)) and zeroes the rows past the new
 * block count inside the meta blocks begun since prev_lens; other rows are
 * untouched.
 * Prefill at prev_lens then this update equals prefill at seq_lens.
 * ORC_EINVAL when prev_lens[b] < 0 or > seq_lens[b]. */
int orc_update_metadata(const void* k_cache, int kv_dt, int num_kv_blocks, int BS, int N, int D,
                        const int32_t* prev_lens, const int32_t* seq_lens, int B,
                        const int32_t* block_tables, int MKBPR,
                        const int32_t* meta_block_tables, int MMBPR, int num_meta_blocks,
                        void* maxblocks, void* minblocks);

/* Group-mean query (a2): qg[b][n][d] = mean over the H/N query heads of group n. */
int orc_group_mean_query(const void* q, int q_dt, int B, int H, int N, int D,
                         double* qg);

/* Quest block scores (a3), double, for j < nb_b: out[(b*N+n)*maxnb + j]; other
 * entries are left untouched.  abs_out (optional) receives sum_d |max-term_d|,
 * the scale used by the score tolerance.  maxnb = MMBPR*BS. */
int orc_quest_scores(const double* qg, const void* maxblocks, const void* minblocks,
                     int meta_dt, const int32_t* meta_block_tables, int MMBPR,
                     int num_meta_blocks, const int32_t* seq_lens, int B, int N,
                     int D, int BS, double* scores, double* abs_out);

/* Full Quest select (a2..a5): selected [B, N, k], ascending in-sequence block
 * indices, -1 padded.  t = tokens_since_metadata_update (-1: no window).
 * scores_f32 (optional, [B, N, MMBPR*BS]) receives the fp32-rounded scores the
 * top-k ranks by. */
int orc_quest_select(const void* q, int q_dt, const void* maxblocks,
                     const void* minblocks, int meta_dt,
                     const int32_t* meta_block_tables, int MMBPR, int num_meta_blocks,
                     const int32_t* seq_lens, int B, int H, int N, int D, int BS,
                     int k, int t, int32_t* selected, float* scores_f32);

/* Forced (sink + window) set of one request (a4): writes the flags into
 * forced[0..nb) and returns |F|, or a negative code. */
int orc_forced_set(int seq_len, int BS, int t, int nb, uint8_t* forced);

/* Probe / prefill-importance selector (a6..a8), one selection per QUERY head:
 * selected [B, H, k].  importance: [B, S_max] fp32 or NULL.  k_scale: [P,BS,N]
 * for int8 KV, else NULL.  probe_out [B,H,MKBPR], imp_out [B,MKBPR] and
 * n_imp_out [B,H] are optional diagnostics. */
int orc_probe_select(const void* q, int q_dt, const void* k_cache,
                     const float* k_scale, int kv_dt, int num_kv_blocks,
                     const int32_t* block_tables, int MKBPR, const int32_t* seq_lens,
                     const float* importance, int S_max, int B, int H, int N, int D,
                     int BS, int k, int n_probe, int32_t* selected, float* probe_out,
                     float* imp_out, int32_t* n_imp_out);

/* Exact attention over the selected blocks (a9), double.  selected
 * [B, sel_heads, k] with sel_heads == N (per KV head) or H (per query head);
 * entries < 0 are ignored; the valid entries of a row must be distinct and
 * < nb_b.  out [B,H,D]; lse [B,H] natural-log log-sum-exp of the scaled
 * logits (-inf and zero output for an empty selection). */
int orc_sparse_attention(const void* q, int q_dt, const void* k_cache,
                         const void* v_cache, const float* k_scale,
                         const float* v_scale, int kv_dt, int num_kv_blocks,
                         const int32_t* block_tables, int MKBPR,
                         const int32_t* seq_lens, const int32_t* selected,
                         int sel_heads, int k, double softmax_scale, int B, int H,
                         int N, int D, int BS, double* out, double* lse);

/* Symmetric per-(b,h) int8 quantisation of a query vector used by the int8 KV
 * path: s_q = max|q| / 127 (fp32), q8 = round-half-even(q / s_q) (fp32).
 * Exposed so the tests can pin it. */
int orc_quantize_query(const void* q, int q_dt, int D, int8_t* q8, float* s_q);

/* Prefill importance (f3), double.  For request b with S = prefill_lens[b]
 * prefill tokens, every query head h and every query position i < S attends
 * causally to the keys s <= i of its KV head h / (H/N):
 *   p[h][i][s] = exp(l_s - lse[h][i]),  l_s = softmax_scale * q[b][i][h] . K[b][s],
 *   lse[h][i]  = log sum_{s<=i} exp(l_s);
 * the per-head attention mass a token received, imp_head[h][s] = sum_{i>=s}
 * p[h][i][s], is accumulated over the heads in ascending order into
 * importance[b][s].  int8 KV: the query row is quantised as by
 * orc_quantize_query and l_s = softmax_scale * s_q * k_scale[s] * (q8 . k8).
 * q is [B, S_max, H, D]; K of position s sits in block_tables[b][s / BS],
 * row s % BS.  Only query positions i >= first_query are summed (0: all), so
 * importance[b][s] is exact for s >= first_query.  importance [B, S_max] is
 * written for every s (0 for s >= S); lse [B, H, S_max] (optional) receives
 * the rows first_query <= i < S.  ORC_EINVAL for S < 0 or
 * S > min(S_max, MKBPR * BS); ORC_ERANGE for a bad table entry. */
int orc_prefill_importance(const void* q, int q_dt, const void* k_cache,
                           const float* k_scale, int kv_dt, int num_kv_blocks,
                           const int32_t* block_tables, int MKBPR,
                           const int32_t* prefill_lens, int S_max, int B, int H, int N,
                           int D, int BS, double softmax_scale, int first_query,
                           double* importance, double* lse);

#ifdef __cplusplus
}
#endif
#endif
