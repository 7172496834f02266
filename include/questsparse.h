/*
 * questsparse -- query-aware sparse KV-block selection and sparse decode
 * attention for one GB300 (sm_103a) GPU.  C ABI.
 *
 * Operations and where they are defined:
 *   qs_prefill_metadata    CANN ops-transformer select_attention_operators page
 *                          (Quest on Ascend 910B), section 'quest_prefill_metadata:
 *                          metadata construction'.
 *   qs_update_metadata     the same page (metadata refreshed while decoding).
 *   qs_block_select_paged  same page, section 'quest_block_select_paged: decode-time
 *                          top-k prediction' (steps 1, 2.1-2.3) and the three
 *                          interfaces ('_in_out' / '_in_out_w': the sink + window
 *                          variant driven by tokens_since_metadata_update).
 *   qs_probe_select        Kestrel-LLM article 10-2 'sparse top-k block selection',
 *                          sections 1 and 2 (probe loop, (k+1)/2 importance budget,
 *                          greedy probe fill, recency insurance).
 *   qs_sparse_decode_attn  Kestrel-LLM 10-2 section 2 (exact attention over the
 *                          selected blocks only, softmax renormalised over that set)
 *                          with the in-sequence -> physical mapping through
 *                          block_tables from the CANN page's top-k section.
 *   qs_sparse_decode_step  select (either mode) followed by the attention.
 *   qs_prefill_importance  Kestrel-LLM 10-2 section 1, signal 2 (the attention each
 *                          prefill token received, per head, summed over heads),
 *                          the input qs_probe_select's importance budget reads.
 *
 * Conventions shared by every call:
 *  - All tensor arguments are DEVICE pointers to contiguous row-major memory
 *    owned by the caller.  The library never allocates device memory; the
 *    scratch a call needs is a caller-provided workspace whose size
 *    qs_workspace_size() returns.  A workspace belongs to one operation and
 *    one set of sizes (B, H, N, D, BS, k, table widths): zero-fill it before
 *    its first use, and again after a call reported a device-side error.  The
 *    kernels rearm the arrival counters they keep in it, so consecutive calls
 *    with the same sizes need no re-zeroing; the rest of it is scratch, so a
 *    call with other sizes needs a freshly zeroed workspace.  Calls that share
 *    a workspace must not overlap in time (use one stream).
 *  - Every call enqueues its kernels on `stream` and returns without waiting.
 *    The returned qs_status reports host-side validation and launch errors only.
 *  - Faults found on the device (a table entry out of range, a bad seq_len, an
 *    out-of-range selected index) do not trap: the kernel skips the bad unit and
 *    stores the first such code into the caller's int32 `dev_status` word
 *    (sticky; 0 = no error).  Read it with qs_read_status().
 *  - Shapes: B requests, H query heads, N KV heads (H % N == 0; query head h
 *    belongs to KV head h / (H/N)), D head dim, BS tokens per KV block.
 *      q                    [B, H, D]                 (fp32, bf16 or fp16)
 *      k_cache, v_cache     [num_kv_blocks, BS, N, D] (fp32, bf16, fp16 or int8)
 *      k_scale, v_scale     [num_kv_blocks, BS, N]    fp32, int8 caches only:
 *                           value = int8 * scale, one scale per (token, KV head)
 *      block_tables         [B, MKBPR] int32, in-sequence block -> physical block
 *      seq_lens             [B] int32, 0 <= seq_len <= MKBPR * BS
 *      maxblocks, minblocks [num_meta_blocks, BS, N, D], dtype of the K cache;
 *                           row r of a request's metadata block slot s holds KV
 *                           block s*BS + r of that request
 *      meta_block_tables    [B, MMBPR] int32, request -> metadata blocks
 *  - Block indices returned by the selectors are IN-SEQUENCE indices (0 is the
 *    first block of the request), ascending, padded with -1.  A request with
 *    nb = ceil(seq_len/BS) < k blocks gets nb indices.
 */
#ifndef QUESTSPARSE_H
#define QUESTSPARSE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* qs_stream_t;

typedef enum {
    QS_OK = 0,
    QS_EINVAL = 1,        /* bad shape, size, pointer or k                    */
    QS_EDTYPE = 2,        /* dtype combination not supported by the call      */
    QS_EUNSUPPORTED = 3,  /* no kernel instantiation for this D / BS / H/N    */
    QS_ECUDA = 4,         /* a CUDA runtime call or kernel launch failed      */
    QS_EWORKSPACE = 5     /* workspace missing or smaller than required       */
} qs_status;

typedef enum { QS_F32 = 0, QS_BF16 = 1, QS_F16 = 2, QS_I8 = 3 } qs_dtype;

/* Codes the kernels store into *dev_status (first error wins). */
typedef enum {
    QS_DEV_OK = 0,
    QS_DEV_EBLOCK_TABLE = 1,  /* block_tables entry outside [0, num_kv_blocks)  */
    QS_DEV_EMETA_TABLE = 2,   /* meta_block_tables entry outside [0, num_meta)  */
    QS_DEV_ESEQ_LEN = 3,      /* seq_len < 0 or > MKBPR*BS (or metadata slots)  */
    QS_DEV_ESELECTED = 4,     /* selected index >= ceil(seq_len/BS)             */
    QS_DEV_EFORCED = 5,       /* more forced window blocks than k               */
    QS_DEV_ETIMEOUT = 6       /* a bounded wait ran out (prefill importance)    */
} qs_dev_code;

typedef enum {
    QS_OP_BLOCK_SELECT = 0,
    QS_OP_PROBE_SELECT = 1,
    QS_OP_SPARSE_ATTN = 2,
    QS_OP_DECODE_STEP_QUEST = 3,
    QS_OP_DECODE_STEP_PROBE = 4
} qs_op;

/* Library version (major*10000 + minor*100 + patch). */
int32_t qs_version(void);

/* Self-check of the device-side bounded wait (no counterpart on the pages):
 * enqueues one small kernel that waits, with the same bounded mbarrier wait
 * the tensor-core prefill-importance passes use, on a barrier that nothing
 * arrives on.  The wait runs out after about a second and the kernel stores
 * QS_DEV_ETIMEOUT into *dev_status (read it with qs_read_status()); the
 * context stays usable.  dev_status: device int32.  Errors: NULL ->
 * QS_EINVAL; a launch failure -> QS_ECUDA. */
qs_status qs_check_bounded_wait(int32_t* dev_status, qs_stream_t stream);

/* Human-readable text for a qs_status or, for values >= 100, for the device
 * code (value - 100).  Never NULL. */
const char* qs_status_string(int32_t code);

/* Copies *dev_status to *host_code, waiting for `stream`; resets the device
 * word to 0 when reset != 0. */
qs_status qs_read_status(const int32_t* dev_status, int32_t* host_code, int32_t reset,
                         qs_stream_t stream);

/* Bytes of workspace `op` needs for these sizes (0 is possible).
 *   max_blocks_per_req: MMBPR*BS for the Quest selector, MKBPR otherwise.
 *   sel_heads: rows of the selection fed to the attention (N or H). */
qs_status qs_workspace_size(qs_op op, int32_t B, int32_t H, int32_t N, int32_t D,
                            int32_t BS, int32_t k, int32_t max_blocks_per_req,
                            int32_t sel_heads, size_t* bytes);

/*
 * Quest metadata (CANN page, 'quest_prefill_metadata: metadata construction').
 * For every request b, in-sequence KV block j < nb_b and KV head n: the
 * channel-wise max and min of K over the block's valid tokens
 * (t < min(BS, seq_len - j*BS)), written to row j % BS, head n of metadata
 * block meta_block_tables[b][j / BS].  Rows j >= nb_b of the metadata blocks
 * the request uses (slots < ceil(nb_b / BS)) are zero-filled; nothing else is
 * written.  Max/min are exact (the results are input elements; -0 orders
 * below +0).  kv_dtype: fp32, bf16 or fp16; maxblocks/minblocks have that
 * dtype.  MMBPR must be >= ceil(MKBPR / BS).
 */
qs_status qs_prefill_metadata(const void* k_cache, qs_dtype kv_dtype, int32_t num_kv_blocks,
                              int32_t BS, int32_t N, int32_t D, const int32_t* seq_lens,
                              int32_t B, const int32_t* block_tables, int32_t MKBPR,
                              const int32_t* meta_block_tables, int32_t MMBPR,
                              int32_t num_meta_blocks, void* maxblocks, void* minblocks,
                              int32_t* dev_status, qs_stream_t stream);

/*
 * Incremental Quest metadata update after decoding (the CANN page's
 * tokens_since_metadata_update: the metadata is refreshed every BS decoded
 * tokens).  The metadata was last built or updated when request b held
 * prev_lens[b] tokens; it now holds seq_lens[b].  Rebuilds, as
 * qs_prefill_metadata would, the rows of blocks prev_lens[b]/BS ..
 * ceil(seq_lens[b]/BS) - 1 (the block that held the last tokens, possibly
 * partial, and every block begun since) and zero-fills the rows past the new
 * block count inside the metadata blocks begun since prev_lens (rows past the
 * block count in metadata blocks already in use were zeroed by the earlier
 * build); no other row is read or written.  Hence qs_prefill_metadata at
 * prev_lens followed by this call leaves exactly what qs_prefill_metadata at
 * seq_lens writes, at a cost proportional to the tokens added.
 * prev_lens: device int32 [B].  A request with prev_lens[b] < 0 or
 * prev_lens[b] > seq_lens[b] is skipped with QS_DEV_ESEQ_LEN.  Other arguments
 * and errors as for qs_prefill_metadata; NULL prev_lens: QS_EINVAL.
 */
qs_status qs_update_metadata(const void* k_cache, qs_dtype kv_dtype, int32_t num_kv_blocks,
                             int32_t BS, int32_t N, int32_t D, const int32_t* prev_lens,
                             const int32_t* seq_lens, int32_t B, const int32_t* block_tables,
                             int32_t MKBPR, const int32_t* meta_block_tables, int32_t MMBPR,
                             int32_t num_meta_blocks, void* maxblocks, void* minblocks,
                             int32_t* dev_status, qs_stream_t stream);

/*
 * Quest block selection (CANN page, 'quest_block_select_paged', steps 1-3).
 * qg[b][n] = mean of the H/N query heads of group n (fp32); block score
 * s_j = sum_d max(qg_d*max_jd, qg_d*min_jd) (fp32) for j < nb_b; the top
 * k - |F| non-forced blocks by (score descending, index ascending) plus the
 * forced set F, written ascending into selected [B, N, k], -1 padded.
 * tokens_since_metadata_update = t: t < 0 disables the window (F empty);
 * t >= 0 forces F = {0} U [w0, nb_b), w0 = min(floor((seq_len - t)/BS), nb_b-1)
 * (the blocks whose metadata the last update, t tokens ago at a multiple of
 * BS, did not cover).  Requires k >= 2 + ceil(t/BS) when t >= 0 (|F| bound).
 * scores_opt: NULL, or [B, N, MMBPR*BS] fp32 that receives s_j for j < nb_b.
 * q_dtype, meta_dtype: fp32, bf16 or fp16.  D in {64, 128}.
 */
qs_status qs_block_select_paged(const void* q, qs_dtype q_dtype, const void* maxblocks,
                                const void* minblocks, qs_dtype meta_dtype,
                                const int32_t* meta_block_tables, int32_t MMBPR,
                                int32_t num_meta_blocks, const int32_t* seq_lens, int32_t B,
                                int32_t H, int32_t N, int32_t D, int32_t BS, int32_t k,
                                int32_t tokens_since_metadata_update, int32_t* selected,
                                float* scores_opt, void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, qs_stream_t stream);

/*
 * Probe / prefill-importance selection (Kestrel-LLM 10-2, sections 1-2), one
 * selection per QUERY head: selected [B, H, k].
 *  probe_j = max over positions ps = p0, p0+step, ... < p_end of q_h . K[ps]
 *           (p0 = j*BS, p_end = min(p0+BS, seq_len), step = max(1,
 *           (p_end-p0)/n_probe); fp32 dot; int8 caches: (s_q*s_k)*int_dot with
 *           q quantised per (b,h) as s_q = max|q|/127, q8 = rint(q/s_q)).
 *  importance: NULL, or [B, importance_stride] fp32 per-token prefill
 *           importance; imp_j = fp32 sum of the block's tokens in order.
 *  Picks: (k+1)/2 blocks by importance (ties to the lower index), the rest by
 *  probe score (ties to the lower index), stopping when blocks run out; then
 *  if block nb-1 is missing and a probe pick exists, it replaces the probe
 *  pick with the lowest probe score (ties: the larger index).  Importance
 *  picks are never evicted.  D in {64, 128}; n_probe >= 1 (values < 1 act as 1).
 */
qs_status qs_probe_select(const void* q, qs_dtype q_dtype, const void* k_cache,
                          const float* k_scale, qs_dtype kv_dtype, int32_t num_kv_blocks,
                          const int32_t* block_tables, int32_t MKBPR, const int32_t* seq_lens,
                          const float* importance, int32_t importance_stride, int32_t B,
                          int32_t H, int32_t N, int32_t D, int32_t BS, int32_t k,
                          int32_t n_probe, int32_t* selected, void* workspace,
                          size_t workspace_bytes, int32_t* dev_status, qs_stream_t stream);

/*
 * Exact decode attention over the selected blocks only (Kestrel-LLM 10-2,
 * section 2; block indices mapped through block_tables per the CANN page).
 * For query head h of request b: T = tokens t < min(BS, seq_len - j*BS) of the
 * blocks j listed in selected[b][s] (s = h / (H/N) when sel_heads == N, s = h
 * when sel_heads == H; entries < 0 skipped; listed blocks must be distinct),
 * logits l = softmax_scale * q_h . K (int8: softmax_scale * s_q*s_k * int_dot),
 * p = softmax of l over T only, out[b][h] = sum p * V (fp32, [B, H, D]).
 * lse_opt: NULL or [B, H] fp32 natural-log log-sum-exp of the logits.  An
 * empty T gives out = 0 and lse = -inf.  Split-K over the selected blocks; the
 * partial results are merged on the device (no host round trip).
 * D in {64, 128}; BS a multiple of 16, <= 4096; H/N (sel_heads == N) in {1,2,4}.
 */
qs_status qs_sparse_decode_attn(const void* q, qs_dtype q_dtype, const void* k_cache,
                                const void* v_cache, const float* k_scale, const float* v_scale,
                                qs_dtype kv_dtype, int32_t num_kv_blocks,
                                const int32_t* block_tables, int32_t MKBPR,
                                const int32_t* seq_lens, const int32_t* selected,
                                int32_t sel_heads, int32_t k, float softmax_scale, int32_t B,
                                int32_t H, int32_t N, int32_t D, int32_t BS, float* out,
                                float* lse_opt, void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, qs_stream_t stream);

/*
 * qs_sparse_decode_attn without a workspace, for callers that cannot allocate
 * device memory (a decode loop that forbids allocations once it is running, a
 * plugin that is handed only input and output pointers).  The pages describe
 * nothing like it; it exists for those callers.  Same arguments, layouts,
 * results and device-side error reporting as qs_sparse_decode_attn.
 *  - Scratch comes from one fixed 4 MiB array in device memory that the
 *    library holds on every GPU that loads it, until the process exits.  A
 *    call needs qs_workspace_size(QS_OP_SPARSE_ATTN, ...) bytes of it: 256
 *    bytes per 64 units of arrival counters plus 2*units + 1024 partial slots
 *    of G*(D+2) floats (units = B*sel_heads, G = H/N when sel_heads == N, else
 *    1).  At H/N = 4, D = 128 that admits at most 495 (request, KV head)
 *    units; sizes that need more than 4 MiB return QS_EWORKSPACE.
 *  - The first call on a device looks up the array's device address; make
 *    that first call outside of any stream capture.
 *  - Once every argument check has passed, a call clears the part of the
 *    array that must start at zero (an async memset on `stream`), then runs
 *    the attention; a rejected call enqueues nothing.  All calls on a device
 *    share the array: calls that overlap on the GPU race -- keep them on one
 *    stream.
 *  - Allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 */
qs_status qs_sparse_decode_attn_noalloc(const void* q, qs_dtype q_dtype, const void* k_cache,
                                        const void* v_cache, const float* k_scale,
                                        const float* v_scale, qs_dtype kv_dtype,
                                        int32_t num_kv_blocks, const int32_t* block_tables,
                                        int32_t MKBPR, const int32_t* seq_lens,
                                        const int32_t* selected, int32_t sel_heads, int32_t k,
                                        float softmax_scale, int32_t B, int32_t H, int32_t N,
                                        int32_t D, int32_t BS, float* out, float* lse_opt,
                                        int32_t* dev_status, qs_stream_t stream);

/* Where the fixed scratch of qs_sparse_decode_attn_noalloc lives on the
 * current device: its device address and its size in bytes (looked up on the
 * first use on a device, like the entry point's first call; allocates
 * nothing).  For callers that want to check the size limit or inspect the
 * array; writing to it between calls is allowed, writing while a call runs
 * races with that call. */
qs_status qs_sparse_decode_attn_noalloc_scratch(void** device_ptr, size_t* bytes);

/* One decode step: block selection followed by the sparse attention.  Quest
 * mode reads maxblocks/minblocks/meta tables and writes selected [B, N, k];
 * probe mode reads importance and writes selected [B, H, k].  The workspace is
 * shared: size it with QS_OP_DECODE_STEP_QUEST/_PROBE.
 *
 * Quest mode can run as ONE fused kernel: every CTA selects the (request, KV
 * head) units its share of the attention touches and streams their K/V at
 * once, with no hand-off between CTAs (a unit split between two CTAs is
 * selected by both, identically).  Otherwise -- and always in probe mode --
 * the selector and the attention run as two kernels on the stream, the
 * attention launched as a programmatic dependent of the selector.
 * Both forms give the same selection and the same attention output, and
 * report the same device-side errors.  fused_select: -1 = the library's
 * choice (currently always two kernels: on GB300 the fused kernel measured
 * slower at every benchmark shape, because each CTA's K/V stream waits for
 * its own metadata scan and top-k), 0 = two kernels, 1 = the fused kernel
 * whenever the sizes fit its shared memory. */
typedef struct {
    int32_t mode;                    /* 0 = Quest, 1 = probe/importance        */
    const void* q; qs_dtype q_dtype;
    const void* k_cache; const void* v_cache;
    const float* k_scale; const float* v_scale; qs_dtype kv_dtype;
    int32_t num_kv_blocks;
    const int32_t* block_tables; int32_t MKBPR;
    const int32_t* seq_lens;
    /* Quest mode */
    const void* maxblocks; const void* minblocks;
    const int32_t* meta_block_tables; int32_t MMBPR; int32_t num_meta_blocks;
    int32_t tokens_since_metadata_update;
    /* probe mode */
    const float* importance; int32_t importance_stride; int32_t n_probe;
    /* sizes */
    int32_t B, H, N, D, BS, k;
    float softmax_scale;
    /* outputs */
    int32_t* selected; float* out; float* lse_opt;
    void* workspace; size_t workspace_bytes;
    int32_t* dev_status;
    int32_t fused_select;            /* Quest mode: -1 auto, 0 off, 1 on     */
} qs_step_params;

qs_status qs_sparse_decode_step(const qs_step_params* params, qs_stream_t stream);

/* How many kernels qs_sparse_decode_step(params) launches: 1 when it takes the
 * fused Quest kernel; 3 when the Quest selector scans (a unit of more metadata
 * rows, MMBPR*BS, than its one-CTA form scores in one load step: 128 rows at
 * D = 128 with bf16/fp16 metadata, 64 with fp32; 256 and 128 at D = 64) and
 * then ranks each unit in a second kernel, before the attention; else 2
 * (selector + attention).  Enqueues nothing and reads no device memory.
 * Returns QS_EINVAL for a NULL argument, QS_EWORKSPACE when the workspace is
 * too small to hold the selector part. */
qs_status qs_step_kernels(const qs_step_params* params, int32_t* kernels);

/*
 * Prefill importance producer (Kestrel-LLM 10-2, section 1, signal 2, and the
 * decode call site in section 2: the attention each prefill token received,
 * reduced per head and summed over the heads into prefill_importance[s] when
 * the prefill ends).  For request b with S = prefill_lens[b] tokens, query
 * head h (KV head n = h / (H/N)) and query position i < S, over the keys
 * s <= i of the request (causal, exact):
 *   l_s = softmax_scale * q[b][i][h] . K[s]   (int8 caches: softmax_scale *
 *         s_q*s_k * int_dot, the query row quantised per (i, h) exactly as the
 *         decode calls do: s_q = max|q|/127, q8 = rint(q/s_q)),
 *   lse = log sum_{s<=i} exp(l_s),   p_s = exp(l_s - lse),
 *   importance[b][s] = sum over h and i >= s of p_s   (fp32, [B, S_max];
 *         0 for s >= S; sum_s importance[b][s] = H * S).
 * q: [B, S_max, H, D] prefill query rows (fp32, bf16 or fp16; equal to
 * kv_dtype unless kv_dtype is int8).  K of position s: row s % BS of KV block
 * block_tables[b][s / BS] of k_cache [num_kv_blocks, BS, N, D] (k_scale
 * [num_kv_blocks, BS, N] fp32 for int8).  lse_opt: NULL or [B, H, S_max] fp32,
 * rows i < S receive lse (natural log).  D in {64, 128}; H/N a power of two
 * <= 64; softmax_scale > 0.  Computed in two passes (row log-sum-exp, then
 * column mass, each recomputing the logits; summation order is the kernel's)
 * on the tensor cores (tcgen05, fp32 accumulation): fp32 operands enter as
 * bf16 high and low parts, three products per q.k term, relative error at
 * most 2^-15 per term (median near 2^-19); bf16/fp16 products are exact; int8 operands enter as bf16
 * (exact), their dot products are exact, and the scales are applied after
 * them.  workspace:
 * qs_prefill_importance_workspace_size bytes (it holds the packed operand
 * tiles), no initial contents needed.  Device errors: a table entry outside
 * [0, num_kv_blocks) -> QS_DEV_EBLOCK_TABLE (that request's importance is then
 * unspecified; nothing outside the buffers is read or written); S < 0 or
 * S > min(S_max, MKBPR*BS) -> QS_DEV_ESEQ_LEN, and that request's importance
 * is left zero; a bounded wait of the tensor-core passes that runs out ->
 * QS_DEV_ETIMEOUT (the call's importance is then unspecified).
 */
qs_status qs_prefill_importance_workspace_size(int32_t B, int32_t H, int32_t N, int32_t D,
                                               int32_t S_max, qs_dtype kv_dtype,
                                               size_t* bytes);
qs_status qs_prefill_importance(const void* q, qs_dtype q_dtype, const void* k_cache,
                                const float* k_scale, qs_dtype kv_dtype,
                                int32_t num_kv_blocks, const int32_t* block_tables,
                                int32_t MKBPR, const int32_t* prefill_lens, int32_t S_max,
                                int32_t B, int32_t H, int32_t N, int32_t D, int32_t BS,
                                float softmax_scale, float* importance, float* lse_opt,
                                void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                qs_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* QUESTSPARSE_H */
