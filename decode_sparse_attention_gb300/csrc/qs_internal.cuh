// Entry points shared between the translation units of the library.
#pragma once

#include "qs_common.cuh"

namespace qs {

size_t select_workspace_bytes(int B, int N, int maxnb);
size_t probe_workspace_bytes(int B, int H, int N, int MKBPR);
size_t attn_workspace_bytes(int B, int H, int N, int D, int sel_heads);

qs_status block_select_impl(const void* q, qs_dtype q_dtype, const void* maxblocks,
                            const void* minblocks, qs_dtype meta_dtype,
                            const int32_t* meta_block_tables, int32_t MMBPR,
                            int32_t num_meta_blocks, const int32_t* seq_lens, int32_t B,
                            int32_t H, int32_t N, int32_t D, int32_t BS, int32_t k, int32_t t,
                            int32_t* selected, float* scores_opt, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream);

qs_status probe_select_impl(const void* q, qs_dtype q_dtype, const void* k_cache,
                            const float* k_scale, qs_dtype kv_dtype, int32_t num_kv_blocks,
                            const int32_t* block_tables, int32_t MKBPR, const int32_t* seq_lens,
                            const float* importance, int32_t importance_stride, int32_t B,
                            int32_t H, int32_t N, int32_t D, int32_t BS, int32_t k,
                            int32_t n_probe, int32_t* selected, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream);

// pdl: launch as a programmatic dependent of the kernel before it on the
// stream (only when that kernel writes nothing the attention reads before
// its grid-dependency wait, i.e. after the selectors).  clear_counters: zero
// the workspace's arrival counters on the stream first (after every argument
// and plan check passed), for a workspace whose contents are unknown.
qs_status sparse_attn_impl(const void* q, qs_dtype q_dtype, const void* k_cache,
                           const void* v_cache, const float* k_scale, const float* v_scale,
                           qs_dtype kv_dtype, int32_t num_kv_blocks, const int32_t* block_tables,
                           int32_t MKBPR, const int32_t* seq_lens, const int32_t* selected,
                           int32_t sel_heads, int32_t k, float softmax_scale, int32_t B, int32_t H,
                           int32_t N, int32_t D, int32_t BS, float* out, float* lse_opt,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                           cudaStream_t stream, bool pdl, bool clear_counters = false);

// Fused Quest decode step (one kernel).  Sets *taken = false, and enqueues
// nothing, when the sizes are outside what the fused kernel serves or the
// inputs would make either kernel of the two-kernel step report an error;
// the caller then runs the two-kernel step.  attn_ws: the attention part of
// the step's workspace.  launch = false only decides (*taken).
// Prefill importance on the tensor cores (every cache dtype): packs the
// operands into ws, writes the column sums of every (request, KV head, part)
// into part and the optional natural log-sum-exps; false on a launch error.
size_t importance_tc_workspace(long long B, long long H, long long N, long long D, long long S_max,
                               bool f32, bool int8, size_t* off_q, size_t* off_k, size_t* off_lse,
                               size_t* off_qs, size_t* off_ks);
// int8 (dt = I8): q holds the quantised query rows [B, S_max, H, D] and
// q_scale their scales [B, S_max, H]; k_scale the cache's [P, BS, N] scales.
bool importance_tc_launch(const void* q, const float* q_scale, Dt dt, const void* k_cache,
                          const float* k_scale, int32_t num_kv_blocks, const int32_t* block_tables,
                          int32_t MKBPR, const int32_t* lens, int32_t S_max, int32_t B, int32_t H,
                          int32_t N, int32_t D, int32_t BS, float scale_log2, float* part, int parts,
                          float* lse_out, uint8_t* ws, int32_t* status, cudaStream_t st);

qs_status quest_step_fused(const qs_step_params* p, void* attn_ws, size_t attn_ws_bytes,
                           cudaStream_t stream, bool* taken, bool launch);

}  // namespace qs
