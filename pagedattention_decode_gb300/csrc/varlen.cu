// varlen.cu -- a8: packed varlen prefill + decode over the paged pool.
//
// "Building a paged inference engine from scratch, and measuring it honestly",
// section 02: one packed tensor holds the step's prefill and decode rows, and
// the attention kernel walks each sequence's block table; section 03 ("Causal
// mask during decode"): query row i of a sequence with q_len new rows and
// kv_len keys sees keys t <= kv_len - q_len + i.
//
// Rows of sequences with q_len == 1 are decode rows and run through the
// split-K decode kernel (decode.cu); chunks with q_len > 1 run on the tcgen05
// tile kernel (prefill_tc.cu).  This file holds the C ABI entry points.
#include <cuda.h>

#include "launch.h"
#include "ptx.cuh"

namespace pkv {

pkv_status run_decode(const void *q, int64_t q_stride, const pkv_cache *cache, const int32_t *tables,
                      int32_t max_blocks, const int32_t *seq_lens, const int32_t *cu_q, int32_t num_seqs,
                      int32_t num_q_heads, float scale, void *out, int32_t out_dtype, void *workspace,
                      size_t workspace_bytes, int32_t *err_word, cudaStream_t stream);
pkv_status decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t hkv, int32_t head_dim,
                                 int32_t device, size_t *bytes);
pkv_status run_decode_window(const void *q, int64_t q_stride, const pkv_cache *cache, const int32_t *tables,
                             int32_t max_blocks, const int32_t *seq_lens, const int32_t *cu_q, int32_t num_seqs,
                             int32_t num_q_heads, float scale, int32_t window, void *out, int32_t out_dtype,
                             void *workspace, size_t workspace_bytes, int32_t *err_word, cudaStream_t stream);
pkv_status run_prefill_tc(const void *q, int64_t q_stride, const pkv_cache *cache, const int32_t *tables,
                          int32_t max_blocks, const int32_t *cu_q, const int32_t *seq_lens, int32_t num_seqs,
                          int32_t total_q, int32_t max_q_len, int32_t num_q_heads, float scale, int32_t causal,
                          int32_t window, void *out, int32_t out_dtype, int32_t *err_word, cudaStream_t stream);
pkv_status check_attention_common(const void *q, int64_t q_stride, const pkv_cache *cache, const int32_t *tables,
                                  int32_t max_blocks, const int32_t *seq_lens, int32_t num_seqs,
                                  int32_t num_q_heads, void *out, int32_t out_dtype, const char *what);

}  // namespace pkv

using namespace pkv;

extern "C" {

pkv_status pkv_attn_varlen_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t device, size_t *bytes) {
    PKV_CHECK_ARG(bytes && num_seqs >= 0 && num_kv_heads > 0 && num_q_heads > 0 && head_dim > 0,
                  PKV_ERR_INVALID_ARG, "bad argument");
    pkv_status st = decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, device, bytes);
    return st == PKV_OK ? ok() : st;
}

static pkv_status varlen_impl(const void *q, int64_t q_token_stride, const pkv_cache *cache,
                              const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *cu_seqlens_q,
                              const int32_t *seq_lens, int32_t num_seqs, int32_t total_q, int32_t max_q_len,
                              int32_t num_q_heads, float scale, int32_t causal, int32_t window, void *out,
                              int32_t out_dtype, void *workspace, size_t workspace_bytes, int32_t *err_word,
                              pkv_stream stream, const char *what) {
    PKV_CHECK_ARG(total_q >= 0 && max_q_len >= 0, PKV_ERR_INVALID_ARG, "negative total_q or max_q_len");
    // with no query rows (total_q == 0: every sequence's row set is empty) q and
    // out hold nothing and may be NULL; the call does nothing
    pkv_status st = check_attention_common(q, q_token_stride, cache, block_tables, max_blocks_per_seq, seq_lens,
                                           total_q > 0 ? num_seqs : 0, num_q_heads, out, out_dtype, what);
    if (st != PKV_OK) return st;
    if (num_seqs == 0 || total_q == 0) return ok();
    PKV_CHECK_ARG(cu_seqlens_q, PKV_ERR_INVALID_ARG, "cu_seqlens_q is NULL");
    PKV_CHECK_ARG(num_seqs <= 65535, PKV_ERR_UNSUPPORTED, "at most 65535 sequences per call");
    // decode rows (q_len == 1) through the split-K decode kernels
    st = run_decode_window(q, q_token_stride, cache, block_tables, max_blocks_per_seq, seq_lens, cu_seqlens_q,
                           num_seqs, num_q_heads, scale, window, out, out_dtype, workspace, workspace_bytes, err_word,
                           stream);
    if (st != PKV_OK) return st;
    if (max_q_len <= 1) return ok();
    st = run_prefill_tc(q, q_token_stride, cache, block_tables, max_blocks_per_seq, cu_seqlens_q, seq_lens, num_seqs,
                        total_q, max_q_len, num_q_heads, scale, causal, window, out, out_dtype, err_word, stream);
    return st == PKV_OK ? ok() : st;
}

pkv_status pkv_attn_varlen(const void *q, int64_t q_token_stride, const pkv_cache *cache, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                           int32_t num_seqs, int32_t total_q, int32_t max_q_len, int32_t num_q_heads, float scale,
                           int32_t causal, void *out, int32_t out_dtype, void *workspace, size_t workspace_bytes,
                           int32_t *err_word, pkv_stream stream) {
    return varlen_impl(q, q_token_stride, cache, block_tables, max_blocks_per_seq, cu_seqlens_q, seq_lens, num_seqs,
                       total_q, max_q_len, num_q_heads, scale, causal, 0, out, out_dtype, workspace, workspace_bytes,
                       err_word, stream, "pkv_attn_varlen");
}

pkv_status pkv_attn_varlen_window(const void *q, int64_t q_token_stride, const pkv_cache *cache,
                                  const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *cu_seqlens_q,
                                  const int32_t *seq_lens, int32_t num_seqs, int32_t total_q, int32_t max_q_len,
                                  int32_t num_q_heads, float scale, int32_t causal, int32_t window, void *out,
                                  int32_t out_dtype, void *workspace, size_t workspace_bytes, int32_t *err_word,
                                  pkv_stream stream) {
    return varlen_impl(q, q_token_stride, cache, block_tables, max_blocks_per_seq, cu_seqlens_q, seq_lens, num_seqs,
                       total_q, max_q_len, num_q_heads, scale, causal, window, out, out_dtype, workspace,
                       workspace_bytes, err_word, stream, "pkv_attn_varlen_window");
}

}  // extern "C"
