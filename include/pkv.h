/*
 * pkv.h -- C ABI of libpkv, the GB300 (sm_103a) paged KV cache attention path.
 *
 * Keys and values live in fixed-size physical blocks of a pool; each sequence
 * reaches its tokens through a block table (logical block -> physical id).
 * This header declares the device calls of that path (slot write, decode
 * attention with split-K, packed varlen prefill/decode attention, block copy)
 * and the host block allocator that produces the block tables and slots.
 *
 * Sources (pages on paged KV caches):
 *  [P1] "Build a paged KV cache manager from scratch" -- block pool with
 *       refcounts, fork, copy-on-write, prefix sharing.
 *  [P2] "How to Implement Paged Attention in PyTorch and vLLM" -- pool layout,
 *       free stack, pos // block_size and pos % block_size, the gather-and-
 *       attend definition, the fused kernels that read block tables directly.
 *  [P3] "nanoserve day 14: the block allocator" -- free stack + handed-out set,
 *       atomic allocate_for, double-free error, exhaustion error.
 *  [P4] "Building a paged inference engine from scratch, and measuring it
 *       honestly" -- packed varlen prefill+decode over a block table, the
 *       causal offset kv_len - q_len + i, per-block-per-head layouts.
 *
 * Conventions (all calls):
 *  - Every call returns a pkv_status; PKV_OK is 0.  No exception or abort
 *    crosses the ABI.  pkv_last_error() gives a thread-local message for the
 *    last failing call of the calling thread.
 *  - Device memory is owned by the caller.  The library allocates no device
 *    memory; scratch for split-K is a caller buffer whose size the matching
 *    *_workspace_size call reports.
 *  - Device calls are asynchronous on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  Argument checks that need no device data are
 *    done on the host before any launch; a failing check launches nothing.
 *    Kernels are launched as programmatic dependents of the work before them
 *    on the stream and wait for that grid (complete, memory visible) before
 *    touching device memory, so inputs written by any earlier kernel on the
 *    stream are seen.  No call synchronises the host or allocates, so a step
 *    of calls can be captured in a CUDA graph.
 *  - `err_word` (optional, may be NULL) is a device int32 the kernels OR bits
 *    into (PKV_DEVERR_*) when they meet bad device-side data (a slot or block
 *    id outside the pool, a wait that ran out).  The offending item is
 *    skipped, never trapped.  Read it after the stream is synchronised; the
 *    caller clears it.
 *  - Cache layout: K and V pools are separate contiguous tensors
 *    [num_blocks, block_size, num_kv_heads, head_dim] of the same 16-bit float
 *    type ([P2] "Build the block allocator and block tables in PyTorch": the
 *    pool tensor, with the layer axis taken out -- one pkv_cache per layer).
 *    A slot is phys * block_size + offset: the row of the pool seen as
 *    [num_blocks * block_size, num_kv_heads, head_dim].
 *  - Query head h reads KV head h / (num_q_heads / num_kv_heads): contiguous
 *    groups ([P2] "Compute reference attention without hiding the layout",
 *    GQA head expansion).
 *
 * Supported shapes on the GPU: head_dim 64 or 128; block_size a multiple of
 * 16 up to 256; num_q_heads / num_kv_heads in {1, 2, 4, 8}; 16-bit types
 * fp16 and bf16; num_kv_heads * head_dim * 2 bytes a multiple of 16.
 * Anything else returns PKV_ERR_UNSUPPORTED before any launch.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(_WIN32)
#define PKV_API __declspec(dllexport)
#else
#define PKV_API __attribute__((visibility("default")))
#endif

struct CUstream_st;
typedef struct CUstream_st *pkv_stream; /* same type as cudaStream_t */

typedef int32_t pkv_status;
#define PKV_OK 0
#define PKV_ERR_INVALID_ARG 1  /* NULL pointer, negative size, misaligned pointer */
#define PKV_ERR_DTYPE 2        /* unknown or mismatched element type */
#define PKV_ERR_SHAPE 3        /* shapes that do not fit together */
#define PKV_ERR_OUT_OF_RANGE 4 /* a host-side id or index outside its range */
#define PKV_ERR_EXHAUSTED 5    /* [P3] KVCacheExhausted: the pool cannot cover a request */
#define PKV_ERR_DOUBLE_FREE 6  /* [P3] freeing an id that is not handed out */
#define PKV_ERR_CUDA 7         /* a CUDA runtime/driver call failed (message has details) */
#define PKV_ERR_WORKSPACE 8    /* workspace NULL or smaller than *_workspace_size */
#define PKV_ERR_UNSUPPORTED 9  /* valid, but outside the shapes compiled for the GPU */

/* bits of the device error word */
#define PKV_DEVERR_SLOT 0x1    /* pkv_write_kv: slot >= num_blocks * block_size (row skipped) */
#define PKV_DEVERR_BLOCK 0x2   /* attention: table entry outside [0, num_blocks) (block 0 read instead; output invalid) */
#define PKV_DEVERR_PAIR 0x4    /* pkv_copy_blocks: src or dst outside [0, num_blocks) (pair skipped) */
#define PKV_DEVERR_TIMEOUT 0x8 /* a bounded wait inside a kernel ran out; the kernel returned early */
#define PKV_DEVERR_LENGTH 0x10 /* a sequence longer than its table, or q_len > kv_len (sequence skipped) */

typedef enum pkv_dtype { PKV_F16 = 0, PKV_BF16 = 1, PKV_F32 = 2 } pkv_dtype;

/* One layer's K and V pools (device pointers, 16-byte aligned). */
typedef struct pkv_cache {
    void *k;              /* [num_blocks, block_size, num_kv_heads, head_dim] */
    void *v;              /* same shape and type as k */
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t dtype;        /* PKV_F16 or PKV_BF16 */
} pkv_cache;

/* ---- library ------------------------------------------------------------ */

/* Version of this ABI (bumped on any incompatible change). */
PKV_API int32_t pkv_abi_version(void);
/* Thread-local message of the last failing call on this thread ("" if none). */
PKV_API const char *pkv_last_error(void);
/* Static name of a status code. */
PKV_API const char *pkv_status_string(pkv_status status);

/* ---- a2: slot write ----------------------------------------------------- */
/*
 * [P2] "Build the block allocator and block tables in PyTorch"
 * (PagedKVCache.append_token) and "How to implement paged attention: the
 * minimal data flow", step 3: the K and V of a new token land at offset
 * pos % block_size of physical block table[pos // block_size].  This call does
 * the write for a batch of tokens whose slots the host already computed.
 *
 *   k, v          device [num_tokens, num_kv_heads, head_dim] of cache->dtype;
 *                 token t's row starts at element t * kv_token_stride (heads
 *                 and dims contiguous); 16-byte aligned rows.
 *   slot_mapping  device int64 [num_tokens]; slot < 0 skips the token; a slot
 *                 >= num_blocks * block_size sets PKV_DEVERR_SLOT and is skipped.
 *   cache         the layer's pools (written in place).
 * Bit-exact copy; duplicate slots in one call race (the caller's error).
 */
PKV_API pkv_status pkv_write_kv(const void *k, const void *v, int64_t kv_token_stride,
                                const int64_t *slot_mapping, int32_t num_tokens,
                                const pkv_cache *cache, int32_t *err_word, pkv_stream stream);

/* ---- a3..a7: decode attention ------------------------------------------- */
/*
 * [P2] "Compute reference attention without hiding the layout" defines the
 * result (gather the sequence's K/V through its table, scale * q.k, softmax
 * over keys, weighted sum of V); "Map the PyTorch design to vLLM
 * PagedAttention" names the fused kernels that walk the block table instead of
 * gathering.  One query row per sequence; every key 0 .. seq_lens[s]-1 is
 * attended (the token written this step included).
 *
 * The kernel splits the concatenated 16-token sub-blocks of all sequences
 * evenly over one CTA per SM; a sequence cut by that split is merged by a
 * second kernel from per-part (max, sum, unnormalised output) records in the
 * workspace (flash-decoding style split-K).
 *
 *   q             device [num_seqs, num_q_heads, head_dim], row s at s * q_token_stride.
 *   block_tables  device int32 [num_seqs, max_blocks_per_seq]; entries past
 *                 ceil(seq_lens[s] / block_size) are never read.
 *   seq_lens      device int32 [num_seqs]; 0 gives an all-zero output row.
 *   scale         multiplies q.k before the softmax (1/sqrt(head_dim) usually).
 *   out           device [num_seqs, num_q_heads, head_dim] of out_dtype, 16-byte aligned
 *                 (PKV_F32, or the cache's dtype).
 *   workspace     device scratch of >= pkv_attn_decode_workspace_size bytes,
 *                 256-byte aligned; its contents on entry do not matter.  That
 *                 size covers the 16-bit, windowed and int8 decode calls alike.
 */
PKV_API pkv_status pkv_attn_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                                  int32_t num_kv_heads, int32_t head_dim,
                                                  int32_t device, size_t *bytes);
PKV_API pkv_status pkv_attn_decode(const void *q, int64_t q_token_stride, const pkv_cache *cache,
                                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                                   const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_heads,
                                   float scale, void *out, int32_t out_dtype, void *workspace,
                                   size_t workspace_bytes, int32_t *err_word, pkv_stream stream);

/*
 * Decode attention without a caller workspace.  The pages have no
 * counterpart to this call: it exists for callers that cannot allocate device
 * memory -- a host program embedding libpkv in a process whose device memory
 * is owned by another runtime's allocator, or a loop that must not call
 * cudaMalloc because it synchronises the device.  Same arguments, result and
 * errors as pkv_attn_decode, minus the workspace.
 *
 * Its scratch is a fixed array of PKV_NOALLOC_SCRATCH_BYTES inside the
 * library's device image, present on every device that loads the library
 * until the process exits.  A call whose split-K records need more (many
 * sequences or query heads) returns PKV_ERR_WORKSPACE and launches nothing.
 * The first call on a device looks up the array's address on the current
 * device (cudaGetSymbolAddress); make that first call before any stream
 * capture.  A reset of the device (cudaDeviceReset, or another teardown of
 * its primary context) loads the library's module again, possibly at another
 * address: the first call after it looks the address up again, so it too
 * belongs before any capture.  All calls share the one array and nothing needs clearing between
 * them, but calls that overlap on the GPU (other streams, other threads) race
 * on it.  The call itself allocates nothing.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (16 * 1024 * 1024)
PKV_API pkv_status pkv_attn_decode_noalloc(const void *q, int64_t q_token_stride, const pkv_cache *cache,
                                           const int32_t *block_tables, int32_t max_blocks_per_seq,
                                           const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_heads,
                                           float scale, void *out, int32_t out_dtype, int32_t *err_word,
                                           pkv_stream stream);

/* ---- a8: packed varlen prefill + decode ---------------------------------- */
/*
 * [P4] section 02 (the paged FlashAttention-2 kernel reads K/V through the
 * block table; the model runner packs prefill and decode rows into one flat
 * tensor) and section 03 ("Causal mask during decode"): query row i (0-based)
 * of sequence s, which has q_len = cu_seqlens_q[s+1] - cu_seqlens_q[s] new
 * rows and kv_len = seq_lens[s] keys (the new rows' keys already written),
 * attends keys t <= kv_len - q_len + i when causal != 0, else all kv_len keys.
 * Rows with q_len == 1 take the split-K decode path; longer chunks run on the
 * tcgen05 tensor cores (accumulators in tensor memory), with the softmax
 * weights entering P V as fp16 (an fp16 cache) or as a bf16 hi + lo pair (a
 * bf16 cache).  q_len > kv_len sets PKV_DEVERR_LENGTH and skips the sequence.
 *
 *   q             device [total_q, num_q_heads, head_dim], row r at r * q_token_stride;
 *                 when max_q_len > 1, q and its row stride must be 16-byte aligned.
 *                 total_q == 0 (every row set empty) is a no-op; q and out may be NULL.
 *   cu_seqlens_q  device int32 [num_seqs + 1], nondecreasing, cu[0] = 0, cu[num_seqs] = total_q.
 *   max_q_len     host upper bound on any q_len (sizes the tile grid).
 *   out           device [total_q, num_q_heads, head_dim] of out_dtype.
 *   workspace     >= pkv_attn_varlen_workspace_size bytes.
 */
PKV_API pkv_status pkv_attn_varlen_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                                  int32_t num_kv_heads, int32_t head_dim,
                                                  int32_t device, size_t *bytes);
PKV_API pkv_status pkv_attn_varlen(const void *q, int64_t q_token_stride, const pkv_cache *cache,
                                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                                   const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                                   int32_t num_seqs, int32_t total_q, int32_t max_q_len,
                                   int32_t num_q_heads, float scale, int32_t causal, void *out,
                                   int32_t out_dtype, void *workspace, size_t workspace_bytes,
                                   int32_t *err_word, pkv_stream stream);

/* ---- sliding-window variants --------------------------------------------- */
/*
 * [P2] "PagedAttention vs sliding-window attention, RadixAttention, and SSMs":
 * with a sliding window each query attends only to the most recent `window`
 * tokens, and paged allocation still holds them.  A row whose last visible key
 * is `last` (L - 1 for a decode row, kv_len - q_len + i for causal chunk row
 * i, kv_len - 1 without causality) sees keys max(0, last - window + 1) .. last.
 * Sub-blocks wholly before the window are never read.  window <= 0 means no
 * window; otherwise arguments, layouts and errors are those of
 * pkv_attn_decode / pkv_attn_varlen (same workspace sizes).
 */
PKV_API pkv_status pkv_attn_decode_window(const void *q, int64_t q_token_stride, const pkv_cache *cache,
                                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                                          const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_heads,
                                          float scale, int32_t window, void *out, int32_t out_dtype,
                                          void *workspace, size_t workspace_bytes, int32_t *err_word,
                                          pkv_stream stream);
PKV_API pkv_status pkv_attn_varlen_window(const void *q, int64_t q_token_stride, const pkv_cache *cache,
                                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                                          const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                                          int32_t num_seqs, int32_t total_q, int32_t max_q_len,
                                          int32_t num_q_heads, float scale, int32_t causal, int32_t window,
                                          void *out, int32_t out_dtype, void *workspace, size_t workspace_bytes,
                                          int32_t *err_word, pkv_stream stream);

/* ---- decode with the step's new key / value written in the same call ------- */
/*
 * [P2] "Build the block allocator and block tables in PyTorch": a decode step
 * first stores the new token's key and value in the slot of position
 * seq_len - 1 of its sequence, then attends over all seq_len keys.  This call
 * does both in one kernel: row s of k_new / v_new ([num_seqs, num_kv_heads,
 * head_dim], row s at s * kv_token_stride, 16-byte aligned) is written to
 * slot table[s][(L - 1) / bs] * bs + (L - 1) % bs of the pools (L =
 * seq_lens[s]; nothing is written when L == 0), and out is what
 * pkv_write_kv with those slots followed by pkv_attn_decode_window(window)
 * gives.  The row is written by the CTA that reads the 16-token sub-block
 * holding it, before that read; no other CTA reads that sub-block.  A block
 * id outside [0, num_blocks) in that table entry sets PKV_DEVERR_BLOCK and
 * the row is not written.  Other arguments, layouts and errors are those of
 * pkv_attn_decode_window (window <= 0: none); same workspace size.
 */
PKV_API pkv_status pkv_attn_decode_append(const void *q, int64_t q_token_stride, const void *k_new,
                                          const void *v_new, int64_t kv_token_stride, const pkv_cache *cache,
                                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                                          const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_heads,
                                          float scale, int32_t window, void *out, int32_t out_dtype,
                                          void *workspace, size_t workspace_bytes, int32_t *err_word,
                                          pkv_stream stream);

/* ---- int8 KV cache --------------------------------------------------------- */
/*
 * [P4] section 02, "INT8 KV cache design": keys and values stored as
 * symmetric int8 with one scale per block per KV head and no zero point; a
 * write re-quantises the block (its earlier rows are dequantised with the
 * stored scale, the new rows join them, the scale becomes max|x| / 127 and
 * every row is re-quantised); the attention kernel dequantises right before
 * its matrix products.  Halves the bytes a decode step reads.
 *
 *   k, v         int8 pools [num_blocks, block_size, num_kv_heads, head_dim]
 *   k_scale,     float32 [num_blocks, num_kv_heads]: value = code * scale
 *   v_scale
 *   dtype        PKV_F16 or PKV_BF16: the type of q, of the new K/V rows given
 *                to pkv_write_kv_int8 and of 16-bit outputs
 * Supported on the GPU: head_dim 128, num_kv_heads a multiple of 4, the other
 * limits of the 16-bit cache.
 */
typedef struct pkv_cache_i8 {
    int8_t *k;
    int8_t *v;
    float *k_scale;
    float *v_scale;
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t dtype;
} pkv_cache_i8;

/*
 * Quantised slot write: rows k[t], v[t] (16-bit of cache->dtype, layout as in
 * pkv_write_kv) go to slot_mapping[t].  Per block written and per KV head the
 * block is re-quantised as above, all integer decisions in binary32 (round
 * half to even, codes clamped to +-127, scale 0 for an all-zero block).  The
 * block's earlier rows are those below the lowest offset the call writes into
 * it.  The slots a call writes into one block must be consecutive entries of
 * slot_mapping (the allocator's order); a later entry with the same slot
 * replaces an earlier one.
 */
PKV_API pkv_status pkv_write_kv_int8(const void *k, const void *v, int64_t kv_token_stride,
                                     const int64_t *slot_mapping, int32_t num_tokens, const pkv_cache_i8 *cache,
                                     int32_t *err_word, pkv_stream stream);
/*
 * Decode attention over an int8 cache (arguments and errors as
 * pkv_attn_decode_window, window <= 0 meaning none): scores use
 * k_scale[block][head] * (q . codes), the softmax weights are multiplied by
 * v_scale[block][head] before the product with the V codes.  Workspace size:
 * pkv_attn_decode_workspace_size.
 */
PKV_API pkv_status pkv_attn_decode_int8(const void *q, int64_t q_token_stride, const pkv_cache_i8 *cache,
                                        const int32_t *block_tables, int32_t max_blocks_per_seq,
                                        const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_heads,
                                        float scale, int32_t window, void *out, int32_t out_dtype,
                                        void *workspace, size_t workspace_bytes, int32_t *err_word,
                                        pkv_stream stream);

/* ---- a10: block copy for copy-on-write ----------------------------------- */
/*
 * [P1] Architecture Overview, copy-on-write: when sequences that share a
 * block diverge, the diverging block is duplicated; [P2] "Map the PyTorch
 * design to vLLM PagedAttention": a shared block is copied only on the first
 * divergent write.  For each (src, dst) pair, block dst of every listed
 * layer's K and V pools becomes a bit copy of block src.
 *
 *   caches         host array [num_layers] of pools with equal geometry.
 *   src_dst_pairs  device int64 [num_pairs, 2]; an id outside the pool sets
 *                  PKV_DEVERR_PAIR and skips the pair.  A dst that is also a
 *                  src, or repeated, races: pkv_check_copy_pairs (host) catches it.
 * Runs before the write of the step's new rows, on the same stream.
 */
PKV_API pkv_status pkv_copy_blocks(const pkv_cache *caches, int32_t num_layers,
                                   const int64_t *src_dst_pairs, int32_t num_pairs,
                                   int32_t *err_word, pkv_stream stream);
/* Host check of a pair list: ids in range, src != dst, no repeated dst, no dst that is a src. */
PKV_API pkv_status pkv_check_copy_pairs(const int64_t *host_pairs, int32_t num_pairs,
                                        int32_t num_blocks);

/* ---- a1, a9: host block allocator ----------------------------------------- */
/*
 * [P3] "What I learned": free ids on a stack, handed-out ids in a set, every
 * id in exactly one of them; allocate pops; allocate_for(n) takes
 * ceil(n / block_size) blocks or none (PKV_ERR_EXHAUSTED); freeing an id that
 * is not handed out is PKV_ERR_DOUBLE_FREE and changes nothing.  [P2]: the
 * stack starts as num_blocks-1 .. 0 (first pop returns 0), reuse is LIFO, a
 * sequence takes a new block when pos % block_size == 0.  [P1] Steps 2-3:
 * refcount 1 on allocation, +1 per retain / share / fork; a release that
 * drops it to 0 pushes the id back on the stack.  Copy-on-write: appending to
 * a non-full tail with refcount > 1 takes a new block, reports the pair
 * (tail, new), releases the tail and writes into the new block; the last
 * holder writes in place.  Shared prefix blocks are whole blocks, retained
 * once per holder.  All calls are serialised by an internal mutex.  Sequence
 * ids are small integers, never reused.
 */
typedef struct pkv_allocator pkv_allocator;

typedef struct pkv_alloc_counters {
    int64_t allocs;     /* blocks popped */
    int64_t frees;      /* blocks pushed back (refcount reached 0) */
    int64_t cow_copies; /* copy-on-write pairs reported */
    int64_t peak_used;  /* most blocks handed out at once */
} pkv_alloc_counters;

PKV_API pkv_status pkv_alloc_create(int32_t num_blocks, int32_t block_size, pkv_allocator **out);
PKV_API void pkv_alloc_destroy(pkv_allocator *a);
/* Make the next pops return order[0], order[1], ...: a permutation of the free ids. */
PKV_API pkv_status pkv_alloc_set_free_order(pkv_allocator *a, const int32_t *order, int32_t n);
PKV_API pkv_status pkv_alloc_allocate(pkv_allocator *a, int32_t *block_id);
/* ceil(num_tokens / block_size) ids into out_ids[capacity], all or nothing. */
PKV_API pkv_status pkv_alloc_allocate_for(pkv_allocator *a, int64_t num_tokens, int32_t *out_ids,
                                          int32_t capacity, int32_t *num_out);
PKV_API pkv_status pkv_alloc_free(pkv_allocator *a, int32_t block_id);
/* Releases every listed id once, in list order; all or nothing. */
PKV_API pkv_status pkv_alloc_free_all(pkv_allocator *a, const int32_t *ids, int32_t n);
PKV_API pkv_status pkv_alloc_retain(pkv_allocator *a, int32_t block_id);
PKV_API int32_t pkv_alloc_refcount(const pkv_allocator *a, int32_t block_id); /* 0 if free */
PKV_API int32_t pkv_alloc_num_free(const pkv_allocator *a);
PKV_API int64_t pkv_alloc_blocks_needed(const pkv_allocator *a, int64_t num_tokens);
PKV_API pkv_status pkv_alloc_counters_get(const pkv_allocator *a, pkv_alloc_counters *out);

/* New sequence holding n_shared whole shared blocks (retained once each); its
 * length is shared_tokens, which must equal n_shared * block_size. */
PKV_API pkv_status pkv_seq_create(pkv_allocator *a, const int32_t *shared_ids, int32_t n_shared,
                                  int64_t shared_tokens, int32_t *seq_id);
/* Child sharing every block of seq (each retained), same length. */
PKV_API pkv_status pkv_seq_fork(pkv_allocator *a, int32_t seq_id, int32_t *child_id);
/* Releases the sequence's blocks in table order; a second free of the same id is a no-op. */
PKV_API pkv_status pkv_seq_free(pkv_allocator *a, int32_t seq_id);
/*
 * Appends counts[i] tokens (1 each if counts is NULL) to seq_ids[i], in order,
 * all or nothing for the whole call.  Writes the slot of every new token into
 * out_slots (call order; capacity slot_capacity) and the copy-on-write pairs
 * (src, dst) into out_pairs[2 * pair_capacity]; *num_pairs gets their count.
 * A sequence may appear once per call.
 */
PKV_API pkv_status pkv_seq_append(pkv_allocator *a, const int32_t *seq_ids, const int32_t *counts,
                                  int32_t n, int64_t *out_slots, int64_t slot_capacity,
                                  int64_t *out_pairs, int32_t pair_capacity, int32_t *num_pairs);
PKV_API pkv_status pkv_seq_len(const pkv_allocator *a, int32_t seq_id, int64_t *len);
PKV_API pkv_status pkv_seq_block_table(const pkv_allocator *a, int32_t seq_id, int32_t *out,
                                       int32_t capacity, int32_t *n);
/* Batch form for a step: row i of tables[n, max_blocks] gets seq_ids[i]'s
 * table padded with -1; seq_lens[i] its length. */
PKV_API pkv_status pkv_seq_fill_tables(const pkv_allocator *a, const int32_t *seq_ids, int32_t n,
                                       int32_t *tables, int32_t max_blocks, int32_t *seq_lens);

/*
 * Prefix sharing ([P1] Step 4, the radix/prefix tree, and Step 2's LRU
 * reclaim).  The trie's children are keyed by one whole block of token ids
 * (only whole blocks are shared).
 *  - pkv_prefix_match walks `tokens` block by block and writes the ids of the
 *    matched blocks (at most `capacity`); it does not retain them: passing them
 *    to pkv_seq_create retains each once ([P1]'s listing retains twice).  With
 *    other threads evicting, use pkv_seq_create_prefixed instead.
 *  - pkv_prefix_insert publishes the whole blocks of a sequence (block_ids[j]
 *    holds tokens j*block_size .. j*block_size + block_size - 1); a new node
 *    takes one reference to its block; an existing key keeps its block.
 *  - pkv_prefix_evict removes up to max_blocks least recently used leaves whose
 *    block is held by the trie alone, releasing those blocks to the free stack;
 *    out_ids gets them in eviction order.
 * Recency is a logical clock advanced by each node a match or insert touches.
 */
PKV_API pkv_status pkv_prefix_match(pkv_allocator *a, const int32_t *tokens, int64_t num_tokens, int32_t *out_ids,
                                    int32_t capacity, int32_t *num_blocks);
/* Match and create in one step (under the allocator's lock, so no eviction can
 * come between them): a new sequence holding the matched whole blocks of
 * `tokens`, each retained once; *shared_tokens gets its length. */
PKV_API pkv_status pkv_seq_create_prefixed(pkv_allocator *a, const int32_t *tokens, int64_t num_tokens,
                                           int32_t *seq_id, int64_t *shared_tokens);
PKV_API pkv_status pkv_prefix_insert(pkv_allocator *a, const int32_t *tokens, int64_t num_tokens,
                                     const int32_t *block_ids, int32_t num_ids);
PKV_API pkv_status pkv_prefix_evict(pkv_allocator *a, int32_t max_blocks, int32_t *out_ids, int32_t *num_evicted);
PKV_API int32_t pkv_prefix_num_nodes(const pkv_allocator *a);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
