/*
 * pkv_oracle.c -- plain, slow CPU reference for the paged KV cache path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only tests, the smoke check and the bench's CPU baseline
 * load it.  It shares no code, header, table or helper with the CUDA path.
 *
 * Everything follows the plain definitions on the pages:
 *
 *  - Slot write.  "How to Implement Paged Attention in PyTorch and vLLM",
 *    section "Build the block allocator and block tables in PyTorch"
 *    (PagedKVCache.append_token): the new K/V row of position pos lands in
 *    physical block table[pos // block_size] at offset pos % block_size.  A
 *    slot is that pair flattened, phys * block_size + offset, i.e. the row
 *    index of the pool seen as [num_blocks * block_size, kv_heads, head_dim].
 *    A negative slot means "no write".
 *
 *  - Attention.  Same page, section "Compute reference attention without
 *    hiding the layout" (reference_paged_attention): gather the sequence's
 *    K/V through its block table into contiguous arrays, map query head h to
 *    KV head h // (q_heads / kv_heads), score = scale * <q, k>, softmax over
 *    keys (computed as exp(s - max s) / sum), output = sum_t p_t v_t.
 *
 *  - Causal limit for packed rows.  "Building a paged inference engine from
 *    scratch, and measuring it honestly", section 03 ("Causal mask during
 *    decode"): query i (0-based) of a sequence with q_len new rows and kv_len
 *    keys sees keys t <= kv_len - q_len + i.
 *
 *  - Block copy.  "Build a paged KV cache manager from scratch", Architecture
 *    Overview (copy-on-write): the diverging block is duplicated; dst becomes
 *    a byte copy of src in every layer.
 *
 * Arithmetic is IEEE binary64.  fp16 / bf16 inputs are decoded exactly from
 * their bit patterns with the format definitions below.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F16 0
#define ORACLE_BF16 1

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    return sign ? -mag : mag;
}

/* bfloat16: the upper 16 bits of an IEEE binary32 (8 exponent bits, bias 127). */
static double decode_bf16(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -133); /* f * 2^-126 * 2^-7 */
    else if (e == 255)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(128 + f), e - 134); /* (1 + f/128) * 2^(e-127) */
    return sign ? -mag : mag;
}

static double decode(uint16_t x, int dtype)
{
    return dtype == ORACLE_BF16 ? decode_bf16(x) : decode_f16(x);
}

/* Exposed for the tests that pin the decoders against numpy's own casts. */
double oracle_decode_f16(uint16_t h) { return decode_f16(h); }
double oracle_decode_bf16(uint16_t b) { return decode_bf16(b); }

/*
 * Slot write: for each token t with slot >= 0, copy its [kv_heads * head_dim]
 * row of k and v into row `slot` of the caches.  Returns the number of tokens
 * written, or -1 (nothing written) if any slot lies outside the pool.
 */
int64_t oracle_write_kv(const uint16_t *k, const uint16_t *v, int64_t num_tokens,
                        int64_t row_elems, const int64_t *slots,
                        uint16_t *k_cache, uint16_t *v_cache, int64_t num_slots)
{
    int64_t written = 0;
    for (int64_t t = 0; t < num_tokens; ++t)
        if (slots[t] >= num_slots)
            return -1;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slots[t];
        if (s < 0)
            continue;
        memcpy(k_cache + s * row_elems, k + t * row_elems, (size_t)row_elems * 2);
        memcpy(v_cache + s * row_elems, v + t * row_elems, (size_t)row_elems * 2);
        ++written;
    }
    return written;
}

/*
 * Block copy of one layer: for each pair (src, dst), block dst of both caches
 * becomes a copy of block src.  Returns -1 (nothing copied) on an id outside
 * the pool.
 */
int oracle_copy_blocks(uint16_t *k_cache, uint16_t *v_cache, int64_t num_blocks,
                       int64_t block_elems, const int64_t *pairs, int64_t num_pairs)
{
    for (int64_t i = 0; i < num_pairs; ++i) {
        int64_t s = pairs[2 * i], d = pairs[2 * i + 1];
        if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks)
            return -1;
    }
    for (int64_t i = 0; i < num_pairs; ++i) {
        int64_t s = pairs[2 * i], d = pairs[2 * i + 1];
        memcpy(k_cache + d * block_elems, k_cache + s * block_elems, (size_t)block_elems * 2);
        memcpy(v_cache + d * block_elems, v_cache + s * block_elems, (size_t)block_elems * 2);
    }
    return 0;
}

/*
 * Paged attention over packed query rows.
 *
 *   q        [total_rows, num_q_heads, head_dim] (row stride q_row_stride elements)
 *   caches   [num_blocks, block_size, num_kv_heads, head_dim]
 *   tables   [num_seqs, max_blocks] int32
 *   kv_lens  [num_seqs]: keys of each sequence (already in the cache)
 *   cu_q     [num_seqs + 1]: sequence s owns query rows cu_q[s] .. cu_q[s+1]-1;
 *            NULL means one query row per sequence (decode).
 *   causal   0: every row sees all kv_len keys; 1: row i sees t <= kv_len - q_len + i.
 *   window   > 0: a row whose last visible key is `last` sees only keys
 *            t >= last - window + 1 (the most recent `window` tokens, its own
 *            included; "How to Implement Paged Attention in PyTorch and vLLM",
 *            section "PagedAttention vs sliding-window attention..."); <= 0: no
 *            window.
 *   out      [total_rows, num_q_heads, head_dim] binary64.
 *
 * A row that sees no key (kv_len == 0) is all zeros.  Returns 0, or -1 on an
 * input the definition does not cover (block id outside the pool, a table
 * too short for kv_len, q_len > kv_len under the causal rule, q heads not a
 * multiple of kv heads).
 */
int oracle_paged_attention(const uint16_t *q, int64_t q_row_stride,
                           const uint16_t *k_cache, const uint16_t *v_cache, int dtype,
                           int64_t num_blocks, int block_size, int num_kv_heads, int head_dim,
                           const int32_t *tables, int max_blocks, const int32_t *kv_lens,
                           const int32_t *cu_q, int num_seqs, int num_q_heads,
                           double scale, int causal, int window, double *out)
{
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return -1;
    const int group = num_q_heads / num_kv_heads;
    const int D = head_dim;

    /* validate first: every table entry that a key position reaches */
    for (int s = 0; s < num_seqs; ++s) {
        int64_t L = kv_lens[s];
        int64_t qlen = cu_q ? (int64_t)cu_q[s + 1] - cu_q[s] : 1;
        if (L < 0 || qlen < 0 || (causal && qlen > L && L > 0))
            return -1;
        if (L > (int64_t)max_blocks * block_size)
            return -1;
        for (int64_t t = 0; t < L; t += block_size) {
            int32_t phys = tables[(int64_t)s * max_blocks + t / block_size];
            if (phys < 0 || phys >= num_blocks)
                return -1;
        }
    }

    int failed = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int s = 0; s < num_seqs; ++s) {
        for (int g = 0; g < num_kv_heads; ++g) {
            const int64_t L = kv_lens[s];
            const int64_t row0 = cu_q ? cu_q[s] : s;
            const int64_t qlen = cu_q ? (int64_t)cu_q[s + 1] - cu_q[s] : 1;

            /* gather K and V of KV head g through the block table */
            double *K = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * D);
            double *V = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * D);
            double *p = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
            double *qd = (double *)malloc(sizeof(double) * (size_t)D);
            if (!K || !V || !p || !qd) {
#pragma omp atomic write
                failed = 1;
                free(K); free(V); free(p); free(qd);
                continue;
            }
            for (int64_t t = 0; t < L; ++t) {
                int64_t phys = tables[(int64_t)s * max_blocks + t / block_size];
                int64_t off = t % block_size;
                const int64_t base = ((phys * block_size + off) * num_kv_heads + g) * D;
                for (int d = 0; d < D; ++d) {
                    K[t * D + d] = decode(k_cache[base + d], dtype);
                    V[t * D + d] = decode(v_cache[base + d], dtype);
                }
            }

            for (int64_t i = 0; i < qlen; ++i) {
                const int64_t row = row0 + i;
                int64_t visible = L; /* keys first .. visible-1 */
                if (causal)
                    visible = L - qlen + i + 1;
                int64_t first = 0;
                if (window > 0 && visible - window > 0)
                    first = visible - window;
                for (int h = g * group; h < (g + 1) * group; ++h) {
                    double *o = out + (row * num_q_heads + h) * (int64_t)D;
                    for (int d = 0; d < D; ++d)
                        o[d] = 0.0;
                    if (visible <= 0)
                        continue;
                    for (int d = 0; d < D; ++d)
                        qd[d] = decode(q[row * q_row_stride + (int64_t)h * D + d], dtype);
                    double mx = -INFINITY;
                    for (int64_t t = first; t < visible; ++t) {
                        double dot = 0.0;
                        for (int d = 0; d < D; ++d)
                            dot += qd[d] * K[t * D + d];
                        p[t] = scale * dot;
                        if (p[t] > mx)
                            mx = p[t];
                    }
                    double Z = 0.0;
                    for (int64_t t = first; t < visible; ++t) {
                        p[t] = exp(p[t] - mx);
                        Z += p[t];
                    }
                    for (int64_t t = first; t < visible; ++t)
                        for (int d = 0; d < D; ++d)
                            o[d] += p[t] * V[t * D + d];
                    for (int d = 0; d < D; ++d)
                        o[d] /= Z;
                }
            }
            free(K); free(V); free(p); free(qd);
        }
    }
    return failed ? -1 : 0;
}

/*
 * ---- int8 KV cache ---------------------------------------------------------
 *
 * "Building a paged inference engine from scratch, and measuring it honestly",
 * section 02 ("INT8 KV cache design"): symmetric int8, one scale per block
 * per KV head, no zero point; on a write the block's existing entries are
 * dequantised with the stored scale, the new entries are added, a new max-abs
 * scale is computed over all of them and everything is requantised.  The page
 * calls this path unverified; this is the plain reading, applied once per
 * call to each block the call writes:
 *
 *   existing rows = rows 0 .. min_off-1 of the block (min_off = the lowest
 *                   offset written into it by this call; rows are appended in
 *                   order, so the rows below are the block's earlier tokens)
 *   new rows      = the rows this call writes (a later token with the same slot
 *                   replaces an earlier one)
 *   scale         = max |x| / 127 over existing (dequantised) and new values,
 *                   per KV head; 0 when that max is 0
 *   code          = clamp(round_half_even(x / scale), -127, 127), 0 if scale 0
 *
 * Every decision that yields an integer is taken in binary32 (the kernel's
 * precision): x as float, dequantised values q * scale as a float product,
 * the max in float, scale = max / 127 and x / scale as IEEE float divisions,
 * rintf for the rounding.  Rows past the highest written offset are left
 * untouched.
 */
static float f32_of(uint16_t x, int dtype) { return (float)decode(x, dtype); }

static int8_t quantize_f32(float x, float scale)
{
    if (scale == 0.0f)
        return 0;
    float r = rintf(x / scale);
    if (r > 127.0f)
        r = 127.0f;
    if (r < -127.0f)
        r = -127.0f;
    return (int8_t)r;
}

/* Quantised slot write.  k/v: [T, Hkv, D] 16-bit of `dtype`; pools int8
 * [nb, bs, Hkv, D]; scales float [nb, Hkv].  Returns 0, or -1 on a slot outside
 * the pool (nothing written). */
int oracle_write_kv_int8(const uint16_t *k, const uint16_t *v, int dtype, int64_t num_tokens,
                         int num_kv_heads, int head_dim, const int64_t *slots,
                         int8_t *kq, int8_t *vq, float *kscale, float *vscale,
                         int64_t num_blocks, int block_size)
{
    const int64_t nslots = num_blocks * block_size;
    for (int64_t t = 0; t < num_tokens; ++t)
        if (slots[t] >= nslots)
            return -1;
    const int H = num_kv_heads, D = head_dim, bs = block_size;
    /* blocks touched, in first-touch order */
    int64_t *blocks = (int64_t *)malloc(sizeof(int64_t) * (size_t)(num_tokens > 0 ? num_tokens : 1));
    int64_t nblk = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        if (slots[t] < 0)
            continue;
        int64_t b = slots[t] / bs, seen = 0;
        for (int64_t i = 0; i < nblk; ++i)
            if (blocks[i] == b)
                seen = 1;
        if (!seen)
            blocks[nblk++] = b;
    }
    float *rows = (float *)malloc(sizeof(float) * (size_t)bs * D);
    int64_t *src = (int64_t *)malloc(sizeof(int64_t) * (size_t)bs);
    for (int which = 0; which < 2; ++which) {
        const uint16_t *x = which ? v : k;
        int8_t *pool = which ? vq : kq;
        float *sc = which ? vscale : kscale;
        for (int64_t bi = 0; bi < nblk; ++bi) {
            const int64_t b = blocks[bi];
            int min_off = bs, max_off = -1;
            for (int o = 0; o < bs; ++o)
                src[o] = -1;
            for (int64_t t = 0; t < num_tokens; ++t) {
                if (slots[t] < 0 || slots[t] / bs != b)
                    continue;
                int o = (int)(slots[t] % bs);
                src[o] = t; /* last writer of an offset wins */
                if (o < min_off)
                    min_off = o;
                if (o > max_off)
                    max_off = o;
            }
            for (int h = 0; h < H; ++h) {
                const float old = sc[b * H + h];
                float amax = 0.0f;
                for (int o = 0; o <= max_off; ++o) {
                    for (int d = 0; d < D; ++d) {
                        float val;
                        if (src[o] >= 0)
                            val = f32_of(x[(src[o] * H + h) * D + d], dtype);
                        else if (o < min_off)
                            val = (float)pool[((b * bs + o) * H + h) * D + d] * old;
                        else
                            val = 0.0f; /* a gap below max_off (not produced by appends) */
                        rows[o * D + d] = val;
                        float a = fabsf(val);
                        if (a > amax)
                            amax = a;
                    }
                }
                const float scale = amax / 127.0f;
                for (int o = 0; o <= max_off; ++o)
                    for (int d = 0; d < D; ++d)
                        pool[((b * bs + o) * H + h) * D + d] = quantize_f32(rows[o * D + d], scale);
                sc[b * H + h] = scale;
            }
        }
    }
    free(blocks);
    free(rows);
    free(src);
    return 0;
}

/* Paged attention over an int8 cache: K = code * k_scale[block][head] (exact in
 * binary64), then the definition of oracle_paged_attention (decode rows only,
 * optional window).  q is 16-bit of `dtype`. */
int oracle_paged_attention_int8(const uint16_t *q, int64_t q_row_stride, int dtype,
                                const int8_t *kq, const int8_t *vq, const float *kscale,
                                const float *vscale, int64_t num_blocks, int block_size,
                                int num_kv_heads, int head_dim, const int32_t *tables, int max_blocks,
                                const int32_t *kv_lens, int num_seqs, int num_q_heads, double scale,
                                int window, double *out)
{
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return -1;
    const int group = num_q_heads / num_kv_heads;
    const int D = head_dim, H = num_kv_heads;
    for (int s = 0; s < num_seqs; ++s) {
        int64_t L = kv_lens[s];
        if (L < 0 || L > (int64_t)max_blocks * block_size)
            return -1;
        for (int64_t t = 0; t < L; t += block_size) {
            int32_t phys = tables[(int64_t)s * max_blocks + t / block_size];
            if (phys < 0 || phys >= num_blocks)
                return -1;
        }
    }
    int failed = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int s = 0; s < num_seqs; ++s) {
        for (int g = 0; g < H; ++g) {
            const int64_t L = kv_lens[s];
            const int64_t first = (window > 0 && L - window > 0) ? L - window : 0;
            const int64_t n = L - first;
            double *K = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * D);
            double *V = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * D);
            double *p = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
            double *qd = (double *)malloc(sizeof(double) * (size_t)D);
            if (!K || !V || !p || !qd) {
#pragma omp atomic write
                failed = 1;
                free(K); free(V); free(p); free(qd);
                continue;
            }
            for (int64_t i = 0; i < n; ++i) {
                const int64_t t = first + i;
                const int64_t phys = tables[(int64_t)s * max_blocks + t / block_size];
                const int64_t off = t % block_size;
                const int64_t base = ((phys * block_size + off) * H + g) * D;
                const double sk = kscale[phys * H + g], sv = vscale[phys * H + g];
                for (int d = 0; d < D; ++d) {
                    K[i * D + d] = (double)kq[base + d] * sk;
                    V[i * D + d] = (double)vq[base + d] * sv;
                }
            }
            for (int h = g * group; h < (g + 1) * group; ++h) {
                double *o = out + ((int64_t)s * num_q_heads + h) * D;
                for (int d = 0; d < D; ++d)
                    o[d] = 0.0;
                if (n <= 0)
                    continue;
                for (int d = 0; d < D; ++d)
                    qd[d] = decode(q[(int64_t)s * q_row_stride + (int64_t)h * D + d], dtype);
                double mx = -INFINITY;
                for (int64_t i = 0; i < n; ++i) {
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += qd[d] * K[i * D + d];
                    p[i] = scale * dot;
                    if (p[i] > mx)
                        mx = p[i];
                }
                double Z = 0.0;
                for (int64_t i = 0; i < n; ++i) {
                    p[i] = exp(p[i] - mx);
                    Z += p[i];
                }
                for (int64_t i = 0; i < n; ++i)
                    for (int d = 0; d < D; ++d)
                        o[d] += p[i] * V[i * D + d];
                for (int d = 0; d < D; ++d)
                    o[d] /= Z;
            }
            free(K); free(V); free(p); free(qd);
        }
    }
    return failed ? -1 : 0;
}
