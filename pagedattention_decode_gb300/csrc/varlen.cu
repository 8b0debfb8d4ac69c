// varlen.cu -- a8: packed varlen prefill + decode over the paged pool.
//
// "Building a paged inference engine from scratch, and measuring it honestly",
// section 02: one packed tensor holds the step's prefill and decode rows, and
// the attention kernel walks each sequence's block table; section 03 ("Causal
// mask during decode"): query row i of a sequence with q_len new rows and
// kv_len keys sees keys t <= kv_len - q_len + i.
//
// Rows of sequences with q_len == 1 are decode rows and run through the
// split-K decode kernel (decode.cu).  Chunks with q_len > 1 run here: one CTA
// per (128 / G query rows, sequence, KV head), so that its M = 128 rows are the
// G query heads of one KV head times 128 / G positions and every K/V tile it
// stages is used by all of them.  A producer warp streams 16-token K and V
// tiles of that KV head through a TMA + mbarrier ring; eight consumer warps
// each own 16 M rows and run the FlashAttention-2 loop on mma.sync m16n8k16
// (S = Q K^T, online softmax in fp32, O += P V with P as a 16-bit hi + lo
// pair).  Warps whose rows cannot see a tile under the causal rule skip it.
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
pkv_status check_attention_common(const void *q, int64_t q_stride, const pkv_cache *cache, const int32_t *tables,
                                  int32_t max_blocks, const int32_t *seq_lens, int32_t num_seqs,
                                  int32_t num_q_heads, void *out, int32_t out_dtype, const char *what);

constexpr int kPfTile = 2048;
constexpr int kPfWarps = 8;       // consumer warps
constexpr int kPfRows = 128;      // M rows per CTA (query rows x query heads of the group)
constexpr int kPfStages = 8;

struct PrefillParams {
    const void *q;
    int64_t q_stride;
    const int32_t *tables;
    int32_t max_blocks;
    const int32_t *seq_lens;
    const int32_t *cu_q;
    int32_t num_blocks, block_size, hkv, group, causal;
    float scale_log2;
    void *out;
    int32_t out_f32;
    int32_t *err;
    int32_t q_tiles;   // gridDim.x
};

template <int D, typename T>
__global__ void __launch_bounds__(32 * (1 + kPfWarps), 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const PrefillParams p) {
    constexpr int HALVES = D / 64;
    constexpr int STAGE = 2 * HALVES * kPfTile;
    extern __shared__ uint8_t smem_raw[];
    __shared__ volatile int s_abort;
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(base + kPfStages * STAGE);
    uint64_t *empty = full + kPfStages;

    const int s = blockIdx.y;
    const int kvh = blockIdx.z;
    const int tile = p.q_tiles - 1 - blockIdx.x;  // longest causal tiles first
    const int q_begin = p.cu_q[s];
    const int q_len = p.cu_q[s + 1] - q_begin;
    const int kv_len = p.seq_lens[s];
    const int G = p.group;
    const int qrows = kPfRows / G;
    const int q0 = tile * qrows;
    if (q_len <= 1 || q0 >= q_len) return;
    if (q_len > kv_len || (int64_t)kv_len > (int64_t)p.max_blocks * p.block_size) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && kvh == 0) set_err(p.err, PKV_DEVERR_LENGTH);
        return;
    }
    const int last_row = min(q_len, q0 + qrows) - 1;
    const int kv_hi = p.causal ? kv_len - q_len + last_row + 1 : kv_len;  // keys this CTA may need
    const int nsb = (kv_hi + 15) / 16;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        s_abort = 0;
        for (int i = 0; i < kPfStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kPfWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ===== producer =====
        if (lane == 0) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
        }
        const uint64_t pol = policy_evict_last();  // re-read by the other q tiles of this sequence
        const int32_t *trow = p.tables + (int64_t)s * p.max_blocks;
        int it = 0;
        bool aborted = false;
        for (int j0 = 0; j0 < nsb && !aborted; j0 += 32) {
            const int jn = min(32, nsb - j0);
            int row = 0;
            if (lane < jn) {
                const int tok = (j0 + lane) * 16;
                const int lb = tok / p.block_size;
                int phys = trow[lb];
                if (phys < 0 || phys >= p.num_blocks) {
                    set_err(p.err, PKV_DEVERR_BLOCK);
                    phys = 0;
                }
                row = phys * p.block_size + (tok - lb * p.block_size);
            }
            for (int j = 0; j < jn; ++j) {
                const int r = __shfl_sync(0xffffffffu, row, j);
                const int stage = it % kPfStages;
                int okw = 1;
                if (lane == 0) okw = mbar_wait(&empty[stage], ((it / kPfStages) & 1) ^ 1, &s_abort);
                okw = __shfl_sync(0xffffffffu, okw, 0);
                if (!okw) {
                    aborted = true;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(&full[stage], STAGE);
                __syncwarp();
                if (lane < 2 * HALVES) {
                    const int which = lane >= HALVES;
                    const int half = which ? lane - HALVES : lane;
                    tma_load_3d(base + stage * STAGE + lane * kPfTile, which ? &tmv : &tmk, &full[stage], 0,
                                kvh * HALVES + half, r, pol);
                }
                ++it;
            }
        }
        if (aborted && lane == 0) {
            s_abort = 1;
            set_err(p.err, PKV_DEVERR_TIMEOUT);
        }
        if (lane == 0) {
            const int first = it > kPfStages ? it - kPfStages : 0;
            for (int k = first; k < it; ++k) {
                volatile int never = 0;
                if (!mbar_wait(&full[k % kPfStages], (k / kPfStages) & 1, &never)) set_err(p.err, PKV_DEVERR_TIMEOUT);
            }
        }
        return;
    }

    // ===== consumers: 16 M rows each = 16 query rows of one query head =====
    const int w = warp - 1;
    const int wph = kPfWarps / G;           // warps per query head
    const int gi = w / wph;                 // query head within the group
    const int r0 = q0 + (w % wph) * 16;     // first query row (within the sequence) of this warp
    const int g = lane >> 2, t4 = lane & 3;
    const int qa = r0 + g, qb = r0 + g + 8;  // this thread's two rows
    const int head = kvh * G + gi;
    const float sl = p.scale_log2;
    // last key each row may see (rows past q_len see everything: never written)
    const int lim_a = (p.causal && qa < q_len) ? kv_len - q_len + qa : kv_len - 1;
    const int lim_b = (p.causal && qb < q_len) ? kv_len - q_len + qb : kv_len - 1;
    const bool warp_live = r0 < q_len;
    const int warp_lim = max(lim_a, lim_b);  // per-lane; the warp max is taken below
    int wl = warp_lim;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) wl = max(wl, __shfl_xor_sync(0xffffffffu, wl, off));

    uint32_t qf[D / 16][4];
    {
        const T *qpa = static_cast<const T *>(p.q) + (int64_t)(q_begin + qa) * p.q_stride + (int64_t)head * D;
        const T *qpb = static_cast<const T *>(p.q) + (int64_t)(q_begin + qb) * p.q_stride + (int64_t)head * D;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int d = kk * 16 + 2 * t4;
            qf[kk][0] = qa < q_len ? *reinterpret_cast<const uint32_t *>(qpa + d) : 0u;
            qf[kk][1] = qb < q_len ? *reinterpret_cast<const uint32_t *>(qpb + d) : 0u;
            qf[kk][2] = qa < q_len ? *reinterpret_cast<const uint32_t *>(qpa + d + 8) : 0u;
            qf[kk][3] = qb < q_len ? *reinterpret_cast<const uint32_t *>(qpb + d + 8) : 0u;
        }
    }
    float o[D / 8][4];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;

    for (int j = 0; j < nsb; ++j) {
        const int stage = j % kPfStages;
        if (!mbar_wait(&full[stage], (j / kPfStages) & 1, &s_abort)) {
            if (lane == 0) {
                s_abort = 1;
                set_err(p.err, PKV_DEVERR_TIMEOUT);
            }
            return;
        }
        const int t0 = j * 16;
        if (warp_live && t0 <= wl) {
            const uint8_t *kb = base + stage * STAGE;
            const uint8_t *vb = kb + HALVES * kPfTile;
            // S[16 rows x 16 tokens] = Q K^T, as two n tiles of 8 tokens
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            {
                const int tok = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int cg = 2 * kk + ((lane >> 3) & 1);
                    uint32_t b[4];
                    ldmatrix_x4(b, smem_u32(kb + (cg >> 3) * kPfTile + tok * 128 + (((cg & 7) ^ (tok & 7)) << 4)));
                    mma_16816<T>(sc[0], qf[kk], b[0], b[1]);
                    mma_16816<T>(sc[1], qf[kk], b[2], b[3]);
                }
            }
            float xs[2][4];
            float bma = -INFINITY, bmb = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int tk = t0 + nt * 8 + 2 * t4;
                xs[nt][0] = (tk <= lim_a) ? sc[nt][0] * sl : -INFINITY;
                xs[nt][1] = (tk + 1 <= lim_a) ? sc[nt][1] * sl : -INFINITY;
                xs[nt][2] = (tk <= lim_b) ? sc[nt][2] * sl : -INFINITY;
                xs[nt][3] = (tk + 1 <= lim_b) ? sc[nt][3] * sl : -INFINITY;
                bma = fmaxf(bma, fmaxf(xs[nt][0], xs[nt][1]));
                bmb = fmaxf(bmb, fmaxf(xs[nt][2], xs[nt][3]));
            }
#pragma unroll
            for (int off = 1; off < 4; off <<= 1) {
                bma = fmaxf(bma, __shfl_xor_sync(0xffffffffu, bma, off));
                bmb = fmaxf(bmb, __shfl_xor_sync(0xffffffffu, bmb, off));
            }
            const float na = fmaxf(ma, bma), nb = fmaxf(mb, bmb);
            const float aa = fast_exp2(ma - na), ab = fast_exp2(mb - nb);
            ma = na;
            mb = nb;
            float ps[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                ps[nt][0] = fast_exp2(xs[nt][0] - na);
                ps[nt][1] = fast_exp2(xs[nt][1] - na);
                ps[nt][2] = fast_exp2(xs[nt][2] - nb);
                ps[nt][3] = fast_exp2(xs[nt][3] - nb);
            }
            la = la * aa + ps[0][0] + ps[0][1] + ps[1][0] + ps[1][1];
            lb = lb * ab + ps[0][2] + ps[0][3] + ps[1][2] + ps[1][3];
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt) {
                o[nt][0] *= aa;
                o[nt][1] *= aa;
                o[nt][2] *= ab;
                o[nt][3] *= ab;
            }
            uint32_t ah[4], al[4];
            ah[0] = pack2<T>(ps[0][0], ps[0][1]);
            ah[1] = pack2<T>(ps[0][2], ps[0][3]);
            ah[2] = pack2<T>(ps[1][0], ps[1][1]);
            ah[3] = pack2<T>(ps[1][2], ps[1][3]);
            {
                float2 r;
                r = unpack2<T>(ah[0]);
                al[0] = pack2<T>(ps[0][0] - r.x, ps[0][1] - r.y);
                r = unpack2<T>(ah[1]);
                al[1] = pack2<T>(ps[0][2] - r.x, ps[0][3] - r.y);
                r = unpack2<T>(ah[2]);
                al[2] = pack2<T>(ps[1][0] - r.x, ps[1][1] - r.y);
                r = unpack2<T>(ah[3]);
                al[3] = pack2<T>(ps[1][2] - r.x, ps[1][3] - r.y);
            }
            // V rows past kv_len hold whatever the pool holds there: zero them
            uint32_t m0 = 0xffffffffu, m1 = 0xffffffffu;
            const int nv = kv_len - t0;
            if (nv < 16) {
                m0 = (2 * t4 < nv ? 0x0000ffffu : 0u) | (2 * t4 + 1 < nv ? 0xffff0000u : 0u);
                m1 = (2 * t4 + 8 < nv ? 0x0000ffffu : 0u) | (2 * t4 + 9 < nv ? 0xffff0000u : 0u);
            }
            {
                const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                for (int np = 0; np < D / 16; ++np) {
                    const int cg = 2 * np + (lane >> 4);
                    uint32_t b[4];
                    ldmatrix_x4_trans(b, smem_u32(vb + (cg >> 3) * kPfTile + tok * 128 + (((cg & 7) ^ (tok & 7)) << 4)));
                    b[0] &= m0;
                    b[1] &= m1;
                    b[2] &= m0;
                    b[3] &= m1;
                    mma_16816<T>(o[2 * np], ah, b[0], b[1]);
                    mma_16816<T>(o[2 * np], al, b[0], b[1]);
                    mma_16816<T>(o[2 * np + 1], ah, b[2], b[3]);
                    mma_16816<T>(o[2 * np + 1], al, b[2], b[3]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
    }
    if (!warp_live) return;
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        la += __shfl_xor_sync(0xffffffffu, la, off);
        lb += __shfl_xor_sync(0xffffffffu, lb, off);
    }
    const float ia = 1.f / la, ib = 1.f / lb;
    const int64_t hq = (int64_t)p.hkv * G;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
        const int d = nt * 8 + 2 * t4;
        if (qa < q_len) {
            const int64_t off = ((int64_t)(q_begin + qa) * hq + head) * D + d;
            if (p.out_f32) {
                *reinterpret_cast<float2 *>(static_cast<float *>(p.out) + off) = make_float2(o[nt][0] * ia, o[nt][1] * ia);
            } else {
                *reinterpret_cast<uint32_t *>(static_cast<T *>(p.out) + off) = pack2<T>(o[nt][0] * ia, o[nt][1] * ia);
            }
        }
        if (qb < q_len) {
            const int64_t off = ((int64_t)(q_begin + qb) * hq + head) * D + d;
            if (p.out_f32) {
                *reinterpret_cast<float2 *>(static_cast<float *>(p.out) + off) = make_float2(o[nt][2] * ib, o[nt][3] * ib);
            } else {
                *reinterpret_cast<uint32_t *>(static_cast<T *>(p.out) + off) = pack2<T>(o[nt][2] * ib, o[nt][3] * ib);
            }
        }
    }
}

template <int D, typename T>
static pkv_status launch_prefill_t(const CUtensorMap &mk, const CUtensorMap &mv, const PrefillParams &p,
                                   int num_seqs, cudaStream_t stream) {
    constexpr int STAGE = 2 * (D / 64) * kPfTile;
    const int smem = kPfStages * STAGE + 1024 + 2 * kPfStages * 8;
    auto kern = prefill_kernel<D, T>;
    PKV_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    dim3 grid(p.q_tiles, num_seqs, p.hkv);
    kern<<<grid, 32 * (1 + kPfWarps), smem, stream>>>(mk, mv, p);
    PKV_CUDA_TRY(cudaGetLastError());
    return PKV_OK;
}

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

pkv_status pkv_attn_varlen(const void *q, int64_t q_token_stride, const pkv_cache *cache, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                           int32_t num_seqs, int32_t total_q, int32_t max_q_len, int32_t num_q_heads, float scale,
                           int32_t causal, void *out, int32_t out_dtype, void *workspace, size_t workspace_bytes,
                           int32_t *err_word, pkv_stream stream) {
    pkv_status st = check_attention_common(q, q_token_stride, cache, block_tables, max_blocks_per_seq, seq_lens,
                                           num_seqs, num_q_heads, out, out_dtype, "pkv_attn_varlen");
    if (st != PKV_OK) return st;
    PKV_CHECK_ARG(total_q >= 0 && max_q_len >= 0, PKV_ERR_INVALID_ARG, "negative total_q or max_q_len");
    if (num_seqs == 0 || total_q == 0) return ok();
    PKV_CHECK_ARG(cu_seqlens_q, PKV_ERR_INVALID_ARG, "cu_seqlens_q is NULL");
    PKV_CHECK_ARG(num_seqs <= 65535, PKV_ERR_UNSUPPORTED, "at most 65535 sequences per call");
    // decode rows (q_len == 1) through the split-K decode kernels
    st = run_decode(q, q_token_stride, cache, block_tables, max_blocks_per_seq, seq_lens, cu_seqlens_q, num_seqs,
                    num_q_heads, scale, out, out_dtype, workspace, workspace_bytes, err_word, stream);
    if (st != PKV_OK) return st;
    if (max_q_len <= 1) return ok();
    CUtensorMap mk, mv;
    st = encode_pool_map(&mk, cache->k, cache);
    if (st != PKV_OK) return st;
    st = encode_pool_map(&mv, cache->v, cache);
    if (st != PKV_OK) return st;
    PrefillParams p{};
    p.q = q;
    p.q_stride = q_token_stride;
    p.tables = block_tables;
    p.max_blocks = max_blocks_per_seq;
    p.seq_lens = seq_lens;
    p.cu_q = cu_seqlens_q;
    p.num_blocks = cache->num_blocks;
    p.block_size = cache->block_size;
    p.hkv = cache->num_kv_heads;
    p.group = num_q_heads / cache->num_kv_heads;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.out = out;
    p.out_f32 = out_dtype == PKV_F32;
    p.err = err_word;
    const int qrows = kPfRows / p.group;
    p.q_tiles = (max_q_len + qrows - 1) / qrows;
    const bool bf = cache->dtype == PKV_BF16;
    if (cache->head_dim == 64)
        st = bf ? launch_prefill_t<64, __nv_bfloat16>(mk, mv, p, num_seqs, stream)
                : launch_prefill_t<64, __half>(mk, mv, p, num_seqs, stream);
    else
        st = bf ? launch_prefill_t<128, __nv_bfloat16>(mk, mv, p, num_seqs, stream)
                : launch_prefill_t<128, __half>(mk, mv, p, num_seqs, stream);
    return st == PKV_OK ? ok() : st;
}

}  // extern "C"
