// decode.cu -- a3..a7: fused gather-and-attend decode over the paged pool.
//
// What it computes is the plain definition in "How to Implement Paged
// Attention in PyTorch and vLLM", section "Compute reference attention without
// hiding the layout": for sequence s and query head h, with KV head
// h / (Hq / Hkv), softmax over t < L_s of scale * <q, K_t> applied to V_t.
// "Map the PyTorch design to vLLM PagedAttention" names fused kernels that read
// the block table during attention instead of gathering; this is one, shaped
// for GB300:
//
//  * Work split (split-K, "flash-decoding"): the 16-token sub-blocks of all
//    sequences are concatenated and cut into equal contiguous ranges, one per
//    CTA, all CTAs resident at once (persistent: one per SM for head_dim 128,
//    two for int8 caches, three for head_dim 64).  A sequence wholly inside
//    one range is finished in place; a sequence cut by a range boundary
//    leaves (running max, running sum, unnormalised output) records in the
//    workspace that decode_merge_kernel combines.  Balance is exact whatever
//    the length mix.  A call of at most 32 sequences and 64 sub-blocks takes
//    a CTA per sequence instead (no cut, nothing to merge, and when the
//    tables' capacity already guarantees the bounds no merge launch): the
//    tiny MHA call went from 22.0 to 16.3-16.6 us per write + decode step
//    (A/B, L2 flushed).
//  * Data movement: one producer warp walks the block tables and issues two
//    TMA tensor loads per 16-token sub-block, K and V, into a ring of
//    shared-memory stages guarded by mbarriers.  Each load is one box of 16
//    token rows x every 128-byte chunk of the CTA's KV heads (a view of the
//    pool with the chunk dimension outside the row dimension), so it lands as
//    one 2 KB, 128-byte-swizzled tile per (KV head, half of head_dim).  A TMA
//    box costs ~50 cycles on the SM besides its bytes: 2 KB boxes, one per tile,
//    held an SM near 25 B/clk (GQA decode call 6,886 GB/s, the mixed step's
//    L2-served decode rows 0.567 ms); one box per K or V of a stage gives
//    7,015 GB/s and 0.371 ms.  Each K/V byte is read from HBM once (GQA: the
//    query heads of a group share it).
//  * Math: one consumer warp per KV head.  Scores for 16 tokens x the group's
//    query heads come from mma.sync m16n8k16 (tokens as M, heads as N, fp32
//    accumulate); the online softmax (running max in base 2, rescaled running
//    sum and accumulator) follows the online-normaliser recurrence of Milakov &
//    Gimelshein (2018) as used by FlashAttention-2; P is transposed in
//    registers (movmatrix) and multiplied with V^T on the tensor cores as a
//    16-bit hi + lo pair, so P keeps ~16 significant bits (with 2 or 4 query
//    heads per KV head both parts share one MMA: the N = 8 columns hold each
//    head twice).  For head_dim 128 and int8 the running max is lazy: it moves
//    only when a scaled score passes it by more than 8 in base 2 (p <= 256).
#include <cuda.h>

#include "launch.h"
#include "ptx.cuh"

#include <type_traits>

namespace pkv {

constexpr int kSub = 16;      // tokens per stage (the mma M dimension)
constexpr int kTile = 2048;   // bytes of one swizzled 16-token x 64-element tile
// Consumer warps (one per KV head) per CTA: 8 at head_dim 128 keeps the
// accumulators in registers (3 warps per SM sub-partition), 16 at head_dim 64.
template <int D>
constexpr int max_heads_per_cta() { return D == 64 ? 4 : 8; }
// 16-bit caches with head_dim 64: three CTAs of up to four KV heads (five
// warps) per SM.  Small D 64 calls are latency-bound, and more, smaller CTAs
// start streaming sooner.  Measured on the GPT-2-shaped step (12 layers, 12
// heads, B 32, contexts 64-1024; ms per step, without / with the new rows
// written by the decode kernel): 1 x 12 heads 0.2214 / 0.2136, 2 x 6
// 0.2196 / 0.2050, 3 x 4 0.2158 / 0.2050, 4 x 3 0.2173 / 0.2071, 6 x 2
// 0.2235 / 0.2127.
constexpr int kD64CtasPerSm = 3;

// int8 cache: two CTAs of up to eight KV heads (nine warps) per SM.  With
// eight KV heads a stage then holds whole 16-token rows of the pool, and
// sixteen consumer warps hide the code conversion.  Measured against the other
// shapes the registers allow (same code; GB/s of codes at GQA 32/8, B 256):
// 2 x 8 heads 6,075 (96 registers, a few bytes spilled), 2 x 4 6,016 and
// 3 x 4 5,990 (128+ registers, no spills), 4 x 4 5,877, 1 x 8 4,820.
constexpr int kI8CtasPerSm = 2;
constexpr int kI8HeadsPerCta = 8;

template <int D, bool I8>
constexpr int cta_threads() { return 32 * (1 + (I8 ? kI8HeadsPerCta : max_heads_per_cta<D>())); }
constexpr int kMinSubBlocksPerCta = 4;
// Calls of at most kWholeSeqMaxSeqs sequences and kWholeSeqMaxSubBlocks
// sub-blocks, launched with a CTA per sequence: CTA c takes sequence c whole,
// so no sequence is cut and the merge has nothing to combine.
constexpr int kWholeSeqMaxSeqs = 32;
constexpr int kWholeSeqMaxSubBlocks = 64;
// The one test of that split, shared by the host (with its bound on the
// sub-blocks), the decode kernel and the merge (with the actual count).
__host__ __device__ __forceinline__ bool whole_seq_split(int64_t sub_blocks, int64_t num_seqs, int64_t grid_x) {
    return sub_blocks <= kWholeSeqMaxSubBlocks && num_seqs <= kWholeSeqMaxSeqs && num_seqs <= grid_x;
}

struct DecodeParams {
    const void *q;
    int64_t q_stride;              // elements between consecutive query rows
    const int32_t *tables;
    int32_t max_blocks;
    const int32_t *seq_lens;
    const int32_t *cu_q;           // varlen mode: only q_len == 1 sequences, row cu_q[s]
    int32_t num_seqs;
    int32_t num_blocks, block_size, hkv, heads_per_cta, group;
    float scale_log2;              // scale * log2(e)
    void *out;
    int32_t out_f32;
    float *ws_o;                   // [num_hg][cmax][2][heads_per_cta * group][D]
    float *ws_ml;                  // [num_hg][cmax][2][heads_per_cta * group][2]
    int32_t *ws_meta;              // [0] total sub-blocks, [1] CTAs used, [2 + s] first sub-block of s
    int32_t cmax;                  // gridDim.x at most (the records' CTA stride)
    int32_t grid_x;                // the decode launch's gridDim.x (the merge recomputes the split with it)
    int32_t *err;
    int32_t stages;
    int32_t window;                // > 0: attend only the last `window` keys
    const float *k_scale;          // int8 cache: [num_blocks, hkv] scales (NULL for 16-bit caches)
    const float *v_scale;
    // append mode (16-bit caches): row s of k_new / v_new is the key / value of
    // position seq_lens[s] - 1 and is written into the pool before the
    // sub-block holding it is loaded; NULL otherwise
    const void *k_new, *v_new;
    int64_t new_stride;            // elements between consecutive new rows
    void *k_pool, *v_pool;         // the pools ([num_blocks * block_size, hkv, D])
};

// First key a decode row of a sequence with L keys attends (sliding window).
__device__ __forceinline__ int decode_first_key(const DecodeParams &p, int L) {
    return (p.window > 0 && L > p.window) ? L - p.window : 0;
}

// Sub-blocks of sequence s handled by the decode kernel (0 when skipped):
// those from the one holding its first attended key to the one holding L-1.
__device__ __forceinline__ int decode_sub_blocks(const DecodeParams &p, int s) {
    if (p.cu_q && p.cu_q[s + 1] - p.cu_q[s] != 1) return 0;
    const int L = p.seq_lens[s];
    if (L <= 0) return 0;
    if ((int64_t)L > (int64_t)p.max_blocks * p.block_size) return 0;
    return (L + kSub - 1) / kSub - decode_first_key(p, L) / kSub;
}

__device__ __forceinline__ bool decode_bad_length(const DecodeParams &p, int s) {
    if (p.cu_q && p.cu_q[s + 1] - p.cu_q[s] != 1) return false;
    const int L = p.seq_lens[s];
    return L < 0 || (int64_t)L > (int64_t)p.max_blocks * p.block_size;
}

// Inclusive block-wide scan of one int per thread; *total gets the block sum.
__device__ __forceinline__ int block_scan(int v, int *warp_sums, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < nw) warp_sums[lane] = w;  // inclusive prefix of warp totals
    }
    __syncthreads();
    const int before = warp > 0 ? warp_sums[warp - 1] : 0;
    *total = warp_sums[nw - 1];
    __syncthreads();
    return x + before;
}

// Two int8 codes -> a packed 16-bit pair.  `x` holds four codes XOR 0x80
// (offset binary); `sel` is a byte_perm selector 0x4?4? naming the bytes for
// the low and high halves.  fp16: bytes under the exponent of 1024 give
// 1024 + u exactly, minus 1152 = the signed code.  bf16: through binary32
// (2^23 + u, minus 2^23 + 128), then an exact narrowing.
template <typename T>
struct IsHalf {
    static constexpr bool value = false;
};
template <>
struct IsHalf<__half> {
    static constexpr bool value = true;
};

template <typename T>
__device__ __forceinline__ uint32_t i8_pair(uint32_t x, uint32_t sel);

template <>
__device__ __forceinline__ uint32_t i8_pair<__half>(uint32_t x, uint32_t sel) {
    uint32_t h = __byte_perm(x, 0x64646464u, sel);
    __half2 v = __hsub2(*reinterpret_cast<__half2 *>(&h), __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
    return *reinterpret_cast<uint32_t *>(&v);
}

// fp16 codes + 1152 (1024 + 128 + code, exact) without the subtraction, for
// the K codes: the decode kernel takes the bias out of the scores (1152 * sum
// of q), which costs them ~1e-4 of relative precision.  V codes enter P V
// without the bias (i8_pair): there it would sit in the fp32 accumulator of O.
__device__ __forceinline__ uint32_t i8_pair_biased(uint32_t x, uint32_t sel) {
    return __byte_perm(x, 0x64646464u, sel);
}

template <>
__device__ __forceinline__ uint32_t i8_pair<__nv_bfloat16>(uint32_t x, uint32_t sel) {
    const float lo = __int_as_float((int)__byte_perm(x, 0x4B000000u, 0x7540u | (sel & 0xFu))) - 8388736.f;
    const float hi = __int_as_float((int)__byte_perm(x, 0x4B000000u, 0x7540u | ((sel >> 8) & 0xFu))) - 8388736.f;
    return pack2<__nv_bfloat16>(lo, hi);
}

__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// The CTA that owns concatenated sub-block x when `ctas` ranges split `total`.
__device__ __forceinline__ int range_owner(int64_t x, int64_t total, int64_t ctas) {
    return (int)(((x + 1) * ctas - 1) / total);
}

// Lazy running max (int8 and head_dim 128): how far (log2 units) a score may
// pass the running max before the max is moved
constexpr float kLazyMax = 8.f;

// AP: append mode (pkv_attn_decode_append), compiled separately so that the
// plain decode carries none of its code
template <int D, typename T, bool I8, bool AP = false>
__global__ void __launch_bounds__(cta_threads<D, I8>(), I8 ? kI8CtasPerSm : (D == 64 ? kD64CtasPerSm : 1))
    decode_splitk_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                         const DecodeParams p) {
    // 2 KB shared tiles per KV head per sub-block: 16 tokens x 64 dims of a
    // 16-bit cache (two for head_dim 128), or 16 tokens x 128 int8 codes
    constexpr int HALVES = I8 ? 1 : D / 64;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_warp[32];
    __shared__ int s_first_seq, s_first_start;
    __shared__ long long s_whole[2];
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int HG = p.heads_per_cta;
    const int tiles = HG * HALVES;                 // 2 KB tiles per K (and per V) in a stage
    const int stage_bytes = 2 * tiles * kTile;
    const int NS = p.stages;
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(base + NS * stage_bytes);
    uint64_t *empty = full + NS;
    float *sscale = reinterpret_cast<float *>(empty + NS);  // int8: [NS][2][hkv] per-stage block scales
    const int hg = blockIdx.y;
    const bool meta_cta = blockIdx.x == 0 && blockIdx.y == 0;
    if (threadIdx.x == 0) {  // descriptors are kernel parameters: no wait needed
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }
    pdl_wait();  // the previous kernel on the stream (e.g. the slot write) is complete

    // ---- 1. total sub-blocks, this CTA's range ------------------------------
    if (tid == 0) {
        s_first_seq = -1;
        s_abort = 0;
    }
    int64_t total = 0;
    int my_n = 0, my_incl = 0;  // this thread's sequence when they all fit one pass
    for (int s0 = 0; s0 < p.num_seqs; s0 += blockDim.x) {
        const int s = s0 + tid;
        const int n = s < p.num_seqs ? decode_sub_blocks(p, s) : 0;
        if (meta_cta && s < p.num_seqs && decode_bad_length(p, s)) set_err(p.err, PKV_DEVERR_LENGTH);
        int chunk;
        const int incl = block_scan(n, s_warp, &chunk);
        if (s0 == 0) {
            my_n = n;
            my_incl = incl;
        }
        total += chunk;
    }
    const bool whole = whole_seq_split(total, p.num_seqs, gridDim.x);
    const int64_t want = (total + kMinSubBlocksPerCta - 1) / kMinSubBlocksPerCta;
    const int ctas = whole ? p.num_seqs : (int)(want < gridDim.x ? want : gridDim.x);
    if (blockIdx.x >= ctas && !meta_cta) return;
    int64_t lo = ctas ? (int64_t)blockIdx.x * total / ctas : 0;
    int64_t hi = ctas ? (int64_t)(blockIdx.x + 1) * total / ctas : 0;
    if (whole) {
        // sequence blockIdx.x, whose bounds thread blockIdx.x found in the one pass
        // (num_seqs <= 32 < blockDim.x); uniform over the CTA
        if (tid == (int)blockIdx.x) {
            s_whole[0] = my_incl - my_n;
            s_whole[1] = my_incl;
        }
        __syncthreads();
        lo = s_whole[0];
        hi = s_whole[1];
    }

    if (p.num_seqs <= (int)blockDim.x) {
        // one pass held every sequence: its prefix sums locate the range start
        // (ordered after s_first_seq = -1 by the scan's barriers; read after
        // the barrier below)
        const int64_t start = my_incl - my_n;
        if (my_n > 0 && start <= lo && lo < start + my_n) {
            s_first_seq = tid;
            s_first_start = (int)start;
        }
        if (meta_cta && tid < p.num_seqs) p.ws_meta[2 + tid] = (int)start;
    } else {
        int64_t carry = 0;
        for (int s0 = 0; s0 < p.num_seqs; s0 += blockDim.x) {
            const int s = s0 + tid;
            const int n = s < p.num_seqs ? decode_sub_blocks(p, s) : 0;
            int chunk;
            const int incl = block_scan(n, s_warp, &chunk);
            const int64_t start = carry + incl - n;
            if (n > 0 && start <= lo && lo < start + n) {
                s_first_seq = s;
                s_first_start = (int)start;
            }
            if (meta_cta && s < p.num_seqs) p.ws_meta[2 + s] = (int)start;
            carry += chunk;
        }
    }
    if (meta_cta && tid == 0) {
        p.ws_meta[0] = (int)total;
        p.ws_meta[1] = ctas;
        p.ws_meta[2 + p.num_seqs] = (int)total;
    }
    if (whole && lo >= hi && blockIdx.x < ctas) {
        // an empty decode row of a call whose merge is not launched: its zero
        // rows (this head group's query heads) come from here
        const int s = blockIdx.x;
        if (!p.cu_q || p.cu_q[s + 1] - p.cu_q[s] == 1) {
            const int64_t qrow = p.cu_q ? (int64_t)p.cu_q[s] : (int64_t)s;
            const int nq = HG * p.group;
            const int64_t ob = (qrow * (int64_t)(p.hkv * p.group) + (int64_t)hg * nq) * D;
            for (int i = tid; i < nq * D; i += blockDim.x) {
                if (p.out_f32)
                    static_cast<float *>(p.out)[ob + i] = 0.f;
                else
                    static_cast<T *>(p.out)[ob + i] = static_cast<T>(0.f);
            }
        }
    }
    if (blockIdx.x >= ctas || lo >= hi) return;

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], HG);
        }
        fence_barrier_init();
    }
    __syncthreads();

    // ---- 2. walk of the range: segments (s, first sub-block, end sub-block) --
    // Both roles walk the same list; `x` counts concatenated sub-blocks.
    if (warp == 0) {
        // ===== producer =====
        const uint64_t pol = policy_evict_first();
        int it = 0;  // loads issued; ring position (stage, phase) kept alongside without a division
        int pstage = 0;
        uint32_t pphase = 0;
        bool aborted = false;
        int s = s_first_seq;
        int sb = (int)(lo - s_first_start);
        int64_t x = lo;
        while (x < hi && !aborted) {
            const int n_s = decode_sub_blocks(p, s);
            if (n_s == 0) {
                ++s;
                continue;
            }
            const int b1 = (int)(sb + (hi - x) < n_s ? sb + (hi - x) : n_s);
            const int32_t *trow = p.tables + (int64_t)s * p.max_blocks;
            const int L = p.seq_lens[s];
            const int sb0 = decode_first_key(p, L) / kSub;  // window: first sub-block
            // append mode: the sub-block holding position L - 1 (the new key);
            // when this segment reaches it, the new row (this head group's
            // part) is loaded into registers now, so its latency passes while
            // the segment's earlier sub-blocks are issued
            const int sb_new = AP ? (L - 1) / kSub : -1;
            constexpr int U = D / 8;                 // 16-byte units per head row
            constexpr int kNewPerLane = 2 * 8 * 16 / 32;  // (K and V) x HG x U / 32, HG * D <= 1024
            uint4 new_row[kNewPerLane];
            const bool has_new = sb_new >= sb0 + sb && sb_new < sb0 + b1;
            if constexpr (AP) {
                if (has_new) {
#pragma unroll
                    for (int i = 0; i < kNewPerLane; ++i) {
                        const int t = lane + 32 * i;
                        if (t < 2 * HG * U) {
                            const int which = t >= HG * U;
                            const int tt = which ? t - HG * U : t;
                            const int head = hg * HG + tt / U;
                            new_row[i] = *(reinterpret_cast<const uint4 *>(
                                               static_cast<const T *>(which ? p.v_new : p.k_new) +
                                               (int64_t)s * p.new_stride + (int64_t)head * D) + tt % U);
                        }
                    }
                }
            }
            for (int j0 = sb; j0 < b1 && !aborted; j0 += 32) {
                const int jn = min(32, b1 - j0);
                int row = 0, pblk = 0;
                if (lane < jn) {
                    const int tok = (sb0 + j0 + lane) * kSub;
                    const int lb = tok / p.block_size;
                    int phys = trow[lb];
                    if (phys < 0 || phys >= p.num_blocks) {
                        set_err(p.err, PKV_DEVERR_BLOCK);
                        phys = 0;
                    }
                    pblk = phys;
                    row = phys * p.block_size + (tok - lb * p.block_size);
                }
                for (int j = 0; j < jn; ++j) {
                    const int r = __shfl_sync(0xffffffffu, row, j);
                    const int rb = __shfl_sync(0xffffffffu, pblk, j);
                    const int stage = pstage;
                    int okw = 1;
                    if (lane == 0) okw = mbar_wait(&empty[stage], pphase ^ 1u, &s_abort);
                    okw = __shfl_sync(0xffffffffu, okw, 0);
                    if (!okw) {
                        aborted = true;
                        break;
                    }
                    if constexpr (AP) {
                        if (sb0 + j0 + j == sb_new) {
                            // this CTA (and no other of its head group) reads the
                            // sub-block holding the new key: write its row for
                            // this group's KV heads first, then let the TMA see it
                            const int tok = L - 1, lb = tok / p.block_size;
                            const int phys = trow[lb];
                            if (phys >= 0 && phys < p.num_blocks) {
                                const int64_t slot = (int64_t)phys * p.block_size + (tok - lb * p.block_size);
#pragma unroll
                                for (int i = 0; i < kNewPerLane; ++i) {
                                    const int t = lane + 32 * i;
                                    if (t < 2 * HG * U) {
                                        const int which = t >= HG * U;
                                        const int tt = which ? t - HG * U : t;
                                        const int head = hg * HG + tt / U;
                                        *(reinterpret_cast<uint4 *>(static_cast<T *>(which ? p.v_pool : p.k_pool) +
                                                                    (slot * p.hkv + head) * D) + tt % U) = new_row[i];
                                    }
                                }
                                asm volatile("fence.proxy.async.global;" ::: "memory");
                            } else if (lane == 0) {
                                set_err(p.err, PKV_DEVERR_BLOCK);
                            }
                            __syncwarp();
                        }
                    }
                    const uint32_t scale_bytes = I8 ? (uint32_t)(8 * p.hkv) : 0u;
                    if (lane == 0) mbar_arrive_expect_tx(&full[stage], stage_bytes + scale_bytes);
                    __syncwarp();
                    if constexpr (I8) {
                        if (lane == 0) {
                            float *ds = sscale + stage * 2 * p.hkv;
                            bulk_copy_g2s(ds, p.k_scale + (int64_t)rb * p.hkv, 4 * p.hkv, &full[stage]);
                            bulk_copy_g2s(ds + p.hkv, p.v_scale + (int64_t)rb * p.hkv, 4 * p.hkv, &full[stage]);
                        }
                    }
                    // one copy for K and one for V: 16 token rows x this
                    // CTA's `tiles` chunks, landing as `tiles` 2 KB tiles
                    uint8_t *sbase = base + stage * stage_bytes;
                    if (lane < 2)
                        tma_load_3d(sbase + lane * tiles * kTile, lane ? &tmv : &tmk, &full[stage], 0, r,
                                    hg * tiles, pol);
                    ++it;
                    if (++pstage == NS) {
                        pstage = 0;
                        pphase ^= 1u;
                    }
                }
            }
            x += b1 - sb;
            ++s;
            sb = 0;
        }
        if (aborted && lane == 0) {
            s_abort = 1;
            set_err(p.err, PKV_DEVERR_TIMEOUT);
        }
        // every load of this CTA is issued: the merge kernel may be scheduled
        pdl_trigger();
        // drain: the last load issued into each stage must land before the CTA exits
        if (lane == 0) {
            const int first = it > NS ? it - NS : 0;
            for (int k = first; k < it; ++k) {
                volatile int never = 0;
                if (!mbar_wait(&full[k % NS], (k / NS) & 1, &never)) set_err(p.err, PKV_DEVERR_TIMEOUT);
            }
        }
        return;
    }
    if (warp > HG) return;

    // ===== consumer: KV head kvh =====
    const int w = warp - 1;
    const int kvh = hg * HG + w;
    const int G = p.group;
    const int g = lane >> 2, t4 = lane & 3;
    const int hA = 2 * t4, hB = 2 * t4 + 1;
    // head_dim 128 and int8: MMA columns G .. 2G - 1 repeat heads 0 .. G - 1
    // (G = 2 or 4) and carry the low 16-bit part of their P, so P V takes one
    // MMA per m tile instead of two; the two parts of O are added at the end
    // of the segment (lanes t4 and t4 + G / 2 hold a head's two parts).  The
    // running max of these kernels is lazy (below).  The head_dim 64 kernel,
    // latency-bound on small calls, keeps the plain form: with these paths
    // compiled in, its GPT-2-shaped step measured 1-2% slower.
    constexpr bool kLazy = I8 || D == 128;
    const bool packlo = kLazy && (G == 2 || G == 4);
    const int gcols = packlo ? 2 * G : G;  // MMA columns that hold a head
    const bool lo_lane = packlo && t4 >= (G >> 1);
    const float sl = p.scale_log2;
    const int qheads_cta = HG * G;
    int stage = 0;  // ring position of the next sub-block and the parity of its fill
    uint32_t phase = 0;
    bool first_seg = true;
    int s = s_first_seq;
    int sb = (int)(lo - s_first_start);
    int64_t x = lo;
    while (x < hi) {
        const int n_s = decode_sub_blocks(p, s);
        if (n_s == 0) {
            ++s;
            continue;
        }
        const int b1 = (int)(sb + (hi - x) < n_s ? sb + (hi - x) : n_s);
        const int L = p.seq_lens[s];
        const int first_key = decode_first_key(p, L);
        const int sb0 = first_key / kSub;
        const int64_t qrow = p.cu_q ? (int64_t)p.cu_q[s] : (int64_t)s;

        // query fragments: B operand (16 dims x 8 heads), head g of the group
        uint32_t qf[D / 16][2];
        {
            const int qcol = g < G ? g : (g < gcols ? g - G : 0);  // the head in column g
            const T *qp = static_cast<const T *>(p.q) + qrow * p.q_stride + (int64_t)(kvh * G + qcol) * D;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                if (g < gcols) {
                    // int8: dims permuted inside each 16-dim step to match the K codes' byte order
                    qf[kk][0] = *reinterpret_cast<const uint32_t *>(qp + kk * 16 + (I8 ? 4 * t4 : 2 * t4));
                    qf[kk][1] = *reinterpret_cast<const uint32_t *>(qp + kk * 16 + (I8 ? 4 * t4 + 2 : 8 + 2 * t4));
                } else {
                    qf[kk][0] = 0u;
                    qf[kk][1] = 0u;
                }
            }
        }
        float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
        // int8 K codes of an fp16 cache enter the score MMAs as code + 1152 (see i8_pair_biased)
        constexpr bool BIAS = I8 && IsHalf<T>::value;
        float qsA = 0.f, qsB = 0.f;
        if constexpr (BIAS) {
            // sum of q over head_dim for heads hA, hB: lane 4g + t4 holds a quarter of head g
            float qs = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const float2 a = unpack2<T>(qf[kk][0]), b = unpack2<T>(qf[kk][1]);
                qs += (a.x + a.y) + (b.x + b.y);
            }
            qs += __shfl_xor_sync(0xffffffffu, qs, 1);
            qs += __shfl_xor_sync(0xffffffffu, qs, 2);
            qsA = __shfl_sync(0xffffffffu, qs, hA * 4);
            qsB = __shfl_sync(0xffffffffu, qs, hB * 4);
        }
        float o[D / 16][4];
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

        bool aborted = false;
        for (int j = sb; j < b1; ++j) {
            if (!mbar_wait(&full[stage], phase, &s_abort)) {
                aborted = true;
                break;
            }
            const uint8_t *kb = base + stage * stage_bytes + (w * HALVES) * kTile;
            const uint8_t *vb = kb + tiles * kTile;
            const int tok0 = (sb0 + j) * kSub;
            const int nv = min(kSub, L - tok0);        // tokens below nv are in the sequence
            const int nlo = first_key - tok0;          // tokens below nlo are outside the window

            // S^T[16 tokens x 8 heads] = K q^T
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
            float ssl = sl, vsc = 1.f;
            if constexpr (I8) {
                const float *st_scale = sscale + stage * 2 * p.hkv;
                ssl = sl * st_scale[kvh];
                vsc = st_scale[p.hkv + kvh];
                // codes of 16 tokens x 32 dims per ldmatrix.x4; thread t of a row holds dims 4t..4t+3
                const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                for (int k2 = 0; k2 < D / 32; ++k2) {
                    const int chunk = 2 * k2 + (lane >> 4);
                    uint32_t r[4];
                    ldmatrix_x4(r, smem_u32(kb + tok * 128 + ((chunk ^ (tok & 7)) << 4)));
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const uint32_t lo = r[2 * u] ^ 0x80808080u, hi = r[2 * u + 1] ^ 0x80808080u;
                        uint32_t a[4];
                        if constexpr (BIAS) {
                            a[0] = i8_pair_biased(lo, 0x4140u);
                            a[1] = i8_pair_biased(hi, 0x4140u);
                            a[2] = i8_pair_biased(lo, 0x4342u);
                            a[3] = i8_pair_biased(hi, 0x4342u);
                        } else {
                            a[0] = i8_pair<T>(lo, 0x4140u);
                            a[1] = i8_pair<T>(hi, 0x4140u);
                            a[2] = i8_pair<T>(lo, 0x4342u);
                            a[3] = i8_pair<T>(hi, 0x4342u);
                        }
                        mma_16816<T>(sc, a, qf[2 * k2 + u][0], qf[2 * k2 + u][1]);
                    }
                }
            } else {
                const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int chunk = ((kk & 3) << 1) + (lane >> 4);
                    uint32_t a[4];
                    ldmatrix_x4(a, smem_u32(kb + (kk >> 2) * kTile + tok * 128 + ((chunk ^ (tok & 7)) << 4)));
                    mma_16816<T>(sc, a, qf[kk][0], qf[kk][1]);
                }
            }
            float x0, x1, x2, x3;
            if constexpr (BIAS) {
                const float kA = 1152.f * qsA * ssl, kB = 1152.f * qsB * ssl;
                x0 = fmaf(sc[0], ssl, -kA);
                x1 = fmaf(sc[1], ssl, -kB);
                x2 = fmaf(sc[2], ssl, -kA);
                x3 = fmaf(sc[3], ssl, -kB);
            } else {
                x0 = sc[0] * ssl;
                x1 = sc[1] * ssl;
                x2 = sc[2] * ssl;
                x3 = sc[3] * ssl;
            }
            if (nv < kSub) {
                if (g >= nv) x0 = x1 = -INFINITY;
                if (g + 8 >= nv) x2 = x3 = -INFINITY;
            }
            if (nlo > 0) {
                if (g < nlo) x0 = x1 = -INFINITY;
                if (g + 8 < nlo) x2 = x3 = -INFINITY;
            }
            if (hA >= gcols) x0 = x2 = 0.f;
            if (hB >= gcols) x1 = x3 = 0.f;
            // kLazy: the running max is lazy.  It moves only when a score of the
            // warp passes it by more than kLazyMax (so every p <= 2^kLazyMax); a
            // vote stands in for the reduction and the rescale on the other
            // tiles.  O, l (and the records) stay relative to the max used.
            bool moved = true;
            if constexpr (kLazy)
                moved = __any_sync(0xffffffffu, !(fmaxf(x0, x2) <= mA + kLazyMax) || !(fmaxf(x1, x3) <= mB + kLazyMax));
            float aA = 1.f, aB = 1.f;
            if (moved) {
                float bA = fmaxf(x0, x2), bB = fmaxf(x1, x3);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    bA = fmaxf(bA, __shfl_xor_sync(0xffffffffu, bA, off));
                    bB = fmaxf(bB, __shfl_xor_sync(0xffffffffu, bB, off));
                }
                if (packlo) {  // both columns of a head keep one running max
                    bA = fmaxf(bA, __shfl_xor_sync(0xffffffffu, bA, G >> 1));
                    bB = fmaxf(bB, __shfl_xor_sync(0xffffffffu, bB, G >> 1));
                }
                const float nA = fmaxf(mA, bA), nB = fmaxf(mB, bB);
                aA = fast_exp2(mA - nA);
                aB = fast_exp2(mB - nB);
                mA = nA;
                mB = nB;
            }
            const float p0 = fast_exp2(x0 - mA), p1 = fast_exp2(x1 - mB);
            const float p2 = fast_exp2(x2 - mA), p3 = fast_exp2(x3 - mB);
            lA = lA * aA + p0 + p2;
            lB = lB * aB + p1 + p3;
            if (moved) {
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    o[mt][0] *= aA;
                    o[mt][1] *= aB;
                    o[mt][2] *= aA;
                    o[mt][3] *= aB;
                }
            }
            // P as the B operand (16 tokens x 8 heads), hi and lo 16-bit parts
            // (int8: P is scaled by the block's V scale, so the codes multiply directly)
            const float q0 = p0 * vsc, q1 = p1 * vsc, q2 = p2 * vsc, q3 = p3 * vsc;
            const uint32_t h01 = pack2<T>(q0, q1), h23 = pack2<T>(q2, q3);
            const float2 r01 = unpack2<T>(h01), r23 = unpack2<T>(h23);
            const uint32_t l01 = pack2<T>(q0 - r01.x, q1 - r01.y), l23 = pack2<T>(q2 - r23.x, q3 - r23.y);
            const uint32_t bh0 = movmatrix_trans(lo_lane ? l01 : h01), bh1 = movmatrix_trans(lo_lane ? l23 : h23);
            uint32_t m01 = 0xffffffffu, m23 = 0xffffffffu;
            if (nv < kSub) {
                m01 = (2 * t4 < nv ? 0x0000ffffu : 0u) | (2 * t4 + 1 < nv ? 0xffff0000u : 0u);
                m23 = (2 * t4 + 8 < nv ? 0x0000ffffu : 0u) | (2 * t4 + 9 < nv ? 0xffff0000u : 0u);
            }
            // O^T[16 dims x 8 heads] += V^T P
            if constexpr (I8) {
                // codes of 16 tokens x 32 dims per ldmatrix.x4.trans; M row g of an
                // m tile is dim 2g, row g + 8 is dim 2g + 1 (see the output mapping)
                auto pv_i8 = [&](auto lo_pass, uint32_t bl0, uint32_t bl1) {
                    const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                    for (int m2 = 0; m2 < D / 32; ++m2) {
                        const int chunk = 2 * m2 + (lane >> 4);
                        uint32_t r[4];
                        ldmatrix_x4_trans(r, smem_u32(vb + tok * 128 + ((chunk ^ (tok & 7)) << 4)));
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const uint32_t lo = r[2 * u] ^ 0x80808080u, hi = r[2 * u + 1] ^ 0x80808080u;
                            // the signed codes themselves (no 1152 bias): O accumulates
                            // only the signal, so the fp32 accumulator keeps its
                            // precision on long sequences (with the bias it held
                            // ~15x the signal, and 2-4k-token rows of the GQA int8
                            // workload missed the binary64 oracle by up to 6.5e-3)
                            uint32_t a[4];
                            a[0] = i8_pair<T>(lo, 0x4240u);
                            a[1] = i8_pair<T>(lo, 0x4341u);
                            a[2] = i8_pair<T>(hi, 0x4240u);
                            a[3] = i8_pair<T>(hi, 0x4341u);
                            mma_16816<T>(o[2 * m2 + u], a, bh0, bh1);
                            if constexpr (decltype(lo_pass)::value) mma_16816<T>(o[2 * m2 + u], a, bl0, bl1);
                        }
                    }
                };
                if (packlo)
                    pv_i8(std::false_type{}, 0u, 0u);
                else
                    pv_i8(std::true_type{}, movmatrix_trans(l01), movmatrix_trans(l23));
            } else if constexpr (!kLazy) {
                const uint32_t bl0 = movmatrix_trans(l01), bl1 = movmatrix_trans(l23);
                const int tok = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    const int cg = mt * 2 + ((lane >> 3) & 1);
                    uint32_t a[4];
                    ldmatrix_x4_trans(a, smem_u32(vb + (cg >> 3) * kTile + tok * 128 + (((cg & 7) ^ (tok & 7)) << 4)));
                    a[0] &= m01;
                    a[1] &= m01;
                    a[2] &= m23;
                    a[3] &= m23;
                    mma_16816<T>(o[mt], a, bh0, bh1);
                    mma_16816<T>(o[mt], a, bl0, bl1);
                }
            } else {
                auto pv16 = [&](auto lo_pass, uint32_t bl0, uint32_t bl1) {
                    const int tok = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        const int cg = mt * 2 + ((lane >> 3) & 1);
                        uint32_t a[4];
                        ldmatrix_x4_trans(a, smem_u32(vb + (cg >> 3) * kTile + tok * 128 + (((cg & 7) ^ (tok & 7)) << 4)));
                        a[0] &= m01;
                        a[1] &= m01;
                        a[2] &= m23;
                        a[3] &= m23;
                        mma_16816<T>(o[mt], a, bh0, bh1);
                        if constexpr (decltype(lo_pass)::value) mma_16816<T>(o[mt], a, bl0, bl1);
                    }
                };
                if (packlo)
                    pv16(std::false_type{}, 0u, 0u);
                else
                    pv16(std::true_type{}, movmatrix_trans(l01), movmatrix_trans(l23));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == NS) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (aborted) {
            if (lane == 0) {
                s_abort = 1;
                set_err(p.err, PKV_DEVERR_TIMEOUT);
            }
            return;
        }
        if (packlo) {  // O of a head = its high-part column + its low-part column
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[mt][e] += __shfl_xor_sync(0xffffffffu, o[mt][e], G >> 1);
        }
        // sum over the 8 lanes holding other tokens of the same heads
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            lA += __shfl_xor_sync(0xffffffffu, lA, off);
            lB += __shfl_xor_sync(0xffffffffu, lB, off);
        }
        const bool complete = (sb == 0 && b1 == n_s);
        if (complete) {
            const float iA = 1.f / lA, iB = 1.f / lB;
            const int64_t ob = (qrow * (int64_t)(p.hkv * G) + (int64_t)kvh * G) * D;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                const int d0 = I8 ? mt * 16 + 2 * g : mt * 16 + g, d1 = I8 ? d0 + 1 : d0 + 8;
                if (p.out_f32) {
                    float *op = static_cast<float *>(p.out) + ob;
                    if (hA < G) {
                        op[hA * D + d0] = o[mt][0] * iA;
                        op[hA * D + d1] = o[mt][2] * iA;
                    }
                    if (hB < G) {
                        op[hB * D + d0] = o[mt][1] * iB;
                        op[hB * D + d1] = o[mt][3] * iB;
                    }
                } else {
                    T *op = static_cast<T *>(p.out) + ob;
                    if (hA < G) {
                        op[hA * D + d0] = static_cast<T>(o[mt][0] * iA);
                        op[hA * D + d1] = static_cast<T>(o[mt][2] * iA);
                    }
                    if (hB < G) {
                        op[hB * D + d0] = static_cast<T>(o[mt][1] * iB);
                        op[hB * D + d1] = static_cast<T>(o[mt][3] * iB);
                    }
                }
            }
        } else {
            const int slot = first_seg ? 0 : 1;
            const int64_t rec = (((int64_t)hg * p.cmax + blockIdx.x) * 2 + slot) * qheads_cta + (int64_t)w * G;
            float *wo = p.ws_o + rec * D;
            float *wml = p.ws_ml + rec * 2;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                const int d0 = I8 ? mt * 16 + 2 * g : mt * 16 + g, d1 = I8 ? d0 + 1 : d0 + 8;
                if (hA < G) {
                    wo[hA * D + d0] = o[mt][0];
                    wo[hA * D + d1] = o[mt][2];
                }
                if (hB < G) {
                    wo[hB * D + d0] = o[mt][1];
                    wo[hB * D + d1] = o[mt][3];
                }
            }
            if (g == 0) {
                if (hA < G) {
                    wml[hA * 2] = mA;
                    wml[hA * 2 + 1] = lA;
                }
                if (hB < G) {
                    wml[hB * 2] = mB;
                    wml[hB * 2 + 1] = lB;
                }
            }
        }
        first_seg = false;
        x += b1 - sb;
        ++s;
        sb = 0;
    }
}

// Combines the records of sequences cut by a range boundary; writes zero rows
// for empty sequences.  Grid: (sequence, group of kMergeHeads query heads).
// For a cut sequence the CTA first turns the per-part running maxima and sums
// of its heads into weights exp2(m_c - M) / sum_c(l_c exp2(m_c - M)) in shared
// memory; then its threads split the parts between them (a 128k-token
// sequence is cut into ~76 parts), each summing float4 outputs of its parts
// with four loads in flight, and the part-groups are added in shared memory.
// Launched as a programmatic dependent of the decode kernel: it is scheduled
// while that kernel drains and waits for its completion before any read.  Its
// CTAs are kept small (256 threads, ~40 registers each) so they fit on an SM
// beside a decode CTA and are waiting there when it finishes; the same code
// with 512 threads, or with more registers, starts later.
constexpr int kMergeThreads = 256;
// Calls of at most this many sequences with fewer than 8 query heads per
// merge CTA (the host picks 8 for 128 sequences or more): the merge
// recomputes the split itself.  Large calls read the decode kernel's
// metadata instead: there 1,024 merge CTAs scanning 256 lengths each beside
// the running decode kernel slowed the GQA decode step from 0.358 to 0.361 ms,
// while the GPT-2-shaped step gained 1-2% (0.2171 -> 0.2150 ms, fused 0.2048
// -> 0.2007; A/B, one box).
constexpr int kMergeScanMaxSeqs = 1024;

template <int D, typename T, int kMergeHeads>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(const DecodeParams p) {
    extern __shared__ float4 s_merge[];  // [groups][kMergeHeads * D / 4] partial sums, then [parts][heads] weights
    __shared__ int s_scan[32];
    __shared__ long long s_start;
    const int s = blockIdx.x;
    // The split of the concatenated sub-blocks into CTA ranges depends only on
    // the call's inputs (lengths, row offsets, window, table width), which the
    // decode kernel read after its own dependency wait.  This grid starts only
    // once every decode CTA has passed that wait, so the inputs are final here:
    // the split is recomputed before this kernel's wait instead of being read
    // back from the decode kernel's metadata after it (one dependent round trip
    // fewer on the call's path).  Every CTA still waits before it exits, so this
    // grid never completes ahead of the decode grid.
    const bool early = kMergeHeads < 8 && p.num_seqs <= kMergeScanMaxSeqs;
    int64_t total = 0, start = 0, n = 0, ctas = 0;
    bool whole = false;  // every sequence went whole to one decode CTA
    if (early) {
        int64_t carry = 0;
        for (int s0 = 0; s0 < p.num_seqs; s0 += blockDim.x) {
            const int t = s0 + threadIdx.x;
            const int v = t < p.num_seqs ? decode_sub_blocks(p, t) : 0;
            int chunk;
            const int incl = block_scan(v, s_scan, &chunk);
            if (t == s) s_start = carry + incl - v;
            carry += chunk;
        }
        __syncthreads();
        total = carry;
        start = s_start;
        n = decode_sub_blocks(p, s);
        const int64_t want = (total + kMinSubBlocksPerCta - 1) / kMinSubBlocksPerCta;
        ctas = want < p.grid_x ? want : p.grid_x;  // as the decode kernel takes it
        whole = whole_seq_split(total, p.num_seqs, p.grid_x);
    }
    pdl_wait();
    pdl_trigger();
    if (p.cu_q && p.cu_q[s + 1] - p.cu_q[s] != 1) return;
    const int64_t qrow = p.cu_q ? (int64_t)p.cu_q[s] : (int64_t)s;
    const int G = p.group, HG = p.heads_per_cta;
    const int hq = p.hkv * G;
    const int h0 = blockIdx.y * kMergeHeads;
    const int nh = min(kMergeHeads, hq - h0);
    if (!early) {
        total = p.ws_meta[0];
        ctas = p.ws_meta[1];
        start = p.ws_meta[2 + s];
        n = p.ws_meta[3 + s] - start;
    }
    const int64_t ob = (qrow * (int64_t)hq + h0) * D;
    if (n == 0) {
        for (int i = threadIdx.x; i < nh * D; i += blockDim.x) {
            if (p.out_f32)
                static_cast<float *>(p.out)[ob + i] = 0.f;
            else
                static_cast<T *>(p.out)[ob + i] = static_cast<T>(0.f);
        }
        return;
    }
    if (whole) return;  // finished by the decode kernel
    const int c0 = range_owner(start, total, ctas);
    const int c1 = range_owner(start + n - 1, total, ctas);
    if (c0 == c1) return;  // finished by the decode kernel
    const int parts = c1 - c0 + 1;
    const int64_t lo0 = (int64_t)c0 * total / ctas;
    const int slot0 = start == lo0 ? 0 : 1;
    auto record = [&](int c, int h) -> int64_t {
        const int hgi = (h / G) / HG;
        const int hl = h - hgi * HG * G;
        const int slot = c == c0 ? slot0 : 0;
        return (((int64_t)hgi * p.cmax + c) * 2 + slot) * (HG * G) + hl;
    };
    constexpr int OUTS = kMergeHeads * D / 4;          // float4 outputs of a full head group
    constexpr int GROUPS = kMergeThreads / OUTS;        // part groups
    float *s_w = reinterpret_cast<float *>(s_merge + GROUPS * OUTS);
    // thread = (part group, output); its first part's output is loaded now, beside the weights' loads
    const int o = threadIdx.x % OUTS, grp = threadIdx.x / OUTS;
    const int hl = o / (D / 4), d4 = o - hl * (D / 4);
    float4 first = make_float4(0.f, 0.f, 0.f, 0.f);
    if (hl < nh && grp < parts) first = *reinterpret_cast<const float4 *>(p.ws_o + record(c0 + grp, h0 + hl) * D + 4 * d4);
    // weights: one warp per head, lanes over the parts
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < nh) {
        const int h = h0 + warp;
        float M = -INFINITY;
        for (int c = lane; c < parts; c += 32) M = fmaxf(M, p.ws_ml[record(c0 + c, h) * 2]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float Lsum = 0.f;
        for (int c = lane; c < parts; c += 32) {
            const int64_t r = record(c0 + c, h);
            const float e = exp2f(p.ws_ml[r * 2] - M);
            s_w[c * kMergeHeads + warp] = e;
            Lsum += p.ws_ml[r * 2 + 1] * e;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, off);
        const float inv = 1.f / Lsum;
        for (int c = lane; c < parts; c += 32) s_w[c * kMergeHeads + warp] *= inv;
    }
    __syncthreads();
    float4 acc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (hl < nh) {
        const int h = h0 + hl;
        int c = grp;
        if (c < parts) {
            const float w = s_w[c * kMergeHeads + hl];
            acc[0].x += w * first.x;
            acc[0].y += w * first.y;
            acc[0].z += w * first.z;
            acc[0].w += w * first.w;
            c += GROUPS;
        }
        for (; c + 3 * GROUPS < parts; c += 4 * GROUPS) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int cc = c + u * GROUPS;
                const float w = s_w[cc * kMergeHeads + hl];
                const float4 v = *reinterpret_cast<const float4 *>(p.ws_o + record(c0 + cc, h) * D + 4 * d4);
                acc[u].x += w * v.x;
                acc[u].y += w * v.y;
                acc[u].z += w * v.z;
                acc[u].w += w * v.w;
            }
        }
#pragma unroll
        for (int u = 0; u < 3; ++u) {
            const int cc = c + u * GROUPS;
            if (cc < parts) {
                const float w = s_w[cc * kMergeHeads + hl];
                const float4 v = *reinterpret_cast<const float4 *>(p.ws_o + record(c0 + cc, h) * D + 4 * d4);
                acc[u].x += w * v.x;
                acc[u].y += w * v.y;
                acc[u].z += w * v.z;
                acc[u].w += w * v.w;
            }
        }
    }
    s_merge[grp * OUTS + o] = make_float4(acc[0].x + acc[1].x + acc[2].x + acc[3].x, acc[0].y + acc[1].y + acc[2].y + acc[3].y,
                                          acc[0].z + acc[1].z + acc[2].z + acc[3].z, acc[0].w + acc[1].w + acc[2].w + acc[3].w);
    __syncthreads();
    if (grp == 0 && hl < nh) {
        float4 r = s_merge[o];
        for (int g2 = 1; g2 < GROUPS; ++g2) {
            const float4 t = s_merge[g2 * OUTS + o];
            r.x += t.x;
            r.y += t.y;
            r.z += t.z;
            r.w += t.w;
        }
        const int64_t off = ob + (int64_t)hl * D + 4 * d4;
        if (p.out_f32) {
            *reinterpret_cast<float4 *>(static_cast<float *>(p.out) + off) = r;
        } else {
            T *op = static_cast<T *>(p.out) + off;
            *reinterpret_cast<uint2 *>(op) = make_uint2(pack2<T>(r.x, r.y), pack2<T>(r.z, r.w));
        }
    }
}

// ---- host side -------------------------------------------------------------

struct DecodePlan {
    int heads_per_cta, num_hg, stages, threads, smem_bytes, cmax;
    size_t meta_bytes, ml_bytes, o_bytes;
};

static int pick_heads_per_cta(int hkv, int head_dim, bool i8) {
    const int halves = i8 ? 1 : head_dim / 64;  // 2 KB tiles per head per K (or V)
    const int cap = i8 ? kI8HeadsPerCta : head_dim == 64 ? max_heads_per_cta<64>() : max_heads_per_cta<128>();
    for (int hg = cap < hkv ? cap : hkv; hg >= 1; --hg)
        if (hkv % hg == 0 && hg * halves * 2 * kTile <= 64 * 1024) return hg;
    return 1;
}

static size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

static pkv_status make_plan(int32_t num_seqs, int32_t num_q_heads, int32_t hkv, int32_t head_dim, int32_t device,
                            DecodePlan *pl, bool i8 = false) {
    int sms = 0;
    pkv_status st = sm_count(device, &sms);
    if (st != PKV_OK) return st;
    pl->heads_per_cta = pick_heads_per_cta(hkv, head_dim, i8);
    pl->num_hg = hkv / pl->heads_per_cta;
    // persistent: all CTAs resident at once -- one per SM over all head
    // groups (head_dim 128), two per SM for int8 (half-size stages: more
    // consumer warps per SM to hide the code conversion), three for head_dim 64
    const int per_sm = i8 ? kI8CtasPerSm : (head_dim == 64 ? kD64CtasPerSm : 1);
    pl->cmax = per_sm * sms / pl->num_hg > 0 ? per_sm * sms / pl->num_hg : 1;
    const int stage_bytes = pl->heads_per_cta * (i8 ? 1 : head_dim / 64) * 2 * kTile;
    int ns = (200 * 1024 / per_sm) / stage_bytes;
    pl->stages = ns > 16 ? 16 : (ns < 2 ? 2 : ns);
    pl->threads = 32 * (1 + pl->heads_per_cta);
    // stages, alignment slack, barriers, and (int8) two scale rows per stage; <= 210 KB (set once per device)
    pl->smem_bytes = pl->stages * stage_bytes + 1024 + 2 * pl->stages * 8 + (i8 ? pl->stages * 8 * hkv : 0);
    const int group = num_q_heads / hkv;
    const size_t recs = (size_t)pl->num_hg * pl->cmax * 2 * pl->heads_per_cta * group;
    pl->meta_bytes = round256(sizeof(int32_t) * (size_t)(num_seqs + 3));
    pl->ml_bytes = round256(recs * 2 * sizeof(float));
    pl->o_bytes = round256(recs * head_dim * sizeof(float));
    return PKV_OK;
}

template <int D, typename T, bool I8 = false, bool AP = false>
static pkv_status launch_decode_t(const CUtensorMap &mk, const CUtensorMap &mv, const DecodeParams &p,
                                  const DecodePlan &pl, cudaStream_t stream) {
    auto kern = decode_splitk_kernel<D, T, I8, AP>;
    // the plan's shared memory depends only on (D, heads per CTA); size for the largest plan once
    static std::atomic<uint64_t> smem_set{0};
    pkv_status st = set_smem_once(reinterpret_cast<const void *>(kern), 210 * 1024, &smem_set);
    if (st != PKV_OK) return st;
    // the table width bounds a head group's sub-blocks (every sequence at its
    // table's capacity): a small call launches only the CTAs its split can use
    // (the split itself takes min(its need, gridDim.x), so results are the same)
    const int64_t bound = (int64_t)p.num_seqs * p.max_blocks * ((p.block_size + kSub - 1) / kSub);
    const int64_t need = (bound + kMinSubBlocksPerCta - 1) / kMinSubBlocksPerCta;
    unsigned grid_x = (unsigned)(need < 1 ? 1 : need < pl.cmax ? need : pl.cmax);
    // a call this small even at its tables' capacity gets a CTA per sequence,
    // each taking its sequence whole (the kernels check the same bounds)
    if (whole_seq_split(bound, p.num_seqs, pl.cmax) && (unsigned)p.num_seqs > grid_x) grid_x = (unsigned)p.num_seqs;
    DecodeParams pg = p;
    pg.grid_x = (int32_t)grid_x;
    st = launch_pdl(kern, dim3(grid_x, pl.num_hg), dim3(pl.threads), (size_t)pl.smem_bytes, stream, mk, mv, pg);
    if (st != PKV_OK) return st;
    // a call the small-call split surely covers (total <= bound, grid = a CTA
    // per sequence) cuts no sequence, and its empty rows are written by the
    // decode kernel: no merge
    if (whole_seq_split(bound, p.num_seqs, grid_x)) return PKV_OK;
    // the merge reads only what the decode kernel wrote: launch it as a
    // programmatic dependent so it is scheduled while the decode kernel drains
    // many sequences: 8 query heads per merge CTA (fewer, mostly idle, CTAs);
    // fewer: 4 (more CTAs share a long sequence's parts); so few that even
    // that leaves SMs idle: 1
    const int hq = p.hkv * p.group;
    const int mh = p.num_seqs >= 128 ? 8 : (int64_t)p.num_seqs * ((hq + 3) / 4) >= pl.cmax * pl.num_hg ? 4 : 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.num_seqs, (hq + mh - 1) / mh);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = (size_t)kMergeThreads * sizeof(float4) + (size_t)p.cmax * mh * sizeof(float);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    auto merge = mh == 8 ? decode_merge_kernel<D, T, 8> : mh == 4 ? decode_merge_kernel<D, T, 4> : decode_merge_kernel<D, T, 1>;
    PKV_CUDA_TRY(cudaLaunchKernelEx(&cfg, merge, pg));
    return PKV_OK;
}

// Shared by pkv_attn_decode[_window|_append] (cu_q == NULL) and pkv_attn_varlen[_window] (q_len == 1 rows).
static pkv_status run_decode_impl(const void *q, int64_t q_stride, const pkv_cache *cache, const int32_t *tables,
                                  int32_t max_blocks, const int32_t *seq_lens, const int32_t *cu_q, int32_t num_seqs,
                                  int32_t num_q_heads, float scale, int32_t window, void *out, int32_t out_dtype,
                                  void *workspace, size_t workspace_bytes, int32_t *err_word, cudaStream_t stream,
                                  const void *k_new, const void *v_new, int64_t new_stride) {
    DecodePlan pl;
    pkv_status st = make_plan(num_seqs, num_q_heads, cache->num_kv_heads, cache->head_dim, -1, &pl);
    if (st != PKV_OK) return st;
    const size_t need = pl.meta_bytes + pl.ml_bytes + pl.o_bytes;
    PKV_CHECK_ARG(workspace && workspace_bytes >= need, PKV_ERR_WORKSPACE,
                  "workspace of %zu bytes given, %zu needed", workspace_bytes, need);
    PKV_CHECK_ARG((reinterpret_cast<uintptr_t>(workspace) & 255) == 0, PKV_ERR_INVALID_ARG,
                  "workspace must be 256-byte aligned");
    CUtensorMap mk, mv;
    const int chunks = pl.heads_per_cta * (cache->head_dim / 64);
    st = encode_pool_rows_map(&mk, cache->k, cache, chunks);
    if (st != PKV_OK) return st;
    st = encode_pool_rows_map(&mv, cache->v, cache, chunks);
    if (st != PKV_OK) return st;
    DecodeParams p{};
    p.q = q;
    p.q_stride = q_stride;
    p.tables = tables;
    p.max_blocks = max_blocks;
    p.seq_lens = seq_lens;
    p.cu_q = cu_q;
    p.num_seqs = num_seqs;
    p.num_blocks = cache->num_blocks;
    p.block_size = cache->block_size;
    p.hkv = cache->num_kv_heads;
    p.heads_per_cta = pl.heads_per_cta;
    p.group = num_q_heads / cache->num_kv_heads;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.out = out;
    p.out_f32 = out_dtype == PKV_F32;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.ws_meta = reinterpret_cast<int32_t *>(ws);
    p.ws_ml = reinterpret_cast<float *>(ws + pl.meta_bytes);
    p.ws_o = reinterpret_cast<float *>(ws + pl.meta_bytes + pl.ml_bytes);
    p.cmax = pl.cmax;
    p.err = err_word;
    p.stages = pl.stages;
    p.window = window > 0 ? window : 0;
    p.k_new = k_new;
    p.v_new = v_new;
    p.new_stride = new_stride;
    p.k_pool = cache->k;
    p.v_pool = cache->v;
    const bool bf = cache->dtype == PKV_BF16;
    if (k_new != nullptr) {
        if (cache->head_dim == 64)
            return bf ? launch_decode_t<64, __nv_bfloat16, false, true>(mk, mv, p, pl, stream)
                      : launch_decode_t<64, __half, false, true>(mk, mv, p, pl, stream);
        return bf ? launch_decode_t<128, __nv_bfloat16, false, true>(mk, mv, p, pl, stream)
                  : launch_decode_t<128, __half, false, true>(mk, mv, p, pl, stream);
    }
    if (cache->head_dim == 64)
        return bf ? launch_decode_t<64, __nv_bfloat16>(mk, mv, p, pl, stream)
                  : launch_decode_t<64, __half>(mk, mv, p, pl, stream);
    return bf ? launch_decode_t<128, __nv_bfloat16>(mk, mv, p, pl, stream)
              : launch_decode_t<128, __half>(mk, mv, p, pl, stream);
}

pkv_status run_decode_window(const void *q, int64_t q_stride, const pkv_cache *cache, const int32_t *tables,
                             int32_t max_blocks, const int32_t *seq_lens, const int32_t *cu_q, int32_t num_seqs,
                             int32_t num_q_heads, float scale, int32_t window, void *out, int32_t out_dtype,
                             void *workspace, size_t workspace_bytes, int32_t *err_word, cudaStream_t stream) {
    return run_decode_impl(q, q_stride, cache, tables, max_blocks, seq_lens, cu_q, num_seqs, num_q_heads, scale,
                           window, out, out_dtype, workspace, workspace_bytes, err_word, stream, nullptr, nullptr, 0);
}

pkv_status run_decode(const void *q, int64_t q_stride, const pkv_cache *cache, const int32_t *tables,
                      int32_t max_blocks, const int32_t *seq_lens, const int32_t *cu_q, int32_t num_seqs,
                      int32_t num_q_heads, float scale, void *out, int32_t out_dtype, void *workspace,
                      size_t workspace_bytes, int32_t *err_word, cudaStream_t stream) {
    return run_decode_window(q, q_stride, cache, tables, max_blocks, seq_lens, cu_q, num_seqs, num_q_heads, scale, 0,
                             out, out_dtype, workspace, workspace_bytes, err_word, stream);
}

pkv_status check_cache_i8(const pkv_cache_i8 *c, const char *what);  // int8_write.cu

static pkv_status run_decode_i8(const void *q, int64_t q_stride, const pkv_cache_i8 *cache, const int32_t *tables,
                                int32_t max_blocks, const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_heads,
                                float scale, int32_t window, void *out, int32_t out_dtype, void *workspace,
                                size_t workspace_bytes, int32_t *err_word, cudaStream_t stream) {
    DecodePlan pl;
    pkv_status st = make_plan(num_seqs, num_q_heads, cache->num_kv_heads, cache->head_dim, -1, &pl, true);
    if (st != PKV_OK) return st;
    const size_t need = pl.meta_bytes + pl.ml_bytes + pl.o_bytes;
    PKV_CHECK_ARG(workspace && workspace_bytes >= need, PKV_ERR_WORKSPACE,
                  "workspace of %zu bytes given, %zu needed", workspace_bytes, need);
    PKV_CHECK_ARG((reinterpret_cast<uintptr_t>(workspace) & 255) == 0, PKV_ERR_INVALID_ARG,
                  "workspace must be 256-byte aligned");
    CUtensorMap mk, mv;
    st = encode_pool_rows_map_i8(&mk, cache->k, cache, pl.heads_per_cta);
    if (st != PKV_OK) return st;
    st = encode_pool_rows_map_i8(&mv, cache->v, cache, pl.heads_per_cta);
    if (st != PKV_OK) return st;
    DecodeParams p{};
    p.q = q;
    p.q_stride = q_stride;
    p.tables = tables;
    p.max_blocks = max_blocks;
    p.seq_lens = seq_lens;
    p.cu_q = nullptr;
    p.num_seqs = num_seqs;
    p.num_blocks = cache->num_blocks;
    p.block_size = cache->block_size;
    p.hkv = cache->num_kv_heads;
    p.heads_per_cta = pl.heads_per_cta;
    p.group = num_q_heads / cache->num_kv_heads;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.out = out;
    p.out_f32 = out_dtype == PKV_F32;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.ws_meta = reinterpret_cast<int32_t *>(ws);
    p.ws_ml = reinterpret_cast<float *>(ws + pl.meta_bytes);
    p.ws_o = reinterpret_cast<float *>(ws + pl.meta_bytes + pl.ml_bytes);
    p.cmax = pl.cmax;
    p.err = err_word;
    p.stages = pl.stages;
    p.window = window > 0 ? window : 0;
    p.k_scale = cache->k_scale;
    p.v_scale = cache->v_scale;
    return cache->dtype == PKV_BF16 ? launch_decode_t<128, __nv_bfloat16, true>(mk, mv, p, pl, stream)
                                    : launch_decode_t<128, __half, true>(mk, mv, p, pl, stream);
}

// Workspace of the 16-bit decode plan (the no-allocation entry point sizes its call with this).
pkv_status decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t hkv, int32_t head_dim,
                                 int32_t device, size_t *bytes) {
    DecodePlan pl;
    pkv_status st = make_plan(num_seqs, num_q_heads, hkv, head_dim, device, &pl);
    if (st != PKV_OK) return st;
    *bytes = pl.meta_bytes + pl.ml_bytes + pl.o_bytes;
    return PKV_OK;
}

// The larger of the 16-bit and int8 plans: one workspace serves every decode call.
static pkv_status decode_workspace_size_any(int32_t num_seqs, int32_t num_q_heads, int32_t hkv, int32_t head_dim,
                                            int32_t device, size_t *bytes) {
    size_t a = 0;
    pkv_status st = decode_workspace_size(num_seqs, num_q_heads, hkv, head_dim, device, &a);
    if (st != PKV_OK) return st;
    DecodePlan pl;
    st = make_plan(num_seqs, num_q_heads, hkv, head_dim, device, &pl, true);
    if (st != PKV_OK) return st;
    const size_t b = pl.meta_bytes + pl.ml_bytes + pl.o_bytes;
    *bytes = a > b ? a : b;
    return PKV_OK;
}

pkv_status check_attention_common(const void *q, int64_t q_stride, const pkv_cache *cache, const int32_t *tables,
                                  int32_t max_blocks, const int32_t *seq_lens, int32_t num_seqs,
                                  int32_t num_q_heads, void *out, int32_t out_dtype, const char *what) {
    pkv_status st = check_cache(cache, what);
    if (st != PKV_OK) return st;
    st = check_attention_shapes(cache, num_q_heads);
    if (st != PKV_OK) return st;
    PKV_CHECK_ARG(num_seqs >= 0 && max_blocks >= 0, PKV_ERR_INVALID_ARG, "%s: negative size", what);
    PKV_CHECK_ARG(out_dtype == PKV_F32 || out_dtype == cache->dtype, PKV_ERR_DTYPE,
                  "%s: out dtype must be F32 or the cache's dtype", what);
    PKV_CHECK_ARG(q_stride >= (int64_t)num_q_heads * cache->head_dim, PKV_ERR_SHAPE,
                  "%s: q_token_stride %lld shorter than a row", what, (long long)q_stride);
    PKV_CHECK_ARG((q_stride % 2) == 0 && (reinterpret_cast<uintptr_t>(q) & 3) == 0, PKV_ERR_INVALID_ARG,
                  "%s: q rows must be 4-byte aligned", what);
    if (num_seqs > 0)
        PKV_CHECK_ARG(q && tables && seq_lens && out, PKV_ERR_INVALID_ARG, "%s: NULL pointer", what);
    PKV_CHECK_ARG(aligned16(out), PKV_ERR_INVALID_ARG, "%s: out must be 16-byte aligned", what);
    return PKV_OK;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

pkv_status pkv_attn_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t device, size_t *bytes) {
    PKV_CHECK_ARG(bytes && num_seqs >= 0 && num_kv_heads > 0 && num_q_heads > 0 && head_dim > 0,
                  PKV_ERR_INVALID_ARG, "bad argument");
    pkv_status st = decode_workspace_size_any(num_seqs, num_q_heads, num_kv_heads, head_dim, device, bytes);
    return st == PKV_OK ? ok() : st;
}

pkv_status pkv_attn_decode(const void *q, int64_t q_token_stride, const pkv_cache *cache, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_heads,
                           float scale, void *out, int32_t out_dtype, void *workspace, size_t workspace_bytes,
                           int32_t *err_word, pkv_stream stream) {
    pkv_status st = check_attention_common(q, q_token_stride, cache, block_tables, max_blocks_per_seq, seq_lens,
                                           num_seqs, num_q_heads, out, out_dtype, "pkv_attn_decode");
    if (st != PKV_OK) return st;
    if (num_seqs == 0) return ok();
    st = run_decode(q, q_token_stride, cache, block_tables, max_blocks_per_seq, seq_lens, nullptr, num_seqs,
                    num_q_heads, scale, out, out_dtype, workspace, workspace_bytes, err_word, stream);
    return st == PKV_OK ? ok() : st;
}

pkv_status pkv_attn_decode_window(const void *q, int64_t q_token_stride, const pkv_cache *cache,
                                  const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                  int32_t num_seqs, int32_t num_q_heads, float scale, int32_t window, void *out,
                                  int32_t out_dtype, void *workspace, size_t workspace_bytes, int32_t *err_word,
                                  pkv_stream stream) {
    pkv_status st = check_attention_common(q, q_token_stride, cache, block_tables, max_blocks_per_seq, seq_lens,
                                           num_seqs, num_q_heads, out, out_dtype, "pkv_attn_decode_window");
    if (st != PKV_OK) return st;
    if (num_seqs == 0) return ok();
    st = run_decode_window(q, q_token_stride, cache, block_tables, max_blocks_per_seq, seq_lens, nullptr, num_seqs,
                           num_q_heads, scale, window, out, out_dtype, workspace, workspace_bytes, err_word, stream);
    return st == PKV_OK ? ok() : st;
}

pkv_status pkv_attn_decode_append(const void *q, int64_t q_token_stride, const void *k_new, const void *v_new,
                                  int64_t kv_token_stride, const pkv_cache *cache, const int32_t *block_tables,
                                  int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs,
                                  int32_t num_q_heads, float scale, int32_t window, void *out, int32_t out_dtype,
                                  void *workspace, size_t workspace_bytes, int32_t *err_word, pkv_stream stream) {
    pkv_status st = check_attention_common(q, q_token_stride, cache, block_tables, max_blocks_per_seq, seq_lens,
                                           num_seqs, num_q_heads, out, out_dtype, "pkv_attn_decode_append");
    if (st != PKV_OK) return st;
    if (num_seqs == 0) return ok();
    PKV_CHECK_ARG(k_new && v_new, PKV_ERR_INVALID_ARG, "pkv_attn_decode_append: k_new and v_new must be non-NULL");
    PKV_CHECK_ARG(kv_token_stride >= (int64_t)cache->num_kv_heads * cache->head_dim, PKV_ERR_SHAPE,
                  "pkv_attn_decode_append: kv_token_stride shorter than a row");
    PKV_CHECK_ARG(aligned16(k_new) && aligned16(v_new) && kv_token_stride % 8 == 0, PKV_ERR_INVALID_ARG,
                  "pkv_attn_decode_append: k_new / v_new rows must be 16-byte aligned");
    st = run_decode_impl(q, q_token_stride, cache, block_tables, max_blocks_per_seq, seq_lens, nullptr, num_seqs,
                         num_q_heads, scale, window, out, out_dtype, workspace, workspace_bytes, err_word, stream, k_new,
                         v_new, kv_token_stride);
    return st == PKV_OK ? ok() : st;
}

pkv_status pkv_attn_decode_int8(const void *q, int64_t q_token_stride, const pkv_cache_i8 *cache,
                                const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                int32_t num_seqs, int32_t num_q_heads, float scale, int32_t window, void *out,
                                int32_t out_dtype, void *workspace, size_t workspace_bytes, int32_t *err_word,
                                pkv_stream stream) {
    pkv_status st = check_cache_i8(cache, "pkv_attn_decode_int8");
    if (st != PKV_OK) return st;
    PKV_CHECK_ARG(cache->head_dim == 128, PKV_ERR_UNSUPPORTED, "int8 decode: head_dim must be 128");
    PKV_CHECK_ARG(cache->num_kv_heads % 4 == 0, PKV_ERR_UNSUPPORTED, "int8 decode: num_kv_heads must be a multiple of 4");
    PKV_CHECK_ARG(cache->block_size % 16 == 0, PKV_ERR_UNSUPPORTED, "int8 decode: block_size must be a multiple of 16");
    PKV_CHECK_ARG(num_q_heads > 0 && num_q_heads % cache->num_kv_heads == 0, PKV_ERR_SHAPE,
                  "num_q_heads must be a multiple of num_kv_heads");
    const int group = num_q_heads / cache->num_kv_heads;
    PKV_CHECK_ARG(group == 1 || group == 2 || group == 4 || group == 8, PKV_ERR_UNSUPPORTED,
                  "query heads per KV head must be 1, 2, 4 or 8");
    PKV_CHECK_ARG(num_seqs >= 0 && max_blocks_per_seq >= 0, PKV_ERR_INVALID_ARG, "negative size");
    PKV_CHECK_ARG(out_dtype == PKV_F32 || out_dtype == cache->dtype, PKV_ERR_DTYPE, "out dtype must be F32 or q's");
    PKV_CHECK_ARG(q_token_stride >= (int64_t)num_q_heads * 128 && q_token_stride % 2 == 0 &&
                      (reinterpret_cast<uintptr_t>(q) & 7) == 0,
                  PKV_ERR_INVALID_ARG, "q rows must be 8-byte aligned and at least one row long");
    PKV_CHECK_ARG(aligned16(out), PKV_ERR_INVALID_ARG, "out must be 16-byte aligned");
    if (num_seqs == 0) return ok();
    PKV_CHECK_ARG(q && block_tables && seq_lens && out, PKV_ERR_INVALID_ARG, "NULL pointer");
    st = run_decode_i8(q, q_token_stride, cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs, num_q_heads,
                       scale, window, out, out_dtype, workspace, workspace_bytes, err_word, stream);
    return st == PKV_OK ? ok() : st;
}

}  // extern "C"
