// prefill_tc.cu -- a8, prefill chunks (q_len > 1) on the 5th-generation tensor
// cores: tcgen05.mma with accumulators in tensor memory (TMEM).
//
// "Building a paged inference engine from scratch, and measuring it honestly",
// sections 02-03: a packed step holds prefill chunks whose keys are read
// through the block table, and query row i of a chunk with q_len rows and
// kv_len keys sees keys t <= kv_len - q_len + i.  For a chunk the work is a
// dense contraction, so it runs here as a FlashAttention-style loop on UMMA:
//
//  * CTA = 128 M rows: the G query heads of one KV head x 128/G query
//    positions (row r -> head r / (128/G), position q0 + r % (128/G)), so every
//    K/V tile staged in shared memory serves all G heads.
//  * Warp 0 streams Q once and then 64-token K and V tiles of the KV head
//    (TMA, 16 tokens x 64 dims x 128-byte swizzle per box, through the block
//    table) into a 2-stage ring.
//  * Warp 1, one thread, issues the MMAs: S = Q K^T (M 128, N 64, K 16 steps,
//    both operands K-major from shared memory) into one of two TMEM score
//    buffers, and O += P V (A = P read from TMEM, B = V as an MN-major shared
//    operand, N = head_dim) into a TMEM accumulator.  Completion is signalled
//    with tcgen05.commit on mbarriers.
//  * Warps 2-5 (one TMEM lane = one M row per thread) read scores from TMEM,
//    apply the causal limit, keep the running max and sum in registers, and
//    write P back over the scores as a 16-bit hi + lo pair (two MMAs keep
//    ~16 significant bits of P).  The running max is only moved when it grows
//    by more than 2^8; then those rows of O are rescaled in TMEM after the
//    previous P V has completed.  The final O row is divided by the sum and
//    stored.
// Two CTAs share an SM (256 TMEM columns and ~97 KB of shared memory each),
// so one CTA's softmax overlaps the other's MMAs.
#include <cuda.h>

#include "launch.h"
#include "ptx.cuh"

namespace pkv {

namespace {

constexpr int kTok = 64;          // keys per score tile
constexpr int kStages = 2;
constexpr int kTmemCols = 256;    // S0 [0,64) S1 [64,128) O [128, 128 + D)
constexpr float kRescaleLog2 = 8.f;

template <typename T>
struct IsBf16 {
    static constexpr bool value = false;
};
template <>
struct IsBf16<__nv_bfloat16> {
    static constexpr bool value = true;
};

struct TcParams {
    const int32_t *tables;
    int32_t max_blocks;
    const int32_t *seq_lens;
    const int32_t *cu_q;
    int32_t num_blocks, block_size, hkv, group, causal;
    float scale_log2;
    void *out;
    int32_t out_f32;
    int32_t *err;
    int32_t q_tiles;
    int32_t window;   // > 0: each row attends only its most recent `window` keys
};

// UMMA shared-memory descriptor, 128-byte swizzle (sm_100 family layout:
// start >> 4 in bits 0-13, LBO >> 4 in 16-29, SBO >> 4 in 32-45, version 1 at
// bit 46, swizzle mode 2 in bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)((lbo & 0x3FFFF) >> 4) << 16) |
           ((uint64_t)((sbo & 0x3FFFF) >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 D, A/B fp16 or bf16, A K-major,
// B K-major or MN-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_f16(int bf16, int b_mn_major, int M, int N) {
    return (1u << 4) | ((uint32_t)bf16 << 7) | ((uint32_t)bf16 << 10) | ((uint32_t)b_mn_major << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

}  // namespace

template <int D, typename T>
__global__ void __launch_bounds__(192, 2)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const TcParams p) {
    constexpr int HALVES = D / 64;
    constexpr int QHALF = 128 * 128;            // bytes of 128 rows x 64 dims
    constexpr int KVHALF = kTok * 128;           // bytes of 64 tokens x 64 dims
    constexpr int STAGE = 2 * HALVES * KVHALF;   // K then V
    constexpr bool BF = IsBf16<T>::value;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bars[2 + 2 * kStages + 6];
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sq = base;
    uint8_t *skv = base + HALVES * QHALF;
    uint64_t *q_full = &bars[0];
    uint64_t *kv_full = &bars[1];
    uint64_t *kv_empty = &bars[1 + kStages];
    uint64_t *s_full = &bars[1 + 2 * kStages];
    uint64_t *p_full = s_full + 2;
    uint64_t *o_done = p_full + 2;
    uint64_t *fin = o_done + 2;  // abort path: completion of every MMA issued

    const int s = blockIdx.y;
    const int kvh = blockIdx.z;
    const int tile = p.q_tiles - 1 - blockIdx.x;  // longest causal tiles first
    const int q_begin = p.cu_q[s];
    const int q_len = p.cu_q[s + 1] - q_begin;
    const int kv_len = p.seq_lens[s];
    const int G = p.group;
    const int R = 128 / G;                        // query positions per CTA
    const int q0 = tile * R;
    if (q_len <= 1 || q0 >= q_len) return;
    if (q_len > kv_len || (int64_t)kv_len > (int64_t)p.max_blocks * p.block_size) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && kvh == 0) set_err(p.err, PKV_DEVERR_LENGTH);
        return;
    }
    const int last_row = min(q_len, q0 + R) - 1;
    const int kv_hi = p.causal ? kv_len - q_len + last_row + 1 : kv_len;
    // window: the CTA's first row has the lowest first key of its rows
    const int lim_first = p.causal ? kv_len - q_len + q0 : kv_len - 1;
    const int lo_first = (p.window > 0 && lim_first - p.window + 1 > 0) ? lim_first - p.window + 1 : 0;
    const int j_first = lo_first / kTok;
    const int nt = (kv_hi + kTok - 1) / kTok - j_first;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        s_abort = 0;
        mbar_init(q_full, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 128);
            mbar_init(&o_done[i], 1);
        }
        mbar_init(fin, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        // ===== producer: Q once, then K/V tiles =====
        const uint64_t pol_q = policy_evict_first();
        const uint64_t pol_kv = policy_evict_last();  // re-read by the other q tiles of the chunk
        if (lane == 0) {
            prefetch_tensormap(&tmq);
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
            mbar_arrive_expect_tx(q_full, (uint32_t)(G * HALVES * R * 128));
        }
        __syncwarp();
        for (int t = lane; t < G * HALVES; t += 32) {
            const int g = t / HALVES, half = t % HALVES;
            tma_load_3d(sq + half * QHALF + g * R * 128, &tmq, q_full, 0, (kvh * G + g) * HALVES + half, q_begin + q0,
                        pol_q);
        }
        const int32_t *trow = p.tables + (int64_t)s * p.max_blocks;
        int issued = 0;
        for (int j = 0; j < nt; ++j) {
            const int stage = j % kStages;
            int okw = 1;
            if (lane == 0) okw = mbar_wait(&kv_empty[stage], ((j / kStages) & 1) ^ 1, &s_abort);
            okw = __shfl_sync(0xffffffffu, okw, 0);
            if (!okw) {
                if (lane == 0) {
                    s_abort = 1;
                    set_err(p.err, PKV_DEVERR_TIMEOUT);
                }
                break;
            }
            const int t0 = (j_first + j) * kTok;
            const int nvalid = min(kTok, kv_len - t0);
            const int nsub = (nvalid + 15) / 16;
            if (lane == 0) mbar_arrive_expect_tx(&kv_full[stage], (uint32_t)(nsub * 2 * HALVES * 2048));
            __syncwarp();
            for (int t = lane; t < nsub * 2 * HALVES; t += 32) {
                const int sub = t / (2 * HALVES), r = t % (2 * HALVES);
                const int which = r / HALVES, half = r % HALVES;
                const int tok = t0 + sub * 16;
                const int lb = tok / p.block_size;
                int phys = trow[lb];
                if (phys < 0 || phys >= p.num_blocks) {
                    set_err(p.err, PKV_DEVERR_BLOCK);
                    phys = 0;
                }
                const int row = phys * p.block_size + (tok - lb * p.block_size);
                uint8_t *dst = skv + stage * STAGE + which * (HALVES * KVHALF) + half * KVHALF + sub * 2048;
                tma_load_3d(dst, which ? &tmv : &tmk, &kv_full[stage], 0, kvh * HALVES + half, row, pol_kv);
            }
            issued = j + 1;
        }
        if (s_abort && lane == 0) {
            // the loads this warp issued must land before the CTA exits
            volatile int never = 0;
            mbar_wait(q_full, 0, &never);
            for (int k = issued > kStages ? issued - kStages : 0; k < issued; ++k)
                mbar_wait(&kv_full[k % kStages], (k / kStages) & 1, &never);
        }
    } else if (warp == 1) {
        // ===== MMA issuer =====
        if (lane == 0) {
            const uint32_t idS = idesc_f16(BF ? 1 : 0, 0, 128, kTok);
            const uint32_t idPV = idesc_f16(BF ? 1 : 0, 1, 128, D);
            const uint32_t sq_a = smem_u32(sq), skv_a = smem_u32(skv);
            bool ok = mbar_wait(q_full, 0, &s_abort);
            auto issue_pv = [&](int i) -> bool {
                const int b = i & 1, stage = i % kStages;
                if (!mbar_wait(&p_full[b], (i >> 1) & 1, &s_abort)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kTok / 16; ++kk) {
                    const uint64_t vd = sw128_desc(skv_a + stage * STAGE + HALVES * KVHALF + kk * 2048, KVHALF, 1024);
                    umma_ts(tmem + 128, tmem + b * 64 + kk * 8, vd, idPV, (i > 0 || kk > 0) ? 1u : 0u);
                    umma_ts(tmem + 128, tmem + b * 64 + 32 + kk * 8, vd, idPV, 1u);
                }
                umma_commit(&o_done[b]);
                umma_commit(&kv_empty[stage]);
                return true;
            };
            for (int j = 0; j < nt && ok; ++j) {
                const int stage = j % kStages, b = j & 1;
                ok = mbar_wait(&kv_full[stage], (j / kStages) & 1, &s_abort);
                if (ok && j >= 2) ok = mbar_wait(&o_done[b], ((j - 2) >> 1) & 1, &s_abort);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int half = kk >> 2, koff = (kk & 3) * 32;
                    const uint64_t ad = sw128_desc(sq_a + half * QHALF + koff, 16, 1024);
                    const uint64_t bd = sw128_desc(skv_a + stage * STAGE + half * KVHALF + koff, 16, 1024);
                    umma_ss(tmem + b * 64, ad, bd, idS, kk > 0 ? 1u : 0u);
                }
                umma_commit(&s_full[b]);
                if (j >= 1) ok = issue_pv(j - 1);
            }
            if (ok) ok = issue_pv(nt - 1);
            if (!ok) {
                s_abort = 1;
                set_err(p.err, PKV_DEVERR_TIMEOUT);
            }
        }
    } else {
        // ===== softmax + epilogue: one M row per thread =====
        const int qw = warp & 3;
        const int row = qw * 32 + lane;
        const uint32_t trow_addr = tmem + ((uint32_t)(qw * 32) << 16);
        const int g = row / R;
        const int qi = q0 + row % R;
        const bool valid = qi < q_len;
        const int lim = (p.causal && valid) ? kv_len - q_len + qi : kv_len - 1;
        const int lo = (p.window > 0 && lim - p.window + 1 > 0) ? lim - p.window + 1 : 0;
        const float sl = p.scale_log2;
        float m_used = -INFINITY, lsum = 0.f;
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            const int b = j & 1;
            // warp-uniform outcome: the tcgen05 ld/st below are warp-collective
            if (!__all_sync(0xffffffffu, mbar_wait(&s_full[b], (j >> 1) & 1, &s_abort))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[64];
            tmem_ld32(trow_addr + b * 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
            tmem_ld32(trow_addr + b * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
            tmem_wait_ld();
            const int t0 = (j_first + j) * kTok;
            // eight independent partial maxima (short dependency chains);
            // tiles every row of the warp sees in full skip the causal select
            float pm[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) pm[u] = -INFINITY;
            if (__all_sync(0xffffffffu, t0 + kTok - 1 <= lim && t0 >= lo)) {
#pragma unroll
                for (int c = 0; c < kTok; ++c) {
                    const float x = __uint_as_float(sr[c]) * sl;
                    sr[c] = __float_as_uint(x);
                    pm[c & 7] = fmaxf(pm[c & 7], x);
                }
            } else {
#pragma unroll
                for (int c = 0; c < kTok; ++c) {
                    const float x = (t0 + c <= lim && t0 + c >= lo) ? __uint_as_float(sr[c]) * sl : -INFINITY;
                    sr[c] = __float_as_uint(x);
                    pm[c & 7] = fmaxf(pm[c & 7], x);
                }
            }
            const float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                                   fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
            const float m_new = fmaxf(m_used, mx);
            const bool need = m_new > m_used + kRescaleLog2;
            const float alpha = need ? fast_exp2(m_used - m_new) : 1.f;
            if (__any_sync(0xffffffffu, need) && j > 0) {
                // the previous P V must be complete before its rows are rescaled
                if (!__all_sync(0xffffffffu, mbar_wait(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1, &s_abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t orr[32];
                    tmem_ld32(trow_addr + 128 + c0, orr);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) orr[c] = __float_as_uint(__uint_as_float(orr[c]) * alpha);
                    tmem_st32(trow_addr + 128 + c0, orr);
                }
                tmem_wait_st();
            }
            if (need) {
                lsum *= alpha;
                m_used = m_new;
            }
            uint32_t ph[32], pl[32];
            float ps[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) ps[u] = 0.f;
            // with a window a row can meet whole tiles before its first key:
            // there m_used is still -inf and those p must be 0, not NaN
            const bool none_yet = m_used == -INFINITY;
#pragma unroll
            for (int c = 0; c < kTok; c += 2) {
                float p0 = fast_exp2(__uint_as_float(sr[c]) - m_used);
                float p1 = fast_exp2(__uint_as_float(sr[c + 1]) - m_used);
                if (none_yet) {
                    p0 = 0.f;
                    p1 = 0.f;
                }
                ps[(c >> 1) & 7] += p0 + p1;
                const uint32_t h = pack2<T>(p0, p1);
                const float2 hf = unpack2<T>(h);
                ph[c / 2] = h;
                pl[c / 2] = pack2<T>(p0 - hf.x, p1 - hf.y);
            }
            lsum += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
            tmem_st32(trow_addr + b * 64, ph);
            tmem_st32(trow_addr + b * 64 + 32, pl);
            // V rows past kv_len in this tile hold stale or unrelated data: zero them
            if (t0 + kTok > kv_len) {
                const int rr = row & (kTok - 1), half = row / kTok;
                if (half < HALVES && rr >= kv_len - t0) {
                    uint4 *dst = reinterpret_cast<uint4 *>(skv + (j % kStages) * STAGE + HALVES * KVHALF +
                                                           half * KVHALF + rr * 128);
#pragma unroll
                    for (int c = 0; c < 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&p_full[b]);
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&o_done[(nt - 1) & 1], ((nt - 1) >> 1) & 1, &s_abort));
        if (ok) {
            tc_fence_after();
            const float inv = 1.f / lsum;
            const int64_t hq = (int64_t)p.hkv * G;
            const int64_t off = ((int64_t)(q_begin + qi) * hq + (int64_t)kvh * G + g) * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t orr[32];
                tmem_ld32(trow_addr + 128 + c0, orr);
                tmem_wait_ld();
                if (valid) {
                    if (p.out_f32) {
                        float4 *op = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + off + c0);
#pragma unroll
                        for (int c = 0; c < 32; c += 4)
                            op[c / 4] = make_float4(__uint_as_float(orr[c]) * inv, __uint_as_float(orr[c + 1]) * inv,
                                                    __uint_as_float(orr[c + 2]) * inv, __uint_as_float(orr[c + 3]) * inv);
                    } else {
                        uint4 *op = reinterpret_cast<uint4 *>(static_cast<T *>(p.out) + off + c0);
#pragma unroll
                        for (int c = 0; c < 32; c += 8)
                            op[c / 8] = make_uint4(
                                pack2<T>(__uint_as_float(orr[c]) * inv, __uint_as_float(orr[c + 1]) * inv),
                                pack2<T>(__uint_as_float(orr[c + 2]) * inv, __uint_as_float(orr[c + 3]) * inv),
                                pack2<T>(__uint_as_float(orr[c + 4]) * inv, __uint_as_float(orr[c + 5]) * inv),
                                pack2<T>(__uint_as_float(orr[c + 6]) * inv, __uint_as_float(orr[c + 7]) * inv));
                    }
                }
            }
        } else if (lane == 0) {
            s_abort = 1;
            set_err(p.err, PKV_DEVERR_TIMEOUT);
        }
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    if (s_abort && warp == 1 && lane == 0) {
        // an abandoned pipeline: let every MMA issued so far land before TMEM is released
        umma_commit(fin);
        volatile int never = 0;
        mbar_wait(fin, 0, &never);
    }
    __syncwarp();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

template <int D, typename T>
static pkv_status launch_prefill_tc_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                                      const TcParams &p, int num_seqs, cudaStream_t stream) {
    constexpr int HALVES = D / 64;
    // + 1 KB for the 1024-byte alignment of the swizzled tiles, + 4 KB of slack after the last stage
    const int smem = HALVES * 128 * 128 + kStages * 2 * HALVES * kTok * 128 + 1024 + 4096;
    auto kern = prefill_tc_kernel<D, T>;
    static std::atomic<uint64_t> smem_set{0};
    pkv_status st = set_smem_once(reinterpret_cast<const void *>(kern), smem, &smem_set);
    if (st != PKV_OK) return st;
    dim3 grid(p.q_tiles, num_seqs, p.hkv);
    kern<<<grid, 192, smem, stream>>>(mq, mk, mv, p);
    PKV_CUDA_TRY(cudaGetLastError());
    return PKV_OK;
}

// Prefill chunks of a varlen call on tcgen05 (rows of q_len == 1 are left to the decode kernel).
pkv_status run_prefill_tc(const void *q, int64_t q_stride, const pkv_cache *cache, const int32_t *tables,
                          int32_t max_blocks, const int32_t *cu_q, const int32_t *seq_lens, int32_t num_seqs,
                          int32_t total_q, int32_t max_q_len, int32_t num_q_heads, float scale, int32_t causal,
                          int32_t window, void *out, int32_t out_dtype, int32_t *err_word, cudaStream_t stream) {
    PKV_CHECK_ARG(aligned16(q) && (q_stride * 2) % 16 == 0, PKV_ERR_INVALID_ARG,
                  "pkv_attn_varlen: q and its row stride must be 16-byte aligned for prefill chunks");
    TcParams p{};
    p.tables = tables;
    p.max_blocks = max_blocks;
    p.seq_lens = seq_lens;
    p.cu_q = cu_q;
    p.num_blocks = cache->num_blocks;
    p.block_size = cache->block_size;
    p.hkv = cache->num_kv_heads;
    p.group = num_q_heads / cache->num_kv_heads;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.out = out;
    p.out_f32 = out_dtype == PKV_F32;
    p.err = err_word;
    p.window = window > 0 ? window : 0;
    const int rows = 128 / p.group;
    p.q_tiles = (max_q_len + rows - 1) / rows;
    CUtensorMap mq, mk, mv;
    pkv_status st = encode_q_map(&mq, q, q_stride, total_q, num_q_heads, cache->head_dim, rows, cache->dtype);
    if (st != PKV_OK) return st;
    st = encode_pool_map(&mk, cache->k, cache);
    if (st != PKV_OK) return st;
    st = encode_pool_map(&mv, cache->v, cache);
    if (st != PKV_OK) return st;
    const bool bf = cache->dtype == PKV_BF16;
    if (cache->head_dim == 64)
        return bf ? launch_prefill_tc_t<64, __nv_bfloat16>(mq, mk, mv, p, num_seqs, stream)
                  : launch_prefill_tc_t<64, __half>(mq, mk, mv, p, num_seqs, stream);
    return bf ? launch_prefill_tc_t<128, __nv_bfloat16>(mq, mk, mv, p, num_seqs, stream)
              : launch_prefill_tc_t<128, __half>(mq, mk, mv, p, num_seqs, stream);
}

}  // namespace pkv
