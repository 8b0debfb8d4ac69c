// prefill_tc.cu -- a8, prefill chunks (q_len > 1) on the 5th-generation tensor
// cores: tcgen05.mma with accumulators in tensor memory (TMEM).
//
// "Building a paged inference engine from scratch, and measuring it honestly",
// sections 02-03: a packed step holds prefill chunks whose keys are read
// through the block table, and query row i of a chunk with q_len rows and
// kv_len keys sees keys t <= kv_len - q_len + i.  For a chunk the work is a
// dense contraction, so it runs here as a FlashAttention-style loop on UMMA:
//
//  * A q tile = 128 M rows: the G query heads of one KV head x 128/G query
//    positions (row r -> head r / (128/G), position q0 + r % (128/G)).  A work
//    item is two consecutive tiles, so every K/V tile staged in shared memory
//    serves 256 rows.
//  * Persistent: one CTA per SM walks its items (c, c + grid, ...; numbered
//    sequence by sequence, a sequence's pairs of tiles from the last to the
//    first, KV head fastest).  Warp 0 finds them in cu_seqlens_q, hands each
//    to the other warps through a two-slot ring in shared memory, and streams
//    Q of both tiles, then 128-token K and V tiles of the KV head (TMA
//    through the block table, 128-byte swizzle, boxes of the largest of 128,
//    64, 32 or 16 rows that divides block_size: L2 -> shared throughput grows
//    with the box) into separate K and V rings.  Barrier phases run on across
//    items, so the next item's loads and first scores overlap the current
//    item's tail.
//  * Warp 1 issues the MMAs (the whole warp walks the loop, an elected lane
//    issues): S = Q K^T (M 128, N 128, K 16 steps, both operands K-major
//    from shared memory) into the tile's TMEM score columns, and O += P V
//    (A = P read from TMEM, B = V as an MN-major shared operand, N =
//    head_dim) into its TMEM accumulator.  Per step it issues P V of tile 0,
//    the next scores of tile 0, P V of tile 1, the next scores of tile 1:
//    while one tile's softmax runs, the tensor pipe works on the other tile.
//    Completion is signalled with tcgen05.commit.
//  * Warps 4-7 (tile 0) and 8-11 (tile 1), one TMEM lane = one M row per
//    thread, read the 128 scores of their row with a single wait for the
//    TMEM loads, apply the causal and window limits, keep the
//    running max and sum in registers, and write P back over the scores as
//    16-bit values (bf16: a hi + lo pair, ~16 significant bits).  The running
//    max comes from the row's first tile with a visible key and is moved only
//    when a step's p could pass 2^15 (their sum tells, so no per-step max is
//    taken): then that row of O is rescaled in TMEM and P written again.  The
//    final O row is divided by the sum and leaves by TMA tensor stores from a
//    shared-memory staging slot (rows of a ragged last tile: plain stores).
// All 512 TMEM columns (per tile: S/P 128, O head_dim) and ~217 KB of shared
// memory; setmaxnreg moves registers from the producer / MMA warpgroup
// (warps 0-3) to the two softmax warpgroups.
#include <cuda.h>

#include <cstring>

#include "launch.h"
#include "ptx.cuh"

namespace pkv {

namespace {

constexpr int kTok = 128;         // keys per step: the N of the score MMA
constexpr int kTiles = 2;         // q tiles of 128 M rows per CTA; every K/V stage serves both
constexpr int kTmemCols = 512;    // 256 columns per tile: scores / P at +0 (128), O at +128 (D)
constexpr float kPSumMax = 32768.f;  // a step's sum of p above this moves the running max

template <typename T>
struct IsBf16 {
    static constexpr bool value = false;
};
template <>
struct IsBf16<__nv_bfloat16> {
    static constexpr bool value = true;
};

struct TcParams {
    const void *q;
    int64_t q_stride;  // elements between query rows
    const int32_t *tables;
    int32_t max_blocks;
    const int32_t *seq_lens;
    const int32_t *cu_q;
    int32_t num_blocks, block_size, hkv, group, causal;
    float scale_log2;
    void *out;
    int32_t out_f32;
    int32_t *err;
    int32_t q_tiles;  // most pairs of q tiles in a sequence (kTiles * 128 / group positions each)
    int32_t window;   // > 0: each row attends only its most recent `window` keys
    int32_t box_rows; // rows per K/V TMA box: 128, 64, 32 or 16, a divisor of block_size
    int32_t num_seqs;
    int32_t out_tma;  // the output map is valid: whole warps' rows leave by TMA stores
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

// The MMA and commit wrappers are executed by a whole, converged warp: the
// warp computes the (uniform) operands and one lane elected inside the
// instruction sequence issues it.  Issuing from a single-lane branch instead
// costs more per MMA than the MMA itself takes on the tensor pipe.
__device__ __forceinline__ void umma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

// Arrives once on `bar` when every MMA issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
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

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]));
}

// max(a, b, c) in one instruction (three-input form of max.f32 on sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Non-blocking test of an mbarrier phase.  A phase that has completed is
// seen at a fraction of the cost of the suspending wait, so every wait of
// this kernel tests first and suspends only when the phase is still open.
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, volatile int *abort) {
    return mbar_test(bar, parity) || mbar_wait(bar, parity, abort);
}

__device__ __forceinline__ void st_shared_f4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
    return v;
}

// Tensor store of a shared-memory box (64-byte swizzle) into the output rows,
// tracked in this thread's bulk group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// This thread's earlier bulk stores have read their shared memory ...
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... or have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void st_shared_u4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

}  // namespace

template <int D>
__host__ __device__ constexpr int prefill_stages() {  // stages of the K ring and of the V ring
    return D == 64 ? 4 : 2;
}

// Registers per thread after the warpgroups re-balance them: the producer /
// MMA warpgroup gives registers back, the two softmax warpgroups (a whole
// row of 128 fp32 scores each per thread) take them.  Their sum must fit the
// launch's registers (kThreads x the kernel's count, 168 x 384): checked on
// the host.  ptxas, head_dim 128 fp16, with each role's code compiled alone:
// at 88 / 208 the producer and MMA warps fit without spills and the softmax
// warps spill 72 bytes (loads) in their step loop; at 72 / 216 the producer
// and MMA warps spill 96 bytes and the softmax 28 more.  88 / 208 took the
// mixed step's prefill chunks from 1,075 to 1,121 TFLOP/s (A/B on one box).
constexpr int kThreads = 384;
constexpr int kRegsLow = 88;
constexpr int kRegsHigh = 208;
constexpr int kRegsAtLaunchMin = (128 * kRegsLow + 256 * kRegsHigh + kThreads - 1) / kThreads;
// Epilogue staging: each softmax warp passes 16 columns of its 32 O rows
// through shared memory (row stride 20 floats: conflict-free 16-byte
// accesses), so the global stores cover 8 rows x 64 contiguous bytes per
// instruction instead of 32 rows x 16 bytes.
constexpr int kStageStride = 20;
constexpr int kStageBytes = 2 * 4 * 32 * kStageStride * 4;

// A work item: the pair of q tiles `pair` (2 x 128 M rows) of KV head `kvh`
// of the prefill chunk of sequence `s`.  The producer warp finds a CTA's
// items and hands them to the other warps through a two-slot ring in shared
// memory; nt0 < 0 marks the end.
struct TcItem {
    int s, kvh, q_begin, q_len, kv_len, q00, j_first, nt0, nt1;
};

template <int D, typename T>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo,
                      const TcParams p) {
    constexpr int HALVES = D / 64;
    constexpr int S = prefill_stages<D>();
    constexpr int QHALF = 128 * 128;            // bytes of 128 rows x 64 dims
    constexpr int QTILE = HALVES * QHALF;
    constexpr int KVHALF = kTok * 128;           // bytes of 128 tokens x 64 dims
    constexpr int KVSTAGE = HALVES * KVHALF;     // one K (or V) tile
    constexpr bool BF = IsBf16<T>::value;
    // P enters P V as a 16-bit operand.  fp16 keeps 11 significant bits of each
    // p in [0, 2^15] (relative error <= 2^-12, far inside the 2e-3 gate); bf16
    // keeps only 8, so there P is split into hi + lo halves and P V takes two
    // MMAs per K step.  P of keys 32c .. 32c + 31 lies in TMEM columns
    // 16c .. 16c + 15 (fp16), or hi in 32c .. 32c + 15 and lo in 32c + 16 ..
    // 32c + 31 (bf16): columns whose scores have already been read.
    constexpr bool LO = BF;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bars[2 + 4 * S + 3 * kTiles + 4 + 1];
    __shared__ TcItem s_item[2];
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sq = base;
    uint8_t *sk = base + kTiles * QTILE;
    uint8_t *sv = sk + S * KVSTAGE;
    float *stage_o = reinterpret_cast<float *>(sv + S * KVSTAGE + 4096);
    uint64_t *q_full = &bars[0];
    uint64_t *q_empty = &bars[1];  // every score MMA of an item has read its Q
    uint64_t *k_full = &bars[2];
    uint64_t *k_empty = &bars[2 + S];
    uint64_t *v_full = &bars[2 + 2 * S];
    uint64_t *v_empty = &bars[2 + 3 * S];
    uint64_t *tile_bars = &bars[2 + 4 * S];  // per tile: s_full, p_full, o_done
    uint64_t *item_full = &bars[2 + 4 * S + 3 * kTiles];
    uint64_t *item_empty = item_full + 2;
    uint64_t *fin = item_full + 4;  // abort path: completion of every MMA issued
    auto s_full = [&](int u) { return tile_bars + u * 3; };
    auto p_full = [&](int u) { return tile_bars + u * 3 + 1; };
    auto o_done = [&](int u) { return tile_bars + u * 3 + 2; };

    pdl_wait();  // the previous kernel on the stream (e.g. the slot write) is complete
    pdl_trigger();
    const int G = p.group;
    const int R = 128 / G;  // query positions per tile
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        s_abort = 0;
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int i = 0; i < S; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int u = 0; u < kTiles; ++u) {
            mbar_init(s_full(u), 1);
            mbar_init(p_full(u), 128);
            mbar_init(o_done(u), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&item_full[i], 1);
            mbar_init(&item_empty[i], 1 + 2 * 4);  // the MMA warp and the eight softmax warps
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
    // steps of tile u in an item, and the step count that both tiles walk
    auto tile_steps = [&](const TcItem &it, int u) -> int {
        const int q0 = it.q00 + u * R;
        if (q0 >= it.q_len) return 0;
        const int last_row = min(it.q_len, q0 + R) - 1;
        const int kv_hi = p.causal ? it.kv_len - it.q_len + last_row + 1 : it.kv_len;
        return (kv_hi + kTok - 1) / kTok - it.j_first;
    };
    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
    if (warp == 0) {
        // ===== producer: finds the items, then Q of both tiles and the K and V tiles of each =====
        const uint64_t pol_q = policy_evict_first();
        const uint64_t pol_kv = policy_evict_last();  // re-read by the other q tiles of the chunk
        if (lane == 0) {
            prefetch_tensormap(&tmq);
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
        }
        const int box = p.box_rows;
        const int32_t *tables = p.tables;
        // Items are numbered sequence by sequence, within a sequence from its
        // last pair of q tiles (the most keys) to its first, KV head fastest;
        // CTA c takes items c, c + gridDim.x, ...  The cursor (s_cur, base)
        // only moves forward: base is the number of the first item of
        // sequence s_cur.
        int s_cur = 0;
        long long base_item = 0;
        long long idx = blockIdx.x;
        int it = 0;           // items published
        int gs = 0;           // K / V steps started (ring position)
        int issued_k = 0, issued_v = 0, q_issued = 0;  // loads issued
        bool ok = true;
        while (ok) {
            TcItem item;
            item.nt0 = -1;
            bool found = false;
            while (s_cur < p.num_seqs) {
                const int sl = s_cur + lane;
                int qb = 0, ql = 0, cnt = 0;
                if (sl < p.num_seqs) {
                    qb = p.cu_q[sl];
                    ql = p.cu_q[sl + 1] - qb;
                    if (ql > 1) cnt = ((ql + kTiles * R - 1) / (kTiles * R)) * p.hkv;
                }
                int inc = cnt;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int t = __shfl_up_sync(0xffffffffu, inc, off);
                    if (lane >= off) inc += t;
                }
                const unsigned hit = __ballot_sync(0xffffffffu, cnt > 0 && idx < base_item + inc);
                if (hit) {
                    const int L = __ffs(hit) - 1;
                    const int cntL = __shfl_sync(0xffffffffu, cnt, L);
                    base_item += __shfl_sync(0xffffffffu, inc, L) - cntL;
                    s_cur += L;
                    item.s = s_cur;
                    item.q_begin = __shfl_sync(0xffffffffu, qb, L);
                    item.q_len = __shfl_sync(0xffffffffu, ql, L);
                    const int r = (int)(idx - base_item);
                    const int npairs = cntL / p.hkv;
                    item.kvh = r % p.hkv;
                    const int pair = npairs - 1 - r / p.hkv;
                    item.q00 = pair * kTiles * R;
                    found = true;
                    break;
                }
                base_item += __shfl_sync(0xffffffffu, inc, 31);
                s_cur += 32;
            }
            if (found) {
                item.kv_len = p.seq_lens[item.s];
                if (item.q_len > item.kv_len || (int64_t)item.kv_len > (int64_t)p.max_blocks * p.block_size) {
                    // flagged once, by the item of the sequence's last pair and KV head 0
                    if (lane == 0 && item.kvh == 0 && item.q00 + kTiles * R >= item.q_len)
                        set_err(p.err, PKV_DEVERR_LENGTH);
                    idx += gridDim.x;
                    continue;
                }
                // the window's first key is lowest for the first row of tile 0,
                // so both tiles walk from j_first
                const int lim_first = p.causal ? item.kv_len - item.q_len + item.q00 : item.kv_len - 1;
                const int lo_first =
                    (p.window > 0 && lim_first - p.window + 1 > 0) ? lim_first - p.window + 1 : 0;
                item.j_first = lo_first / kTok;
                item.nt0 = tile_steps(item, 0);
                item.nt1 = tile_steps(item, 1);
            }
            // publish the item (or the end mark)
            if (lane == 0) {
                ok = mbar_wait(&item_empty[it & 1], ((it >> 1) & 1) ^ 1, &s_abort);
                if (ok) {
                    s_item[it & 1] = item;
                    mbar_arrive(&item_full[it & 1]);
                }
            }
            ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
            ++it;
            if (!ok || !found) break;
            idx += gridDim.x;
            const int nt = max(item.nt0, item.nt1);
            // Q of both tiles, once the previous item's score MMAs have read theirs
            const int ntiles = item.nt1 > 0 ? 2 : 1;
            if (lane == 0 && q_issued > 0) ok = mbar_wait(q_empty, (q_issued - 1) & 1, &s_abort);
            if (!__shfl_sync(0xffffffffu, (int)ok, 0)) {
                ok = false;
                break;
            }
            if (lane == 0) mbar_arrive_expect_tx(q_full, (uint32_t)(ntiles * G * HALVES * R * 128));
            __syncwarp();
            for (int t = lane; t < ntiles * G * HALVES; t += 32) {
                const int u = t / (G * HALVES), g = (t / HALVES) % G, half = t % HALVES;
                tma_load_3d(sq + u * QTILE + half * QHALF + g * R * 128, &tmq, q_full, 0,
                            (item.kvh * G + g) * HALVES + half, item.q_begin + item.q00 + u * R, pol_q);
            }
            ++q_issued;
            // K and V tiles: a tile has at most (128 / 16) * HALVES <= 16 boxes:
            // lane t issues box t of K and of V (sub-block t / HALVES, half t %
            // HALVES).  Its block-table entry is read one step ahead.
            const int32_t *trow = tables + (int64_t)item.s * p.max_blocks;
            auto boxes_of = [&](int j) {
                const int nvalid = min(kTok, item.kv_len - (item.j_first + j) * kTok);
                return ((nvalid + box - 1) / box) * HALVES;
            };
            auto lookup = [&](int j) -> int {
                if (j >= nt || lane >= boxes_of(j)) return 0;
                const int tok = (item.j_first + j) * kTok + (lane / HALVES) * box;
                return trow[tok / p.block_size];
            };
            int phys_next = lookup(0);
            for (int j = 0; j < nt; ++j, ++gs) {
                const int stage = gs % S;
                int phys = phys_next;
                phys_next = lookup(j + 1);
                const int nbox = boxes_of(j);
                const int t0 = (item.j_first + j) * kTok;
                int row = 0;
                if (lane < nbox) {
                    const int tok = t0 + (lane / HALVES) * box;  // box | block_size: a box never leaves its block
                    const int lb = tok / p.block_size;
                    if (phys < 0 || phys >= p.num_blocks) {
                        set_err(p.err, PKV_DEVERR_BLOCK);
                        phys = 0;
                    }
                    row = phys * p.block_size + (tok - lb * p.block_size);
                }
                const uint32_t dst_off =
                    (uint32_t)(stage * KVSTAGE + (lane % HALVES) * KVHALF + (lane / HALVES) * box * 128);
                int okw = 1;
                if (lane == 0) okw = wait_phase(&k_empty[stage], ((gs / S) & 1) ^ 1, &s_abort);
                if (!__shfl_sync(0xffffffffu, okw, 0)) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(&k_full[stage], (uint32_t)(nbox * box * 128));
                __syncwarp();
                if (lane < nbox)
                    tma_load_3d(sk + dst_off, &tmk, &k_full[stage], 0, item.kvh * HALVES + lane % HALVES, row, pol_kv);
                ++issued_k;
                if (lane == 0) okw = wait_phase(&v_empty[stage], ((gs / S) & 1) ^ 1, &s_abort);
                if (!__shfl_sync(0xffffffffu, okw, 0)) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(&v_full[stage], (uint32_t)(nbox * box * 128));
                __syncwarp();
                if (lane < nbox)
                    tma_load_3d(sv + dst_off, &tmv, &v_full[stage], 0, item.kvh * HALVES + lane % HALVES, row, pol_kv);
                ++issued_v;
            }
        }
        if (!ok && lane == 0) {
            // gave up: the loads this warp issued must land before the CTA exits
            s_abort = 1;
            set_err(p.err, PKV_DEVERR_TIMEOUT);
            volatile int never = 0;
            if (q_issued > 0) mbar_wait(q_full, (q_issued - 1) & 1, &never);
            for (int k = issued_k > S ? issued_k - S : 0; k < issued_k; ++k)
                mbar_wait(&k_full[k % S], (k / S) & 1, &never);
            for (int k = issued_v > S ? issued_v - S : 0; k < issued_v; ++k)
                mbar_wait(&v_full[k % S], (k / S) & 1, &never);
        }
    } else if (warp == 1) {
        // ===== MMA issuer: the whole warp walks the loop, one elected lane issues =====
        // every lane waits on the same phase; the vote keeps the warp converged
        auto wait = [&](uint64_t *bar, uint32_t parity) {
            return __all_sync(0xffffffffu, wait_phase(bar, parity, &s_abort));
        };
        const uint32_t idS = idesc_f16(BF ? 1 : 0, 0, 128, kTok);
        const uint32_t idPV = idesc_f16(BF ? 1 : 0, 1, 128, D);
        const uint32_t sq_a = smem_u32(sq), sk_a = smem_u32(sk), sv_a = smem_u32(sv);
        // g: ring position of the K / V step
        auto issue_s = [&](int u, int g) {
            const uint32_t kst = sk_a + (g % S) * KVSTAGE;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int half = kk >> 2, koff = (kk & 3) * 32;
                const uint64_t ad = sw128_desc(sq_a + u * QTILE + half * QHALF + koff, 16, 1024);
                const uint64_t bd = sw128_desc(kst + half * KVHALF + koff, 16, 1024);
                umma_ss(tmem + u * 256, ad, bd, idS, kk > 0 ? 1u : 0u);
            }
            umma_commit(s_full(u));
        };
        auto issue_pv = [&](int u, int g, bool first) {
            const uint32_t vst = sv_a + (g % S) * KVSTAGE;
            const uint32_t ts = tmem + u * 256, to = tmem + u * 256 + 128;
#pragma unroll
            for (int kk = 0; kk < kTok / 16; ++kk) {
                const uint64_t vd = sw128_desc(vst + kk * 2048, KVHALF, 1024);
                const uint32_t col = LO ? (kk >> 1) * 32 + (kk & 1) * 8 : kk * 8;
                umma_ts(to, ts + col, vd, idPV, (!first || kk > 0) ? 1u : 0u);
                if (LO) umma_ts(to, ts + col + 16, vd, idPV, 1u);
            }
            umma_commit(o_done(u));
        };
        int gc = 0;              // ring position of the current item's first step
        int tb[kTiles] = {0, 0}; // steps of each tile in earlier items
        bool ok = true;
        for (int it = 0; ok; ++it) {
            ok = wait(&item_full[it & 1], (it >> 1) & 1);
            if (!ok) break;
            const TcItem item = s_item[it & 1];
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[it & 1]);
            if (item.nt0 < 0) break;
            const int nt0 = item.nt0, nt1 = item.nt1, nt = max(nt0, nt1);
            auto steps_of = [&](int u) { return u ? nt1 : nt0; };
            // V rows past kv_len (only in the last step) are cleared by the first
            // tile whose P V reads that step
            const int zt = nt0 == nt ? 0 : 1;
            ok = wait(q_full, it & 1) && wait(&k_full[gc % S], (gc / S) & 1);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int u = 0; u < kTiles; ++u) {
                if (!ok || steps_of(u) == 0) continue;
                // the scores overwrite the tile's last P of the previous item
                if (tb[u] > 0) {
                    ok = wait(o_done(u), (tb[u] - 1) & 1);
                    if (!ok) continue;
                    tc_fence_after();
                }
                issue_s(u, gc);
            }
            if (!ok) break;
            umma_commit(&k_empty[gc % S]);
            if (nt == 1) umma_commit(q_empty);  // every score MMA of the item issued
            for (int j = 0; j < nt && ok; ++j) {
                const int g = gc + j;
                const int j1 = j + 1;
                const bool last_partial = (item.j_first + j1) * kTok > item.kv_len;
                // V of the step is tested before P (it has mostly landed long before):
                // once P arrives, only its own wait stands before the P V issue
                ok = wait(&v_full[g % S], (g / S) & 1);
                bool k_ready = false;
#pragma unroll
                for (int u = 0; u < kTiles; ++u) {
                    if (!ok || j >= steps_of(u)) continue;
                    const uint32_t ph = (uint32_t)(tb[u] + j) & 1;
                    ok = wait(p_full(u), ph);
                    // the last step's V rows past kv_len are cleared by tile zt
                    if (ok && u != zt && last_partial) ok = wait(p_full(zt), (uint32_t)(tb[zt] + j) & 1);
                    if (!ok) continue;
                    tc_fence_after();
                    issue_pv(u, g, j == 0);
                    // every P V that reads the stage's V issued: its release is committed
                    // here, in the shadow of the next wait
                    if (u == kTiles - 1 || j >= nt1) umma_commit(&v_empty[g % S]);
                    if (j1 < steps_of(u)) {
                        if (!k_ready) ok = k_ready = wait(&k_full[(g + 1) % S], ((g + 1) / S) & 1);
                        // the scores overwrite P of step j: its P V must have completed
                        if (ok) ok = wait(o_done(u), ph);
                        if (!ok) continue;
                        tc_fence_after();
                        issue_s(u, g + 1);
                    }
                }
                if (!ok) break;
                if (k_ready) umma_commit(&k_empty[(g + 1) % S]);
                if (j1 == nt - 1) umma_commit(q_empty);  // every score MMA of the item issued
            }
            tb[0] += nt0;
            tb[1] += nt1;
            gc += nt;
        }
        if (!ok && lane == 0) {
            s_abort = 1;
            set_err(p.err, PKV_DEVERR_TIMEOUT);
        }
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
        // ===== softmax + epilogue: warps 4-7 tile 0, warps 8-11 tile 1, one M row per thread =====
        const int u = (warp - 4) >> 2;
        const int qw = warp & 3;  // a warp reaches TMEM lanes 32 * (warp % 4) .. + 31
        const int row = qw * 32 + lane;
        const uint32_t trow_addr = tmem + ((uint32_t)(qw * 32) << 16) + u * 256;
        const float sl = p.scale_log2;
        int tbu = 0;  // steps of this tile in earlier items
        int gcs = 0;  // ring position of the current item's first step
        bool ok = true;
        for (int it = 0; ok; ++it) {
            ok = __all_sync(0xffffffffu, wait_phase(&item_full[it & 1], (it >> 1) & 1, &s_abort));
            if (!ok) break;
            // the item is read from shared memory where it is used (few values
            // stay live across the steps) and released after the epilogue
            const volatile TcItem &item = s_item[it & 1];
            const int nt0 = item.nt0, nt1 = item.nt1;
            if (nt0 < 0) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&item_empty[it & 1]);
                break;
            }
            const int nt = max(nt0, nt1);
            const int ntu = u ? nt1 : nt0;
            const int j_first = item.j_first;
            int lim, lo;
            bool valid;
            {
                const int kv_len = item.kv_len, q_len = item.q_len;
                const int qi = item.q00 + u * R + row % R;
                valid = qi < q_len;
                lim = (p.causal && valid) ? kv_len - q_len + qi : kv_len - 1;
                lo = (p.window > 0 && lim - p.window + 1 > 0) ? lim - p.window + 1 : 0;
            }
            // the step whose V rows past kv_len this tile clears (the item's last
            // step, when it is partial and this tile is the first to read it), or -1
            const int zt = nt0 == nt ? 0 : 1;
            const int jzero = (u == zt && (j_first + nt) * kTok > item.kv_len) ? nt - 1 : -1;
            float m_used = -INFINITY, lsum = 0.f;
            for (int j = 0; j < ntu; ++j) {
                const int gpos = gcs + j;
                // warp-uniform outcome: the tcgen05 ld/st below are warp-collective
                if (!__all_sync(0xffffffffu, wait_phase(s_full(u), (tbu + j) & 1, &s_abort))) {
                    ok = false;
                    break;
                }
                // the scores of step j were issued after P V of step j - 1 completed,
                // so O is settled here and may be rescaled
                tc_fence_after();
                const int t0 = (j_first + j) * kTok;
                // every row of the warp sees every key of the tile: no masking
                const bool whole = __all_sync(0xffffffffu, t0 + kTok - 1 <= lim && t0 >= lo);
                // the row's 128 scores, read with one wait (each wait exposes the
                // whole TMEM load latency)
                uint32_t sr[kTok];
#pragma unroll
                for (int c0 = 0; c0 < kTok; c0 += 32)
                    tmem_ld32(trow_addr + c0, *reinterpret_cast<uint32_t(*)[32]>(&sr[c0]));
                tmem_wait_ld();
                if (!whole) {
                    // keys t0 + c with c > lim - t0 (causal limit) or c < lo - t0
                    // (window start) are invisible; the start only matters on
                    // steps that begin before it
                    const int hi_c = lim - t0, lo_c = lo - t0;
#pragma unroll
                    for (int c = 0; c < kTok; ++c)
                        if (c > hi_c) sr[c] = __float_as_uint(-INFINITY);
                    if (__any_sync(0xffffffffu, lo_c > 0)) {
#pragma unroll
                        for (int c = 0; c < kTok; ++c)
                            if (c < lo_c) sr[c] = __float_as_uint(-INFINITY);
                    }
                }
                // the row max of the raw scores times the scale (positive): eight
                // independent chains of three-input maxima
                auto row_max = [&]() -> float {
                    float pm[8];
    #pragma unroll
                    for (int v = 0; v < 8; ++v) pm[v] = fmaxf(__uint_as_float(sr[v]), __uint_as_float(sr[8 + v]));
    #pragma unroll
                    for (int c = 16; c < kTok; c += 16)
    #pragma unroll
                        for (int v = 0; v < 8; ++v)
                            pm[v] = fmax3(pm[v], __uint_as_float(sr[c + v]), __uint_as_float(sr[c + 8 + v]));
                    return fmaxf(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], fmax3(pm[5], pm[6], pm[7]))) * sl;
                };
                // The running max m_used is taken from the row's first tile with
                // a visible key and is moved only when p would leave the range
                // where it is exact enough and finite as a 16-bit value: every p of
                // a step is at most the step's sum, so a sum <= 2^15 proves all p
                // <= 2^15.  Otherwise (or on inf / NaN) the row takes the exact
                // max, O and the row sum are rescaled, and P is written again (a
                // second pass of the loop below).
                const bool fresh = m_used == -INFINITY;
                if (__any_sync(0xffffffffu, fresh) && fresh) m_used = row_max();
                float step_sum;
    #pragma unroll 1
                for (int pass = 0;; ++pass) {
                    // p = 2^(s * scale - m_used), written back over the scores as
                    // 16-bit values (the scale and shift, and the row sum, as packed
                    // fp32 pairs).  While a row has met no key yet (a window can
                    // start past whole tiles) every score and m_used are -inf: the
                    // shift is then taken as -inf too, so every p is 0, not NaN.
                    const float neg_m = m_used == -INFINITY ? -INFINITY : -m_used;
                    const float2 sl2 = make_float2(sl, sl), nm2 = make_float2(neg_m, neg_m);
                    float2 ps[4];
    #pragma unroll
                    for (int v = 0; v < 4; ++v) ps[v] = make_float2(0.f, 0.f);
    #pragma unroll
                    for (int c0 = 0; c0 < kTok; c0 += 32) {
                        uint32_t ph[16], pl[16];
    #pragma unroll
                        for (int c = 0; c < 32; c += 2) {
                            const float2 x = __ffma2_rn(
                                make_float2(__uint_as_float(sr[c0 + c]), __uint_as_float(sr[c0 + c + 1])), sl2, nm2);
                            const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
                            ps[(c >> 1) & 3] = __fadd2_rn(ps[(c >> 1) & 3], make_float2(p0, p1));
                            const uint32_t h = pack2<T>(p0, p1);
                            ph[c / 2] = h;
                            if (LO) {
                                const float2 hf = unpack2<T>(h);
                                pl[c / 2] = pack2<T>(p0 - hf.x, p1 - hf.y);
                            }
                        }
                        if (LO) {
                            tmem_st16(trow_addr + c0, ph);
                            tmem_st16(trow_addr + c0 + 16, pl);
                        } else {
                            tmem_st16(trow_addr + c0 / 2, ph);
                        }
                    }
                    const float2 ps01 = __fadd2_rn(ps[0], ps[1]), ps23 = __fadd2_rn(ps[2], ps[3]);
                    const float2 ps4 = __fadd2_rn(ps01, ps23);
                    step_sum = ps4.x + ps4.y;
                    const bool over = pass == 0 && !(step_sum <= kPSumMax);
                    if (!__any_sync(0xffffffffu, over)) break;
                    tmem_wait_st();
                    float alpha = 1.f;
                    if (over) {
                        const float m_new = fmaxf(m_used, row_max());
                        alpha = fast_exp2(m_used - m_new);
                        lsum *= alpha;
                        m_used = m_new;
                    }
                    if (j > 0) {
    #pragma unroll
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t orr[32];
                            tmem_ld32(trow_addr + 128 + c0, orr);
                            tmem_wait_ld();
    #pragma unroll
                            for (int c = 0; c < 32; ++c) orr[c] = __float_as_uint(__uint_as_float(orr[c]) * alpha);
                            tmem_st32(trow_addr + 128 + c0, orr);
                        }
                    }
                }
                lsum += step_sum;
                // V rows past kv_len in the last tile hold stale or unrelated data:
                // zero them, once the tile's TMA load (which may cover some of
                // them) has landed
                if (j == jzero) {
                    if (!wait_phase(&v_full[gpos % S], (gpos / S) & 1, &s_abort)) {
                        s_abort = 1;
                        set_err(p.err, PKV_DEVERR_TIMEOUT);
                    }
                    if (row >= item.kv_len - t0) {
    #pragma unroll
                        for (int half = 0; half < HALVES; ++half) {
                            uint4 *dst = reinterpret_cast<uint4 *>(sv + (gpos % S) * KVSTAGE + half * KVHALF + row * 128);
    #pragma unroll
                            for (int c = 0; c < 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(p_full(u));
            }
            if (!ok) break;
            if (ntu > 0) {
                ok = __all_sync(0xffffffffu, wait_phase(o_done(u), (tbu + ntu - 1) & 1, &s_abort));
                if (!ok) break;
                tc_fence_after();
                const float inv = 1.f / lsum;
                const int64_t hq = (int64_t)p.hkv * G;
                // shared-window address: the staging accesses are issued as
                // shared-memory instructions, not generic ones
                const uint32_t stg = smem_u32(stage_o) + (uint32_t)((warp - 4) * 32 * kStageStride * 4);
                // The warp's 32 rows are min(32, R) consecutive positions of 32 / min(32, R)
                // consecutive heads.  When all of them lie inside the chunk they leave by
                // tensor stores: 64 bytes of each row at a time into the warp's staging
                // rows (a 64-byte-swizzled box, 512-byte aligned: chunk k of row r at
                // k ^ ((r >> 1) & 3), conflict-free), then one store issued by one lane
                // while the warp goes on.  The epilogue had been ~9k cycles of every
                // item's critical path (clock trace).
                const int q_first = item.q00 + u * R;
                const int wp0 = (qw * 32) % R, wpos = R < 32 ? R : 32;
                if (p.out_tma && q_first + wp0 + wpos <= item.q_len) {
                    const int pos0 = item.q_begin + q_first + wp0, head0 = item.kvh * G + (qw * 32) / R;
                    const uint32_t myrow = stg + (uint32_t)lane * 64u;
                    const uint32_t sw = (uint32_t)(lane >> 1) & 3u;
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t orr[32];
                        tmem_ld32(trow_addr + 128 + c0, orr);
                        tmem_wait_ld();
                        if (p.out_f32) {
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                if (lane == 0) bulk_wait_read();  // the previous store has read the rows
                                __syncwarp();
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    const int c = h * 16 + k * 4;
                                    st_shared_f4(myrow + (((uint32_t)k ^ sw) << 4), __uint_as_float(orr[c]) * inv,
                                                 __uint_as_float(orr[c + 1]) * inv, __uint_as_float(orr[c + 2]) * inv,
                                                 __uint_as_float(orr[c + 3]) * inv);
                                }
                                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                                __syncwarp();
                                if (lane == 0) tma_store_3d(&tmo, stg, c0 + h * 16, pos0, head0);
                            }
                        } else {
                            if (lane == 0) bulk_wait_read();
                            __syncwarp();
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const int c = k * 8;
                                st_shared_u4(myrow + (((uint32_t)k ^ sw) << 4),
                                             pack2<T>(__uint_as_float(orr[c]) * inv, __uint_as_float(orr[c + 1]) * inv),
                                             pack2<T>(__uint_as_float(orr[c + 2]) * inv, __uint_as_float(orr[c + 3]) * inv),
                                             pack2<T>(__uint_as_float(orr[c + 4]) * inv, __uint_as_float(orr[c + 5]) * inv),
                                             pack2<T>(__uint_as_float(orr[c + 6]) * inv, __uint_as_float(orr[c + 7]) * inv));
                            }
                            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                            __syncwarp();
                            if (lane == 0) tma_store_3d(&tmo, stg, c0, pos0, head0);
                        }
                    }
                } else {
                if (lane == 0) bulk_wait_read();  // the rows may still be read by an earlier tensor store
                __syncwarp();
                const int rr = lane >> 2, c4 = lane & 3;
                // the output rows this lane stores: rows k * 8 + rr of the warp
                int64_t row_off[4];
                bool row_ok[4];
                {
                    const int q_len = item.q_len, q_first = item.q00 + u * R, q_row0 = item.q_begin + q_first;
                    const int64_t head0 = (int64_t)item.kvh * G;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int rw = qw * 32 + k * 8 + rr;  // M row of the tile
                        const int pos = rw % R;
                        row_ok[k] = q_first + pos < q_len;
                        row_off[k] = ((int64_t)(q_row0 + pos) * hq + head0 + rw / R) * D + c4 * 4;
                    }
                }
                // a loop, not unrolled: the epilogue runs once per item, and its
                // code has to come into the instruction cache each time
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t orr[32];
                    tmem_ld32(trow_addr + 128 + c0, orr);
                    tmem_wait_ld();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        // this thread's row, 16 columns, into the staging rows
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const int c = h * 16 + q4 * 4;
                            st_shared_f4(stg + (uint32_t)((lane * kStageStride + q4 * 4) * 4),
                                         __uint_as_float(orr[c]) * inv, __uint_as_float(orr[c + 1]) * inv,
                                         __uint_as_float(orr[c + 2]) * inv, __uint_as_float(orr[c + 3]) * inv);
                        }
                        __syncwarp();
                        // rows k * 8 + rr of the warp, 4 columns per lane: 8 rows x 16 columns per store
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int r = k * 8 + rr;
                            const float4 v = ld_shared_f4(stg + (uint32_t)((r * kStageStride + c4 * 4) * 4));
                            if (row_ok[k]) {
                                const int64_t off = row_off[k] + c0 + h * 16;
                                if (p.out_f32)
                                    *reinterpret_cast<float4 *>(static_cast<float *>(p.out) + off) = v;
                                else
                                    *reinterpret_cast<uint2 *>(static_cast<T *>(p.out) + off) =
                                        make_uint2(pack2<T>(v.x, v.y), pack2<T>(v.z, v.w));
                            }
                        }
                        __syncwarp();
                    }
                }
                }
                // O of this tile has been read: the next item's first P V (which
                // overwrites O) waits for this warp's next arrival on p_full
                tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[it & 1]);
            tbu += ntu;
            gcs += nt;
        }
        if (!ok && lane == 0) {
            s_abort = 1;
            set_err(p.err, PKV_DEVERR_TIMEOUT);
        }
        // the output rows this warp handed to tensor stores are written before the CTA leaves
        if (lane == 0) bulk_wait_all();
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    if (warp == 1 && __all_sync(0xffffffffu, s_abort != 0)) {
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
                                      const CUtensorMap &mo, const TcParams &p, int num_seqs, cudaStream_t stream) {
    constexpr int HALVES = D / 64;
    // Q of both tiles + the K and V rings, + 1 KB for the 1024-byte alignment
    // of the swizzled tiles, + 4 KB of slack after the last stage, + the
    // epilogue staging rows
    const int smem = kTiles * HALVES * 128 * 128 + 2 * prefill_stages<D>() * HALVES * kTok * 128 + 1024 + 4096 +
                     kStageBytes;
    auto kern = prefill_tc_kernel<D, T>;
    static std::atomic<uint64_t> smem_set{0};
    pkv_status st = set_smem_once(reinterpret_cast<const void *>(kern), smem, &smem_set);
    if (st != PKV_OK) return st;
    // persistent: one CTA per SM (fewer if there cannot be that many items)
    int sms = 0;
    st = sm_count(-1, &sms);
    if (st != PKV_OK) return st;
    const int64_t most_items = (int64_t)p.q_tiles * num_seqs * p.hkv;
    dim3 grid((unsigned)(most_items < sms ? most_items : sms));
    // the register re-balancing inside the kernel needs at least
    // kRegsAtLaunchMin registers per thread at launch, or it would wait forever
    static std::atomic<int> regs{0};
    if (regs.load() == 0) {
        cudaFuncAttributes fa{};
        PKV_CUDA_TRY(cudaFuncGetAttributes(&fa, reinterpret_cast<const void *>(kern)));
        regs.store(fa.numRegs);
    }
    PKV_CHECK_ARG(regs.load() >= kRegsAtLaunchMin, PKV_ERR_UNSUPPORTED,
                  "prefill kernel built with %d registers per thread, needs >= %d", regs.load(), kRegsAtLaunchMin);
    return launch_pdl(kern, grid, dim3(kThreads), (size_t)smem, stream, mq, mk, mv, mo, p);
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
    p.q_tiles = (max_q_len + kTiles * rows - 1) / (kTiles * rows);
    p.num_seqs = num_seqs;
    p.box_rows = cache->block_size % 128 == 0  ? 128
                 : cache->block_size % 64 == 0 ? 64
                 : cache->block_size % 32 == 0 ? 32
                                               : 16;
    p.q = q;
    p.q_stride = q_stride;
    CUtensorMap mq, mk, mv;
    pkv_status st = encode_q_map(&mq, q, q_stride, total_q, num_q_heads, cache->head_dim, rows, cache->dtype);
    if (st != PKV_OK) return st;
    st = encode_pool_map(&mk, cache->k, cache, p.box_rows);
    if (st != PKV_OK) return st;
    st = encode_pool_map(&mv, cache->v, cache, p.box_rows);
    if (st != PKV_OK) return st;
    // output rows by tensor stores: a warp's 32 rows are min(32, 128 / G) positions of
    // 32 / min(32, 128 / G) heads (the output must be 16-byte aligned; out is contiguous)
    CUtensorMap mo;
    memset(&mo, 0, sizeof(mo));
    const int wrows = rows < 32 ? rows : 32;
    p.out_tma = 0;
    if (aligned16(out)) {
        st = encode_out_map(&mo, out, total_q, num_q_heads, cache->head_dim, out_dtype, out_dtype == PKV_F32 ? 16 : 32,
                            wrows, 32 / wrows);
        if (st != PKV_OK) return st;
        p.out_tma = 1;
    }
    const bool bf = cache->dtype == PKV_BF16;
    if (cache->head_dim == 64)
        return bf ? launch_prefill_tc_t<64, __nv_bfloat16>(mq, mk, mv, mo, p, num_seqs, stream)
                  : launch_prefill_tc_t<64, __half>(mq, mk, mv, mo, p, num_seqs, stream);
    return bf ? launch_prefill_tc_t<128, __nv_bfloat16>(mq, mk, mv, mo, p, num_seqs, stream)
              : launch_prefill_tc_t<128, __half>(mq, mk, mv, mo, p, num_seqs, stream);
}

}  // namespace pkv
