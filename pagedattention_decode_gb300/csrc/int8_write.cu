// int8_write.cu -- quantised slot write for the int8 KV cache.
//
// "Building a paged inference engine from scratch, and measuring it honestly",
// section 02 (INT8 KV cache design): symmetric int8, one scale per block per
// KV head, no zero point; a write dequantises the block's existing entries
// with the stored scale, adds the new entries, recomputes the max-abs scale
// and requantises everything.  Applied once per call to each block the call
// writes: the rows below the lowest offset written are the block's earlier
// tokens.  Every decision that yields an integer is taken in IEEE binary32
// with correctly rounded division and no contraction, so the codes and scales
// match a plain binary32 implementation bit for bit.
//
// One CTA per slot_mapping entry; only the first entry of a run of consecutive
// entries in the same block does the work (the allocator emits a block's
// slots consecutively).  Its warps take (K or V, KV head) pairs; lanes walk
// head_dim.
#include "launch.h"
#include "ptx.cuh"

namespace pkv {

__device__ __forceinline__ int8_t quantize(float x, float scale) {
    if (scale == 0.f) return 0;
    float r = rintf(__fdiv_rn(x, scale));
    r = fminf(fmaxf(r, -127.f), 127.f);
    return (int8_t)(int)r;
}

// grid (slot_mapping entry, group of 8 (K or V, KV head) jobs); one warp per
// job, each lane owning 4 consecutive dims (one 32-bit word of codes).
template <typename T>
__global__ void __launch_bounds__(256) write_kv_int8_kernel(const T *__restrict__ k, const T *__restrict__ v,
                                                            int64_t stride, const int64_t *__restrict__ slots,
                                                            int32_t num_tokens, int8_t *kq, int8_t *vq, float *ks,
                                                            float *vs, int32_t num_blocks, int32_t bs, int32_t H,
                                                            int32_t D, int32_t *err) {
    __shared__ int32_t src[256];  // offset -> token of its last writer in this run, or -1
    __shared__ int32_t s_min, s_max;
    pdl_wait();
    pdl_trigger();
    const int64_t t = blockIdx.x;
    const int64_t nslots = (int64_t)num_blocks * bs;
    const int64_t slot = slots[t];
    if (slot < 0) return;
    if (slot >= nslots) {
        if (threadIdx.x == 0 && blockIdx.y == 0) set_err(err, PKV_DEVERR_SLOT);
        return;
    }
    const int64_t blk = slot / bs;
    if (t > 0) {
        const int64_t prev = slots[t - 1];
        if (prev >= 0 && prev < nslots && prev / bs == blk) return;  // not the first of its run
    }
    if (threadIdx.x == 0) {
        for (int o = 0; o < bs; ++o) src[o] = -1;
        int mn = bs, mx = -1;
        for (int64_t u = t; u < num_tokens; ++u) {
            const int64_t su = slots[u];
            if (su < 0 || su >= nslots || su / bs != blk) break;
            const int o = (int)(su % bs);
            src[o] = (int32_t)u;
            mn = min(mn, o);
            mx = max(mx, o);
        }
        s_min = mn;
        s_max = mx;
    }
    __syncthreads();
    const int job = blockIdx.y * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (job >= 2 * H) return;
    const int lane = threadIdx.x & 31;
    const int min_off = s_min, max_off = s_max;
    const int which = job / H, h = job % H;
    const T *x = which ? v : k;
    int8_t *pool = (which ? vq : kq) + (blk * bs * H + h) * (int64_t)D;
    float *sc = (which ? vs : ks) + blk * H + h;
    const float old = *sc;
    // the 4 values of row o at dims 4*d4 .. 4*d4+3, in binary32
    auto row4 = [&](int o, int d4, float (&f)[4]) {
        const int32_t s = src[o];
        if (s >= 0) {
            const T *xp = x + (int64_t)s * stride + (int64_t)h * D + 4 * d4;
            const uint2 raw = *reinterpret_cast<const uint2 *>(xp);
            const float2 a = unpack2<T>(raw.x), b = unpack2<T>(raw.y);
            f[0] = a.x;
            f[1] = a.y;
            f[2] = b.x;
            f[3] = b.y;
        } else if (o < min_off) {
            const char4 c = *reinterpret_cast<const char4 *>(pool + (int64_t)o * H * D + 4 * d4);
            f[0] = __fmul_rn((float)c.x, old);
            f[1] = __fmul_rn((float)c.y, old);
            f[2] = __fmul_rn((float)c.z, old);
            f[3] = __fmul_rn((float)c.w, old);
        } else {
            f[0] = f[1] = f[2] = f[3] = 0.f;
        }
    };
    if (max_off < 16 && D <= 128) {
        // up to 16 rows x 4 dims per lane held in registers: every load in flight at once
        float f[16][4];
#pragma unroll
        for (int o = 0; o < 16; ++o)
            if (o <= max_off && lane < D / 4) row4(o, lane, f[o]);
        float amax = 0.f;
#pragma unroll
        for (int o = 0; o < 16; ++o)
            if (o <= max_off && lane < D / 4)
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(f[o][0]), fabsf(f[o][1])), fmaxf(fabsf(f[o][2]), fabsf(f[o][3]))));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float scale = __fdiv_rn(amax, 127.f);
#pragma unroll
        for (int o = 0; o < 16; ++o)
            if (o <= max_off && lane < D / 4) {
                char4 c;
                c.x = quantize(f[o][0], scale);
                c.y = quantize(f[o][1], scale);
                c.z = quantize(f[o][2], scale);
                c.w = quantize(f[o][3], scale);
                *reinterpret_cast<char4 *>(pool + (int64_t)o * H * D + 4 * lane) = c;
            }
        __syncwarp();
        if (lane == 0) *sc = scale;
        return;
    }
    float amax = 0.f;
    for (int o = 0; o <= max_off; ++o)
        for (int d4 = lane; d4 < D / 4; d4 += 32) {
            float f[4];
            row4(o, d4, f);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3]))));
        }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float scale = __fdiv_rn(amax, 127.f);
    for (int o = 0; o <= max_off; ++o)
        for (int d4 = lane; d4 < D / 4; d4 += 32) {
            float f[4];
            row4(o, d4, f);  // read before this lane overwrites the same codes
            char4 c;
            c.x = quantize(f[0], scale);
            c.y = quantize(f[1], scale);
            c.z = quantize(f[2], scale);
            c.w = quantize(f[3], scale);
            *reinterpret_cast<char4 *>(pool + (int64_t)o * H * D + 4 * d4) = c;
        }
    __syncwarp();
    if (lane == 0) *sc = scale;
}

pkv_status check_cache_i8(const pkv_cache_i8 *c, const char *what) {
    PKV_CHECK_ARG(c, PKV_ERR_INVALID_ARG, "%s: cache descriptor is NULL", what);
    PKV_CHECK_ARG(c->k && c->v && c->k_scale && c->v_scale, PKV_ERR_INVALID_ARG, "%s: NULL pool or scale", what);
    PKV_CHECK_ARG(aligned16(c->k) && aligned16(c->v) && aligned16(c->k_scale) && aligned16(c->v_scale),
                  PKV_ERR_INVALID_ARG, "%s: pools and scales must be 16-byte aligned", what);
    PKV_CHECK_ARG(c->dtype == PKV_F16 || c->dtype == PKV_BF16, PKV_ERR_DTYPE, "%s: dtype must be F16 or BF16",
                  what);
    PKV_CHECK_ARG(c->num_blocks > 0 && c->block_size > 0 && c->num_kv_heads > 0 && c->head_dim > 0, PKV_ERR_SHAPE,
                  "%s: cache geometry must be positive", what);
    PKV_CHECK_ARG((int64_t)c->num_blocks * c->block_size < (int64_t)1 << 31, PKV_ERR_SHAPE,
                  "%s: num_blocks * block_size must be < 2^31", what);
    PKV_CHECK_ARG(c->block_size <= 256, PKV_ERR_UNSUPPORTED, "%s: block_size must be <= 256", what);
    return PKV_OK;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

pkv_status pkv_write_kv_int8(const void *k, const void *v, int64_t kv_token_stride, const int64_t *slot_mapping,
                             int32_t num_tokens, const pkv_cache_i8 *cache, int32_t *err_word, pkv_stream stream) {
    pkv_status st = check_cache_i8(cache, "pkv_write_kv_int8");
    if (st != PKV_OK) return st;
    PKV_CHECK_ARG(num_tokens >= 0, PKV_ERR_INVALID_ARG, "num_tokens %d < 0", num_tokens);
    if (num_tokens == 0) return ok();
    PKV_CHECK_ARG(k && v && slot_mapping, PKV_ERR_INVALID_ARG, "k, v and slot_mapping must be non-NULL");
    const int64_t row = (int64_t)cache->num_kv_heads * cache->head_dim;
    PKV_CHECK_ARG(kv_token_stride >= row, PKV_ERR_SHAPE, "kv_token_stride shorter than a row");
    PKV_CHECK_ARG(cache->head_dim % 4 == 0 && aligned16(k) && aligned16(v) && kv_token_stride % 4 == 0,
                  PKV_ERR_INVALID_ARG, "k/v rows must be 16-byte aligned, head_dim a multiple of 4");
    const dim3 grid((unsigned)num_tokens, (unsigned)((2 * cache->num_kv_heads + 7) / 8));
    st =
        cache->dtype == PKV_BF16
            ? launch_pdl(write_kv_int8_kernel<__nv_bfloat16>, grid, dim3(256), 0, stream,
                         static_cast<const __nv_bfloat16 *>(k), static_cast<const __nv_bfloat16 *>(v), kv_token_stride,
                         slot_mapping, num_tokens, cache->k, cache->v, cache->k_scale, cache->v_scale,
                         cache->num_blocks, cache->block_size, cache->num_kv_heads, cache->head_dim, err_word)
            : launch_pdl(write_kv_int8_kernel<__half>, grid, dim3(256), 0, stream, static_cast<const __half *>(k),
                         static_cast<const __half *>(v), kv_token_stride, slot_mapping, num_tokens, cache->k,
                         cache->v, cache->k_scale, cache->v_scale, cache->num_blocks, cache->block_size,
                         cache->num_kv_heads, cache->head_dim, err_word);
    return st == PKV_OK ? ok() : st;
}

}  // extern "C"
