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

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) {
    return __half2float(x);
}
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}

__device__ __forceinline__ int8_t quantize(float x, float scale) {
    if (scale == 0.f) return 0;
    float r = rintf(__fdiv_rn(x, scale));
    r = fminf(fmaxf(r, -127.f), 127.f);
    return (int8_t)(int)r;
}

template <typename T>
__global__ void __launch_bounds__(128) write_kv_int8_kernel(const T *__restrict__ k, const T *__restrict__ v,
                                                            int64_t stride, const int64_t *__restrict__ slots,
                                                            int32_t num_tokens, int8_t *kq, int8_t *vq, float *ks,
                                                            float *vs, int32_t num_blocks, int32_t bs, int32_t H,
                                                            int32_t D, int32_t *err) {
    __shared__ int32_t src[256];  // offset -> token of its last writer in this run, or -1
    __shared__ int32_t s_min, s_max;
    const int64_t t = blockIdx.x;
    const int64_t nslots = (int64_t)num_blocks * bs;
    const int64_t slot = slots[t];
    if (slot < 0) return;
    if (slot >= nslots) {
        if (threadIdx.x == 0) set_err(err, PKV_DEVERR_SLOT);
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
    const int min_off = s_min, max_off = s_max;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int job = warp; job < 2 * H; job += nw) {
        const int which = job / H, h = job % H;
        const T *x = which ? v : k;
        int8_t *pool = (which ? vq : kq) + (blk * bs * H + h) * (int64_t)D;
        float *sc = (which ? vs : ks) + blk * H + h;
        const float old = *sc;
        auto value = [&](int o, int d) -> float {
            const int32_t s = src[o];
            if (s >= 0) return to_f32<T>(x[(int64_t)s * stride + (int64_t)h * D + d]);
            if (o < min_off) return __fmul_rn((float)pool[(int64_t)o * H * D + d], old);
            return 0.f;
        };
        float amax = 0.f;
        for (int o = 0; o <= max_off; ++o)
            for (int d = lane; d < D; d += 32) amax = fmaxf(amax, fabsf(value(o, d)));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float scale = __fdiv_rn(amax, 127.f);
        for (int o = 0; o <= max_off; ++o)
            for (int d = lane; d < D; d += 32) {
                const float val = value(o, d);  // read before this lane overwrites the same code
                pool[(int64_t)o * H * D + d] = quantize(val, scale);
            }
        __syncwarp();
        if (lane == 0) *sc = scale;
    }
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
    if (cache->dtype == PKV_BF16)
        write_kv_int8_kernel<__nv_bfloat16><<<num_tokens, 128, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(k), static_cast<const __nv_bfloat16 *>(v), kv_token_stride,
            slot_mapping, num_tokens, cache->k, cache->v, cache->k_scale, cache->v_scale, cache->num_blocks,
            cache->block_size, cache->num_kv_heads, cache->head_dim, err_word);
    else
        write_kv_int8_kernel<__half><<<num_tokens, 128, 0, stream>>>(
            static_cast<const __half *>(k), static_cast<const __half *>(v), kv_token_stride, slot_mapping, num_tokens,
            cache->k, cache->v, cache->k_scale, cache->v_scale, cache->num_blocks, cache->block_size,
            cache->num_kv_heads, cache->head_dim, err_word);
    PKV_CUDA_TRY(cudaGetLastError());
    return ok();
}

}  // extern "C"
