// write_copy.cu -- a2 slot write and a10 block copy: plain HBM-bound byte moves.
//
// Slot write ("How to Implement Paged Attention in PyTorch and vLLM",
// PagedKVCache.append_token): the K/V row of a new token goes to row `slot` of
// the pool viewed as [num_blocks * block_size, kv_heads * head_dim].  One warp
// moves one token's K and V rows with 16-byte loads and stores.
//
// Block copy ("Build a paged KV cache manager from scratch", copy-on-write):
// block dst of every layer's K and V becomes a copy of block src.  A CTA
// copies one 16 KB chunk of one block of one layer for one pair.
#include "launch.h"
#include "ptx.cuh"

namespace pkv {

__global__ void write_kv_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v, int64_t src_stride16,
                                const int64_t *__restrict__ slots, int32_t num_tokens, uint4 *__restrict__ kc,
                                uint4 *__restrict__ vc, int64_t num_slots, int32_t row16, int32_t *err) {
    pdl_wait();
    pdl_trigger();
    const int warps = blockDim.x >> 5;
    const int64_t t = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= num_tokens) return;
    const int64_t slot = slots[t];
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (lane == 0) set_err(err, PKV_DEVERR_SLOT);
        return;
    }
    const uint4 *ks = k + t * src_stride16;
    const uint4 *vs = v + t * src_stride16;
    uint4 *kd = kc + slot * row16;
    uint4 *vd = vc + slot * row16;
    for (int i = lane; i < row16; i += 32) {
        uint4 a = __ldg(ks + i);
        uint4 b = __ldg(vs + i);
        kd[i] = a;
        vd[i] = b;
    }
}

constexpr int kMaxLayersPerLaunch = 32;
struct LayerPtrs {
    uint4 *k[kMaxLayersPerLaunch];
    uint4 *v[kMaxLayersPerLaunch];
};

// grid: x = chunk of the block (16 KB each), y = pair, z = layer
__global__ void copy_blocks_kernel(LayerPtrs layers, const int64_t *__restrict__ pairs, int32_t num_blocks,
                                   int64_t block16, int32_t chunk16, int32_t *err) {
    pdl_wait();
    pdl_trigger();
    const int64_t src = pairs[2 * (int64_t)blockIdx.y];
    const int64_t dst = pairs[2 * (int64_t)blockIdx.y + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.z == 0) set_err(err, PKV_DEVERR_PAIR);
        return;
    }
    const int64_t begin = (int64_t)blockIdx.x * chunk16;
    const int64_t end = (begin + chunk16 < block16 ? begin + chunk16 : block16);
    const uint4 *ks = layers.k[blockIdx.z] + src * block16;
    const uint4 *vs = layers.v[blockIdx.z] + src * block16;
    uint4 *kd = layers.k[blockIdx.z] + dst * block16;
    uint4 *vd = layers.v[blockIdx.z] + dst * block16;
    for (int64_t i = begin + threadIdx.x; i < end; i += blockDim.x) {
        uint4 a = ks[i];
        uint4 b = vs[i];
        kd[i] = a;
        vd[i] = b;
    }
}

}  // namespace pkv

using namespace pkv;

extern "C" {

pkv_status pkv_write_kv(const void *k, const void *v, int64_t kv_token_stride, const int64_t *slot_mapping,
                        int32_t num_tokens, const pkv_cache *cache, int32_t *err_word, pkv_stream stream) {
    pkv_status st = check_cache(cache, "pkv_write_kv");
    if (st != PKV_OK) return st;
    PKV_CHECK_ARG(num_tokens >= 0, PKV_ERR_INVALID_ARG, "num_tokens %d < 0", num_tokens);
    if (num_tokens == 0) return ok();
    PKV_CHECK_ARG(k && v && slot_mapping, PKV_ERR_INVALID_ARG, "k, v and slot_mapping must be non-NULL");
    const int64_t row = (int64_t)cache->num_kv_heads * cache->head_dim;
    PKV_CHECK_ARG(kv_token_stride >= row, PKV_ERR_SHAPE, "kv_token_stride %lld < row of %lld elements",
                  (long long)kv_token_stride, (long long)row);
    PKV_CHECK_ARG(aligned16(k) && aligned16(v) && (kv_token_stride * 2) % 16 == 0, PKV_ERR_INVALID_ARG,
                  "k/v rows must start on 16-byte boundaries");
    const int warps = 8;
    dim3 grid((unsigned)((num_tokens + warps - 1) / warps));
    st = launch_pdl(
        write_kv_kernel, grid, dim3(warps * 32), 0, stream, static_cast<const uint4 *>(k),
        static_cast<const uint4 *>(v), (int64_t)(kv_token_stride * 2 / 16), slot_mapping, num_tokens,
        static_cast<uint4 *>(cache->k), static_cast<uint4 *>(cache->v), (int64_t)cache->num_blocks * cache->block_size,
        (int32_t)(row * 2 / 16), err_word);
    return st == PKV_OK ? ok() : st;
}

pkv_status pkv_copy_blocks(const pkv_cache *caches, int32_t num_layers, const int64_t *src_dst_pairs,
                           int32_t num_pairs, int32_t *err_word, pkv_stream stream) {
    PKV_CHECK_ARG(num_layers >= 0 && num_pairs >= 0, PKV_ERR_INVALID_ARG, "negative count");
    if (num_layers == 0 || num_pairs == 0) return ok();
    PKV_CHECK_ARG(caches && src_dst_pairs, PKV_ERR_INVALID_ARG, "caches and src_dst_pairs must be non-NULL");
    PKV_CHECK_ARG(num_pairs <= 65535, PKV_ERR_UNSUPPORTED, "at most 65535 pairs per call (got %d)", num_pairs);
    for (int32_t l = 0; l < num_layers; ++l) {
        pkv_status st = check_cache(&caches[l], "pkv_copy_blocks");
        if (st != PKV_OK) return st;
        PKV_CHECK_ARG(caches[l].num_blocks == caches[0].num_blocks && caches[l].block_size == caches[0].block_size &&
                          caches[l].num_kv_heads == caches[0].num_kv_heads &&
                          caches[l].head_dim == caches[0].head_dim && caches[l].dtype == caches[0].dtype,
                      PKV_ERR_SHAPE, "layer %d has a different pool geometry than layer 0", l);
    }
    const int64_t block16 = (int64_t)caches[0].block_size * caches[0].num_kv_heads * caches[0].head_dim * 2 / 16;
    const int32_t chunk16 = 1024;  // 16 KB per CTA
    const unsigned chunks = (unsigned)((block16 + chunk16 - 1) / chunk16);
    for (int32_t l0 = 0; l0 < num_layers; l0 += kMaxLayersPerLaunch) {
        const int n = num_layers - l0 < kMaxLayersPerLaunch ? num_layers - l0 : kMaxLayersPerLaunch;
        LayerPtrs lp{};
        for (int i = 0; i < n; ++i) {
            lp.k[i] = static_cast<uint4 *>(caches[l0 + i].k);
            lp.v[i] = static_cast<uint4 *>(caches[l0 + i].v);
        }
        dim3 grid(chunks, (unsigned)num_pairs, (unsigned)n);
        const pkv_status st = launch_pdl(copy_blocks_kernel, grid, dim3(256), 0, stream, lp, src_dst_pairs,
                                         caches[0].num_blocks, block16, chunk16, err_word);
        if (st != PKV_OK) return st;
    }
    return ok();
}

}  // extern "C"
