// launch.cpp -- see launch.h.
#include "launch.h"

#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

namespace pkv {

pkv_status check_cache(const pkv_cache *c, const char *what) {
    PKV_CHECK_ARG(c, PKV_ERR_INVALID_ARG, "%s: cache descriptor is NULL", what);
    PKV_CHECK_ARG(c->k && c->v, PKV_ERR_INVALID_ARG, "%s: cache k/v pointer is NULL", what);
    PKV_CHECK_ARG(aligned16(c->k) && aligned16(c->v), PKV_ERR_INVALID_ARG,
                  "%s: cache pointers must be 16-byte aligned", what);
    PKV_CHECK_ARG(c->dtype == PKV_F16 || c->dtype == PKV_BF16, PKV_ERR_DTYPE,
                  "%s: cache dtype %d is not F16 or BF16", what, c->dtype);
    PKV_CHECK_ARG(c->num_blocks > 0 && c->block_size > 0 && c->num_kv_heads > 0 && c->head_dim > 0,
                  PKV_ERR_SHAPE, "%s: cache geometry must be positive (%d, %d, %d, %d)", what,
                  c->num_blocks, c->block_size, c->num_kv_heads, c->head_dim);
    PKV_CHECK_ARG((int64_t)c->num_blocks * c->block_size < (int64_t)1 << 31, PKV_ERR_SHAPE,
                  "%s: num_blocks * block_size must be < 2^31", what);
    PKV_CHECK_ARG(((int64_t)c->num_kv_heads * c->head_dim * 2) % 16 == 0, PKV_ERR_UNSUPPORTED,
                  "%s: a token row (num_kv_heads * head_dim * 2 bytes) must be a multiple of 16", what);
    return PKV_OK;
}

pkv_status check_attention_shapes(const pkv_cache *c, int32_t num_q_heads) {
    PKV_CHECK_ARG(num_q_heads > 0 && num_q_heads % c->num_kv_heads == 0, PKV_ERR_SHAPE,
                  "num_q_heads %d is not a multiple of num_kv_heads %d", num_q_heads, c->num_kv_heads);
    const int group = num_q_heads / c->num_kv_heads;
    PKV_CHECK_ARG(group == 1 || group == 2 || group == 4 || group == 8, PKV_ERR_UNSUPPORTED,
                  "query heads per KV head must be 1, 2, 4 or 8 (got %d)", group);
    PKV_CHECK_ARG(c->head_dim == 64 || c->head_dim == 128, PKV_ERR_UNSUPPORTED,
                  "head_dim must be 64 or 128 (got %d)", c->head_dim);
    PKV_CHECK_ARG(c->block_size % 16 == 0 && c->block_size <= 256, PKV_ERR_UNSUPPORTED,
                  "block_size must be a multiple of 16 up to 256 (got %d)", c->block_size);
    return PKV_OK;
}

pkv_status sm_count(int32_t device, int *count) {
    static std::atomic<int> cached[64] = {};
    int dev = device;
    if (dev < 0) PKV_CUDA_TRY(cudaGetDevice(&dev));
    if (dev >= 0 && dev < 64 && cached[dev].load(std::memory_order_relaxed) > 0) {
        *count = cached[dev].load(std::memory_order_relaxed);
        return PKV_OK;
    }
    PKV_CUDA_TRY(cudaDeviceGetAttribute(count, cudaDevAttrMultiProcessorCount, dev));
    if (dev >= 0 && dev < 64) cached[dev].store(*count, std::memory_order_relaxed);
    return PKV_OK;
}

pkv_status set_smem_once(const void *kernel, int bytes, std::atomic<uint64_t> *done) {
    int dev = 0;
    PKV_CUDA_TRY(cudaGetDevice(&dev));
    const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
    if (bit && (done->load(std::memory_order_acquire) & bit)) return PKV_OK;
    PKV_CUDA_TRY(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
    if (bit) done->fetch_or(bit, std::memory_order_acq_rel);
    return PKV_OK;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

pkv_status encode_pool_map(CUtensorMap *map, void *base, const pkv_cache *c, int rows) {
    auto fn = encode_fn();
    PKV_CHECK_ARG(fn, PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    PKV_CHECK_ARG(rows == 16 || rows == 32 || rows == 64 || rows == 128, PKV_ERR_INVALID_ARG, "pool box of %d rows", rows);
    const int tiles = c->num_kv_heads * c->head_dim / 64;
    cuuint64_t dims[3] = {64, (cuuint64_t)tiles, (cuuint64_t)c->num_blocks * c->block_size};
    cuuint64_t strides[2] = {128, (cuuint64_t)c->num_kv_heads * c->head_dim * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, c->dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    PKV_CHECK_ARG(r == CUDA_SUCCESS, PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PKV_OK;
}

// The pool seen as [head chunks][token rows][64 elements] (innermost last): a
// box of 16 token rows x `chunks` consecutive 128-byte chunks (one KV head's
// half of head_dim each) is one TMA copy that lands chunk by chunk, each as
// 16 swizzled 128-byte lines in a 2 KB tile of its own -- the layout the
// decode consumers read with ldmatrix.  The chunk stride (128 bytes) is
// smaller than the row stride: the dimensions are listed in the order the
// box is laid out in shared memory, not by stride.
pkv_status encode_pool_rows_map(CUtensorMap *map, void *base, const pkv_cache *c, int chunks) {
    auto fn = encode_fn();
    PKV_CHECK_ARG(fn, PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const int tiles = c->num_kv_heads * c->head_dim / 64;
    PKV_CHECK_ARG(chunks >= 1 && chunks <= tiles && chunks <= 256, PKV_ERR_INVALID_ARG, "pool box of %d chunks",
                  chunks);
    cuuint64_t dims[3] = {64, (cuuint64_t)c->num_blocks * c->block_size, (cuuint64_t)tiles};
    cuuint64_t strides[2] = {(cuuint64_t)c->num_kv_heads * c->head_dim * 2, 128};
    cuuint32_t box[3] = {64, 16, (cuuint32_t)chunks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, c->dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    PKV_CHECK_ARG(r == CUDA_SUCCESS, PKV_ERR_CUDA, "cuTensorMapEncodeTiled (pool rows) failed (%d)", (int)r);
    return PKV_OK;
}

// The int8 pool the same way: chunks are whole KV heads (128 codes).
pkv_status encode_pool_rows_map_i8(CUtensorMap *map, void *base, const pkv_cache_i8 *c, int heads) {
    auto fn = encode_fn();
    PKV_CHECK_ARG(fn, PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    PKV_CHECK_ARG(heads >= 1 && heads <= c->num_kv_heads, PKV_ERR_INVALID_ARG, "int8 pool box of %d heads", heads);
    cuuint64_t dims[3] = {(cuuint64_t)c->head_dim, (cuuint64_t)c->num_blocks * c->block_size,
                          (cuuint64_t)c->num_kv_heads};
    cuuint64_t strides[2] = {(cuuint64_t)c->num_kv_heads * c->head_dim, (cuuint64_t)c->head_dim};
    cuuint32_t box[3] = {128, 16, (cuuint32_t)heads};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    PKV_CHECK_ARG(r == CUDA_SUCCESS, PKV_ERR_CUDA, "cuTensorMapEncodeTiled (int8 pool rows) failed (%d)", (int)r);
    return PKV_OK;
}

// Packed output rows [total_q][Hq][D] seen as [heads][rows][D] (innermost
// last): a box of `cols` elements (64 bytes) x `rows` consecutive rows x
// `heads` consecutive heads is the part of a q tile one warp holds, staged
// in shared memory with the 64-byte swizzle.  The head stride is smaller than
// the row stride: the dimensions follow the order the box has in shared
// memory.
pkv_status encode_out_map(CUtensorMap *map, void *out, int total_q, int hq, int d, int out_dtype, int cols, int rows,
                          int heads) {
    auto fn = encode_fn();
    PKV_CHECK_ARG(fn, PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const int esz = out_dtype == PKV_F32 ? 4 : 2;
    PKV_CHECK_ARG(cols * esz == 64 && rows >= 1 && rows <= 256 && heads >= 1 && heads <= hq, PKV_ERR_INVALID_ARG,
                  "output box %d x %d x %d", cols, rows, heads);
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)total_q, (cuuint64_t)hq};
    cuuint64_t strides[2] = {(cuuint64_t)hq * d * esz, (cuuint64_t)d * esz};
    cuuint32_t box[3] = {(cuuint32_t)cols, (cuuint32_t)rows, (cuuint32_t)heads};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt = out_dtype == PKV_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : out_dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = fn(map, dt, 3, out, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    PKV_CHECK_ARG(r == CUDA_SUCCESS, PKV_ERR_CUDA, "cuTensorMapEncodeTiled (output rows) failed (%d)", (int)r);
    return PKV_OK;
}

pkv_status encode_q_map(CUtensorMap *map, const void *q, int64_t q_stride, int total_q, int hq, int d, int rows,
                        int dtype) {
    auto fn = encode_fn();
    PKV_CHECK_ARG(fn, PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[3] = {64, (cuuint64_t)hq * d / 64, (cuuint64_t)total_q};
    cuuint64_t strides[2] = {128, (cuuint64_t)q_stride * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                    const_cast<void *>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    PKV_CHECK_ARG(r == CUDA_SUCCESS, PKV_ERR_CUDA, "cuTensorMapEncodeTiled (q) failed (%d)", (int)r);
    return PKV_OK;
}

}  // namespace pkv
