// launch.h -- host-side helpers shared by the .cu files of libpkv: argument
// validation, the device's SM count, and TMA tensor-map encoding for the pools.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <utility>

#include "internal.h"

namespace pkv {

inline int dtype_bytes(int32_t dt) { return dt == PKV_F32 ? 4 : (dt == PKV_F16 || dt == PKV_BF16) ? 2 : 0; }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

#define PKV_CUDA_TRY(expr)                                                              \
    do {                                                                                \
        cudaError_t e_ = (expr);                                                        \
        if (e_ != cudaSuccess)                                                          \
            return pkv::fail(PKV_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_));     \
    } while (0)

// Launches `kernel` as a programmatic dependent of the work before it on the
// stream: its CTAs may be scheduled while the previous kernel finishes.  Every
// kernel of this library begins with griddepcontrol.wait (pdl_wait) before it
// touches global memory, which waits for the whole previous grid and its
// memory operations, so this is safe after any kernel, ours or the caller's.
template <typename... KArgs, typename... Args>
pkv_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                      Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    PKV_CUDA_TRY(cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...));
    return PKV_OK;
}

// Checks a pool descriptor: pointers, geometry, type.
pkv_status check_cache(const pkv_cache *c, const char *what);
// Shapes compiled for the attention kernels.
pkv_status check_attention_shapes(const pkv_cache *c, int32_t num_q_heads);
// SM count of `device` (-1: current device), cached per device.
pkv_status sm_count(int32_t device, int *count);

// Sets a kernel's max dynamic shared memory once per device (the attribute
// persists for the process); `done` is that kernel's per-device flag set.
pkv_status set_smem_once(const void *kernel, int bytes, std::atomic<uint64_t> *done);

// 3-D tensor map over a pool seen as [rows = num_blocks * block_size]
// x [num_kv_heads * head_dim / 64 tiles of 64 elements] x [64 elements], box
// = `rows` (16, 32, 64 or 128) rows x 1 tile x 64 elements, 128-byte swizzle
// (a 2 to 16 KB shared tile).
pkv_status encode_pool_map(CUtensorMap *map, void *base, const pkv_cache *c, int rows = 16);

// The same for an int8 pool with head_dim 128: box = 16 rows x 1 head x 128
// codes (one 2 KB shared tile per KV head per 16 tokens).
// [chunks][rows][64] views: one box = 16 token rows x `chunks` 128-byte chunks
pkv_status encode_pool_rows_map(CUtensorMap *map, void *base, const pkv_cache *c, int chunks);
// [heads][rows][D] view of packed output rows: one box = 64 bytes x rows x heads
pkv_status encode_out_map(CUtensorMap *map, void *out, int total_q, int hq, int d, int out_dtype, int cols, int rows,
                          int heads);
pkv_status encode_pool_rows_map_i8(CUtensorMap *map, void *base, const pkv_cache_i8 *c, int heads);

// 3-D tensor map over packed query rows [total_q][Hq * D / 64][64] (row
// stride q_stride elements), box = `rows` rows x 1 x 64 elements, 128-byte
// swizzle: one head-half of `rows` consecutive query rows per load.
pkv_status encode_q_map(CUtensorMap *map, const void *q, int64_t q_stride, int total_q, int hq, int d, int rows,
                        int dtype);

}  // namespace pkv
