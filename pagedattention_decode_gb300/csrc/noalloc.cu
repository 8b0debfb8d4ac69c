// noalloc.cu -- decode attention for callers that cannot allocate device memory.
//
// pkv_attn_decode needs a caller-provided workspace for its split-K records.
// Some callers have no way to provide one: a C or C++ host program that embeds
// libpkv inside a process whose device memory belongs to another runtime's
// caching allocator (and so has no allocator handle of its own), or a latency-
// critical loop that must not call cudaMalloc because it synchronises the
// device and takes an unbounded time.  For them this file keeps the scratch in
// a fixed array that is part of the library's own device image.
//
// The array is created on a device when the library's module is loaded there
// and stays until the process exits, on every device that loads the library.
// All calls share it: the kernels write every byte they later read, so nothing
// is cleared between calls, and two calls that run on the GPU at the same time
// (on different streams, or from different host threads) race on it.
#include <cuda.h>

#include <mutex>

#include "launch.h"

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

// The scratch itself.  In host code this name is only a stand-in for the
// symbol, never a device address: the address is looked up per device below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 256;
std::mutex g_scratch_mu;
// Per device: the address found for the context that was current then, and
// that context's process-unique id.  cudaDeviceReset (or any teardown of the
// primary context) loads the module again, possibly at another address, in a
// context with a new id, so the next call looks the address up again.
struct ScratchEntry {
    unsigned long long ctx_id;
    void *ptr;
};
ScratchEntry g_scratch[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Id of the current context, or 0 (and a lookup on every call) when the
// driver does not offer it.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;
}
}  // namespace

// Device address of the scratch array on `device`, which must be current.
// Set-up: the first call on a device (and the first after the device's
// context was re-created) looks it up with cudaGetSymbolAddress and keeps it.
static pkv_status scratch_address(int device, void **out) {
    PKV_CHECK_ARG(device >= 0 && device < kMaxDevices, PKV_ERR_UNSUPPORTED, "device ordinal %d", device);
    // cudaGetDevice already made the device's primary context current
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> g(g_scratch_mu);
    ScratchEntry &e = g_scratch[device];
    if (e.ptr == nullptr || id == 0 || e.ctx_id != id) {
        void *p = nullptr;
        cudaError_t r = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        PKV_CHECK_ARG(r == cudaSuccess && p != nullptr, PKV_ERR_CUDA,
                      "cudaGetSymbolAddress of the no-allocation scratch on device %d: %s", device,
                      cudaGetErrorString(r));
        e.ptr = p;
        e.ctx_id = id;
    }
    *out = e.ptr;
    return PKV_OK;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

pkv_status pkv_attn_decode_noalloc(const void *q, int64_t q_token_stride, const pkv_cache *cache,
                                   const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                   int32_t num_seqs, int32_t num_q_heads, float scale, void *out, int32_t out_dtype,
                                   int32_t *err_word, pkv_stream stream) {
    pkv_status st = check_attention_common(q, q_token_stride, cache, block_tables, max_blocks_per_seq, seq_lens,
                                           num_seqs, num_q_heads, out, out_dtype, "pkv_attn_decode_noalloc");
    if (st != PKV_OK) return st;
    if (num_seqs == 0) return ok();
    size_t need = 0;
    st = decode_workspace_size(num_seqs, num_q_heads, cache->num_kv_heads, cache->head_dim, -1, &need);
    if (st != PKV_OK) return st;
    PKV_CHECK_ARG(need <= (size_t)PKV_NOALLOC_SCRATCH_BYTES, PKV_ERR_WORKSPACE,
                  "pkv_attn_decode_noalloc: this call needs %zu bytes of scratch but the fixed array holds %d; "
                  "use pkv_attn_decode with a workspace for it",
                  need, PKV_NOALLOC_SCRATCH_BYTES);
    int dev = 0;
    PKV_CUDA_TRY(cudaGetDevice(&dev));
    void *ws = nullptr;
    st = scratch_address(dev, &ws);
    if (st != PKV_OK) return st;
    st = run_decode(q, q_token_stride, cache, block_tables, max_blocks_per_seq, seq_lens, nullptr, num_seqs,
                    num_q_heads, scale, out, out_dtype, ws, (size_t)PKV_NOALLOC_SCRATCH_BYTES, err_word, stream);
    return st == PKV_OK ? ok() : st;
}

}  // extern "C"
