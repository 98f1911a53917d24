// dattn_decode_noalloc: the fused decode with its scratch memory in a fixed device array.
//
// dattn_decode needs a caller-provided workspace: per-head counters plus fp32 partial
// triples for heads that are split across CTAs. Some callers cannot provide one. Code that
// runs inside another program's allocator regime (a plugin or custom op handed only input
// and output pointers, or a framework whose caching allocator owns all device memory) must
// not call cudaMalloc. Latency-critical code cannot afford cudaMalloc either, because it may
// synchronise the device. This entry point lets such callers decode without any allocation.
// The scratch lives in a file-scope __device__ array that every GPU loading this library
// holds until the process exits.
//
// Limits and behaviour:
//  - The array holds kStaticScratchBytes (8 MiB). A problem that needs more workspace than
//    that is rejected with DATTN_ERR_WORKSPACE before anything is launched. The size needed
//    is dattn_workspace_size(B, Hq, Hkv, head_dim, 0, num_splits).
//  - The first call on a device looks up the array's device address on that device
//    (cudaGetSymbolAddress, with the device current) and caches it. Make that first call
//    before any stream capture on the device, because the lookup may load the module.
//  - Every call on a device shares the one array, which keeps the last call's contents.
//    Each call clears the counter region on its stream before the kernel runs. Calls that
//    overlap on the GPU (different streams, no ordering between them) race on the array and
//    give wrong results.
//  - Nothing here calls cudaMalloc, cudaFree or any allocating library routine.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dattn {
namespace {

constexpr size_t kStaticScratchBytes = 8u << 20;

// Device code could name this array directly. Host code must not: on the host the name
// refers to a host-side stand-in, not a device address. Use the address from
// cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDev] = {};

// Device address of the scratch array on the current device, looked up once per device.
dattn_status_t scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return DATTN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDev) return DATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
            return DATTN_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return DATTN_OK;
}

}  // namespace
}  // namespace dattn

extern "C" dattn_status_t dattn_decode_noalloc(const dattn_kv_layout* layout,
                                               const void* k_pool,
                                               const void* v_pool, const dattn_bf16* q,
                                               int32_t B, int32_t Hq, float scale,
                                               const int32_t* seq_lens,
                                               const dattn_sparse* sparse, int32_t num_splits,
                                               float* out, float* m_g, float* e_g,
                                               int32_t* dev_err, void* stream) {
    using namespace dattn;
    if (layout == nullptr) return DATTN_ERR_INVALID_ARG;
    const size_t need = dattn_workspace_size(B, Hq, layout->num_kv_heads, layout->head_dim, 0,
                                             num_splits);
    if (need == 0)  // invalid shape: let the full validation name the error, with no launch
        return dattn_decode(layout, k_pool, v_pool, q, B, Hq, scale, seq_lens, sparse,
                            num_splits, nullptr, 0, out, m_g, e_g, dev_err, stream);
    if (need > kStaticScratchBytes) return DATTN_ERR_WORKSPACE;
    void* scratch = nullptr;
    dattn_status_t st = scratch_address(&scratch);
    if (st != DATTN_OK) return st;
    // the per-head counters must start at zero; the rest is written before it is read
    const size_t counters = attn_counter_bytes(B * layout->num_kv_heads);
    if (counters > 0 &&
        cudaMemsetAsync(scratch, 0, counters, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return DATTN_ERR_CUDA;
    return dattn_decode(layout, k_pool, v_pool, q, B, Hq, scale, seq_lens, sparse, num_splits,
                        scratch, kStaticScratchBytes, out, m_g, e_g, dev_err, stream);
}
