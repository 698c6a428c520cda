// kvq_noalloc.cu -- decode attention for callers that cannot allocate device memory.
//
// kvq_decode_attention needs a caller-provided workspace for the partial results of its
// split context.  Some callers cannot provide one: code running where device allocation
// is not allowed (inside an allocator callback or a memory-pool hook, a plugin whose host
// forbids cudaMalloc, a region that must not synchronise the device as a cudaMalloc may).
// kvq_decode_attention_noalloc runs the same decode with its scratch in a fixed-size
// array that the library itself holds in device memory, so the caller passes only the
// cache, the queries and the output.
#include <cstdint>
#include <mutex>

#include "kvq_decode.cuh"
#include "kvq_internal.cuh"
#include "kvq_launch.h"

// The library's own decode scratch: KVQ_NOALLOC_SCRATCH_BYTES (16 MiB) of device memory,
// held by every GPU that loads the library until the process exits.  Its name in host
// code is not a device address: the kernel gets the address from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device (with
// that device current) and remembered.  Returns nullptr when the lookup fails.
void* scratch_address(int device) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[device] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[device] = p;
    }
    return g_scratch_ptr[device];
}

}  // namespace

extern "C" int kvq_decode_attention_noalloc(const kvq_config* cfg, const void* cache, int32_t layer,
                                            const void* q, float softmax_scale, float* out,
                                            kvq_stream_t stream) {
    if (!cfg || !cache || !q || !out) return KVQ_ERR_ARG;
    kvq::Layout lo;
    int rc = kvq::make_layout(cfg, cfg->max_tokens, &lo);
    if (rc != KVQ_OK) return rc;
    if (layer < 0 || layer >= lo.L) return KVQ_ERR_ARG;
    kvq::DecodePlan plan;
    rc = kvq::make_plan(lo, &plan);
    if (rc != KVQ_OK) return rc;
    if (plan.ws_total > static_cast<int64_t>(KVQ_NOALLOC_SCRATCH_BYTES)) return KVQ_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(cache) % 256 || reinterpret_cast<uintptr_t>(q) % 16 ||
        reinterpret_cast<uintptr_t>(out) % 16)
        return KVQ_ERR_ALIGN;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices) return KVQ_ERR_CUDA;
    uint8_t* ws = static_cast<uint8_t*>(scratch_address(device));
    if (!ws) return KVQ_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the scratch keeps the previous call's contents: only the status word must start at
    // zero (the partial results are always written before they are read)
    if (cudaMemsetAsync(ws, 0, 4, s) != cudaSuccess) return KVQ_ERR_CUDA;
    return kvq::launch_decode(lo, plan, static_cast<const uint8_t*>(cache), layer, q, softmax_scale, out, ws, s);
}
