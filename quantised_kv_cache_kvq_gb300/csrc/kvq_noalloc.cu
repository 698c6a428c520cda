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

#include <cuda.h>

#include "kvq_decode.cuh"
#include "kvq_internal.cuh"
#include "kvq_launch.h"

// The library's own decode scratch: KVQ_NOALLOC_SCRATCH_BYTES (16 MiB) of device memory,
// held by every GPU that loads the library until the process exits.  Its name in host
// code is not a device address: the kernel gets the address from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

// The scratch's device address is a property of the module loaded into one CUDA context.
// After cudaDeviceReset (or any release of the primary context) the module is loaded
// again and the array may sit elsewhere, so a remembered address is only reused while the
// device's current context is the one it was looked up in.  Contexts are told apart by
// the driver's context ID (cuCtxGetId, unique for the life of the process), reached
// through the runtime's driver entry points so that the library needs no link to the
// driver library.  Without those entry points the address is looked up on every call.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct ScratchEntry {
    unsigned long long ctx_id;
    void* ptr;
};

std::mutex g_mutex;
ScratchEntry g_scratch[kMaxDevices] = {};
bool g_entry_points_tried = false;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// ID of the calling thread's current context; false when it cannot be had.
bool current_context_id(unsigned long long* id) {
    if (!g_entry_points_tried) {
        g_entry_points_tried = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f);
    }
    if (!g_ctx_get_current || !g_ctx_get_id) return false;
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return g_ctx_get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch in the current context of `device`, remembered per
// (device, context).  Returns nullptr when the lookup fails.
void* scratch_address(int device) {
    std::lock_guard<std::mutex> lock(g_mutex);
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    if (have_id && g_scratch[device].ptr != nullptr && g_scratch[device].ctx_id == id) return g_scratch[device].ptr;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch[device].ctx_id = have_id ? id : 0ull;
    g_scratch[device].ptr = have_id ? p : nullptr;
    return p;
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
    if (lo.PG > 0 && !lo.table) return KVQ_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(cache) % 256 || reinterpret_cast<uintptr_t>(q) % 16 ||
        reinterpret_cast<uintptr_t>(out) % 16 || reinterpret_cast<uintptr_t>(lo.table) % 4)
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
