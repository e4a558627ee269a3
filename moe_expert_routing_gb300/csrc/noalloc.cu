// smoe_route_noalloc: the routing step with its scratch in a fixed device array instead of a
// caller-provided workspace.
//
// Some callers cannot call cudaMalloc.  A plugin running inside a host application that owns
// the whole device-memory budget (an inference server with a preallocated arena, a game or
// visualisation engine) may be forbidden to allocate; other callers cannot afford the implicit
// device-wide synchronisation a cudaMalloc may cause in the middle of a latency-critical loop.
// For them this entry point needs nothing but its inputs and outputs: the split-K partial
// router logits live in g_route_scratch below, a file-scope device array of
// kNoallocScratchFloats floats (4 MiB) that every GPU which loads the library holds until the
// process exits.  A call needs B * E <= kNoallocScratchFloats.  Up to 256 tokens at 128
// experts the call uses the same split-K partials as smoe_route and returns identical
// results; beyond that the number of partials is capped to what fits, which changes only the
// fp32 summation order of the logits.
//
// Set-up: the first call on a device (with that device current) looks up the array's device
// address with cudaGetSymbolAddress and caches it, keyed by the unique id of the device's
// current CUDA context; make that first call before any stream capture.  A device reset (or
// any teardown of the context) gives the next call a new context id, so the address is looked
// up again (again a first call: before any capture).  In host code the name g_route_scratch
// is only a host-side stand-in for the symbol, never a usable device address, which is why
// the looked-up address is passed to the kernels.
//
// Sharing: every call on a device uses the same array and leaves the last call's partial
// logits in it.  Nothing has to start at zero (each call overwrites every partial it reads),
// but calls whose work overlaps on the GPU (different streams, no ordering) race on the array
// and must be serialised by the caller.
#include "smoe_internal.cuh"

#include <algorithm>
#include <mutex>

namespace smoe {
namespace {

constexpr size_t kNoallocScratchFloats = 1u << 20;   // 4 MiB: splits * B * E partial logits

static __device__ __align__(256) float g_route_scratch[kNoallocScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
float* g_scratch_ptr[kMaxDevices] = {nullptr};
unsigned long long g_scratch_ctx[kMaxDevices] = {0};   // context id the address belongs to

// Unique id of the calling thread's current CUDA context (0 if there is none yet or the driver
// cannot say).
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    }();
    static PFN_cuCtxGetId_v12000 get_id = []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    }();
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_route_scratch in the current device's context (looked up once per
// context).
cudaError_t scratch_for_current_device(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    // before the runtime's first use of the device there is no current context (id 0): the
    // look-up below creates it, and its id is read afterwards
    const unsigned long long ctx = current_context_id();
    if (!g_scratch_ptr[dev] || ctx == 0 || g_scratch_ctx[dev] != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_route_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = static_cast<float*>(p);
        g_scratch_ctx[dev] = current_context_id();
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace smoe

using namespace smoe;

extern "C" SMOE_API smoe_status smoe_route_noalloc(const smoe_layer_desc* desc, const uint16_t* x,
                                                   const float* gate_w, const float* gate_bias, int32_t B,
                                                   int32_t* topk_idx, float* topk_w, void* stream) {
    const smoe_status st = check_desc(desc);
    if (st != SMOE_OK) return st;
    if (B < 0) return SMOE_ERR_INVALID_ARG;
    if (B == 0) return SMOE_OK;
    if (!x || !gate_w || !topk_idx || !topk_w) return SMOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(gate_w) & 15u))
        return SMOE_ERR_UNSUPPORTED;
    // the partial logits of this call must fit the fixed array: at least one split of B x E,
    // and no more splits than fit
    const size_t per_split = (size_t)B * desc->num_experts;
    if (per_split > kNoallocScratchFloats) return SMOE_ERR_UNSUPPORTED;
    const int cap = (int)std::min<size_t>(kNoallocScratchFloats / per_split, 1 << 20);
    float* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return SMOE_ERR_CUDA;
    return launch_route(*desc, x, gate_w, gate_bias, B, topk_idx, topk_w, scratch,
                        static_cast<cudaStream_t>(stream), cap) == cudaSuccess
               ? SMOE_OK
               : SMOE_ERR_CUDA;
}
