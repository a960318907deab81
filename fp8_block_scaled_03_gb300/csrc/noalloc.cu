// noalloc.cu -- per-tensor quantisation for callers that cannot allocate
// device memory.
//
// A per-tensor scale needs the amax of the whole tensor before any code can
// be written, so the usual entry point (fp8_quantize with PER_TENSOR) keeps
// one partial maximum per CTA in the caller's workspace.  Some callers have
// no way to provide that workspace: code that only receives the input and
// output buffers from a host framework whose allocator owns all device
// memory, plugin or custom-op interfaces that hand over tensors but no
// scratch, and real-time or embedded callers that forbid allocation once
// they are running.  This entry point keeps the partials in a fixed array
// that lives inside the library instead, so the caller passes only x, q
// and the scale.
#include <mutex>

#include <cuda.h>

#include "../../include/fp8bs.h"
#include "common.cuh"
#include "internal.h"

namespace fp8bs {
namespace {

constexpr int kNoAllocPartials = FP8BS_NOALLOC_MAX_PARTIALS;
constexpr int64_t kTasksPerPartial = 64;   // warp tasks (1024 columns of one row) per amax CTA

// One amax partial per CTA of the first pass.  The array (16 KB) is part of
// the library's device module: it is committed on a GPU when that module is
// loaded there (at the first call on that device under lazy module loading)
// and held until the context ends.  Each call
// writes the slots it reads before reading them, so stale contents from an
// earlier call never matter; calls that overlap on the GPU share it and race.
static __device__ __align__(256) uint32_t g_amax_scratch[kNoAllocPartials];

std::mutex g_mu;

// Device address of g_amax_scratch, cached per device together with the
// unique id of the context it was looked up in.  In host code the array's
// name is only a host-side stand-in, so the kernels must be given this
// address instead.  A context that is destroyed and created again (after
// cudaDeviceReset, or when the primary context is released) loads the module
// afresh, possibly at another address; its id differs from the cached one
// (ids are never reused within a process), so the address is looked up again.
struct ScratchEntry {
    unsigned long long ctx_id;
    void* ptr;
};
ScratchEntry g_scratch[64] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <class Fn>
Fn driver_fn(const char* name) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(p);
}

// Id of the calling thread's current context; false if there is none yet or
// the driver does not say.
bool current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (get_current == nullptr || get_id == nullptr) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

int scratch_for_current_device(uint32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return FP8BS_ECUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    unsigned long long id = 0;
    if (current_context_id(&id) && g_scratch[dev].ptr != nullptr && g_scratch[dev].ctx_id == id) {
        *out = static_cast<uint32_t*>(g_scratch[dev].ptr);
        return FP8BS_OK;
    }
    // First call in this context: the lookup loads the module (and with it
    // the array) if lazy loading has not done so yet.
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_amax_scratch) != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();
        return FP8BS_ECUDA;
    }
    // Cached only when the context can be identified; otherwise every call
    // looks the address up, which is correct, only slower.
    g_scratch[dev] = current_context_id(&id) ? ScratchEntry{id, p} : ScratchEntry{0, nullptr};
    *out = static_cast<uint32_t*>(p);
    return FP8BS_OK;
}

}  // namespace
}  // namespace fp8bs

using namespace fp8bs;

extern "C" int fp8_quantize_per_tensor_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ld_x, void* q,
                                               float* scale, fp8bs_stream_t stream) {
    if (rows < 0 || cols < 0 || cols % 8 != 0 || ld_x < cols || ld_x % 8 != 0) return FP8BS_EINVAL;
    if (rows == 0 || cols == 0) return FP8BS_OK;
    if (x == nullptr || q == nullptr || scale == nullptr) return FP8BS_EINVAL;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(q) & 15u) ||
        (reinterpret_cast<uintptr_t>(scale) & 3u))
        return FP8BS_EALIGN;
    const int64_t tasks = rows * ceil_div(cols, 1024);
    const int64_t nparts = ceil_div(tasks, kTasksPerPartial);
    if (nparts > kNoAllocPartials) return FP8BS_EINVAL;   // larger than the built-in scratch serves
    uint32_t* partials = nullptr;
    const int rc = scratch_for_current_device(&partials);
    if (rc != FP8BS_OK) return rc;
    const int err = launch_quantize_per_tensor_scratch(static_cast<const uint16_t*>(x), rows, cols, ld_x,
                                                       static_cast<uint8_t*>(q), scale, partials, (int)nparts,
                                                       reinterpret_cast<cudaStream_t>(stream));
    if (err != 0) {
        (void)cudaGetLastError();
        return FP8BS_ECUDA;
    }
    return FP8BS_OK;
}

// Test hook: the address the entry point would use in the current context
// (through its cache) and the address a fresh lookup gives.  Lets a test
// check, without launching anything, that the cache follows a context that
// was destroyed and created again.
extern "C" int fp8bs_test_noalloc_scratch(void** cached, void** looked_up) {
    if (cached == nullptr || looked_up == nullptr) return FP8BS_EINVAL;
    uint32_t* p = nullptr;
    const int rc = scratch_for_current_device(&p);
    if (rc != FP8BS_OK) return rc;
    void* q = nullptr;
    if (cudaGetSymbolAddress(&q, g_amax_scratch) != cudaSuccess) {
        (void)cudaGetLastError();
        return FP8BS_ECUDA;
    }
    *cached = p;
    *looked_up = q;
    return FP8BS_OK;
}
