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

#include "../../include/fp8bs.h"
#include "common.cuh"
#include "internal.h"

namespace fp8bs {
namespace {

constexpr int kNoAllocPartials = FP8BS_NOALLOC_MAX_PARTIALS;
constexpr int64_t kTasksPerPartial = 64;   // warp tasks (1024 columns of one row) per amax CTA

// One amax partial per CTA of the first pass.  Every GPU that loads the
// library holds this array (16 KB) until the process exits.  Each call
// writes the slots it reads before reading them, so stale contents from an
// earlier call never matter; calls that overlap on the GPU share it and race.
static __device__ __align__(256) uint32_t g_amax_scratch[kNoAllocPartials];

std::mutex g_mu;
void* g_scratch_ptr[64] = {nullptr};

// Device address of g_amax_scratch on the current device, looked up once per
// device.  In host code the array's name is only a host-side stand-in, so
// the kernels must be given this address instead.
int scratch_for_current_device(uint32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return FP8BS_ECUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_amax_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            return FP8BS_ECUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = static_cast<uint32_t*>(g_scratch_ptr[dev]);
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
