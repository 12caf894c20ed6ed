// pi_noalloc.cu -- pi_sparse_fc2_noalloc: FC2 for callers that cannot
// allocate device memory.
//
// pi_sparse_fc2 needs a caller-provided workspace for its per-split partial
// sums.  Some callers cannot provide one: a plug-in running inside a host
// framework that owns the whole device memory pool and gives its plug-ins no
// way to allocate, or a service with a fixed device-memory budget that forbids
// any allocation after start-up.  For them this variant keeps the partial sums
// in a file-scope device array of fixed size instead (every GPU that loads the
// library holds it until the process exits).
//
// Host code never passes the array's name to a kernel: in host code that name
// is only a stand-in for the device symbol.  The device address is looked up
// with cudaGetSymbolAddress once per device, the first time the entry point is
// called with that device current.
#include <cuda_runtime.h>

#include <mutex>

#include "pi_internal.h"

namespace pi {
namespace {

// 8 MiB of fp32 partial sums: the FC2 partials of the path the plan takes
// must fit (the predictor's and FC1's partials do not enter this call).
constexpr size_t kNoallocScratchFloats = (size_t(8) << 20) / sizeof(float);

static __device__ __align__(256) float g_fc2_scratch[kNoallocScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch_addr[kMaxDevices] = {};

// Device address of g_fc2_scratch on the current device (looked up once).
cudaError_t scratch_address(float** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_fc2_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = static_cast<float*>(ptr);
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace pi

using namespace pi;

extern "C" pi_status pi_sparse_fc2_noalloc(const pi_layer_desc* desc, const float* h, const int32_t* idx,
                                           const int32_t* d_count, const pi_layer_weights* w, float* y,
                                           void* stream) {
    Plan p;
    if (!desc || !make_plan(*desc, &p)) return PI_ERR_INVALID_ARG;
    if (!fc2_args_ok(p, h, idx, d_count, w, y)) return PI_ERR_INVALID_ARG;
    // every partial-sum slot the reduction reads is written by the same call
    // first, so nothing in the array has to start at zero
    if (fc2_part_floats(p) > kNoallocScratchFloats) return PI_ERR_WORKSPACE;
    float* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return PI_ERR_CUDA;
    const cudaError_t e =
        launch_fc2(p, h, idx, d_count, layer_ptrs(w), nullptr, scratch, y, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PI_OK : PI_ERR_CUDA;
}
