// Routing without any device allocation: the router kernels of the forward, run with their
// scratch (the sigmoid scores and the split-K partial logits) in a fixed array that is part of
// the library image, so the call needs no cudaMalloc, cudaFree or allocator of any kind.
//
// Some callers cannot allocate device memory when they route: code that runs while a CUDA graph
// is being captured (allocation is not a capturable operation), runtimes that own every byte of
// device memory through their own pool and forbid a library from allocating behind their back,
// and latency-critical loops where a first-call allocation is not acceptable. This entry point is
// for them; coli_moe_forward remains the general path.
#include <mutex>

#include "colimoe_internal.cuh"

namespace colimoe {
namespace {

// Largest T * E this entry point accepts, and the scratch it needs for that size.
// The partial logits take the router's fixed cap, the same the forward's workspace holds, so both
// calls choose the same split count and add the partials in the same order.
constexpr size_t kMaxScores = 262144;              // T * E <= 262144, e.g. 1024 tokens x 256 experts
constexpr size_t kMaxPartials = kRouterPartialFloats;          // split-K partial logits
constexpr size_t kScratchFloats = kMaxScores + kMaxPartials;   // 5 MiB

// One copy per device that loads the library, resident until the process exits.
__device__ __align__(256) float g_route_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
struct DeviceSetup {
    float *scratch = nullptr;   // device address of g_route_scratch on this device
    int num_sms = 0;
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mutex;

// Looks up the array's device address on the current device (once per device).
int setup_current_device(DeviceSetup **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        set_create_error("route_static: no usable current CUDA device");
        return COLI_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    DeviceSetup &d = g_setup[dev];
    if (!d.scratch) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
            set_create_error("route_static: cudaGetDeviceProperties failed: %s", cudaGetErrorString(cudaGetLastError()));
            return COLI_ERR_CUDA;
        }
        if (prop.major != 10 || prop.minor != 3) {
            set_create_error("route_static: device %d is sm_%d%d; this library is built for sm_103a (GB300) only", dev,
                             prop.major, prop.minor);
            return COLI_ERR_UNSUPPORTED_ARCH;
        }
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_route_scratch);
        if (e != cudaSuccess || !ptr) {
            cudaGetLastError();
            set_create_error("route_static: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
            return COLI_ERR_CUDA;
        }
        d.num_sms = prop.multiProcessorCount;
        d.scratch = static_cast<float *>(ptr);
    }
    *out = &d;
    return COLI_OK;
}

}  // namespace
}  // namespace colimoe

using namespace colimoe;

extern "C" int coli_moe_route_static(const void *x_bf16, int32_t T, int32_t H, const float *router_w,
                                     const float *router_bias, int32_t E, int32_t top_k, int32_t *idx_out,
                                     float *weights_out, void *cuda_stream) {
    if (T == 0) return COLI_OK;
    if (T < 0 || E < 1 || E > 1024 || H < 128 || H % 128 || top_k < 1 || top_k > 32 || top_k > E) {
        set_create_error("route_static: need T >= 0, 1 <= E <= 1024, H a positive multiple of 128, "
                         "1 <= top_k <= min(E, 32)");
        return COLI_ERR_INVALID_ARG;
    }
    if ((size_t)T * (size_t)E > kMaxScores) {
        set_create_error("route_static: T * E = %lld exceeds the fixed scratch limit of %lld (T <= %lld for E = %d)",
                         (long long)T * E, (long long)kMaxScores, (long long)(kMaxScores / (size_t)E), E);
        return COLI_ERR_INVALID_ARG;
    }
    if (!x_bf16 || !router_w || !idx_out || !weights_out || (reinterpret_cast<uintptr_t>(x_bf16) & 15) ||
        (reinterpret_cast<uintptr_t>(router_w) & 15)) {
        set_create_error("route_static: x, router_w, idx_out and weights_out must be non-NULL device pointers "
                         "(x and router_w 16-byte aligned)");
        return COLI_ERR_INVALID_ARG;
    }
    DeviceSetup *d = nullptr;
    const int rc = setup_current_device(&d);
    if (rc != COLI_OK) return rc;
    cudaGetLastError();
    const int n = launch_router(static_cast<const __nv_bfloat16 *>(x_bf16), T, H, router_w, router_bias, E, top_k,
                                d->scratch, idx_out, weights_out, d->scratch + kMaxScores, d->num_sms,
                                nullptr, 0, nullptr, static_cast<cudaStream_t>(cuda_stream));
    if (n < 0) {
        set_create_error("route_static: kernel launch failed: %s", cudaGetErrorString(cudaGetLastError()));
        return COLI_ERR_CUDA;
    }
    return COLI_OK;
}
