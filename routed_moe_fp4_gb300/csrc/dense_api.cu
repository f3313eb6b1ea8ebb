// C ABI of the FP8 dense projection (coli_dense_* in colimoe.h): argument checks, the workspace
// for the activation terms, the choice between the CUDA-core kernel of gemv_fp8.cu (a few tokens)
// and the two launches of gemm_fp8.cu. No host synchronisation and no allocation inside a forward.
#include <stdarg.h>
#include <stdio.h>

#include <new>

#include "colimoe_internal.cuh"

using namespace colimoe;

struct coli_dense {
    int32_t max_tokens = 0, max_k = 0;
    cudaStream_t stream = nullptr;
    int num_sms = 0;
    uint8_t *xq = nullptr;     // [2][max_tokens][max_k] E4M3 terms of x
    float *xs = nullptr;       // [max_tokens] token scales
    float *part = nullptr;     // split-K partial sums
    int *cnt = nullptr;        // split-K arrival counters [SMs]
    int *err = nullptr;        // device error word
    uint64_t wait_ns = 0;
    int32_t path = COLI_DENSE_AUTO;   // forced kernel path, or the automatic choice
    int32_t last_path = COLI_DENSE_AUTO;
    char msg[256] = {0};
};

namespace {

thread_local char g_dense_err[256] = "no error";

void dense_err(coli_dense_t *d, const char *fmt, ...) {
    char *dst = d ? d->msg : g_dense_err;
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(dst, 256, fmt, ap);
    va_end(ap);
}

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

void free_dense(coli_dense_t *d) {
    if (d->xq) cudaFree(d->xq);
    if (d->xs) cudaFree(d->xs);
    if (d->part) cudaFree(d->part);
    if (d->cnt) cudaFree(d->cnt);
    if (d->err) cudaFree(d->err);
    delete d;
}

}  // namespace

extern "C" {

int coli_dense_create(int32_t max_tokens, int32_t max_k, void *cuda_stream, coli_dense_t **out) {
    if (!out) return COLI_ERR_INVALID_ARG;
    *out = nullptr;
    if (max_tokens < 1 || max_k < 128 || max_k % 128 || (double)max_tokens * max_k > 4.0e9) {
        dense_err(nullptr, "invalid dense config: need max_tokens >= 1, max_k a positive multiple of 128");
        return COLI_ERR_INVALID_ARG;
    }
    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
        cudaGetLastError();
        dense_err(nullptr, "no CUDA device available");
        return COLI_ERR_UNSUPPORTED_ARCH;
    }
    if (prop.major != 10 || prop.minor != 3) {
        dense_err(nullptr, "device %d (%s) is sm_%d%d; this library is built for sm_103a (GB300) only", dev,
                  prop.name, prop.major, prop.minor);
        return COLI_ERR_UNSUPPORTED_ARCH;
    }
    if (!fp8_available()) {
        dense_err(nullptr, "no tensor-map encoder in the driver: the FP8 GEMM cannot run");
        return COLI_ERR_UNSUPPORTED_ARCH;
    }
    coli_dense_t *d = new (std::nothrow) coli_dense_t();
    if (!d) return COLI_ERR_OUT_OF_MEMORY;
    d->max_tokens = max_tokens;
    d->max_k = max_k;
    d->stream = static_cast<cudaStream_t>(cuda_stream);
    d->num_sms = prop.multiProcessorCount;
    const size_t tk = (size_t)max_tokens * max_k;
    const size_t part = (size_t)(max_tokens < kSplitMaxTokens ? max_tokens : kSplitMaxTokens) * 128 * d->num_sms;
    if (cudaMalloc(&d->xq, 2 * tk + 256) != cudaSuccess || cudaMalloc(&d->xs, 4 * (size_t)max_tokens + 256) != cudaSuccess ||
        cudaMalloc(&d->part, 4 * part + 256) != cudaSuccess || cudaMalloc(&d->cnt, 4 * (size_t)d->num_sms + 256) != cudaSuccess ||
        cudaMemset(d->cnt, 0, 4 * (size_t)d->num_sms) != cudaSuccess ||
        cudaMalloc(&d->err, 256) != cudaSuccess || cudaMemset(d->err, 0, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        free_dense(d);
        dense_err(nullptr, "dense workspace allocation failed");
        return COLI_ERR_OUT_OF_MEMORY;
    }
    *out = d;
    return COLI_OK;
}

int coli_dense_forward(coli_dense_t *d, const void *x_bf16, int32_t T, int32_t K, const uint8_t *w_e4m3,
                       const float *w_scale, int32_t N, void *out_bf16) {
    if (!d) return COLI_ERR_INVALID_ARG;
    if (T == 0) return COLI_OK;
    if (T < 0 || T > d->max_tokens || K < 128 || K > d->max_k || K % 128 || N < 128 || N % 128) {
        dense_err(d, "need 0 <= T <= max_tokens, K a multiple of 128 up to max_k, N a positive multiple of 128");
        return COLI_ERR_INVALID_ARG;
    }
    if (!x_bf16 || !w_e4m3 || !w_scale || !out_bf16 || !al16(x_bf16) || !al16(w_e4m3) || !al16(out_bf16) ||
        (reinterpret_cast<uintptr_t>(w_scale) & 3)) {
        dense_err(d, "x, w, out must be non-NULL 16-byte aligned device pointers, w_scale 4-byte aligned");
        return COLI_ERR_INVALID_ARG;
    }
    if (x_bf16 == out_bf16) {
        dense_err(d, "out may not alias x");
        return COLI_ERR_INVALID_ARG;
    }
    cudaGetLastError();
    DenseArgs a;
    a.x = static_cast<const __nv_bfloat16 *>(x_bf16);
    a.T = T;
    a.K = K;
    a.N = N;
    a.w = w_e4m3;
    a.w_scale = w_scale;
    a.xq = d->xq;
    a.xs = d->xs;
    a.out = static_cast<__nv_bfloat16 *>(out_bf16);
    a.part = d->part;
    a.cnt = d->cnt;
    a.err = d->err;
    a.wait_ns = d->wait_ns;
    // A few tokens on a small matrix: the CUDA-core kernel (one launch, latency-bound work); else
    // the tensor-core GEMM
    const bool gemv_ok = dense_gemv_supported(T, K, N, d->num_sms);
    if (d->path == COLI_DENSE_CUDA_CORES && !gemv_ok) {
        dense_err(d, "the CUDA-core path needs K <= 8192 and one block's weight rows within shared memory");
        return COLI_ERR_INVALID_ARG;
    }
    const bool gemv = d->path == COLI_DENSE_CUDA_CORES || (d->path == COLI_DENSE_AUTO && gemv_ok &&
                                                           T <= dense_gemv_max_tokens(K, N));
    const int n = gemv ? launch_dense_gemv(a, d->num_sms, d->stream) : launch_dense_fp8(a, d->num_sms, d->stream);
    d->last_path = gemv ? COLI_DENSE_CUDA_CORES : COLI_DENSE_TENSOR;
    if (n == -2) {
        dense_err(d, "tensor maps for the FP8 GEMM could not be encoded");
        return COLI_ERR_INVALID_ARG;
    }
    if (n < 0) {
        dense_err(d, "kernel launch failed: %s", cudaGetErrorString(cudaGetLastError()));
        return COLI_ERR_CUDA;
    }
    return COLI_OK;
}

void coli_dense_destroy(coli_dense_t *d) {
    if (!d) return;
    cudaStreamSynchronize(d->stream);
    free_dense(d);
}

const char *coli_dense_last_error(const coli_dense_t *d) { return d ? d->msg : g_dense_err; }

int coli_dense_set_path(coli_dense_t *d, int32_t path) {
    if (!d) return COLI_ERR_INVALID_ARG;
    if (path < COLI_DENSE_AUTO || path > COLI_DENSE_TENSOR) {
        dense_err(d, "unknown dense path %d", path);
        return COLI_ERR_INVALID_ARG;
    }
    d->path = path;
    return COLI_OK;
}

int coli_dense_last_path(const coli_dense_t *d) { return d ? d->last_path : COLI_DENSE_AUTO; }

int coli_dense_device_error(coli_dense_t *d, int32_t *code) {
    if (!d || !code) return COLI_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(d->stream) != cudaSuccess ||
        cudaMemcpy(code, d->err, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(d->err, 0, sizeof(int)) != cudaSuccess) {
        dense_err(d, "stream error: %s", cudaGetErrorString(cudaGetLastError()));
        return COLI_ERR_CUDA;
    }
    return COLI_OK;
}

}  // extern "C"
