// A5 weighted combine fused with the shared expert ("the CUDA tier wired into the DeepSeek V4
// engine", What it is: fused routed+shared MoE).
//
// out[t][m] = bf16_rn( y[shared row of t][m] + sum_{j=0..k-1} w[t][j] * y[inv_row[t][j]][m] ),
// accumulated in fp32 in that fixed order (no atomics), so the result is the same on every run.
#include "colimoe_internal.cuh"

namespace colimoe {
namespace {

__global__ void __launch_bounds__(256)
combine_kernel(const float *__restrict__ y, const int32_t *__restrict__ inv_row, const float *__restrict__ w,
               int T, int H, int top_k, int shared_base, __nv_bfloat16 *__restrict__ out) {
    pdl_begin();
    const int t = blockIdx.y;
    const int v = blockIdx.x * blockDim.x + threadIdx.x;   // float4 column index
    if (v >= H / 4) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (shared_base >= 0) acc = __ldg(reinterpret_cast<const float4 *>(y + (size_t)(shared_base + t) * H) + v);
    for (int j = 0; j < top_k; ++j) {
        const float wj = __ldg(w + (size_t)t * top_k + j);
        const int r = __ldg(inv_row + (size_t)t * top_k + j);
        const float4 yv = __ldg(reinterpret_cast<const float4 *>(y + (size_t)r * H) + v);
        acc.x = fmaf(wj, yv.x, acc.x);
        acc.y = fmaf(wj, yv.y, acc.y);
        acc.z = fmaf(wj, yv.z, acc.z);
        acc.w = fmaf(wj, yv.w, acc.w);
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t *>(&lo);
    packed.y = *reinterpret_cast<uint32_t *>(&hi);
    reinterpret_cast<uint2 *>(out + (size_t)t * H)[v] = packed;
}

// dst[0..bytes) = src[0..bytes), 16 bytes per thread step (both 16-byte aligned, bytes a multiple
// of 16); used to pull x from device-mapped host memory.
__global__ void __launch_bounds__(256) copy16(uint4 *__restrict__ dst, const uint4 *__restrict__ src, size_t n) {
    pdl_begin();
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

}  // namespace

int launch_copy(void *dst, const void *src, size_t bytes, int num_sms, cudaStream_t st) {
    const size_t n = bytes / 16;
    const size_t blocks = (n + 255) / 256 < (size_t)num_sms * 4 ? (n + 255) / 256 : (size_t)num_sms * 4;
    launch_pdl(copy16, dim3((unsigned)(blocks ? blocks : 1)), dim3(256), 0, st, static_cast<uint4 *>(dst),
               static_cast<const uint4 *>(src), n);
    return cudaPeekAtLastError() == cudaSuccess ? 1 : -1;
}

int launch_combine(const float *y, const int32_t *inv_row, const float *w, int T, int H, int top_k,
                   bool with_shared, __nv_bfloat16 *out, cudaStream_t st) {
    const dim3 grid((H / 4 + 255) / 256, T);
    launch_pdl(combine_kernel, grid, dim3(256), 0, st, y, inv_row, w, T, H, top_k, with_shared ? T * top_k : -1, out);
    return cudaPeekAtLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace colimoe
