// Block-wide exclusive scan shared by the single-block planning kernels (permute.cu, bank.cu).
#pragma once

namespace colimoe {

// Exclusive block scan of one value per thread (blockDim.x == 1024). Returns the exclusive
// prefix; *total receives the block sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int *smem_warp, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) smem_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = smem_warp[lane];
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        smem_warp[lane] = wi - w;          // exclusive prefix of warp sums
        if (lane == 31) smem_warp[32] = wi;
    }
    __syncthreads();
    const int res = smem_warp[warp] + incl - v;
    *total = smem_warp[32];
    __syncthreads();
    return res;
}

// The same scan for a 64-bit value that packs several counters into bit fields: one scan (three
// barriers) instead of one per counter, as long as no field's block sum overflows into the next.
__device__ __forceinline__ unsigned long long block_exclusive_scan64(unsigned long long v,
                                                                     unsigned long long *smem_warp,
                                                                     unsigned long long *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) smem_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const unsigned long long w = smem_warp[lane];
        unsigned long long wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        smem_warp[lane] = wi - w;
        if (lane == 31) smem_warp[32] = wi;
    }
    __syncthreads();
    const unsigned long long res = smem_warp[warp] + incl - v;
    *total = smem_warp[32];
    __syncthreads();
    return res;
}

}  // namespace colimoe
