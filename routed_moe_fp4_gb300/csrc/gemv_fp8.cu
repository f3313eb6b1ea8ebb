// FP8 dense projection for a few tokens on the CUDA cores:
// out[t][n] = bf16(sum_k x[t][k] * e4m3(w[n][k]) * w_scale[n/128][k/128]) (the dense weight format of
// "DeepSeek V4 Flash CPU inference with NVMe expert streaming", the review question on config-driven
// V4 sizes; the dense-on-GPU tier of "DeepSeek V4 Flash support -- CUDA/VRAM expert tiering").
//
// With one to eight tokens the projection reads each weight byte once and does one multiply-add
// per token with it, so it is bound by HBM and by latency, not by tensor throughput. One kernel
// does it all: every block owns a contiguous range of weight rows, copies them into shared memory
// with bulk copies issued at its start (before the dependency wait, since no kernel of a forward
// writes the weights), and its threads split K, sixteen features each, holding those features of
// the pass's tokens in registers. Per row a thread multiplies sixteen weights by them in fp32
// (packed two-lane FMAs, two rows at a time for independent work), scales by the row's block
// scale, and the warp sums the partials of its 32 threads; the block's warps add theirs in a fixed
// order at the end of the pass. No activation terms, no K split across blocks, no arrival counters.
//
// Arithmetic: an E4M3 byte becomes an fp32 equal to its value times 2^-120, by moving the sign to
// bit 31 and the exponent and mantissa bits to bits 26..20 (subnormals included: they land on fp32
// subnormals). x is scaled per token by a power of two that puts the block's largest |x| in
// [2^60, 2^61), so every product of a weight and an x element is exact and normal; the sums are
// fp32; the two powers of two are undone before the single rounding to bf16. The NaN codes
// (S.1111.111) make the row's results NaN, as in the tensor-core path.
#include <cuda_bf16.h>

#include "colimoe_internal.cuh"
#include "sm103_ptx.cuh"

namespace colimoe {
namespace {

constexpr int kKpt = 16;                    // features per thread: one 16-byte word of a weight row
constexpr int kMaxChunks = 16;              // bulk copies (and mbarriers) per block
constexpr uint32_t kChunkBytes = 16384;     // rows per copy: as many as fit 16 KB (at least one)
constexpr size_t kSmemLimit = 227 * 1024;

struct GemvFp8Params {
    const __nv_bfloat16 *x;      // [T][K]
    int T, K, N;
    const uint8_t *w;            // [N][K]
    const float *w_scale;        // [N/128][K/128]
    __nv_bfloat16 *out;          // [T][N]
    int rows_max;                // rows of the largest block
    int chunk_rows;              // rows per bulk copy
    int *err;
    uint64_t wait_ns;
};

// Byte 3 of v as fp32 (E4M3 value times 2^-120): sign to bit 31, exponent and mantissa to bits 26..20.
__device__ __forceinline__ float e4m3_top(uint32_t v) {
    return __uint_as_float((uint32_t)((int32_t)v >> 4) & 0x87F00000u);
}

// Non-zero when a byte of w is an E4M3 NaN code (low seven bits all set).
__device__ __forceinline__ uint32_t e4m3_nan_bytes(uint32_t w) {
    const uint32_t v = ~w & 0x7F7F7F7Fu;   // a zero byte marks a NaN code
    return (v - 0x01010101u) & ~v & 0x80808080u;
}

// One splitting level of the warp sum: lanes with bit `o` set keep the upper half of the NV
// values, the others the lower half, and each adds its partner's copy of the half it kept.
template <int TP, int NV>
__device__ __forceinline__ void split_level(float (&v)[TP], int lane) {
    constexpr int o = 16 * NV / TP, h = NV / 2;
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < h; ++j) {
        const float send = up ? v[j] : v[j + h];
        const float keep = up ? v[j + h] : v[j];
        v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
}

// Sums v[t] over the warp's 32 lanes for each of the TP tokens in a fixed order; lane l returns the
// sum of token l / (32 / TP).
template <int TP>
__device__ __forceinline__ float warp_token_sums(float (&v)[TP], int lane) {
    if constexpr (TP >= 8) split_level<TP, 8>(v, lane);
    if constexpr (TP >= 4) split_level<TP, 4>(v, lane);
    if constexpr (TP >= 2) split_level<TP, 2>(v, lane);
    float s = v[0];
#pragma unroll
    for (int o = 16 / TP; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

template <int TP>
__global__ void __launch_bounds__(TP == 8 ? 256 : 512, 1) gemv_fp8(const GemvFp8Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kMaxChunks * 8);
    uint8_t *wsm = smem + 256;                                        // [rows_max][K] weight rows
    const int NW = blockDim.x >> 5;
    float *red = reinterpret_cast<float *>(wsm + (size_t)p.rows_max * p.K);   // [NW][rows_max][TP]
    float *xm = red + (size_t)NW * p.rows_max * TP;                   // [NW][TP] warp maxima of |x|
    float *omul = xm + NW * TP;                                       // [TP] output multipliers

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r0 = (int)((long long)blockIdx.x * p.N / gridDim.x);
    const int rows = (int)((long long)(blockIdx.x + 1) * p.N / gridDim.x) - r0;
    const int nch = (rows + p.chunk_rows - 1) / p.chunk_rows;
    if (tid == 0) {
        for (int c = 0; c < nch; ++c) ptx::mbar_init(ptx::smem_addr(&bar[c]), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        const uint64_t pol = ptx::policy_evict_first();
        for (int c = 0; c < nch; ++c) {
            const uint32_t bytes = (uint32_t)min(p.chunk_rows, rows - c * p.chunk_rows) * (uint32_t)p.K;
            const uint32_t b = ptx::smem_addr(&bar[c]);
            ptx::mbar_arrive_expect_tx(b, bytes);
            ptx::bulk_g2s_hint(ptx::smem_addr(wsm + (size_t)c * p.chunk_rows * p.K),
                               p.w + ((size_t)r0 + (size_t)c * p.chunk_rows) * p.K, bytes, b, pol);
        }
    }
    pdl_wait();       // x may be the previous kernel's output
    pdl_trigger();
    __syncthreads();  // the barriers' initialisation, before any thread waits on them

    const int k0 = tid * kKpt;
    const bool act = k0 < p.K;
    const int kb = k0 >> 7;                                           // the thread's 128-feature block
    int waited = 0;                                                   // chunks known to have landed
    for (int t0 = 0; t0 < p.T; t0 += TP) {
        // ---- this pass's tokens: 16 features each, in fp32 pairs, and the block's max |x| per token
        float2 xs[TP][kKpt / 2];
#pragma unroll
        for (int t = 0; t < TP; ++t) {
            uint32_t m = 0;
            if (act && t0 + t < p.T) {
                const uint4 *src = reinterpret_cast<const uint4 *>(p.x + (size_t)(t0 + t) * p.K + k0);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 u = src[h];
                    const uint32_t q[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        xs[t][4 * h + j] = make_float2(__uint_as_float(q[j] << 16), __uint_as_float(q[j] & 0xFFFF0000u));
                        m = max(m, max(q[j] << 17 >> 1, (q[j] & 0x7FFF0000u)));   // |x| bits, ordered
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < kKpt / 2; ++j) xs[t][j] = make_float2(0.f, 0.f);
            }
            m = __reduce_max_sync(0xffffffffu, m);
            if (lane == 0) xm[warp * TP + t] = __uint_as_float(m);
        }
        __syncthreads();
#pragma unroll
        for (int t = 0; t < TP; ++t) {
            uint32_t m = 0;
            for (int w = 0; w < NW; ++w) m = max(m, __float_as_uint(xm[w * TP + t]));
            // biased exponent of the block's max |x|, kept where both multipliers are normal floats
            const uint32_t eb = min(max((m >> 23) & 0xFFu, 1u), 253u);
            const float in_mul = __uint_as_float((254u - eb) << 23);     // 2^(127 - eb)
            if (tid == 0) omul[t] = __uint_as_float(eb << 23);            // 2^(eb - 127)
#pragma unroll
            for (int j = 0; j < kKpt / 2; ++j)
                xs[t][j] = make_float2((xs[t][j].x * in_mul) * 0x1p60f, (xs[t][j].y * in_mul) * 0x1p60f);
        }

        // ---- rows, two at a time: exact products, fp32 sums, block scale, warp sums per token
        int cur_rb = -1;
        float sc = 0.f;
        for (int r = 0; r < rows; r += 2) {
            const int nr = r + 1 < rows ? 2 : 1;
            while (waited * p.chunk_rows < r + nr)
                ptx::mbar_wait(ptx::smem_addr(&bar[waited++]), 0, p.err, ptx::kErrWaitFull, abort_flag, p.wait_ns);
            const bool live = act && !*abort_flag;
            float acc[2][TP];
            uint32_t nan[2] = {0u, 0u};
            float rsc[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int rr = i < nr ? r + i : r;                    // a lone last row is done twice
                const int rb = (r0 + rr) >> 7;
                if (rb != cur_rb) {
                    cur_rb = rb;
                    sc = act ? __ldg(p.w_scale + (size_t)rb * (p.K >> 7) + kb) : 0.f;
                }
                rsc[i] = sc;
                uint4 wv = make_uint4(0u, 0u, 0u, 0u);
                if (live) wv = *reinterpret_cast<const uint4 *>(wsm + (size_t)rr * p.K + k0);
                const uint32_t wq[4] = {wv.x, wv.y, wv.z, wv.w};
                float2 a2[TP];
#pragma unroll
                for (int t = 0; t < TP; ++t) a2[t] = make_float2(0.f, 0.f);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t w = wq[q];
                    nan[i] |= e4m3_nan_bytes(w);
                    const float2 lo = make_float2(e4m3_top(w << 24), e4m3_top(w << 16));
                    const float2 hi = make_float2(e4m3_top(w << 8), e4m3_top(w));
#pragma unroll
                    for (int t = 0; t < TP; ++t) {
                        a2[t] = __ffma2_rn(lo, xs[t][2 * q], a2[t]);
                        a2[t] = __ffma2_rn(hi, xs[t][2 * q + 1], a2[t]);
                    }
                }
#pragma unroll
                for (int t = 0; t < TP; ++t) acc[i][t] = a2[t].x + a2[t].y;
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
#pragma unroll
                for (int t = 0; t < TP; ++t) acc[i][t] = nan[i] ? __uint_as_float(0x7FC00000u) : acc[i][t] * rsc[i];
                const float s = warp_token_sums<TP>(acc[i], lane);
                if (i < nr && (lane & (32 / TP - 1)) == 0)
                    red[((size_t)warp * p.rows_max + r + i) * TP + lane / (32 / TP)] = s;
            }
        }
        __syncthreads();

        // ---- the warps' sums in warp order, undo the two powers of two, round once
        for (int i = tid; i < rows * TP; i += blockDim.x) {
            const int t = i / rows, r = i - t * rows;
            if (t0 + t >= p.T) continue;
            float s = 0.f;
            for (int w = 0; w < NW; ++w) s += red[((size_t)w * p.rows_max + r) * TP + t];
            p.out[(size_t)(t0 + t) * p.N + r0 + r] = __float2bfloat16_rn((s * 0x1p60f) * omul[t]);
        }
        __syncthreads();
    }
    // copies still in flight after a wait gave up land before the block's shared memory goes away
    if (tid == 0 && *abort_flag)
        for (int c = 0; c < nch; ++c) ptx::mbar_wait(ptx::smem_addr(&bar[c]), 0, nullptr, 0, nullptr, p.wait_ns);
}

template <int TP>
int launch_tp(const GemvFp8Params &p, int grid, int threads, size_t smem, cudaStream_t st) {
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(gemv_fp8<TP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit) !=
            cudaSuccess)
            return -1;
        attr = true;
    }
    launch_pdl(gemv_fp8<TP>, dim3(grid), dim3(threads), smem, st, p);
    return cudaPeekAtLastError() == cudaSuccess ? 1 : -1;
}

int gemv_tp_max(int K) { return K <= 4096 ? 8 : 4; }

size_t gemv_smem(int K, int N, int num_sms, int tp) {
    const int grid = N < num_sms ? N : num_sms;
    const size_t rows_max = ((size_t)N + grid - 1) / grid;
    const size_t nw = ((size_t)K / kKpt + 31) / 32;
    return 256 + rows_max * K + (nw * rows_max * tp + nw * tp + tp) * sizeof(float);
}

}  // namespace

bool dense_gemv_supported(int T, int K, int N, int num_sms) {
    if (T < 1 || K > 8192 || K % 128 || N < 1) return false;
    const int grid = N < num_sms ? N : num_sms;
    const size_t rows_max = ((size_t)N + grid - 1) / grid;
    const size_t chunk_rows = kChunkBytes / K > 0 ? kChunkBytes / K : 1;
    if ((rows_max + chunk_rows - 1) / chunk_rows > (size_t)kMaxChunks) return false;
    return gemv_smem(K, N, num_sms, gemv_tp_max(K)) <= kSmemLimit;
}

int dense_gemv_max_tokens(int K, int N) {
    // Measured on a GB300 (K 4096 and 7168, N 512 to 4096, 1 to 8 tokens, L2 flushed): the tensor
    // path costs 13-19 us whatever the size at these token counts (the activation split, the K
    // split and its tail), the CUDA-core kernel 9-10 us plus time that grows with the weight bytes
    // and the tokens. These are the token counts below which the CUDA-core kernel was faster.
    const double mib = (double)N * K / (1024.0 * 1024.0);
    return mib <= 4.0 ? 8 : mib <= 7.0 ? 4 : mib <= 14.0 ? 2 : 0;
}

int launch_dense_gemv(const DenseArgs &a, int num_sms, cudaStream_t st) {
    if (!dense_gemv_supported(a.T, a.K, a.N, num_sms)) return -2;
    const int tp_max = gemv_tp_max(a.K);
    const int tp = a.T >= tp_max ? tp_max : a.T > 2 ? (a.T > 4 ? 8 : 4) : a.T;   // tokens per pass
    GemvFp8Params p;
    p.x = a.x;
    p.T = a.T;
    p.K = a.K;
    p.N = a.N;
    p.w = a.w;
    p.w_scale = a.w_scale;
    p.out = a.out;
    const int grid = a.N < num_sms ? a.N : num_sms;
    p.rows_max = (a.N + grid - 1) / grid;
    p.chunk_rows = (int)(kChunkBytes / a.K > 0 ? kChunkBytes / a.K : 1);
    p.err = a.err;
    p.wait_ns = a.wait_ns ? a.wait_ns : ptx::kWaitLimitNs;
    const int threads = ((a.K / kKpt + 31) / 32) * 32;
    const size_t smem = gemv_smem(a.K, a.N, num_sms, tp);
    switch (tp) {
        case 1: return launch_tp<1>(p, grid, threads, smem, st);
        case 2: return launch_tp<2>(p, grid, threads, smem, st);
        case 4: return launch_tp<4>(p, grid, threads, smem, st);
        default: return launch_tp<8>(p, grid, threads, smem, st);
    }
}

}  // namespace colimoe
