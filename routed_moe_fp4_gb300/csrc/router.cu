// A1 router: fp32 logits, sigmoid scores, bias-adjusted top-k with warp shuffles, renormalised
// weights ("the CUDA tier wired into the DeepSeek V4 engine", What it is: route on device).
//
// logits[t][e] = sum_h x[t][h] * Wr[e][h] in fp32 (x is bf16, exact in fp32); s = 1/(1+exp(-z)).
// key = fp32(s + b); the top_k largest keys in descending order, bit-identical keys going to
// the lower expert index; w_j = s_j / S, S the fp32 sum of the chosen s in slot order, one
// IEEE division each. Built without fast-math: every add, divide and expf is the IEEE/accurate one.
#include "colimoe_internal.cuh"
#include "sm103_ptx.cuh"
#include "topk.cuh"

#include <float.h>

#include <algorithm>

namespace colimoe {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float sigmoidf_ieee(float z) {
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-z)));
}

// Small T: one expert per block, its router row split over eight warps, up to 8 tokens per block
// row. Lanes read the row as float4, four loads issued before use; the eight warp partials are
// added in warp order (deterministic).
constexpr int kSmallTok = 8;
constexpr int kSmallWarps = 8;

__global__ void __launch_bounds__(kSmallWarps * 32)
router_logits_small(const __nv_bfloat16 *__restrict__ x, int T, int H, const float *__restrict__ wr,
                    int E, float *__restrict__ scores) {
    pdl_begin();
    __shared__ float part[kSmallWarps][kSmallTok];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x;
    const int t0 = blockIdx.y * kSmallTok;
    const int nt = min(kSmallTok, T - t0);
    float acc[kSmallTok];
#pragma unroll
    for (int t = 0; t < kSmallTok; ++t) acc[t] = 0.f;
    const int nv = H / (4 * kSmallWarps);                    // float4 per warp slice
    const float4 *wrow = reinterpret_cast<const float4 *>(wr + (size_t)e * H) + warp * nv;
    const uint2 *xbase = reinterpret_cast<const uint2 *>(x + (size_t)t0 * H) + warp * nv;
    for (int c0 = lane; c0 < nv; c0 += 128) {
        float4 wv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = c0 + 32 * u;
            wv[u] = c < nv ? __ldg(wrow + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int t = 0; t < kSmallTok; ++t) {
            if (t < nt) {
                float a = acc[t];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c = c0 + 32 * u;
                    if (c < nv) {
                        const uint2 xv = __ldg(xbase + (size_t)t * (H / 4) + c);
                        a = fmaf(bf16_lo(xv.x), wv[u].x, a);
                        a = fmaf(bf16_hi(xv.x), wv[u].y, a);
                        a = fmaf(bf16_lo(xv.y), wv[u].z, a);
                        a = fmaf(bf16_hi(xv.y), wv[u].w, a);
                    }
                }
                acc[t] = a;
            }
        }
    }
#pragma unroll
    for (int t = 0; t < kSmallTok; ++t) {
        float a = acc[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0) part[warp][t] = a;
    }
    __syncthreads();
    if (warp == 0 && lane < nt) {
        float a = part[0][lane];
#pragma unroll
        for (int w = 1; w < kSmallWarps; ++w) a += part[w][lane];
        scores[(size_t)(t0 + lane) * E + e] = sigmoidf_ieee(a);
    }
}

// Large T: logits on the tensor cores (tcgen05.mma kind::f16, fp32 accumulate in TMEM). x is bf16,
// exact as an MMA operand. Each router weight is split into three bf16 values that carry its whole
// fp32 significand: hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid) (both differences
// are exact in fp32); the three products of every element accumulate into the same fp32
// accumulator. A block computes a tile of 128 tokens (M) x 64 experts (N) over one K range.
//
// The tensor cores' fp32 accumulation loses low bits at every step, so over a long K (21504
// products at H = 7168) the error would reach about 1e-4 of a logit. The accumulator is therefore
// restarted every kRtChunk stages (128 K): two TMEM buffers alternate, and drain warps add each
// finished chunk into fp32 registers (round to nearest, chunk order fixed).
//
// Roles: warp 0 issues TMA (x as bf16 in the 128-byte swizzled layout the MMA reads; the fp32
// router rows as two plain 128-byte boxes), warp 1 allocates TMEM and issues the MMAs, warps 2-9
// split the fp32 rows into the three bf16 planes (swizzled stores, then a proxy fence; two warps per
// scheduler, so that one's shared-memory latency hides behind the other's arithmetic), warps 10-13
// drain the accumulator chunks and write the result: warp w covers tokens 32 (w % 4) .. + 31. Four
// stages; every wait is bounded (a wait that runs out records kErrWaitRouter and the block winds
// down).
//
// gridDim.z splits H into slices of `hs` columns: with one split the block writes sigmoid(logit)
// to `out` ([T][E]); with several it writes its partial logits to out + z * T * E and
// router_split_reduce sums them in split order (deterministic) and applies the sigmoid.
constexpr int kRtM = 128, kRtN = 64, kRtK = 64, kRtNS = 4, kRtThreads = 448, kRtChunk = 2;
constexpr int kRtConv = 256;                    // plane-splitting threads (warps 2-9)
constexpr uint32_t kRtX = kRtM * 128;          // 16 KB: 128 tokens x 64 bf16, swizzled
constexpr uint32_t kRtW = kRtN * 256;          // 16 KB: 64 experts x 64 fp32, two boxes of 32
constexpr uint32_t kRtP = kRtN * 128;          // 8 KB: one bf16 plane, 64 experts x 64, swizzled
constexpr uint32_t kRtOffW = kRtX, kRtOffP = kRtX + kRtW;
constexpr uint32_t kRtStage = kRtX + kRtW + 3 * kRtP;   // 57344, a multiple of 1024
constexpr uint32_t kRtIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kRtN >> 3) << 17) |
                              ((uint32_t)(kRtM >> 4) << 24);   // bf16 x bf16 -> fp32, M x N
constexpr size_t kRtSmem = kRtNS * kRtStage + 1024 + 256;

__device__ __forceinline__ uint64_t rt_desc(uint32_t saddr) {   // K-major, 128-byte swizzle
    uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat16 lo, __nv_bfloat16 hi) {
    return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}

__global__ void __launch_bounds__(kRtThreads, 1)
router_logits_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w, int T, int E,
                 int H, int hs, float *__restrict__ out, int *err) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kRtNS * kRtStage);
    uint64_t *tma_full = bar, *conv_full = bar + kRtNS, *empty = bar + 2 * kRtNS, *acc_full = bar + 3 * kRtNS,
             *acc_empty = bar + 3 * kRtNS + 2, *drain = bar + 3 * kRtNS + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 3 * kRtNS + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRtNS; ++s) {
            ptx::mbar_init(ptx::smem_addr(&tma_full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&conv_full[s]), kRtConv);
            ptx::mbar_init(ptx::smem_addr(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_addr(&acc_full[b]), 1);
            ptx::mbar_init(ptx::smem_addr(&acc_empty[b]), 4);
        }
        ptx::mbar_init(ptx::smem_addr(drain), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), 2 * kRtN);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_begin();
    const int t0 = blockIdx.x * kRtM, e0 = blockIdx.y * kRtN;
    const int kb = blockIdx.z * hs, nk = (min(H, kb + hs) - kb) / kRtK;
    const int nchunk = (nk + kRtChunk - 1) / kRtChunk;
    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            ptx::prefetch_tmap(&tm_x);
            ptx::prefetch_tmap(&tm_w);
            int k = 0;
            for (; k < nk && !*abort_flag; ++k) {
                const int s = k % kRtNS;
                if (!ptx::mbar_wait(ptx::smem_addr(&empty[s]), ((k / kRtNS) & 1u) ^ 1u, err, ptx::kErrWaitRouter,
                                    abort_flag))
                    break;
                const uint32_t fb = ptx::smem_addr(&tma_full[s]), st = ptx::smem_addr(smem + s * kRtStage);
                const int kx = kb + k * kRtK;
                ptx::mbar_arrive_expect_tx(fb, kRtX + kRtW);
                ptx::tma_load_2d(st, &tm_x, kx, t0, fb);
                ptx::tma_load_2d(st + kRtOffW, &tm_w, kx, e0, fb);
                ptx::tma_load_2d(st + kRtOffW + kRtW / 2, &tm_w, kx + 32, e0, fb);
            }
            // copies still in flight after a wait gave up: let them land before the block exits
            for (int i = k > kRtNS ? k - kRtNS : 0; i < k; ++i)
                ptx::mbar_wait(ptx::smem_addr(&tma_full[i % kRtNS]), (i / kRtNS) & 1u, nullptr, 0, nullptr);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t acc = 0, d = tmem;
            for (int k = 0; k < nk && !*abort_flag; ++k) {
                const int s = k % kRtNS, c = k / kRtChunk, b = c & 1;
                if (k % kRtChunk == 0) {   // a new chunk: its buffer must have been drained
                    if (!ptx::mbar_wait(ptx::smem_addr(&acc_empty[b]), ((c >> 1) & 1u) ^ 1u, err,
                                        ptx::kErrWaitRouter, abort_flag))
                        break;
                    ptx::tc_fence_after();
                    acc = 0;
                    d = tmem + b * kRtN;
                }
                if (!ptx::mbar_wait(ptx::smem_addr(&conv_full[s]), (k / kRtNS) & 1u, err, ptx::kErrWaitRouter,
                                    abort_flag))
                    break;
                ptx::tc_fence_after();
                const uint32_t st = ptx::smem_addr(smem + s * kRtStage);
#pragma unroll
                for (int kk = 0; kk < kRtK / 16; ++kk) {
                    const uint64_t a = rt_desc(st + 32 * kk);
#pragma unroll
                    for (int pl = 0; pl < 3; ++pl) {
                        ptx::mma_bf16(d, a, rt_desc(st + kRtOffP + pl * kRtP + 32 * kk), kRtIdesc, acc);
                        acc = 1;
                    }
                }
                ptx::mma_commit(ptx::smem_addr(&empty[s]));
                if (k % kRtChunk == kRtChunk - 1 || k == nk - 1) ptx::mma_commit(ptx::smem_addr(&acc_full[b]));
            }
            ptx::mma_commit(ptx::smem_addr(drain));
            ptx::mbar_wait(ptx::smem_addr(drain), 0, nullptr, 0, nullptr);
        }
    } else if (warp < 2 + kRtConv / 32) {
        // ---------------------------------------------------------------- plane split
        const int ct = threadIdx.x - 64;   // 0..kRtConv-1
        for (int k = 0; k < nk && !*abort_flag; ++k) {
            const int s = k % kRtNS;
            if (!ptx::mbar_wait(ptx::smem_addr(&tma_full[s]), (k / kRtNS) & 1u, err, ptx::kErrWaitRouter, abort_flag))
                break;
            uint8_t *st = smem + s * kRtStage;
#pragma unroll
            for (int i = 0; i < kRtN * 8 / kRtConv; ++i) {
                const int ci = ct + kRtConv * i, r = ci >> 3, c = ci & 7;   // expert row r, 8-element chunk c
                const float4 *src = reinterpret_cast<const float4 *>(st + kRtOffW + (c >> 2) * (kRtW / 2) + r * 128 +
                                                                     (c & 3) * 32);
                const float4 u = src[0], v = src[1];
                const float w[8] = {u.x, u.y, u.z, u.w, v.x, v.y, v.z, v.w};
                uint32_t ph[4], pm[4], pl[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    __nv_bfloat16 h2[2], m2[2], l2[2];
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const float x0 = w[2 * j + q];
                        h2[q] = __float2bfloat16_rn(x0);
                        const float r1 = x0 - __bfloat162float(h2[q]);
                        m2[q] = __float2bfloat16_rn(r1);
                        l2[q] = __float2bfloat16_rn(r1 - __bfloat162float(m2[q]));
                    }
                    ph[j] = bf16x2_bits(h2[0], h2[1]);
                    pm[j] = bf16x2_bits(m2[0], m2[1]);
                    pl[j] = bf16x2_bits(l2[0], l2[1]);
                }
                const uint32_t off = r * 128 + ((c ^ (r & 7)) << 4);
                *reinterpret_cast<uint4 *>(st + kRtOffP + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
                *reinterpret_cast<uint4 *>(st + kRtOffP + kRtP + off) = make_uint4(pm[0], pm[1], pm[2], pm[3]);
                *reinterpret_cast<uint4 *>(st + kRtOffP + 2 * kRtP + off) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(ptx::smem_addr(&conv_full[s]));
        }
    } else {
        // ---------------------------------------------------------------- chunk drain and output
        const int q = warp & 3, t = t0 + 32 * q + lane;
        float sum[kRtN];
#pragma unroll
        for (int j = 0; j < kRtN; ++j) sum[j] = 0.f;
        bool ok = true;
        for (int c = 0; c < nchunk; ++c) {
            const int b = c & 1;
            if (!ptx::mbar_wait(ptx::smem_addr(&acc_full[b]), (c >> 1) & 1u, err, ptx::kErrWaitRouter, abort_flag)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
#pragma unroll
            for (int g = 0; g < kRtN / 16; ++g) {
                uint32_t r[16];
                ptx::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + b * kRtN + 16 * g, r);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) sum[16 * g + j] += __uint_as_float(r[j]);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&acc_empty[b]));
        }
        if (ok && t < T) {
            const bool split = gridDim.z > 1;
            float *dst = out + (split ? (size_t)blockIdx.z * T * E : 0) + (size_t)t * E;
#pragma unroll
            for (int j = 0; j < kRtN; ++j) {
                const int e = e0 + j;
                if (e < E) dst[e] = split ? sum[j] : sigmoidf_ieee(sum[j]);
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 2 * kRtN);
    }
}

__global__ void __launch_bounds__(256)
router_split_reduce(const float *__restrict__ part, int n, int splits, float *__restrict__ scores) {
    pdl_begin();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        float a = part[i];
        for (int z = 1; z < splits; ++z) a += part[(size_t)z * n + i];
        scores[i] = sigmoidf_ieee(a);
    }
}

// Top-k: one warp per token (topk_token).
template <int NPL>
__global__ void __launch_bounds__(256)
router_topk(const float *__restrict__ scores, const float *__restrict__ bias, int T, int E, int top_k,
            int32_t *__restrict__ idx, float *__restrict__ w, int32_t *__restrict__ zero, int n_zero) {
    pdl_begin();
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < n_zero; i += blockDim.x) zero[i] = 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    topk_token<NPL>(scores, bias, E, top_k, t, lane, idx, w, nullptr);
}

}  // namespace

int launch_router(const __nv_bfloat16 *x, int T, int H, const float *router_w, const float *router_b,
                  int E, int top_k, float *scores, int32_t *idx, float *w, float *partial,
                  int num_sms, int32_t *zero, int n_zero, int *err, cudaStream_t st, bool with_topk) {
    int n = 0;
    if (!zero) n_zero = 0;
    if (T < 64) {
        dim3 grid(E, (T + kSmallTok - 1) / kSmallTok);
        launch_pdl(router_logits_small, grid, dim3(kSmallWarps * 32), 0, st, x, T, H, router_w, E, scores);
        ++n;
    } else {
        const int tiles = ((T + kRtM - 1) / kRtM) * ((E + kRtN - 1) / kRtN);
        int splits = (num_sms + tiles - 1) / tiles;                // one block per SM
        splits = std::min(splits, std::max(1, H / (8 * kRtK)));   // at least 8 K chunks per split
        // the partials fit the fixed cap, whatever buffer the caller holds beyond it
        splits = (int)std::min<size_t>((size_t)splits, std::max<size_t>(1, kRouterPartialFloats / ((size_t)T * E)));
        const int chunks = H / kRtK;
        const int hs = ((chunks + splits - 1) / splits) * kRtK;
        splits = (H + hs - 1) / hs;
        CUtensorMap mx, mw;
        if (!tensor_map_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, H, T, (uint64_t)H * 2, kRtK, kRtM,
                           CU_TENSOR_MAP_SWIZZLE_128B) ||
            !tensor_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, router_w, H, E, (uint64_t)H * 4, 32, kRtN,
                           CU_TENSOR_MAP_SWIZZLE_NONE))
            return -1;
        static bool attr = false;
        if (!attr) {
            if (cudaFuncSetAttribute(router_logits_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRtSmem) !=
                cudaSuccess)
                return -1;
            attr = true;
        }
        dim3 grid((T + kRtM - 1) / kRtM, (E + kRtN - 1) / kRtN, splits);
        launch_pdl(router_logits_tc, grid, dim3(kRtThreads), kRtSmem, st, mx, mw, T, E, H, hs,
                   splits > 1 ? partial : scores, err);
        ++n;
        if (splits > 1) {
            const int cnt = T * E;
            launch_pdl(router_split_reduce, dim3(std::min((cnt + 255) / 256, 4 * num_sms)), dim3(256), 0, st,
                       (const float *)partial, cnt, splits, scores);
            ++n;
        }
    }
    if (!with_topk) return cudaPeekAtLastError() == cudaSuccess ? n : -1;
    const int npl = (E + 31) / 32;
    const dim3 grid((T + 7) / 8);
    auto topk = npl <= 1 ? router_topk<1> : npl <= 2 ? router_topk<2> : npl <= 4 ? router_topk<4>
              : npl <= 8 ? router_topk<8> : npl <= 16 ? router_topk<16> : router_topk<32>;
    launch_pdl(topk, grid, dim3(256), 0, st, (const float *)scores, router_b, T, E, top_k, idx, w, zero, n_zero);
    ++n;
    return cudaPeekAtLastError() == cudaSuccess ? n : -1;
}

}  // namespace colimoe
