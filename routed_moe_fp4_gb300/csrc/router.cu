// A1 router: fp32 logits, sigmoid scores, bias-adjusted top-k with warp shuffles, renormalised
// weights ("the CUDA tier wired into the DeepSeek V4 engine", What it is: route on device).
//
// logits[t][e] = sum_h x[t][h] * Wr[e][h] in fp32 (x is bf16, exact in fp32); s = 1/(1+exp(-z)).
// key = fp32(s + b); the top_k largest keys in descending order, bit-identical keys going to
// the lower expert index; w_j = s_j / S, S the fp32 sum of the chosen s in slot order, one
// IEEE division each. Built without fast-math: every add, divide and expf is the IEEE/accurate one.
#include "colimoe_internal.cuh"
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

// Large T: a 64 tokens x 64 experts tile per block, 4 x 4 outputs per thread, K chunks of 32.
constexpr int kTileT = 64, kTileE = 64, kTileK = 32;

// gridDim.z splits H into slices of `hs` columns: with one split the block writes sigmoid(logit)
// to `out` ([T][E]); with several it writes its partial logits to out + z * T * E and
// router_split_reduce sums them in split order (deterministic) and applies the sigmoid.
__global__ void __launch_bounds__(256)
router_logits_tiled(const __nv_bfloat16 *__restrict__ x, int T, int H, const float *__restrict__ wr,
                    int E, int hs, float *__restrict__ out) {
    pdl_begin();
    __shared__ float xs[kTileK][kTileT + 4];
    __shared__ float ws[kTileK][kTileE + 4];
    const int tid = threadIdx.x;
    const int tt = blockIdx.x * kTileT, ee = blockIdx.y * kTileE;
    const int kb = blockIdx.z * hs, ke = min(H, kb + hs);
    const bool split = gridDim.z > 1;
    const int ty = tid / 16, tx = tid % 16;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    const int lr = tid / 4, lk = (tid % 4) * 8;   // loader: row (token / expert), 8 k values
    for (int k0 = kb; k0 < ke; k0 += kTileK) {
        {   // x tile: 64 tokens x 32 k as bf16 -> fp32, transposed
            const int t = tt + lr;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (t < T) v = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)t * H + k0 + lk));
            xs[lk + 0][lr] = bf16_lo(v.x); xs[lk + 1][lr] = bf16_hi(v.x);
            xs[lk + 2][lr] = bf16_lo(v.y); xs[lk + 3][lr] = bf16_hi(v.y);
            xs[lk + 4][lr] = bf16_lo(v.z); xs[lk + 5][lr] = bf16_hi(v.z);
            xs[lk + 6][lr] = bf16_lo(v.w); xs[lk + 7][lr] = bf16_hi(v.w);
        }
        {   // router tile: 64 experts x 32 k, transposed
            const int e = ee + lr;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (e < E) {
                const float4 *p = reinterpret_cast<const float4 *>(wr + (size_t)e * H + k0 + lk);
                a = __ldg(p);
                b = __ldg(p + 1);
            }
            ws[lk + 0][lr] = a.x; ws[lk + 1][lr] = a.y; ws[lk + 2][lr] = a.z; ws[lk + 3][lr] = a.w;
            ws[lk + 4][lr] = b.x; ws[lk + 5][lr] = b.y; ws[lk + 6][lr] = b.z; ws[lk + 7][lr] = b.w;
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < kTileK; ++k) {
            const float4 av = *reinterpret_cast<const float4 *>(&xs[k][ty * 4]);
            const float4 bv = *reinterpret_cast<const float4 *>(&ws[k][tx * 4]);
            const float a[4] = {av.x, av.y, av.z, av.w};
            const float b[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    float *dst = out + (split ? (size_t)blockIdx.z * T * E : 0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = tt + ty * 4 + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = ee + tx * 4 + j;
            if (e < E) dst[(size_t)t * E + e] = split ? acc[i][j] : sigmoidf_ieee(acc[i][j]);
        }
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
                  int E, int top_k, float *scores, int32_t *idx, float *w, float *partial, size_t partial_floats,
                  int num_sms, int32_t *zero, int n_zero, cudaStream_t st, bool with_topk) {
    int n = 0;
    if (!zero) n_zero = 0;
    if (T < 64) {
        dim3 grid(E, (T + kSmallTok - 1) / kSmallTok);
        launch_pdl(router_logits_small, grid, dim3(kSmallWarps * 32), 0, st, x, T, H, router_w, E, scores);
        ++n;
    } else {
        const int tiles = ((T + kTileT - 1) / kTileT) * ((E + kTileE - 1) / kTileE);
        int splits = (2 * num_sms + tiles - 1) / tiles;          // aim for two blocks per SM
        splits = std::min(splits, std::max(1, H / (8 * kTileK)));  // at least 8 K chunks per split
        while (splits > 1 && (size_t)splits * T * E > partial_floats) --splits;
        const int chunks = H / kTileK;
        const int hs = ((chunks + splits - 1) / splits) * kTileK;
        splits = (H + hs - 1) / hs;
        dim3 grid((T + kTileT - 1) / kTileT, (E + kTileE - 1) / kTileE, splits);
        launch_pdl(router_logits_tiled, grid, dim3(256), 0, st, x, T, H, router_w, E, hs,
                   splits > 1 ? partial : scores);
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
