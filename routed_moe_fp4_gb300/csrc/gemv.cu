// A3/A4 for small token counts: weight-streaming GEMV kernels over the touched experts.
//
// gate/up: h[row][i] = silu(g) * u, g = sum_k Wg[i][k] x[row][k], u = sum_k Wu[i][k] x[row][k]
//          ("DeepSeek V4 Flash CPU inference with NVMe expert streaming": the dual gate+up
//          matvec; FP4 E2M1 experts with UE8M0 group-32 scales)
// down:    y[row][m] = sum_i Wd[m][i] h[row][i]
//
// Work is a flat list of (touched group, block of weight rows) items; each block walks a
// contiguous range of it, so every block streams the same number of weight bytes. A warp owns
// four weight rows; lane l reads the 16-byte code chunks l, l+32, ... of each row (one chunk =
// one 32-element scale group), so a warp reads 512 contiguous bytes per row per step.
//
// Arithmetic: each activation row is staged in shared memory as fp16 after multiplying it by a
// power of two that puts its largest magnitude in [2^8, 2^9) (exact; undone at the end). E2M1
// codes become exact fp16 pairs (cvt.rn.f16x2.e2m1x2); the products of one 32-element group
// are accumulated with HFMA2 (16 terms per half, |sum| < 6 * 2^9 * 16 < 65504), then converted
// to fp32, scaled by the group's UE8M0 factor (fp32 bits s << 23) and summed in fp32.
#include "colimoe_internal.cuh"

namespace colimoe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTB = 2;                    // tokens per staged chunk
constexpr int kGateUpI = 2 * kWarps;      // i-values per gate/up item (2 per warp)
constexpr int kDownM = 4 * kWarps;        // output rows per down item (4 per warp)

__device__ __forceinline__ void e2m1x8_to_h2(uint32_t w, uint32_t (&o)[4]) {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]) : "r"(w));
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ float h2_sum(uint32_t v) {
    const __half2 h = *reinterpret_cast<const __half2 *>(&v);
    const float2 f = __half22float2(h);
    return f.x + f.y;
}

__device__ __forceinline__ float ue8m0(uint32_t s) { return __uint_as_float(s << 23); }

__device__ __forceinline__ uint4 ld_stream(const uint8_t *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Stages rows [0, n) of `src` (bf16, K used columns, row stride `ld` elements) into xs as fp16,
// layout [kTB][4][K/32] of 16-byte units: unit (q, c) of token t holds elements 32c + 8q ..
// 32c + 8q + 7. Missing rows are zero. inv[t] receives the power of two that undoes the staging
// scale.
__device__ void stage_rows(const __nv_bfloat16 *__restrict__ src, int n, int K, int ld, uint4 *xs, float *inv) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NC = K / 32;
    if (warp < kTB) {
        const int t = warp;
        uint4 *dst = xs + (size_t)t * 4 * NC;
        if (t >= n) {
            for (int v = lane; v < K / 8; v += 32) dst[(v & 3) * NC + (v >> 2)] = make_uint4(0, 0, 0, 0);
            if (lane == 0) inv[t] = 0.f;
            return;
        }
        const uint4 *row = reinterpret_cast<const uint4 *>(src + (size_t)t * ld);
        uint32_t mx = 0;   // max |bf16| bit pattern (monotone for non-negative floats)
        for (int v = lane; v < K / 8; v += 32) {
            const uint4 q = row[v];
            const uint32_t a[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                mx = max(mx, a[i] & 0x7FFFu);
                mx = max(mx, (a[i] >> 16) & 0x7FFFu);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        // exponent of the largest magnitude; scale = 2^(8 - e) clamped to the normal fp32 range
        const int e = (int)((mx >> 7) & 0xFF) - 127;
        int se = 8 - e;
        se = max(-126, min(126, se));
        const float scale = (mx == 0 || mx >= 0x7F80u) ? 1.0f : __uint_as_float((uint32_t)(se + 127) << 23);
        if (lane == 0) inv[t] = (mx == 0 || mx >= 0x7F80u) ? 1.0f : __uint_as_float((uint32_t)(127 - se) << 23);
        for (int v = lane; v < K / 8; v += 32) {
            const uint4 q = row[v];
            const uint32_t a[4] = {q.x, q.y, q.z, q.w};
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float lo = __uint_as_float(a[i] << 16) * scale;
                const float hi = __uint_as_float(a[i] & 0xFFFF0000u) * scale;
                const __half2 hv = __floats2half2_rn(lo, hi);
                o[i] = *reinterpret_cast<const uint32_t *>(&hv);
            }
            dst[(v & 3) * NC + (v >> 2)] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// Dot products of four weight rows with NT staged tokens. rowp[r] points at the code bytes of
// row r, sclp[r] at its scale bytes. Returns warp-reduced sums in acc (valid on every lane).
template <int NT>
__device__ __forceinline__ void rows4_dot(const uint8_t *const (&rowp)[4], const uint8_t *const (&sclp)[4],
                                          int NC, const uint4 *xs, float (&acc)[4][NT]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
    int c = lane;
    uint4 cur[4];
    uint32_t csc[4];
    if (c < NC) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            cur[r] = ld_stream(rowp[r] + (size_t)c * 16);
            csc[r] = __ldg(sclp[r] + c);
        }
    }
    for (; c < NC; c += 32) {
        uint4 nxt[4];
        uint32_t nsc[4];
        const bool more = c + 32 < NC;
        if (more) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                nxt[r] = ld_stream(rowp[r] + (size_t)(c + 32) * 16);
                nsc[r] = __ldg(sclp[r] + c + 32);
            }
        }
        uint32_t hacc[4][NT];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int t = 0; t < NT; ++t) hacc[r][t] = 0u;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 xv[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) xv[t] = xs[(size_t)t * 4 * NC + q * NC + c];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint32_t word = q == 0 ? cur[r].x : q == 1 ? cur[r].y : q == 2 ? cur[r].z : cur[r].w;
                uint32_t v[4];
                e2m1x8_to_h2(word, v);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    hacc[r][t] = hfma2_u32(v[0], xv[t].x, hacc[r][t]);
                    hacc[r][t] = hfma2_u32(v[1], xv[t].y, hacc[r][t]);
                    hacc[r][t] = hfma2_u32(v[2], xv[t].z, hacc[r][t]);
                    hacc[r][t] = hfma2_u32(v[3], xv[t].w, hacc[r][t]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float s = ue8m0(csc[r]);
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[r][t] = fmaf(s, h2_sum(hacc[r][t]), acc[r][t]);
        }
        if (more) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                cur[r] = nxt[r];
                csc[r] = nsc[r];
            }
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[r][t] = warp_sum(acc[r][t]);
}

template <int NT>
__device__ __forceinline__ void gateup_item(const FfnArgs &a, const uint8_t *gu_c, const uint8_t *gu_s, int Ig,
                                            int i, int out_row0, const uint4 *xs, const float *inv) {
    const int lane = threadIdx.x & 31;
    const int H = a.H;
    const uint8_t *rowp[4] = {gu_c + (size_t)i * (H / 2), gu_c + (size_t)(i + 1) * (H / 2),
                              gu_c + (size_t)(Ig + i) * (H / 2), gu_c + (size_t)(Ig + i + 1) * (H / 2)};
    const uint8_t *sclp[4] = {gu_s + (size_t)i * (H / 32), gu_s + (size_t)(i + 1) * (H / 32),
                              gu_s + (size_t)(Ig + i) * (H / 32), gu_s + (size_t)(Ig + i + 1) * (H / 32)};
    float acc[4][NT];
    rows4_dot<NT>(rowp, sclp, H / 32, xs, acc);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int ii = 0; ii < 2; ++ii) {
            if (lane == t * 2 + ii) {
                const float g = acc[ii][t] * inv[t];
                const float u = acc[2 + ii][t] * inv[t];
                const float hval = __fdiv_rn(g, 1.0f + expf(-g)) * u;
                a.h[(size_t)(out_row0 + t) * a.I_max + i + ii] = __float2bfloat16_rn(hval);
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads, 2)
gemv_gateup(FfnArgs a, int items_per_group) {
    extern __shared__ uint4 smem[];
    uint4 *xs = smem;
    float *inv = reinterpret_cast<float *>(smem + (size_t)kTB * 4 * (a.H / 32));
    const long total = (long)(*a.n_touched) * items_per_group;
    const long beg = total * blockIdx.x / gridDim.x;
    const long end = total * (blockIdx.x + 1) / gridDim.x;
    const int warp = threadIdx.x >> 5;
    int staged_g = -1, staged_n0 = -1;
    for (long it = beg; it < end; ++it) {
        const int g = a.touched[it / items_per_group];
        const int i0 = (int)(it % items_per_group) * kGateUpI;
        const bool sh = g == a.E;
        const int Ig = sh ? a.I_s : a.I;
        if (i0 >= Ig) continue;
        const ExpertSet &es = sh ? a.shared : a.routed;
        const size_t ge = sh ? 0 : (size_t)g;
        const uint8_t *gu_c = es.gu_codes + ge * 2 * Ig * (a.H / 2);
        const uint8_t *gu_s = es.gu_scales + ge * 2 * Ig * (a.H / 32);
        const int r0 = a.off[g], n = a.cnt[g];
        for (int n0 = 0; n0 < n; n0 += kTB) {
            if (g != staged_g || n0 != staged_n0) {
                __syncthreads();
                stage_rows(a.xp + (size_t)(r0 + n0) * a.H, min(kTB, n - n0), a.H, a.H, xs, inv);
                __syncthreads();
                staged_g = g;
                staged_n0 = n0;
            }
            const int nt = min(kTB, n - n0);
            const int i = i0 + warp * 2;
            if (nt == 1) gateup_item<1>(a, gu_c, gu_s, Ig, i, r0 + n0, xs, inv);
            else gateup_item<2>(a, gu_c, gu_s, Ig, i, r0 + n0, xs, inv);
        }
    }
}

template <int NT>
__device__ __forceinline__ void down_item(const FfnArgs &a, const uint8_t *d_c, const uint8_t *d_s, int Ig,
                                          int m, int out_row0, const uint4 *xs, const float *inv) {
    const int lane = threadIdx.x & 31;
    const uint8_t *rowp[4], *sclp[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        rowp[r] = d_c + (size_t)(m + r) * (Ig / 2);
        sclp[r] = d_s + (size_t)(m + r) * (Ig / 32);
    }
    float acc[4][NT];
    rows4_dot<NT>(rowp, sclp, Ig / 32, xs, acc);
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int r = 0; r < 4; ++r)
            if (lane == t * 4 + r) a.y[(size_t)(out_row0 + t) * a.H + m + r] = acc[r][t] * inv[t];
}

__global__ void __launch_bounds__(kThreads, 2)
gemv_down(FfnArgs a, int items_per_group) {
    extern __shared__ uint4 smem[];
    uint4 *xs = smem;
    float *inv = reinterpret_cast<float *>(smem + (size_t)kTB * 4 * (a.I_max / 32));
    const long total = (long)(*a.n_touched) * items_per_group;
    const long beg = total * blockIdx.x / gridDim.x;
    const long end = total * (blockIdx.x + 1) / gridDim.x;
    const int warp = threadIdx.x >> 5;
    int staged_g = -1, staged_n0 = -1;
    for (long it = beg; it < end; ++it) {
        const int g = a.touched[it / items_per_group];
        const int m0 = (int)(it % items_per_group) * kDownM;
        const bool sh = g == a.E;
        const int Ig = sh ? a.I_s : a.I;
        const ExpertSet &es = sh ? a.shared : a.routed;
        const size_t ge = sh ? 0 : (size_t)g;
        const uint8_t *d_c = es.d_codes + ge * (size_t)a.H * (Ig / 2);
        const uint8_t *d_s = es.d_scales + ge * (size_t)a.H * (Ig / 32);
        const int r0 = a.off[g], n = a.cnt[g];
        for (int n0 = 0; n0 < n; n0 += kTB) {
            if (g != staged_g || n0 != staged_n0) {
                __syncthreads();
                // h rows have stride I_max; stage the first Ig columns of each
                stage_rows(a.h + (size_t)(r0 + n0) * a.I_max, min(kTB, n - n0), Ig, a.I_max, xs, inv);
                __syncthreads();
                staged_g = g;
                staged_n0 = n0;
            }
            const int nt = min(kTB, n - n0);
            const int m = m0 + warp * 4;
            if (nt == 1) down_item<1>(a, d_c, d_s, Ig, m, r0 + n0, xs, inv);
            else down_item<2>(a, d_c, d_s, Ig, m, r0 + n0, xs, inv);
        }
    }
}

}  // namespace

int launch_ffn_gemv(const FfnArgs &a, int num_sms, cudaEvent_t mid, cudaStream_t st) {
    const int blocks = 2 * num_sms;
    const size_t smem_gu = (size_t)kTB * 4 * (a.H / 32) * sizeof(uint4) + kTB * sizeof(float);
    const size_t smem_dn = (size_t)kTB * 4 * (a.I_max / 32) * sizeof(uint4) + kTB * sizeof(float);
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(gemv_gateup, cudaFuncAttributeMaxDynamicSharedMemorySize, 100 * 1024);
        cudaFuncSetAttribute(gemv_down, cudaFuncAttributeMaxDynamicSharedMemorySize, 100 * 1024);
        attr_set = true;
    }
    const int gu_items = (max(a.I, a.I_s) + kGateUpI - 1) / kGateUpI;
    gemv_gateup<<<blocks, kThreads, smem_gu, st>>>(a, gu_items);
    if (mid) cudaEventRecord(mid, st);
    const int dn_items = a.H / kDownM;
    gemv_down<<<blocks, kThreads, smem_dn, st>>>(a, dn_items);
    return cudaPeekAtLastError() == cudaSuccess ? 2 : -1;
}

}  // namespace colimoe
