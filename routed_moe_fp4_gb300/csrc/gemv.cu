// A3/A4 for small token counts: weight-streaming GEMV kernels over the touched experts.
//
// gate/up: h[row][i] = silu(g) * u, g = sum_k Wg[i][k] x[row][k], u = sum_k Wu[i][k] x[row][k]
//          ("DeepSeek V4 Flash CPU inference with NVMe expert streaming": the dual gate+up
//          matvec; FP4 E2M1 experts with UE8M0 group-32 scales)
// down:    y[row][m] = sum_i Wd[m][i] h[row][i]
//
// Structure: one persistent block per SM walks a contiguous range of a flat list of (touched
// group, block of weight rows) items, so every block streams about the same number of weight
// bytes. A producer warp streams each item's code and scale rows (contiguous in the packed
// layout) into a ring of shared-memory stages with 1-D bulk TMA copies; eight consumer warps
// take a stage when its mbarrier completes, compute, and release it. Every wait is bounded.
//
// Arithmetic: activation rows are pre-scaled by a power of two that puts their largest magnitude
// in [2^8, 2^9) and stored as fp16 (undone at the end). A bf16 element keeps its value exactly
// unless it lies more than about 2^22 below the row's largest magnitude, where fp16 holds it as a
// subnormal with fewer significant bits or flushes it to zero; such elements contribute below
// 2^-22 of the row's scale to any sum, which the error bar of the layer absorbs. E2M1 codes become
// exact fp16 pairs (cvt.rn.f16x2.e2m1x2); the products of one 32-element group are summed with
// HFMA2 in two chains (8 terms per half each, |sum| < 6 * 2^9 * 8 < 65504), converted to fp32,
// scaled by the group's UE8M0 factor (fp32 bits s << 23) and summed in fp32. Blocks split the
// items by cost (one unit per weight pass plus one per 4-token pass over the stage), so a group
// with many rows, such as the shared expert, does not leave a long tail on a few blocks.
//
// Activation layout (fp16 rows, K elements, NC = K/32): 16-byte unit (q, c), holding elements
// 32c + 8q .. 32c + 8q + 7, sits at unit index q * NC + c, so lane c of a warp reads unit
// q * NC + c for q = 0..3 and each load instruction covers 512 contiguous bytes.
#include "colimoe_internal.cuh"
#include "sm103_ptx.cuh"

namespace colimoe {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kIB = kConsumerWarps;            // i-values per gate/up item (one per consumer warp)
constexpr int kMB = 4 * kConsumerWarps;        // output rows per down item (four per consumer warp)
constexpr int kTB = kGemvCostTokens;           // tokens per pass over a resident stage
constexpr uint32_t kSmemBudget = 200 * 1024;

enum Mode { kGateUp = 0, kDown = 1 };

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
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&v));
    return f.x + f.y;
}

__device__ __forceinline__ float ue8m0(uint32_t s) { return __uint_as_float(s << 23); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

struct ItemInfo {
    int g, blk, Ig;
    bool valid;
    const ExpertSet *es;
    size_t ge;
};

template <int MODE>
__device__ __forceinline__ ItemInfo decode_item(const FfnArgs &a, long it, int ipg) {
    ItemInfo r;
    r.g = a.touched[it / ipg];
    r.blk = (int)(it % ipg);
    const bool sh = r.g == a.E;
    r.Ig = sh ? a.I_s : a.I;
    r.es = sh ? &a.shared : &a.routed;
    r.ge = sh ? 0 : (size_t)r.g;
    r.valid = MODE == kGateUp ? r.blk * kIB < r.Ig : true;
    return r;
}

// Dot products of R weight rows (codes/scales in shared memory) with NT activation rows (global,
// permuted fp16 layout). Returns warp-reduced sums (valid on every lane).
template <int R, int NT>
__device__ __forceinline__ void dot_rows(const uint8_t *const (&codes)[R], const uint8_t *const (&scales)[R], int NC,
                                         const uint4 *const (&xrow)[NT], float (&acc)[R][NT]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
    for (int c = lane; c < NC; c += 32) {
        uint4 cw[R];
        float sc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            cw[r] = *reinterpret_cast<const uint4 *>(codes[r] + (size_t)c * 16);
            sc[r] = ue8m0(scales[r][c]);
        }
        uint32_t hacc[R][NT], hacc2[R][NT];   // two chains per (row, token) for ILP
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int t = 0; t < NT; ++t) hacc[r][t] = hacc2[r][t] = 0u;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 xv[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) xv[t] = __ldg(xrow[t] + q * NC + c);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t word = q == 0 ? cw[r].x : q == 1 ? cw[r].y : q == 2 ? cw[r].z : cw[r].w;
                uint32_t v[4];
                e2m1x8_to_h2(word, v);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    hacc[r][t] = hfma2_u32(v[0], xv[t].x, hacc[r][t]);
                    hacc2[r][t] = hfma2_u32(v[1], xv[t].y, hacc2[r][t]);
                    hacc[r][t] = hfma2_u32(v[2], xv[t].z, hacc[r][t]);
                    hacc2[r][t] = hfma2_u32(v[3], xv[t].w, hacc2[r][t]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int t = 0; t < NT; ++t)
                acc[r][t] = fmaf(sc[r], h2_sum(hacc[r][t]) + h2_sum(hacc2[r][t]), acc[r][t]);
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[r][t] = warp_sum(acc[r][t]);
}

template <int NT>
__device__ __forceinline__ void gateup_compute(const FfnArgs &a, const uint8_t *stage, const ItemInfo &itm, int r0,
                                               int n0) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, NC = H / 32;
    const uint8_t *codes[2] = {stage + (size_t)warp * (H / 2), stage + (size_t)(kIB + warp) * (H / 2)};
    const uint8_t *sbase = stage + (size_t)2 * kIB * (H / 2);
    const uint8_t *scales[2] = {sbase + (size_t)warp * NC, sbase + (size_t)(kIB + warp) * NC};
    const uint4 *xrow[NT];
    int tok[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        tok[t] = a.src_token[r0 + n0 + t];
        xrow[t] = reinterpret_cast<const uint4 *>(a.xh + (size_t)tok[t] * H);
    }
    float acc[2][NT];
    dot_rows<2, NT>(codes, scales, NC, xrow, acc);
    const int i = itm.blk * kIB + warp;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        if (lane == t) {
            const float inv = a.xinv[tok[t]];
            const float g = acc[0][t] * inv, u = acc[1][t] * inv;
            const float hval = __fdiv_rn(g, 1.0f + expf(-g)) * u;
            a.h[(size_t)(r0 + n0 + t) * a.I_max + i] = __float2bfloat16_rn(hval);
        }
    }
}

template <int NT>
__device__ __forceinline__ void down_compute(const FfnArgs &a, const uint8_t *stage, const ItemInfo &itm, int r0,
                                             int n0) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Ig = itm.Ig, NC = Ig / 32;
    const uint8_t *codes[4], *scales[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        codes[r] = stage + (size_t)(4 * warp + r) * (Ig / 2);
        scales[r] = stage + (size_t)kMB * (Ig / 2) + (size_t)(4 * warp + r) * NC;
    }
    const uint4 *xrow[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) xrow[t] = reinterpret_cast<const uint4 *>(a.hh + (size_t)(r0 + n0 + t) * a.I_max);
    float acc[4][NT];
    dot_rows<4, NT>(codes, scales, NC, xrow, acc);
    const int m = itm.blk * kMB + 4 * warp;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int r = 0; r < 4; ++r)
            if (lane == t * 4 + r) a.y[(size_t)(r0 + n0 + t) * a.H + m + r] = acc[r][t] * a.hinv[r0 + n0 + t];
}

// First flat item index (group-major, ipg items per group) whose cost start is >= target, where
// item (u, b) of touched group u starts at ipg * P[u] + b * (P[u+1] - P[u]) cost units.
// Executed by one full warp; the result is valid on every lane.
__device__ long item_at_cost(const int32_t *__restrict__ P, int nt, int ipg, long target) {
    const int lane = threadIdx.x & 31;
    if (nt <= 0) return 0;
    int lo = 0, hi = nt;                 // find the last u in [0, nt) with ipg * P[u] <= target
    while (hi - lo > 1) {
        const int step = (hi - lo + 31) / 32;
        const int u = lo + lane * step;
        const bool ok = u < hi && (long)ipg * P[u] <= target;
        const unsigned b = __ballot_sync(0xffffffffu, ok);
        const int last = 31 - __clz(b);  // lane 0 always qualifies (P[lo] <= target holds)
        lo = lo + last * step;
        hi = min(hi, lo + step);
    }
    const long c0 = (long)ipg * P[lo];
    const int per = P[lo + 1] - P[lo];
    long b = (target - c0 + per - 1) / per;
    if (b >= ipg) return (long)(lo + 1) * ipg;
    return (long)lo * ipg + b;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
gemv_tma(FfnArgs a, int ipg, int nst, uint32_t stage_stride) {
    pdl_trigger();
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)nst * stage_stride);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * nst);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    long *range = reinterpret_cast<long *>(bars + 2 * nst + 1);
    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            ptx::mbar_init(ptx::smem_addr(&bars[s]), 1);                       // full: producer
            ptx::mbar_init(ptx::smem_addr(&bars[nst + s]), kConsumerWarps);    // empty: consumers
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    pdl_wait();   // everything above is on-chip set-up
    if (warp == 0) {   // this block's share of the total cost, as a range of flat items
        const int nt = *a.n_touched;
        const long total = (long)ipg * a.touched_cost[nt];
        const long b0 = item_at_cost(a.touched_cost, nt, ipg, total * blockIdx.x / gridDim.x);
        const long b1 = item_at_cost(a.touched_cost, nt, ipg, total * (blockIdx.x + 1) / gridDim.x);
        if (lane == 0) {
            range[0] = b0;
            range[1] = b1;
        }
    }
    __syncthreads();
    const long beg = range[0], end = range[1];
    const int H = a.H;
    int issued = 0;

    if (warp == kConsumerWarps) {
        if (lane == 0) {   // producer
            const uint64_t pol = ptx::policy_evict_first();
            for (long it = beg; it < end; ++it) {
                const ItemInfo itm = decode_item<MODE>(a, it, ipg);
                if (!itm.valid) continue;
                const int slot = issued % nst;
                const uint32_t ph = (uint32_t)(issued / nst) & 1u;
                if (!ptx::mbar_wait(ptx::smem_addr(&bars[nst + slot]), ph ^ 1u, a.err, ptx::kErrWaitEmpty, abort_flag))
                    break;
                const uint32_t full = ptx::smem_addr(&bars[slot]);
                const uint32_t dst = ptx::smem_addr(smem + (size_t)slot * stage_stride);
                if (MODE == kGateUp) {
                    const int Ig = itm.Ig, i0 = itm.blk * kIB;
                    const uint8_t *gc = itm.es->gu_codes + itm.ge * 2 * Ig * (size_t)(H / 2);
                    const uint8_t *gs = itm.es->gu_scales + itm.ge * 2 * Ig * (size_t)(H / 32);
                    const uint32_t cb = kIB * (H / 2), sb = kIB * (H / 32);
                    ptx::mbar_arrive_expect_tx(full, 2 * (cb + sb));
                    ptx::bulk_g2s_hint(dst, gc + (size_t)i0 * (H / 2), cb, full, pol);
                    ptx::bulk_g2s_hint(dst + cb, gc + (size_t)(Ig + i0) * (H / 2), cb, full, pol);
                    ptx::bulk_g2s_hint(dst + 2 * cb, gs + (size_t)i0 * (H / 32), sb, full, pol);
                    ptx::bulk_g2s_hint(dst + 2 * cb + sb, gs + (size_t)(Ig + i0) * (H / 32), sb, full, pol);
                } else {
                    const int Ig = itm.Ig, m0 = itm.blk * kMB;
                    const uint8_t *dc = itm.es->d_codes + itm.ge * (size_t)H * (Ig / 2);
                    const uint8_t *ds = itm.es->d_scales + itm.ge * (size_t)H * (Ig / 32);
                    const uint32_t cb = kMB * (Ig / 2), sb = kMB * (Ig / 32);
                    ptx::mbar_arrive_expect_tx(full, cb + sb);
                    ptx::bulk_g2s_hint(dst, dc + (size_t)m0 * (Ig / 2), cb, full, pol);
                    ptx::bulk_g2s_hint(dst + cb, ds + (size_t)m0 * (Ig / 32), sb, full, pol);
                }
                ++issued;
            }
        }
    } else {   // consumers
        int used = 0;
        for (long it = beg; it < end; ++it) {
            const ItemInfo itm = decode_item<MODE>(a, it, ipg);
            if (!itm.valid) continue;
            const int slot = used % nst;
            const uint32_t ph = (uint32_t)(used / nst) & 1u;
            if (!ptx::mbar_wait(ptx::smem_addr(&bars[slot]), ph, a.err, ptx::kErrWaitFull, abort_flag)) break;
            const uint8_t *stage = smem + (size_t)slot * stage_stride;
            const int r0 = a.off[itm.g], n = a.cnt[itm.g];
            for (int n0 = 0; n0 < n; n0 += kTB) {
                const int nt = min(kTB, n - n0);
                if (MODE == kGateUp) {
                    if (nt == 1) gateup_compute<1>(a, stage, itm, r0, n0);
                    else if (nt == 2) gateup_compute<2>(a, stage, itm, r0, n0);
                    else if (nt == 3) gateup_compute<3>(a, stage, itm, r0, n0);
                    else gateup_compute<4>(a, stage, itm, r0, n0);
                } else {
                    if (nt == 1) down_compute<1>(a, stage, itm, r0, n0);
                    else if (nt == 2) down_compute<2>(a, stage, itm, r0, n0);
                    else if (nt == 3) down_compute<3>(a, stage, itm, r0, n0);
                    else down_compute<4>(a, stage, itm, r0, n0);
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&bars[nst + slot]));
            ++used;
        }
    }
    __syncthreads();
    // After an abort the producer waits (bounded) for the copies it issued, so no TMA write
    // lands in shared memory after the block has exited.
    if (*abort_flag && warp == kConsumerWarps && lane == 0) {
        for (int j = issued > nst ? issued - nst : 0; j < issued; ++j)
            ptx::mbar_wait(ptx::smem_addr(&bars[j % nst]), (uint32_t)(j / nst) & 1u, nullptr, 0, nullptr);
    }
}

// Rows of bf16 -> fp16 scaled by a power of two (largest magnitude in [2^8, 2^9)), written in the
// permuted unit layout; inv[row] receives the inverse scale. One warp per row. Rows >= split use
// K2 columns, the others K1.
__global__ void __launch_bounds__(256)
prep_rows_f16(const __nv_bfloat16 *__restrict__ src, int src_ld, int nrows, int K1, int split, int K2,
              __half *__restrict__ dst, int dst_ld, float *__restrict__ inv) {
    pdl_begin();
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= nrows) return;
    const int K = row >= split ? K2 : K1;
    const int NC = K / 32;
    const uint4 *in = reinterpret_cast<const uint4 *>(src + (size_t)row * src_ld);
    uint4 *out = reinterpret_cast<uint4 *>(dst + (size_t)row * dst_ld);
    uint32_t mx = 0;
    for (int v = lane; v < K / 8; v += 32) {
        const uint4 q = in[v];
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) mx = max(mx, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const bool plain = mx == 0 || mx >= 0x7F80u;   // all zero, or inf/nan present: no scaling
    int se = 8 - ((int)((mx >> 7) & 0xFF) - 127);
    se = max(-126, min(126, se));
    const float scale = plain ? 1.0f : __uint_as_float((uint32_t)(se + 127) << 23);
    if (lane == 0) inv[row] = plain ? 1.0f : __uint_as_float((uint32_t)(127 - se) << 23);
    for (int v = lane; v < K / 8; v += 32) {
        const uint4 q = in[v];
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 hv = __floats2half2_rn(__uint_as_float(w[i] << 16) * scale,
                                                 __uint_as_float(w[i] & 0xFFFF0000u) * scale);
            o[i] = *reinterpret_cast<const uint32_t *>(&hv);
        }
        out[(v & 3) * NC + (v >> 2)] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

template <int MODE>
uint32_t stage_bytes(const FfnArgs &a) {
    const int Imax = a.I_max;
    const uint32_t b = MODE == kGateUp ? 2u * kIB * (uint32_t)(a.H / 2 + a.H / 32)
                                       : (uint32_t)kMB * (uint32_t)(Imax / 2 + Imax / 32);
    return (b + 127u) & ~127u;
}

template <int MODE>
int launch_mode(const FfnArgs &a, int num_sms, cudaStream_t st) {
    const uint32_t stride = stage_bytes<MODE>(a);
    int nst = (int)(kSmemBudget / stride);
    nst = nst > 8 ? 8 : nst;
    if (nst < 2) return -2;
    const size_t smem = (size_t)nst * stride + (2 * nst + 4) * sizeof(uint64_t);
    if (cudaFuncSetAttribute(gemv_tma<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return -1;
    const int ipg = MODE == kGateUp ? (a.I_max + kIB - 1) / kIB : a.H / kMB;
    launch_pdl(gemv_tma<MODE>, dim3(num_sms), dim3(kThreads), smem, st, a, ipg, nst, stride);
    return cudaPeekAtLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace

int launch_ffn_gemv(const FfnArgs &a, int num_sms, cudaEvent_t mid, cudaStream_t st) {
    int n = 0, r;
    // tokens -> scaled fp16 (gate/up activations)
    launch_pdl(prep_rows_f16, dim3((a.T + 7) / 8), dim3(256), 0, st, a.x, a.H, a.T, a.H, a.T, a.H, a.xh, a.H, a.xinv);
    ++n;
    if ((r = launch_mode<kGateUp>(a, num_sms, st)) < 0) return r;
    n += r;
    if (mid) cudaEventRecord(mid, st);
    // h rows -> scaled fp16 (down activations); shared rows (from T*k on) have I_s columns
    launch_pdl(prep_rows_f16, dim3((a.rows + 7) / 8), dim3(256), 0, st, (const __nv_bfloat16 *)a.h, a.I_max, a.rows,
               a.I, a.T * a.top_k, a.I_s, a.hh, a.I_max, a.hinv);
    ++n;
    if ((r = launch_mode<kDown>(a, num_sms, st)) < 0) return r;
    n += r;
    return cudaPeekAtLastError() == cudaSuccess ? n : -1;
}

}  // namespace colimoe
