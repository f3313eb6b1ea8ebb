// A3/A4 on the tensor cores with native MXFP4 weights: block-scaled tcgen05.mma
// (kind::mxf8f6f4, E2M1 weights x E4M3 activations, UE8M0 scales per 32 elements, fp32 accumulate).
// ("DeepSeek V4 Flash CPU inference with NVMe expert streaming": FP4 E2M1 experts with UE8M0
// group-32 scales; the gate/up pair and the down projection. "the CUDA tier wired into the
// DeepSeek V4 engine": expert-grouped GEMM rows.)
//
// The weights never pass through the ALU: TMA copies the packed E2M1 codes into shared memory in
// the unpacked 16-value/16-byte form the MMA reads (tensor-map type 16U4_ALIGN16B, 128-byte
// swizzle), and the UE8M0 scale bytes go to TMEM, where the MMA applies them per 32-element block.
//
// Activations are split into E4M3 terms that the MMA multiplies exactly, each term with its own
// UE8M0 scale per 32 elements:
//   x (bf16, 8 significant bits): two terms reproduce it (the residual of a 4-bit rounding of an
//     8-bit value fits in 4 bits), up to elements 2^14 below their block maximum;
//   h (fp32, from the gate/up epilogue): three terms, relative error about 2^-12.
// The terms are stacked along N (term t at activation rows [t * bh, (t + 1) * bh) of the tile), so
// one MMA per weight matrix and 32-wide K block covers all of them; the epilogue adds the term
// columns. Block-scaled MMAs carry a large fixed cost each, which makes their count per stage the
// quantity to minimise.
//
// Swap-AB tiles: 128 weight rows (M) x up to 32 (gate/up) or 64 (down) tokens of one group (N).
// One persistent block per SM; warp roles:
//   warp 0     TMA producer (weight codes, activation terms) into a 4-stage ring, 128 K per stage;
//              the activation box is 16, 32 or 64 rows high, the smallest that holds the tile
//   warp 1     TMEM owner and MMA issuer; accumulators double buffered (2 x 192 columns)
//   warps 2-5  scale loaders: the stage's UE8M0 bytes -> TMEM (tcgen05.st). The MMA reads weight
//              row 32q + i from lane 32q + i, column q, and activation row n from lane 32q + n%32,
//              column n/32, in each lane quarter q; warp q loads its 32 weight rows' bytes with
//              16-byte loads that cover four stages, one group ahead
//   warps 6-9  epilogue: gate/up -> SwiGLU -> three E4M3 terms of h (scales from warp-wide block
//              maxima: a warp holds the 32 consecutive i-values of one scale block); down -> y
// Every barrier wait is bounded (sm103_ptx.cuh).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp8.h>

#include "colimoe_internal.cuh"
#include "sm103_ptx.cuh"

namespace colimoe {
namespace {

constexpr int BM = 128, BK = 128;
constexpr int kBnGateUp = kNtileMx, kBnDown = 2 * kNtileMx;   // tokens per tile
constexpr int NS = 4;
constexpr int kThreads = 320;
constexpr uint32_t kASmem = BM * BK;           // 16 KB: one unpacked E2M1 tile
constexpr uint32_t kATx = BM * BK / 2;         // 8 KB of packed codes per tile
constexpr uint32_t kBSmemMax = 3 * 64 * BK;    // activation terms stacked along N: up to 192 rows
// stage: A0 | A1 | B (terms stacked: term t at rows [t * bh, (t + 1) * bh))
constexpr uint32_t kOffA0 = 0, kOffA1 = kASmem, kOffB = 2 * kASmem;
constexpr uint32_t kStageBytes = 2 * kASmem + kBSmemMax;   // 57344
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 192;             // per accumulator buffer: matrices x terms x box rows
constexpr uint32_t kSfCol0 = 384;              // scale-factor columns: 16 per stage
constexpr int kBoxRows[3] = {16, 32, 64};      // activation box heights (16-row steps of the tile)
constexpr int kXTerms = 2, kHTerms = 3;

enum Mode { kGateUp = 0, kDown = 1 };

struct MxParams {
    int E, H, I, I_s, I_max, rows;
    int mode, m_tiles, nterms, bn;
    const int32_t *cnt, *off, *touched, *n_touched, *ntile_prefix, *ntile_owner;
    const uint8_t *w_scales_routed, *w_scales_shared;   // UE8M0 bytes of the weight rows
    const uint8_t *act_scales;                          // [nterms][rows][K/32]
    int act_ld;                                         // K of the activation terms (H or I_max)
    // gate/up epilogue outputs: h terms and their scales
    uint8_t *hq;                                        // [3][rows][I_max]
    uint8_t *hs;                                        // [3][rows][I_max/32]
    float *y;                                           // down epilogue output [rows][H]
    int *err;
};

struct TileInfo {
    int g, mt, row0, n_valid, Ig, nk;
    int box, bh;            // activation box map index and height (rows per term)
    bool valid, shared;
    size_t ge;
};

__device__ __forceinline__ TileInfo decode_tile(const MxParams &p, int t) {
    TileInfo ti;
    ti.mt = t % p.m_tiles;
    const int r = t / p.m_tiles;
    const int u = p.ntile_owner[r];
    ti.g = p.touched[u];
    const int nt = r - p.ntile_prefix[u];
    ti.shared = ti.g == p.E;
    ti.Ig = ti.shared ? p.I_s : p.I;
    ti.ge = ti.shared ? 0 : (size_t)ti.g;
    ti.row0 = p.off[ti.g] + nt * p.bn;
    ti.n_valid = min(p.bn, p.cnt[ti.g] - nt * p.bn);
    ti.valid = p.mode == kGateUp ? ti.mt * BM < ti.Ig : true;
    ti.nk = (p.mode == kGateUp ? p.H : ti.Ig) / BK;
    ti.box = ti.n_valid <= 16 ? 0 : ti.n_valid <= 32 ? 1 : 2;
    ti.bh = 16 << ti.box;
    return ti;
}

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Block-scaled instruction descriptor: A E2M1 (5), B E4M3 (0), UE8M0 scales, M x N, scale-factor
// byte ids for A and B (the K block of the 32-wide MMA within the 128-wide stage).
__device__ __forceinline__ uint32_t idesc_mx(int N, int sf_id) {
    return ((uint32_t)sf_id << 4) | (5u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
           ((uint32_t)(BM >> 4) << 24) | ((uint32_t)sf_id << 29);
}

__device__ __forceinline__ void mma_mx(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n}\n"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void tmem_st_x4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ void tmem_st_x1(uint32_t taddr, uint32_t a) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(a) : "memory");
}

__device__ __forceinline__ void tmem_st_x2(uint32_t taddr, uint32_t a, uint32_t b) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1,%2};" ::"r"(taddr), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// One E4M3 term of a warp-wide block of 32 values (one per lane): scale byte s with
// |v| / 2^(s-127) < 256, the E4M3 code of v / 2^(s-127) (round to nearest even), and the
// residual v - code * 2^(s-127) (exact in fp32).
__device__ __forceinline__ uint8_t e4m3_term(float v, float &resid, uint32_t &sbyte) {
    const float amax = warp_max(fabsf(v));
    const uint32_t ef = (__float_as_uint(amax) >> 23) & 0xFF;
    uint32_t s = (amax > 0.f && ef < 255) ? (ef > 8 ? ef - 7 : 1) : 127;
    s = min(s, 253u);
    const float scale = __uint_as_float(s << 23);            // 2^(s-127)
    const float inv = __uint_as_float((254u - s) << 23);     // 2^(127-s)
    uint16_t q2;
    asm("{\n .reg .b16 t;\n cvt.rn.satfinite.e4m3x2.f32 t, %1, %1;\n mov.b16 %0, t;\n}\n" : "=h"(q2) : "f"(v * inv));
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(q2));
    const float back = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFF)));
    resid = v - back * scale;
    sbyte = s;
    return (uint8_t)(q2 & 0xFF);
}

// Activation term maps: [term][box height index].
struct BMaps {
    CUtensorMap m[3][3];
};

__global__ void __launch_bounds__(kThreads, 1)
gemm_mx(const __grid_constant__ CUtensorMap tm_a_routed, const __grid_constant__ CUtensorMap tm_a_shared,
        const __grid_constant__ BMaps tm_b, const MxParams p) {
    pdl_trigger();
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + NS * kStageBytes);
    // barriers: tma_full[NS], sf_full[NS], empty[NS], acc_full[2], acc_empty[2], drain
    uint64_t *tma_full = bar, *sf_full = bar + NS, *empty = bar + 2 * NS, *acc_full = bar + 3 * NS,
             *acc_empty = bar + 3 * NS + 2, *drain = bar + 3 * NS + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 3 * NS + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool gu = p.mode == kGateUp;
    const int n_a = gu ? 2 : 1;
    const int nterms = p.nterms;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(ptx::smem_addr(&tma_full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&sf_full[s]), 128);
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
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();   // everything above is on-chip set-up
    const int total_tiles = p.m_tiles * p.ntile_prefix[*p.n_touched];

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            ptx::prefetch_tmap(&tm_a_routed);
            const uint64_t pol = ptx::policy_evict_first();
            uint32_t it = 0;
            for (int t = blockIdx.x; t < total_tiles && !*abort_flag; t += gridDim.x) {
                const TileInfo ti = decode_tile(p, t);
                if (!ti.valid) continue;
                const uint32_t tx = n_a * kATx + nterms * ti.bh * BK;
                const CUtensorMap *ta = ti.shared ? &tm_a_shared : &tm_a_routed;
                const int rpe = gu ? 2 * ti.Ig : p.H;
                const int arow = (int)ti.ge * rpe + ti.mt * BM;
                for (int k = 0; k < ti.nk; ++k, ++it) {
                    const int s = it % NS;
                    if (!ptx::mbar_wait(ptx::smem_addr(&empty[s]), ((it / NS) & 1u) ^ 1u, p.err, ptx::kErrWaitEmpty,
                                        abort_flag))
                        break;
                    const uint32_t fb = ptx::smem_addr(&tma_full[s]);
                    const uint32_t st = ptx::smem_addr(smem + s * kStageBytes);
                    ptx::mbar_arrive_expect_tx(fb, tx);
                    ptx::tma_load_2d_hint(st + kOffA0, ta, k * BK, arow, fb, pol);
                    if (gu) ptx::tma_load_2d_hint(st + kOffA1, ta, k * BK, arow + ti.Ig, fb, pol);
                    for (int tt = 0; tt < nterms; ++tt)
                        ptx::tma_load_2d(st + kOffB + tt * ti.bh * BK, &tm_b.m[tt][ti.box], k * BK, ti.row0, fb);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, tcount = 0;
            for (int t = blockIdx.x; t < total_tiles && !*abort_flag; t += gridDim.x) {
                const TileInfo ti = decode_tile(p, t);
                if (!ti.valid) continue;
                const uint32_t buf = tcount & 1u, use = tcount >> 1;
                if (!ptx::mbar_wait(ptx::smem_addr(&acc_empty[buf]), (use & 1u) ^ 1u, p.err, ptx::kErrWaitAccum,
                                    abort_flag))
                    break;
                ++tcount;
                ptx::tc_fence_after();
                const int n_mma = nterms * ti.bh;       // terms stacked along N
                bool ok = true;
                for (int k = 0; k < ti.nk; ++k, ++it) {
                    const int s = it % NS;
                    const uint32_t ph = (it / NS) & 1u;
                    if (!ptx::mbar_wait(ptx::smem_addr(&tma_full[s]), ph, p.err, ptx::kErrWaitFull, abort_flag) ||
                        !ptx::mbar_wait(ptx::smem_addr(&sf_full[s]), ph, p.err, ptx::kErrWaitFull, abort_flag)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_addr(smem + s * kStageBytes);
                    const uint32_t sf = tmem + kSfCol0 + s * 16;
#pragma unroll
                    for (int kb = 0; kb < BK / 32; ++kb) {
                        const uint32_t idesc = idesc_mx(n_mma, kb);
                        const uint64_t bd = sw128_desc(sa + kOffB + kb * 32);
                        for (int a = 0; a < n_a; ++a) {
                            const uint64_t ad = sw128_desc(sa + (a ? kOffA1 : kOffA0) + kb * 32);
                            const uint32_t d = tmem + buf * kAccCols + (uint32_t)(a * n_mma);
                            mma_mx(d, ad, bd, idesc, sf + 4 * a, sf + 8, (k > 0 || kb > 0) ? 1u : 0u);
                        }
                    }
                    ptx::mma_commit(ptx::smem_addr(&empty[s]));
                }
                if (!ok) break;
                ptx::mma_commit(ptx::smem_addr(&acc_full[buf]));
            }
            ptx::mma_commit(ptx::smem_addr(drain));
            ptx::mbar_wait(ptx::smem_addr(drain), 0, nullptr, 0, nullptr);
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------------ scale loaders
        // TMEM scale layout the MMA reads (M = 128): weight row 32q + i takes its four K-block
        // bytes from lane 32q + i, column base + q; activation row n takes them from lane
        // 32q + n % 32, column base + n / 32, in every lane quarter q. Warp `quad` writes quarter
        // quad: its own 32 weight rows and a copy of the activation rows.
        const int quad = warp & 3;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        const int kba = p.act_ld / 32;                   // scale bytes per activation row
        uint32_t it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total_tiles && ok && !*abort_flag; t += gridDim.x) {
            const TileInfo ti = decode_tile(p, t);
            if (!ti.valid) continue;
            const int K = gu ? p.H : ti.Ig;
            const int kb_row = K / 32;                   // scale bytes per weight row
            const uint8_t *ws = ti.shared ? p.w_scales_shared : p.w_scales_routed;
            const int rpe = gu ? 2 * ti.Ig : p.H;
            const size_t wrow = ti.ge * (size_t)rpe + (size_t)ti.mt * BM + quad * 32 + lane;
            const uint8_t *wp[2] = {ws + wrow * kb_row, n_a > 1 ? ws + (wrow + ti.Ig) * kb_row : nullptr};
            // activation row n = lane + 32c of the stacked B tile: term n / bh, token n % bh
            const int nb_rows = nterms * ti.bh, nb_cols = (nb_rows + 31) / 32;
            const uint8_t *bp[6];
#pragma unroll
            for (int c = 0; c < 6; ++c) {
                const int n = lane + 32 * c;
                const int tt = n / ti.bh, j = n % ti.bh;
                bp[c] = (n < nb_rows && j < ti.n_valid) ? p.act_scales + ((size_t)tt * p.rows + ti.row0 + j) * kba
                                                        : nullptr;
            }
            // one 16-byte load covers four stages when the rows' scale bytes allow it
            const bool vec = (kb_row % 16 == 0) && (kba % 16 == 0) && (ti.nk % 4 == 0);
            auto put = [&](int s, uint32_t a0, uint32_t a1, const uint32_t (&b)[6]) {
                const uint32_t col = lane_base + kSfCol0 + s * 16;
                tmem_st_x1(col + quad, a0);
                if (n_a > 1) tmem_st_x1(col + 4 + quad, a1);
                tmem_st_x2(col + 8, b[0], b[1]);
                if (nb_cols > 2) tmem_st_x2(col + 10, b[2], b[3]);
                if (nb_cols > 4) tmem_st_x2(col + 12, b[4], b[5]);
                tmem_st_wait();
                ptx::tc_fence_before();
                ptx::mbar_arrive(ptx::smem_addr(&sf_full[s]));
            };
            auto ld16 = [](const uint8_t *q, int g) {
                return q ? __ldg(reinterpret_cast<const uint4 *>(q) + g) : make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu,
                                                                                  0x7F7F7F7Fu, 0x7F7F7F7Fu);
            };
            auto ld4 = [](const uint8_t *q, int k) {
                return q ? __ldg(reinterpret_cast<const uint32_t *>(q) + k) : 0x7F7F7F7Fu;
            };
            if (vec) {
                uint4 ca[2], cb[6];
                ca[0] = ld16(wp[0], 0);
                ca[1] = ld16(wp[1], 0);
#pragma unroll
                for (int i = 0; i < 6; ++i) cb[i] = ld16(bp[i], 0);
                for (int g = 0; g < ti.nk / 4 && ok; ++g) {
                    uint4 na[2], nb[6];
                    const bool more = g + 1 < ti.nk / 4;
                    if (more) {
                        na[0] = ld16(wp[0], g + 1);
                        na[1] = ld16(wp[1], g + 1);
#pragma unroll
                        for (int i = 0; i < 6; ++i) nb[i] = ld16(bp[i], g + 1);
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int s = it % NS;
                        if (!ptx::mbar_wait(ptx::smem_addr(&empty[s]), ((it / NS) & 1u) ^ 1u, p.err,
                                            ptx::kErrWaitEmpty, abort_flag)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        auto pick = [j](const uint4 &v) { return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w; };
                        const uint32_t b[6] = {pick(cb[0]), pick(cb[1]), pick(cb[2]), pick(cb[3]), pick(cb[4]),
                                               pick(cb[5])};
                        put(s, pick(ca[0]), pick(ca[1]), b);
                        ++it;
                    }
                    if (more) {
                        ca[0] = na[0];
                        ca[1] = na[1];
#pragma unroll
                        for (int i = 0; i < 6; ++i) cb[i] = nb[i];
                    }
                }
            } else {
                for (int k = 0; k < ti.nk && ok; ++k) {
                    const uint32_t a0 = ld4(wp[0], k), a1 = ld4(wp[1], k);
                    uint32_t b[6];
#pragma unroll
                    for (int i = 0; i < 6; ++i) b[i] = ld4(bp[i], k);
                    const int s = it % NS;
                    if (!ptx::mbar_wait(ptx::smem_addr(&empty[s]), ((it / NS) & 1u) ^ 1u, p.err, ptx::kErrWaitEmpty,
                                        abort_flag)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    put(s, a0, a1, b);
                    ++it;
                }
            }
        }
    } else {
        // ------------------------------------------------------------------ epilogue
        const int quad = warp & 3;
        const int m = quad * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        uint32_t tcount = 0;
        for (int t = blockIdx.x; t < total_tiles && !*abort_flag; t += gridDim.x) {
            const TileInfo ti = decode_tile(p, t);
            if (!ti.valid) continue;
            const uint32_t buf = tcount & 1u, use = tcount >> 1;
            if (!ptx::mbar_wait(ptx::smem_addr(&acc_full[buf]), use & 1u, p.err, ptx::kErrWaitAccum, abort_flag))
                break;
            ++tcount;
            ptx::tc_fence_after();
            const int mrow = ti.mt * BM + m;
            const uint32_t acc = lane_base + buf * kAccCols;
            const int ncols = nterms * ti.bh;           // accumulator columns per matrix
            for (int c0 = 0; c0 < ti.n_valid; c0 += 16) {
                if (gu) {
                    uint32_t g0[16], g1[16], u0[16], u1[16];
                    ptx::tmem_ld16(acc + c0, g0);
                    ptx::tmem_ld16(acc + ti.bh + c0, g1);
                    ptx::tmem_ld16(acc + ncols + c0, u0);
                    ptx::tmem_ld16(acc + ncols + ti.bh + c0, u1);
                    ptx::tmem_ld_wait();
                    for (int j = 0; j < 16 && c0 + j < ti.n_valid; ++j) {
                        const float g = __uint_as_float(g0[j]) + __uint_as_float(g1[j]);
                        const float u = __uint_as_float(u0[j]) + __uint_as_float(u1[j]);
                        float v = __fdiv_rn(g, 1.0f + expf(-g)) * u;
                        const size_t row = (size_t)ti.row0 + c0 + j;
#pragma unroll
                        for (int tt = 0; tt < kHTerms; ++tt) {
                            uint32_t sb;
                            float r;
                            const uint8_t q = e4m3_term(v, r, sb);
                            p.hq[((size_t)tt * p.rows + row) * p.I_max + mrow] = q;
                            if (lane == 0) p.hs[((size_t)tt * p.rows + row) * (p.I_max / 32) + mrow / 32] = (uint8_t)sb;
                            v = r;
                        }
                    }
                } else {
                    uint32_t d0[16], d1[16], d2[16];
                    ptx::tmem_ld16(acc + c0, d0);
                    ptx::tmem_ld16(acc + ti.bh + c0, d1);
                    ptx::tmem_ld16(acc + 2 * ti.bh + c0, d2);
                    ptx::tmem_ld_wait();
                    for (int j = 0; j < 16 && c0 + j < ti.n_valid; ++j)
                        p.y[((size_t)ti.row0 + c0 + j) * p.H + mrow] =
                            (__uint_as_float(d0[j]) + __uint_as_float(d1[j])) + __uint_as_float(d2[j]);
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&acc_empty[buf]));
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// UE8M0 byte s for a block maximum: |v| / 2^(s-127) < 256 (same rule as e4m3_term).
__device__ __forceinline__ uint32_t block_scale_byte(float amax) {
    const uint32_t ef = (__float_as_uint(amax) >> 23) & 0xFF;
    const uint32_t s = (amax > 0.f && ef < 255) ? (ef > 8 ? ef - 7 : 1) : 127;
    return min(s, 253u);
}

// x rows (expert-grouped, via src_token) -> two E4M3 terms with UE8M0 scales per 32 elements.
// One thread per (row, 32-element block): it reads the block's 64 bytes, finds its maximum, and
// writes 32 code bytes per term and one scale byte per term; a warp covers 2 KB of one row.
__global__ void __launch_bounds__(256)
quant_x_rows(const __nv_bfloat16 *__restrict__ x, int H, const int32_t *__restrict__ src_token, int rows,
             uint8_t *__restrict__ xq, uint8_t *__restrict__ xs) {
    pdl_begin();
    const int nb = H / 32;
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long)rows * nb) return;
    const int row = (int)(i / nb), b = (int)(i % nb);
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)src_token[row] * H + b * 32);
    float v[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 u = __ldg(src + q);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[q * 8 + 2 * j] = __uint_as_float(w[j] << 16);
            v[q * 8 + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
#pragma unroll
    for (int tt = 0; tt < kXTerms; ++tt) {
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(v[e]));
        const uint32_t sb = block_scale_byte(amax);
        const float scale = __uint_as_float(sb << 23), inv = __uint_as_float((254u - sb) << 23);
        uint32_t packed[8];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
            uint16_t q2;
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(q2) : "f"(v[e + 1] * inv), "f"(v[e] * inv));
            uint32_t h2;
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(q2));
            const float2 back = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
            v[e] -= back.x * scale;                // residuals for the next term (exact)
            v[e + 1] -= back.y * scale;
            if (e % 4 == 0) packed[e / 4] = q2;
            else packed[e / 4] |= (uint32_t)q2 << 16;
        }
        uint4 *dst = reinterpret_cast<uint4 *>(xq + ((size_t)tt * rows + row) * H + b * 32);
        dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        xs[((size_t)tt * rows + row) * nb + b] = (uint8_t)sb;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &ptr, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// Packed E2M1 rows of K elements: unpacked into 16-values-per-16-bytes smem, 128 x 128 boxes.
bool map_codes(CUtensorMap *m, const void *base, uint64_t K, uint64_t rows) {
    auto enc = encoder();
    if (!enc || (reinterpret_cast<uintptr_t>(base) & 31)) return false;
    const cuuint64_t dims[2] = {K, rows};
    const cuuint64_t strides[1] = {K / 2};
    const cuuint32_t box[2] = {BK, BM};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E4M3 activation rows (bytes): 128 x box_rows boxes with the 128-byte swizzle.
bool map_act(CUtensorMap *m, const void *base, uint64_t K, uint64_t rows, uint32_t box_rows) {
    auto enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {K, rows};
    const cuuint64_t strides[1] = {K};
    const cuuint32_t box[2] = {BK, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool mx_available() { return encoder() != nullptr; }

int launch_quant_x(const FfnArgs &a, cudaStream_t st) {
    const long qthreads = (long)a.rows * (a.H / 32);
    launch_pdl(quant_x_rows, dim3((unsigned)((qthreads + 255) / 256)), dim3(256), 0, st, a.x, a.H, a.src_token,
               a.rows, a.xq, a.xqs);
    return cudaPeekAtLastError() == cudaSuccess ? 1 : -1;
}


bool mx_supported(const FfnArgs &a) {
    auto al = [](const void *p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 31) == 0; };
    return mx_available() && al(a.routed.gu_codes) && al(a.routed.d_codes) && al(a.shared.gu_codes) &&
           al(a.shared.d_codes);
}

// The three box heights of one activation term.
bool map_term(CUtensorMap (&m)[3], const void *base, uint64_t K, uint64_t rows) {
    for (int b = 0; b < 3; ++b)
        if (!map_act(&m[b], base, K, rows, kBoxRows[b])) return false;
    return true;
}

int launch_ffn_mx(const FfnArgs &a, int num_sms, void *sched, cudaEvent_t mid, cudaStream_t st) {
    if (!mx_supported(a)) return -2;
    // n-tile prefixes and owners were written by the permute scan (NtileLayout)
    const NtileLayout nl = ntile_layout(sched, a.E, a.rows);
    int32_t *prefix_gu = nl.prefix_small, *owner_gu = nl.owner_small;
    int32_t *prefix_dn = nl.prefix_large, *owner_dn = nl.owner_large;
    int n = 0;

    const size_t smem = NS * kStageBytes + 1024 + 256;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(gemm_mx, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return -1;
        attr = true;
    }
    MxParams p{};
    p.E = a.E;
    p.H = a.H;
    p.I = a.I;
    p.I_s = a.I_s;
    p.I_max = a.I_max;
    p.rows = a.rows;
    p.cnt = a.cnt;
    p.off = a.off;
    p.touched = a.touched;
    p.n_touched = a.n_touched;
    p.hq = a.hq;
    p.hs = a.hqs;
    p.y = a.y;
    p.err = a.err;

    CUtensorMap tar, tas;
    BMaps tb;
    // gate/up: A = gate/up code rows, B = two terms of x
    p.mode = kGateUp;
    p.bn = kBnGateUp;
    p.ntile_prefix = prefix_gu;
    p.ntile_owner = owner_gu;
    p.m_tiles = (a.I_max + BM - 1) / BM;
    p.nterms = kXTerms;
    p.w_scales_routed = a.routed.gu_scales;
    p.w_scales_shared = a.shared.gu_scales;
    p.act_scales = a.xqs;
    p.act_ld = a.H;
    bool ok = map_codes(&tar, a.routed.gu_codes, a.H, (uint64_t)a.E * 2 * a.I) &&
              map_term(tb.m[0], a.xq, a.H, a.rows) && map_term(tb.m[1], a.xq + (size_t)a.rows * a.H, a.H, a.rows);
    for (int b = 0; b < 3; ++b) tb.m[2][b] = tb.m[1][b];
    if (a.shared.gu_codes) ok = ok && map_codes(&tas, a.shared.gu_codes, a.H, 2 * (uint64_t)a.I_s);
    else tas = tar;
    if (!ok) return -2;
    launch_pdl(gemm_mx, dim3(num_sms), dim3(kThreads), smem, st, tar, tas, tb, p);
    ++n;
    if (mid) cudaEventRecord(mid, st);

    // down: A = down code rows, B = three terms of h
    p.mode = kDown;
    p.bn = kBnDown;
    p.ntile_prefix = prefix_dn;
    p.ntile_owner = owner_dn;
    p.m_tiles = a.H / BM;
    p.nterms = kHTerms;
    p.w_scales_routed = a.routed.d_scales;
    p.w_scales_shared = a.shared.d_scales;
    p.act_scales = a.hqs;
    p.act_ld = a.I_max;
    ok = map_codes(&tar, a.routed.d_codes, a.I, (uint64_t)a.E * a.H);
    for (int t = 0; t < kHTerms && ok; ++t)
        ok = map_term(tb.m[t], a.hq + (size_t)t * a.rows * a.I_max, a.I_max, a.rows);
    if (a.shared.d_codes) ok = ok && map_codes(&tas, a.shared.d_codes, a.I_s, (uint64_t)a.H);
    else tas = tar;
    if (!ok) return -2;
    launch_pdl(gemm_mx, dim3(num_sms), dim3(kThreads), smem, st, tar, tas, tb, p);
    ++n;
    return cudaPeekAtLastError() == cudaSuccess ? n : -1;
}

}  // namespace colimoe
