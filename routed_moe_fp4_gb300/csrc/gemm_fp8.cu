// FP8 dense projection: out[t][n] = bf16(sum_k x[t][k] * e4m3(w[n][k]) * w_scale[n/128][k/128]).
//
// The pages give the model's dense weights as FP8 E4M3 with one scale per 128 x 128 block ("DeepSeek
// V4 Flash CPU inference with NVMe expert streaming", the review question on config-driven V4
// sizes) and run the five per-layer dense matmuls on the GPU with the CPU path's numerics
// ("DeepSeek V4 Flash support -- CUDA/VRAM expert tiering", the dense-on-GPU tier comment).
//
// GB300 design. The weights go to the 5th-generation tensor cores as stored (tcgen05.mma
// kind::f8f6f4, E4M3 x E4M3, 32 K per instruction). The activations become two E4M3 terms per
// element after a per-token power-of-two scale: x = 2^e (q1 + q2), |x| 2^-e < 256, which keeps about
// 8 significant bits (bf16 has 8). The two terms are stacked along N, so one MMA covers both.
// The block scale varies along K every 128 elements and is an arbitrary fp32, so it cannot ride in
// the MMA's power-of-two scale factors. Each 128-K block is therefore accumulated on its own, into
// one of two TMEM buffers, and the epilogue warps fold it into fp32 registers: acc += s * (p1 + p2).
// This runs while the tensor cores fill the other buffer. The token scale 2^e is applied once,
// when out is written.
//
// Roles (one persistent block per SM): warp 0 issues TMA, warp 1 allocates TMEM and issues MMAs,
// the other warps fold the partial sums: 8 of them (16 for 128-token tiles), each TMEM lane
// quarter shared by 2 (4) warps that split the tile's tokens. Tiles are 128 weight rows x BN
// tokens; every wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "colimoe_internal.cuh"
#include "sm103_ptx.cuh"

namespace colimoe {
namespace {

constexpr int BM = 128;            // weight rows per tile (MMA M)
constexpr int KB = 128;            // K per stage: one scale block, one 128-byte swizzle row
constexpr uint32_t kASmem = BM * KB;                       // 16 KB
// Per token-tile size BN: a stage holds the weights and both terms of BN tokens; as many stages
// as fit in 200 KB (more bytes in flight when the stages are small); as many TMEM
// accumulator buffers (2 x BN columns each) as fit in 512 columns, up to 8, so the tensor cores
// can run ahead of the fold.
template <int BN> struct Fp8Cfg {
    static constexpr int EPI = BN >= 128 ? 16 : 8;         // fold warps
    static constexpr int THREADS = 64 + 32 * EPI;
    static constexpr uint32_t kStage = kASmem + 2 * BN * KB;
    static constexpr int NS = (200 * 1024) / kStage > 12 ? 12 : (200 * 1024) / kStage;
    static constexpr int NBUF = 512 / (2 * BN) > 8 ? 8 : 512 / (2 * BN);
};
constexpr int kTmemCols = 512;

struct Fp8Params {
    int T, K, N, n_blocks, t_tiles;
    int ksplit, kper;              // K split into ksplit ranges of kper 128-blocks (ksplit 1: none)
    const float *w_scale;          // [N/128][K/128]
    const float *x_scale;          // [T] 2^e per token
    __nv_bfloat16 *out;            // [T][N]
    float *part;                   // [ksplit][T][N] partial sums of a split K
    int *cnt;                      // [n_blocks * t_tiles] arrivals of the splits of a tile
    int *err;
    uint64_t wait_ns;
};

// Tile `tile` = (K range sp, token block tb, weight block nb), weight blocks fastest.
struct Fp8Tile {
    int nb, tb, sp, k0, k1, id;
};
__device__ __forceinline__ Fp8Tile fp8_tile(const Fp8Params &p, int tile) {
    Fp8Tile t;
    const int per = p.n_blocks * p.t_tiles, r = tile % per;
    t.sp = tile / per;
    t.nb = r % p.n_blocks;
    t.tb = r / p.n_blocks;
    t.id = r;
    t.k0 = t.sp * p.kper;
    t.k1 = min(p.K / KB, t.k0 + p.kper);
    return t;
}

// 32 lanes x 32 bits, 32 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// kind::f8f6f4 instruction descriptor: fp32 accumulator, A and B E4M3 (format 0), K-major, M x N.
__device__ __forceinline__ uint32_t idesc_f8(int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void mma_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

template <int BN>
__global__ void __launch_bounds__(Fp8Cfg<BN>::THREADS, 1)
gemm_fp8(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x0,
         const __grid_constant__ CUtensorMap tm_x1, const Fp8Params p) {
    // The quantisation kernel before this one signals only after its own dependency wait, so the
    // weights (which no kernel of this forward writes) may be loaded before this kernel's wait.
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int NS = Fp8Cfg<BN>::NS, NBUF = Fp8Cfg<BN>::NBUF, kEpiWarps = Fp8Cfg<BN>::EPI;
    constexpr uint32_t kStageBytes = Fp8Cfg<BN>::kStage;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + NS * kStageBytes);
    uint64_t *full = bar, *empty = bar + NS, *acc_full = bar + 2 * NS, *acc_empty = bar + 2 * NS + NBUF,
             *drain = bar + 2 * NS + 2 * NBUF;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *last_flag = abort_flag + 1;
    constexpr int NC = 2 * BN;                                // MMA N: both terms
    constexpr uint32_t kBBytes = NC * KB;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(ptx::smem_addr(&full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&empty[s]), 1);
        }
        for (int b = 0; b < NBUF; ++b) {
            ptx::mbar_init(ptx::smem_addr(&acc_full[b]), 1);
            ptx::mbar_init(ptx::smem_addr(&acc_empty[b]), kEpiWarps);
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
    const int total = p.n_blocks * p.t_tiles * p.ksplit;

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            ptx::prefetch_tmap(&tm_w);
            const uint64_t pol = ptx::policy_evict_first();
            auto issue_w = [&](const Fp8Tile &tl, int k, int s) {
                const uint32_t fb = ptx::smem_addr(&full[s]);
                ptx::mbar_arrive_expect_tx(fb, kASmem + kBBytes);
                ptx::tma_load_2d_hint(ptx::smem_addr(smem + s * kStageBytes), &tm_w, k * KB, tl.nb * BM, fb, pol);
            };
            auto issue_x = [&](const Fp8Tile &tl, int k, int s) {
                const uint32_t fb = ptx::smem_addr(&full[s]);
                const uint32_t st = ptx::smem_addr(smem + s * kStageBytes) + kASmem;
                ptx::tma_load_2d(st, &tm_x0, k * KB, tl.tb * BN, fb);
                ptx::tma_load_2d(st + BN * KB, &tm_x1, k * KB, tl.tb * BN, fb);
            };
            const int first = blockIdx.x;
            const Fp8Tile tf = fp8_tile(p, first);
            const int pre = first < total ? min(NS, tf.k1 - tf.k0) : 0;
            for (int k = 0; k < pre; ++k) issue_w(tf, tf.k0 + k, k);
            pdl_wait();
            pdl_trigger();
            for (int k = 0; k < pre; ++k) issue_x(tf, tf.k0 + k, k);
            uint32_t it = 0;
            for (int tile = first; tile < total && !*abort_flag; tile += gridDim.x) {
                const Fp8Tile tl = fp8_tile(p, tile);
                for (int k = tl.k0; k < tl.k1; ++k, ++it) {
                    if (tile == first && k - tl.k0 < pre) continue;
                    const int s = it % NS;
                    if (!ptx::mbar_wait(ptx::smem_addr(&empty[s]), ((it / NS) & 1u) ^ 1u, p.err, ptx::kErrWaitEmpty,
                                        abort_flag, p.wait_ns))
                        break;
                    issue_w(tl, k, s);
                    issue_x(tl, k, s);
                }
            }
            const uint32_t issued = it > (uint32_t)pre ? it : (uint32_t)pre;
            for (uint32_t i = issued > (uint32_t)NS ? issued - NS : 0; i < issued; ++i)
                ptx::mbar_wait(ptx::smem_addr(&full[i % NS]), (i / NS) & 1u, nullptr, 0, nullptr);
        } else {
            pdl_wait();
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        pdl_wait();
        if (lane == 0) {
            const uint64_t desc0 = sw128_desc(ptx::smem_addr(smem));
            const uint32_t idesc = idesc_f8(NC);
            uint32_t it = 0, u = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok && !*abort_flag; tile += gridDim.x) {
                const Fp8Tile tl = fp8_tile(p, tile);
                for (int k = tl.k0; k < tl.k1; ++k, ++it, ++u) {
                    const int s = it % NS, b = u % NBUF;
                    if (!ptx::mbar_wait(ptx::smem_addr(&acc_empty[b]), ((u / NBUF) & 1u) ^ 1u, p.err,
                                        ptx::kErrWaitAccum, abort_flag, p.wait_ns) ||
                        !ptx::mbar_wait(ptx::smem_addr(&full[s]), (it / NS) & 1u, p.err, ptx::kErrWaitFull,
                                        abort_flag, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint64_t a = desc0 + (uint64_t)(s * (kStageBytes >> 4));
                    const uint64_t bd = a + (kASmem >> 4);
                    const uint32_t d = tmem + b * NC;
#pragma unroll
                    for (int j = 0; j < KB / 32; ++j) mma_f8(d, a + 2 * j, bd + 2 * j, idesc, j > 0 ? 1u : 0u);
                    ptx::mma_commit(ptx::smem_addr(&empty[s]));
                    ptx::mma_commit(ptx::smem_addr(&acc_full[b]));
                }
            }
            ptx::mma_commit(ptx::smem_addr(drain));
            ptx::mbar_wait(ptx::smem_addr(drain), 0, nullptr, 0, nullptr);
        }
    } else {
        // ------------------------------------------------------------------ fold + store
        pdl_wait();
        constexpr int H2 = BN / (kEpiWarps / 4);               // tokens of this warp
        const int quad = warp & 3, half = (warp - 2) >> 2;     // lane quarter, token slice
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        uint32_t u = 0;
        // Every epilogue warp walks every tile of the block, also after an abort (its waits then
        // return at once), so that the split-K named barriers below are always met by all eight.
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const Fp8Tile tl = fp8_tile(p, tile);
            const int t0 = tl.tb * BN + half * H2;
            const int n = tl.nb * BM + quad * 32 + lane;
            const float *wsc = p.w_scale + (size_t)tl.nb * (p.K / KB);
            float acc[H2];
#pragma unroll
            for (int j = 0; j < H2; ++j) acc[j] = 0.f;
            float s_next = __ldg(wsc + tl.k0);
            bool ok = true;
            for (int k = tl.k0; k < tl.k1; ++k, ++u) {
                const int b = u % NBUF;
                const float s = s_next;
                if (k + 1 < tl.k1) s_next = __ldg(wsc + k + 1);
                if (!ptx::mbar_wait(ptx::smem_addr(&acc_full[b]), (u / NBUF) & 1u, p.err, ptx::kErrWaitAccum,
                                    abort_flag, p.wait_ns)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t base = lane_base + b * NC + half * H2;
                // columns per TMEM load: 32, or 16 when 16 fold warps share the registers
                constexpr int CH = H2 < 16 ? 8 : (kEpiWarps > 8 || H2 < 32) ? 16 : 32;
#pragma unroll
                for (int c = 0; c < H2; c += CH) {
                    uint32_t r0[CH], r1[CH];
                    if constexpr (CH == 32) {
                        tmem_ld32(base + c, r0);
                        tmem_ld32(base + BN + c, r1);
                    } else if constexpr (CH == 16) {
                        ptx::tmem_ld16(base + c, r0);
                        ptx::tmem_ld16(base + BN + c, r1);
                    } else {
                        ptx::tmem_ld8(base + c, r0);
                        ptx::tmem_ld8(base + BN + c, r1);
                    }
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < CH; ++j)
                        acc[c + j] = fmaf(s, __uint_as_float(r0[j]) + __uint_as_float(r1[j]), acc[c + j]);
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&acc_empty[b]));
            }
            if (BN > kSplitMaxTokens || p.ksplit == 1) {   // the host splits K only for small T
                if (!ok) continue;
#pragma unroll
                for (int j = 0; j < H2; ++j) {
                    const int t = t0 + j;
                    if (t < p.T) p.out[(size_t)t * p.N + n] = __float2bfloat16_rn(acc[j] * __ldg(p.x_scale + t));
                }
                continue;
            }
            // Split K: every split stores its partial sums; the last split of the tile to arrive adds
            // them in split order (the same result whichever arrives last) and writes out.
            if (ok) {
#pragma unroll
                for (int j = 0; j < H2; ++j)
                    if (t0 + j < p.T) p.part[((size_t)tl.sp * p.T + t0 + j) * p.N + n] = acc[j];
            }
            __threadfence();
            asm volatile("bar.sync 1, %0;" ::"r"(32 * kEpiWarps) : "memory");
            if (warp == 2 && lane == 0)
                *last_flag = !*abort_flag && atomicAdd(p.cnt + tl.id, 1) == p.ksplit - 1;
            asm volatile("bar.sync 1, %0;" ::"r"(32 * kEpiWarps) : "memory");
            if (*last_flag && ok) {
                __threadfence();
                // sum[j] over the splits in split order; each split's H2 values are loaded together
                float sum[H2];
#pragma unroll
                for (int j = 0; j < H2; ++j) sum[j] = 0.f;
                for (int s2 = 0; s2 < p.ksplit; ++s2) {
                    float v[H2];
#pragma unroll
                    for (int j = 0; j < H2; ++j)
                        v[j] = s2 == tl.sp ? acc[j]
                             : t0 + j < p.T ? __ldcg(p.part + ((size_t)s2 * p.T + t0 + j) * p.N + n) : 0.f;
#pragma unroll
                    for (int j = 0; j < H2; ++j) sum[j] += v[j];
                }
#pragma unroll
                for (int j = 0; j < H2; ++j)
                    if (t0 + j < p.T)
                        p.out[(size_t)(t0 + j) * p.N + n] = __float2bfloat16_rn(sum[j] * __ldg(p.x_scale + t0 + j));
                if (warp == 2 && lane == 0) p.cnt[tl.id] = 0;
            }
            asm volatile("bar.sync 1, %0;" ::"r"(32 * kEpiWarps) : "memory");   // last_flag reuse
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// x [T][K] bf16 -> two E4M3 terms [2][T][K] and the token scale 2^e ([T]): e = floor(log2 max|x|) - 7,
// so |x| 2^-e < 256 (within E4M3's 448); q1 = e4m3(x 2^-e), q2 = e4m3(x 2^-e - q1). One block per token.
// Block 0 also clears the split-K arrival counters (left non-zero only by a forward that gave up).
__global__ void __launch_bounds__(256) quant_x_e4m3(const __nv_bfloat16 *__restrict__ x, int T, int K,
                                                    uint8_t *__restrict__ xq, float *__restrict__ xs, int *cnt,
                                                    int n_cnt) {
    pdl_wait();
    pdl_trigger();
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < n_cnt; i += 256) cnt[i] = 0;
    const int t = blockIdx.x;
    const __nv_bfloat16 *row = x + (size_t)t * K;
    float amax = 0.f;
    for (int i = threadIdx.x * 8; i < K; i += 256 * 8) {
        const uint4 v = *reinterpret_cast<const uint4 *>(row + i);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(h[j]);
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
    amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax)));
    __shared__ float wmax[8];
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) amax = fmaxf(amax, wmax[w]);
    // 2^-e as an fp32 bit pattern: biased exponent of amax minus 7, kept in the normal range
    const int ea = amax > 0.f ? (int)((__float_as_uint(amax) >> 23) & 0xFF) : 127;
    const int eb = min(max(ea - 7, 1), 254);                  // biased exponent of 2^e
    const float scale = __uint_as_float((uint32_t)eb << 23), inv = __uint_as_float((uint32_t)(254 - eb) << 23);
    if (threadIdx.x == 0) xs[t] = scale;
    uint8_t *q1 = xq + (size_t)t * K, *q2 = xq + (size_t)T * K + (size_t)t * K;
    for (int i = threadIdx.x * 8; i < K; i += 256 * 8) {
        const uint4 v = *reinterpret_cast<const uint4 *>(row + i);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
        uint32_t a[2] = {0, 0}, c[2] = {0, 0};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(h[j]);
            const float v0 = f.x * inv, v1 = f.y * inv;
            uint16_t p1, p2;
            uint32_t back;
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(p1) : "f"(v1), "f"(v0));
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(back) : "h"(p1));
            const float2 bf = __half22float2(*reinterpret_cast<const __half2 *>(&back));
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(p2) : "f"(v1 - bf.y), "f"(v0 - bf.x));
            a[j >> 1] |= (uint32_t)p1 << (16 * (j & 1));
            c[j >> 1] |= (uint32_t)p2 << (16 * (j & 1));
        }
        *reinterpret_cast<uint2 *>(q1 + i) = make_uint2(a[0], a[1]);
        *reinterpret_cast<uint2 *>(q2 + i) = make_uint2(c[0], c[1]);
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

// Rows of K bytes, boxes of 128 bytes x box_rows with the 128-byte swizzle.
bool map_bytes(CUtensorMap *m, const void *base, uint64_t K, uint64_t rows, uint32_t box_rows) {
    auto enc = encoder();
    if (!enc || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
    const cuuint64_t dims[2] = {K, rows};
    const cuuint64_t strides[1] = {K};
    const cuuint32_t box[2] = {KB, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN>
int launch_gemm(const DenseArgs &a, int num_sms, cudaStream_t st) {
    const size_t smem = Fp8Cfg<BN>::NS * Fp8Cfg<BN>::kStage + 1024 + 512;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(gemm_fp8<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return -1;
        attr = true;
    }
    CUtensorMap tw, tx0, tx1;
    if (!map_bytes(&tw, a.w, a.K, a.N, BM) || !map_bytes(&tx0, a.xq, a.K, a.T, BN) ||
        !map_bytes(&tx1, a.xq + (size_t)a.T * a.K, a.K, a.T, BN))
        return -2;
    Fp8Params p;
    p.T = a.T;
    p.K = a.K;
    p.N = a.N;
    p.n_blocks = a.N / BM;
    p.t_tiles = (a.T + BN - 1) / BN;
    // Few tiles (small T): split K so that every SM streams weights; the partials fit the
    // workspace because ksplit x n_blocks <= SMs.
    const int nk = a.K / KB, tiles0 = p.n_blocks * p.t_tiles;
    int ksplit = 1;
    if (a.T <= kSplitMaxTokens && 2 * tiles0 <= num_sms) ksplit = min(nk, num_sms / tiles0);
    p.kper = (nk + ksplit - 1) / ksplit;
    p.ksplit = (nk + p.kper - 1) / p.kper;
    p.part = a.part;
    p.cnt = a.cnt;
    p.w_scale = a.w_scale;
    p.x_scale = a.xs;
    p.out = a.out;
    p.err = a.err;
    p.wait_ns = a.wait_ns ? a.wait_ns : ptx::kWaitLimitNs;
    const int tiles = tiles0 * p.ksplit;
    launch_pdl(gemm_fp8<BN>, dim3(tiles < num_sms ? tiles : num_sms), dim3(Fp8Cfg<BN>::THREADS), smem, st, tw, tx0,
               tx1, p);
    return cudaPeekAtLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace

bool fp8_available() { return encoder() != nullptr; }

int launch_dense_fp8(const DenseArgs &a, int num_sms, cudaStream_t st) {
    if (!encoder()) return -2;
    launch_pdl(quant_x_e4m3, dim3(a.T), dim3(256), 0, st, a.x, a.T, a.K, a.xq, a.xs, a.cnt, num_sms);
    if (cudaPeekAtLastError() != cudaSuccess) return -1;
    // tokens per tile: 16 for decode-sized T, else 64 or 128 (the MMA's N is twice that)
    const int n = a.T <= 16 ? launch_gemm<16>(a, num_sms, st)
                : a.T <= 64 ? launch_gemm<64>(a, num_sms, st) : launch_gemm<128>(a, num_sms, st);
    return n < 0 ? n : n + 1;
}

}  // namespace colimoe
