// A3/A4 for larger token counts: grouped GEMMs on the 5th-generation tensor cores (tcgen05).
//
// gate/up: for each touched group, D_g = Wg x^T and D_u = Wu x^T over tiles of 128 weight rows
//          (i-values) x 128 tokens; the epilogue writes h = silu(D_g) * D_u as bf16.
// down:    D = Wd h^T over tiles of 128 output features x 128 tokens; the epilogue writes y (fp32).
// ("DeepSeek V4 Flash CPU inference with NVMe expert streaming": FP4 E2M1 experts with UE8M0
// group-32 scales, the gate/up pair and the down projection; "the CUDA tier wired into the
// DeepSeek V4 engine": expert-grouped GEMM rows.)
//
// Swap-AB: the weights are the M operand (128 rows per tile) and the tokens of one group the N
// operand, so a group with few tokens still fills the 128-row MMA. One persistent block per SM;
// warp roles:
//   warp 0      TMA producer: packed E2M1 code rows (uint8 tensor map, 32 B x 128 rows per K step)
//               and the group's activation rows (bf16, 128-byte swizzle, 64 x 128 per K step)
//   warp 1      TMEM allocation and the MMA issuer (tcgen05.mma kind::f16, bf16 x bf16 -> fp32)
//   warps 2-5   dequantisers: E2M1 codes and their UE8M0 scales -> exact bf16 weights, written in
//               the 128-byte-swizzled K-major layout the MMA reads (e2m1 -> fp16 -> bf16 bits,
//               times 2^(s-127) by bf16 multiplies by powers of two)
//   warps 6-9   epilogue: tcgen05.ld of the fp32 accumulators, SwiGLU / store
// The accumulators are double buffered in TMEM (2 x 256 columns) so the epilogue of one tile
// overlaps the MMAs of the next. Every barrier wait is bounded (see sm103_ptx.cuh).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "colimoe_internal.cuh"
#include "sm103_ptx.cuh"

namespace colimoe {
namespace {

constexpr int BM = 128, BN = 128, BK = 64;
constexpr int NS = 3;                          // pipeline stages
constexpr int kThreads = 320;
constexpr int kDequantThreads = 128;
constexpr uint32_t kABytes = BM * BK * 2;      // one bf16 weight tile per K step: 16 KB
constexpr uint32_t kBBytes = BN * BK * 2;      // activation tile: 16 KB
constexpr uint32_t kCBytes = BM * BK / 2;      // packed codes: 4 KB
// stage layout: A0 | A1 | B | C0 | C1 (A1/C1 hold the up matrix in gate/up mode)
constexpr uint32_t kOffA0 = 0, kOffA1 = kABytes, kOffB = 2 * kABytes, kOffC0 = 2 * kABytes + kBBytes,
                   kOffC1 = kOffC0 + kCBytes;
constexpr uint32_t kStageBytes = kOffC1 + kCBytes;     // 57344, a multiple of 1024
constexpr uint32_t kTmemCols = 512;

enum Mode { kGateUp = 0, kDown = 1 };

struct TileInfo {
    int g, mt, row0, n_valid, Ig, nk;
    bool valid, shared;
    size_t ge;
};

struct GemmParams {
    int E, H, I, I_s, I_max;
    int mode, m_tiles;
    const int32_t *cnt, *off, *touched, *n_touched, *ntile_prefix, *ntile_owner;
    const uint8_t *scales_routed, *scales_shared;   // gate/up or down scales
    __nv_bfloat16 *h;
    float *y;
    int *err;
};

__device__ __forceinline__ TileInfo decode_tile(const GemmParams &p, int t) {
    TileInfo ti;
    ti.mt = t % p.m_tiles;
    const int r = t / p.m_tiles;
    const int u = p.ntile_owner[r];
    ti.g = p.touched[u];
    const int nt = r - p.ntile_prefix[u];
    ti.shared = ti.g == p.E;
    ti.Ig = ti.shared ? p.I_s : p.I;
    ti.ge = ti.shared ? 0 : (size_t)ti.g;
    ti.row0 = p.off[ti.g] + nt * BN;
    ti.n_valid = min(BN, p.cnt[ti.g] - nt * BN);
    ti.valid = p.mode == kGateUp ? ti.mt * BM < ti.Ig : true;
    ti.nk = (p.mode == kGateUp ? p.H : ti.Ig) / BK;
    return ti;
}

// tcgen05 shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);   // start address
    d |= (uint64_t)1 << 16;                            // leading byte offset (unused for SW128 K-major)
    d |= (uint64_t)(1024 >> 4) << 32;                  // stride byte offset: next 8-row atom
    d |= (uint64_t)1 << 46;                            // descriptor version for sm_100 family
    d |= (uint64_t)2 << 61;                            // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B (K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
    uint32_t r;
    asm("{\n .reg .b8 b;\n cvt.u8.u32 b, %1;\n cvt.rn.f16x2.e2m1x2 %0, b;\n}\n" : "=r"(r) : "r"(byte));
    return r;
}

// Two E2M1 codes (one byte) times 2^(s-127) as a bf16 pair. fp16 bits >> 3 (sign kept) is the bf16
// of the value times 2^-112; bf16 multiplies by 2^(s-15) (and, for s > 142, a second factor)
// restore it and apply the scale. Every step is exact except the flush of results below the
// smallest normal bf16 (scales s <= 1 only).
__device__ __forceinline__ uint32_t e2m1x2_to_bf16x2(uint32_t byte, __nv_bfloat162 f1, __nv_bfloat162 f2, bool two) {
    const uint32_t f = e2m1x2_to_f16x2(byte);
    const uint32_t b = ((f >> 3) & 0x0FFF0FFFu) | (f & 0x80008000u);
    __nv_bfloat162 r = __hmul2(*reinterpret_cast<const __nv_bfloat162 *>(&b), f1);
    if (two) r = __hmul2(r, f2);
    return *reinterpret_cast<const uint32_t *>(&r);
}

__device__ __forceinline__ __nv_bfloat162 bf16_pair(uint32_t bits) {
    const uint32_t b2 = bits | (bits << 16);
    return *reinterpret_cast<const __nv_bfloat162 *>(&b2);
}

// Factors for a UE8M0 byte: 2^(s-15) [x 2^(s-142) when s > 142]; s = 0 -> 0, s = 255 -> inf.
__device__ __forceinline__ void scale_factors(uint32_t s, __nv_bfloat162 &f1, __nv_bfloat162 &f2, bool &two) {
    two = false;
    f2 = bf16_pair(0x3F80);
    if (s == 0) {
        f1 = bf16_pair(0);
    } else if (s == 255) {
        f1 = bf16_pair(0x7F80);
    } else if (s <= 142) {
        f1 = bf16_pair((s + 112) << 7);          // exponent field (s - 15) + 127
    } else {
        f1 = bf16_pair(254u << 7);                // 2^127
        f2 = bf16_pair((s - 142 + 127) << 7);     // 2^(s - 142)
        two = true;
    }
}

// Dequantises one 64-element row of packed codes (32 bytes at `codes` + 32p) into row p of the
// 128-byte-swizzled bf16 tile `a`. sc holds the row's two group scale bytes.
__device__ __forceinline__ void dequant_row(const uint8_t *codes, uint8_t *a, int p, uint32_t sc) {
    const uint4 c0 = *reinterpret_cast<const uint4 *>(codes + p * 32);
    const uint4 c1 = *reinterpret_cast<const uint4 *>(codes + p * 32 + 16);
    __nv_bfloat162 fa1, fa2, fb1, fb2;
    bool ta, tb;
    scale_factors(sc & 0xFF, fa1, fa2, ta);
    scale_factors((sc >> 8) & 0xFF, fb1, fb2, tb);
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    uint8_t *row = a + (p >> 3) * 1024 + (p & 7) * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j) {           // 16-byte unit j holds elements 8j .. 8j+7
        const __nv_bfloat162 f1 = j < 4 ? fa1 : fb1, f2 = j < 4 ? fa2 : fb2;
        const bool two = j < 4 ? ta : tb;
        uint4 o;
        o.x = e2m1x2_to_bf16x2(w[j] & 0xFF, f1, f2, two);
        o.y = e2m1x2_to_bf16x2((w[j] >> 8) & 0xFF, f1, f2, two);
        o.z = e2m1x2_to_bf16x2((w[j] >> 16) & 0xFF, f1, f2, two);
        o.w = e2m1x2_to_bf16x2(w[j] >> 24, f1, f2, two);
        *reinterpret_cast<uint4 *>(row + ((j ^ (p & 7)) << 4)) = o;
    }
}

__global__ void __launch_bounds__(kThreads, 1)
gemm_tc(const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_c_routed,
        const __grid_constant__ CUtensorMap tm_c_shared, const GemmParams p) {
    pdl_trigger();
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + NS * kStageBytes);
    // barriers: tma_full[NS], a_full[NS], empty[NS], acc_full[2], acc_empty[2], drain
    uint64_t *tma_full = bar, *a_full = bar + NS, *empty = bar + 2 * NS, *acc_full = bar + 3 * NS,
             *acc_empty = bar + 3 * NS + 2, *drain = bar + 3 * NS + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 3 * NS + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(ptx::smem_addr(&tma_full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&a_full[s]), kDequantThreads);
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
    const bool gu = p.mode == kGateUp;
    const uint32_t tx_bytes = kBBytes + (gu ? 2 : 1) * kCBytes;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            ptx::prefetch_tmap(&tm_b);
            ptx::prefetch_tmap(&tm_c_routed);
            ptx::prefetch_tmap(&tm_c_shared);
            const uint64_t pol = ptx::policy_evict_first();
            uint32_t it = 0;
            for (int t = blockIdx.x; t < total_tiles && !*abort_flag; t += gridDim.x) {
                const TileInfo ti = decode_tile(p, t);
                if (!ti.valid) continue;
                const CUtensorMap *tc = ti.shared ? &tm_c_shared : &tm_c_routed;
                // code rows of this tile within the expert array (rows of 32-byte K steps)
                const int rows_per_expert = gu ? 2 * ti.Ig : p.H;
                const int crow0 = (int)ti.ge * rows_per_expert + ti.mt * BM;
                for (int k = 0; k < ti.nk; ++k, ++it) {
                    const int s = it % NS;
                    const uint32_t ph = (it / NS) & 1u;
                    if (!ptx::mbar_wait(ptx::smem_addr(&empty[s]), ph ^ 1u, p.err, ptx::kErrWaitEmpty, abort_flag))
                        break;
                    const uint32_t fb = ptx::smem_addr(&tma_full[s]);
                    uint8_t *st = smem + s * kStageBytes;
                    ptx::mbar_arrive_expect_tx(fb, tx_bytes);
                    ptx::tma_load_2d(ptx::smem_addr(st + kOffB), &tm_b, k * BK, ti.row0, fb);
                    ptx::tma_load_2d_hint(ptx::smem_addr(st + kOffC0), tc, k * (BK / 2), crow0, fb, pol);
                    if (gu) ptx::tma_load_2d_hint(ptx::smem_addr(st + kOffC1), tc, k * (BK / 2), crow0 + ti.Ig, fb, pol);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t it = 0, tcount = 0;
            for (int t = blockIdx.x; t < total_tiles && !*abort_flag; t += gridDim.x) {
                const TileInfo ti = decode_tile(p, t);
                if (!ti.valid) continue;
                const uint32_t buf = tcount & 1u, use = tcount >> 1;
                ++tcount;
                if (!ptx::mbar_wait(ptx::smem_addr(&acc_empty[buf]), (use & 1u) ^ 1u, p.err, ptx::kErrWaitAccum,
                                    abort_flag))
                    break;
                ptx::tc_fence_after();
                const int n_mma = (ti.n_valid + 15) & ~15;
                const uint32_t idesc = idesc_bf16(BM, n_mma);
                const uint32_t d0 = tmem + buf * 256, d1 = d0 + 128;
                bool ok = true;
                for (int k = 0; k < ti.nk; ++k, ++it) {
                    const int s = it % NS;
                    const uint32_t ph = (it / NS) & 1u;
                    if (!ptx::mbar_wait(ptx::smem_addr(&tma_full[s]), ph, p.err, ptx::kErrWaitFull, abort_flag) ||
                        !ptx::mbar_wait(ptx::smem_addr(&a_full[s]), ph, p.err, ptx::kErrWaitFull, abort_flag)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_addr(smem + s * kStageBytes);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t db = sw128_desc(sa + kOffB + kk * 32);
                        const uint32_t accum = (k > 0 || kk > 0) ? 1u : 0u;
                        ptx::mma_bf16(d0, sw128_desc(sa + kOffA0 + kk * 32), db, idesc, accum);
                        if (gu) ptx::mma_bf16(d1, sw128_desc(sa + kOffA1 + kk * 32), db, idesc, accum);
                    }
                    ptx::mma_commit(ptx::smem_addr(&empty[s]));   // frees the stage when these MMAs finish
                }
                if (!ok) break;
                ptx::mma_commit(ptx::smem_addr(&acc_full[buf]));
            }
            // drain: arrives once every MMA this thread issued has completed (at once if none is
            // in flight), so TMEM is never released under a running MMA
            ptx::mma_commit(ptx::smem_addr(drain));
            ptx::mbar_wait(ptx::smem_addr(drain), 0, nullptr, 0, nullptr);
        }
    } else if (warp < 6) {
        // ---------------------------------------------------------------- dequantisers
        const int q = threadIdx.x - 64;   // 0..127: the weight row this thread converts
        uint32_t it = 0;
        for (int t = blockIdx.x; t < total_tiles && !*abort_flag; t += gridDim.x) {
            const TileInfo ti = decode_tile(p, t);
            if (!ti.valid) continue;
            const uint8_t *sbase = ti.shared ? p.scales_shared : p.scales_routed;
            const int K = gu ? p.H : ti.Ig;
            const int rows_per_expert = gu ? 2 * ti.Ig : p.H;
            const size_t r_first = (size_t)ti.ge * rows_per_expert + ti.mt * BM + q;
            const uint16_t *s0p = reinterpret_cast<const uint16_t *>(sbase + r_first * (K / 32));
            const uint16_t *s1p = reinterpret_cast<const uint16_t *>(sbase + (r_first + ti.Ig) * (K / 32));
            uint32_t sc0 = __ldg(s0p), sc1 = gu ? __ldg(s1p) : 0u;
            bool ok = true;
            for (int k = 0; k < ti.nk; ++k, ++it) {
                // prefetch the next K step's scales
                uint32_t nsc0 = 0, nsc1 = 0;
                if (k + 1 < ti.nk) {
                    nsc0 = __ldg(s0p + k + 1);
                    if (gu) nsc1 = __ldg(s1p + k + 1);
                }
                const int s = it % NS;
                const uint32_t ph = (it / NS) & 1u;
                if (!ptx::mbar_wait(ptx::smem_addr(&tma_full[s]), ph, p.err, ptx::kErrWaitFull, abort_flag)) {
                    ok = false;
                    break;
                }
                uint8_t *st = smem + s * kStageBytes;
                dequant_row(st + kOffC0, st + kOffA0, q, sc0);
                if (gu) dequant_row(st + kOffC1, st + kOffA1, q, sc1);
                ptx::fence_proxy_async_smem();   // generic-proxy writes -> visible to the tensor core
                ptx::mbar_arrive(ptx::smem_addr(&a_full[s]));
                sc0 = nsc0;
                sc1 = nsc1;
            }
            if (!ok) break;
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int quad = warp & 3;              // TMEM lane quarter this warp may access
        const int m = quad * 32 + lane;         // accumulator row = weight row within the tile
        uint32_t tcount = 0;
        for (int t = blockIdx.x; t < total_tiles && !*abort_flag; t += gridDim.x) {
            const TileInfo ti = decode_tile(p, t);
            if (!ti.valid) continue;
            const uint32_t buf = tcount & 1u, use = tcount >> 1;
            ++tcount;
            if (!ptx::mbar_wait(ptx::smem_addr(&acc_full[buf]), use & 1u, p.err, ptx::kErrWaitAccum, abort_flag))
                break;
            ptx::tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + buf * 256;
            const int mrow = ti.mt * BM + m;
            for (int c0 = 0; c0 < ti.n_valid; c0 += 16) {
                uint32_t r0[16];
                ptx::tmem_ld16(taddr + c0, r0);
                if (gu) {
                    uint32_t r1[16];
                    ptx::tmem_ld16(taddr + 128 + c0, r1);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c0 + j < ti.n_valid) {
                            const float g = __uint_as_float(r0[j]), u = __uint_as_float(r1[j]);
                            const float hv = __fdiv_rn(g, 1.0f + expf(-g)) * u;
                            p.h[(size_t)(ti.row0 + c0 + j) * p.I_max + mrow] = __float2bfloat16_rn(hv);
                        }
                    }
                } else {
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < ti.n_valid) p.y[(size_t)(ti.row0 + c0 + j) * p.H + mrow] = __uint_as_float(r0[j]);
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

// ---- host side ------------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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

bool make_map(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    auto enc = get_encode();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct NtileArgs {
    const int32_t *cnt, *touched, *n_touched;
    int32_t *prefix, *owner;
};

// n-tile bookkeeping for the grouped GEMM: prefix[u] = sum of ceil(cnt / BN) over touched groups
// before u, owner[r] = the touched group of n-tile r. One block.
__global__ void __launch_bounds__(1024) gemm_ntiles(NtileArgs a) {
    pdl_begin();
    __shared__ int part[1024];
    const int nt = *a.n_touched;
    int carry = 0;
    for (int u0 = 0; u0 < nt; u0 += 1024) {
        const int u = u0 + threadIdx.x;
        const int c = u < nt ? (a.cnt[a.touched[u]] + BN - 1) / BN : 0;
        part[threadIdx.x] = c;
        __syncthreads();
        for (int o = 1; o < 1024; o <<= 1) {   // Hillis-Steele inclusive scan
            const int v = threadIdx.x >= o ? part[threadIdx.x - o] : 0;
            __syncthreads();
            part[threadIdx.x] += v;
            __syncthreads();
        }
        const int excl = carry + part[threadIdx.x] - c;
        if (u < nt) {
            a.prefix[u] = excl;
            for (int r = 0; r < c; ++r) a.owner[excl + r] = u;
        }
        carry += part[1023];
        __syncthreads();
    }
    if (threadIdx.x == 0) a.prefix[nt] = carry;
}

}  // namespace

bool gemm_available() { return get_encode() != nullptr; }

size_t gemm_sched_bytes(int E, int max_rows) {
    // prefix [E + 2] and owner [max_rows / BN + E + 1]
    return sizeof(int32_t) * ((size_t)E + 2 + (size_t)max_rows / BN + E + 2);
}

int launch_ffn_gemm(const FfnArgs &a, int num_sms, void *sched, cudaEvent_t mid, cudaStream_t st) {
    if (!gemm_available()) return -2;
    int32_t *prefix = static_cast<int32_t *>(sched);
    int32_t *owner = prefix + a.E + 2;
    NtileArgs na{a.cnt, a.touched, a.n_touched, prefix, owner};
    launch_pdl(gemm_ntiles, dim3(1), dim3(1024), 0, st, na);

    const size_t smem = NS * kStageBytes + 1024 + 256;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return -1;
        attr = true;
    }
    const int max_rows = a.rows;   // rows of xp / h / y used by this forward
    CUtensorMap tb, tcr, tcs;
    GemmParams p{};
    p.E = a.E;
    p.H = a.H;
    p.I = a.I;
    p.I_s = a.I_s;
    p.I_max = a.I_max;
    p.cnt = a.cnt;
    p.off = a.off;
    p.touched = a.touched;
    p.n_touched = a.n_touched;
    p.ntile_prefix = prefix;
    p.ntile_owner = owner;
    p.h = a.h;
    p.y = a.y;
    p.err = a.err;

    // gate/up: B = expert-grouped activation rows [rows][H], codes [E*2I][H/2]
    p.mode = kGateUp;
    p.m_tiles = (a.I_max + BM - 1) / BM;
    p.scales_routed = a.routed.gu_scales;
    p.scales_shared = a.shared.gu_scales;
    bool ok = make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.xp, a.H, max_rows, (uint64_t)a.H * 2, BK, BN,
                       CU_TENSOR_MAP_SWIZZLE_128B) &&
              make_map(&tcr, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.routed.gu_codes, a.H / 2, (uint64_t)a.E * 2 * a.I,
                       a.H / 2, BK / 2, BM, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (a.shared.gu_codes)
        ok = ok && make_map(&tcs, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.shared.gu_codes, a.H / 2, 2 * (uint64_t)a.I_s,
                            a.H / 2, BK / 2, BM, CU_TENSOR_MAP_SWIZZLE_NONE);
    else
        tcs = tcr;
    if (!ok) return -2;
    launch_pdl(gemm_tc, dim3(num_sms), dim3(kThreads), smem, st, tb, tcr, tcs, p);
    if (mid) cudaEventRecord(mid, st);

    // down: B = h rows [rows][I_max], codes [E*H][I/2]
    p.mode = kDown;
    p.m_tiles = a.H / BM;
    p.scales_routed = a.routed.d_scales;
    p.scales_shared = a.shared.d_scales;
    ok = make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.h, a.I_max, max_rows, (uint64_t)a.I_max * 2, BK, BN,
                  CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map(&tcr, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.routed.d_codes, a.I / 2, (uint64_t)a.E * a.H, a.I / 2,
                  BK / 2, BM, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (a.shared.d_codes)
        ok = ok && make_map(&tcs, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.shared.d_codes, a.I_s / 2, (uint64_t)a.H,
                            a.I_s / 2, BK / 2, BM, CU_TENSOR_MAP_SWIZZLE_NONE);
    else
        tcs = tcr;
    if (!ok) return -2;
    launch_pdl(gemm_tc, dim3(num_sms), dim3(kThreads), smem, st, tb, tcr, tcs, p);
    return cudaPeekAtLastError() == cudaSuccess ? 3 : -1;
}

}  // namespace colimoe
