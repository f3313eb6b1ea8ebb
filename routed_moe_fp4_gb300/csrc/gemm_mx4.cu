// A3/A4 on the tensor cores with FP4 on both sides: block-scaled tcgen05.mma kind::mxf4
// (E2M1 x E2M1, UE8M0 scale per 32 elements, fp32 accumulate, 64 K per instruction).
// ("DeepSeek V4 Flash CPU inference with NVMe expert streaming": FP4 E2M1 experts with UE8M0
// group-32 scales; the gate/up pair and the down projection. "the CUDA tier wired into the
// DeepSeek V4 engine": expert-grouped GEMM rows.)
//
// The weight codes go from HBM to the tensor cores as they are stored: a plain byte TMA with the
// 128-byte swizzle puts 256 packed E2M1 values of each weight row in one 128-byte shared-memory row
// (K = 256 per stage, 128 contiguous bytes read per row), and kind::mxf4 reads them packed. The
// UE8M0 scale bytes go to TMEM. Each MMA instruction covers 64 K, twice what the E2M1 x E4M3 kind
// covers, and block-scaled MMAs cost a roughly fixed time per instruction, so this path moves
// twice the weight bytes per instruction.
//
// Activations become four E2M1 terms, each with its own UE8M0 scale per 32 elements (the residual
// of one term is the input of the next): about 2e-4 relative error for Gaussian data, and exact
// for values with few significant bits. x terms come from quant_x4_rows (T < 64) or
// quant_x4_tokens; h terms are made in the gate/up epilogue, where a warp holds the 32 consecutive
// i-values of one scale block (with 32- and 48-token tiles the epilogue writes fp32 h and
// quant_h_rows makes them). The terms are stacked along N (term t at activation rows
// [t * bh, (t + 1) * bh)); the epilogue adds them.
//
// Tiles: 128 weight rows (M) x 16 (gate/up) or up to 32 (down) tokens of one group. One persistent
// block per SM; warp roles: TMA producer (warp 0), TMEM owner and MMA issuer (warp 1), scale
// loaders (warps 2-5; weight row 32q + i reads its scales from lane 32q + i, column (word) * 4 + q;
// activation row n from lane 32q + n % 32, column n / 32 of its word, in every lane quarter q; the
// words of one stage sit 4 columns apart; the scale bytes arrive by TMA with each stage when every
// scale row is a whole number of 16-byte chunks, else the loaders fetch them four stages ahead),
// epilogue (warps 6-13: two per lane quarter, taking alternate 8-column groups of the tile's
// tokens). Four stages,
// double-buffered accumulators, bounded waits. A stage covers 256 K (512 K for down tiles of up to
// 16 rows, which leave half of the slot free otherwise); the last stage of a K that is not a
// multiple of it is partial.
//
// Big tiles, for launches with many rows per expert (48 on average or more): the tensor pipe then
// bounds the launch, and with 16- or 32-token tiles every expert's weights are read into shared
// memory once per tile, more often than the L2 can serve at the pipe's rate. A big tile holds 48
// tokens (N = 4 x 48 = 192 per MMA) and two 128-row weight matrices that share them: the gate and
// up rows of 128 i-values, or two consecutive 128-row blocks of the down matrix (256 rows of
// hidden). Both accumulators (2 x 192 TMEM columns) live in one buffer; the scale factors take
// columns 384-511. The epilogue first moves its sums of the term columns into registers and frees
// the buffer, so the next tile's MMAs start while it computes. In the scale area an activation
// word has 8 columns (a row n < 192 reads column n / 32 of its word).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "colimoe_internal.cuh"
#include "sm103_ptx.cuh"

namespace colimoe {
namespace {

constexpr int BM = 128, BK = 256, MK = 64;     // weight rows, K per stage, K per MMA
constexpr int kBnGateUp = kNtileMx4, kBnDown = 2 * kNtileMx4;   // tokens per tile
constexpr int kTerms = 4;                      // E2M1 terms per activation
constexpr int kThreads = 448;                  // 14 warps: see the role list above
constexpr int kBnBig = 48;                     // tokens of a big tile
constexpr uint32_t kASmem = BM * BK / 2;       // 16 KB: 128 rows x 256 packed codes
constexpr uint32_t kOffA0 = 0, kOffA1 = kASmem, kOffB = 2 * kASmem;
// A stage: two weight tiles and up to 4 terms x 32 rows (48 in big tiles), a multiple of 1024 bytes.
// Small-tile launches keep the smaller stage, which leaves more of the SM's unified L1 to the
// scale loaders' reads.
template <bool BIG> constexpr uint32_t stage_bytes() { return 2 * kASmem + kTerms * (BIG ? kBnBig : 32) * (BK / 2); }
// Ring stages: four; three for big tiles, whose 56 KB stages would otherwise leave the unified L1
// too small to hold the scale loaders' sectors between stages.
template <bool BIG> constexpr int num_stages() { return BIG ? 3 : 4; }
template <bool BIG> constexpr size_t smem_bytes() { return num_stages<BIG>() * (size_t)stage_bytes<BIG>() + 1024 + 256; }
// Scales by TMA (SFT): each stage also holds the 16-byte chunk of every scale row it reads (the
// stage's 8 scale bytes lie in it; a 512-K stage reads all 16): two weight matrices x 128 rows,
// then the activation rows as [term][row], after the terms.
constexpr uint32_t kScW = 2 * BM * 16;   // weight-scale chunks of a stage
template <bool BIG> constexpr uint32_t sc_off() { return stage_bytes<BIG>(); }
template <bool BIG> constexpr uint32_t stage_bytes_sft() {
    return stage_bytes<BIG>() + kScW + kTerms * (BIG ? kBnBig : 32) * 16;
}
template <bool BIG> constexpr size_t smem_bytes_sft() {
    return num_stages<BIG>() * (size_t)stage_bytes_sft<BIG>() + 1024 + 256;
}
static_assert(stage_bytes_sft<false>() % 1024 == 0 && stage_bytes_sft<true>() % 1024 == 0, "1 KB-aligned stages");
static_assert(smem_bytes_sft<false>() <= 232448 && smem_bytes_sft<true>() <= 232448, "shared memory per block");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 128;             // per accumulator buffer (two buffers; big tiles: one)
// Scale-factor columns, 32 per stage (64 for NVFP4): after the two 128-column accumulator buffers,
// or after the 384 accumulator columns of a big tile.
template <bool BIG> constexpr uint32_t sf_col0() { return BIG ? 384 : 256; }
constexpr uint32_t kSfStage = 32;
constexpr uint32_t kSfStageNv = 64;
constexpr int kSfAhead = 4;                   // stages the scale loads run ahead (2 for NVFP4)
constexpr int kEpiWarps = 8;                  // two per TMEM lane quarter, alternate 8-column groups

enum Mode { kGateUp = 0, kDown = 1 };

struct Mx4Params {
    int E, H, I, I_s, I_max, rows;
    int mode, m_tiles, bn;
    int nbuf;                           // accumulator buffers: 2, or 1 when a tile needs more than 128 columns
    const int2 *ntile_rec;              // per n-tile: {first row, group | rows << 16}
    const int32_t *ntile_count;         // number of n-tiles
    const uint8_t *w_scales_routed, *w_scales_shared;
    const uint8_t *act_scales;          // [kTerms][rows][K/32]
    int act_ld;                         // K of the activation terms (H or I_max)
    uint8_t *hq;                        // [kTerms][rows][I_max/2] packed E2M1 terms of h
    uint8_t *hs;                        // [kTerms][rows][I_max/32]
    float *y;
    int *err;
    uint64_t wait_ns;                   // limit of the pipeline waits (the drains always allow the full limit)
};

// A separate parameter, so that the kernels keep the parameter layout of Mx4Params. NVFP4: the
// experts' fp32 matrix scales, the activations' power-of-two scales per (term, row)
// ([kTerms][rows]), and fp32 h out of the gate/up launch (act_scales then holds E4M3 bytes per
// 16). A few-token MXFP4 forward: per-group counters that the gate/up epilogue warps raise once
// each per stored tile of h terms, and the groups' row counts, so that its down launch starts on
// a group as soon as that group's h is complete instead of after the whole gate/up launch.
struct NvParams {
    const float *w_global_routed, *w_global_shared, *act_global;
    float *hf;
    int32_t *h_ready;                   // [E+1], zeroed by the x-term kernel; null: not used
    const int32_t *grp_rows;            // [E+1] rows per group (the permutation's counts)
};

// A down tile of at most 16 rows uses wide stages: 512 K, two 128-byte chunks of weights (in the
// A0 and A1 slots) and of activation terms (two halves of the B slot), eight MMAs.
struct TileInfo {
    int g, mt, row0, n_valid, Ig, K, nk, box, bh, kst;
    bool valid, shared, wide;
    size_t ge;
};



// Tile t = (n-tile t / m_tiles, m-tile t % m_tiles); `rec` is the n-tile's record.
__device__ __forceinline__ int2 tile_rec(const Mx4Params &p, int t, int total_tiles) {
    return t < total_tiles ? __ldg(p.ntile_rec + t / p.m_tiles) : make_int2(0, 0);
}

template <bool NV, bool BIG>
__device__ __forceinline__ TileInfo decode_tile(const Mx4Params &p, int t, int2 rec) {
    TileInfo ti;
    ti.mt = t % p.m_tiles;
    ti.g = rec.y & 0xFFFF;
    ti.shared = ti.g == p.E;
    ti.Ig = ti.shared ? p.I_s : p.I;
    ti.ge = ti.shared ? 0 : (size_t)ti.g;
    ti.row0 = rec.x;
    ti.n_valid = rec.y >> 16;
    ti.valid = p.mode == kGateUp ? ti.mt * BM < ti.Ig : true;
    ti.K = p.mode == kGateUp ? p.H : ti.Ig;
    ti.box = ti.n_valid <= 16 ? 0 : ti.n_valid <= 32 ? 1 : 2;   // 48-row boxes in big tiles only
    ti.bh = 16 * (ti.box + 1);
    ti.wide = !NV && p.mode == kDown && ti.box == 0 && !BIG;
    ti.kst = ti.wide ? 2 * BK : BK;
    ti.nk = (ti.K + ti.kst - 1) / ti.kst;
#ifdef COLI_BOUNDS_CHECK
    // Debug build: a tile whose records would reach outside the buffers is recorded (kErrBounds)
    // and skipped by every role alike (all of them decode the same records), never trapped. The
    // weight rows of an m-tile must lie inside its expert's matrix; the activation rows inside
    // the rows the permutation laid out; the group inside the experts plus the shared one.
    if (ti.valid && ti.n_valid > 0) {   // n_valid 0: the zero record of an index past the last tile
        const bool gu = p.mode == kGateUp;
        const int mrows = BIG && !gu ? 2 * BM : BM;
        const bool bad = ti.g > p.E || ti.n_valid < 1 || ti.n_valid > ti.bh || ti.row0 < 0 ||
                         ti.row0 + ti.n_valid > p.rows || (gu ? ti.mt * BM + BM > ti.Ig : ti.mt * mrows + mrows > p.H);
        if (bad) {
            ptx::record_error(p.err, ptx::kErrBounds);
            ti.valid = false;
        }
    }
#endif
    return ti;
}

// Scale words of one stage for one loader lane: its gate (a0) and up (a1) weight rows, and the
// activation rows lane + 32c (c < nbc); nbc == 0 marks an empty ring slot.
// In a wide stage a0 / a1 hold the weight words 0-1 / 2-3, and b[c] / b[c + 2] the words 0-1 / 2-3
// of activation column c (c < 2).
// NVFP4 stages hold four words per operand row (one per 64-K MMA) and are never wide.
template <bool NV, bool BIG> struct SfStageT {
    static constexpr int W = NV ? 4 : 2;
    static constexpr int C = BIG ? 6 : 4;   // activation column groups: 4 x 48 rows in a big tile
    uint32_t a0[W], a1[W], b[C][W];
    int nbc;
    bool wide;
};

// Position of a scale loader in the (tile, stage) sequence of its block, with the row pointers of
// the current tile.
struct SfCursor {
    int t, k, nk, K, nbc, tA, tB;
    bool wide;
    bool vw, va;                        // NVFP4: weight / activation scale rows are 16-byte aligned
    int2 recA, recB;                    // records of the next two tiles (tA < tB), loaded ahead
    const uint8_t *wp0, *wp1, *bp[6];
};

// Moves the cursor to the first valid tile at or after cur.t; false when there is none.
template <bool NV, bool BIG>
__device__ __forceinline__ bool sf_tile(const Mx4Params &p, SfCursor &c, int total_tiles, int quad, int lane) {
    const bool gu = p.mode == kGateUp;
    for (; c.t < total_tiles; c.t += gridDim.x) {
        const int2 rec = c.t == c.tA ? c.recA : c.t == c.tB ? c.recB : tile_rec(p, c.t, total_tiles);
        const TileInfo ti = decode_tile<NV, BIG>(p, c.t, rec);
        if (!ti.valid) continue;
        if (c.tB == c.t + (int)gridDim.x) {            // keep the next two records in flight
            c.tA = c.tB;
            c.recA = c.recB;
        } else {
            c.tA = c.t + gridDim.x;
            c.recA = tile_rec(p, c.tA, total_tiles);
        }
        c.tB = c.t + 2 * gridDim.x;
        c.recB = tile_rec(p, c.tB, total_tiles);
        constexpr int sdiv = NV ? 16 : 32;               // elements per scale byte
        const int kb_row = ti.K / sdiv, kba = p.act_ld / sdiv;
        const uint8_t *ws = ti.shared ? p.w_scales_shared : p.w_scales_routed;
        const int rpe = gu ? 2 * ti.Ig : p.H;
        const int mrows = BIG && !gu ? 2 * BM : BM;       // rows of the tile's m-block
        const size_t wrow = ti.ge * (size_t)rpe + (size_t)ti.mt * mrows + quad * 32 + lane;
        c.wp0 = ws + wrow * kb_row;
        c.wp1 = gu ? ws + (wrow + ti.Ig) * kb_row : BIG ? ws + (wrow + BM) * kb_row : nullptr;
        c.nbc = (kTerms * ti.bh + 31) / 32;
#pragma unroll
        for (int q = 0; q < SfStageT<NV, BIG>::C; ++q) {
            const int n = lane + 32 * q;
            const int tt = n / ti.bh, j = n % ti.bh;
            c.bp[q] = (q < c.nbc && j < ti.n_valid) ? p.act_scales + ((size_t)tt * p.rows + ti.row0 + j) * kba
                                                    : nullptr;
        }
        c.k = 0;
        c.nk = ti.nk;
        c.K = ti.K;
        c.wide = ti.wide;
        c.vw = kb_row % 16 == 0;
        c.va = kba % 16 == 0;
        return true;
    }
    return false;
}

template <bool NV, bool BIG>
__device__ __forceinline__ bool sf_next(const Mx4Params &p, SfCursor &c, int total_tiles, int quad, int lane) {
    if (++c.k < c.nk) return true;
    c.t += gridDim.x;
    return sf_tile<NV, BIG>(p, c, total_tiles, quad, lane);
}

// Issues the loads of the cursor's stage: 8 scale bytes per row (16 in a wide stage; fewer in the
// last stage of a K that is not a multiple of the stage; a missing word reads as scale 1).
template <bool NV, bool BIG>
__device__ __forceinline__ void sf_fetch(const SfCursor &c, SfStageT<NV, BIG> &s, int n_a) {
    if constexpr (NV) {   // four words (16 scale bytes) per row and stage; a missing word reads as 1.0
        const int nw = min(BK, c.K - c.k * BK) / 64;
        const int w0 = c.k * 4;
        // a full stage of a 16-byte aligned row is one 16-byte load; other rows, and the last stage
        // of a K that is not a multiple of 256, load word by word
        auto ld4 = [&](const uint8_t *q, bool vec, uint32_t (&o)[4]) {
            if (!q) {
#pragma unroll
                for (int w = 0; w < 4; ++w) o[w] = 0x38383838u;
            } else if (vec && nw == 4) {
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(q) + c.k);
                o[0] = v.x;
                o[1] = v.y;
                o[2] = v.z;
                o[3] = v.w;
            } else {
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    o[w] = w < nw ? __ldg(reinterpret_cast<const uint32_t *>(q) + w0 + w) : 0x38383838u;
            }
        };
        ld4(c.wp0, c.vw, s.a0);
        ld4(n_a > 1 ? c.wp1 : nullptr, c.vw, s.a1);
#pragma unroll
        for (int q = 0; q < 4; ++q) ld4(c.bp[q], c.va, s.b[q]);
        s.nbc = c.nbc;
        s.wide = false;
        return;
    } else {
    const int kst = c.wide ? 2 * BK : BK;
    const int nw = min(kst, c.K - c.k * kst) / 128;         // valid words of this stage (1 to 4)
    const int w0 = c.k * (kst / 128);
    auto ld = [&](const uint8_t *q, int w) -> uint32_t {
        return (q && w < nw) ? __ldg(reinterpret_cast<const uint32_t *>(q) + w0 + w) : 0x7F7F7F7Fu;
    };
    // full stages of 16-byte aligned rows: one 8-byte (16 in a wide stage) load per row
    if (c.wide && nw == 4 && c.vw && c.va) {
        const uint4 a = __ldg(reinterpret_cast<const uint4 *>(c.wp0) + c.k);
        s.a0[0] = a.x;
        s.a0[1] = a.y;
        s.a1[0] = a.z;
        s.a1[1] = a.w;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint4 v = c.bp[q] ? __ldg(reinterpret_cast<const uint4 *>(c.bp[q]) + c.k)
                                    : make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
            s.b[q][0] = v.x;
            s.b[q][1] = v.y;
            s.b[q + 2][0] = v.z;
            s.b[q + 2][1] = v.w;
        }
    } else if (!c.wide && nw == 2 && c.vw && c.va) {
        auto ld2 = [&](const uint8_t *q, uint32_t (&o)[2]) {
            const uint2 v = q ? __ldg(reinterpret_cast<const uint2 *>(q) + c.k) : make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
            o[0] = v.x;
            o[1] = v.y;
        };
        ld2(c.wp0, s.a0);
        ld2(n_a > 1 ? c.wp1 : nullptr, s.a1);
#pragma unroll
        for (int q = 0; q < SfStageT<NV, BIG>::C; ++q) ld2(c.bp[q], s.b[q]);
    } else if (c.wide) {
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            s.a0[w] = ld(c.wp0, w);
            s.a1[w] = ld(c.wp0, w + 2);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                s.b[q][w] = ld(c.bp[q], w);
                s.b[q + 2][w] = ld(c.bp[q], w + 2);
            }
        }
    } else {
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            s.a0[w] = ld(c.wp0, w);
            s.a1[w] = n_a > 1 ? ld(c.wp1, w) : 0x7F7F7F7Fu;
#pragma unroll
            for (int q = 0; q < SfStageT<NV, BIG>::C; ++q) s.b[q][w] = ld(c.bp[q], w);
        }
    }
    s.nbc = c.nbc;
    s.wide = c.wide;
    }
}

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Block-scaled descriptor, kind::mxf4: A and B E2M1 (1), UE8M0, M x N; sf_id 0 or 2 selects the
// scale byte pair of the 64-wide MMA within a 128-wide scale word.
__device__ __forceinline__ uint32_t idesc_mx4(int N, int sf_id) {
    return ((uint32_t)sf_id << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
           ((uint32_t)(BM >> 4) << 24) | ((uint32_t)sf_id << 29);
}

__device__ __forceinline__ void mma_mx4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                        uint32_t sfb, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n}\n"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
}

// kind::mxf4nvf4 with UE4M3 scales per 16 (scale_vec::4X): one scale word per row per MMA.
__device__ __forceinline__ uint32_t idesc_nv4(int N) {
    return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void mma_nv4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                        uint32_t sfb, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}\n"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void tmem_st_x1(uint32_t taddr, uint32_t a) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(a) : "memory");
}

// 32 lanes x 16 consecutive columns.
__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Writes one stage's scale words of this loader lane to TMEM at column `col` of its lane quarter.
// NVFP4: A0 words at +4w, A1 at +16 + 4w, activation words at +32 + 4w. Lane 32q + i reads only
// column 4w + q of a weight group, so each word is written to all four columns of its group: one
// 16-column store per operand. MXFP4: weight words 0-3 (a0 then a1; in a wide stage a1 holds
// words 2-3) at +4w, each written to its whole 4-column group; the activation words of column
// group c at +16 + 4w + c (a wide stage's words 2-3 at +24 + 4w + c); big tiles: activation word
// w of column group c at +16 + 8w + c (c < 6). Columns a stage does not use take any value.
template <bool NV, bool BIG>
__device__ __forceinline__ void store_sf_stage(uint32_t col, const SfStageT<NV, BIG> &w, int n_a) {
    uint32_t r[16];
    if constexpr (NV) {
#pragma unroll
        for (int j = 0; j < 16; ++j) r[j] = w.a0[j >> 2];
        tmem_st_x16(col, r);
        if (n_a > 1) {
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = w.a1[j >> 2];
            tmem_st_x16(col + 16, r);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) r[j] = w.b[j & 3][j >> 2];
        tmem_st_x16(col + 32, r);
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) r[j] = j < 8 ? w.a0[(j >> 2) & 1] : w.a1[(j >> 2) & 1];
        tmem_st_x16(col, r);
        if constexpr (BIG) {
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = (j & 7) < 6 ? w.b[j & 7][j >> 3] : 0x7F7F7F7Fu;
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j)
                r[j] = j < 8 ? w.b[j & 3][(j >> 2) & 1] : w.b[((j & 3) + 2) & 3][(j >> 2) & 1];
        }
        tmem_st_x16(col + 16, r);
    }
}

// Largest of 32 non-negative floats across the warp: their bit patterns order like unsigned
// integers, so one integer warp reduction serves.
__device__ __forceinline__ float warp_max_abs(float a) {
    return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(a)));
}

// UE8M0 byte for an E2M1 term of a block with maximum amax: |v| / 2^(s-127) < 4.
__device__ __forceinline__ uint32_t e2m1_scale_byte(float amax) {
    const uint32_t ef = (__float_as_uint(amax) >> 23) & 0xFF;
    const uint32_t s = (amax > 0.f && ef < 255) ? (ef > 2 ? ef - 1 : 1) : 127;
    return min(s, 253u);
}

// Two values -> one byte of E2M1 codes (lo in bits 0-3) and their decoded values.
__device__ __forceinline__ uint32_t e2m1_pair(float lo, float hi, float &blo, float &bhi) {
    uint32_t b;
    asm("{\n .reg .b8 q;\n cvt.rn.satfinite.e2m1x2.f32 q, %1, %2;\n cvt.u32.u8 %0, q;\n}\n"
        : "=r"(b) : "f"(hi), "f"(lo));
    uint32_t h2;
    asm("{\n .reg .b8 q;\n cvt.u8.u32 q, %1;\n cvt.rn.f16x2.e2m1x2 %0, q;\n}\n" : "=r"(h2) : "r"(b));
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
    blo = f.x;
    bhi = f.y;
    return b;
}

// One token's value of h at i = mrow (lane = i mod 32): SwiGLU of the gate and up sums, then four
// E2M1 terms, each with its UE8M0 scale per 32 consecutive i (one warp), stored to hq / hs. Called
// by all lanes of a warp together. Not inlined: a big tile's epilogue finishes 24 tokens per warp,
// and as many inlined copies overflow the instruction cache the MMA and TMA warps share.
__device__ __noinline__ void finish_h(float g, float u, size_t row, int mrow, int lane, uint8_t *hq, uint8_t *hs,
                                      int rows, int I_max) {
    float v = __fdiv_rn(g, 1.0f + expf(-g)) * u;
#pragma unroll
    for (int tt = 0; tt < kTerms; ++tt) {
        const uint32_t sb = e2m1_scale_byte(warp_max_abs(fabsf(v)));
        const float scale = __uint_as_float(sb << 23), inv = __uint_as_float((254u - sb) << 23);
        float back, unused;
        const uint32_t code = e2m1_pair(v * inv, 0.f, back, unused) & 0xF;
        v -= back * scale;
        const uint32_t hi = __shfl_down_sync(0xffffffffu, code, 1);
        if ((lane & 1) == 0) hq[((size_t)tt * rows + row) * (I_max / 2) + mrow / 2] = (uint8_t)(code | (hi << 4));
        if (lane == 0) hs[((size_t)tt * rows + row) * (I_max / 32) + mrow / 32] = (uint8_t)sb;
    }
}

template <bool BIG> struct BMaps4 {
    CUtensorMap m[kTerms][BIG ? 3 : 2];   // [term][box height 16 / 32 / 48]
};

// SFT launches: the weight scales (routed, shared: [rows][K/32] bytes, 16 x 128 boxes) and the
// activation scales ([kTerms][rows][K/32] bytes, 16 x box height x kTerms boxes, by box height).
template <bool BIG> struct ScMaps {
    CUtensorMap w_routed, w_shared, act[BIG ? 3 : 2];
};

// SFT: the scale bytes come by TMA with each stage (ScMaps), and the scale loaders read them from
// shared memory; otherwise the loaders fetch them from global memory, stages ahead.
template <int MODE, bool NV, bool BIG, bool SFT>
__global__ void __launch_bounds__(kThreads, 1)
gemm_mx4(const __grid_constant__ CUtensorMap tm_a_routed, const __grid_constant__ CUtensorMap tm_a_shared,
         const __grid_constant__ BMaps4<BIG> tm_b, const Mx4Params p, const __grid_constant__ NvParams q,
         const __grid_constant__ ScMaps<BIG> tm_sc) {
    constexpr uint32_t kStageBytes = SFT ? stage_bytes_sft<BIG>() : stage_bytes<BIG>(), kSfCol0 = sf_col0<BIG>();
    constexpr uint32_t kOffSc = sc_off<BIG>();
    constexpr int NS = num_stages<BIG>();
    // The kernel before this one in the stream (an x- or h-term kernel, or the gate/up launch
    // before the down launch) signals its dependents only after its own dependency wait, so every kernel up
    // to the permutation has completed when this one starts: its tile records can be read, and the
    // first weight stages issued, before the wait. Activation terms and scales, and all writes,
    // come after it.
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + NS * kStageBytes);
    uint64_t *tma_full = bar, *sf_full = bar + NS, *empty = bar + 2 * NS, *acc_full = bar + 3 * NS,
             *acc_empty = bar + 3 * NS + 2, *drain = bar + 3 * NS + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 3 * NS + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr bool gu = MODE == kGateUp;
    constexpr int n_a = gu || BIG ? 2 : 1;          // weight matrices: gate and up, or two down row blocks
    constexpr int mrows = BIG && !gu ? 2 * BM : BM; // weight rows of one m-tile
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(ptx::smem_addr(&tma_full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&sf_full[s]), 128);
            ptx::mbar_init(ptx::smem_addr(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
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
    const int total_tiles = p.m_tiles * *p.ntile_count;   // a permutation output: see above

    // The down launch of a few-token forward (h counters given) does not wait for the gate/up
    // launch to finish: its producer waits, per tile, for the group's counter, and no other role
    // reads what the gate/up launch writes.
    const bool early = !gu && q.h_ready != nullptr;
    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            ptx::prefetch_tmap(&tm_a_routed);
            ptx::prefetch_tmap(&tm_a_shared);
            const uint64_t pol = ptx::policy_evict_first();
            // stage k of tile ti into slot s: the weights (A, with the stage's byte count) and the
            // activation terms (B) are issued separately
            auto issue_a = [&](const TileInfo &ti, int k, int s) {
                const uint32_t bbytes = kTerms * ti.bh * (BK / 2);   // one 128-byte K chunk of the terms
                const CUtensorMap *ta = ti.shared ? &tm_a_shared : &tm_a_routed;
                const int rpe = gu ? 2 * ti.Ig : p.H;
                const int arow = (int)ti.ge * rpe + ti.mt * mrows;
                const uint32_t fb = ptx::smem_addr(&tma_full[s]);
                const uint32_t st = ptx::smem_addr(smem + s * kStageBytes);
                const int x0 = k * (ti.kst / 2);                      // byte offset along K
                const bool two = !gu && ti.wide && ti.K - k * ti.kst > BK;   // second K chunk
                // SFT: the scale chunks of the weight rows (one per matrix) and of the activation
                // rows (one box of kTerms x bh rows), 16 bytes each, on the same barrier
                const uint32_t scbytes = SFT ? n_a * BM * 16 + kTerms * ti.bh * 16 : 0;
                ptx::mbar_arrive_expect_tx(fb, (n_a == 2 || two ? 2 : 1) * kASmem + (two ? 2 : 1) * bbytes + scbytes);
                ptx::tma_load_2d_hint(st + kOffA0, ta, x0, arow, fb, pol);
                if (n_a == 2) ptx::tma_load_2d_hint(st + kOffA1, ta, x0, arow + (gu ? ti.Ig : BM), fb, pol);
                if (two) ptx::tma_load_2d_hint(st + kOffA1, ta, x0 + BK / 2, arow, fb, pol);
                if constexpr (SFT) {   // byte offset of the stage's chunk along a scale row
                    const CUtensorMap *tw = ti.shared ? &tm_sc.w_shared : &tm_sc.w_routed;
                    const int xs = NV || ti.wide ? k * 16 : (k * 8) & ~15;   // NVFP4: 16 bytes a stage
                    ptx::tma_load_2d(st + kOffSc, tw, xs, arow, fb);
                    if (n_a == 2) ptx::tma_load_2d(st + kOffSc + BM * 16, tw, xs, arow + (gu ? ti.Ig : BM), fb);
                }
            };
            auto issue_b = [&](const TileInfo &ti, int k, int s) {
                const uint32_t bbytes = kTerms * ti.bh * (BK / 2);
                const uint32_t fb = ptx::smem_addr(&tma_full[s]);
                const uint32_t st = ptx::smem_addr(smem + s * kStageBytes);
                const int x0 = k * (ti.kst / 2);
                const bool two = !gu && ti.wide && ti.K - k * ti.kst > BK;
                if constexpr (SFT)   // the activation rows' scale chunks, [term][row]
                    ptx::tma_load_3d(st + kOffSc + kScW, &tm_sc.act[ti.box], NV || ti.wide ? k * 16 : (k * 8) & ~15,
                                     ti.row0, 0, fb);
#pragma unroll
                for (int tt = 0; tt < kTerms; ++tt) {
                    ptx::tma_load_2d(st + kOffB + tt * ti.bh * (BK / 2), &tm_b.m[tt][ti.box], x0, ti.row0, fb);
                    if (two)
                        ptx::tma_load_2d(st + kOffB + bbytes + tt * ti.bh * (BK / 2), &tm_b.m[tt][ti.box],
                                         x0 + BK / 2, ti.row0, fb);
                }
            };
            // the group's h terms are all stored: every epilogue warp of each of its gate/up tiles
            // (row tiles of kBnGateUp tokens, m-tiles of BM rows of its intermediate size) has
            // raised the counter; then TMA may load them (proxy fence after the acquire). A wait
            // that runs out records kErrWaitH and aborts; the loads are still issued, so that every
            // stage's barrier completes.
            auto h_wait = [&](const TileInfo &ti) {
                const int c = __ldg(q.grp_rows + ti.g);
                const int target = kEpiWarps * ((c + kBnGateUp - 1) / kBnGateUp) * ((ti.Ig + BM - 1) / BM);
                ptx::wait_counter(q.h_ready + ti.g, target, p.err, ptx::kErrWaitH, abort_flag, p.wait_ns);
                ptx::fence_proxy_async_global();
            };
            // before the wait: the weights of the first stages of the first tile (all slots are free)
            int t0 = blockIdx.x, pre = 0;
            int2 rec = tile_rec(p, t0, total_tiles);
            TileInfo ti0 = decode_tile<NV, BIG>(p, t0, rec);
            while (t0 < total_tiles && !ti0.valid) {
                t0 += gridDim.x;
                ti0 = decode_tile<NV, BIG>(p, t0, tile_rec(p, t0, total_tiles));
            }
            if (t0 < total_tiles) {
                pre = min(NS, ti0.nk);
                for (int k = 0; k < pre; ++k) issue_a(ti0, k, k);
            }
            if (early) {
                pdl_trigger();
                if (t0 < total_tiles) h_wait(ti0);
            } else {
                pdl_wait();
                pdl_trigger();
            }
            for (int k = 0; k < pre; ++k) issue_b(ti0, k, k);
            uint32_t it = 0;
            for (int t = blockIdx.x; t < total_tiles && !*abort_flag; t += gridDim.x) {
                const int2 cur = rec;
                rec = tile_rec(p, t + gridDim.x, total_tiles);   // in flight during this tile
                const TileInfo ti = decode_tile<NV, BIG>(p, t, cur);
                if (!ti.valid) continue;
                if (early && t != t0) h_wait(ti);
                for (int k = 0; k < ti.nk; ++k, ++it) {
                    if (t == t0 && k < pre) continue;             // issued above
                    const int s = it % NS;
                    if (!ptx::mbar_wait(ptx::smem_addr(&empty[s]), ((it / NS) & 1u) ^ 1u, p.err, ptx::kErrWaitEmpty,
                                        abort_flag, p.wait_ns))
                        break;
                    issue_a(ti, k, s);
                    issue_b(ti, k, s);
                }
            }
            // copies still in flight (only after a wait gave up): let them land before the block
            // exits, with the full limit
            const uint32_t issued = it > (uint32_t)pre ? it : (uint32_t)pre;
            for (uint32_t i = issued > (uint32_t)NS ? issued - NS : 0; i < issued; ++i)
                ptx::mbar_wait(ptx::smem_addr(&tma_full[i % NS]), (i / NS) & 1u, nullptr, 0, nullptr);
        } else if (!early) {
            pdl_wait();
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint64_t desc0 = sw128_desc(ptx::smem_addr(smem));   // stage 0, matrix A0
            uint32_t it = 0, tcount = 0;
            int2 rec = tile_rec(p, blockIdx.x, total_tiles);
            for (int t = blockIdx.x; t < total_tiles && !*abort_flag; t += gridDim.x) {
                const int2 cur = rec;
                rec = tile_rec(p, t + gridDim.x, total_tiles);   // in flight during this tile
                const TileInfo ti = decode_tile<NV, BIG>(p, t, cur);
                if (!ti.valid) continue;
                const uint32_t buf = p.nbuf == 2 ? tcount & 1u : 0u, use = p.nbuf == 2 ? tcount >> 1 : tcount;
                if (!ptx::mbar_wait(ptx::smem_addr(&acc_empty[buf]), (use & 1u) ^ 1u, p.err, ptx::kErrWaitAccum,
                                    abort_flag, p.wait_ns))
                    break;
                ++tcount;
                ptx::tc_fence_after();
                const int n_mma = kTerms * ti.bh;
                const uint32_t id0 = idesc_mx4(n_mma, 0), id2 = idesc_mx4(n_mma, 2);
                const uint32_t d0 = tmem + buf * kAccCols, d1 = d0 + (uint32_t)n_mma;
                uint32_t acc = 0;
                bool ok = true;
                for (int k = 0; k < ti.nk; ++k, ++it) {
                    const int s = it % NS;
                    const uint32_t ph = (it / NS) & 1u;
                    if (!ptx::mbar_wait(ptx::smem_addr(&tma_full[s]), ph, p.err, ptx::kErrWaitFull, abort_flag,
                                        p.wait_ns) ||
                        !ptx::mbar_wait(ptx::smem_addr(&sf_full[s]), ph, p.err, ptx::kErrWaitFull, abort_flag,
                                        p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    // descriptors of this stage: the start-address field advances by 32 B (2) per MMA
                    const uint64_t a0 = desc0 + (uint64_t)(s * (kStageBytes >> 4));
                    const uint64_t a1 = a0 + (kOffA1 >> 4), b = a0 + (kOffB >> 4);
                    const int nsteps = min(ti.kst, ti.K - k * ti.kst) / 64;   // 2, 4, 6 or 8
                    if constexpr (NV) {   // one scale word per MMA, four words per operand and stage
                        const uint32_t sfa = tmem + kSfCol0 + s * kSfStageNv, sfb = sfa + 32;
                        const uint32_t idn = idesc_nv4(n_mma);
                        for (int j = 0; j < nsteps; ++j) {
                            mma_nv4(d0, a0 + 2 * j, b + 2 * j, idn, sfa + 4 * j, sfb + 4 * j, acc);
                            if (gu) mma_nv4(d1, a1 + 2 * j, b + 2 * j, idn, sfa + 16 + 4 * j, sfb + 4 * j, acc);
                            acc = 1;
                        }
                        ptx::mma_commit(ptx::smem_addr(&empty[s]));
                        continue;
                    }
                    const uint32_t sfa = tmem + kSfCol0 + s * kSfStage, sfb = sfa + 16;
                    constexpr uint32_t bws = BIG ? 8 : 4;                  // activation word stride
                    auto step = [&](int j) {
                        const uint32_t id = (j & 1) ? id2 : id0;
                        const uint32_t sw = 4 * (j >> 1);                  // scale word j / 2
                        if (n_a == 2) {
                            const uint32_t bw = bws * (j >> 1);
                            mma_mx4(d0, a0 + 2 * j, b + 2 * j, id, sfa + sw, sfb + bw, acc);
                            mma_mx4(d1, a1 + 2 * j, b + 2 * j, id, sfa + 8 + sw, sfb + bw, acc);
                        } else if (j < 4) {
                            mma_mx4(d0, a0 + 2 * j, b + 2 * j, id, sfa + sw, sfb + sw, acc);
                        } else {                                           // second chunk of a wide stage
                            constexpr uint64_t kHalfB = (kTerms * 16 * (BK / 2)) >> 4;
                            mma_mx4(d0, a1 + 2 * (j - 4), b + kHalfB + 2 * (j - 4), id, sfa + sw, sfb + sw, acc);
                        }
                        acc = 1;
                    };
                    step(0);
                    step(1);
                    if (nsteps > 2) {
                        step(2);
                        step(3);
                    }
                    if (!gu && nsteps > 4) {
                        step(4);
                        step(5);
                        if (nsteps > 6) {
                            step(6);
                            step(7);
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
    } else if (warp < 6 && SFT) {
        // ------------------------------------------------------------------ scale loaders (SFT)
        // Each stage's scale chunks arrive by TMA with its weights: once the stage has landed,
        // this lane takes its weight row's words (row quad * 32 + lane of each matrix) and those
        // of activation columns lane + 32c from shared memory, and writes them to the stage's TMEM
        // scale columns. (The TMA into a slot is issued only after the MMAs that read the slot's
        // previous scale columns have completed.)
        const int quad = warp & 3, m = quad * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        uint32_t it = 0;
        bool run = true;
        int2 rec = tile_rec(p, blockIdx.x, total_tiles);
        for (int t = blockIdx.x; t < total_tiles && run; t += gridDim.x) {
            const int2 cur = rec;
            rec = tile_rec(p, t + gridDim.x, total_tiles);
            const TileInfo ti = decode_tile<NV, BIG>(p, t, cur);
            if (!ti.valid) continue;
            for (int k = 0; k < ti.nk; ++k, ++it) {
                const int s = it % NS;
                // warp-uniform: the TMEM stores below are warp-wide
                if (__any_sync(0xffffffffu, *abort_flag != 0) ||
                    !__all_sync(0xffffffffu, ptx::mbar_wait(ptx::smem_addr(&tma_full[s]), (it / NS) & 1u, p.err,
                                                             ptx::kErrWaitFull, abort_flag, p.wait_ns))) {
                    run = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint8_t *sc = smem + s * kStageBytes + kOffSc;
                const uint8_t *sa = sc + kScW;
                SfStageT<NV, BIG> w;
                if constexpr (NV) {   // four words per row, one per 64-K MMA
                    const uint4 a0 = *reinterpret_cast<const uint4 *>(sc + m * 16);
                    const uint4 a1 = n_a > 1 ? *reinterpret_cast<const uint4 *>(sc + BM * 16 + m * 16)
                                             : make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
                    w.a0[0] = a0.x;
                    w.a0[1] = a0.y;
                    w.a0[2] = a0.z;
                    w.a0[3] = a0.w;
                    w.a1[0] = a1.x;
                    w.a1[1] = a1.y;
                    w.a1[2] = a1.z;
                    w.a1[3] = a1.w;
#pragma unroll
                    for (int c = 0; c < SfStageT<NV, BIG>::C; ++c) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(sa + (lane + 32 * c) * 16);
                        w.b[c][0] = v.x;
                        w.b[c][1] = v.y;
                        w.b[c][2] = v.z;
                        w.b[c][3] = v.w;
                    }
                } else if (ti.wide) {   // 16 bytes per row: words 0-1 and 2-3
                    const uint4 a = *reinterpret_cast<const uint4 *>(sc + m * 16);
                    w.a0[0] = a.x;
                    w.a0[1] = a.y;
                    w.a1[0] = a.z;
                    w.a1[1] = a.w;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(sa + (lane + 32 * c) * 16);
                        w.b[c][0] = v.x;
                        w.b[c][1] = v.y;
                        w.b[c + 2][0] = v.z;
                        w.b[c + 2][1] = v.w;
                    }
                } else {         // the stage's 8 bytes: the chunk's half k & 1
                    const int h = (k & 1) * 8;
                    const uint2 a0 = *reinterpret_cast<const uint2 *>(sc + m * 16 + h);
                    w.a0[0] = a0.x;
                    w.a0[1] = a0.y;
                    if (n_a > 1) {
                        const uint2 a1 = *reinterpret_cast<const uint2 *>(sc + BM * 16 + m * 16 + h);
                        w.a1[0] = a1.x;
                        w.a1[1] = a1.y;
                    } else {
                        w.a1[0] = w.a1[1] = 0x7F7F7F7Fu;
                    }
#pragma unroll
                    for (int c = 0; c < SfStageT<NV, BIG>::C; ++c) {
                        const uint2 v = *reinterpret_cast<const uint2 *>(sa + (lane + 32 * c) * 16 + h);
                        w.b[c][0] = v.x;
                        w.b[c][1] = v.y;
                    }
                }
                store_sf_stage<NV, BIG>(lane_base + kSfCol0 + s * (NV ? kSfStageNv : kSfStage), w, n_a);
                tmem_st_wait();
                ptx::tc_fence_before();
                ptx::mbar_arrive(ptx::smem_addr(&sf_full[s]));
            }
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------------ scale loaders
        // The scale words of stage it + kSfAhead are fetched while stage it is stored, so the
        // global-load latency overlaps kSfAhead stages of MMA work. Each ring slot keeps its
        // registers (the loop is unrolled over the slots): nothing waits on a load until the
        // slot's words are stored.
        const int quad = warp & 3;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        SfCursor cur;
        cur.t = blockIdx.x;
        cur.tA = cur.tB = -1;
        bool live = sf_tile<NV, BIG>(p, cur, total_tiles, quad, lane);   // tile records: readable before the wait
        if (live) {   // this lane's weight-scale rows of the first tile into L2 meanwhile
            for (int o = 0; o < cur.K / 32; o += 128) {
                asm volatile("prefetch.global.L2 [%0];" ::"l"(cur.wp0 + o));
                if (n_a > 1) asm volatile("prefetch.global.L2 [%0];" ::"l"(cur.wp1 + o));
            }
        }
        pdl_wait();
        constexpr int kAhead = NV ? 2 : BIG ? 3 : kSfAhead;
        SfStageT<NV, BIG> ring[kAhead];
#pragma unroll
        for (int d = 0; d < kAhead; ++d) {
            ring[d].nbc = 0;
            if (live) {
                sf_fetch(cur, ring[d], n_a);
                live = sf_next<NV, BIG>(p, cur, total_tiles, quad, lane);
            }
        }
        uint32_t it = 0;
        bool run = true;
        while (run) {
#pragma unroll
            for (int d = 0; d < kAhead; ++d) {
                if (!run || ring[d].nbc == 0 || *abort_flag) {
                    run = false;
                    continue;
                }
                const int s = it % NS;
                if (!ptx::mbar_wait(ptx::smem_addr(&empty[s]), ((it / NS) & 1u) ^ 1u, p.err, ptx::kErrWaitEmpty,
                                    abort_flag, p.wait_ns)) {
                    run = false;
                    continue;
                }
                ptx::tc_fence_after();
                store_sf_stage<NV, BIG>(lane_base + kSfCol0 + s * (NV ? kSfStageNv : kSfStage), ring[d], n_a);
                tmem_st_wait();
                ptx::tc_fence_before();
                ptx::mbar_arrive(ptx::smem_addr(&sf_full[s]));
                ++it;
                ring[d].nbc = 0;
                if (live) {
                    sf_fetch(cur, ring[d], n_a);
                    live = sf_next<NV, BIG>(p, cur, total_tiles, quad, lane);
                }
            }
        }
    } else {
        // ------------------------------------------------------------------ epilogue
        if (!early) pdl_wait();   // early: it writes only y, which nothing before it reads
        const int quad = warp & 3;
        const int half = (warp - 6) >> 2;             // this warp's 8-column groups: half, half + 2, ...
        const int m = quad * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        uint32_t tcount = 0;
        int2 rec = tile_rec(p, blockIdx.x, total_tiles);
        for (int t = blockIdx.x; t < total_tiles && !*abort_flag; t += gridDim.x) {
            const int2 cur = rec;
            rec = tile_rec(p, t + gridDim.x, total_tiles);
            const TileInfo ti = decode_tile<NV, BIG>(p, t, cur);
            if (!ti.valid) continue;
            const uint32_t buf = p.nbuf == 2 ? tcount & 1u : 0u, use = p.nbuf == 2 ? tcount >> 1 : tcount;
            if (!ptx::mbar_wait(ptx::smem_addr(&acc_full[buf]), use & 1u, p.err, ptx::kErrWaitAccum, abort_flag,
                                p.wait_ns))
                break;
            ++tcount;
            ptx::tc_fence_after();
            const int mrow = ti.mt * mrows + m;
            const uint32_t acc = lane_base + buf * kAccCols;
            const int ncols = kTerms * ti.bh;
            if constexpr (BIG) {
                // Big tile: this warp's token groups c0 = 8 * half + 16 * gi (gi < 3). First the
                // sums of the term columns of both matrices into registers; then the buffer is
                // released and the next tile's MMAs run while the values are finished and stored.
                float s0[3][8], s1[3][8];
#pragma unroll
                for (int gi = 0; gi < 3; ++gi) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) s0[gi][j] = s1[gi][j] = 0.f;
                    const int c0 = 8 * half + 16 * gi;
                    if (c0 >= ti.n_valid) continue;
#pragma unroll
                    for (int tt = 0; tt < kTerms; ++tt) {
                        uint32_t r[8], r1[8];
                        ptx::tmem_ld8(acc + tt * ti.bh + c0, r);
                        ptx::tmem_ld8(acc + ncols + tt * ti.bh + c0, r1);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            s0[gi][j] += __uint_as_float(r[j]);
                            s1[gi][j] += __uint_as_float(r1[j]);
                        }
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&acc_empty[buf]));
#pragma unroll
                for (int gi = 0; gi < 3; ++gi) {
                    const int c0 = 8 * half + 16 * gi;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (c0 + j >= ti.n_valid) break;
                        const size_t row = (size_t)ti.row0 + c0 + j;
                        if (!gu) {            // two 128-row blocks of the down output
                            p.y[row * p.H + mrow] = s0[gi][j];
                            p.y[row * p.H + mrow + BM] = s1[gi][j];
                        } else if (q.hf) {    // h in fp32; quant_h_rows makes its terms
                            const float g = s0[gi][j];
                            q.hf[row * p.I_max + mrow] = __fdiv_rn(g, 1.0f + expf(-g)) * s1[gi][j];
                        } else {
                            finish_h(s0[gi][j], s1[gi][j], row, mrow, lane, p.hq, p.hs, p.rows, p.I_max);
                        }
                    }
                }
                continue;
            }
            float wg = 1.f;   // NVFP4: the matrix scale of this tile's expert
            if constexpr (NV) wg = __ldg(ti.shared ? q.w_global_shared : q.w_global_routed + ti.ge);
            for (int c0 = 8 * half; c0 < ti.n_valid; c0 += 16) {
                float v0[8], v1[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) v0[j] = v1[j] = 0.f;
#pragma unroll
                for (int tt = 0; tt < kTerms; ++tt) {   // add the term columns (gate and up: one wait)
                    uint32_t r[8], r1[8];
                    ptx::tmem_ld8(acc + tt * ti.bh + c0, r);
                    if (gu) ptx::tmem_ld8(acc + ncols + tt * ti.bh + c0, r1);
                    if constexpr (NV) {   // each term column times its power-of-two scale for that row
                        float ag[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            ag[j] = c0 + j < ti.n_valid
                                        ? __ldg(q.act_global + (size_t)tt * p.rows + ti.row0 + c0 + j) : 0.f;
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 8; ++j) v0[j] = fmaf(__uint_as_float(r[j]), ag[j], v0[j]);
                        if (gu) {
#pragma unroll
                            for (int j = 0; j < 8; ++j) v1[j] = fmaf(__uint_as_float(r1[j]), ag[j], v1[j]);
                        }
                    } else {
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 8; ++j) v0[j] += __uint_as_float(r[j]);
                        if (gu) {
#pragma unroll
                            for (int j = 0; j < 8; ++j) v1[j] += __uint_as_float(r1[j]);
                        }
                    }
                }
                for (int j = 0; j < 8 && c0 + j < ti.n_valid; ++j) {
                    const size_t row = (size_t)ti.row0 + c0 + j;
                    if (!gu) {
                        if constexpr (NV) p.y[row * p.H + mrow] = v0[j] * wg;
                        else p.y[row * p.H + mrow] = v0[j];
                        continue;
                    }
                    // h in fp32, and the next kernel splits it into terms: NVFP4, and MXFP4 launches
                    // with 32-token tiles (the MXFP4 instantiation that takes them holds the code)
                    if (NV || (!SFT && q.hf)) {
                        const float g = v0[j] * wg, u = v1[j] * wg;
                        q.hf[row * p.I_max + mrow] = __fdiv_rn(g, 1.0f + expf(-g)) * u;
                        continue;
                    }
                    float v = __fdiv_rn(v0[j], 1.0f + expf(-v0[j])) * v1[j];
#pragma unroll
                    for (int tt = 0; tt < kTerms; ++tt) {
                        const uint32_t sb = e2m1_scale_byte(warp_max_abs(fabsf(v)));
                        const float scale = __uint_as_float(sb << 23), inv = __uint_as_float((254u - sb) << 23);
                        float back, unused;
                        const uint32_t code = e2m1_pair(v * inv, 0.f, back, unused) & 0xF;
                        v -= back * scale;
                        const uint32_t hi = __shfl_down_sync(0xffffffffu, code, 1);
                        if ((lane & 1) == 0)
                            p.hq[((size_t)tt * p.rows + row) * (p.I_max / 2) + mrow / 2] = (uint8_t)(code | (hi << 4));
                        if (lane == 0) p.hs[((size_t)tt * p.rows + row) * (p.I_max / 32) + mrow / 32] = (uint8_t)sb;
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&acc_empty[buf]));
            if (gu && q.h_ready) {   // this warp's share of the tile's h terms is stored
                __threadfence();
                __syncwarp();
                if (lane == 0) ptx::red_release_add(q.h_ready + ti.g, 1);
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// The four E2M1 terms of one 32-element block of one expert-grouped x row.
__device__ __forceinline__ void quant_x4_block(const __nv_bfloat16 *__restrict__ x, int H,
                                               const int32_t *__restrict__ src_token, int rows,
                                               uint8_t *__restrict__ xq, uint8_t *__restrict__ xs, int row, int b) {
    const int nb = H / 32;
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
    for (int tt = 0; tt < kTerms; ++tt) {
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(v[e]));
        const uint32_t sb = e2m1_scale_byte(amax);
        const float scale = __uint_as_float(sb << 23), inv = __uint_as_float((254u - sb) << 23);
        uint32_t packed[4] = {0, 0, 0, 0};
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
            float blo, bhi;
            const uint32_t byte = e2m1_pair(v[e] * inv, v[e + 1] * inv, blo, bhi);
            v[e] -= blo * scale;
            v[e + 1] -= bhi * scale;
            packed[e / 8] |= byte << (8 * ((e / 2) % 4));
        }
        *reinterpret_cast<uint4 *>(xq + ((size_t)tt * rows + row) * (H / 2) + b * 16) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
        xs[((size_t)tt * rows + row) * nb + b] = (uint8_t)sb;
    }
}

// Expert-grouped x rows -> four E2M1 terms (packed, two codes per byte) with UE8M0 scales per 32
// elements. One thread per (row, 32-element block), grid-stride over a grid that is resident at
// once: the gate/up GEMM launched after it (programmatically) takes SMs as soon as every block of
// this kernel has started, so blocks still queued behind a larger grid would be left to fewer and
// fewer SMs (measured: 1.1 ms lost on the 4096-token layer).
__global__ void __launch_bounds__(256)
quant_x4_rows(const __nv_bfloat16 *__restrict__ x, int H, const int32_t *__restrict__ src_token, int rows,
              uint8_t *__restrict__ xq, uint8_t *__restrict__ xs, int32_t *__restrict__ h_ready, int n_groups) {
    // signals the next kernel (the gate/up GEMM) only after the wait: that kernel reads the
    // permutation's tile records before its own wait
    pdl_wait();
    pdl_trigger();
    // the per-group h counters start at zero for this forward's gate/up epilogues (which wait
    // for this kernel to complete before they store anything)
    if (h_ready)
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_groups; i += gridDim.x * blockDim.x) h_ready[i] = 0;
    const int nb = H / 32;
    const long n = (long)rows * nb;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x)
        quant_x4_block(x, H, src_token, rows, xq, xs, (int)(i / nb), (int)(i % nb));
}

// Many tokens (T >= 64): the same terms, made once per token and stored to each of its grouped
// rows: rows inv_row[t][j] (j < top_k) and, with the shared expert, its row T * top_k + t (the
// permutation places the shared rows after the routed ones, in token order). Thread i quantises
// 32-element block b of token t and writes all its copies: top_k + 1 times less arithmetic than
// one quantisation per grouped row (0.24 -> 0.11 ms on the 4096-token layer; for a few tokens the
// per-row kernel above is 1-2 us faster, its threads' chains being shorter). Every grouped row gets
// the same bytes either way. A resident grid too.
__global__ void __launch_bounds__(256)
quant_x4_tokens(const __nv_bfloat16 *__restrict__ x, int H, int T, int top_k, const int32_t *__restrict__ inv_row,
                int with_shared, int rows, uint8_t *__restrict__ xq, uint8_t *__restrict__ xs,
                int32_t *__restrict__ h_ready, int n_groups) {
    // signals the next kernel (the gate/up GEMM) only after the wait: that kernel reads the
    // permutation's tile records before its own wait
    pdl_wait();
    pdl_trigger();
    if (h_ready)   // as in quant_x4_rows
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_groups; i += gridDim.x * blockDim.x) h_ready[i] = 0;
    const int nb = H / 32, copies = top_k + with_shared;
    const long n = (long)T * nb;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        const int t = (int)(i / nb), b = (int)(i % nb);
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * H + b * 32);
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
        for (int tt = 0; tt < kTerms; ++tt) {
            float amax = 0.f;
#pragma unroll
            for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(v[e]));
            const uint32_t sb = e2m1_scale_byte(amax);
            const float scale = __uint_as_float(sb << 23), inv = __uint_as_float((254u - sb) << 23);
            uint32_t packed[4] = {0, 0, 0, 0};
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                float blo, bhi;
                const uint32_t byte = e2m1_pair(v[e] * inv, v[e + 1] * inv, blo, bhi);
                v[e] -= blo * scale;
                v[e + 1] -= bhi * scale;
                packed[e / 8] |= byte << (8 * ((e / 2) % 4));
            }
            const uint4 codes = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            for (int j = 0; j < copies; ++j) {
                const int r = j < top_k ? __ldg(inv_row + (size_t)t * top_k + j) : T * top_k + t;
                *reinterpret_cast<uint4 *>(xq + ((size_t)tt * rows + r) * (H / 2) + b * 16) = codes;
                xs[((size_t)tt * rows + r) * nb + b] = (uint8_t)sb;
            }
        }
    }
}

// h rows (fp32, [rows][I_max], from a gate/up launch with 32-token or big tiles) -> four E2M1
// terms with UE8M0 scales per 32 elements, the values the fused epilogue makes for the other
// launches (the same scale bytes and codes from the same fp32 h). One thread per (row, 32-element
// block) of a resident grid; routed rows hold I values, the shared expert's rows (from off[E]
// on) I_s, and blocks past a row's width are never read. Moving this work out of the gate/up
// epilogue measured 28 % off that launch with big tiles (the epilogue warps had become its
// bound) and 10 % with 32-token tiles.
__global__ void __launch_bounds__(256)
quant_h_rows(const float *__restrict__ hf, const int32_t *__restrict__ off_shared, int I, int I_s, int I_max,
             int rows, uint8_t *__restrict__ hq, uint8_t *__restrict__ hs) {
    // signals the down GEMM only after the wait: it reads tile records before its own wait
    pdl_wait();
    pdl_trigger();
    const int nb = I_max / 32, shared0 = *off_shared;
    const long n = (long)rows * nb;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        const int row = (int)(i / nb), b = (int)(i % nb);
        if (b * 32 >= (row >= shared0 ? I_s : I)) continue;
        const float4 *src = reinterpret_cast<const float4 *>(hf + (size_t)row * I_max + b * 32);
        float v[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 f = src[q];
            v[4 * q] = f.x;
            v[4 * q + 1] = f.y;
            v[4 * q + 2] = f.z;
            v[4 * q + 3] = f.w;
        }
#pragma unroll
        for (int tt = 0; tt < kTerms; ++tt) {
            float amax = 0.f;
#pragma unroll
            for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(v[e]));
            const uint32_t sb = e2m1_scale_byte(amax);
            const float scale = __uint_as_float(sb << 23), inv = __uint_as_float((254u - sb) << 23);
            uint32_t packed[4] = {0, 0, 0, 0};
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                float blo, bhi;
                const uint32_t byte = e2m1_pair(v[e] * inv, v[e + 1] * inv, blo, bhi);
                v[e] -= blo * scale;
                v[e + 1] -= bhi * scale;
                packed[e / 8] |= byte << (8 * ((e / 2) % 4));
            }
            *reinterpret_cast<uint4 *>(hq + ((size_t)tt * rows + row) * (I_max / 2) + b * 16) =
                make_uint4(packed[0], packed[1], packed[2], packed[3]);
            hs[((size_t)tt * rows + row) * nb + b] = (uint8_t)sb;
        }
    }
}

// NVFP4 activation terms: rows -> four E2M1 terms, each with an E4M3 scale per 16 elements under
// a power-of-two scale per (term, row): G = 2^ceil(log2(max|v| / (6 * 448))) keeps every group's
// scale max|v_group| / (6 G), rounded up to an E4M3 value, within E4M3's range, and |v| / (scale
// G) <= 6 within E2M1's. The next term takes the exact residual. x rows are gathered through
// src_token (K = H); h rows come from the gate/up launch in fp32, K = I for routed rows and I_s
// for the shared expert's rows (from off[E] on). One block of 128 threads per row; a thread owns
// whole groups, up to four (K <= 8192).
template <bool FROM_X>
__device__ __forceinline__ void quant_row_nv(const __nv_bfloat16 *__restrict__ x, const float *__restrict__ hf,
                                             const int32_t *__restrict__ src_token, const int32_t *__restrict__ off_shared,
                                             int K_routed, int K_shared, int ld_in, int rows, int ld_out,
                                             uint8_t *__restrict__ q, uint8_t *__restrict__ qs, float *__restrict__ gs,
                                             int row) {
    const int tid = threadIdx.x;
    const int K = FROM_X ? K_routed : (row >= *off_shared ? K_shared : K_routed);
    const int ng = K / 16;
    float v[4][16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int g = tid + 128 * i;
#pragma unroll
        for (int e = 0; e < 16; e += 8) {
            if (g < ng) {
                if constexpr (FROM_X) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(x + (size_t)src_token[row] * ld_in + g * 16 + e);
                    const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float2 f = __bfloat1622float2(h2[j]);
                        v[i][e + 2 * j] = f.x;
                        v[i][e + 2 * j + 1] = f.y;
                    }
                } else {
                    const float4 a = *reinterpret_cast<const float4 *>(hf + (size_t)row * ld_in + g * 16 + e);
                    const float4 b = *reinterpret_cast<const float4 *>(hf + (size_t)row * ld_in + g * 16 + e + 4);
                    v[i][e] = a.x; v[i][e + 1] = a.y; v[i][e + 2] = a.z; v[i][e + 3] = a.w;
                    v[i][e + 4] = b.x; v[i][e + 5] = b.y; v[i][e + 6] = b.z; v[i][e + 7] = b.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) v[i][e + j] = 0.f;
            }
        }
    }
    __shared__ float red[4];
    for (int t = 0; t < kTerms; ++t) {
        float am[4], tm = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            am[i] = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) am[i] = fmaxf(am[i], fabsf(v[i][e]));
            tm = fmaxf(tm, am[i]);
        }
        tm = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(tm)));
        if ((tid & 31) == 0) red[tid >> 5] = tm;
        __syncthreads();
        const float M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
        __syncthreads();
        // G = 2^ceil(log2(M / 2688)) as an fp32 bit pattern (M = 0: G = 1)
        float G = 1.f;
        if (M > 0.f) {
            const float r = M * (1.0f / 2688.0f);
            uint32_t eb = (__float_as_uint(r) >> 23) & 0xFF;
            if ((__float_as_uint(r) & 0x7FFFFF) != 0 || eb == 0) ++eb;   // round the power up
            G = __uint_as_float(min(max(eb, 1u), 254u) << 23);
        }
        if (tid == 0) gs[(size_t)t * rows + row] = G;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int g = tid + 128 * i;
            if (g >= ng) continue;
            // the group's E4M3 scale: am / (6 G) rounded up to an E4M3 value (0 for an empty group)
            const float ratio = am[i] / (6.0f * G);
            uint16_t sb2;
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(sb2) : "f"(0.f), "f"(ratio));
            uint32_t sb = sb2 & 0xFF, back;
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(back) : "h"((uint16_t)sb));
            if (__half2float(__ushort_as_half((uint16_t)(back & 0xFFFF))) < ratio) {   // next code up
                ++sb;
                asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(back) : "h"((uint16_t)sb));
            }
            const float scale = __half2float(__ushort_as_half((uint16_t)(back & 0xFFFF))) * G;
            qs[((size_t)t * rows + row) * (ld_out / 16) + g] = (uint8_t)sb;
            // codes of v / scale (by the rounded reciprocal: a quotient a hair above 6 saturates,
            // and the next term takes whatever this one leaves)
            const float inv = scale > 0.f ? __frcp_rn(scale) : 0.f;
            uint32_t packed[2] = {0, 0};
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
                float b0 = 0.f, b1 = 0.f;
                const uint32_t code = e2m1_pair(v[i][e] * inv, v[i][e + 1] * inv, b0, b1);
                v[i][e] -= b0 * scale;
                v[i][e + 1] -= b1 * scale;
                packed[e >> 3] |= code << (4 * (e & 7));
            }
            *reinterpret_cast<uint2 *>(q + ((size_t)t * rows + row) * (ld_out / 2) + g * 8) =
                make_uint2(packed[0], packed[1]);
        }
    }
}

template <bool FROM_X>
__global__ void __launch_bounds__(128)
quant_rows_nv(const __nv_bfloat16 *__restrict__ x, const float *__restrict__ hf, const int32_t *__restrict__ src_token,
              const int32_t *__restrict__ off_shared, int K_routed, int K_shared, int ld_in, int rows, int ld_out,
              uint8_t *__restrict__ q, uint8_t *__restrict__ qs, float *__restrict__ gs) {
    pdl_wait();
    pdl_trigger();
    // grid-stride over rows on a grid resident at once (see quant_x4_tokens)
    for (int row = blockIdx.x; row < rows; row += gridDim.x)
        quant_row_nv<FROM_X>(x, hf, src_token, off_shared, K_routed, K_shared, ld_in, rows, ld_out, q, qs, gs, row);
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

// Rows of packed 4-bit codes (K/2 bytes each), 128-byte x box_rows boxes with the 128-byte swizzle.
bool map_packed(CUtensorMap *m, const void *base, uint64_t K, uint64_t rows, uint32_t box_rows) {
    auto enc = encoder();
    if (!enc || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
    const cuuint64_t dims[2] = {K / 2, rows};
    const cuuint64_t strides[1] = {K / 2};
    const cuuint32_t box[2] = {BK / 2, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scale bytes [rows][K/sdiv] (weights; sdiv elements per scale byte, 32 or 16) in 16-byte x
// 128-row boxes: one chunk per row and stage.
bool map_w_scales(CUtensorMap *m, const void *base, uint64_t K, uint64_t rows, int sdiv) {
    auto enc = encoder();
    if (!enc || (reinterpret_cast<uintptr_t>(base) & 15) || (K / sdiv) % 16) return false;
    const cuuint64_t dims[2] = {K / sdiv, rows};
    const cuuint64_t strides[1] = {K / sdiv};
    const cuuint32_t box[2] = {16, BM};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Activation scale bytes [kTerms][rows][K/sdiv] in boxes of 16 bytes x box_rows x kTerms: one
// chunk per column of a stage's B operand, term by term. Rows past the last read as zero.
bool map_act_scales(CUtensorMap *m, const void *base, uint64_t K, uint64_t rows, uint32_t box_rows, int sdiv) {
    auto enc = encoder();
    if (!enc || (reinterpret_cast<uintptr_t>(base) & 15) || (K / sdiv) % 16) return false;
    const cuuint64_t dims[3] = {K / sdiv, rows, kTerms};
    const cuuint64_t strides[2] = {K / sdiv, rows * (K / sdiv)};
    const cuuint32_t box[3] = {16, box_rows, kTerms};
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool BIG>
bool map_sc(ScMaps<BIG> &m, int sdiv, const void *w_routed, uint64_t K_routed, uint64_t rows_routed,
            const void *w_shared, uint64_t K_shared, uint64_t rows_shared, const void *act, uint64_t K_act,
            uint64_t rows_act) {
    if (!map_w_scales(&m.w_routed, w_routed, K_routed, rows_routed, sdiv)) return false;
    if (w_shared) {
        if (!map_w_scales(&m.w_shared, w_shared, K_shared, rows_shared, sdiv)) return false;
    } else {
        m.w_shared = m.w_routed;
    }
    for (int h = 0; h < (BIG ? 3 : 2); ++h)
        if (!map_act_scales(&m.act[h], act, K_act, rows_act, 16u * (h + 1), sdiv)) return false;
    return true;
}

template <bool BIG>
bool map_terms(BMaps4<BIG> &b, const uint8_t *base, uint64_t K, uint64_t rows) {
    for (int t = 0; t < kTerms; ++t)
        for (int h = 0; h < (BIG ? 3 : 2); ++h)
            if (!map_packed(&b.m[t][h], base + (size_t)t * rows * (K / 2), K, rows, 16u * (h + 1))) return false;
    return true;
}

}  // namespace

bool tensor_map_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t rows,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
    auto enc = encoder();
    if (!enc || (reinterpret_cast<uintptr_t>(base) & 15) || (row_bytes & 15)) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool mx4_available() { return encoder() != nullptr; }

bool mx4_supported(const FfnArgs &a) { return encoder() != nullptr && a.H % 128 == 0; }

namespace {
// Big tiles pay when experts average 48 rows or more; the down launch's row blocks of 256 need H a
// multiple of 256.
bool big_tiles(int T, int top_k, int E, int H) { return (long)T * top_k >= (long)kBnBig * E && H % (2 * BM) == 0; }
}  // namespace

int mx4_ntile(int T, int top_k, int E, int H) { return big_tiles(T, top_k, E, H) ? kBnBig / 2 : kNtileMx4; }

int launch_quant_x4(const FfnArgs &a, int num_sms, cudaStream_t st) {
    if (a.T < kSmallRouteTokens) {
        const long threads = (long)a.rows * (a.H / 32);
        const long blocks = std::min<long>((threads + 255) / 256, 4L * num_sms);   // 4 blocks of 256 fit an SM
        launch_pdl(quant_x4_rows, dim3((unsigned)blocks), dim3(256), 0, st, a.x, a.H, a.src_token, a.rows, a.xq,
                   a.xqs, a.h_ready, a.E + 1);
    } else {
        const long threads = (long)a.T * (a.H / 32);
        const long blocks = std::min<long>((threads + 255) / 256, 4L * num_sms);
        launch_pdl(quant_x4_tokens, dim3((unsigned)blocks), dim3(256), 0, st, a.x, a.H, a.T, a.top_k,
                   (const int32_t *)a.inv_row, a.rows > a.T * a.top_k ? 1 : 0, a.rows, a.xq, a.xqs, a.h_ready, a.E + 1);
    }
    return cudaPeekAtLastError() == cudaSuccess ? 1 : -1;
}

namespace {

template <bool NV, bool BIG>
int launch_ffn_impl(const FfnArgs &a, int num_sms, void *sched, cudaEvent_t mid, cudaStream_t st) {
    const NtileLayout nl = a.tiles ? *a.tiles : ntile_layout(sched, a.E, a.rows);
    const uint64_t slots = a.w_slots ? a.w_slots : a.E;   // weight sets the routed arrays hold
    const dim3 grid(a.grid ? a.grid : num_sms);
    constexpr size_t smem = smem_bytes<BIG>();
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(gemm_mx4<kGateUp, NV, BIG, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess ||
            cudaFuncSetAttribute(gemm_mx4<kDown, NV, BIG, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return -1;
        if (cudaFuncSetAttribute(gemm_mx4<kGateUp, NV, BIG, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem_bytes_sft<BIG>()) != cudaSuccess ||
            cudaFuncSetAttribute(gemm_mx4<kDown, NV, BIG, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem_bytes_sft<BIG>()) != cudaSuccess)
            return -1;
        attr = true;
    }
    Mx4Params p{};
    p.E = a.E;
    p.H = a.H;
    p.I = a.I;
    p.I_s = a.I_s;
    p.I_max = a.I_max;
    p.rows = a.rows;
    p.wait_ns = a.wait_ns ? a.wait_ns : ptx::kWaitLimitNs;
    p.hq = a.hq;
    p.hs = a.hqs;
    p.y = a.y;
    p.err = a.err;
    NvParams q{};
    // gate/up with 32-token or big tiles writes fp32 h, and quant_h_rows makes its terms (not in
    // an expert bank's rounds, each of which computes only its own rows)
    const bool gu32 = BIG || (long)a.T * a.top_k >= 16L * a.E;
    const bool split_h = !NV && gu32 && !a.tiles;
    q.hf = NV || split_h ? a.hf : nullptr;
    q.grp_rows = a.cnt;
    CUtensorMap tar, tas;
    BMaps4<BIG> tb;
    // gate/up
    // Many tokens per expert: gate/up tiles of 32 tokens (N = 128 per matrix, half the MMAs per
    // token) with one accumulator buffer (gate + up fill 256 TMEM columns); more still: big tiles
    // of 48 tokens for both launches (the permutation then lays out 48-row tiles as its large ones).
    p.mode = kGateUp;
    p.bn = BIG ? kBnBig : gu32 ? kBnDown : kBnGateUp;
    p.nbuf = gu32 ? 1 : 2;
    p.ntile_rec = gu32 ? nl.rec_large : nl.rec_small;
    p.ntile_count = gu32 ? nl.count + 1 : nl.count;
    p.m_tiles = (a.I_max + BM - 1) / BM;
    p.w_scales_routed = a.routed.gu_scales;
    p.w_scales_shared = a.shared.gu_scales;
    q.w_global_routed = a.routed.gu_global;
    q.w_global_shared = a.shared.gu_global;
    p.act_scales = a.xqs;
    q.act_global = a.xg;
    p.act_ld = a.H;
    bool ok = map_packed(&tar, a.routed.gu_codes, a.H, slots * 2 * a.I, BM) &&
              map_terms(tb, a.xq, a.H, a.rows);
    if (a.shared.gu_codes) ok = ok && map_packed(&tas, a.shared.gu_codes, a.H, 2 * (uint64_t)a.I_s, BM);
    else tas = tar;
    if (!ok) return -2;
    // Scales by TMA whenever every scale row is a whole number of 16-byte chunks (H, I, I_s and
    // I_max multiples of 512 for MXFP4, of 256 for NVFP4), else loaded by the scale warps
    // themselves; and for the 32-token gate/up tiles the warps' own loads too, which measured
    // faster there (512 tokens: 440 against 463 us), while TMA-fed scales were faster for every
    // other tile shape.
    ScMaps<BIG> sc{};
    const int sdiv = NV ? 16 : 32, kq = 16 * sdiv;
    const bool sft = a.H % kq == 0 && a.I % kq == 0 && a.I_max % kq == 0 && (!a.shared.gu_codes || a.I_s % kq == 0);
    const bool sft_gu = sft && (BIG || !gu32);
    // A few tokens per expert (16-token gate/up tiles storing the h terms themselves, scale bytes
    // by TMA): the down launch starts on each group once its gate/up tiles are done. Measured
    // against waiting for the whole gate/up launch, on one box: 4, 8 and 16 tokens 2-3 % faster,
    // 2 and 64 tokens 5 % and 1 % slower. With a static tile assignment the blocks that start early
    // take their first tiles and then wait on groups still in the gate/up launch, while drawing
    // HBM bandwidth from its last wave; the blocks that start late keep their full share.
    q.h_ready = !NV && !BIG && !gu32 && !a.tiles && sft && a.T >= 4 && a.T < kSmallRouteTokens ? a.h_ready : nullptr;
    if (sft_gu && !map_sc(sc, sdiv, a.routed.gu_scales, a.H, slots * 2 * a.I,
                          a.shared.gu_codes ? a.shared.gu_scales : nullptr, a.H, 2 * (uint64_t)a.I_s, a.xqs, a.H,
                          a.rows))
        return -2;
    if (sft_gu)
        launch_k(a.pdl_gate_up, gemm_mx4<kGateUp, NV, BIG, true>, grid, dim3(kThreads), smem_bytes_sft<BIG>(), st, tar,
                 tas, tb, p, q, sc);
    else
        launch_k(a.pdl_gate_up, gemm_mx4<kGateUp, NV, BIG, false>, grid, dim3(kThreads), smem, st, tar, tas, tb, p, q,
                 sc);
    int n = 1;
    if (mid) cudaEventRecord(mid, st);
    if (split_h) {
        const long items = (long)a.rows * (a.I_max / 32);
        const long blocks = std::max(1L, std::min((items + 255) / 256, 4L * num_sms));   // a resident grid
        launch_pdl(quant_h_rows, dim3((unsigned)blocks), dim3(256), 0, st, (const float *)a.hf, a.off + a.E, a.I, a.I_s,
                   a.I_max, a.rows, a.hq, a.hqs);
        ++n;
    }
    if constexpr (NV) {   // h (fp32) -> four terms with E4M3 scales per 16 under a scale per (term, row)
        launch_pdl(quant_rows_nv<false>, dim3((unsigned)std::min(a.rows, 4 * num_sms)), dim3(128), 0, st,
                   (const __nv_bfloat16 *)nullptr,
                   (const float *)a.hf, (const int32_t *)nullptr, a.off + a.E, a.I, a.I_s, a.I_max, a.rows, a.I_max,
                   a.hq, a.hqs, a.hg);
        ++n;
    }
    // down
    p.mode = kDown;
    p.bn = BIG ? kBnBig : kBnDown;
    p.nbuf = BIG ? 1 : 2;
    p.ntile_rec = nl.rec_large;
    p.ntile_count = nl.count + 1;
    p.m_tiles = BIG ? a.H / (2 * BM) : a.H / BM;
    p.w_scales_routed = a.routed.d_scales;
    p.w_scales_shared = a.shared.d_scales;
    q.w_global_routed = a.routed.d_global;
    q.w_global_shared = a.shared.d_global;
    p.act_scales = a.hqs;
    q.act_global = a.hg;
    p.act_ld = a.I_max;
    ok = map_packed(&tar, a.routed.d_codes, a.I, slots * a.H, BM) && map_terms(tb, a.hq, a.I_max, a.rows);
    if (a.shared.d_codes) ok = ok && map_packed(&tas, a.shared.d_codes, a.I_s, (uint64_t)a.H, BM);
    else tas = tar;
    if (!ok) return -2;
    if constexpr (!NV && !BIG) {
        // 32-token down tiles: two 128-row blocks of the down matrix share each tile's terms (the
        // big-tile kernel, its tiles up to 32 rows here), so the terms are read into shared memory
        // half as often per weight byte
        if (gu32 && !a.tiles && a.H % (2 * BM) == 0) {
            static bool attr2 = false;
            if (!attr2) {
                if (cudaFuncSetAttribute(gemm_mx4<kDown, false, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bytes<true>()) != cudaSuccess ||
                    cudaFuncSetAttribute(gemm_mx4<kDown, false, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bytes_sft<true>()) != cudaSuccess)
                    return -1;
                attr2 = true;
            }
            p.nbuf = 1;
            p.m_tiles = a.H / (2 * BM);
            BMaps4<true> tb2;
            ScMaps<true> sc2{};
            if (!map_terms(tb2, a.hq, a.I_max, a.rows)) return -2;
            if (sft) {
                if (!map_sc(sc2, sdiv, a.routed.d_scales, a.I, slots * a.H, a.shared.d_codes ? a.shared.d_scales : nullptr,
                            a.I_s, (uint64_t)a.H, a.hqs, a.I_max, a.rows))
                    return -2;
                launch_pdl(gemm_mx4<kDown, false, true, true>, grid, dim3(kThreads), smem_bytes_sft<true>(), st, tar, tas,
                           tb2, p, q, sc2);
            } else {
                launch_pdl(gemm_mx4<kDown, false, true, false>, grid, dim3(kThreads), smem_bytes<true>(), st, tar, tas,
                           tb2, p, q, sc2);
            }
            ++n;
            return cudaPeekAtLastError() == cudaSuccess ? n : -1;
        }
    }
    if (sft) {
        if (!map_sc(sc, sdiv, a.routed.d_scales, a.I, slots * a.H, a.shared.d_codes ? a.shared.d_scales : nullptr,
                    a.I_s, (uint64_t)a.H, a.hqs, a.I_max, a.rows))
            return -2;
        launch_pdl(gemm_mx4<kDown, NV, BIG, true>, grid, dim3(kThreads), smem_bytes_sft<BIG>(), st, tar, tas, tb, p, q,
                   sc);
    } else {
        launch_pdl(gemm_mx4<kDown, NV, BIG, false>, grid, dim3(kThreads), smem, st, tar, tas, tb, p, q, sc);
    }
    ++n;
    return cudaPeekAtLastError() == cudaSuccess ? n : -1;
}

}  // namespace

int launch_ffn_mx4(const FfnArgs &a, int num_sms, void *sched, cudaEvent_t mid, cudaStream_t st) {
    if (!mx4_supported(a)) return -2;
    // An expert bank's rounds bring their own 16/32-row records, so banked forwards stay small.
    if (!a.tiles && big_tiles(a.T, a.top_k, a.E, a.H)) return launch_ffn_impl<false, true>(a, num_sms, sched, mid, st);
    return launch_ffn_impl<false, false>(a, num_sms, sched, mid, st);
}

bool nv4_supported(const FfnArgs &a) {
    return mx4_supported(a) && a.H <= 8192 && a.I_max <= 8192 && a.routed.gu_global && a.routed.d_global;
}

int launch_quant_x_nv(const FfnArgs &a, int num_sms, cudaStream_t st) {
    launch_pdl(quant_rows_nv<true>, dim3((unsigned)std::min(a.rows, 4 * num_sms)), dim3(128), 0, st, a.x,
               (const float *)nullptr,
               a.src_token, a.off + a.E, a.H, a.H, a.H, a.rows, a.H, a.xq, a.xqs, a.xg);
    return cudaPeekAtLastError() == cudaSuccess ? 1 : -1;
}

int launch_ffn_nv4(const FfnArgs &a, int num_sms, void *sched, cudaEvent_t mid, cudaStream_t st) {
    if (!nv4_supported(a)) return -2;
    return launch_ffn_impl<true, false>(a, num_sms, sched, mid, st);
}

}  // namespace colimoe
