// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <utility>

#include "colimoe.h"

namespace colimoe {

// One expert set in the packed MXFP4 layout (see colimoe.h).
// NVFP4 sets (the format variant) use the same codes, E4M3 scales per 16 ([E][rows][K/16]) and
// one fp32 scale per expert and matrix (gu_global, d_global: [E] device arrays, else null).
struct ExpertSet {
    const uint8_t *gu_codes;    // [E][2I][H/2]
    const uint8_t *gu_scales;   // [E][2I][H/32]
    const uint8_t *d_codes;     // [E][H][I/2]
    const uint8_t *d_scales;    // [E][H][I/32]
    const float *gu_global = nullptr, *d_global = nullptr;
};

// Device workspace, sized at create for (max_tokens, max_top_k).
struct Workspace {
    float *scores = nullptr;        // [Tm][E]
    float *logit_part = nullptr;    // [kRouterPartialFloats] split-K partial router logits
    int32_t *idx = nullptr;         // [Tm][km]
    float *w = nullptr;             // [Tm][km]
    int32_t *inv_row = nullptr;     // [Tm][km]
    int32_t *src_token = nullptr;   // [Tm*km + Tm]
    int32_t *cnt = nullptr;         // [E+1]
    int32_t *off = nullptr;         // [E+2]
    int32_t *touched = nullptr;     // [E+1] non-empty groups, ascending
    int32_t *touched_cost = nullptr;  // [E+2] exclusive prefix of per-group work cost
    int32_t *n_touched = nullptr;   // [1]
    __nv_bfloat16 *h = nullptr;     // [Tm*km + Tm][I_max] SwiGLU output rows (GEMV path)
    float *y = nullptr;             // [Tm*km + Tm][H] expert output rows
    // Activation terms of the block-scaled path: four packed E2M1 terms of x ([4][rows][H/2]) and
    // of h ([4][rows][I_max/2]); scales per 32 elements (UE8M0) or per 16 (E4M3, NVFP4 layer),
    // [terms][rows][K/32 or K/16].
    uint8_t *xq = nullptr;          // 2 * rows * H bytes
    uint8_t *xqs = nullptr;         // 4 * rows * H/16
    uint8_t *hq = nullptr;          // 2 * rows * I_max
    uint8_t *hqs = nullptr;         // 4 * rows * I_max/16
    float *xg = nullptr;            // NVFP4 path: [4][rows] power-of-two scale per x term and row
    float *hg = nullptr;            // [4][rows] the same for the h terms
    float *hf = nullptr;            // [rows][I_max] fp32 h between the NVFP4 GEMMs
    __half *xh = nullptr;           // [Tm][H] tokens as scaled fp16, permuted unit layout (GEMV path)
    float *xinv = nullptr;          // [Tm] inverse scales of xh
    __half *hh = nullptr;           // [Tm*km + Tm][I_max] h rows as scaled fp16 (GEMV path)
    float *hinv = nullptr;          // [Tm*km + Tm]
    int *err = nullptr;             // device error word (0 = none), see sm103_ptx.cuh
    __nv_bfloat16 *x_stage = nullptr;    // [Tm][H] forward_host input staging
    __nv_bfloat16 *out_stage = nullptr;  // [Tm][H] forward_host output staging
    void *tile_sched = nullptr;     // n-tile layout of the block-scaled GEMM (NtileLayout)
    size_t tile_sched_bytes = 0;
    int32_t *h_ready = nullptr;     // [E+1] per group: epilogue warps that have stored a gate/up
                                    // tile's h terms (FP4 path, few tokens: the down launch's start)
};

struct NtileLayout;

// Arguments of the expert FFN stage: groups 0..E-1 are the routed experts, group E the
// shared expert. Group g owns rows [off[g], off[g] + cnt[g]) of xp / h / y.
struct FfnArgs {
    ExpertSet routed;
    ExpertSet shared;
    int E, H, I, I_s, I_max;
    int T, top_k;
    int rows;                       // T*k + (shared ? T : 0), known on the host
    const int32_t *cnt;
    const int32_t *off;
    const int32_t *touched;
    const int32_t *n_touched;
    const int32_t *touched_cost;    // [n_touched + 1] exclusive prefix of per-group cost
    const int32_t *src_token;
    const int32_t *inv_row;         // [T][k] grouped row of each (token, slot)
    const __nv_bfloat16 *x;         // [T][H] input tokens
    __half *xh;                     // GEMV path: scaled fp16 tokens and inverse scales
    float *xinv;
    __nv_bfloat16 *h;               // [rows][I_max]
    __half *hh;                     // GEMV path: scaled fp16 h rows and inverse scales
    float *hinv;
    float *y;                       // [rows][H]
    uint8_t *xq, *xqs, *hq, *hqs;   // block-scaled paths: activation terms and scales
    float *xg, *hg, *hf;            // NVFP4 path: per (term, row) scales of x and h, fp32 h
    int *err;
    uint64_t wait_ns;               // FP4 path: limit of the pipeline waits (0 = the default, 2 s)
    // FP4 path over an expert bank (bank.cu): the tile layout of one round, whose records name
    // bank slots instead of experts; the number of slots `routed` holds; the grid (0 = one block
    // per SM); false when the gate/up launch must not overlap the kernel before it.
    const NtileLayout *tiles = nullptr;
    int w_slots = 0;
    int grid = 0;
    bool pdl_gate_up = true;
    int32_t *h_ready = nullptr;     // [E+1] the workspace's per-group h counters (null: not used)
};

// Programmatic dependent launch. Every kernel of the library is launched with programmatic
// stream serialisation (launch_pdl), so its launch and prologue may overlap the kernel before it
// in the stream. Each kernel therefore begins with pdl_begin() (or, for kernels with an on-chip
// prologue, pdl_trigger() first and pdl_wait() before its first global-memory access):
// pdl_trigger lets the next kernel be scheduled once every block of this one has started;
// pdl_wait returns when the kernel before this one has completed and its writes are visible.
// Since every kernel waits, completion of one kernel implies completion of all earlier ones. A
// kernel that signals only after its own wait (the x- and h-term kernels quant_x4_rows,
// quant_x4_tokens, quant_h_rows and quant_rows_nv, and gemm_mx4) starts its dependent only once
// everything before itself has completed; gemm_mx4 relies on that to read the permutation's
// outputs, and issue weight loads, before its wait. One exception: the down launch of a forward
// of 4 to 63 tokens does not wait for the gate/up launch before it; it waits per expert on
// counters that the gate/up epilogues release (gemm_mx4.cu), and writes only y, which the combine
// reads after its own wait.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_begin() {
    pdl_trigger();
    pdl_wait();
}

// `pdl` false: an ordinary launch, which starts only after all earlier work of the stream (and
// the events it waits on) has completed; griddepcontrol.wait then returns at once.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t st, Args &&...args) {
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args &&...args) {
    return launch_k(true, kernel, grid, block, smem, st, std::forward<Args>(args)...);
}

// Records the text coli_moe_last_error(NULL) returns (printf-style).
void set_create_error(const char *fmt, ...);

// A 2-D tensor map (cuTensorMapEncodeTiled, taken from the driver at first use): `rows` rows of
// `inner` elements of type dt, `row_bytes` apart, boxes of box_inner x box_rows. False when the
// driver offers no encoder or rejects the arguments (base and row_bytes must be 16-byte aligned).
bool tensor_map_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t rows,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle);

// Launchers. Each returns the number of kernels it enqueued, or -1 on a launch error
// (the CUDA error is then available from cudaGetLastError()).
// `partial` holds split-K partial logits for larger T: at least kRouterPartialFloats fp32. The
// split count depends only on (T, E, H, num_sms) and keeps splits * T * E within that fixed cap,
// so every caller that passes such a buffer adds the partial logits in the same order and gets
// bit-identical scores. `zero` (may be null): n_zero ints the router's last kernel clears (the
// permute histogram). `err` (may be null): the device error word the tensor-core logits kernel
// records a timed-out wait in. with_topk false: the logits and scores only (route_permute_small
// takes the top-k).
constexpr size_t kRouterPartialFloats = size_t(1) << 20;   // 4 MiB
int launch_router(const __nv_bfloat16 *x, int T, int H, const float *router_w, const float *router_b,
                  int E, int top_k, float *scores, int32_t *idx, float *w, float *partial,
                  int num_sms, int32_t *zero, int n_zero, int *err, cudaStream_t st, bool with_topk = true);
// Small T: the top-k of A1 and all of A2 (launch_permute) in one launch.
// Returns -2 outside T < kSmallRouteTokens, top_k <= 32, E <= 1024.
constexpr int kSmallRouteTokens = 64;
int launch_route_permute_small(const float *router_b, int T, int E, int top_k, bool with_shared, int cost_tokens,
                               int ntile, Workspace &ws, cudaStream_t st);
// `cost_tokens`: rows per unit of work cost in ws.touched_cost (see permute_scan). `ntile`: when
// non-zero, also write the block-scaled GEMM's n-tile layout (NtileLayout, tiles of `ntile` and
// 2 * `ntile` rows) into ws.tile_sched.
int launch_permute(const int32_t *idx, int T, int E, int top_k, bool with_shared, int cost_tokens, int ntile,
                   Workspace &ws, cudaStream_t st);
// Rows per cost unit the GEMV kernels assume.
constexpr int kGemvCostTokens = 4;

// Token tiles of the block-scaled GEMM: gate/up tiles of n rows, down tiles of 2n rows; with many
// rows per expert both launches take 48-row tiles (the records of 2 x 24).
constexpr int kNtileMx4 = 16;   // E2M1 weights x E2M1 activation terms (gemm_mx4.cu)
constexpr int kNtileMin = 16;   // the layout below is sized for tiles of at least this many rows
// The permute scan writes, per tile size, an exclusive prefix of ceil(cnt / size) over the touched
// groups, the owning group of each tile, one record per tile ({first row, group | rows << 16},
// so a kernel decodes a tile with one load) and the number of tiles. A tile size s >= kNtileMin
// gives at most rows / s + E + 1 tiles.
struct NtileLayout {
    int2 *rec_small, *rec_large;
    int32_t *prefix_small, *owner_small, *prefix_large, *owner_large, *count;   // count[0] small, [1] large
};
__host__ __device__ inline size_t ntile_max(int E, int rows) { return (size_t)rows / kNtileMin + (size_t)E + 2; }
__host__ __device__ inline size_t ntile_layout_ints(int E, int rows) {
    return 4 * ntile_max(E, rows) + 2 * ((size_t)E + 2) + 2 * ntile_max(E, rows) + 2;
}
__host__ __device__ inline NtileLayout ntile_layout(void *base, int E, int rows) {
    const size_t nm = ntile_max(E, rows);
    NtileLayout l;
    l.rec_small = static_cast<int2 *>(base);
    l.rec_large = l.rec_small + nm;
    l.prefix_small = reinterpret_cast<int32_t *>(l.rec_large + nm);
    l.owner_small = l.prefix_small + E + 2;
    l.prefix_large = l.owner_small + nm;
    l.owner_large = l.prefix_large + E + 2;
    l.count = l.owner_large + nm;
    return l;
}
// `mid` (may be null): an event recorded between the gate/up and the down kernels.
int launch_ffn_gemv(const FfnArgs &a, int num_sms, cudaEvent_t mid, cudaStream_t st);
int launch_combine(const float *y, const int32_t *inv_row, const float *w, int T, int H, int top_k,
                   bool with_shared, __nv_bfloat16 *out, cudaStream_t st);
// Device copy of `bytes` (a multiple of 16, both pointers 16-byte aligned), e.g. from mapped host memory.
int launch_copy(void *dst, const void *src, size_t bytes, int num_sms, cudaStream_t st);

// Expert residency bank (bank.cu). Device state and per-round buffers of one bank.
struct BankDev {
    int E, S, R;                    // experts, slots, rounds the buffers hold
    size_t nm;                      // n-tiles per round and tile size (ntile_max)
    int32_t *slot_of;               // [E] slot of a resident expert, -1 otherwise
    int32_t *expert_in;             // [S] expert in a slot, -1 when empty
    uint32_t *usage;                // [E] forwards that routed to the expert
    int32_t *last_use;              // [S] the forward that last used the slot
    long long *stats;               // [3] forwards, experts found in place, experts copied
    int2 *copies;                   // [R][S] {expert, slot} refills of each round
    int32_t *ncopy;                 // [R]
    int2 *rec_small, *rec_large;    // [R][nm] n-tile records of each round ({row0, slot | n << 16})
    int32_t *counts;                // [R][2] small and large n-tile counts of each round
};
// Byte sizes of one expert's four arrays (gate/up codes and scales, down codes and scales).
struct ExpertBytes {
    uint64_t seg[4];
};
// The layout of round r's tiles, as the FP4 GEMM reads it.
inline NtileLayout bank_round_layout(const BankDev &b, int r) {
    NtileLayout l{};
    l.rec_small = b.rec_small + (size_t)r * b.nm;
    l.rec_large = b.rec_large + (size_t)r * b.nm;
    l.count = b.counts + 2 * r;
    return l;
}
// Plans one forward over the bank from the permutation's cnt/off (after the permute, same
// stream): cache forward when `cache`, else transient groups of G slots; R rounds are cleared.
int launch_bank_plan(const BankDev &b, const int32_t *cnt, const int32_t *off, bool cache, int G, int R, int ntile,
                     int *err, cudaStream_t st);
// Copies round r's refills from the source experts (device-accessible, e.g. mapped host memory)
// into their slots.
int launch_bank_refill(const BankDev &b, int r, const ExpertSet &src, const ExpertSet &dst, const ExpertBytes &eb,
                       int blocks, int *err, cudaStream_t st);

// FP8 dense projection (gemm_fp8.cu): out [T][N] bf16 = x [T][K] bf16 times the E4M3 weights
// w [N][K] with fp32 scales w_scale [N/128][K/128]; K and N multiples of 128. xq ([2][T][K]) and
// xs ([T]) are workspace for the two E4M3 terms of x and the per-token scales.
struct DenseArgs {
    const __nv_bfloat16 *x;
    int T, K, N;
    const uint8_t *w;
    const float *w_scale;
    uint8_t *xq;
    float *xs;
    __nv_bfloat16 *out;
    float *part;          // split-K partial sums: min(max_tokens, kSplitMaxTokens) x 128 x SMs floats
    int *cnt;             // SMs split-K arrival counters
    int *err;
    uint64_t wait_ns;
};
constexpr int kSplitMaxTokens = 64;   // the FP8 GEMM splits K only up to this many tokens
bool fp8_available();
int launch_dense_fp8(const DenseArgs &a, int num_sms, cudaStream_t st);
// The CUDA-core projection for few tokens (gemv_fp8.cu): one kernel, no workspace. Supported when
// K <= 8192 and one block's weight rows fit in shared memory; launch returns -2 otherwise. The
// automatic choice takes it for up to dense_gemv_max_tokens(K, N) tokens (0 for large matrices).
bool dense_gemv_supported(int T, int K, int N, int num_sms);
int dense_gemv_max_tokens(int K, int N);
int launch_dense_gemv(const DenseArgs &a, int num_sms, cudaStream_t st);

// Block-scaled tcgen05 GEMM path with FP4 on both sides (gemm_mx4.cu): E2M1 weights x four E2M1
// activation terms.
bool mx4_available();
bool mx4_supported(const FfnArgs &a);
// The n-tile size the permutation must lay out for a forward of the MXFP4 layer (see kNtileMx4).
int mx4_ntile(int T, int top_k, int E, int H);
int launch_ffn_mx4(const FfnArgs &a, int num_sms, void *sched, cudaEvent_t mid, cudaStream_t st);
// Expert-grouped activation rows -> four packed E2M1 terms + UE8M0 scales (ws.xq / ws.xqs).
int launch_quant_x4(const FfnArgs &a, int num_sms, cudaStream_t st);
// NVFP4 variant (routed and shared sets carry E4M3 scales per 16 and fp32 globals): the x terms
// (E4M3 scales per 16 under a power-of-two scale per (term, row)); then both GEMMs with the h
// terms between them (`mid`, may be null, is recorded after the gate/up launch). Each returns the
// kernels enqueued, -1 on a launch error; launch_ffn_nv4 -2 when the shapes are unsupported.
bool nv4_supported(const FfnArgs &a);
int launch_quant_x_nv(const FfnArgs &a, int num_sms, cudaStream_t st);
int launch_ffn_nv4(const FfnArgs &a, int num_sms, void *sched, cudaEvent_t mid, cudaStream_t st);

}  // namespace colimoe
