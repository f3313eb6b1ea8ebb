/*
 * colimoe.h -- C ABI of the GB300 routed MXFP4 mixture-of-experts layer (libcolimoe.so).
 *
 * One routed MoE layer of a DeepSeek-V4-style decoder on one NVIDIA GB300 (sm_103a):
 *   A1 router   fp32 logits x.Wr^T, s = sigmoid(logit), key = fp32(s + b), top-k keys
 *               (ties -> lower expert index, descending order), w_j = s_j / sum_j s_j in fp32
 *               ("the CUDA tier wired into the DeepSeek V4 engine", What it is: route on device)
 *   A2 permute  per-expert histogram, exclusive scan, stable scatter of (token, slot) pairs
 *               into expert-grouped rows, inverse map (same list: expert-grouped GEMM rows)
 *   A3 gate/up  h = silu(Wg x) * (Wu x) per expert on its rows, MXFP4 weights
 *   A4 down     y = Wd h
 *               ("DeepSeek V4 Flash CPU inference with NVMe expert streaming": FP4 E2M1 experts
 *               with UE8M0 group-32 scales; the dual gate+up matvec; hidden 4096 x moe_inter 2048)
 *   A5 combine  out = y_shared + sum_j w_j y_j, rounded to bf16
 *               ("the CUDA tier wired into the DeepSeek V4 engine": fused routed+shared MoE)
 *
 * Style follows "DeepSeek V4: the CUDA kernels, as a tier rather than an engine": a header that
 * needs only <stdint.h>; the caller calls in and the library never calls out; the device is
 * checked up front. There is no CPU fallback: every failure is an error code.
 *
 * Conventions
 *  - Return codes: COLI_OK (0) or a negative COLI_ERR_*. Nothing throws across the ABI.
 *    After an error, coli_moe_last_error() describes it.
 *  - Pointers marked "device" must point to GB300 device memory (cudaMalloc or equivalent);
 *    "host" pointers to host memory. The caller owns every pointer it passes; the library owns
 *    only the handle and its workspace.
 *  - A handle is bound to one device and one CUDA stream (given at create). coli_moe_forward
 *    enqueues all its work on that stream and returns without synchronising; it allocates
 *    nothing. Forwards on one handle must not overlap on the device (they share the workspace).
 *
 * Weight format (MXFP4, OCP Microscaling v1.0 FP4 E2M1 elements, UE8M0 scale per 32 elements):
 *  - A matrix of R rows and K columns is stored K-major: codes [R][K/2] bytes, element k of a row
 *    in byte k/2, low nibble for even k and high nibble for odd k; scales [R][K/32] bytes, byte
 *    s giving the fp32 whose bit pattern is s << 23 (2^(s-127); s=0 -> +0, s=255 -> +inf, the
 *    edges the pages' MXFP4 decode reproduces).
 *  - Element value = E2M1(code) * UE8M0(scale of its group of 32 along K).
 */
#ifndef COLIMOE_H
#define COLIMOE_H

#include <stdint.h>

#if defined(__GNUC__)
#define COLI_API __attribute__((visibility("default")))
#else
#define COLI_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

enum {
    COLI_OK = 0,
    COLI_ERR_INVALID_ARG = -1,      /* a NULL or out-of-range argument; nothing was enqueued */
    COLI_ERR_UNSUPPORTED_ARCH = -2, /* the current device is not an sm_103 GB300 */
    COLI_ERR_OUT_OF_MEMORY = -3,    /* workspace allocation failed at create */
    COLI_ERR_CUDA = -4,             /* a CUDA runtime/driver call or kernel launch failed */
};

/* FFN path selection for coli_moe_set_ffn_path. */
enum {
    COLI_FFN_AUTO = 0,      /* COLI_FFN_GEMM_MXF4 whenever a tensor-map encoder is available (always on
                               a GB300 with its driver), else COLI_FFN_GEMV */
    COLI_FFN_GEMV = 1,      /* weight-streaming GEMV kernels on the CUDA cores: the small-T comparison
                               path of the crossover measurement */
    COLI_FFN_GEMM_MXF4 = 2, /* block-scaled tcgen05 GEMM with FP4 on both sides (kind::mxf4, 64 K per
                               instruction): E2M1 weights from HBM as stored, activations as four
                               E2M1 terms with UE8M0 scales per 32 elements (about 3e-4 RMS relative
                               error on x and h). Follows the hardware's UE8M0 decoding, which
                               differs from the format above only for scale bytes 0 and 255. */
};

typedef struct coli_moe coli_moe_t;

/* One set of MXFP4 experts (device pointers, caller-owned). With E experts of hidden H and
 * intermediate I:
 *   gate_up_codes  [E][2I][H/2]   rows 0..I-1 are the gate matrix, rows I..2I-1 the up matrix
 *   gate_up_scales [E][2I][H/32]
 *   down_codes     [E][H][I/2]
 *   down_scales    [E][H][I/32]
 * The shared expert uses the same struct with E = 1 and I = shared_inter.
 * Every pointer must be 16-byte aligned. */
typedef struct {
    const uint8_t *gate_up_codes;
    const uint8_t *gate_up_scales;
    const uint8_t *down_codes;
    const uint8_t *down_scales;
} coli_mxfp4_experts;

typedef struct {
    int32_t num_experts;   /* E, 1..1024 */
    int32_t hidden;        /* H, a multiple of 128 */
    int32_t inter;         /* I, a multiple of 128 */
    int32_t shared_inter;  /* I_s, a multiple of 128, or 0 for a layer without shared expert */
    int32_t max_tokens;    /* largest T a forward will be given, >= 1 */
    int32_t max_top_k;     /* largest top_k a forward will be given, 1..min(E, 32) */
} coli_moe_config;

/* Creates a handle on the current CUDA device, bound to `cuda_stream` (a cudaStream_t; NULL =
 * the legacy default stream). Checks that the device is sm_103 and allocates the workspace for
 * (max_tokens, max_top_k). On success *out receives the handle; on failure *out is set to NULL
 * and the error text is available from coli_moe_last_error(NULL). */
COLI_API int coli_moe_create(const coli_moe_config *cfg, void *cuda_stream, coli_moe_t **out);

/* One forward pass of the layer (A1..A5), enqueued on the handle's stream.
 *   x_bf16         device, bf16 [T][H] row-major, 16-byte aligned
 *   T              tokens, 0..max_tokens (0: nothing is enqueued, returns COLI_OK)
 *   router_w       device, fp32 [E][H], 16-byte aligned
 *   router_bias    device, fp32 [E], or NULL for a zero bias
 *   packed_experts the E routed experts (device pointers), I = cfg.inter
 *   shared_expert  the shared expert (E = 1, I = cfg.shared_inter), or NULL for none; must be
 *                  NULL when cfg.shared_inter == 0
 *   top_k          1..cfg.max_top_k
 *   out_bf16       device, bf16 [T][H], 16-byte aligned; may not overlap x_bf16
 * Errors: COLI_ERR_INVALID_ARG for bad arguments (nothing enqueued), COLI_ERR_CUDA when a launch
 * fails. Device-side execution errors surface on the stream as usual in CUDA. */
COLI_API int coli_moe_forward(coli_moe_t *h, const void *x_bf16, int32_t T,
                     const float *router_w, const float *router_bias,
                     const coli_mxfp4_experts *packed_experts,
                     const coli_mxfp4_experts *shared_expert,
                     int32_t top_k, void *out_bf16);

/* The same forward with x and out in HOST memory, synchronising the handle's stream before
 * returning. Page-locked (pinned, device-mapped) buffers are used in place: a kernel reads x
 * across the host link into a per-handle staging buffer and the combine writes out directly.
 * Other host memory is copied to and from the staging buffers. Weights and router arguments are
 * device pointers as above. */
COLI_API int coli_moe_forward_host(coli_moe_t *h, const void *x_bf16_host, int32_t T,
                          const float *router_w, const float *router_bias,
                          const coli_mxfp4_experts *packed_experts,
                          const coli_mxfp4_experts *shared_expert,
                          int32_t top_k, void *out_bf16_host);

/* Releases the handle and its workspace (synchronises its stream first). NULL is a no-op. Every
 * expert bank created on h must be destroyed first: a bank keeps h's stream and shapes. */
COLI_API void coli_moe_destroy(coli_moe_t *h);

/* Text of the last error on this handle (or of the last failed create when h is NULL). The
 * string stays valid until the next call on the same handle. Never returns NULL. */
COLI_API const char *coli_moe_last_error(const coli_moe_t *h);

/* Forces the FFN path (COLI_FFN_AUTO / _GEMV / _GEMM_MXF4). Returns
 * COLI_ERR_INVALID_ARG for an unknown value. All paths compute the same result within rounding. */
COLI_API int coli_moe_set_ffn_path(coli_moe_t *h, int32_t path);

/* Routing of the last forward, copied to HOST buffers (synchronises the stream). Any field may
 * be NULL to skip it. Sizes use that forward's T, k and the handle's E:
 *   scores    fp32  [T][E]   sigmoid scores s
 *   idx       int32 [T][k]   chosen experts, descending key
 *   weights   fp32  [T][k]   renormalised weights
 *   cnt       int32 [E+1]    rows per group; group E is the shared expert (T rows, or 0)
 *   off       int32 [E+2]    exclusive prefix of cnt
 *   src_token int32 [T*k+T]  token of each expert-grouped row (shared rows are 0..T-1)
 *   inv_row   int32 [T][k]   row of (token, slot)                                             */
typedef struct {
    float *scores;
    int32_t *idx;
    float *weights;
    int32_t *cnt;
    int32_t *off;
    int32_t *src_token;
    int32_t *inv_row;
} coli_moe_routing;

COLI_API int coli_moe_debug_routing(coli_moe_t *h, coli_moe_routing *dst);

/* Kernel launches the last forward enqueued (for launch accounting). */
COLI_API int32_t coli_moe_last_launch_count(const coli_moe_t *h);

/* FFN path (COLI_FFN_GEMV / _GEMM_MXF4) the last forward ran; COLI_FFN_AUTO
 * before the first forward, after a forward with T = 0, or for a NULL handle. */
COLI_API int32_t coli_moe_last_ffn_path(const coli_moe_t *h);

/* Device error word. Kernels that wait on barriers bound every wait (about two seconds); a wait
 * that runs out makes the kernel stop, record a code here (1: waiting for a weight stage,
 * 2: waiting for a free stage, 3: waiting for an MMA, 4: waiting for an accumulator) and return,
 * leaving that forward's output incomplete. Banked forwards (coli_moe_forward_banked) also record
 * 21 when a cache forward finds no free slot and 22 when a refill entry names an expert or slot
 * out of range; neither happens for arguments the host accepted, and the entry is skipped rather
 * than copied. The first code recorded is kept. Synchronises the stream, writes the code (0 = no
 * error) to *code and clears it. */
COLI_API int coli_moe_device_error(coli_moe_t *h, int32_t *code);

/* Limit, in nanoseconds, of the bounded barrier waits inside the COLI_FFN_GEMM_MXF4 kernels
 * (0 restores the default of two seconds; negative values are rejected). It exists to exercise
 * the failure path without a fault: with a limit far below a memory latency, a wait runs out,
 * the kernel records its code in the device error word, lets its copies and MMAs in flight
 * finish (with the full limit), frees TMEM and returns. The forward's output is then incomplete,
 * the context stays usable, and later forwards with the default limit are correct. */
COLI_API int coli_moe_set_wait_limit(coli_moe_t *h, int64_t ns);

/* Stage timing. With profiling enabled (enable != 0) every forward records CUDA events on the
 * handle's stream between its stages; coli_moe_stage_times then synchronises the stream and
 * writes the last forward's stage durations in milliseconds to ms[0..COLI_STAGES-1]:
 * router, permute, FFN gate/up, FFN down, combine. Returns COLI_ERR_INVALID_ARG when profiling
 * is off or no forward has run since it was enabled. */
#define COLI_STAGES 5
COLI_API int coli_moe_set_profiling(coli_moe_t *h, int32_t enable);
COLI_API int coli_moe_stage_times(coli_moe_t *h, float *ms);

/* Test hook for the failure path of coli_moe_create, host only (touches no device). Runs create's
 * workspace allocation sequence for cfg with a host allocator that fails at allocation number
 * fail_at (0-based; negative: never), and frees what was allocated the way create does when an
 * allocation fails (or, when none failed, the way destroy does). Writes the number of allocations
 * attempted to *allocations and the number of blocks still allocated afterwards to *still_live
 * (0: nothing leaked). Returns COLI_ERR_OUT_OF_MEMORY when the sequence failed, COLI_OK when it
 * completed, COLI_ERR_INVALID_ARG for a NULL pointer or a config create would reject outright. */
COLI_API int coli_moe_test_alloc_failure(const coli_moe_config *cfg, int32_t fail_at, int32_t *allocations,
                                         int32_t *still_live);

/* Routing with no device allocation. Runs the router of coli_moe_forward (A1: scores, bias-
 * adjusted top-k, renormalised weights) on the given stream and writes idx_out [T][top_k] (int32)
 * and weights_out [T][top_k] (fp32), device pointers owned by the caller, identical to the idx and
 * weights coli_moe_forward computes for the same inputs, whatever max_tokens the forward's handle
 * was created with: both calls choose the router's split of H from T, E, H and the SM count alone,
 * and so add the same partial logits in the same order. The pages have no counterpart to this call.
 *
 * Who it is for: callers that cannot let a library allocate device memory while they route -- code
 * running while a CUDA graph is being captured, runtimes whose own pool owns all device memory,
 * loops where a first-call allocation is not acceptable. It calls no cudaMalloc, cudaFree or other
 * allocating routine. Its scratch (scores and split-K partial logits) is a fixed 5 MiB array inside
 * the library image, present on every device that loads the library until the process exits.
 *
 * Limits and behaviour:
 *  - T * E <= 262144 (for example 1024 tokens with 256 experts); larger sizes are rejected with
 *    COLI_ERR_INVALID_ARG and a message from coli_moe_last_error(NULL). Also 1 <= E <= 1024, H a
 *    positive multiple of 128, 1 <= top_k <= min(E, 32); T = 0 returns COLI_OK at once.
 *  - The first call on a device, with that device current, looks up the array's device address
 *    (cudaGetSymbolAddress) and the device's properties; make that first call before any stream
 *    capture begins. Later calls only enqueue kernels.
 *  - Every call shares the one array: calls whose kernels overlap on the GPU (different streams,
 *    or different host threads on one device) race and may corrupt each other's results. Nothing
 *    in the array needs to start at zero: each call overwrites all the scratch it reads.
 *  - x_bf16 [T][H] bf16, router_w [E][H] fp32 (both 16-byte aligned), router_bias [E] or NULL. */
COLI_API int coli_moe_route_static(const void *x_bf16, int32_t T, int32_t H, const float *router_w,
                                   const float *router_bias, int32_t E, int32_t top_k, int32_t *idx_out,
                                   float *weights_out, void *cuda_stream);

/* ---------------------------------------------------------------------------------------------
 * Expert residency bank. The routed experts' master copy stays in page-locked host memory (or any
 * memory the device can read); a bank of S device slots holds the experts a layer uses most, and
 * each forward refills it route-aware on the device: the plan, the copies over the host link and
 * the GEMMs are stream-ordered device work, and the host never waits for the routing.
 * The pages keep the most used routed experts of each layer resident on the GPU, ranked by usage
 * ("DeepSeek V4 Flash support -- CUDA/VRAM expert tiering", summary item 1), refill that cache in
 * place, and for a batched prefill refill a transient per-layer bank in slot-sized groups, one
 * group's uploads overlapped with the neighbouring group's compute ("the CUDA tier wired into the
 * DeepSeek V4 engine", What it is: engine tier and prefill MoE).
 *
 * Policy, per forward with T tokens and top_k (readings of the pages, which give no more):
 *  - cache forward, when min(T * top_k, E) <= S: touched experts already resident compute in place
 *    (round 0, with the shared expert). Each other touched expert, in increasing expert order, is
 *    copied into the slot that is empty or holds an untouched expert and comes first by (occupied,
 *    usage of its expert, forward that last used the slot, slot index), where usage counts the
 *    forwards that routed to the expert; those compute in round 1, their copies overlapping
 *    round 0.
 *  - transient forward otherwise: with G = S / 2 the touched experts, in increasing order, form
 *    groups of G; group r computes in round r from slots (r mod 2) * G + i (i its place in the
 *    group), and its copies overlap round r - 1. An expert already in its slot is not copied.
 * Results are bit-identical to coli_moe_forward with the same experts resident in device memory
 * (the same FP4 path, COLI_FFN_GEMM_MXF4, computes both).
 */
typedef struct coli_expert_bank coli_expert_bank_t;

/* Creates a bank of `slots` device slots (2 <= slots <= E) for handle h, bound to h's shapes.
 * host_experts: the E routed experts in the coli_mxfp4_experts layout, in page-locked host memory
 * mapped for the device (cudaHostAlloc, or cudaHostRegister with cudaHostRegisterMapped) or in
 * device memory; pointers 16-byte aligned. The caller owns that memory and keeps it alive and
 * unchanged for the bank's life. The bank allocates slots x (one expert's bytes) of device memory,
 * its state and per-round buffers, one copy stream and its events; it starts empty. Synchronises
 * h's stream. Errors: COLI_ERR_INVALID_ARG (bad slots or pointers, host memory not page-locked),
 * COLI_ERR_OUT_OF_MEMORY, COLI_ERR_UNSUPPORTED_ARCH (no FP4 tensor-map path on this device). */
COLI_API int coli_bank_create(coli_moe_t *h, int32_t slots, const coli_mxfp4_experts *host_experts,
                              coli_expert_bank_t **out);
/* Waits for the bank's work and frees it. NULL-safe. Call it before coli_moe_destroy of the
 * bank's handle. */
COLI_API void coli_bank_destroy(coli_expert_bank_t *bank);

/* coli_moe_forward with the routed experts taken from the bank (arguments as there, the shared
 * expert in device memory). Enqueues on h's stream (and the bank's copy stream, joined back into
 * h's stream before the combine) and returns without synchronising; allocates nothing. Works
 * under stream capture. Forwards on one bank must not overlap. */
COLI_API int coli_moe_forward_banked(coli_moe_t *h, coli_expert_bank_t *bank, const void *x_bf16, int32_t T,
                                     const float *router_w, const float *router_bias,
                                     const coli_mxfp4_experts *shared_expert, int32_t top_k, void *out_bf16);

/* Blocks of 1024 threads that copy experts while another round computes (1 .. SMs - 1; default
 * 16); the GEMM of that round runs on the other SMs. */
COLI_API int coli_bank_set_copy_blocks(coli_expert_bank_t *bank, int32_t blocks);

/* Bank state after the forwards enqueued so far (synchronises h's stream). Each output may be
 * NULL: slot_of [E] (slot of a resident expert, -1 if none), expert_in [S] (-1: empty), usage [E]
 * (forwards that routed to the expert), last_use [S] (the forward, counted from 1, that last used
 * the slot), stats [3] = {forwards, touched experts found in their slot, experts copied}. */
COLI_API int coli_bank_state(coli_expert_bank_t *bank, int32_t *slot_of, int32_t *expert_in, uint32_t *usage,
                             int32_t *last_use, int64_t *stats);

/* ---------------------------------------------------------------------------------------------
 * NVFP4 experts (the format variant of the layer; the pages use MXFP4 only). Same layer, with each
 * matrix stored as E2M1 codes (the layout above), one E4M3 scale byte per 16 elements along K
 * (positive values; [rows][K/16]) and one fp32 scale per matrix: element = e2m1(code) *
 * e4m3(scale) * global. The weights go to the tensor cores as stored (tcgen05 kind::mxf4nvf4,
 * scale_vec::4X); the activations are split into four E2M1 terms with E4M3 scales per 16 under a
 * power-of-two scale per term and row. */
typedef struct {
    const uint8_t *gate_up_codes;        /* [E][2I][H/2] */
    const uint8_t *gate_up_scales;       /* [E][2I][H/16] E4M3 */
    const float *gate_up_global;         /* [E] fp32, one per expert's gate/up matrix */
    const uint8_t *down_codes;           /* [E][H][I/2] */
    const uint8_t *down_scales;          /* [E][H][I/16] E4M3 */
    const float *down_global;            /* [E] fp32 */
} coli_nvfp4_experts;                    /* all device pointers; the shared expert: E = 1 */

/* coli_moe_forward with NVFP4 experts (H and I up to 8192). Same conventions and errors. */
COLI_API int coli_moe_forward_nvfp4(coli_moe_t *h, const void *x_bf16, int32_t T, const float *router_w,
                                    const float *router_bias, const coli_nvfp4_experts *packed_experts,
                                    const coli_nvfp4_experts *shared_expert, int32_t top_k, void *out_bf16);

/* ---------------------------------------------------------------------------------------------
 * FP8 dense projection: out[t][n] = bf16(sum_k x[t][k] * e4m3(w[n][k]) * w_scale[n/128][k/128]),
 * the weight format the pages give for the model's dense matrices: FP8 E4M3 with one fp32 scale
 * per 128 x 128 block ("DeepSeek V4 Flash CPU inference with NVMe expert streaming", the review
 * question on config-driven V4 sizes; the five per-layer dense matmuls of "DeepSeek V4 Flash
 * support -- CUDA/VRAM expert tiering", dense-on-GPU tier comment). E4M3 is the OCP 8-bit float
 * (bias 7, subnormals, max 448, S.1111.111 NaN); the output is the exact sum rounded once, up to the
 * activation split (x enters as two E4M3 terms under a per-token power-of-two scale, about 2^-9
 * relative per element) and fp32 accumulation; on the CUDA-core path (below) the products are
 * exact and only the fp32 sums round.
 *
 * A dense handle holds the workspace for up to max_tokens rows of up to max_k features and is
 * bound to one stream. Layout: x bf16 [T][K], w E4M3 codes [N][K] (K-major rows), w_scale fp32
 * [N/128][K/128], out bf16 [T][N]; all device pointers owned by the caller; K and N multiples of 128.
 * coli_dense_forward enqueues one kernel (CUDA-core path) or two (tensor-core path) on the stream,
 * returns without synchronising and allocates nothing; forwards on one handle must not overlap on
 * the device. */
typedef struct coli_dense coli_dense_t;
COLI_API int coli_dense_create(int32_t max_tokens, int32_t max_k, void *cuda_stream, coli_dense_t **out);
COLI_API int coli_dense_forward(coli_dense_t *d, const void *x_bf16, int32_t T, int32_t K, const uint8_t *w_e4m3,
                                const float *w_scale, int32_t N, void *out_bf16);
COLI_API void coli_dense_destroy(coli_dense_t *d);
/* Text of the last error on d (or of the last failed coli_dense_create when d is NULL). */
COLI_API const char *coli_dense_last_error(const coli_dense_t *d);
/* Synchronises d's stream, returns the device error word (0: none; a bounded wait that ran out
 * records its code, as for coli_moe_device_error) and clears it. */
COLI_API int coli_dense_device_error(coli_dense_t *d, int32_t *code);
/* Kernel path of coli_dense_forward. */
enum {
    COLI_DENSE_AUTO = 0,        /* COLI_DENSE_CUDA_CORES where it measured faster: up to 8 tokens for
                                   N x K <= 4 MiB, 4 for <= 7 MiB, 2 for <= 14 MiB; else
                                   COLI_DENSE_TENSOR */
    COLI_DENSE_CUDA_CORES = 1,  /* one kernel: each block copies its weight rows into shared memory and
                                   multiplies them by the tokens in fp32 (exact products); needs
                                   K <= 8192 and ceil(N / SMs) x K bytes within shared memory */
    COLI_DENSE_TENSOR = 2       /* two E4M3 terms of x, then the tcgen05 E4M3 GEMM (kind::f8f6f4) */
};
/* Forces the path (COLI_DENSE_AUTO restores the automatic choice). COLI_ERR_INVALID_ARG for an
 * unknown path; a forward on a forced CUDA-core path whose shape it does not support returns
 * COLI_ERR_INVALID_ARG. */
COLI_API int coli_dense_set_path(coli_dense_t *d, int32_t path);
/* Path the last forward on d ran (COLI_DENSE_AUTO before the first). */
COLI_API int coli_dense_last_path(const coli_dense_t *d);

#ifdef __cplusplus
}
#endif
#endif /* COLIMOE_H */
