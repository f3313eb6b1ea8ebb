// The C ABI (colimoe.h) and the host orchestration of one forward: argument checks, the
// workspace, and the stream-ordered launch sequence A1 router -> A2 permute -> A3/A4 expert
// FFN -> A5 combine. No host synchronisation and no allocation inside a forward.
#include <stdarg.h>
#include <stdlib.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <type_traits>

#include "colimoe_internal.cuh"

using namespace colimoe;

struct coli_moe {
    coli_moe_config cfg;
    cudaStream_t stream = nullptr;
    int device = 0;
    int num_sms = 0;
    int I_max = 0;
    int ffn_path = COLI_FFN_AUTO;
    Workspace ws;
    // shape of the last forward (for coli_moe_debug_routing)
    int last_T = 0, last_k = 0;
    bool last_shared = false;
    int32_t last_launches = 0;
    int32_t last_path = COLI_FFN_AUTO;
    uint64_t wait_ns = 0;           // coli_moe_set_wait_limit (0 = default)
    bool profiling = false;
    bool stage_valid = false;
    cudaEvent_t ev[COLI_STAGES + 1] = {};
    char err[512] = {0};
};

namespace {

thread_local char g_create_err[512] = "no error";

void set_err(coli_moe_t *h, const char *fmt, ...) {
    char *dst = h ? h->err : g_create_err;
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(dst, 512, fmt, ap);
    va_end(ap);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Workspace memory goes through this interface, so that the failure path of create (every block
// allocated so far freed, nothing leaked) can be exercised without a device: the default is
// cudaMalloc / cudaFree / cudaMemset; coli_moe_test_alloc_failure substitutes a host allocator
// that fails at a chosen allocation.
struct WsAllocator {
    bool (*alloc)(void **p, size_t bytes, void *ctx);
    void (*release)(void *p, void *ctx);
    bool (*zero)(void *p, size_t bytes, void *ctx);
    void *ctx;
};

bool dev_alloc(void **p, size_t bytes, void *) { return cudaMalloc(p, bytes) == cudaSuccess; }
void dev_release(void *p, void *) { cudaFree(p); }
bool dev_zero(void *p, size_t bytes, void *) { return cudaMemset(p, 0, bytes) == cudaSuccess; }
constexpr WsAllocator kDeviceAllocator{dev_alloc, dev_release, dev_zero, nullptr};

void free_ws(Workspace &ws, const WsAllocator &A = kDeviceAllocator) {
    void *ptrs[] = {ws.xq, ws.xqs, ws.hq, ws.hqs, ws.xg, ws.hg, ws.hf, ws.scores, ws.logit_part, ws.idx,  ws.w,  ws.inv_row, ws.src_token, ws.cnt, ws.off, ws.touched, ws.touched_cost,
                    ws.n_touched, ws.h, ws.y, ws.xh, ws.xinv, ws.hh, ws.hinv, ws.err, ws.x_stage,
                    ws.out_stage, ws.tile_sched, ws.h_ready};
    for (void *p : ptrs)
        if (p) A.release(p, A.ctx);
    ws = Workspace();
}

// Allocates the whole workspace for (max_tokens, max_top_k); on any failure frees what it had
// allocated and returns false.
bool alloc_workspace(Workspace &ws, const coli_moe_config &c, int I_max, const WsAllocator &A) {
    auto alloc = [&](auto **p, size_t count) {
        void *q = nullptr;
        if (!A.alloc(&q, count * sizeof(**p) + 256, A.ctx)) return false;
        *p = static_cast<std::remove_reference_t<decltype(*p)>>(q);
        return true;
    };
    const size_t Tm = c.max_tokens, km = c.max_top_k, E = c.num_experts, H = c.hidden;
    const size_t rows = Tm * km + Tm;
    bool ok = alloc(&ws.scores, Tm * E) && alloc(&ws.logit_part, kRouterPartialFloats) && alloc(&ws.idx, Tm * km) &&
              alloc(&ws.w, Tm * km) && alloc(&ws.inv_row, Tm * km) && alloc(&ws.src_token, rows) &&
              alloc(&ws.cnt, E + 1) && alloc(&ws.off, E + 2) && alloc(&ws.touched, E + 1) &&
              alloc(&ws.touched_cost, E + 2) && alloc(&ws.n_touched, 4) && alloc(&ws.h, rows * (size_t)I_max) &&
              alloc(&ws.y, rows * H) && alloc(&ws.xh, Tm * H) && alloc(&ws.xinv, Tm) &&
              alloc(&ws.hh, rows * (size_t)I_max) && alloc(&ws.hinv, rows) && alloc(&ws.err, 4) &&
              alloc(&ws.x_stage, Tm * H) && alloc(&ws.out_stage, Tm * H) && alloc(&ws.xq, 2 * rows * H) &&
              alloc(&ws.xqs, 4 * rows * (H / 16)) && alloc(&ws.hq, 2 * rows * (size_t)I_max) &&
              alloc(&ws.hqs, 4 * rows * (size_t)(I_max / 16)) && alloc(&ws.xg, 4 * rows) && alloc(&ws.hg, 4 * rows) &&
              alloc(&ws.hf, rows * (size_t)I_max) && alloc(&ws.h_ready, E + 1);
    if (ok) ok = A.zero(ws.err, sizeof(int), A.ctx);
    if (ok) {
        ws.tile_sched_bytes = ntile_layout_ints((int)E, (int)rows) * sizeof(int32_t);
        ok = A.alloc(&ws.tile_sched, ws.tile_sched_bytes + 256, A.ctx);
    }
    if (!ok) free_ws(ws, A);
    return ok;
}

bool valid_experts(const coli_mxfp4_experts *e) {
    return e && e->gate_up_codes && e->gate_up_scales && e->down_codes && e->down_scales &&
           aligned16(e->gate_up_codes) && aligned16(e->gate_up_scales) && aligned16(e->down_codes) &&
           aligned16(e->down_scales);
}

ExpertSet to_set(const coli_mxfp4_experts *e) {
    ExpertSet s{};
    if (e) {
        s.gu_codes = e->gate_up_codes;
        s.gu_scales = e->gate_up_scales;
        s.d_codes = e->down_codes;
        s.d_scales = e->down_scales;
    }
    return s;
}

enum FfnKind { kFfnGemv, kFfnMx4 };

// The FFN kernels a forward uses: the FP4 x FP4 block-scaled GEMM whenever it can run (weights go
// to the tensor cores as stored, 64 K per instruction, at every token count); the CUDA-core GEMV
// only when forced, or when no tensor-map encoder is available.
FfnKind pick_ffn(const coli_moe_t *h) {
    switch (h->ffn_path) {
        case COLI_FFN_GEMV: return kFfnGemv;
        case COLI_FFN_GEMM_MXF4: return kFfnMx4;
        default: break;
    }
    return mx4_available() ? kFfnMx4 : kFfnGemv;
}

// Argument checks every forward shares (T > 0 here).
int check_forward(coli_moe_t *h, const void *x_bf16, int32_t T, const float *router_w,
                  const coli_mxfp4_experts *shared, int32_t top_k, const void *out_bf16) {
    const coli_moe_config &c = h->cfg;
    if (T < 0 || T > c.max_tokens) {
        set_err(h, "T=%d outside [0, max_tokens=%d]", T, c.max_tokens);
        return COLI_ERR_INVALID_ARG;
    }
    if (top_k < 1 || top_k > c.max_top_k) {
        set_err(h, "top_k=%d outside [1, max_top_k=%d]", top_k, c.max_top_k);
        return COLI_ERR_INVALID_ARG;
    }
    if (!x_bf16 || !router_w || !out_bf16 || !aligned16(x_bf16) || !aligned16(router_w) || !aligned16(out_bf16)) {
        set_err(h, "x, router_w and out must be non-NULL, 16-byte aligned device pointers");
        return COLI_ERR_INVALID_ARG;
    }
    const size_t bytes = (size_t)T * (size_t)c.hidden * sizeof(uint16_t);
    const uintptr_t xb = reinterpret_cast<uintptr_t>(x_bf16), ob = reinterpret_cast<uintptr_t>(out_bf16);
    if (xb < ob + bytes && ob < xb + bytes) {   // x is const across the ABI: writing out may not touch it
        set_err(h, "out_bf16 may not overlap x_bf16");
        return COLI_ERR_INVALID_ARG;
    }
    if (shared && (c.shared_inter == 0 || !valid_experts(shared))) {
        set_err(h, c.shared_inter == 0 ? "shared_expert given but cfg.shared_inter is 0"
                                       : "shared_expert must hold four non-NULL 16-byte aligned device pointers");
        return COLI_ERR_INVALID_ARG;
    }
    return COLI_OK;
}

// A1 router and A2 permute (with the n-tile layout of tile size `ntile` when non-zero). Returns
// false on a launch error.
bool run_front(coli_moe_t *h, const void *x_bf16, int32_t T, const float *router_w, const float *router_bias,
               int32_t top_k, bool with_shared, int ntile, int &launches) {
    const int E = h->cfg.num_experts, H = h->cfg.hidden;
    Workspace &ws = h->ws;
    cudaStream_t st = h->stream;
    const __nv_bfloat16 *x = static_cast<const __nv_bfloat16 *>(x_bf16);
    int n;
    if (T < kSmallRouteTokens) {
        // logits, then top-k and the whole permutation in one single-block launch
        n = launch_router(x, T, H, router_w, router_bias, E, top_k, ws.scores, ws.idx, ws.w, ws.logit_part,
                          h->num_sms, nullptr, 0, ws.err, st, false);
        if (n < 0) return false;
        launches += n;
        if (h->profiling) cudaEventRecord(h->ev[1], st);
        n = launch_route_permute_small(router_bias, T, E, top_k, with_shared, kGemvCostTokens, ntile, ws, st);
        if (n < 0) return false;
        launches += n;
        return true;
    }
    n = launch_router(x, T, H, router_w, router_bias, E, top_k, ws.scores, ws.idx, ws.w, ws.logit_part,
                      h->num_sms, ws.cnt, E + 1, ws.err, st);
    if (n < 0) return false;
    launches += n;
    if (h->profiling) cudaEventRecord(h->ev[1], st);
    n = launch_permute(ws.idx, T, E, top_k, with_shared, kGemvCostTokens, ntile, ws, st);
    if (n < 0) return false;
    launches += n;
    return true;
}

// The FFN stage's arguments over the handle's workspace.
FfnArgs ffn_args(coli_moe_t *h, const void *x_bf16, int32_t T, int32_t top_k, int rows,
                 const coli_mxfp4_experts *packed, const coli_mxfp4_experts *shared) {
    const coli_moe_config &c = h->cfg;
    Workspace &ws = h->ws;
    FfnArgs a{};
    a.routed = to_set(packed);
    a.shared = to_set(shared);
    a.E = c.num_experts;
    a.H = c.hidden;
    a.I = c.inter;
    a.I_s = c.shared_inter;
    a.I_max = h->I_max;
    a.T = T;
    a.top_k = top_k;
    a.rows = rows;
    a.cnt = ws.cnt;
    a.off = ws.off;
    a.touched = ws.touched;
    a.n_touched = ws.n_touched;
    a.touched_cost = ws.touched_cost;
    a.src_token = ws.src_token;
    a.inv_row = ws.inv_row;
    a.x = static_cast<const __nv_bfloat16 *>(x_bf16);
    a.xh = ws.xh;
    a.xinv = ws.xinv;
    a.h = ws.h;
    a.hh = ws.hh;
    a.hinv = ws.hinv;
    a.y = ws.y;
    a.xq = ws.xq;
    a.xqs = ws.xqs;
    a.hq = ws.hq;
    a.hqs = ws.hqs;
    a.xg = ws.xg;
    a.hg = ws.hg;
    a.hf = ws.hf;
    a.err = ws.err;
    a.wait_ns = h->wait_ns;
    a.h_ready = ws.h_ready;
    return a;
}

int launch_failed(coli_moe_t *h) {
    const cudaError_t e = cudaGetLastError();
    set_err(h, "kernel launch failed: %s", cudaGetErrorString(e));
    return COLI_ERR_CUDA;
}

int forward_impl(coli_moe_t *h, const void *x_bf16, int32_t T, const float *router_w, const float *router_bias,
                 const coli_mxfp4_experts *packed, const coli_mxfp4_experts *shared, int32_t top_k,
                 void *out_bf16) {
    if (T == 0) {
        h->last_launches = 0;
        h->last_path = COLI_FFN_AUTO;
        return COLI_OK;
    }
    int rc = check_forward(h, x_bf16, T, router_w, shared, top_k, out_bf16);
    if (rc != COLI_OK) return rc;
    if (!valid_experts(packed)) {
        set_err(h, "packed_experts must hold four non-NULL 16-byte aligned device pointers");
        return COLI_ERR_INVALID_ARG;
    }
    cudaGetLastError();   // clear a stale error so launch checks below see only our own
    cudaStream_t st = h->stream;
    const int H = h->cfg.hidden;
    const bool with_shared = shared != nullptr;
    Workspace &ws = h->ws;
    int launches = 0, n;
    const FfnKind ffn = pick_ffn(h);
    const int ntile = ffn == kFfnMx4 ? mx4_ntile(T, top_k, h->cfg.num_experts, H) : 0;
    const int rows = T * top_k + (with_shared ? T : 0);
    const bool prof = h->profiling;
    h->stage_valid = false;
    if (prof) cudaEventRecord(h->ev[0], st);
    if (!run_front(h, x_bf16, T, router_w, router_bias, top_k, with_shared, ntile, launches))
        return launch_failed(h);
    {
        FfnArgs a = ffn_args(h, x_bf16, T, top_k, rows, packed, shared);
        // The gate/up GEMM overlaps its launch and prologue with the kernels before it only for
        // small T. For larger T that programmatic launch cost more than it saved: measured with
        // 512 tokens, 0.788 against 0.742 ms per layer, and with 4096 tokens 4.96 against 3.81 ms,
        // every kernel's own time unchanged.
        a.pdl_gate_up = T < kSmallRouteTokens;
        if (ffn == kFfnMx4) {   // the activation terms belong to the permute stage
            n = launch_quant_x4(a, h->num_sms, st);
            if (n < 0) return launch_failed(h);
            launches += n;
        }
        if (prof) cudaEventRecord(h->ev[2], st);
        cudaEvent_t mid = prof ? h->ev[3] : nullptr;
        if (ffn == kFfnMx4) {
            n = launch_ffn_mx4(a, h->num_sms, ws.tile_sched, mid, st);
            if (n == -2) {
                set_err(h, "FP4 block-scaled GEMM path unavailable (needs a tensor-map encoder)");
                return COLI_ERR_INVALID_ARG;
            }
        } else {
            n = launch_ffn_gemv(a, h->num_sms, mid, st);
        }
        if (n < 0) return launch_failed(h);
        launches += n;
    }
    if (prof) cudaEventRecord(h->ev[4], st);
    n = launch_combine(ws.y, ws.inv_row, ws.w, T, H, top_k, with_shared, static_cast<__nv_bfloat16 *>(out_bf16), st);
    if (n < 0) return launch_failed(h);
    launches += n;
    if (prof) {
        cudaEventRecord(h->ev[5], st);
        h->stage_valid = true;
    }
    h->last_T = T;
    h->last_k = top_k;
    h->last_shared = with_shared;
    h->last_launches = launches;
    h->last_path = ffn == kFfnGemv ? COLI_FFN_GEMV : COLI_FFN_GEMM_MXF4;
    return COLI_OK;
}

}  // namespace

void colimoe::set_create_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_create_err, sizeof g_create_err, fmt, ap);
    va_end(ap);
}

extern "C" {

int coli_moe_create(const coli_moe_config *cfg, void *cuda_stream, coli_moe_t **out) {
    if (!out) {
        set_err(nullptr, "out is NULL");
        return COLI_ERR_INVALID_ARG;
    }
    *out = nullptr;
    if (!cfg) {
        set_err(nullptr, "cfg is NULL");
        return COLI_ERR_INVALID_ARG;
    }
    const coli_moe_config c = *cfg;
    if (c.num_experts < 1 || c.num_experts > 1024 || c.hidden < 128 || c.hidden % 128 || c.inter < 128 ||
        c.inter % 128 || c.shared_inter < 0 || c.shared_inter % 128 || c.max_tokens < 1 || c.max_top_k < 1 ||
        c.max_top_k > 32 || c.max_top_k > c.num_experts) {
        set_err(nullptr,
                "invalid config: need 1<=E<=1024, H and I positive multiples of 128, I_s a multiple of 128 "
                "(or 0), max_tokens>=1, 1<=max_top_k<=min(E,32)");
        return COLI_ERR_INVALID_ARG;
    }
    if ((double)c.max_tokens * (c.max_top_k + 1) > 2.0e9 / 4) {
        set_err(nullptr, "max_tokens too large for 32-bit row indexing");
        return COLI_ERR_INVALID_ARG;
    }
    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
        cudaGetLastError();
        set_err(nullptr, "no CUDA device available");
        return COLI_ERR_UNSUPPORTED_ARCH;
    }
    if (prop.major != 10 || prop.minor != 3) {
        set_err(nullptr, "device %d (%s) is sm_%d%d; this library is built for sm_103a (GB300) only", dev, prop.name,
                prop.major, prop.minor);
        return COLI_ERR_UNSUPPORTED_ARCH;
    }
    coli_moe_t *h = new (std::nothrow) coli_moe_t();
    if (!h) {
        set_err(nullptr, "host allocation failed");
        return COLI_ERR_OUT_OF_MEMORY;
    }
    h->cfg = c;
    h->stream = static_cast<cudaStream_t>(cuda_stream);
    h->device = dev;
    h->num_sms = prop.multiProcessorCount;
    h->I_max = c.inter > c.shared_inter ? c.inter : c.shared_inter;
    const bool ok = alloc_workspace(h->ws, c, h->I_max, kDeviceAllocator);
    if (!ok) {
        cudaGetLastError();
        delete h;
        set_err(nullptr, "workspace allocation failed (max_tokens=%d, max_top_k=%d)", c.max_tokens, c.max_top_k);
        return COLI_ERR_OUT_OF_MEMORY;
    }
    *out = h;
    return COLI_OK;
}

int coli_moe_forward(coli_moe_t *h, const void *x_bf16, int32_t T, const float *router_w, const float *router_bias,
                     const coli_mxfp4_experts *packed_experts, const coli_mxfp4_experts *shared_expert,
                     int32_t top_k, void *out_bf16) {
    if (!h) return COLI_ERR_INVALID_ARG;
    return forward_impl(h, x_bf16, T, router_w, router_bias, packed_experts, shared_expert, top_k, out_bf16);
}

int coli_moe_forward_host(coli_moe_t *h, const void *x_bf16_host, int32_t T, const float *router_w,
                          const float *router_bias, const coli_mxfp4_experts *packed_experts,
                          const coli_mxfp4_experts *shared_expert, int32_t top_k, void *out_bf16_host) {
    if (!h) return COLI_ERR_INVALID_ARG;
    if (T == 0) return COLI_OK;
    if (T < 0 || T > h->cfg.max_tokens || !x_bf16_host || !out_bf16_host) {
        set_err(h, "forward_host: need 0<=T<=max_tokens and non-NULL host buffers");
        return COLI_ERR_INVALID_ARG;
    }
    const size_t bytes = (size_t)T * h->cfg.hidden * sizeof(uint16_t);
    // Page-locked host buffers are device-mapped: a kernel pulls x across the host link into the
    // staging buffer (one read of each byte; the forward reads x many times), and the combine
    // writes out in place. Other host memory goes through copies.
    cudaPointerAttributes ax, ao;
    const bool mapped = cudaPointerGetAttributes(&ax, x_bf16_host) == cudaSuccess && ax.type == cudaMemoryTypeHost &&
                        ax.devicePointer && aligned16(ax.devicePointer) &&
                        cudaPointerGetAttributes(&ao, out_bf16_host) == cudaSuccess && ao.type == cudaMemoryTypeHost &&
                        ao.devicePointer && aligned16(ao.devicePointer);
    cudaGetLastError();
    void *out_dev = h->ws.out_stage;
    if (mapped) {
        if (launch_copy(h->ws.x_stage, ax.devicePointer, bytes, h->num_sms, h->stream) < 0) {
            set_err(h, "host-to-device copy kernel failed: %s", cudaGetErrorString(cudaGetLastError()));
            return COLI_ERR_CUDA;
        }
        out_dev = ao.devicePointer;
    } else if (cudaMemcpyAsync(h->ws.x_stage, x_bf16_host, bytes, cudaMemcpyHostToDevice, h->stream) != cudaSuccess) {
        set_err(h, "host-to-device copy failed: %s", cudaGetErrorString(cudaGetLastError()));
        return COLI_ERR_CUDA;
    }
    const int rc = forward_impl(h, h->ws.x_stage, T, router_w, router_bias, packed_experts, shared_expert, top_k,
                                out_dev);
    if (rc != COLI_OK) return rc;
    if (!mapped &&
        cudaMemcpyAsync(out_bf16_host, h->ws.out_stage, bytes, cudaMemcpyDeviceToHost, h->stream) != cudaSuccess) {
        set_err(h, "device-to-host copy failed: %s", cudaGetErrorString(cudaGetLastError()));
        return COLI_ERR_CUDA;
    }
    const cudaError_t e = cudaStreamSynchronize(h->stream);
    if (e != cudaSuccess) {
        set_err(h, "forward failed on the device: %s", cudaGetErrorString(e));
        return COLI_ERR_CUDA;
    }
    return COLI_OK;
}

void coli_moe_destroy(coli_moe_t *h) {
    if (!h) return;
    cudaStreamSynchronize(h->stream);
    for (cudaEvent_t &e : h->ev)
        if (e) cudaEventDestroy(e);
    free_ws(h->ws);
    delete h;
}

const char *coli_moe_last_error(const coli_moe_t *h) { return h ? h->err : g_create_err; }

int coli_moe_set_ffn_path(coli_moe_t *h, int32_t path) {
    if (!h || path < COLI_FFN_AUTO || path > COLI_FFN_GEMM_MXF4) {
        if (h) set_err(h, "unknown FFN path %d", path);
        return COLI_ERR_INVALID_ARG;
    }
    h->ffn_path = path;
    return COLI_OK;
}

int coli_moe_debug_routing(coli_moe_t *h, coli_moe_routing *dst) {
    if (!h || !dst) return COLI_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) {
        set_err(h, "stream error: %s", cudaGetErrorString(cudaGetLastError()));
        return COLI_ERR_CUDA;
    }
    const size_t T = h->last_T, k = h->last_k, E = h->cfg.num_experts;
    const size_t rows = T * k + (h->last_shared ? T : 0);
    struct Copy {
        void *dst;
        const void *src;
        size_t bytes;
    } copies[] = {
        {dst->scores, h->ws.scores, T * E * 4}, {dst->idx, h->ws.idx, T * k * 4},  {dst->weights, h->ws.w, T * k * 4},
        {dst->cnt, h->ws.cnt, (E + 1) * 4},     {dst->off, h->ws.off, (E + 2) * 4}, {dst->src_token, h->ws.src_token, rows * 4},
        {dst->inv_row, h->ws.inv_row, T * k * 4},
    };
    for (const Copy &c : copies) {
        if (!c.dst || c.bytes == 0) continue;
        if (cudaMemcpy(c.dst, c.src, c.bytes, cudaMemcpyDeviceToHost) != cudaSuccess) {
            set_err(h, "copy failed: %s", cudaGetErrorString(cudaGetLastError()));
            return COLI_ERR_CUDA;
        }
    }
    return COLI_OK;
}

int32_t coli_moe_last_launch_count(const coli_moe_t *h) { return h ? h->last_launches : 0; }

int32_t coli_moe_last_ffn_path(const coli_moe_t *h) { return h ? h->last_path : COLI_FFN_AUTO; }

int coli_moe_set_wait_limit(coli_moe_t *h, int64_t ns) {
    if (!h || ns < 0) return COLI_ERR_INVALID_ARG;
    h->wait_ns = (uint64_t)ns;
    return COLI_OK;
}

int coli_moe_device_error(coli_moe_t *h, int32_t *code) {
    if (!h || !code) return COLI_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess ||
        cudaMemcpy(code, h->ws.err, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(h->ws.err, 0, sizeof(int32_t)) != cudaSuccess) {
        set_err(h, "stream error: %s", cudaGetErrorString(cudaGetLastError()));
        return COLI_ERR_CUDA;
    }
    return COLI_OK;
}

int coli_moe_set_profiling(coli_moe_t *h, int32_t enable) {
    if (!h) return COLI_ERR_INVALID_ARG;
    if (enable && !h->ev[0]) {
        for (cudaEvent_t &e : h->ev) {
            if (cudaEventCreate(&e) != cudaSuccess) {
                set_err(h, "cudaEventCreate failed: %s", cudaGetErrorString(cudaGetLastError()));
                return COLI_ERR_CUDA;
            }
        }
    }
    h->profiling = enable != 0;
    h->stage_valid = false;
    return COLI_OK;
}

int coli_moe_stage_times(coli_moe_t *h, float *ms) {
    if (!h || !ms) return COLI_ERR_INVALID_ARG;
    if (!h->profiling || !h->stage_valid) {
        set_err(h, "no profiled forward: enable profiling with coli_moe_set_profiling first");
        return COLI_ERR_INVALID_ARG;
    }
    if (cudaEventSynchronize(h->ev[COLI_STAGES]) != cudaSuccess) {
        set_err(h, "stream error: %s", cudaGetErrorString(cudaGetLastError()));
        return COLI_ERR_CUDA;
    }
    for (int i = 0; i < COLI_STAGES; ++i) {
        if (cudaEventElapsedTime(&ms[i], h->ev[i], h->ev[i + 1]) != cudaSuccess) {
            set_err(h, "cudaEventElapsedTime failed: %s", cudaGetErrorString(cudaGetLastError()));
            return COLI_ERR_CUDA;
        }
    }
    return COLI_OK;
}

namespace {
// Host stand-in for the device allocator: malloc / free, failing at allocation number fail_at.
struct FakeAllocs {
    int fail_at, count = 0, live = 0, peak = 0;
};
bool fake_alloc(void **p, size_t bytes, void *ctx) {
    FakeAllocs &f = *static_cast<FakeAllocs *>(ctx);
    if (f.count++ == f.fail_at) return false;
    *p = malloc(16);   // only the bookkeeping matters: no workspace byte is touched
    if (!*p) return false;
    f.peak = ++f.live > f.peak ? f.live : f.peak;
    return true;
}
void fake_release(void *p, void *ctx) {
    --static_cast<FakeAllocs *>(ctx)->live;
    free(p);
}
bool fake_zero(void *, size_t, void *) { return true; }
}  // namespace

int coli_moe_test_alloc_failure(const coli_moe_config *cfg, int32_t fail_at, int32_t *allocations,
                                int32_t *still_live) {
    if (!cfg || !allocations || !still_live || cfg->num_experts < 1 || cfg->max_tokens < 1 || cfg->max_top_k < 1 ||
        cfg->hidden < 128 || cfg->inter < 128)
        return COLI_ERR_INVALID_ARG;
    FakeAllocs f{fail_at};
    Workspace ws;
    const int I_max = cfg->inter > cfg->shared_inter ? cfg->inter : cfg->shared_inter;
    const bool ok = alloc_workspace(ws, *cfg, I_max, WsAllocator{fake_alloc, fake_release, fake_zero, &f});
    *allocations = f.count;
    if (ok) free_ws(ws, WsAllocator{fake_alloc, fake_release, fake_zero, &f});
    *still_live = f.live;
    return ok ? COLI_OK : COLI_ERR_OUT_OF_MEMORY;
}

}  // extern "C"

// ------------------------------------------------------------------------------------------------
// NVFP4 experts.

namespace {

bool valid_nv(const coli_nvfp4_experts *e) {
    return e && e->gate_up_codes && e->gate_up_scales && e->gate_up_global && e->down_codes && e->down_scales &&
           e->down_global && aligned16(e->gate_up_codes) && aligned16(e->gate_up_scales) &&
           aligned16(e->down_codes) && aligned16(e->down_scales);
}

ExpertSet nv_set(const coli_nvfp4_experts *e) {
    ExpertSet s{};
    if (e) {
        s.gu_codes = e->gate_up_codes;
        s.gu_scales = e->gate_up_scales;
        s.d_codes = e->down_codes;
        s.d_scales = e->down_scales;
        s.gu_global = e->gate_up_global;
        s.d_global = e->down_global;
    }
    return s;
}

}  // namespace

extern "C" int coli_moe_forward_nvfp4(coli_moe_t *h, const void *x_bf16, int32_t T, const float *router_w,
                                      const float *router_bias, const coli_nvfp4_experts *packed,
                                      const coli_nvfp4_experts *shared, int32_t top_k, void *out_bf16) {
    if (!h) return COLI_ERR_INVALID_ARG;
    if (T == 0) {
        h->last_launches = 0;
        return COLI_OK;
    }
    int rc = check_forward(h, x_bf16, T, router_w, nullptr, top_k, out_bf16);
    if (rc != COLI_OK) return rc;
    if (!valid_nv(packed) || (shared && (h->cfg.shared_inter == 0 || !valid_nv(shared)))) {
        set_err(h, "NVFP4 experts need six non-NULL pointers (codes and scales 16-byte aligned), and a shared "
                   "expert only with cfg.shared_inter > 0");
        return COLI_ERR_INVALID_ARG;
    }
    cudaGetLastError();
    const bool with_shared = shared != nullptr;
    const int rows = T * top_k + (with_shared ? T : 0);
    int launches = 0;
    cudaStream_t st = h->stream;
    const bool prof = h->profiling;
    h->stage_valid = false;
    FfnArgs a = ffn_args(h, x_bf16, T, top_k, rows, nullptr, nullptr);
    a.routed = nv_set(packed);
    a.shared = nv_set(shared);
    a.pdl_gate_up = T < kSmallRouteTokens;   // as in coli_moe_forward: a plain launch from 64 tokens on
    if (!nv4_supported(a)) {
        set_err(h, "NVFP4 path unavailable (needs a tensor-map encoder, H and I up to 8192)");
        return COLI_ERR_INVALID_ARG;
    }
    if (prof) cudaEventRecord(h->ev[0], st);
    if (!run_front(h, x_bf16, T, router_w, router_bias, top_k, with_shared, kNtileMx4, launches))
        return launch_failed(h);
    int n = launch_quant_x_nv(a, h->num_sms, st);
    if (n < 0) return launch_failed(h);
    launches += n;
    if (prof) cudaEventRecord(h->ev[2], st);
    n = launch_ffn_nv4(a, h->num_sms, h->ws.tile_sched, prof ? h->ev[3] : nullptr, st);
    if (n < 0) return launch_failed(h);
    launches += n;
    if (prof) cudaEventRecord(h->ev[4], st);
    n = launch_combine(h->ws.y, h->ws.inv_row, h->ws.w, T, h->cfg.hidden, top_k, with_shared,
                       static_cast<__nv_bfloat16 *>(out_bf16), st);
    if (n < 0) return launch_failed(h);
    launches += n;
    if (prof) {
        cudaEventRecord(h->ev[5], st);
        h->stage_valid = true;
    }
    h->last_T = T;
    h->last_k = top_k;
    h->last_shared = with_shared;
    h->last_launches = launches;
    h->last_path = COLI_FFN_GEMM_MXF4;
    return COLI_OK;
}

// ------------------------------------------------------------------------------------------------
// Expert residency bank (kernels and policy in bank.cu).

struct coli_expert_bank {
    coli_moe_t *h = nullptr;
    int S = 0, R = 0, copy_blocks = 16;
    BankDev dev{};
    ExpertSet src{};                 // device-accessible addresses of the master experts
    ExpertSet slots{};               // [S] experts in device memory
    ExpertBytes eb{};
    cudaStream_t copy = nullptr;
    cudaEvent_t ev_plan = nullptr;
    cudaEvent_t *ev_fill = nullptr, *ev_done = nullptr;   // [R] each
    void *mem[12] = {};
};

namespace {

void free_bank(coli_expert_bank_t *b) {
    if (b->copy) cudaStreamSynchronize(b->copy);
    for (void *p : b->mem)
        if (p) cudaFree(p);
    if (b->ev_plan) cudaEventDestroy(b->ev_plan);
    for (int r = 0; r < b->R; ++r) {
        if (b->ev_fill && b->ev_fill[r]) cudaEventDestroy(b->ev_fill[r]);
        if (b->ev_done && b->ev_done[r]) cudaEventDestroy(b->ev_done[r]);
    }
    delete[] b->ev_fill;
    delete[] b->ev_done;
    if (b->copy) cudaStreamDestroy(b->copy);
    delete b;
}

// The device-readable address of caller memory: mapped page-locked host memory or device memory.
const uint8_t *device_view(const void *p) {
    cudaPointerAttributes at;
    if (!p || cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (at.type == cudaMemoryTypeHost) return static_cast<const uint8_t *>(at.devicePointer);
    if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return static_cast<const uint8_t *>(p);
    return nullptr;
}

}  // namespace

extern "C" {

int coli_bank_create(coli_moe_t *h, int32_t slots, const coli_mxfp4_experts *host_experts,
                     coli_expert_bank_t **out) {
    if (!h || !out) return COLI_ERR_INVALID_ARG;
    *out = nullptr;
    const coli_moe_config &c = h->cfg;
    const int E = c.num_experts;
    if (slots < 2 || slots > E) {
        set_err(h, "bank slots=%d outside [2, E=%d]", slots, E);
        return COLI_ERR_INVALID_ARG;
    }
    if (!valid_experts(host_experts)) {
        set_err(h, "host_experts must hold four non-NULL 16-byte aligned pointers");
        return COLI_ERR_INVALID_ARG;
    }
    if (!mx4_available()) {
        set_err(h, "the expert bank runs on the FP4 block-scaled path, which needs a tensor-map encoder");
        return COLI_ERR_UNSUPPORTED_ARCH;
    }
    ExpertSet src;
    src.gu_codes = device_view(host_experts->gate_up_codes);
    src.gu_scales = device_view(host_experts->gate_up_scales);
    src.d_codes = device_view(host_experts->down_codes);
    src.d_scales = device_view(host_experts->down_scales);
    if (!src.gu_codes || !src.gu_scales || !src.d_codes || !src.d_scales || !aligned16(src.gu_codes) ||
        !aligned16(src.gu_scales) || !aligned16(src.d_codes) || !aligned16(src.d_scales)) {
        set_err(h, "host_experts must be page-locked host memory mapped for the device, or device memory");
        return COLI_ERR_INVALID_ARG;
    }
    coli_expert_bank_t *b = new (std::nothrow) coli_expert_bank_t();
    if (!b) return COLI_ERR_OUT_OF_MEMORY;
    b->h = h;
    b->S = slots;
    b->src = src;
    const uint64_t H = c.hidden, I = c.inter;
    b->eb.seg[0] = 2 * I * (H / 2);
    b->eb.seg[1] = 2 * I * (H / 32);
    b->eb.seg[2] = H * (I / 2);
    b->eb.seg[3] = H * (I / 32);
    const long cap = std::min<long>((long)c.max_tokens * c.max_top_k, E);
    const int G = slots / 2;
    b->R = std::max<int>(2, (int)((cap + G - 1) / G));
    const int rows = c.max_tokens * c.max_top_k + c.max_tokens;
    BankDev &d = b->dev;
    d.E = E;
    d.S = slots;
    d.R = b->R;
    d.nm = ntile_max(E, rows);
    bool ok = true;
    auto get = [&](int i, size_t bytes) -> void * {
        if (ok && cudaMalloc(&b->mem[i], bytes + 256) != cudaSuccess) ok = false;
        return ok ? b->mem[i] : nullptr;
    };
    b->slots.gu_codes = static_cast<const uint8_t *>(get(0, slots * b->eb.seg[0]));
    b->slots.gu_scales = static_cast<const uint8_t *>(get(1, slots * b->eb.seg[1]));
    b->slots.d_codes = static_cast<const uint8_t *>(get(2, slots * b->eb.seg[2]));
    b->slots.d_scales = static_cast<const uint8_t *>(get(3, slots * b->eb.seg[3]));
    d.slot_of = static_cast<int32_t *>(get(4, sizeof(int32_t) * E));
    d.expert_in = static_cast<int32_t *>(get(5, sizeof(int32_t) * slots));
    d.usage = static_cast<uint32_t *>(get(6, sizeof(uint32_t) * E));
    d.last_use = static_cast<int32_t *>(get(7, sizeof(int32_t) * slots));
    d.stats = static_cast<long long *>(get(8, sizeof(long long) * 4));
    d.copies = static_cast<int2 *>(get(9, sizeof(int2) * (size_t)b->R * slots));
    d.ncopy = static_cast<int32_t *>(get(10, sizeof(int32_t) * (size_t)b->R + sizeof(int32_t) * 2 * b->R));
    d.counts = d.ncopy ? d.ncopy + b->R : nullptr;
    int2 *recs = static_cast<int2 *>(get(11, sizeof(int2) * 2 * d.nm * (size_t)b->R));
    d.rec_small = recs;
    d.rec_large = recs ? recs + d.nm * (size_t)b->R : nullptr;
    if (ok) {
        cudaStream_t st = h->stream;
        ok = cudaMemsetAsync(d.slot_of, 0xFF, sizeof(int32_t) * E, st) == cudaSuccess &&
             cudaMemsetAsync(d.expert_in, 0xFF, sizeof(int32_t) * slots, st) == cudaSuccess &&
             cudaMemsetAsync(d.usage, 0, sizeof(uint32_t) * E, st) == cudaSuccess &&
             cudaMemsetAsync(d.last_use, 0, sizeof(int32_t) * slots, st) == cudaSuccess &&
             cudaMemsetAsync(d.stats, 0, sizeof(long long) * 4, st) == cudaSuccess &&
             cudaStreamSynchronize(st) == cudaSuccess;
    }
    if (ok) ok = cudaStreamCreateWithFlags(&b->copy, cudaStreamNonBlocking) == cudaSuccess;
    if (ok) {
        b->ev_fill = new (std::nothrow) cudaEvent_t[b->R]();
        b->ev_done = new (std::nothrow) cudaEvent_t[b->R]();
        ok = b->ev_fill && b->ev_done &&
             cudaEventCreateWithFlags(&b->ev_plan, cudaEventDisableTiming) == cudaSuccess;
        for (int r = 0; ok && r < b->R; ++r)
            ok = cudaEventCreateWithFlags(&b->ev_fill[r], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&b->ev_done[r], cudaEventDisableTiming) == cudaSuccess;
    }
    if (!ok) {
        cudaGetLastError();
        free_bank(b);
        set_err(h, "bank allocation failed (%d slots)", slots);
        return COLI_ERR_OUT_OF_MEMORY;
    }
    b->copy_blocks = std::min(16, h->num_sms - 1);
    *out = b;
    return COLI_OK;
}

void coli_bank_destroy(coli_expert_bank_t *bank) {
    if (!bank) return;
    cudaStreamSynchronize(bank->h->stream);
    free_bank(bank);
}

int coli_bank_set_copy_blocks(coli_expert_bank_t *bank, int32_t blocks) {
    if (!bank || blocks < 1 || blocks > bank->h->num_sms - 1) {
        if (bank) set_err(bank->h, "copy blocks %d outside [1, SMs - 1]", blocks);
        return COLI_ERR_INVALID_ARG;
    }
    bank->copy_blocks = blocks;
    return COLI_OK;
}

int coli_bank_state(coli_expert_bank_t *bank, int32_t *slot_of, int32_t *expert_in, uint32_t *usage,
                    int32_t *last_use, int64_t *stats) {
    if (!bank) return COLI_ERR_INVALID_ARG;
    coli_moe_t *h = bank->h;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) {
        set_err(h, "stream error: %s", cudaGetErrorString(cudaGetLastError()));
        return COLI_ERR_CUDA;
    }
    const BankDev &d = bank->dev;
    struct Copy {
        void *dst;
        const void *src;
        size_t bytes;
    } copies[] = {{slot_of, d.slot_of, sizeof(int32_t) * d.E}, {expert_in, d.expert_in, sizeof(int32_t) * d.S},
                  {usage, d.usage, sizeof(uint32_t) * d.E},     {last_use, d.last_use, sizeof(int32_t) * d.S},
                  {stats, d.stats, sizeof(int64_t) * 3}};
    for (const Copy &c : copies) {
        if (!c.dst) continue;
        if (cudaMemcpy(c.dst, c.src, c.bytes, cudaMemcpyDeviceToHost) != cudaSuccess) {
            set_err(h, "copy failed: %s", cudaGetErrorString(cudaGetLastError()));
            return COLI_ERR_CUDA;
        }
    }
    return COLI_OK;
}

int coli_moe_forward_banked(coli_moe_t *h, coli_expert_bank_t *bank, const void *x_bf16, int32_t T,
                            const float *router_w, const float *router_bias,
                            const coli_mxfp4_experts *shared_expert, int32_t top_k, void *out_bf16) {
    if (!h) return COLI_ERR_INVALID_ARG;
    if (!bank || bank->h != h) {
        set_err(h, "bank is NULL or belongs to another handle");
        return COLI_ERR_INVALID_ARG;
    }
    if (T == 0) {
        h->last_launches = 0;
        return COLI_OK;
    }
    int rc = check_forward(h, x_bf16, T, router_w, shared_expert, top_k, out_bf16);
    if (rc != COLI_OK) return rc;
    cudaGetLastError();
    cudaStream_t st = h->stream, cs = bank->copy;
    const int E = h->cfg.num_experts, S = bank->S;
    const bool with_shared = shared_expert != nullptr;
    const int rows = T * top_k + (with_shared ? T : 0);
    const long cap = std::min<long>((long)T * top_k, E);
    const bool cache = cap <= S;
    const int G = cache ? S : S / 2;
    const int R = cache ? 2 : (int)((cap + G - 1) / G);
    int launches = 0, n;
    h->stage_valid = false;
    if (!run_front(h, x_bf16, T, router_w, router_bias, top_k, with_shared, kNtileMx4, launches))
        return launch_failed(h);
    Workspace &ws = h->ws;
    n = launch_bank_plan(bank->dev, ws.cnt, ws.off, cache, G, R, kNtileMx4, ws.err, st);
    if (n < 0) return launch_failed(h);
    launches += n;
    FfnArgs a = ffn_args(h, x_bf16, T, top_k, rows, nullptr, shared_expert);
    a.routed = bank->slots;
    a.w_slots = S;
    n = launch_quant_x4(a, h->num_sms, st);
    if (n < 0) return launch_failed(h);
    launches += n;
    if (cudaEventRecord(bank->ev_plan, st) != cudaSuccess || cudaStreamWaitEvent(cs, bank->ev_plan, 0) != cudaSuccess)
        return launch_failed(h);
    // Refills on the copy stream: round r's copies overlap round r - 1's GEMMs. A round's copies
    // may reuse slots of round r - 2 only, so they wait for that round's down projection.
    auto refill = [&](int r) -> bool {
        if (r >= 2 && cudaStreamWaitEvent(cs, bank->ev_done[r - 2], 0) != cudaSuccess) return false;
        const int blocks = r == 0 ? h->num_sms : bank->copy_blocks;   // round 0's copies run alone
        if (launch_bank_refill(bank->dev, r, bank->src, bank->slots, bank->eb, blocks, ws.err, cs) < 0) return false;
        ++launches;
        return cudaEventRecord(bank->ev_fill[r], cs) == cudaSuccess;
    };
    const int first_fill = cache ? 1 : 0;   // a cache forward's round 0 computes resident experts
    for (int r = first_fill; r < std::min(R, 2); ++r)
        if (!refill(r)) return launch_failed(h);
    for (int r = 0; r < R; ++r) {
        const bool waits = r >= first_fill;
        if (waits && cudaStreamWaitEvent(st, bank->ev_fill[r], 0) != cudaSuccess) return launch_failed(h);
        const NtileLayout nl = bank_round_layout(bank->dev, r);
        a.tiles = &nl;
        a.grid = r + 1 < R ? h->num_sms - bank->copy_blocks : 0;   // the copy blocks take the rest
        a.pdl_gate_up = !waits;
        n = launch_ffn_mx4(a, h->num_sms, nullptr, nullptr, st);
        if (n == -2) {
            set_err(h, "FP4 block-scaled GEMM path unavailable (needs a tensor-map encoder)");
            return COLI_ERR_INVALID_ARG;
        }
        if (n < 0) return launch_failed(h);
        launches += n;
        if (cudaEventRecord(bank->ev_done[r], st) != cudaSuccess) return launch_failed(h);
        if (r + 2 < R && !refill(r + 2)) return launch_failed(h);
    }
    n = launch_combine(ws.y, ws.inv_row, ws.w, T, h->cfg.hidden, top_k, with_shared,
                       static_cast<__nv_bfloat16 *>(out_bf16), st);
    if (n < 0) return launch_failed(h);
    launches += n;
    h->last_T = T;
    h->last_k = top_k;
    h->last_shared = with_shared;
    h->last_launches = launches;
    h->last_path = COLI_FFN_GEMM_MXF4;
    return COLI_OK;
}

}  // extern "C"
