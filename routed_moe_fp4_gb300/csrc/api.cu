// The C ABI (colimoe.h) and the host orchestration of one forward: argument checks, the
// workspace, and the stream-ordered launch sequence A1 router -> A2 permute -> A3/A4 expert
// FFN -> A5 combine. No host synchronisation and no allocation inside a forward.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <new>

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

void free_ws(Workspace &ws) {
    void *ptrs[] = {ws.xq, ws.xqs, ws.hq, ws.hqs, ws.scores, ws.logit_part, ws.idx,  ws.w,  ws.inv_row, ws.src_token, ws.cnt, ws.off, ws.touched, ws.touched_cost,
                    ws.n_touched, ws.xp, ws.h, ws.y, ws.xh, ws.xinv, ws.hh, ws.hinv, ws.err, ws.x_stage,
                    ws.out_stage, ws.tile_sched};
    for (void *p : ptrs)
        if (p) cudaFree(p);
    ws = Workspace();
}

template <typename T>
bool alloc(T **p, size_t count) {
    return cudaMalloc(reinterpret_cast<void **>(p), count * sizeof(T) + 256) == cudaSuccess;
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

enum FfnKind { kFfnGemv, kFfnMx, kFfnBf16, kFfnMx4 };

bool mx_pointers_ok(const coli_mxfp4_experts *r, const coli_mxfp4_experts *s) {
    auto al = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31) == 0; };
    return al(r->gate_up_codes) && al(r->down_codes) && (!s || (al(s->gate_up_codes) && al(s->down_codes)));
}

// The FFN kernels a forward uses: the FP4 x FP4 block-scaled GEMM whenever it can run (weights go
// to the tensor cores as stored, 64 K per instruction, at every token count); then the E2M1 x E4M3
// block-scaled GEMM; otherwise the bf16 GEMM when tokens per touched expert are many, the GEMV
// when they are few.
FfnKind pick_ffn(const coli_moe_t *h, int T, int top_k, const coli_mxfp4_experts *r, const coli_mxfp4_experts *s) {
    switch (h->ffn_path) {
        case COLI_FFN_GEMV: return kFfnGemv;
        case COLI_FFN_GEMM: return kFfnMx;
        case COLI_FFN_GEMM_BF16: return kFfnBf16;
        case COLI_FFN_GEMM_MXF4: return kFfnMx4;
        default: break;
    }
    if (mx4_available()) return kFfnMx4;
    if (mx_available() && mx_pointers_ok(r, s)) return kFfnMx;
    if (!gemm_available()) return kFfnGemv;
    const double E = h->cfg.num_experts;
    const double touched = E * (1.0 - pow(1.0 - (double)top_k / E, (double)T));
    return (double)T * top_k / (touched > 0 ? touched : 1.0) > 3.0 ? kFfnBf16 : kFfnGemv;
}

int forward_impl(coli_moe_t *h, const void *x_bf16, int32_t T, const float *router_w, const float *router_bias,
                 const coli_mxfp4_experts *packed, const coli_mxfp4_experts *shared, int32_t top_k,
                 void *out_bf16) {
    const coli_moe_config &c = h->cfg;
    if (T == 0) {
        h->last_launches = 0;
        h->last_path = COLI_FFN_AUTO;
        return COLI_OK;
    }
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
    if (x_bf16 == out_bf16) {
        set_err(h, "out_bf16 may not alias x_bf16");
        return COLI_ERR_INVALID_ARG;
    }
    if (!valid_experts(packed)) {
        set_err(h, "packed_experts must hold four non-NULL 16-byte aligned device pointers");
        return COLI_ERR_INVALID_ARG;
    }
    if (shared && (c.shared_inter == 0 || !valid_experts(shared))) {
        set_err(h, c.shared_inter == 0 ? "shared_expert given but cfg.shared_inter is 0"
                                       : "shared_expert must hold four non-NULL 16-byte aligned device pointers");
        return COLI_ERR_INVALID_ARG;
    }
    cudaGetLastError();   // clear a stale error so launch checks below see only our own
    cudaStream_t st = h->stream;
    const int E = c.num_experts, H = c.hidden;
    const bool with_shared = shared != nullptr;
    Workspace &ws = h->ws;
    int launches = 0, n;
    const FfnKind ffn = pick_ffn(h, T, top_k, packed, shared);
    const bool gemm = ffn == kFfnBf16;
    const int ntile = ffn == kFfnMx ? kNtileMx : ffn == kFfnMx4 ? kNtileMx4 : 0;
    const int rows = T * top_k + (with_shared ? T : 0);
    const bool prof = h->profiling;
    h->stage_valid = false;
    if (prof) cudaEventRecord(h->ev[0], st);

    if (T < kSmallRouteTokens) {
        // logits, then top-k and the whole permutation in one single-block launch
        n = launch_router(static_cast<const __nv_bfloat16 *>(x_bf16), T, H, router_w, router_bias, E, top_k,
                          ws.scores, ws.idx, ws.w, ws.logit_part, ws.logit_part_floats, h->num_sms, nullptr, 0, st,
                          false);
        if (n < 0) goto launch_fail;
        launches += n;
        if (prof) cudaEventRecord(h->ev[1], st);
        n = launch_route_permute_small(router_bias, T, E, top_k, with_shared, kGemvCostTokens, ntile, ws, st);
        if (n < 0) goto launch_fail;
        launches += n;
        if (gemm) {
            n = launch_gather(static_cast<const __nv_bfloat16 *>(x_bf16), H, rows, ws, st);
            if (n < 0) goto launch_fail;
            launches += n;
        }
    } else {
        n = launch_router(static_cast<const __nv_bfloat16 *>(x_bf16), T, H, router_w, router_bias, E, top_k,
                          ws.scores, ws.idx, ws.w, ws.logit_part, ws.logit_part_floats, h->num_sms, ws.cnt, E + 1,
                          st);
        if (n < 0) goto launch_fail;
        launches += n;
        if (prof) cudaEventRecord(h->ev[1], st);
        n = launch_permute(ws.idx, T, E, top_k, with_shared, static_cast<const __nv_bfloat16 *>(x_bf16), H, gemm,
                           kGemvCostTokens, ntile, ws, st);
        if (n < 0) goto launch_fail;
        launches += n;
    }
    {
        FfnArgs a{};
        a.routed = to_set(packed);
        a.shared = to_set(shared);
        a.E = E;
        a.H = H;
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
        a.x = static_cast<const __nv_bfloat16 *>(x_bf16);
        a.xp = ws.xp;
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
        a.err = ws.err;
        a.wait_ns = h->wait_ns;
        if (ffn == kFfnMx || ffn == kFfnMx4) {   // the activation terms belong to the permute stage
            n = ffn == kFfnMx ? launch_quant_x(a, st) : launch_quant_x4(a, st);
            if (n < 0) goto launch_fail;
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
        } else if (ffn == kFfnMx) {
            n = launch_ffn_mx(a, h->num_sms, ws.tile_sched, mid, st);
            if (n == -2) {
                set_err(h, "block-scaled GEMM path unavailable (needs 32-byte aligned code pointers and a "
                           "tensor-map encoder)");
                return COLI_ERR_INVALID_ARG;
            }
        } else if (gemm) {
            n = launch_ffn_gemm(a, h->num_sms, ws.tile_sched, mid, st);
            if (n == -2) {
                set_err(h, "tensor-core grouped GEMM path is not available for this configuration");
                return COLI_ERR_INVALID_ARG;
            }
        } else {
            n = launch_ffn_gemv(a, h->num_sms, mid, st);
        }
        if (n < 0) goto launch_fail;
        launches += n;
    }
    if (prof) cudaEventRecord(h->ev[4], st);
    n = launch_combine(ws.y, ws.inv_row, ws.w, T, H, top_k, with_shared, static_cast<__nv_bfloat16 *>(out_bf16), st);
    if (n < 0) goto launch_fail;
    launches += n;
    if (prof) {
        cudaEventRecord(h->ev[5], st);
        h->stage_valid = true;
    }
    h->last_T = T;
    h->last_k = top_k;
    h->last_shared = with_shared;
    h->last_launches = launches;
    h->last_path = ffn == kFfnGemv ? COLI_FFN_GEMV : ffn == kFfnMx ? COLI_FFN_GEMM
                 : ffn == kFfnBf16 ? COLI_FFN_GEMM_BF16 : COLI_FFN_GEMM_MXF4;
    return COLI_OK;

launch_fail : {
    const cudaError_t e = cudaGetLastError();
    set_err(h, "kernel launch failed: %s", cudaGetErrorString(e));
    return COLI_ERR_CUDA;
}
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
    const size_t Tm = c.max_tokens, km = c.max_top_k, E = c.num_experts, H = c.hidden;
    const size_t rows = Tm * km + Tm;
    Workspace &ws = h->ws;
    ws.logit_part_floats = 4 * (Tm > 1024 ? Tm : 1024) * E;
    bool ok = alloc(&ws.scores, Tm * E) && alloc(&ws.logit_part, ws.logit_part_floats) && alloc(&ws.idx, Tm * km) && alloc(&ws.w, Tm * km) &&
              alloc(&ws.inv_row, Tm * km) && alloc(&ws.src_token, rows) && alloc(&ws.cnt, E + 1) &&
              alloc(&ws.off, E + 2) && alloc(&ws.touched, E + 1) && alloc(&ws.touched_cost, E + 2) && alloc(&ws.n_touched, 4) &&
              alloc(&ws.xp, rows * H) && alloc(&ws.h, rows * (size_t)h->I_max) && alloc(&ws.y, rows * H) &&
              alloc(&ws.xh, Tm * H) && alloc(&ws.xinv, Tm) && alloc(&ws.hh, rows * (size_t)h->I_max) &&
              alloc(&ws.hinv, rows) && alloc(&ws.err, 4) && alloc(&ws.x_stage, Tm * H) &&
              alloc(&ws.out_stage, Tm * H);
    if (ok)
        ok = alloc(&ws.xq, 2 * rows * H) && alloc(&ws.xqs, 4 * rows * (H / 32)) &&
             alloc(&ws.hq, 3 * rows * (size_t)h->I_max) && alloc(&ws.hqs, 4 * rows * (size_t)(h->I_max / 32));
    if (ok) ok = cudaMemset(ws.err, 0, sizeof(int)) == cudaSuccess;
    if (ok) {
        ws.tile_sched_bytes = gemm_sched_bytes((int)E, (int)rows);
        const size_t mx_bytes = ntile_layout_ints((int)E, (int)rows) * sizeof(int32_t);
        if (mx_bytes > ws.tile_sched_bytes) ws.tile_sched_bytes = mx_bytes;
        ok = cudaMalloc(&ws.tile_sched, ws.tile_sched_bytes + 256) == cudaSuccess;
    }
    if (!ok) {
        cudaGetLastError();
        free_ws(ws);
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

}  // extern "C"
