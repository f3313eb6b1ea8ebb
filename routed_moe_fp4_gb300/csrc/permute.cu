// A2 permute: per-expert histogram, exclusive scan, deterministic scatter into expert-grouped
// rows and the inverse map ("the CUDA tier wired into the DeepSeek V4 engine", What it is:
// expert-grouped GEMM rows).
//
// The row of (token t, slot j) with e = idx[t][j] is off[e] + #{t' < t : e in idx[t']}: a stable
// grouping by (expert, token), computed without atomics on positions, so it is the same on every
// run. Group E is the shared expert with rows off[E] + t for every token t.
#include "colimoe_internal.cuh"
#include "block_scan.cuh"
#include "topk.cuh"

namespace colimoe {
namespace {

__global__ void permute_count(const int32_t *__restrict__ idx, int n, int32_t *__restrict__ cnt) {
    pdl_begin();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        atomicAdd(&cnt[idx[i]], 1);
}

// One block of 1024 threads; groups g = 0..E (E <= 1024 + shared handled as the last entry).
// Also lists the non-empty groups in ascending order (touched) with an exclusive prefix of their
// work cost, 1 + ceil(rows / cost_tokens) per weight pass (touched_cost[n_touched] = total), which
// the expert-FFN kernels use to split work evenly across blocks.
// cnt[0..E] (E = the shared expert) must be complete and visible to the block.
__device__ void scan_groups(const int32_t *cnt, int32_t *__restrict__ off, int32_t *__restrict__ touched,
                            int32_t *__restrict__ touched_cost, int32_t *__restrict__ n_touched, int E,
                            int cost_tokens, NtileLayout nl, int ntile) {
    __shared__ int smem[33];
    __shared__ int s_nt;
    const int G = E + 1;
    int base = 0, tbase = 0, cbase = 0;
    for (int g0 = 0; g0 < G; g0 += 1024) {
        const int g = g0 + threadIdx.x;
        const int c = g < G ? cnt[g] : 0;
        const int cost = c > 0 ? 1 + (c + cost_tokens - 1) / cost_tokens : 0;
        int tot, ttot, ctot;
        const int ex = block_exclusive_scan(c, smem, &tot);
        const int tex = block_exclusive_scan(c > 0 ? 1 : 0, smem, &ttot);
        const int cex = block_exclusive_scan(cost, smem, &ctot);
        if (g < G) {
            off[g] = base + ex;
            if (c > 0) {
                touched[tbase + tex] = g;
                touched_cost[tbase + tex] = cbase + cex;
            }
        }
        base += tot;
        tbase += ttot;
        cbase += ctot;
    }
    if (threadIdx.x == 0) {
        off[G] = base;
        *n_touched = tbase;
        touched_cost[tbase] = cbase;
        s_nt = tbase;
    }
    if (!ntile) return;
    // n-tiles of the block-scaled GEMM for both tile sizes, over the touched groups in order
    __syncthreads();
    const int nt = s_nt;
    int c_small = 0, c_large = 0;
    for (int u0 = 0; u0 < nt; u0 += 1024) {
        const int u = u0 + threadIdx.x;
        const int c = u < nt ? cnt[touched[u]] : 0;
        const int ns = (c + ntile - 1) / ntile, nlg = (c + 2 * ntile - 1) / (2 * ntile);
        int tot_s, tot_l;
        const int ex_s = block_exclusive_scan(ns, smem, &tot_s);
        const int ex_l = block_exclusive_scan(nlg, smem, &tot_l);
        if (u < nt) {
            const int g = touched[u], o = off[g];
            nl.prefix_small[u] = c_small + ex_s;
            nl.prefix_large[u] = c_large + ex_l;
            for (int r = 0; r < ns; ++r) {
                nl.owner_small[c_small + ex_s + r] = u;
                nl.rec_small[c_small + ex_s + r] = make_int2(o + r * ntile, g | (min(ntile, c - r * ntile) << 16));
            }
            for (int r = 0; r < nlg; ++r) {
                nl.owner_large[c_large + ex_l + r] = u;
                nl.rec_large[c_large + ex_l + r] =
                    make_int2(o + r * 2 * ntile, g | (min(2 * ntile, c - r * 2 * ntile) << 16));
            }
        }
        c_small += tot_s;
        c_large += tot_l;
    }
    if (threadIdx.x == 0) {
        nl.prefix_small[nt] = c_small;
        nl.prefix_large[nt] = c_large;
        nl.count[0] = c_small;
        nl.count[1] = c_large;
    }
}

__global__ void __launch_bounds__(1024)
permute_scan(int32_t *__restrict__ cnt, int32_t *__restrict__ off, int32_t *__restrict__ touched,
             int32_t *__restrict__ touched_cost, int32_t *__restrict__ n_touched, int E, int shared_rows,
             int cost_tokens, NtileLayout nl, int ntile) {
    pdl_begin();
    if (threadIdx.x == 0) cnt[E] = shared_rows;
    __syncthreads();
    scan_groups(cnt, off, touched, touched_cost, n_touched, E, cost_tokens, nl, ntile);
}

// Small T (T < kSmallRouteTokens, k <= 32): A1's top-k and all of A2 in one block of 1024 threads,
// after the router's logits kernel. Warp w takes tokens w and w + 32. The histogram, offsets and
// touched list stay in shared memory (the global copies are written, never read back); the scans
// are those of permute_scan; one warp per touched group scatters its rows in token order (ballot
// over 32 tokens at a time). Same outputs as router_topk + permute_count + permute_scan +
// permute_scatter.
template <int NPL>
__global__ void __launch_bounds__(1024)
route_permute_small(const float *__restrict__ scores, const float *__restrict__ bias, int T, int E, int top_k,
                    int32_t *__restrict__ idx, float *__restrict__ w, int32_t *__restrict__ cnt,
                    int32_t *__restrict__ off, int32_t *__restrict__ touched, int32_t *__restrict__ touched_cost,
                    int32_t *__restrict__ n_touched, int shared_rows, int cost_tokens, NtileLayout nl, int ntile,
                    int32_t *__restrict__ src_token, int32_t *__restrict__ inv_row) {
    pdl_begin();
    __shared__ int idx_s[(kSmallRouteTokens - 1) * 32];
    __shared__ int cnt_s[1025], off_s[1026], touched_s[1025];
    __shared__ unsigned long long smem[33];
    __shared__ int s_nt;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = E + 1;
    for (int t = warp; t < T; t += 32) topk_token<NPL>(scores, bias, E, top_k, t, lane, idx, w, idx_s);
    for (int g = threadIdx.x; g < G; g += blockDim.x) cnt_s[g] = g == E ? shared_rows : 0;
    __syncthreads();
    for (int i = threadIdx.x; i < T * top_k; i += blockDim.x) atomicAdd(&cnt_s[idx_s[i]], 1);
    __syncthreads();
    // groups: offsets, touched list and GEMV costs, in one scan of three 21-bit fields (row count,
    // touched flag, cost: their sums stay below 2^21 with T < 64 tokens and k <= 32)
    constexpr unsigned long long kF = (1ull << 21) - 1;
    int base = 0, tbase = 0, cbase = 0;
    for (int g0 = 0; g0 < G; g0 += 1024) {
        const int g = g0 + threadIdx.x;
        const int c = g < G ? cnt_s[g] : 0;
        const int cost = c > 0 ? 1 + (c + cost_tokens - 1) / cost_tokens : 0;
        unsigned long long tot3;
        const unsigned long long ex3 = block_exclusive_scan64(
            (unsigned long long)c | ((unsigned long long)(c > 0) << 21) | ((unsigned long long)cost << 42), smem, &tot3);
        const int ex = (int)(ex3 & kF), tex = (int)((ex3 >> 21) & kF), cex = (int)(ex3 >> 42);
        const int tot = (int)(tot3 & kF), ttot = (int)((tot3 >> 21) & kF), ctot = (int)(tot3 >> 42);
        if (g < G) {
            cnt[g] = c;
            off[g] = off_s[g] = base + ex;
            if (c > 0) {
                touched[tbase + tex] = touched_s[tbase + tex] = g;
                touched_cost[tbase + tex] = cbase + cex;
            }
        }
        base += tot;
        tbase += ttot;
        cbase += ctot;
    }
    if (threadIdx.x == 0) {
        off[G] = off_s[G] = base;
        *n_touched = tbase;
        touched_cost[tbase] = cbase;
        s_nt = tbase;
    }
    __syncthreads();
    const int nt = s_nt;
    if (ntile) {   // n-tiles of the block-scaled GEMM for both tile sizes, over the touched groups
        int c_small = 0, c_large = 0;
        for (int u0 = 0; u0 < nt; u0 += 1024) {
            const int u = u0 + threadIdx.x;
            const int g = u < nt ? touched_s[u] : 0;
            const int c = u < nt ? cnt_s[g] : 0;
            const int ns = (c + ntile - 1) / ntile, nlg = (c + 2 * ntile - 1) / (2 * ntile);
            unsigned long long tot2;
            const unsigned long long ex2 =
                block_exclusive_scan64((unsigned long long)ns | ((unsigned long long)nlg << 32), smem, &tot2);
            const int ex_s = (int)(ex2 & 0xFFFFFFFFull), ex_l = (int)(ex2 >> 32);
            const int tot_s = (int)(tot2 & 0xFFFFFFFFull), tot_l = (int)(tot2 >> 32);
            if (u < nt) {
                const int o = off_s[g];
                nl.prefix_small[u] = c_small + ex_s;
                nl.prefix_large[u] = c_large + ex_l;
                for (int r = 0; r < ns; ++r) {
                    nl.owner_small[c_small + ex_s + r] = u;
                    nl.rec_small[c_small + ex_s + r] = make_int2(o + r * ntile, g | (min(ntile, c - r * ntile) << 16));
                }
                for (int r = 0; r < nlg; ++r) {
                    nl.owner_large[c_large + ex_l + r] = u;
                    nl.rec_large[c_large + ex_l + r] =
                        make_int2(o + r * 2 * ntile, g | (min(2 * ntile, c - r * 2 * ntile) << 16));
                }
            }
            c_small += tot_s;
            c_large += tot_l;
        }
        if (threadIdx.x == 0) {
            nl.prefix_small[nt] = c_small;
            nl.prefix_large[nt] = c_large;
            nl.count[0] = c_small;
            nl.count[1] = c_large;
        }
    }
    // stable scatter
    for (int u = warp; u < nt; u += 32) {
        const int g = touched_s[u];
        int run = off_s[g];
        if (g == E) {                        // shared expert: rows off[E] + t
            for (int t = lane; t < T; t += 32) src_token[run + t] = t;
            continue;
        }
        for (int t0 = 0; t0 < T; t0 += 32) {
            const int t = t0 + lane;
            int slot = -1;
            if (t < T)
                for (int j = 0; j < top_k; ++j)
                    if (idx_s[t * top_k + j] == g) slot = j;
            const unsigned bal = __ballot_sync(0xffffffffu, slot >= 0);
            if (slot >= 0) {
                const int row = run + __popc(bal & ((1u << lane) - 1u));
                src_token[row] = t;
                inv_row[t * top_k + slot] = row;
            }
            run += __popc(bal);
        }
    }
}

// Block e scans the tokens in order and places the (t, j) pairs routed to expert e.
// Block E writes the shared expert's identity rows.
__global__ void __launch_bounds__(256)
permute_scatter(const int32_t *__restrict__ idx, int T, int E, int top_k, const int32_t *__restrict__ cnt,
                const int32_t *__restrict__ off, int32_t *__restrict__ src_token, int32_t *__restrict__ inv_row) {
    pdl_begin();
    const int e = blockIdx.x;
    if (e == E) {
        const int base = off[E];
        for (int t = threadIdx.x; t < cnt[E]; t += blockDim.x) src_token[base + t] = t;
        return;
    }
    if (cnt[e] == 0) return;
    __shared__ int warp_tot[8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int running = off[e];
    for (int t0 = 0; t0 < T; t0 += 256) {
        const int t = t0 + threadIdx.x;
        int slot = -1;
        if (t < T) {
            for (int j = 0; j < top_k; ++j)
                if (idx[(size_t)t * top_k + j] == e) slot = j;
        }
        const unsigned ballot = __ballot_sync(0xffffffffu, slot >= 0);
        const int in_warp = __popc(ballot & ((1u << lane) - 1u));
        if (lane == 0) warp_tot[warp] = __popc(ballot);
        __syncthreads();
        int before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            before += (w < warp) ? warp_tot[w] : 0;
            total += warp_tot[w];
        }
        if (slot >= 0) {
            const int row = running + before + in_warp;
            src_token[row] = t;
            inv_row[(size_t)t * top_k + slot] = row;
        }
        running += total;
        __syncthreads();
    }
}

}  // namespace

int launch_route_permute_small(const float *router_b, int T, int E, int top_k, bool with_shared, int cost_tokens,
                               int ntile, Workspace &ws, cudaStream_t st) {
    if (T < 1 || T >= kSmallRouteTokens || top_k > 32 || E > 1024) return -2;
    const int rows = T * top_k + (with_shared ? T : 0);
    const int npl = (E + 31) / 32;
    auto kern = npl <= 1 ? route_permute_small<1> : npl <= 2 ? route_permute_small<2> : npl <= 4 ? route_permute_small<4>
              : npl <= 8 ? route_permute_small<8> : npl <= 16 ? route_permute_small<16> : route_permute_small<32>;
    launch_pdl(kern, dim3(1), dim3(1024), 0, st, (const float *)ws.scores, router_b, T, E, top_k, ws.idx, ws.w,
               ws.cnt, ws.off, ws.touched, ws.touched_cost, ws.n_touched, with_shared ? T : 0, cost_tokens,
               ntile_layout(ws.tile_sched, E, rows), ntile, ws.src_token, ws.inv_row);
    return cudaPeekAtLastError() == cudaSuccess ? 1 : -1;
}

int launch_permute(const int32_t *idx, int T, int E, int top_k, bool with_shared, int cost_tokens, int ntile,
                   Workspace &ws, cudaStream_t st) {
    const int n = T * top_k;
    const int rows = n + (with_shared ? T : 0);
    // ws.cnt was cleared by the router's last kernel
    launch_pdl(permute_count, dim3((n + 255) / 256), dim3(256), 0, st, idx, n, ws.cnt);
    launch_pdl(permute_scan, dim3(1), dim3(1024), 0, st, ws.cnt, ws.off, ws.touched, ws.touched_cost, ws.n_touched, E,
               with_shared ? T : 0, cost_tokens, ntile_layout(ws.tile_sched, E, rows), ntile);
    launch_pdl(permute_scatter, dim3(E + 1), dim3(256), 0, st, idx, T, E, top_k, (const int32_t *)ws.cnt,
               (const int32_t *)ws.off, ws.src_token, ws.inv_row);
    return cudaPeekAtLastError() == cudaSuccess ? 3 : -1;
}

}  // namespace colimoe
