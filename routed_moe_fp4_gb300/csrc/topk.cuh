// A1 top-k of one token by one warp, shared by the router's top-k kernel (router.cu) and the
// small-T route + permute kernel (permute.cu).
//
// key = fp32(s + b); lane l holds experts l, l+32, ...; k rounds of a warp arg-max on (key
// descending, expert ascending), so bit-identical keys go to the lower expert index. A key that is
// NaN never wins a comparison; only when every remaining key is NaN is the lowest free expert
// taken. w_j = s_j / S with S the fp32 sum of the chosen s in slot order, one IEEE division each.
#pragma once

#include <float.h>
#include <limits.h>

#include "colimoe_internal.cuh"

namespace colimoe {

// Lane j writes idx[t][j] and w[t][j] (and idx_sm[t * k + j] when idx_sm is non-null).
template <int NPL>
__device__ __forceinline__ void topk_token(const float *__restrict__ scores, const float *__restrict__ bias, int E,
                                           int top_k, int t, int lane, int32_t *__restrict__ idx,
                                           float *__restrict__ w, int *idx_sm) {
    float key[NPL], sc[NPL];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
            sc[i] = scores[(size_t)t * E + e];
            key[i] = __fadd_rn(sc[i], bias ? bias[e] : 0.0f);
        } else {
            sc[i] = 0.f;
            key[i] = -INFINITY;
            taken |= 1u << i;          // padding slots are never chosen
        }
    }
    float my_s = 0.f;              // lane j keeps slot j's score and expert (top_k <= 32)
    int my_e = 0;
    for (int j = 0; j < top_k; ++j) {
        float bk = -INFINITY, bs = 0.f;
        int be = INT_MAX;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            const int e = lane + 32 * i;
            const bool free_ = !((taken >> i) & 1u);
            if (free_ && (key[i] > bk || (key[i] == bk && e < be))) {
                bk = key[i];
                be = e;
                bs = sc[i];
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            const float os = __shfl_xor_sync(0xffffffffu, bs, o);
            if (ok > bk || (ok == bk && oe < be)) {
                bk = ok;
                be = oe;
                bs = os;
            }
        }
        if (be == INT_MAX) {           // only NaN keys left: take the lowest free expert
            int cand = INT_MAX;
            float cs = 0.f;
#pragma unroll
            for (int i = NPL - 1; i >= 0; --i)
                if (!((taken >> i) & 1u)) { cand = lane + 32 * i; cs = sc[i]; }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const int oc = __shfl_xor_sync(0xffffffffu, cand, o);
                const float os = __shfl_xor_sync(0xffffffffu, cs, o);
                if (oc < cand) { cand = oc; cs = os; }
            }
            be = cand;
            bs = cs;
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (lane == j) {
            my_s = bs;
            my_e = be;
        }
    }
    // S in slot order, the same chain on every lane; then lane j writes slot j
    float S = 0.0f;
    for (int j = 0; j < top_k; ++j) S = __fadd_rn(S, __shfl_sync(0xffffffffu, my_s, j));
    if (lane < top_k) {
        idx[(size_t)t * top_k + lane] = my_e;
        w[(size_t)t * top_k + lane] = __fdiv_rn(my_s, S);
        if (idx_sm) idx_sm[t * top_k + lane] = my_e;
    }
}

}  // namespace colimoe
