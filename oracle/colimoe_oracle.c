/*
 * colimoe_oracle.c -- plain, slow CPU oracle of the routed MXFP4 MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY (see colimoe_oracle.h). Floating point is fp64 except where
 * the definition fixes fp32: the routing key s + b, the renormalisation sum and the
 * division. Build without -ffast-math and with -ffp-contract=off so that every fp32
 * operation is one IEEE operation.
 *
 * COLI_ORACLE_MUTANT=n (n > 0) plants one known mistake; the tests use such builds to
 * show that the oracle's pins catch each of them. The default build carries none.
 */
#include "colimoe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef COLI_ORACLE_MUTANT
#define COLI_ORACLE_MUTANT 0
#endif
#define MUT(n) (COLI_ORACLE_MUTANT == (n))

int32_t coli_oracle_mutant(void) { return COLI_ORACLE_MUTANT; }

int32_t coli_oracle_threads(void) {
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------------------
 * Formats
 * E2M1 (OCP Microscaling v1.0 FP4): bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa;
 * exponent 0 is subnormal (0 or 0.5). The 8 magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6.
 */
static const double kE2M1[16] = {
    0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
    -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0,
};
#if COLI_ORACLE_MUTANT == 12
static const double kE2M1_m12[16] = {
    0.0, 0.5, 1.0, 1.5, 2.0, 4.0, 3.0, 6.0,
    -0.0, -0.5, -1.0, -1.5, -2.0, -4.0, -3.0, -6.0,
};
#define E2M1_TABLE kE2M1_m12
#else
#define E2M1_TABLE kE2M1
#endif

double coli_oracle_e2m1(int code) { return E2M1_TABLE[code & 15]; }

/* UE8M0: the fp32 whose bit pattern is s << 23, i.e. 2^(s-127) for s in 1..254, +0 for
 * s = 0 and +inf for s = 255 (the edges the pages' MXFP4 decode reproduces). */
double coli_oracle_e8m0(int s) {
    uint32_t bits = ((uint32_t)(s & 255)) << 23;
    if (MUT(2)) bits = ((uint32_t)((s & 255) - ((s & 255) > 0))) << 23;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

double coli_oracle_mxfp4(const uint8_t *codes, const uint8_t *scales, int64_t K, int64_t row, int64_t k) {
    uint8_t byte = codes[row * (K / 2) + k / 2];
    int even = (k % 2) == 0;
    if (MUT(1)) even = !even;
    int nib = even ? (byte & 15) : (byte >> 4);
    return coli_oracle_e2m1(nib) * coli_oracle_e8m0(scales[row * (K / 32) + k / 32]);
}

double coli_oracle_bf16(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Nearest bf16 (8 significant bits, fp32 exponent range), ties to the even significand. */
uint16_t coli_oracle_round_bf16(double v) {
    if (isnan(v)) return 0x7FC0;
    if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
    double a = fabs(v);
    int e;
    frexp(a, &e);                       /* a = m * 2^e, m in [0.5, 1) */
    int q = e - 8;                      /* quantum exponent: 8 significant bits */
    if (q < -133) q = -133;             /* subnormal bf16 spacing is 2^-133 */
    double scaled = ldexp(a, -q);
    double r = MUT(16) ? floor(scaled) : nearbyint(scaled);   /* FE_TONEAREST: ties to even */
    double res = ldexp(r, q);
    uint16_t out;
    if (res > 3.3895313892515355e38) {  /* above the largest finite bf16 -> infinity */
        out = 0x7F80;
    } else {
        float f = (float)res;           /* exact: res has <= 8 significant bits */
        uint32_t u;
        memcpy(&u, &f, sizeof u);
        out = (uint16_t)(u >> 16);
    }
    return (uint16_t)(out | (signbit(v) ? 0x8000 : 0));
}

/* ------------------------------------------------------------------------------------
 * Router */
void coli_oracle_router_logits(const uint16_t *x, int32_t T, int32_t H, const float *router_w,
                               int32_t E, double *logits) {
    int32_t Hsum = MUT(15) ? H - 1 : H;
#pragma omp parallel for schedule(static)
    for (int64_t te = 0; te < (int64_t)T * E; ++te) {
        int64_t t = te / E, e = te % E;
        double acc = 0.0;
        for (int32_t h = 0; h < Hsum; ++h)
            acc += coli_oracle_bf16(x[t * H + h]) * (double)router_w[e * H + h];
        logits[te] = acc;
    }
}

void coli_oracle_sigmoid(const double *logits, int64_t n, float *s) {
    for (int64_t i = 0; i < n; ++i) {
        double z = logits[i];
        double v = MUT(13) ? 1.0 / (1.0 + exp(z)) : 1.0 / (1.0 + exp(-z));
        s[i] = (float)v;
    }
}

void coli_oracle_route(const float *s, const float *router_b, int32_t T, int32_t E, int32_t top_k,
                       int32_t *idx, float *w) {
    float *key = (float *)malloc(sizeof(float) * (size_t)E);
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    for (int32_t t = 0; t < T; ++t) {
        const float *st = s + (int64_t)t * E;
        for (int32_t e = 0; e < E; ++e) {
            float b = (router_b && !MUT(3)) ? router_b[e] : 0.0f;
            key[e] = st[e] + b;          /* one fp32 addition */
            taken[e] = 0;
        }
        /* selection: k passes, each the largest remaining key, ties to the lower index */
        for (int32_t j = 0; j < top_k; ++j) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || key[e] > key[best] || (MUT(5) && key[e] == key[best])) best = e;
            }
            taken[best] = 1;
            idx[(int64_t)t * top_k + j] = best;
        }
        if (MUT(18)) {                   /* ascending instead of descending order */
            for (int32_t j = 0; j < top_k / 2; ++j) {
                int32_t a = idx[(int64_t)t * top_k + j];
                idx[(int64_t)t * top_k + j] = idx[(int64_t)t * top_k + top_k - 1 - j];
                idx[(int64_t)t * top_k + top_k - 1 - j] = a;
            }
        }
        /* renormalisation: S summed in fp32 in slot order, then one fp32 division each */
        float S = 0.0f;
        for (int32_t j = 0; j < top_k; ++j) {
            int32_t e = idx[(int64_t)t * top_k + j];
            S = S + (MUT(4) ? key[e] : st[e]);
        }
        for (int32_t j = 0; j < top_k; ++j) {
            int32_t e = idx[(int64_t)t * top_k + j];
            float num = MUT(4) ? key[e] : st[e];
            w[(int64_t)t * top_k + j] = MUT(6) ? num : num / S;
        }
    }
    free(key);
    free(taken);
}

/* ------------------------------------------------------------------------------------
 * Permute: stable grouping of the (token, slot) pairs by expert, tokens ascending. */
void coli_oracle_permute(const int32_t *idx, int32_t T, int32_t E, int32_t top_k, int32_t with_shared,
                         int32_t *cnt, int32_t *off, int32_t *src_token, int32_t *inv_row) {
    for (int32_t e = 0; e <= E; ++e) cnt[e] = 0;
    for (int64_t i = 0; i < (int64_t)T * top_k; ++i) cnt[idx[i]]++;
    cnt[E] = with_shared ? T : 0;
    off[0] = 0;
    for (int32_t g = 0; g <= E; ++g) off[g + 1] = off[g] + cnt[g];
    if (MUT(17))                          /* inclusive instead of exclusive prefix */
        for (int32_t g = 0; g < E; ++g) off[g] = off[g] + cnt[g];
    for (int32_t e = 0; e < E; ++e) {
        int32_t next = 0;
        for (int32_t tt = 0; tt < T; ++tt) {
            int32_t t = MUT(9) ? T - 1 - tt : tt;
            for (int32_t j = 0; j < top_k; ++j) {
                if (idx[(int64_t)t * top_k + j] != e) continue;
                int32_t row = off[e] + next++;
                src_token[row] = t;
                inv_row[(int64_t)t * top_k + j] = row;
            }
        }
    }
    for (int32_t t = 0; t < T && with_shared; ++t) src_token[off[E] + t] = t;
}

/* ------------------------------------------------------------------------------------
 * Expert FFN on one row: SwiGLU MLP with MXFP4 weights, everything in fp64. */
void coli_oracle_expert_row(const uint16_t *x_row, int32_t H, int32_t I,
                            const uint8_t *gu_codes, const uint8_t *gu_scales,
                            const uint8_t *d_codes, const uint8_t *d_scales,
                            double *y, double *h_out) {
    double *xv = (double *)malloc(sizeof(double) * (size_t)H);
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    for (int32_t k = 0; k < H; ++k) xv[k] = coli_oracle_bf16(x_row[k]);
    for (int32_t i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int32_t k = 0; k < H; ++k) {
            g += coli_oracle_mxfp4(gu_codes, gu_scales, H, i, k) * xv[k];
            u += coli_oracle_mxfp4(gu_codes, gu_scales, H, (int64_t)I + i, k) * xv[k];
        }
        if (MUT(8)) { double tmp = g; g = u; u = tmp; }
        double silu = MUT(7) ? g / (1.0 + exp(g)) : g / (1.0 + exp(-g));
        h[i] = silu * u;
    }
    int32_t Ksum = MUT(14) ? I - 32 : I;
    for (int32_t m = 0; m < H; ++m) {
        double acc = 0.0;
        for (int32_t i = 0; i < Ksum; ++i) acc += coli_oracle_mxfp4(d_codes, d_scales, I, m, i) * h[i];
        y[m] = acc;
    }
    if (h_out) memcpy(h_out, h, sizeof(double) * (size_t)I);
    free(h);
    free(xv);
}

/* out_row = round_bf16(y_shared + sum_j w_j * y_j), fp64 sum in that order. */
static void combine_row(int32_t H, int32_t top_k, const float *w_t, const double *const *y_slot,
                        const double *y_shared, uint16_t *out_row, double *out_f64_row) {
    for (int32_t m = 0; m < H; ++m) {
        double acc = (y_shared && !MUT(10)) ? y_shared[m] : 0.0;
        for (int32_t j = 0; j < top_k; ++j) {
            int32_t jw = MUT(11) ? (j + 1) % top_k : j;
            acc += (double)w_t[jw] * y_slot[j][m];
        }
        out_row[m] = coli_oracle_round_bf16(acc);
        if (out_f64_row) out_f64_row[m] = acc;
    }
}

static const uint8_t *off_ptr(const uint8_t *base, int64_t e, int64_t per) { return base + e * per; }

void coli_oracle_tokens_output(const uint16_t *x, int32_t H, int32_t I, int32_t I_s,
                               const int32_t *idx, const float *w, int32_t top_k,
                               const uint8_t *gu_codes, const uint8_t *gu_scales,
                               const uint8_t *d_codes, const uint8_t *d_scales,
                               const uint8_t *sh_gu_codes, const uint8_t *sh_gu_scales,
                               const uint8_t *sh_d_codes, const uint8_t *sh_d_scales,
                               const int32_t *tokens, int32_t n_tokens,
                               uint16_t *out, double *out_f64) {
    const int64_t gu_c = 2LL * I * (H / 2), gu_s = 2LL * I * (H / 32);
    const int64_t d_c = (int64_t)H * (I / 2), d_s = (int64_t)H * (I / (MUT(32) ? 16 : 32));
    const int with_shared = sh_gu_codes != NULL && I_s > 0 && !MUT(33);
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t n = 0; n < n_tokens; ++n) {
        int32_t t = tokens[n];
        const uint16_t *xr = x + (int64_t)t * H;
        double *ys = (double *)malloc(sizeof(double) * (size_t)H * (size_t)(top_k + 1));
        const double **slot = (const double **)malloc(sizeof(double *) * (size_t)top_k);
        for (int32_t j = 0; j < top_k; ++j) {
            int64_t e = idx[(int64_t)t * top_k + j];
            double *yj = ys + (int64_t)j * H;
            coli_oracle_expert_row(xr, H, I, off_ptr(gu_codes, e, gu_c), off_ptr(gu_scales, e, gu_s),
                                   off_ptr(d_codes, e, d_c), off_ptr(d_scales, e, d_s), yj, NULL);
            slot[j] = yj;
        }
        double *ysh = NULL;
        if (with_shared) {
            ysh = ys + (int64_t)top_k * H;
            coli_oracle_expert_row(xr, H, I_s, sh_gu_codes, sh_gu_scales, sh_d_codes, sh_d_scales, ysh, NULL);
        }
        combine_row(H, top_k, w + (int64_t)t * top_k, slot, ysh, out + (int64_t)n * H,
                    out_f64 ? out_f64 + (int64_t)n * H : NULL);
        free(slot);
        free(ys);
    }
}

void coli_oracle_moe_forward(const uint16_t *x, int32_t T, int32_t H, int32_t E, int32_t I, int32_t I_s,
                             const float *router_w, const float *router_b, int32_t top_k,
                             const uint8_t *gu_codes, const uint8_t *gu_scales,
                             const uint8_t *d_codes, const uint8_t *d_scales,
                             const uint8_t *sh_gu_codes, const uint8_t *sh_gu_scales,
                             const uint8_t *sh_d_codes, const uint8_t *sh_d_scales,
                             float *s, int32_t *idx, float *w,
                             int32_t *cnt, int32_t *off, int32_t *src_token, int32_t *inv_row,
                             uint16_t *out, double *out_f64) {
    const int with_shared = sh_gu_codes != NULL && I_s > 0;
    double *logits = (double *)malloc(sizeof(double) * (size_t)T * (size_t)E);
    coli_oracle_router_logits(x, T, H, router_w, E, logits);
    coli_oracle_sigmoid(logits, (int64_t)T * E, s);
    free(logits);
    coli_oracle_route(s, router_b, T, E, top_k, idx, w);
    coli_oracle_permute(idx, T, E, top_k, with_shared, cnt, off, src_token, inv_row);

    /* expert FFN over the expert-grouped rows, group by group */
    const int64_t rows = off[E + 1];
    const int64_t gu_c = 2LL * I * (H / 2), gu_s = 2LL * I * (H / 32);
    const int64_t d_c = (int64_t)H * (I / 2), d_s = (int64_t)H * (I / 32);
    double *Y = (double *)malloc(sizeof(double) * (size_t)(rows > 0 ? rows : 1) * (size_t)H);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        int32_t g = 0;
        while (off[g + 1] <= r) ++g;          /* the group that holds row r */
        const uint16_t *xr = x + (int64_t)src_token[r] * H;
        if (g < E)
            coli_oracle_expert_row(xr, H, I, off_ptr(gu_codes, g, gu_c), off_ptr(gu_scales, g, gu_s),
                                   off_ptr(d_codes, g, d_c), off_ptr(d_scales, g, d_s), Y + r * H, NULL);
        else
            coli_oracle_expert_row(xr, H, I_s, sh_gu_codes, sh_gu_scales, sh_d_codes, sh_d_scales,
                                   Y + r * H, NULL);
    }
    /* combine: gather each token's rows through inv_row */
    const double **slot = (const double **)malloc(sizeof(double *) * (size_t)top_k);
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < top_k; ++j) slot[j] = Y + (int64_t)inv_row[(int64_t)t * top_k + j] * H;
        const double *ysh = with_shared ? Y + ((int64_t)off[E] + t) * H : NULL;
        combine_row(H, top_k, w + (int64_t)t * top_k, slot, ysh, out + (int64_t)t * H,
                    out_f64 ? out_f64 + (int64_t)t * H : NULL);
    }
    free(slot);
    free(Y);
}

/* ------------------------------------------------------------------------------------
 * Expert residency bank: S device slots, each holding one routed expert, and what one
 * forward does to them. The pages keep the most used routed experts of each layer
 * resident on the GPU, ranked by usage ("DeepSeek V4 Flash support -- CUDA/VRAM expert
 * tiering", summary item 1), refill that cache in place, and for a batched prefill route
 * on the device and refill a transient per-layer bank route-aware in slot-sized groups,
 * one group's uploads overlapped with the neighbouring group ("the CUDA tier wired into
 * the DeepSeek V4 engine", the engine-tier and prefill-MoE items).
 *
 * Readings (the pages give no rule beyond the above):
 *  - Cache forward, when T*top_k or E (whichever is smaller) fits in S: touched experts
 *    already resident compute in place (round 0, with the shared expert); each other
 *    touched expert, in increasing expert order, takes the slot that is empty or holds an
 *    untouched expert and is smallest by (occupied, usage of its expert, the forward that
 *    last used the slot, slot index); usage[e] counts the forwards that routed to e.
 *    Those refills form round 1.
 *  - Transient forward otherwise: with G = S/2, the touched experts in increasing order
 *    form groups of G; group r is round r and takes slots (r mod 2)*G + i, i its place in
 *    the group, so a group's refill never touches the slots the previous group computes
 *    on. An expert already in its slot is not copied; one that moves leaves its old slot
 *    empty.
 * stats: [0] forwards, [1] touched experts found in their slot, [2] experts copied.
 * Per expert e: round_of (-1 when untouched), slot_for (the slot it computes from in this
 * forward), copied (1 when its weights are copied in this forward). */
static int bank_key_less(int32_t a, int32_t b, const int32_t *expert_in, const uint32_t *usage,
                         const int32_t *last_use) {
    const int32_t oa = expert_in[a], ob = expert_in[b];
    if ((oa >= 0) != (ob >= 0)) return oa < 0;           /* empty slots first */
    if (oa >= 0) {
        if (usage[oa] != usage[ob]) return MUT(20) ? usage[oa] > usage[ob] : usage[oa] < usage[ob];
        if (last_use[a] != last_use[b]) return last_use[a] < last_use[b];
    }
    return a < b;
}

void coli_oracle_bank_plan(int32_t E, int32_t S, int32_t T, int32_t top_k, const int32_t *cnt,
                           int32_t *slot_of, int32_t *expert_in, uint32_t *usage, int32_t *last_use,
                           int64_t *stats, int32_t *round_of, int32_t *slot_for, int32_t *copied) {
    const int32_t step = (int32_t)++stats[0];
    for (int32_t e = 0; e < E; ++e) {
        round_of[e] = -1;
        slot_for[e] = -1;
        copied[e] = 0;
        if (cnt[e] > 0) usage[e]++;
    }
    const int64_t cap = (int64_t)T * top_k < E ? (int64_t)T * top_k : E;
    if (cap <= S) {
        for (int32_t e = 0; e < E; ++e) {                /* resident: compute in place */
            if (cnt[e] <= 0 || slot_of[e] < 0) continue;
            round_of[e] = 0;
            slot_for[e] = slot_of[e];
            last_use[slot_of[e]] = step;
            stats[1]++;
        }
        for (int32_t e = 0; e < E; ++e) {                /* the rest take the cheapest slots */
            if (cnt[e] <= 0 || slot_of[e] >= 0) continue;
            int32_t best = -1;
            for (int32_t s = 0; s < S; ++s) {
                const int32_t occ = expert_in[s];
                if (occ >= 0 && cnt[occ] > 0 && !MUT(19)) continue;
                if (best < 0 || bank_key_less(s, best, expert_in, usage, last_use)) best = s;
            }
            if (best < 0) return;                        /* cannot happen while cap <= S */
            if (expert_in[best] >= 0) slot_of[expert_in[best]] = -1;
            expert_in[best] = e;
            slot_of[e] = best;
            last_use[best] = step;
            round_of[e] = 1;
            slot_for[e] = best;
            copied[e] = 1;
            stats[2]++;
        }
        return;
    }
    const int32_t G = MUT(22) ? S : S / 2;
    int32_t q = 0;
    for (int32_t e = 0; e < E; ++e) {
        if (cnt[e] <= 0) continue;
        const int32_t r = q / G;
        const int32_t s = ((r % 2) * G + q % G) % S;     /* below 2G <= S: the modulus only keeps
                                                           a planted wrong G in bounds */
        ++q;
        round_of[e] = r;
        slot_for[e] = s;
        last_use[s] = step;
        if (expert_in[s] == e) {
            stats[1]++;
            continue;
        }
        if (expert_in[s] >= 0) slot_of[expert_in[s]] = -1;
        if (slot_of[e] >= 0 && !MUT(21)) expert_in[slot_of[e]] = -1;
        expert_in[s] = e;
        slot_of[e] = s;
        copied[e] = 1;
        stats[2]++;
    }
}

/* ------------------------------------------------------------------------------------
 * FP8 dense projection. The pages give the model's dense weights as FP8 E4M3 with one scale
 * per 128 x 128 block ("DeepSeek V4 Flash CPU inference with NVMe expert streaming", the
 * review question on config-driven V4 sizes), and move the five per-layer dense matmuls to
 * the GPU with numerics identical to the CPU path ("DeepSeek V4 Flash support -- CUDA/VRAM
 * expert tiering", the dense-on-GPU tier comment). E4M3 is the OCP 8-bit float: sign, four
 * exponent bits with bias 7, three mantissa bits, subnormals at exponent 0, no infinities,
 * S.1111.111 is NaN. Reading: a block scale multiplies its block's decoded values. */
double coli_oracle_e4m3(int code) {
    code &= 255;
    const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double mag;
    if (e == 0 && !MUT(24)) mag = ldexp(m / 8.0, -6);
    else mag = ldexp(1.0 + m / 8.0, e - (MUT(23) ? 8 : 7));
    return sign ? -mag : mag;
}

void coli_oracle_fp8_linear(const uint16_t *x, int32_t T, int32_t K, const uint8_t *w, const float *w_scale,
                            int32_t N, uint16_t *out, double *out_f64) {
    const int64_t kb = (K + 127) / 128, nb = (N + 127) / 128;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < (int64_t)T * N; ++i) {
        const int64_t t = i / N, n = i % N;
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            int64_t si = (n / 128) * kb + k / 128;
            if (MUT(25)) si = (k / 128) * nb + n / 128;
            if (MUT(26)) si = (n / 128) * kb;
            acc += coli_oracle_bf16(x[t * K + k]) * coli_oracle_e4m3(w[n * K + k]) * (double)w_scale[si];
        }
        out[i] = coli_oracle_round_bf16(acc);
        if (out_f64) out_f64[i] = acc;
    }
}

/* ------------------------------------------------------------------------------------
 * NVFP4 experts: E2M1 elements with an E4M3 scale per 16 elements along K and one fp32 scale
 * per matrix (NVIDIA's two-level FP4 format; the pages use MXFP4 only, so this is the format
 * variant of the same layer). Element value = e2m1(code) * e4m3(scale byte) * global. */
double coli_oracle_nvfp4(const uint8_t *codes, const uint8_t *scales, float global, int64_t K, int64_t row,
                         int64_t k) {
    const uint8_t byte = codes[row * (K / 2) + k / 2];
    const int code = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
    const int64_t si = MUT(27) ? row * (K / 16) + k / 32 : row * (K / 16) + k / 16;
    return E2M1_TABLE[code] * coli_oracle_e4m3(scales[si]) * (MUT(28) ? 1.0 : (double)global);
}

static void expert_row_nv(const uint16_t *x_row, int32_t H, int32_t I, const uint8_t *gu_codes,
                          const uint8_t *gu_scales, float gu_global, const uint8_t *d_codes,
                          const uint8_t *d_scales, float d_global, double *y) {
    double *xv = (double *)malloc(sizeof(double) * (size_t)H);
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    for (int32_t k = 0; k < H; ++k) xv[k] = coli_oracle_bf16(x_row[k]);
    for (int32_t i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int32_t k = 0; k < H; ++k) {
            g += coli_oracle_nvfp4(gu_codes, gu_scales, gu_global, H, i, k) * xv[k];
            u += coli_oracle_nvfp4(gu_codes, gu_scales, gu_global, H, (int64_t)I + i, k) * xv[k];
        }
        h[i] = g / (1.0 + exp(-g)) * u;
    }
    for (int32_t m = 0; m < H; ++m) {
        double acc = 0.0;
        for (int32_t i = 0; i < I; ++i) acc += coli_oracle_nvfp4(d_codes, d_scales, d_global, I, m, i) * h[i];
        y[m] = acc;
    }
    free(h);
    free(xv);
}

void coli_oracle_tokens_output_nv(const uint16_t *x, int32_t H, int32_t I, int32_t I_s,
                                  const int32_t *idx, const float *w, int32_t top_k,
                                  const uint8_t *gu_codes, const uint8_t *gu_scales, const float *gu_global,
                                  const uint8_t *d_codes, const uint8_t *d_scales, const float *d_global,
                                  const uint8_t *sh_gu_codes, const uint8_t *sh_gu_scales, float sh_gu_global,
                                  const uint8_t *sh_d_codes, const uint8_t *sh_d_scales, float sh_d_global,
                                  const int32_t *tokens, int32_t n_tokens, uint16_t *out, double *out_f64) {
    const int64_t gu_c = 2LL * I * (H / 2), gu_s = 2LL * I * (H / (MUT(29) ? 32 : 16));
    const int64_t d_c = (int64_t)H * (I / 2), d_s = (int64_t)H * (I / 16);
    const int with_shared = sh_gu_codes != NULL && I_s > 0 && !MUT(31);
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t n = 0; n < n_tokens; ++n) {
        int32_t t = tokens[n];
        const uint16_t *xr = x + (int64_t)t * H;
        double *ys = (double *)malloc(sizeof(double) * (size_t)H * (size_t)(top_k + 1));
        const double **slot = (const double **)malloc(sizeof(double *) * (size_t)top_k);
        for (int32_t j = 0; j < top_k; ++j) {
            int64_t e = idx[(int64_t)t * top_k + j];
            double *yj = ys + (int64_t)j * H;
            expert_row_nv(xr, H, I, off_ptr(gu_codes, e, gu_c), off_ptr(gu_scales, e, gu_s),
                          gu_global[MUT(30) ? 0 : e],
                          off_ptr(d_codes, e, d_c), off_ptr(d_scales, e, d_s), d_global[e], yj);
            slot[j] = yj;
        }
        double *ysh = NULL;
        if (with_shared) {
            ysh = ys + (int64_t)top_k * H;
            expert_row_nv(xr, H, I_s, sh_gu_codes, sh_gu_scales, sh_gu_global, sh_d_codes, sh_d_scales,
                          sh_d_global, ysh);
        }
        combine_row(H, top_k, w + (int64_t)t * top_k, slot, ysh, out + (int64_t)n * H,
                    out_f64 ? out_f64 + (int64_t)n * H : NULL);
        free(slot);
        free(ys);
    }
}
