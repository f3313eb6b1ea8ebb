/*
 * colimoe_oracle.h -- plain, slow CPU oracle of the routed MXFP4 MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark may load this code; the library never links it and shares no code,
 * header, table or constant with it.
 *
 * Sources (pages of the colibri project):
 *  - "DeepSeek V4 Flash CPU inference with NVMe expert streaming": experts are FP4 E2M1
 *    with UE8M0 scales per group of 32 (the review reply on config-driven V4 sizes);
 *    doubled E2M1 values are integers (the AVX2 kernel-series comment); the 16-entry
 *    E2M1 table is 64 bytes as fp32 (the GB10 NEON rows16 note); hidden 4096 x moe_inter
 *    2048 shapes (GB10 kernel bench table).
 *  - "DeepSeek V4: the CUDA kernels, as a tier rather than an engine": the UE8M0 scale is
 *    built as an fp32 bit pattern, s=0 -> +0 and s=255 -> +inf (the #819 MXFP4 decode note).
 *  - "the CUDA tier wired into the DeepSeek V4 engine": route on device, expert-grouped
 *    GEMM rows, fused routed+shared MoE ("What it is" list).
 *  The layer's arithmetic (fp32 logits, sigmoid scores, bias-adjusted top-k with ties to
 *  the lower index, weights renormalised to sum 1, SwiGLU, shared-expert add) is the
 *  plain definition of a DeepSeek-V4-style routed MoE layer; the pages leave it open.
 *
 * Layouts (row-major, K-major weight rows):
 *  x         bf16 bits [T][H]
 *  router_w  fp32 [E][H];  router_b fp32 [E] or NULL (zero bias)
 *  gate_up   codes [E][2I][H/2], scales [E][2I][H/32] (gate rows 0..I-1, up rows I..2I-1)
 *  down      codes [E][H][I/2],  scales [E][H][I/32]
 *  element k of a row sits in byte k/2: the low nibble for even k, the high nibble for odd k.
 */
#ifndef COLIMOE_ORACLE_H
#define COLIMOE_ORACLE_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

/* --- formats --- */
double coli_oracle_e2m1(int code);          /* value of a 4-bit E2M1 code */
double coli_oracle_e8m0(int s);             /* value of a UE8M0 scale byte */
double coli_oracle_mxfp4(const uint8_t *codes, const uint8_t *scales, int64_t K,
                         int64_t row, int64_t k);   /* one decoded weight */
double coli_oracle_bf16(uint16_t bits);     /* bf16 bits -> value */
uint16_t coli_oracle_round_bf16(double v);  /* round to nearest even bf16 */

/* --- router --- */
/* logits[t][e] = sum_h x[t][h] * Wr[e][h] in fp64 (exact products). */
void coli_oracle_router_logits(const uint16_t *x, int32_t T, int32_t H, const float *router_w,
                               int32_t E, double *logits);
/* s = sigmoid(z) in fp64, returned rounded to fp32. */
void coli_oracle_sigmoid(const double *logits, int64_t n, float *s);
/* Given fp32 scores s[T][E]: key = fp32(s + b); pick the top_k largest keys (ties -> lower
 * expert index) in descending key order; w_j = s_j / S with S the fp32 sum of the chosen
 * s in slot order and an IEEE fp32 division. */
void coli_oracle_route(const float *s, const float *router_b, int32_t T, int32_t E, int32_t top_k,
                       int32_t *idx, float *w);

/* --- permute --- */
/* cnt[E+1] (cnt[E] = T when with_shared, else 0), off[E+2] exclusive prefix of cnt,
 * src_token[T*k + T] (shared rows are tokens in order), inv_row[T][k].
 * Routed row of (t, j) with e = idx[t][j]: off[e] + #{t' < t : e in idx[t']}. */
void coli_oracle_permute(const int32_t *idx, int32_t T, int32_t E, int32_t top_k, int32_t with_shared,
                         int32_t *cnt, int32_t *off, int32_t *src_token, int32_t *inv_row);

/* --- expert FFN --- */
/* One expert on one activation row: g = Wg x, u = Wu x, h = silu(g)*u, y = Wd h, all fp64.
 * The weights point at that expert's arrays. h_out may be NULL. */
void coli_oracle_expert_row(const uint16_t *x_row, int32_t H, int32_t I,
                            const uint8_t *gu_codes, const uint8_t *gu_scales,
                            const uint8_t *d_codes, const uint8_t *d_scales,
                            double *y, double *h_out);

/* out[t] = round_bf16(y_shared(x_t) + sum_j w[t][j] * y_{idx[t][j]}(x_t)) for the listed tokens.
 * shared_* may be NULL (no shared expert). out_f64 (may be NULL) receives the unrounded sums.
 * Rows are written at out[i] for token tokens[i]. Uses OpenMP over tokens when built with it. */
void coli_oracle_tokens_output(const uint16_t *x, int32_t H, int32_t I, int32_t I_s,
                               const int32_t *idx, const float *w, int32_t top_k,
                               const uint8_t *gu_codes, const uint8_t *gu_scales,
                               const uint8_t *d_codes, const uint8_t *d_scales,
                               const uint8_t *sh_gu_codes, const uint8_t *sh_gu_scales,
                               const uint8_t *sh_d_codes, const uint8_t *sh_d_scales,
                               const int32_t *tokens, int32_t n_tokens,
                               uint16_t *out, double *out_f64);

/* Whole layer through the permuted path: router, route, permute, per-row expert FFN over the
 * expert-grouped rows, combine. Every buffer is caller-owned. */
void coli_oracle_moe_forward(const uint16_t *x, int32_t T, int32_t H, int32_t E, int32_t I, int32_t I_s,
                             const float *router_w, const float *router_b, int32_t top_k,
                             const uint8_t *gu_codes, const uint8_t *gu_scales,
                             const uint8_t *d_codes, const uint8_t *d_scales,
                             const uint8_t *sh_gu_codes, const uint8_t *sh_gu_scales,
                             const uint8_t *sh_d_codes, const uint8_t *sh_d_scales,
                             float *s, int32_t *idx, float *w,
                             int32_t *cnt, int32_t *off, int32_t *src_token, int32_t *inv_row,
                             uint16_t *out, double *out_f64);

int32_t coli_oracle_threads(void);   /* threads an OpenMP region uses (1 without OpenMP) */
int32_t coli_oracle_mutant(void);    /* planted-mistake id this build carries (0 = none) */

/* --- expert residency bank --- */
/* One forward's effect on a bank of S device slots (2 <= S <= E) for the touched set
 * {e : cnt[e] > 0}. State (in/out): slot_of[E] (-1: not resident), expert_in[S] (-1: empty),
 * usage[E], last_use[S], stats[3] = {forwards, found in place, copied}. Out per expert:
 * round_of, slot_for, copied. See the definition for the policy and its readings. */
void coli_oracle_bank_plan(int32_t E, int32_t S, int32_t T, int32_t top_k, const int32_t *cnt,
                           int32_t *slot_of, int32_t *expert_in, uint32_t *usage, int32_t *last_use,
                           int64_t *stats, int32_t *round_of, int32_t *slot_for, int32_t *copied);

/* --- FP8 dense projection --- */
double coli_oracle_e4m3(int code);          /* value of an OCP E4M3 byte (NaN for S.1111.111) */
/* out[t][n] = round_bf16(sum_k x[t][k] * e4m3(w[n][k]) * w_scale[n/128][k/128]) in fp64.
 * x bf16 bits [T][K]; w E4M3 codes [N][K]; w_scale fp32 [ceil(N/128)][ceil(K/128)];
 * out_f64 (may be NULL) receives the unrounded sums. OpenMP over outputs when built with it. */
void coli_oracle_fp8_linear(const uint16_t *x, int32_t T, int32_t K, const uint8_t *w, const float *w_scale,
                            int32_t N, uint16_t *out, double *out_f64);

/* --- NVFP4 experts (format variant) --- */
/* One weight of an NVFP4 matrix: e2m1(code) * e4m3(scale of its group of 16 along K) * global;
 * codes [R][K/2] (low nibble = even k), scales [R][K/16] E4M3 bytes. */
double coli_oracle_nvfp4(const uint8_t *codes, const uint8_t *scales, float global, int64_t K, int64_t row,
                         int64_t k);
/* coli_oracle_tokens_output with NVFP4 experts: scales [E][rows][K/16], one fp32 global per
 * expert and matrix (gate/up, down); the shared expert's globals as scalars. */
void coli_oracle_tokens_output_nv(const uint16_t *x, int32_t H, int32_t I, int32_t I_s,
                                  const int32_t *idx, const float *w, int32_t top_k,
                                  const uint8_t *gu_codes, const uint8_t *gu_scales, const float *gu_global,
                                  const uint8_t *d_codes, const uint8_t *d_scales, const float *d_global,
                                  const uint8_t *sh_gu_codes, const uint8_t *sh_gu_scales, float sh_gu_global,
                                  const uint8_t *sh_d_codes, const uint8_t *sh_d_scales, float sh_d_global,
                                  const int32_t *tokens, int32_t n_tokens, uint16_t *out, double *out_f64);

#ifdef __cplusplus
}
#endif
#endif
