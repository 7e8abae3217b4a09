/* CPU oracle of one int4 routed-expert MoE layer (colibrì-style), TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, single-purpose C.  Only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it; the product library never links it and shares no code with
 * it.  Each function cites the passage of the source pages it follows:
 *   [P1] "colibrì 架构概述" (blog.chen3feng.top, colibri-analysis/01): §3.1 quantisation,
 *        §4 kernel layer, §5 token lifecycle (moe step), §6 design decisions.
 *   [P2] colibrì README.zh-TW (git.wopr.ltd): "絕不為同一次硬碟讀取等待兩遍" (batch union,
 *        three matrices stored adjacently), "如實呈現推測式解碼" (draft and verify compute
 *        the same function).
 *   [P3] "colibrì: движок GLM-5.2 …" (ai4coding.ru): "Что реализовано" (DeepSeek-V3 sigmoid
 *        router, shared expert, Q8_0-style int8 activations for the integer dot kernels).
 *
 * Precision.  Every quantity that decides an integer (activation q8 codes, router top-k,
 * the SwiGLU output h that is re-quantised to int8) is computed in fp32 following one
 * canonical order of operations (the "canonical arithmetic" below), which the CUDA path
 * follows too, so those integers can be compared bit for bit.  Final outputs are also
 * evaluated in fp64 from the same integer codes (orc_moe_forward's y64) and the fp32 result
 * is judged against that.
 *
 * Canonical arithmetic (fp32, every operation rounded to nearest even, no contraction):
 *   pairwise32(p[0..31])  = pairwise tree over adjacent pairs: level 1 sums (p0+p1),(p2+p3)…,
 *                           level 2 sums adjacent level-1 results, …, five levels.
 *   canon_dot(a,b,n)      = 32 contiguous groups of G = ceil(n/32) elements; p_g is an fma
 *                           chain p = fma(a_j, b_j, p) over ascending j from +0; empty groups
 *                           are +0; result pairwise32(p).
 *   canon_blocksum(d,A,nb)= the same with 32 contiguous groups of G = ceil(nb/32) blocks and
 *                           p = fma(d_b, (float)A_b, p).
 *   exp                   = own fp32 exp (orc_exp), identical operations on both sides.
 *
 * Parity pins: every function here is checked in tests/test_oracle_pins.py against facts that
 * do not come from this file (closed forms, brute-force integer sums, a full stable sort, fp64
 * evaluations within derived error bounds, a forced all-experts dense loop, identical-expert
 * and batch-invariance identities, and the pages' ≈0.3% IDOT accuracy figure).  The fp32
 * end-to-end value of a full layer has no printed worked example on the pages: beyond those
 * invariants it is "parity unpinned" by a page value.
 */
#ifndef COLI_ORACLE_H
#define COLI_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int d, f, n_experts, top_k, n_shared, qblock;
  float routed_scale, rms_eps;
  int has_norm;
  int wbits; /* expert code width: 4 (int4 records), 8 or 2 (orc_expert_ffn_bits's layout) */
} orc_cfg;

/* optional intermediates; any NULL entry is skipped.  P = T*K + n_shared*T pairs. */
typedef struct {
  float* xn;          /* [T,d]  layer input after RMSNorm (copy of x without norm) */
  int8_t* qx;         /* [T,d]  activation q8 codes                                 */
  float* dx;          /* [T,d/32] activation block scales                           */
  float* logits;      /* [T,E]                                                       */
  float* scores;      /* [T,E]  sigmoid(logits)                                      */
  int32_t* ids;       /* [T,K]  selected experts, rank order                         */
  float* w;           /* [T,K]  renormalised routing weights                         */
  int32_t* n_union;   /* [1]    number of union slots (routed distinct + shared)     */
  int32_t* union_ids; /* [<=E+1] expert id per union slot (shared = E, last)          */
  int32_t* offsets;   /* [n_union+1] pair ranges per union slot                       */
  int32_t* pair_token;/* [P]                                                          */
  int32_t* pair_rank; /* [P]    k of the pair, -1 for the shared expert               */
  int32_t* inv;       /* [T,K]  pair index of (t, ids[t,k])                           */
  float* g;           /* [P,f]                                                        */
  float* u;           /* [P,f]                                                        */
  float* h;           /* [P,f]  SiLU(g)*u                                             */
  int8_t* qh;         /* [P,f]  h q8 codes                                            */
  float* dh;          /* [P,f/32]                                                     */
  float* e;           /* [P,d]  expert outputs (fp32)                                 */
  int32_t* Ag;        /* [P,f,d/32] per-block int32 dots, gate                        */
  int32_t* Au;        /* [P,f,d/32] up                                                */
  int32_t* Ad;        /* [P,d,f/32] down                                              */
} orc_dump;

/* ---- formats (P1 §3.1: int4 packed, two 4-bit values per byte, one f32 scale per row) ---- */
void orc_quantize_i4_rows(const float* w, int64_t rows, int cols, uint8_t* packed, float* scales);
int orc_i4_get(const uint8_t* row, int j);
void orc_pack_i4_row(const int8_t* q, int cols, uint8_t* packed_row);

/* ---- activation int8 blocks (P1 §3.1 IDOT; P3 "Что реализовано", Q8_0-style) ---- */
void orc_quantize_q8(const float* x, int64_t n, int8_t* q, float* d);

/* ---- canonical fp32 arithmetic ---- */
float orc_exp(float x);
void orc_exp_n(const float* x, float* y, int64_t n);
float orc_sigmoid(float x);
float orc_silu_mul(float g, float u);
float orc_pairwise32(const float* p);
float orc_canon_dot(const float* a, const float* b, int n);
float orc_canon_blocksum(const float* d, const int32_t* A, int nb);

/* ---- integer dot of one 32-element block (P1 §4 dot_i4i8) ---- */
int32_t orc_block_dot(const uint8_t* wrow, const int8_t* qx, int b);

/* int8 rows (P1 §3.1 "int8", quantize_rows / dot_i8i8): one f32 scale per row, s = max|w|/127,
 * codes round(w/s) half away from zero in [-127, 127]; block dots exact in int32; the matvec
 * applies the same canonical fp32 epilogue as the int4 one. */
void orc_quantize_i8_rows(const float* w, int64_t rows, int cols, int8_t* q, float* scales);
int32_t orc_i8_block_dot(const int8_t* wrow, const int8_t* qx, int b);
void orc_i8_matvec(const int8_t* W, const float* s, int rows, int cols, const int8_t* qx,
                   const float* dx, float* out, int32_t* A);

/* int2 rows (P1 §3.1 "int2 packed", pack_int2 / matmul_i2): four 2-bit two's-complement codes
 * per byte, element 4i+k in bits 2k..2k+1 of byte i; one f32 scale per row, s = max|w|,
 * codes round(w/s) half away from zero in [-1, 1] (-2 decodes but is never written); block
 * dots with int8 activation codes exact in int32; the matvec's fp32 epilogue is the int4 one. */
int orc_i2_get(const uint8_t* row, int j);
void orc_pack_i2_row(const int8_t* q, int cols, uint8_t* packed_row);
void orc_quantize_i2_rows(const float* w, int64_t rows, int cols, uint8_t* packed, float* scales);
int32_t orc_i2_block_dot(const uint8_t* wrow, const int8_t* qx, int b);
void orc_i2_matvec(const uint8_t* W, const float* s, int rows, int cols, const int8_t* qx,
                   const float* dx, float* out, int32_t* A);

/* ---- int4 x int8 matrix-vector product with dequant-on-use (P1 §3.1, matmul_i4 + IDOT) ---- */
void orc_i4_matvec(const uint8_t* W, const float* s, int rows, int cols, const int8_t* qx,
                   const float* dx, float* out, int32_t* A);

/* ---- router (P1 §5, the moe step: sigmoid routing picks the top 8; P3 DeepSeek-V3-style) ---- */
void orc_topk(const float* sel, int E, int K, int32_t* ids);
void orc_route_token(const float* Wr, const float* bias, const float* x, int E, int d, int K,
                     float routed_scale, float* logits, float* scores, int32_t* ids, float* w);

/* ---- RMSNorm (P1 §4 kernel layer "rmsnorm") ---- */
void orc_rmsnorm(const float* x, const float* gamma, int d, float eps, float* out);

/* ---- batch union (P2: each distinct expert is read once per batch) ---- */
int orc_union_bucket(const int32_t* ids, int T, int K, int E, int n_shared, int32_t* union_ids,
                     int32_t* offsets, int32_t* pair_token, int32_t* pair_rank, int32_t* inv);

/* ---- one routed or shared expert on one token: gate/up, SiLU, re-quantise, down (P1 §5) ----
 * rec: [gate f*d/2 | up f*d/2 | down d*f/2] bytes; sc: [s_g f | s_u f | s_d d]. */
void orc_expert_ffn(const uint8_t* rec, const float* sc, int d, int f, const int8_t* qx,
                    const float* dx, int8_t* qh, float* dh, float* e, float* g_out,
                    float* u_out, float* h_out, int32_t* Ag, int32_t* Au, int32_t* Ad);
/* one expert with int8 (bits 8), int4 (4) or int2 (2) rows: the int4 record layout at bits/8
 * bytes per weight, the same steps as orc_expert_ffn (g_out, u_out, h_out may be NULL).
 * Returns -1 for another width. */
int orc_expert_ffn_bits(int bits, const uint8_t* rec, const float* sc, int d, int f,
                        const int8_t* qx, const float* dx, int8_t* qh, float* dh, float* e,
                        float* g_out, float* u_out, float* h_out);

/* ---- full layer ----
 * rec[id], sc[id] for id in 0..E (E = shared); entries of experts nobody selects may be NULL.
 * y: fp32 canonical result.  y64 (optional): fp64 evaluation from the same integer codes.
 * Returns 0, or -1 if a selected expert's weights are missing / arguments are invalid. */
int orc_moe_forward(const orc_cfg* cfg, const float* x, int T, const float* Wr, const float* bias,
                    const float* gamma, const uint8_t* const* rec, const float* const* sc, float* y,
                    double* y64, const orc_dump* dump);

/* fp64 dequant-on-use reference with unquantised activations (the comparator for the
 * pages' "≈0.3% RMS error" of the integer-dot path, P1 §3.1 and §6).  Routing (ids, w) is
 * taken as given so both paths combine the same experts. */
int orc_moe_dequant64(const orc_cfg* cfg, const float* xn, int T, const int32_t* ids,
                      const float* w, const uint8_t* const* rec, const float* const* sc,
                      const float* x_resid, double* y);

int orc_num_threads(void);
void orc_set_num_threads(int n); /* threads of the parallel loops; results do not depend on it */

#ifdef __cplusplus
}
#endif
#endif
