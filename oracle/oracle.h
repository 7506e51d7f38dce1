/*
 * oracle.h -- plain CPU oracle for the streamed NF4-LoRA hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, imports or
 * calls this code; it exists so the tests, the smoke check and the bench's
 * CPU-baseline leg can check the CUDA path against an independent, slow,
 * obviously correct implementation.  It shares no code, header, table or
 * constant generator with the CUDA library.
 *
 * Method (Poros, "Blockwise residency for frozen-base QLoRA"):
 *   - frozen NF4 base weight W, 4-bit NormalFloat codes with one fp32 absmax
 *     per 64 consecutive weights of a row (Poros docs, "Limitations" page,
 *     section "What 0.00e+00 means": NF4 is the only bitwise precision);
 *   - each linear computes y = x W'^T + (alpha/r) B A dropout(x)
 *     (research page, "Poros": the backward "propagates gradients only to
 *     the adapters and block inputs");
 *   - the backward recomputes each block's forward with the same dropout
 *     masks (research page, paragraph "RNG state capture"); here the masks
 *     come from a counter-based Philox4x32-10 keyed by (seed, step, layer,
 *     linear, micro-batch), so a recompute regenerates them exactly.
 *
 * Floating point: every sum and product is done in double; values are
 * rounded to bf16 only where the method stores a bf16 tensor (x, y, dY,
 * dequantised weights, the normalised / activation inputs of the linears).
 *
 * Layouts (row-major unless stated):
 *   W       bf16 bits  [N, K]
 *   codes   uint8      [N, K/2]; byte j of row n holds k = 2j in the high
 *                      nibble and k = 2j+1 in the low nibble
 *   absmax  float      [K/64, N]   (block-major: absmax[kb*N + n])
 *   mask    uint32     [M, K/32];  bit (k & 31) of word (m*K + k)/32 is 1
 *                      when element (m, k) is kept
 *   A       float      [r, K];  B float [N, r]
 */
#ifndef WS_ORACLE_H
#define WS_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The 16 NormalFloat levels as fp32 literals, ascending. */
extern const float orc_nf4_levels[16];

/* bf16 helpers (round-to-nearest-even, NaN not produced by the oracle). */
uint16_t orc_f32_to_bf16(float f);
double   orc_bf16_to_f64(uint16_t b);
/* Round a double to bf16 the way a double->float->bf16 chain would not:
 * a single rounding of the exact double value to the nearest bf16. */
uint16_t orc_f64_to_bf16(double d);

/* ---- NF4 codec --------------------------------------------------------- */
/* K % 64 == 0.  absmax_b = max |w| over the 64-block (fp32);
 * v = w / absmax (IEEE fp32 division); code = #{i : v > mid_i} with
 * mid_i = fp32(fp32(c_i + c_{i+1}) * 0.5).  A zero block gives code 7. */
void orc_quantize_nf4(const uint16_t* W, int64_t N, int64_t K,
                      uint8_t* codes, float* absmax);
/* w' = bf16_RN( fp32(c[code]) * fp32(absmax) ), one rounding. */
void orc_dequant_nf4(const uint8_t* codes, const float* absmax,
                     int64_t N, int64_t K, uint16_t* Wq);

/* ---- Philox4x32-10 (Salmon et al., SC'11) ------------------------------ */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2],
                       uint32_t out[4]);
/* keep threshold T = ceil(p * 2^32); keep <=> word >= T. */
uint64_t orc_keep_threshold(double p);
/* Dropout mask of one linear's LoRA input [M, K] (K % 32 == 0).
 * key = (seed_lo, seed_hi); counter = (e >> 2, linear | microbatch << 8,
 * layer, step); word (e & 3) decides element e = m*K + k. */
void orc_dropout_mask(uint64_t seed, uint32_t step, uint32_t layer,
                      uint32_t linear, uint32_t microbatch, double p,
                      int64_t M, int64_t K, uint32_t* bits);

/* ---- LoRA linear -------------------------------------------------------- */
/* scale = (alpha / r) / (1 - p).  Rows: the oracle may evaluate a subset of
 * output rows (rows != NULL, nrows entries) so full-size checks stay cheap.
 * y[nrows, N] and U[nrows, r] are unrounded doubles. */
void orc_lora_fwd_rows(int64_t M, int64_t N, int64_t K, int r,
                       const uint16_t* x, const uint16_t* Wq,
                       const float* A, const float* B, const uint32_t* mask,
                       double scale, const int64_t* rows, int64_t nrows,
                       double* y, double* U);
/* Full backward.  G = dY B; dX = dY W' + scale (G A) (.) m;
 * dA = scale G^T (m (.) x); dB = scale dY^T ((m (.) x) A^T).
 * dX may be NULL (skipped); dX rows subset as in the forward. */
void orc_lora_bwd(int64_t M, int64_t N, int64_t K, int r,
                  const uint16_t* x, const uint16_t* Wq,
                  const float* A, const float* B, const uint32_t* mask,
                  const uint16_t* dY, double scale,
                  const int64_t* rows, int64_t nrows,
                  double* dX, double* dA, double* dB);

/* ---- Causal attention core with grouped kv heads (scaled dot-product
 * attention; query head h reads kv head h / (nh / nkv)).  n_seq sequences of
 * S tokens, token t = b*S + i; q, o [M, nh*d]; k, v [M, nkv*d]; M = n_seq*S.
 *   o_i = sum_{j<=i} p_ij v_j,  p_ij = exp(q_i.k_j / sqrt(d) - lse_i),
 *   lse_i = log sum_{j<=i} exp(q_i.k_j / sqrt(d))   (lse [nh, M], may be NULL).
 * The backward overwrites dq, dk, dv with the gradients for upstream dO. */
void orc_attention_fwd(int64_t n_seq, int64_t S, int64_t nh, int64_t nkv, int64_t d,
                       const double* q, const double* k, const double* v, double* o,
                       double* lse);
void orc_attention_bwd(int64_t n_seq, int64_t S, int64_t nh, int64_t nkv, int64_t d,
                       const double* q, const double* k, const double* v, const double* dO,
                       double* dq, double* dk, double* dv);

/* ---- Synthetic stack (RMSNorm -> q,k,v -> repeat(v) or attention -> o -> residual;
 *      RMSNorm -> gate,up -> SiLU(gate)*up -> down -> residual) ---------- */
typedef struct {
  int64_t M, H, KV, I, head_dim;
  int n_layers;
  int r;
  double alpha, p, eps;
  uint64_t seed;
  int round_bf16;   /* 1: round to bf16 at the stored-bf16 points; 0: exact */
  int attn;         /* 0: repeat(v) in place of attention; 1: causal attention core */
} orc_stack_cfg;

/* Linear ids inside a layer. */
enum { ORC_Q = 0, ORC_K = 1, ORC_V = 2, ORC_O = 3, ORC_GATE = 4, ORC_UP = 5,
       ORC_DOWN = 6, ORC_NLIN = 7 };

/* Per-linear parameters, indexed [layer * 7 + linear]. */
typedef struct {
  const uint16_t* const* Wq;  /* dequantised base weights, bf16 bits [N,K] */
  const float* const* A;      /* [r, K] */
  const float* const* B;      /* [N, r] */
} orc_stack_params;

/* One forward + backward of the whole stack from h0 [M, H].
 * loss: 0.5 * mean(h_L^2).  dA/dB: double arrays per linear (caller-owned,
 * same indexing as params; may be NULL to skip the backward).
 * h_out (optional, [M,H]) receives the final residual stream. */
void orc_stack_fwd_bwd(const orc_stack_cfg* cfg, uint32_t step,
                       const orc_stack_params* prm, const double* h0,
                       double* loss, double* h_out,
                       double* const* dA, double* const* dB);
/* The same for micro-batch `microbatch` of a step with gradient
 * accumulation over n_micro micro-batches: the dropout keys carry the
 * micro-batch index, and the step loss is the mean over the micro-batches,
 * so this call returns its share 0.5 mean(h_L^2) / n_micro and the
 * gradients of that share (the step's gradient is the sum over the
 * micro-batches). */
void orc_stack_fwd_bwd_mb(const orc_stack_cfg* cfg, uint32_t step, uint32_t microbatch,
                          int n_micro, const orc_stack_params* prm, const double* h0,
                          double* loss, double* h_out,
                          double* const* dA, double* const* dB);

/* The stack's pointwise / row pieces on their own (x in double):
 * RMSNorm with unit gain -> bf16 bits, rstd per row;
 * act = bf16(SiLU(g) * u) for bf16 g, u;
 * repeat of kv heads: vr[m, hh*hd + d] = v[m, (hh / (H/KV))*hd + d]. */
void orc_rmsnorm_bf16(int64_t M, int64_t H, double eps, const double* x, uint16_t* y,
                      double* rstd);
void orc_silu_mul_bf16(int64_t n, const uint16_t* g, const uint16_t* u, uint16_t* act);
void orc_repeat_kv(int64_t M, int64_t H, int64_t KV, int64_t head_dim, const uint16_t* v,
                   uint16_t* vr);
/* The same pieces as the stack computes them, in double; round_bf16 != 0
 * rounds each output to bf16 where the stack stores bf16 (the normalised
 * row; the SwiGLU input gradients dg, du; the repeat's input gradient dv).
 *   SwiGLU:    act = g sigmoid(g) u (unrounded);
 *   RMSNorm:   y = x rstd, rstd = 1 / sqrt(mean(x^2) + eps) per row;
 *   its backward ADDS rstd dy - rstd^3 x (dy . x) / H to dx;
 *   SwiGLU backward: du = d g sigmoid(g), dg = d u sigmoid(g)(1 + g(1 - sigmoid(g)));
 *   repeat backward: dv[m, kh*hd + d] = sum_t dvr[m, (kh*rep + t)*hd + d]. */
void orc_silu_mul_f64(int64_t n, const double* g, const double* u, double* act);
void orc_rmsnorm_f64(int64_t M, int64_t H, double eps, int round_bf16, const double* x,
                     double* y, double* rstd);
void orc_rmsnorm_bwd_add(int64_t M, int64_t H, const double* x, const double* rstd,
                         const double* dy, double* dx);
void orc_silu_mul_bwd(int64_t n, int round_bf16, const double* dact, const double* g,
                      const double* u, double* dg, double* du);
void orc_repeat_kv_bwd(int64_t M, int64_t H, int64_t KV, int64_t head_dim, int round_bf16,
                       const double* dvr, double* dv);

/* PyTorch-default Adam (betas 0.9/0.999, eps 1e-8, no weight decay,
 * bias-corrected), one step t >= 1, in double. */
void orc_adam_step(int64_t n, double* p, const double* g, double* m,
                   double* v, int64_t t, double lr, double beta1,
                   double beta2, double eps);

/* Threads the oracle uses (OpenMP), for reporting. */
int orc_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
