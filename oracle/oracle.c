/*
 * oracle.c -- plain CPU oracle for the streamed NF4-LoRA hot path.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).  Slow on purpose: straight loops
 * over the definitions, double accumulation, no blocking or reordering
 * beyond what the definitions state.  Build with -ffp-contract=off so the
 * fp32 steps of the NF4 codec are plain IEEE operations on any host.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* The 16-level NormalFloat (NF4) table of QLoRA, as the decimal values it is
 * published with, read as fp32 literals (Poros docs, "Limitations" page:
 * NF4 is the bitwise-gated precision; the levels themselves are the NF4
 * data type of Dettmers et al., "QLoRA", 2023, section 3). */
const float orc_nf4_levels[16] = {
    -1.0f,    -0.6962f, -0.5251f, -0.3949f, -0.2844f, -0.1848f,
    -0.0911f, 0.0f,     0.0796f,  0.1609f,  0.2461f,  0.3379f,
    0.4407f,  0.5626f,  0.7230f,  1.0f};

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---- bf16 ---------------------------------------------------------------- */
static uint32_t f32_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}
static float bits_f32(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

uint16_t orc_f32_to_bf16(float f) {
  uint32_t u = f32_bits(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0; /* NaN */
  /* round to nearest, ties to even, on the 16 dropped bits */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

double orc_bf16_to_f64(uint16_t b) { return (double)bits_f32((uint32_t)b << 16); }

uint16_t orc_f64_to_bf16(double d) {
  if (d == 0.0) return signbit(d) ? 0x8000 : 0x0000;
  double a = fabs(d);
  int e;
  double q;
  if (a < 1.1754943508222875e-38) {
    /* bf16 subnormal range: a fixed quantum of 2^-133 */
    q = nearbyint(ldexp(a, 133));        /* one rounding, RNE          */
    e = -133;
  } else {
    double m = frexp(a, &e);             /* a = m * 2^e, m in [0.5, 1) */
    q = nearbyint(ldexp(m, 8));          /* 8 significant bits, RNE    */
    e -= 8;
  }
  double r = ldexp(q, e);                /* exactly representable      */
  float rf = (float)r;                   /* exact (or inf past the top) */
  uint16_t b = (uint16_t)(f32_bits(rf) >> 16);
  return d < 0 ? (uint16_t)(b | 0x8000) : b;
}

static double bf(uint16_t b) { return orc_bf16_to_f64(b); }

/* ---- NF4 codec ----------------------------------------------------------- */
void orc_quantize_nf4(const uint16_t* W, int64_t N, int64_t K, uint8_t* codes,
                      float* absmax) {
  float mid[15];
  for (int i = 0; i < 15; ++i) {
    volatile float s = orc_nf4_levels[i] + orc_nf4_levels[i + 1];
    mid[i] = s * 0.5f;
  }
  const int64_t nkb = K / 64;
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t kb = 0; kb < nkb; ++kb) {
      const uint16_t* w = W + n * K + kb * 64;
      float amax = 0.0f;
      for (int i = 0; i < 64; ++i) {
        float a = fabsf(bits_f32((uint32_t)w[i] << 16));
        if (a > amax) amax = a;
      }
      absmax[kb * N + n] = amax;
      uint8_t c[64];
      for (int i = 0; i < 64; ++i) {
        if (amax == 0.0f) {
          c[i] = 7;
          continue;
        }
        volatile float v = bits_f32((uint32_t)w[i] << 16) / amax;
        int code = 0;
        for (int j = 0; j < 15; ++j)
          if (v > mid[j]) ++code;
        c[i] = (uint8_t)code;
      }
      uint8_t* dst = codes + n * (K / 2) + kb * 32;
      for (int j = 0; j < 32; ++j)
        dst[j] = (uint8_t)((c[2 * j] << 4) | c[2 * j + 1]);
    }
  }
}

void orc_dequant_nf4(const uint8_t* codes, const float* absmax, int64_t N,
                     int64_t K, uint16_t* Wq) {
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t k = 0; k < K; ++k) {
      uint8_t byte = codes[n * (K / 2) + k / 2];
      int code = (k & 1) ? (byte & 15) : (byte >> 4);
      float a = absmax[(k / 64) * N + n];
      volatile float prod = orc_nf4_levels[code] * a;
      Wq[n * K + k] = orc_f32_to_bf16(prod);
    }
  }
}

/* ---- Philox4x32-10 ------------------------------------------------------- */
/* Round function and key schedule of Philox4x32 (Salmon, Moraes, Dror,
 * Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11, section 4.2):
 * two 32x32->64 multiplies per round by the multipliers below, the high
 * halves xored with the other counter words and the key, and the key bumped
 * by the Weyl constants (golden ratio, sqrt(3)-1) between rounds. */
#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2],
                       uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += PHILOX_W0;
      k1 += PHILOX_W1;
    }
    uint64_t p0 = (uint64_t)PHILOX_M0 * c0;
    uint64_t p1 = (uint64_t)PHILOX_M1 * c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0;
    c1 = n1;
    c2 = n2;
    c3 = n3;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

uint64_t orc_keep_threshold(double p) {
  double t = ceil(p * 4294967296.0);
  if (t < 0) t = 0;
  if (t > 4294967296.0) t = 4294967296.0;
  return (uint64_t)t;
}

void orc_dropout_mask(uint64_t seed, uint32_t step, uint32_t layer,
                      uint32_t linear, uint32_t microbatch, double p,
                      int64_t M, int64_t K, uint32_t* bits) {
  const uint64_t T = orc_keep_threshold(p);
  const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  const int64_t words = K / 32;
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t wi = 0; wi < words; ++wi) {
      uint32_t word = 0;
      for (int b = 0; b < 32; ++b) {
        int64_t e = m * K + wi * 32 + b;
        uint32_t ctr[4] = {(uint32_t)(e >> 2), linear | (microbatch << 8),
                           layer, step};
        uint32_t r[4];
        orc_philox4x32_10(ctr, key, r);
        if ((uint64_t)r[e & 3] >= T) word |= 1u << b;
      }
      bits[m * words + wi] = word;
    }
  }
}

static int mask_bit(const uint32_t* mask, int64_t K, int64_t m, int64_t k) {
  if (!mask) return 1;
  return (mask[(m * K + k) >> 5] >> ((m * K + k) & 31)) & 1;
}

/* ---- LoRA linear ----------------------------------------------------------- */
void orc_lora_fwd_rows(int64_t M, int64_t N, int64_t K, int r,
                       const uint16_t* x, const uint16_t* Wq, const float* A,
                       const float* B, const uint32_t* mask, double scale,
                       const int64_t* rows, int64_t nrows, double* y,
                       double* U) {
  (void)M;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < nrows; ++i) {
    const int64_t m = rows ? rows[i] : i;
    double* xm = (double*)malloc(sizeof(double) * K);
    double* xd = (double*)malloc(sizeof(double) * K);
    double u[64];
    for (int64_t k = 0; k < K; ++k) {
      xm[k] = bf(x[m * K + k]);
      xd[k] = mask_bit(mask, K, m, k) ? xm[k] : 0.0;
    }
    for (int j = 0; j < r; ++j) {
      double s = 0.0;
      for (int64_t k = 0; k < K; ++k) s += xd[k] * (double)A[j * K + k];
      u[j] = s;
      if (U) U[i * r + j] = s;
    }
    for (int64_t n = 0; n < N; ++n) {
      const uint16_t* w = Wq + n * K;
      double s = 0.0;
      for (int64_t k = 0; k < K; ++k) s += xm[k] * bf(w[k]);
      double l = 0.0;
      for (int j = 0; j < r; ++j) l += u[j] * (double)B[n * r + j];
      y[i * N + n] = s + scale * l;
    }
    free(xm);
    free(xd);
  }
}

void orc_lora_bwd(int64_t M, int64_t N, int64_t K, int r, const uint16_t* x,
                  const uint16_t* Wq, const float* A, const float* B,
                  const uint32_t* mask, const uint16_t* dY, double scale,
                  const int64_t* rows, int64_t nrows, double* dX, double* dA,
                  double* dB) {
  /* G = dY B  [M, r];  U = (m.x) A^T  [M, r] */
  double* G = (double*)calloc((size_t)(M * r), sizeof(double));
  double* U = (double*)calloc((size_t)(M * r), sizeof(double));
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    for (int j = 0; j < r; ++j) {
      double s = 0.0;
      for (int64_t n = 0; n < N; ++n) s += bf(dY[m * N + n]) * (double)B[n * r + j];
      G[m * r + j] = s;
      double u = 0.0;
      for (int64_t k = 0; k < K; ++k)
        if (mask_bit(mask, K, m, k)) u += bf(x[m * K + k]) * (double)A[j * K + k];
      U[m * r + j] = u;
    }
  }
  if (dA) {
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < K; ++k) {
      for (int j = 0; j < r; ++j) {
        double s = 0.0;
        for (int64_t m = 0; m < M; ++m)
          if (mask_bit(mask, K, m, k)) s += G[m * r + j] * bf(x[m * K + k]);
        dA[j * K + k] = scale * s;
      }
    }
  }
  if (dB) {
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
      for (int j = 0; j < r; ++j) {
        double s = 0.0;
        for (int64_t m = 0; m < M; ++m) s += bf(dY[m * N + n]) * U[m * r + j];
        dB[n * r + j] = scale * s;
      }
    }
  }
  if (dX) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
      const int64_t m = rows ? rows[i] : i;
      double* acc = dX + i * K;
      for (int64_t k = 0; k < K; ++k) acc[k] = 0.0;
      for (int64_t n = 0; n < N; ++n) {
        double d = bf(dY[m * N + n]);
        if (d == 0.0) continue;
        const uint16_t* w = Wq + n * K;
        for (int64_t k = 0; k < K; ++k) acc[k] += d * bf(w[k]);
      }
      for (int64_t k = 0; k < K; ++k) {
        if (!mask_bit(mask, K, m, k)) continue;
        double l = 0.0;
        for (int j = 0; j < r; ++j) l += G[m * r + j] * (double)A[j * K + k];
        acc[k] += scale * l;
      }
    }
  }
  free(G);
  free(U);
}

/* ---- Synthetic stack -------------------------------------------------------- */
/* A tensor the method stores in bf16: round it, unless the exact mode is on
 * (the exact mode exists so finite differences can check the backward). */
static double rb(const orc_stack_cfg* c, double v) {
  return c->round_bf16 ? orc_bf16_to_f64(orc_f64_to_bf16(v)) : v;
}

/* y[M,N] = x[M,K] W'^T + scale ((m.x) A^T) B^T, x held as doubles. */
static void lin_fwd(const orc_stack_cfg* c, int64_t N, int64_t K,
                    const double* x, const uint16_t* Wq, const float* A,
                    const float* B, const uint32_t* mask, double scale,
                    double* y) {
  const int64_t M = c->M;
  const int r = c->r;
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    double u[64];
    for (int j = 0; j < r; ++j) {
      double s = 0.0;
      for (int64_t k = 0; k < K; ++k)
        if (mask_bit(mask, K, m, k)) s += x[m * K + k] * (double)A[j * K + k];
      u[j] = s;
    }
    for (int64_t n = 0; n < N; ++n) {
      double s = 0.0;
      const uint16_t* w = Wq + n * K;
      for (int64_t k = 0; k < K; ++k) s += x[m * K + k] * bf(w[k]);
      double l = 0.0;
      for (int j = 0; j < r; ++j) l += u[j] * (double)B[n * r + j];
      y[m * N + n] = s + scale * l;
    }
  }
}

/* Backward of lin_fwd for dY[M,N]; dX[M,K] is ADDED to (accumulates). */
static void lin_bwd(const orc_stack_cfg* c, int64_t N, int64_t K,
                    const double* x, const uint16_t* Wq, const float* A,
                    const float* B, const uint32_t* mask, double scale,
                    const double* dY, double* dX, double* dA, double* dB) {
  const int64_t M = c->M;
  const int r = c->r;
  double* G = (double*)calloc((size_t)(M * r), sizeof(double));
  double* U = (double*)calloc((size_t)(M * r), sizeof(double));
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    for (int j = 0; j < r; ++j) {
      double g = 0.0, u = 0.0;
      for (int64_t n = 0; n < N; ++n) g += dY[m * N + n] * (double)B[n * r + j];
      for (int64_t k = 0; k < K; ++k)
        if (mask_bit(mask, K, m, k)) u += x[m * K + k] * (double)A[j * K + k];
      G[m * r + j] = g;
      U[m * r + j] = u;
    }
  }
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < K; ++k)
    for (int j = 0; j < r; ++j) {
      double s = 0.0;
      for (int64_t m = 0; m < M; ++m)
        if (mask_bit(mask, K, m, k)) s += G[m * r + j] * x[m * K + k];
      dA[j * K + k] = scale * s;
    }
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n)
    for (int j = 0; j < r; ++j) {
      double s = 0.0;
      for (int64_t m = 0; m < M; ++m) s += dY[m * N + n] * U[m * r + j];
      dB[n * r + j] = scale * s;
    }
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    double* acc = dX + m * K;
    for (int64_t n = 0; n < N; ++n) {
      double d = dY[m * N + n];
      if (d == 0.0) continue;
      const uint16_t* w = Wq + n * K;
      for (int64_t k = 0; k < K; ++k) acc[k] += d * bf(w[k]);
    }
    for (int64_t k = 0; k < K; ++k) {
      if (!mask_bit(mask, K, m, k)) continue;
      double l = 0.0;
      for (int j = 0; j < r; ++j) l += G[m * r + j] * (double)A[j * K + k];
      acc[k] += scale * l;
    }
  }
  free(G);
  free(U);
}

/* RMSNorm with unit gain: y = x / sqrt(mean(x^2) + eps). */
static void rmsnorm_fwd(const orc_stack_cfg* c, int64_t H, const double* x,
                        double* y, double* rstd) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < c->M; ++m) {
    double ss = 0.0;
    for (int64_t i = 0; i < H; ++i) ss += x[m * H + i] * x[m * H + i];
    double rs = 1.0 / sqrt(ss / (double)H + c->eps);
    rstd[m] = rs;
    for (int64_t i = 0; i < H; ++i) y[m * H + i] = rb(c, x[m * H + i] * rs);
  }
}

/* dx += d/dx of RMSNorm for upstream dy: rstd*dy - rstd^3 x sum(dy x)/H. */
static void rmsnorm_bwd(const orc_stack_cfg* c, int64_t H, const double* x,
                        const double* rstd, const double* dy, double* dx) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < c->M; ++m) {
    double dot = 0.0;
    for (int64_t i = 0; i < H; ++i) dot += dy[m * H + i] * x[m * H + i];
    double rs = rstd[m];
    double coef = rs * rs * rs * dot / (double)H;
    for (int64_t i = 0; i < H; ++i)
      dx[m * H + i] += rs * dy[m * H + i] - coef * x[m * H + i];
  }
}

static double sigmoid(double g) { return 1.0 / (1.0 + exp(-g)); }

/* SwiGLU product act = SiLU(g) u = g sigmoid(g) u, and its partial
 * derivatives for an upstream gradient d: d/du = d g sigmoid(g),
 * d/dg = d u sigmoid(g) (1 + g (1 - sigmoid(g))). */
static double silu_mul1(double g, double u) { return g * sigmoid(g) * u; }
static void silu_mul_bwd1(double d, double g, double u, double* dg, double* du) {
  const double sg = sigmoid(g);
  *du = d * g * sg;
  *dg = d * u * sg * (1.0 + g * (1.0 - sg));
}

/* Backward of the kv-head repeat: kv head kh collects the rep query heads
 * kh*rep .. kh*rep + rep - 1 that read it. */
static double repeat_kv_bwd1(const double* dvr_row, int64_t rep, int64_t hd, int64_t kh,
                             int64_t d) {
  double sum = 0.0;
  for (int64_t t = 0; t < rep; ++t) sum += dvr_row[(kh * rep + t) * hd + d];
  return sum;
}

/* ---- causal attention core ------------------------------------------------ */
/* Scaled dot-product attention of Vaswani et al. (2017), causal, with grouped
 * kv heads (Ainslie et al. 2023): query head h reads kv head h / (nh / nkv).
 * Tokens are n_seq sequences of S, token t = b*S + i; q and o are [M, nh*d],
 * k and v are [M, nkv*d] (M = n_seq*S), row-major.  For query i of sequence
 * b and head h, over the keys j <= i of the same sequence:
 *   s_j = (q_i . k_j) / sqrt(d),  p_j = exp(s_j - lse_i),
 *   lse_i = log sum_{j<=i} exp(s_j),  o_i = sum_j p_j v_j.
 * lse is stored [nh, M]. */
static void attn_row_probs(int64_t S, int64_t nh, int64_t nkv, int64_t d, int64_t b, int64_t h,
                           int64_t i, const double* q, const double* k, double* p,
                           double* lse_out) {
  const int64_t g = h / (nh / nkv);
  const double sc = 1.0 / sqrt((double)d);
  const double* qi = q + ((b * S + i) * nh + h) * d;
  double mx = -INFINITY;
  for (int64_t j = 0; j <= i; ++j) {
    const double* kj = k + ((b * S + j) * nkv + g) * d;
    double s = 0.0;
    for (int64_t t = 0; t < d; ++t) s += qi[t] * kj[t];
    p[j] = s * sc;
    if (p[j] > mx) mx = p[j];
  }
  double l = 0.0;
  for (int64_t j = 0; j <= i; ++j) l += exp(p[j] - mx);
  const double lse = mx + log(l);
  for (int64_t j = 0; j <= i; ++j) p[j] = exp(p[j] - lse);
  if (lse_out) *lse_out = lse;
}

void orc_attention_fwd(int64_t n_seq, int64_t S, int64_t nh, int64_t nkv, int64_t d,
                       const double* q, const double* k, const double* v, double* o,
                       double* lse) {
  const int64_t M = n_seq * S;
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int64_t b = 0; b < n_seq; ++b)
    for (int64_t h = 0; h < nh; ++h) {
      const int64_t g = h / (nh / nkv);
      double* p = (double*)malloc(sizeof(double) * (size_t)S);
      for (int64_t i = 0; i < S; ++i) {
        double l;
        attn_row_probs(S, nh, nkv, d, b, h, i, q, k, p, &l);
        if (lse) lse[h * M + b * S + i] = l;
        double* oi = o + ((b * S + i) * nh + h) * d;
        for (int64_t t = 0; t < d; ++t) {
          double acc = 0.0;
          for (int64_t j = 0; j <= i; ++j) acc += p[j] * v[((b * S + j) * nkv + g) * d + t];
          oi[t] = acc;
        }
      }
      free(p);
    }
}

/* Gradients of the attention above for the upstream gradient dO [M, nh*d],
 * by the chain rule through the softmax:
 *   dv_j += p_ij dO_i,  dp_ij = dO_i . v_j,  D_i = sum_j p_ij dp_ij,
 *   ds_ij = p_ij (dp_ij - D_i),
 *   dq_i = sum_j ds_ij k_j / sqrt(d),  dk_j += ds_ij q_i / sqrt(d).
 * dk and dv sum over the query heads that share a kv head.  dq, dk, dv are
 * overwritten. */
void orc_attention_bwd(int64_t n_seq, int64_t S, int64_t nh, int64_t nkv, int64_t d,
                       const double* q, const double* k, const double* v, const double* dO,
                       double* dq, double* dk, double* dv) {
  const int64_t M = n_seq * S, rep = nh / nkv;
  const double sc = 1.0 / sqrt((double)d);
  memset(dq, 0, sizeof(double) * (size_t)(M * nh * d));
  memset(dk, 0, sizeof(double) * (size_t)(M * nkv * d));
  memset(dv, 0, sizeof(double) * (size_t)(M * nkv * d));
  /* one (sequence, kv head) per task: its dk, dv rows have one writer */
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int64_t b = 0; b < n_seq; ++b)
    for (int64_t g = 0; g < nkv; ++g) {
      double* p = (double*)malloc(sizeof(double) * (size_t)S);
      double* dp = (double*)malloc(sizeof(double) * (size_t)S);
      for (int64_t h = g * rep; h < (g + 1) * rep; ++h)
        for (int64_t i = 0; i < S; ++i) {
          attn_row_probs(S, nh, nkv, d, b, h, i, q, k, p, NULL);
          const double* dOi = dO + ((b * S + i) * nh + h) * d;
          const double* qi = q + ((b * S + i) * nh + h) * d;
          double D = 0.0;
          for (int64_t j = 0; j <= i; ++j) {
            const double* vj = v + ((b * S + j) * nkv + g) * d;
            double s = 0.0;
            for (int64_t t = 0; t < d; ++t) s += dOi[t] * vj[t];
            dp[j] = s;
            D += p[j] * s;
          }
          double* dqi = dq + ((b * S + i) * nh + h) * d;
          for (int64_t j = 0; j <= i; ++j) {
            const double ds = p[j] * (dp[j] - D);
            const double* kj = k + ((b * S + j) * nkv + g) * d;
            double* dkj = dk + ((b * S + j) * nkv + g) * d;
            double* dvj = dv + ((b * S + j) * nkv + g) * d;
            for (int64_t t = 0; t < d; ++t) {
              dqi[t] += sc * ds * kj[t];
              dkj[t] += sc * ds * qi[t];
              dvj[t] += p[j] * dOi[t];
            }
          }
        }
      free(p);
      free(dp);
    }
}

typedef struct {
  double *h, *a, *rstd1, *q, *k, *v, *vr, *h1, *b, *rstd2, *g, *u, *act;
  uint32_t* mask[ORC_NLIN];
} layer_saved;

void orc_stack_fwd_bwd(const orc_stack_cfg* c, uint32_t step,
                       const orc_stack_params* prm, const double* h0,
                       double* loss, double* h_out, double* const* dA,
                       double* const* dB) {
  orc_stack_fwd_bwd_mb(c, step, 0, 1, prm, h0, loss, h_out, dA, dB);
}

void orc_stack_fwd_bwd_mb(const orc_stack_cfg* c, uint32_t step, uint32_t microbatch,
                          int n_micro, const orc_stack_params* prm, const double* h0,
                          double* loss, double* h_out, double* const* dA,
                          double* const* dB) {
  const int64_t M = c->M, H = c->H, KV = c->KV, I = c->I, hd = c->head_dim;
  const int L = c->n_layers;
  const int64_t rep = H / KV;
  const double scale = (c->alpha / c->r) / (1.0 - c->p);
  const int64_t nK[ORC_NLIN] = {H, H, H, H, H, H, I};
  const int64_t nN[ORC_NLIN] = {H, KV, KV, H, I, I, H};

  layer_saved* S = (layer_saved*)calloc((size_t)L, sizeof(layer_saved));
  double* h = (double*)malloc(sizeof(double) * M * H);
  memcpy(h, h0, sizeof(double) * M * H);
  double* scratch = (double*)malloc(sizeof(double) * M * (H > I ? H : I));

  for (int l = 0; l < L; ++l) {
    layer_saved* s = &S[l];
    for (int li = 0; li < ORC_NLIN; ++li) {
      s->mask[li] = (uint32_t*)malloc(sizeof(uint32_t) * M * nK[li] / 32);
      orc_dropout_mask(c->seed, step, (uint32_t)l, (uint32_t)li, microbatch, c->p, M,
                       nK[li], s->mask[li]);
    }
    const int base = l * ORC_NLIN;
    s->h = (double*)malloc(sizeof(double) * M * H);
    memcpy(s->h, h, sizeof(double) * M * H);
    s->a = (double*)malloc(sizeof(double) * M * H);
    s->rstd1 = (double*)malloc(sizeof(double) * M);
    rmsnorm_fwd(c, H, h, s->a, s->rstd1);
    /* q and k: with the attention core they are kept (bf16, as stored);
     * with the repeat(v) stand-in nothing reads them, so they are computed
     * for fidelity and dropped. */
    s->q = (double*)malloc(sizeof(double) * M * H);
    lin_fwd(c, H, H, s->a, prm->Wq[base + ORC_Q], prm->A[base + ORC_Q],
            prm->B[base + ORC_Q], s->mask[ORC_Q], scale, s->q);
    s->k = (double*)malloc(sizeof(double) * M * KV);
    lin_fwd(c, KV, H, s->a, prm->Wq[base + ORC_K], prm->A[base + ORC_K],
            prm->B[base + ORC_K], s->mask[ORC_K], scale, s->k);
    for (int64_t i = 0; i < M * H; ++i) s->q[i] = rb(c, s->q[i]);
    for (int64_t i = 0; i < M * KV; ++i) s->k[i] = rb(c, s->k[i]);
    s->v = (double*)malloc(sizeof(double) * M * KV);
    lin_fwd(c, KV, H, s->a, prm->Wq[base + ORC_V], prm->A[base + ORC_V],
            prm->B[base + ORC_V], s->mask[ORC_V], scale, s->v);
    for (int64_t i = 0; i < M * KV; ++i) s->v[i] = rb(c, s->v[i]);
    s->vr = (double*)malloc(sizeof(double) * M * H);
    if (c->attn) {
      /* causal attention over the M tokens (one sequence), output stored bf16 */
      orc_attention_fwd(1, M, H / hd, KV / hd, hd, s->q, s->k, s->v, s->vr, NULL);
      for (int64_t i = 0; i < M * H; ++i) s->vr[i] = rb(c, s->vr[i]);
    } else {
      /* repeat_kv: query head hh reads kv head hh / rep */
      for (int64_t m = 0; m < M; ++m)
        for (int64_t hh = 0; hh < H / hd; ++hh)
          for (int64_t d = 0; d < hd; ++d)
            s->vr[m * H + hh * hd + d] = s->v[m * KV + (hh / rep) * hd + d];
    }
    double* o = scratch;
    lin_fwd(c, H, H, s->vr, prm->Wq[base + ORC_O], prm->A[base + ORC_O],
            prm->B[base + ORC_O], s->mask[ORC_O], scale, o);
    s->h1 = (double*)malloc(sizeof(double) * M * H);
    for (int64_t i = 0; i < M * H; ++i) s->h1[i] = h[i] + rb(c, o[i]);
    s->b = (double*)malloc(sizeof(double) * M * H);
    s->rstd2 = (double*)malloc(sizeof(double) * M);
    rmsnorm_fwd(c, H, s->h1, s->b, s->rstd2);
    s->g = (double*)malloc(sizeof(double) * M * I);
    s->u = (double*)malloc(sizeof(double) * M * I);
    lin_fwd(c, I, H, s->b, prm->Wq[base + ORC_GATE], prm->A[base + ORC_GATE],
            prm->B[base + ORC_GATE], s->mask[ORC_GATE], scale, s->g);
    lin_fwd(c, I, H, s->b, prm->Wq[base + ORC_UP], prm->A[base + ORC_UP],
            prm->B[base + ORC_UP], s->mask[ORC_UP], scale, s->u);
    s->act = (double*)malloc(sizeof(double) * M * I);
    for (int64_t i = 0; i < M * I; ++i) {
      s->g[i] = rb(c, s->g[i]);
      s->u[i] = rb(c, s->u[i]);
      s->act[i] = rb(c, silu_mul1(s->g[i], s->u[i]));
    }
    double* d = scratch;
    lin_fwd(c, H, I, s->act, prm->Wq[base + ORC_DOWN], prm->A[base + ORC_DOWN],
            prm->B[base + ORC_DOWN], s->mask[ORC_DOWN], scale, d);
    for (int64_t i = 0; i < M * H; ++i) h[i] = s->h1[i] + rb(c, d[i]);
  }

  double ss = 0.0;
  for (int64_t i = 0; i < M * H; ++i) ss += h[i] * h[i];
  /* this micro-batch's share of the step loss (1/n_micro) sum_mb 0.5 mean(h^2) */
  *loss = 0.5 * ss / (double)(M * H) / (double)n_micro;
  if (h_out) memcpy(h_out, h, sizeof(double) * M * H);

  if (dA && dB) {
    double* dh = (double*)malloc(sizeof(double) * M * H);
    for (int64_t i = 0; i < M * H; ++i) dh[i] = h[i] / ((double)(M * H) * (double)n_micro);
    double* dYb = (double*)malloc(sizeof(double) * M * (H > I ? H : I));
    double* dx = (double*)malloc(sizeof(double) * M * (H > I ? H : I));
    double* dx2 = (double*)malloc(sizeof(double) * M * H);
    for (int l = L - 1; l >= 0; --l) {
      layer_saved* s = &S[l];
      const int base = l * ORC_NLIN;
      /* down: dY = bf16(dh2) */
      for (int64_t i = 0; i < M * H; ++i) dYb[i] = rb(c, dh[i]);
      double* dact = dx;
      memset(dact, 0, sizeof(double) * M * I);
      lin_bwd(c, H, I, s->act, prm->Wq[base + ORC_DOWN], prm->A[base + ORC_DOWN],
              prm->B[base + ORC_DOWN], s->mask[ORC_DOWN], scale, dYb, dact,
              dA[base + ORC_DOWN], dB[base + ORC_DOWN]);
      /* SiLU(g) * u backward; dg, du stored bf16 (they are GEMM operands) */
      double* dg = (double*)malloc(sizeof(double) * M * I);
      double* du = (double*)malloc(sizeof(double) * M * I);
      for (int64_t i = 0; i < M * I; ++i) {
        double gi, ui;
        silu_mul_bwd1(dact[i], s->g[i], s->u[i], &gi, &ui);
        dg[i] = rb(c, gi);
        du[i] = rb(c, ui);
      }
      double* db = dx2;
      memset(db, 0, sizeof(double) * M * H);
      lin_bwd(c, I, H, s->b, prm->Wq[base + ORC_GATE], prm->A[base + ORC_GATE],
              prm->B[base + ORC_GATE], s->mask[ORC_GATE], scale, dg, db,
              dA[base + ORC_GATE], dB[base + ORC_GATE]);
      lin_bwd(c, I, H, s->b, prm->Wq[base + ORC_UP], prm->A[base + ORC_UP],
              prm->B[base + ORC_UP], s->mask[ORC_UP], scale, du, db,
              dA[base + ORC_UP], dB[base + ORC_UP]);
      free(dg);
      free(du);
      /* dh1 = dh2 + RMSNorm2 backward */
      rmsnorm_bwd(c, H, s->h1, s->rstd2, db, dh);
      /* o: dY = bf16(dh1) */
      for (int64_t i = 0; i < M * H; ++i) dYb[i] = rb(c, dh[i]);
      double* dvr = dx;
      memset(dvr, 0, sizeof(double) * M * H);
      lin_bwd(c, H, H, s->vr, prm->Wq[base + ORC_O], prm->A[base + ORC_O],
              prm->B[base + ORC_O], s->mask[ORC_O], scale, dYb, dvr,
              dA[base + ORC_O], dB[base + ORC_O]);
      double* da = dx2;
      memset(da, 0, sizeof(double) * M * H);
      if (c->attn) {
        /* attention backward from the bf16-stored upstream gradient; dq, dk,
         * dv are stored bf16 (GEMM operands) */
        for (int64_t i = 0; i < M * H; ++i) dvr[i] = rb(c, dvr[i]);
        double* dq = (double*)malloc(sizeof(double) * M * H);
        double* dk = (double*)malloc(sizeof(double) * M * KV);
        double* dv = (double*)malloc(sizeof(double) * M * KV);
        orc_attention_bwd(1, M, H / hd, KV / hd, hd, s->q, s->k, s->v, dvr, dq, dk, dv);
        for (int64_t i = 0; i < M * H; ++i) dq[i] = rb(c, dq[i]);
        for (int64_t i = 0; i < M * KV; ++i) {
          dk[i] = rb(c, dk[i]);
          dv[i] = rb(c, dv[i]);
        }
        lin_bwd(c, KV, H, s->a, prm->Wq[base + ORC_V], prm->A[base + ORC_V],
                prm->B[base + ORC_V], s->mask[ORC_V], scale, dv, da,
                dA[base + ORC_V], dB[base + ORC_V]);
        lin_bwd(c, KV, H, s->a, prm->Wq[base + ORC_K], prm->A[base + ORC_K],
                prm->B[base + ORC_K], s->mask[ORC_K], scale, dk, da,
                dA[base + ORC_K], dB[base + ORC_K]);
        lin_bwd(c, H, H, s->a, prm->Wq[base + ORC_Q], prm->A[base + ORC_Q],
                prm->B[base + ORC_Q], s->mask[ORC_Q], scale, dq, da,
                dA[base + ORC_Q], dB[base + ORC_Q]);
        free(dq);
        free(dk);
        free(dv);
      } else {
        /* repeat_kv backward: sum over the rep query heads of each kv head */
        double* dv = dYb;
        for (int64_t m = 0; m < M; ++m)
          for (int64_t kh = 0; kh < KV / hd; ++kh)
            for (int64_t d = 0; d < hd; ++d)
              dv[m * KV + kh * hd + d] = rb(c, repeat_kv_bwd1(dvr + m * H, rep, hd, kh, d));
        lin_bwd(c, KV, H, s->a, prm->Wq[base + ORC_V], prm->A[base + ORC_V],
                prm->B[base + ORC_V], s->mask[ORC_V], scale, dv, da,
                dA[base + ORC_V], dB[base + ORC_V]);
        /* q and k receive no gradient: their outputs are unused */
        memset(dA[base + ORC_Q], 0, sizeof(double) * c->r * H);
        memset(dB[base + ORC_Q], 0, sizeof(double) * H * c->r);
        memset(dA[base + ORC_K], 0, sizeof(double) * c->r * H);
        memset(dB[base + ORC_K], 0, sizeof(double) * KV * c->r);
      }
      /* dh = dh1 + RMSNorm1 backward */
      rmsnorm_bwd(c, H, s->h, s->rstd1, da, dh);
    }
    free(dh);
    free(dYb);
    free(dx);
    free(dx2);
  }

  for (int l = 0; l < L; ++l) {
    layer_saved* s = &S[l];
    for (int li = 0; li < ORC_NLIN; ++li) free(s->mask[li]);
    free(s->h);
    free(s->a);
    free(s->rstd1);
    free(s->q);
    free(s->k);
    free(s->v);
    free(s->vr);
    free(s->h1);
    free(s->b);
    free(s->rstd2);
    free(s->g);
    free(s->u);
    free(s->act);
  }
  free(S);
  free(h);
  free(scratch);
}

/* ---- stack pieces on their own ------------------------------------------------ */
void orc_rmsnorm_bf16(int64_t M, int64_t H, double eps, const double* x, uint16_t* y,
                      double* rstd) {
  orc_stack_cfg c;
  memset(&c, 0, sizeof(c));
  c.M = M;
  c.eps = eps;
  c.round_bf16 = 1;
  double* out = (double*)malloc(sizeof(double) * M * H);
  rmsnorm_fwd(&c, H, x, out, rstd);
  for (int64_t i = 0; i < M * H; ++i) y[i] = orc_f64_to_bf16(out[i]);
  free(out);
}

void orc_silu_mul_bf16(int64_t n, const uint16_t* g, const uint16_t* u, uint16_t* act) {
  for (int64_t i = 0; i < n; ++i) act[i] = orc_f64_to_bf16(silu_mul1(bf(g[i]), bf(u[i])));
}

void orc_silu_mul_f64(int64_t n, const double* g, const double* u, double* act) {
  for (int64_t i = 0; i < n; ++i) act[i] = silu_mul1(g[i], u[i]);
}

void orc_rmsnorm_f64(int64_t M, int64_t H, double eps, int round_bf16, const double* x,
                     double* y, double* rstd) {
  orc_stack_cfg c;
  memset(&c, 0, sizeof(c));
  c.M = M;
  c.eps = eps;
  c.round_bf16 = round_bf16;
  rmsnorm_fwd(&c, H, x, y, rstd);
}

void orc_rmsnorm_bwd_add(int64_t M, int64_t H, const double* x, const double* rstd,
                         const double* dy, double* dx) {
  orc_stack_cfg c;
  memset(&c, 0, sizeof(c));
  c.M = M;
  rmsnorm_bwd(&c, H, x, rstd, dy, dx);
}

void orc_silu_mul_bwd(int64_t n, int round_bf16, const double* dact, const double* g,
                      const double* u, double* dg, double* du) {
  for (int64_t i = 0; i < n; ++i) {
    double a, b;
    silu_mul_bwd1(dact[i], g[i], u[i], &a, &b);
    dg[i] = round_bf16 ? bf(orc_f64_to_bf16(a)) : a;
    du[i] = round_bf16 ? bf(orc_f64_to_bf16(b)) : b;
  }
}

void orc_repeat_kv_bwd(int64_t M, int64_t H, int64_t KV, int64_t head_dim, int round_bf16,
                       const double* dvr, double* dv) {
  const int64_t rep = H / KV;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t kh = 0; kh < KV / head_dim; ++kh)
      for (int64_t d = 0; d < head_dim; ++d) {
        const double v = repeat_kv_bwd1(dvr + m * H, rep, head_dim, kh, d);
        dv[m * KV + kh * head_dim + d] = round_bf16 ? bf(orc_f64_to_bf16(v)) : v;
      }
}

void orc_repeat_kv(int64_t M, int64_t H, int64_t KV, int64_t head_dim, const uint16_t* v,
                   uint16_t* vr) {
  const int64_t rep = H / KV;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t hh = 0; hh < H / head_dim; ++hh)
      for (int64_t d = 0; d < head_dim; ++d)
        vr[m * H + hh * head_dim + d] = v[m * KV + (hh / rep) * head_dim + d];
}

/* ---- Adam -------------------------------------------------------------------- */
void orc_adam_step(int64_t n, double* p, const double* g, double* m, double* v,
                   int64_t t, double lr, double beta1, double beta2,
                   double eps) {
  const double bc1 = 1.0 - pow(beta1, (double)t);
  const double bc2 = 1.0 - pow(beta2, (double)t);
  for (int64_t i = 0; i < n; ++i) {
    m[i] = beta1 * m[i] + (1.0 - beta1) * g[i];
    v[i] = beta2 * v[i] + (1.0 - beta2) * g[i] * g[i];
    double mhat = m[i] / bc1;
    double vhat = v[i] / bc2;
    p[i] -= lr * mhat / (sqrt(vhat) + eps);
  }
}
