// attention.cu -- causal softmax attention with grouped kv heads on the
// tcgen05 tensor cores: forward, and a backward in two kernels (dQ; dK/dV per
// query head) plus a fixed-order sum over the query heads of each kv group.
//
// The research page "Poros" says the learning problem is unchanged by
// streaming and the model keeps its own attention kernels; the core is
// scaled dot-product attention (Vaswani et al., 2017), causal, with query
// head h reading kv head h / (nh / nkv) (grouped-query attention, Ainslie et
// al., 2023).  Tokens are n_seq sequences of S, token t = b*S + i; q and the
// output are [M, nh*D], k and v [M, nkv*D] bf16 row-major (M = n_seq*S);
// D = 64 or 128.
//
// Forward, one CTA per (128 queries, head, sequence), 64 keys per step:
//   pass 1: S = Q K_j^T on the tensor cores (fp32 in tensor memory); the
//           softmax warps keep the row maximum m of S log2e/sqrt(D);
//   pass 2: S again, P = exp2(S log2e/sqrt(D) - m) in (0, 1], the row sum l,
//           P split as P_hi + P_lo (two bf16 parts, about 16 significant
//           bits together) and O += P_hi V_j + P_lo V_j.
// With the maximum known no rescaling of O is needed; the epilogue divides
// by l and writes O as bf16 (and fp32 when asked), lse = (m + log2 l) ln 2.
//
// Backward with D_i = dO_i . O_i (fp32 O from the forward):
//   dQ kernel, one CTA per (128 queries, head, sequence), 64 keys per step:
//     S = Q K_j^T, dP = dO V_j^T, P as in the forward, dS = P (dP - D_i),
//     dQ += dS_hi K_j + dS_lo K_j; dq = dQ / sqrt(D) as bf16.  It also
//     stores D_i for the next kernel.
//   dK/dV kernel, one CTA per (128 keys, query head, sequence), 64 queries
//     per step, on the transposed problem: S^T = K Q_i^T, dP^T = V dO_i^T,
//     dV += P^T dO_i, dK += dS^T Q_i (hi/lo parts again), written in fp32
//     per query head;
//   a pointwise kernel sums the query heads of each kv group in head order
//   and rounds dk, dv to bf16.
// Every sum has one fixed order: the results are identical run to run.
//
// Warp roles in every kernel (192 threads): warp 0 issues the TMA loads,
// warp 1 (one lane) the MMAs, warps 2-5 own one row of the 128-row tile each
// (tensor-memory lane quarter warp % 4) and do the softmax / gradient
// arithmetic and the epilogue.  Every wait is bounded (see common.cuh).
#define WS_ATTN_TU 1
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace ws {

cudaError_t attn_read_and_clear_dev_error(uint32_t* flags) {
  cudaError_t e = cudaMemcpyFromSymbol(flags, g_dev_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  const uint32_t zero = 0;
  return cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(uint32_t));
}

namespace {

constexpr int kAtThreads = 192;
constexpr int kBig = 128;    // rows of the CTA's fixed tile (queries, or keys in dK/dV)
constexpr int kStep = 64;    // rows of one step's tile (keys, or queries in dK/dV)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Byte offset of 16-byte chunk c (0..7) of row r in a tile of 128-byte rows
// under the 128-byte swizzle (the layout TMA writes and the MMA reads).
WS_DEVINL uint32_t sw_off(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// K-major operand: a tile of R rows x D columns stored as D/64 boxes of
// R x 128 bytes; contraction step ks covers columns 16 ks .. 16 ks + 15.
WS_DEVINL uint64_t kmaj_desc(uint32_t base, int R, int ks) {
  return smem_desc_sw128(base + (uint32_t)((ks >> 2) * R * 128 + (ks & 3) * 32), 16, 1024);
}
// MN-major B operand from a tile of 64 rows x D columns, read as N = D
// columns and K = the 64 rows; contraction step ks covers rows 16 ks ..
// 16 ks + 15.  The 64-column boxes lie 64 x 128 bytes apart.
WS_DEVINL uint64_t mn_desc(uint32_t base, int ks) {
  return smem_desc_sw128(base + (uint32_t)(ks * 2048), kStep * 128, 1024);
}

// 2^x with the hardware approximation (relative error about 2^-22; results
// below 2^-126 flush to zero, which is what a zero weight needs anyway).
WS_DEVINL float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One answer per warp: true only if v holds in every lane.  The row warps
// wait on barriers lane by lane; deciding to stop as a warp keeps their
// later warp-wide steps (__syncwarp, tensor-memory loads) convergent.
WS_DEVINL bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// bf16 high part of x and the bf16 rounding of the remainder.
WS_DEVINL void split2(float x, float& hi, float& lo) {
  hi = bf16_lo(pack_bf16x2(x, 0.0f));
  lo = x - hi;
}

// Write one row of 64 fp32 values as bf16 hi/lo parts into two K-major
// 128-row x 64-column tiles (row r).
WS_DEVINL void put_row_hilo(uint8_t* hi_tile, uint8_t* lo_tile, int r, const float (&v)[kStep]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float h0, l0, h1, l1;
      split2(v[c * 8 + 2 * e], h0, l0);
      split2(v[c * 8 + 2 * e + 1], h1, l1);
      h[e] = pack_bf16x2(h0, h1);
      l[e] = pack_bf16x2(l0, l1);
    }
    sts128(hi_tile + sw_off(r, c), h[0], h[1], h[2], h[3]);
    sts128(lo_tile + sw_off(r, c), l[0], l[1], l[2], l[3]);
  }
}

// 64 fp32 columns of this thread's tensor-memory row.
WS_DEVINL void tmem_row64(uint32_t taddr, float (&v)[kStep]) {
  uint32_t a[32], b[32];
  tmem_ld_32x32b_x32(taddr, a);
  tmem_ld_32x32b_x32(taddr + 32u, b);
  tmem_ld_wait();
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    v[e] = __uint_as_float(a[e]);
    v[32 + e] = __uint_as_float(b[e]);
  }
}

struct AttnFwdArgs {
  CUtensorMap tq;  // q [M, nh*D], box {64, 128}
  CUtensorMap tk;  // k [M, nkv*D], box {64, 64}
  CUtensorMap tv;  // v [M, nkv*D], box {64, 64}
  int S, nh, nkv;
  int64_t M;
  float sl2;       // log2(e) / sqrt(D)
  uint16_t* o;     // [M, nh*D] bf16
  float* o32;      // [M, nh*D] fp32 or NULL
  float* lse;      // [nh, M] natural log-sum-exp
};

// Shared-memory plan of the forward: Q tile, ring of K/V step tiles, two
// P buffers (hi, lo), barriers.
template <int D>
struct FwdSmem {
  static constexpr uint32_t Q = kBig * D * 2;
  static constexpr uint32_t T = kStep * D * 2;
  static constexpr int NSLOT = 4;
  static constexpr uint32_t P = kBig * kStep * 2;
  static constexpr uint32_t OFF_RING = Q;
  static constexpr uint32_t OFF_P = OFF_RING + NSLOT * T;
  static constexpr uint32_t OFF_BAR = OFF_P + 4 * P;
  static constexpr uint32_t BYTES = OFF_BAR + 256 + 1024;
};

template <int D>
__global__ void __launch_bounds__(kAtThreads, 1) k_attn_fwd(const __grid_constant__ AttnFwdArgs a) {
  using L = FwdSmem<D>;
  constexpr int NS = L::NSLOT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* ring = smem + L::OFF_RING;
  uint8_t* sP = smem + L::OFF_P;  // [buf][hi, lo]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* qfull = bars;
  uint64_t* full = bars + 1;           // [NS]
  uint64_t* empty = full + NS;         // [NS]
  uint64_t* s_full = empty + NS;       // [2]
  uint64_t* s_empty = s_full + 2;      // [2]
  uint64_t* p_full = s_empty + 2;      // [2]
  uint64_t* p_empty = p_full + 2;      // [2]
  uint64_t* o_full = p_empty + 2;
  uint64_t* drain = o_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* skip_flag = tmem_slot + 2;

  const int warp = (int)warp_id(), lane = (int)lane_id();
  // heads vary fastest and the longest tiles (the last queries) come first,
  // so a second wave, if any, holds the shortest tiles
  const int h = (int)blockIdx.x, qt = (int)(gridDim.y - 1 - blockIdx.y), b = (int)blockIdx.z;
  const int S = a.S;
  const int g = h / (a.nh / a.nkv);
  const int64_t row0 = (int64_t)b * S + (int64_t)qt * kBig;
  const int qend = min(S, (qt + 1) * kBig);        // local end of this tile's queries
  const int J = (qend + kStep - 1) / kStep;        // key steps (causal)
  constexpr uint32_t TM_S = 0, TM_O = 2 * kStep;   // tensor-memory columns
  constexpr uint32_t TM_COLS = 256;

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    *skip_flag = (*(volatile uint32_t*)&g_dev_error != 0u) ? 1u : 0u;
    mbar_init(qfull, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 4);
      mbar_init(&p_full[i], 4);
      mbar_init(&p_empty[i], 1);
    }
    mbar_init(o_full, 1);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_launch_dependents();
  const bool run = *skip_flag == 0u;

  if (warp == 0) {
    if (lane == 0 && run) {
      // Q once, then the key/value tiles in the order the MMA warp uses
      // them: K_0..K_{J-1}; then K_0, K_1, V_0, K_2, V_1, ..., V_{J-1}.
      mbar_arrive_expect_tx(qfull, L::Q);
#pragma unroll
      for (int bx = 0; bx < D / 64; ++bx)
        tma_load_2d(sQ + bx * kBig * 128, &a.tq, qfull, h * D + bx * 64, (int)row0);
      int n = 0;
      auto load = [&](const CUtensorMap* m, int j) {
        const int st = n % NS;
        const uint32_t ph = (uint32_t)(n / NS) & 1u;
        if (*abort_flag || !mbar_wait(&empty[st], ph ^ 1u, DERR_TIMEOUT_EMPTY)) {
          *abort_flag = 1u;
          return false;
        }
        mbar_arrive_expect_tx(&full[st], L::T);
        uint8_t* dst = ring + st * L::T;
        const int y = (int)((int64_t)b * S + (int64_t)j * kStep);
#pragma unroll
        for (int bx = 0; bx < D / 64; ++bx)
          tma_load_2d(dst + bx * kStep * 128, m, &full[st], g * D + bx * 64, y);
        ++n;
        return true;
      };
      bool ok = true;
      for (int j = 0; j < J && ok; ++j) ok = load(&a.tk, j);
      for (int j = 0; j < J && ok; ++j) {
        ok = load(&a.tk, j);
        if (ok && j >= 1) ok = load(&a.tv, j - 1);
      }
      if (ok) ok = load(&a.tv, J - 1);
      // nothing may land after the CTA is gone
      for (int i = (n > NS ? n - NS : 0); i < n; ++i)
        mbar_wait(&full[i % NS], (uint32_t)(i / NS) & 1u, DERR_TIMEOUT_DRAIN);
      mbar_wait(qfull, 0u, DERR_TIMEOUT_DRAIN);
    }
  } else if (warp == 1) {
    if (lane == 0 && run) {
      constexpr uint32_t idS = idesc_bf16_f32(kBig, kStep, 0u);
      constexpr uint32_t idO = idesc_bf16_f32(kBig, D, 1u);
      const uint32_t aQ = smem_u32(sQ);
      int n = 0, u = 0;
      bool ok = mbar_wait(qfull, 0u, DERR_TIMEOUT_FULL);
      auto take = [&]() {
        const int st = n % NS;
        if (*abort_flag || !mbar_wait(&full[st], (uint32_t)(n / NS) & 1u, DERR_TIMEOUT_FULL)) {
          *abort_flag = 1u;
          return -1;
        }
        tc_fence_after();
        return st;
      };
      auto issue_S = [&]() {
        const int sb = u & 1;
        if (*abort_flag ||
            !mbar_wait(&s_empty[sb], ((uint32_t)(u >> 1) & 1u) ^ 1u, DERR_TIMEOUT_EMPTY)) {
          *abort_flag = 1u;
          return false;
        }
        const int st = take();
        if (st < 0) return false;
        const uint32_t bK = smem_u32(ring + st * L::T);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          tc_mma_f16(tmem + TM_S + sb * kStep, kmaj_desc(aQ, kBig, ks), kmaj_desc(bK, kStep, ks),
                     idS, ks > 0 ? 1u : 0u);
        tc_commit(&empty[st]);
        tc_commit(&s_full[sb]);
        ++n;
        ++u;
        return true;
      };
      for (int j = 0; j < J && ok; ++j) ok = issue_S();
      if (ok) ok = issue_S();
      for (int j = 0; j < J && ok; ++j) {
        if (j + 1 < J) ok = issue_S();
        if (!ok) break;
        const int pb = j & 1;
        if (*abort_flag || !mbar_wait(&p_full[pb], (uint32_t)(j >> 1) & 1u, DERR_TIMEOUT_BFULL)) {
          *abort_flag = 1u;
          break;
        }
        const int st = take();
        if (st < 0) break;
        const uint32_t bV = smem_u32(ring + st * L::T);
        const uint32_t aHi = smem_u32(sP + (2 * pb) * L::P);
        const uint32_t aLo = smem_u32(sP + (2 * pb + 1) * L::P);
#pragma unroll
        for (int ks = 0; ks < kStep / 16; ++ks)
          tc_mma_f16(tmem + TM_O, kmaj_desc(aHi, kBig, ks), mn_desc(bV, ks), idO,
                     (j > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < kStep / 16; ++ks)
          tc_mma_f16(tmem + TM_O, kmaj_desc(aLo, kBig, ks), mn_desc(bV, ks), idO, 1u);
        tc_commit(&empty[st]);
        tc_commit(&p_empty[pb]);
        ++n;
      }
      tc_commit(o_full);
      tc_commit(drain);
      mbar_wait(drain, 0u, DERR_TIMEOUT_DRAIN);
    }
  } else if (run) {
    // ---- softmax warps: thread <-> query row r of the tile
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int qi = qt * kBig + r;                     // local query index
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    const float sl2 = a.sl2;
    int u = 0;
    bool ok = true;
    auto get_S = [&](float (&v)[kStep]) {
      const int sb = u & 1;
      if (!warp_all(!*abort_flag &&
                    mbar_wait(&s_full[sb], (uint32_t)(u >> 1) & 1u, DERR_TIMEOUT_ACC))) {
        *abort_flag = 1u;
        return false;
      }
      tc_fence_after();
      tmem_row64(trow + TM_S + sb * kStep, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[sb]);
      ++u;
      return true;
    };
    // pass 1: row maximum of the scaled scores (base 2)
    float m2 = -INFINITY;
    for (int j = 0; j < J && ok; ++j) {
      float v[kStep];
      if (!(ok = get_S(v))) break;
#pragma unroll
      for (int c = 0; c < kStep; ++c)
        if (j * kStep + c <= qi) m2 = fmaxf(m2, v[c] * sl2);
    }
    // pass 2: p = 2^(s - max) in (0, 1] as bf16 hi/lo operands; the row sum
    // l in column order; O = (sum_j p_j v_j) / l in the epilogue
    float l = 0.0f;
    for (int j = 0; j < J && ok; ++j) {
      float v[kStep];
      if (!(ok = get_S(v))) break;
#pragma unroll
      for (int c = 0; c < kStep; ++c) {
        v[c] = (j * kStep + c > qi) ? 0.0f : ex2(v[c] * sl2 - m2);
        l += v[c];
      }
      const int pb = j & 1;
      if (!warp_all(!*abort_flag && mbar_wait(&p_empty[pb], ((uint32_t)(j >> 1) & 1u) ^ 1u,
                                                      DERR_TIMEOUT_BEMPTY))) {
        *abort_flag = 1u;
        ok = false;
        break;
      }
      put_row_hilo(sP + (2 * pb) * L::P, sP + (2 * pb + 1) * L::P, r, v);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[pb]);
    }
    const float lse2 = m2 + log2f(l);
    // epilogue: O row divided by the row sum, lse
    if (warp_all(ok && mbar_wait_backoff(o_full, 0u, DERR_TIMEOUT_ACC) && !*abort_flag)) {
      tc_fence_after();
      const int64_t row = row0 + r;
      const bool valid = qi < S && row < a.M;
      const int64_t ld = (int64_t)a.nh * D;
      // 32-byte stores need 32-byte aligned rows
      const bool v8 = (reinterpret_cast<uintptr_t>(a.o) & 31u) == 0u && (ld & 15) == 0 &&
                      (!a.o32 || (reinterpret_cast<uintptr_t>(a.o32) & 31u) == 0u);
#pragma unroll
      for (int cc = 0; cc < D; cc += 32) {
        uint32_t acc[32];
        tmem_ld_32x32b_x32(trow + TM_O + cc, acc);
        tmem_ld_wait();
        if (!valid) continue;
        float ov[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) ov[e] = __fdiv_rn(__uint_as_float(acc[e]), l);
        uint16_t* dst = a.o + row * ld + h * D + cc;
        if (v8) {
          // whole 32-byte sectors per store (a warp's lanes hold different rows)
#pragma unroll
          for (int e = 0; e < 32; e += 16)
            st_global_v8(dst + e, pack_bf16x2(ov[e], ov[e + 1]), pack_bf16x2(ov[e + 2], ov[e + 3]),
                         pack_bf16x2(ov[e + 4], ov[e + 5]), pack_bf16x2(ov[e + 6], ov[e + 7]),
                         pack_bf16x2(ov[e + 8], ov[e + 9]), pack_bf16x2(ov[e + 10], ov[e + 11]),
                         pack_bf16x2(ov[e + 12], ov[e + 13]), pack_bf16x2(ov[e + 14], ov[e + 15]));
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 8)
            *reinterpret_cast<uint4*>(dst + e) =
                make_uint4(pack_bf16x2(ov[e], ov[e + 1]), pack_bf16x2(ov[e + 2], ov[e + 3]),
                           pack_bf16x2(ov[e + 4], ov[e + 5]), pack_bf16x2(ov[e + 6], ov[e + 7]));
        }
        if (a.o32) {
          float* d32 = a.o32 + row * ld + h * D + cc;
          if (v8) {
#pragma unroll
            for (int e = 0; e < 32; e += 8)
              st_global_v8(d32 + e, __float_as_uint(ov[e]), __float_as_uint(ov[e + 1]),
                           __float_as_uint(ov[e + 2]), __float_as_uint(ov[e + 3]),
                           __float_as_uint(ov[e + 4]), __float_as_uint(ov[e + 5]),
                           __float_as_uint(ov[e + 6]), __float_as_uint(ov[e + 7]));
          } else {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(d32 + e) = make_float4(ov[e], ov[e + 1], ov[e + 2], ov[e + 3]);
          }
        }
      }
      if (valid) a.lse[(int64_t)h * a.M + row] = lse2 * kLn2;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TM_COLS);
}

// ------------------------------------------------------------------------------ backward: dQ
struct AttnDqArgs {
  CUtensorMap tq;   // q [M, nh*D], box {64, 128}
  CUtensorMap tdo;  // dO [M, nh*D], box {64, 128}
  CUtensorMap tk;   // k [M, nkv*D], box {64, 64}
  CUtensorMap tv;   // v [M, nkv*D], box {64, 64}
  int S, nh, nkv;
  int64_t M;
  float sl2;          // log2(e) / sqrt(D)
  float scale;        // 1 / sqrt(D)
  const float* lse;   // [nh, M]
  const float* Dvec;  // [nh, M]: dO . O per row
  uint16_t* dq;       // [M, nh*D] bf16
};

template <int D>
struct DqSmem {
  static constexpr uint32_t Q = kBig * D * 2;
  static constexpr uint32_t T = kStep * D * 2;
  static constexpr int NSLOT = 4;
  static constexpr uint32_t P = kBig * kStep * 2;
  static constexpr uint32_t OFF_DO = Q;
  static constexpr uint32_t OFF_RING = 2 * Q;
  static constexpr uint32_t OFF_DS = OFF_RING + NSLOT * T;
  static constexpr uint32_t OFF_BAR = OFF_DS + 4 * P;
  static constexpr uint32_t BYTES = OFF_BAR + 256 + 1024;
};

// dQ of one (128 queries, head, sequence) tile; `a` lives in the kernel's
// parameter space (its tensor maps are read by TMA from there).
template <int D>
WS_DEVINL void attn_dq_tile(const AttnDqArgs& a, uint8_t* smem, int qt, int h, int b) {
  using L = DqSmem<D>;
  constexpr int NS = L::NSLOT;
  uint8_t* sQ = smem;
  uint8_t* sdO = smem + L::OFF_DO;
  uint8_t* ring = smem + L::OFF_RING;
  uint8_t* sdS = smem + L::OFF_DS;  // [buf][hi, lo]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* qfull = bars;
  uint64_t* full = bars + 1;        // [NS]
  uint64_t* empty = full + NS;      // [NS]
  uint64_t* t_full = empty + NS;    // [2] S and dP of a step
  uint64_t* t_empty = t_full + 2;   // [2]
  uint64_t* d_full = t_empty + 2;   // [2] dS written
  uint64_t* d_empty = d_full + 2;   // [2]
  uint64_t* acc_full = d_empty + 2;
  uint64_t* drain = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* skip_flag = tmem_slot + 2;

  const int warp = (int)warp_id(), lane = (int)lane_id();
  const int S = a.S;
  const int g = h / (a.nh / a.nkv);
  const int64_t row0 = (int64_t)b * S + (int64_t)qt * kBig;
  const int qend = min(S, (qt + 1) * kBig);
  const int J = (qend + kStep - 1) / kStep;
  constexpr uint32_t TM_S = 0, TM_DP = 2 * kStep, TM_DQ = 4 * kStep;
  constexpr uint32_t TM_COLS = 512;

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    *skip_flag = (*(volatile uint32_t*)&g_dev_error != 0u) ? 1u : 0u;
    mbar_init(qfull, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&t_full[i], 1);
      mbar_init(&t_empty[i], 4);
      mbar_init(&d_full[i], 4);
      mbar_init(&d_empty[i], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_launch_dependents();
  const bool run = *skip_flag == 0u;

  if (warp == 0) {
    if (lane == 0 && run) {
      mbar_arrive_expect_tx(qfull, 2 * L::Q);
#pragma unroll
      for (int bx = 0; bx < D / 64; ++bx) {
        tma_load_2d(sQ + bx * kBig * 128, &a.tq, qfull, h * D + bx * 64, (int)row0);
        tma_load_2d(sdO + bx * kBig * 128, &a.tdo, qfull, h * D + bx * 64, (int)row0);
      }
      int n = 0;
      bool ok = true;
      for (int j = 0; j < J && ok; ++j)
        for (int w = 0; w < 2 && ok; ++w) {  // K_j then V_j
          const int st = n % NS;
          if (*abort_flag ||
              !mbar_wait(&empty[st], ((uint32_t)(n / NS) & 1u) ^ 1u, DERR_TIMEOUT_EMPTY)) {
            *abort_flag = 1u;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[st], L::T);
          const int y = (int)((int64_t)b * S + (int64_t)j * kStep);
#pragma unroll
          for (int bx = 0; bx < D / 64; ++bx)
            tma_load_2d(ring + st * L::T + bx * kStep * 128, w == 0 ? &a.tk : &a.tv, &full[st],
                        g * D + bx * 64, y);
          ++n;
        }
      for (int i = (n > NS ? n - NS : 0); i < n; ++i)
        mbar_wait(&full[i % NS], (uint32_t)(i / NS) & 1u, DERR_TIMEOUT_DRAIN);
      mbar_wait(qfull, 0u, DERR_TIMEOUT_DRAIN);
    }
  } else if (warp == 1) {
    if (lane == 0 && run) {
      constexpr uint32_t idT = idesc_bf16_f32(kBig, kStep, 0u);
      constexpr uint32_t idQ = idesc_bf16_f32(kBig, D, 1u);
      const uint32_t aQ = smem_u32(sQ), adO = smem_u32(sdO);
      bool ok = mbar_wait(qfull, 0u, DERR_TIMEOUT_FULL);
      auto wait_full = [&](int n) {
        const int st = n % NS;
        if (*abort_flag || !mbar_wait(&full[st], (uint32_t)(n / NS) & 1u, DERR_TIMEOUT_FULL)) {
          *abort_flag = 1u;
          return -1;
        }
        tc_fence_after();
        return st;
      };
      // S_j and dP_j into buffer j & 1; V_j's slot is released at once, K_j's
      // after dQ_j has read it.
      auto issue_T = [&](int j) {
        const int sb = j & 1;
        if (*abort_flag ||
            !mbar_wait(&t_empty[sb], ((uint32_t)(j >> 1) & 1u) ^ 1u, DERR_TIMEOUT_EMPTY)) {
          *abort_flag = 1u;
          return false;
        }
        const int sk = wait_full(2 * j);
        if (sk < 0) return false;
        const uint32_t bK = smem_u32(ring + sk * L::T);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          tc_mma_f16(tmem + TM_S + sb * kStep, kmaj_desc(aQ, kBig, ks), kmaj_desc(bK, kStep, ks),
                     idT, ks > 0 ? 1u : 0u);
        const int sv = wait_full(2 * j + 1);
        if (sv < 0) return false;
        const uint32_t bV = smem_u32(ring + sv * L::T);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          tc_mma_f16(tmem + TM_DP + sb * kStep, kmaj_desc(adO, kBig, ks),
                     kmaj_desc(bV, kStep, ks), idT, ks > 0 ? 1u : 0u);
        tc_commit(&empty[sv]);
        tc_commit(&t_full[sb]);
        return true;
      };
      if (ok) ok = issue_T(0);
      for (int j = 0; j < J && ok; ++j) {
        if (j + 1 < J && !(ok = issue_T(j + 1))) break;
        const int db = j & 1;
        if (*abort_flag || !mbar_wait(&d_full[db], (uint32_t)(j >> 1) & 1u, DERR_TIMEOUT_BFULL)) {
          *abort_flag = 1u;
          break;
        }
        tc_fence_after();
        const int sk = (2 * j) % NS;
        const uint32_t bK = smem_u32(ring + sk * L::T);
        const uint32_t aHi = smem_u32(sdS + (2 * db) * L::P);
        const uint32_t aLo = smem_u32(sdS + (2 * db + 1) * L::P);
#pragma unroll
        for (int ks = 0; ks < kStep / 16; ++ks)
          tc_mma_f16(tmem + TM_DQ, kmaj_desc(aHi, kBig, ks), mn_desc(bK, ks), idQ,
                     (j > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < kStep / 16; ++ks)
          tc_mma_f16(tmem + TM_DQ, kmaj_desc(aLo, kBig, ks), mn_desc(bK, ks), idQ, 1u);
        tc_commit(&empty[sk]);
        tc_commit(&d_empty[db]);
      }
      tc_commit(acc_full);
      tc_commit(drain);
      mbar_wait(drain, 0u, DERR_TIMEOUT_DRAIN);
    }
  } else if (run) {
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int qi = qt * kBig + r;
    const int64_t row = row0 + r;
    const bool valid = qi < S && row < a.M;
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    const int64_t ld = (int64_t)a.nh * D;
    // this row's D_i = dO_i . O_i and log-sum-exp (base 2)
    float Di = 0.0f, lse2 = 0.0f;
    if (valid) {
      Di = a.Dvec[(int64_t)h * a.M + row];
      lse2 = a.lse[(int64_t)h * a.M + row] * kLog2e;
    }
    const float sl2 = a.sl2;
    bool ok = true;
    for (int j = 0; j < J; ++j) {
      const int sb = j & 1;
      if (!warp_all(!*abort_flag &&
                    mbar_wait(&t_full[sb], (uint32_t)(j >> 1) & 1u, DERR_TIMEOUT_ACC) &&
                    mbar_wait(&d_empty[sb], ((uint32_t)(j >> 1) & 1u) ^ 1u,
                                      DERR_TIMEOUT_BEMPTY))) {
        *abort_flag = 1u;
        ok = false;
        break;
      }
      tc_fence_after();
      float s[kStep], dp[kStep];
      tmem_row64(trow + TM_S + sb * kStep, s);
      tmem_row64(trow + TM_DP + sb * kStep, dp);
      tc_fence_before();
#pragma unroll
      for (int c = 0; c < kStep; ++c) {
        // rows past the sequence hold no query: zero, so nothing overflows
        const float p = (!valid || j * kStep + c > qi) ? 0.0f : ex2(s[c] * sl2 - lse2);
        s[c] = p * (dp[c] - Di);
      }
      put_row_hilo(sdS + (2 * sb) * L::P, sdS + (2 * sb + 1) * L::P, r, s);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&t_empty[sb]);
        mbar_arrive(&d_full[sb]);
      }
    }
    if (warp_all(ok && mbar_wait_backoff(acc_full, 0u, DERR_TIMEOUT_ACC) && !*abort_flag)) {
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < D; cc += 32) {
        uint32_t acc[32];
        tmem_ld_32x32b_x32(trow + TM_DQ + cc, acc);
        tmem_ld_wait();
        if (!valid) continue;
        uint16_t* dst = a.dq + row * ld + h * D + cc;
        const float sc = a.scale;
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack_bf16x2(sc * __uint_as_float(acc[2 * e]), sc * __uint_as_float(acc[2 * e + 1]));
        if ((reinterpret_cast<uintptr_t>(a.dq) & 31u) == 0u && (ld & 15) == 0) {
          // whole 32-byte sectors per store
          st_global_v8(dst, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
          st_global_v8(dst + 16, pk[8], pk[9], pk[10], pk[11], pk[12], pk[13], pk[14], pk[15]);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            *reinterpret_cast<uint4*>(dst + 8 * e) = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TM_COLS);
}

// ------------------------------------------------------------------------- backward: dK, dV
struct AttnDkvArgs {
  CUtensorMap tk;   // k [M, nkv*D], box {64, 128}
  CUtensorMap tv;   // v [M, nkv*D], box {64, 128}
  CUtensorMap tq;   // q [M, nh*D], box {64, 64}
  CUtensorMap tdo;  // dO [M, nh*D], box {64, 64}
  int S, nh, nkv;
  int64_t M;
  float sl2, scale;
  const float* lse;   // [nh, M]
  const float* Dvec;  // [nh, M]
  float* dk_part;     // [nh, M, D] fp32: this query head's share of dk
  float* dv_part;     // [nh, M, D]
};

template <int D>
struct DkvSmem {
  static constexpr uint32_t KT = kBig * D * 2;   // K or V tile
  static constexpr uint32_t T = kStep * D * 2;   // Q or dO step tile
  static constexpr int NSTAGE = 2;
  static constexpr uint32_t STAGE = 2 * T;       // Q_i and dO_i
  static constexpr uint32_t P = kBig * kStep * 2;
  static constexpr uint32_t OFF_V = KT;
  static constexpr uint32_t OFF_RING = 2 * KT;
  static constexpr uint32_t OFF_PD = OFF_RING + NSTAGE * STAGE;  // P^T hi, lo, dS^T hi, lo
  static constexpr uint32_t OFF_BAR = OFF_PD + 4 * P;
  static constexpr uint32_t BYTES = OFF_BAR + 256 + 1024;
};

// dK, dV shares of one query head for one (128 keys, head, sequence) tile.
template <int D>
WS_DEVINL void attn_dkv_tile(const AttnDkvArgs& a, uint8_t* smem, int kt, int h, int b) {
  using L = DkvSmem<D>;
  constexpr int NS = L::NSTAGE;
  uint8_t* sK = smem;
  uint8_t* sV = smem + L::OFF_V;
  uint8_t* ring = smem + L::OFF_RING;
  uint8_t* sPD = smem + L::OFF_PD;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* kvfull = bars;
  uint64_t* full = bars + 1;        // [NS]
  uint64_t* empty = full + NS;      // [NS]
  uint64_t* t_full = empty + NS;    // [2] S^T and dP^T of a step
  uint64_t* t_empty = t_full + 2;   // [2]
  uint64_t* pd_full = t_empty + 2;  // P^T and dS^T written
  uint64_t* pd_empty = pd_full + 1;
  uint64_t* acc_full = pd_empty + 1;
  uint64_t* drain = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* skip_flag = tmem_slot + 2;

  const int warp = (int)warp_id(), lane = (int)lane_id();
  const int S = a.S;
  const int g = h / (a.nh / a.nkv);
  const int64_t krow0 = (int64_t)b * S + (int64_t)kt * kBig;
  const int i0 = kt * kBig / kStep;                  // first query step that sees these keys
  const int nsteps = (S + kStep - 1) / kStep - i0;   // query steps
  constexpr uint32_t TM_S = 0, TM_DP = 2 * kStep, TM_DV = 4 * kStep, TM_DK = 4 * kStep + D;
  constexpr uint32_t TM_COLS = 512;
  static_assert(TM_DK + D <= TM_COLS, "tensor memory");

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    *skip_flag = (*(volatile uint32_t*)&g_dev_error != 0u) ? 1u : 0u;
    mbar_init(kvfull, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&t_full[i], 1);
      mbar_init(&t_empty[i], 4);
    }
    mbar_init(pd_full, 4);
    mbar_init(pd_empty, 1);
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_launch_dependents();
  const bool run = *skip_flag == 0u && nsteps > 0;

  if (warp == 0) {
    if (lane == 0 && run) {
      mbar_arrive_expect_tx(kvfull, 2 * L::KT);
#pragma unroll
      for (int bx = 0; bx < D / 64; ++bx) {
        tma_load_2d(sK + bx * kBig * 128, &a.tk, kvfull, g * D + bx * 64, (int)krow0);
        tma_load_2d(sV + bx * kBig * 128, &a.tv, kvfull, g * D + bx * 64, (int)krow0);
      }
      int n = 0;
      for (int s = 0; s < nsteps; ++s) {
        const int st = s % NS;
        if (*abort_flag ||
            !mbar_wait(&empty[st], ((uint32_t)(s / NS) & 1u) ^ 1u, DERR_TIMEOUT_EMPTY)) {
          *abort_flag = 1u;
          break;
        }
        mbar_arrive_expect_tx(&full[st], L::STAGE);
        const int y = (int)((int64_t)b * S + (int64_t)(i0 + s) * kStep);
        uint8_t* dst = ring + st * L::STAGE;
#pragma unroll
        for (int bx = 0; bx < D / 64; ++bx) {
          tma_load_2d(dst + bx * kStep * 128, &a.tq, &full[st], h * D + bx * 64, y);
          tma_load_2d(dst + L::T + bx * kStep * 128, &a.tdo, &full[st], h * D + bx * 64, y);
        }
        n = s + 1;
      }
      for (int i = (n > NS ? n - NS : 0); i < n; ++i)
        mbar_wait(&full[i % NS], (uint32_t)(i / NS) & 1u, DERR_TIMEOUT_DRAIN);
      mbar_wait(kvfull, 0u, DERR_TIMEOUT_DRAIN);
    }
  } else if (warp == 1) {
    if (lane == 0 && run) {
      constexpr uint32_t idT = idesc_bf16_f32(kBig, kStep, 0u);
      constexpr uint32_t idG = idesc_bf16_f32(kBig, D, 1u);
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV);
      bool ok = mbar_wait(kvfull, 0u, DERR_TIMEOUT_FULL);
      auto issue_T = [&](int s) {
        const int sb = s & 1, st = s % NS;
        if (*abort_flag ||
            !mbar_wait(&t_empty[sb], ((uint32_t)(s >> 1) & 1u) ^ 1u, DERR_TIMEOUT_EMPTY) ||
            !mbar_wait(&full[st], (uint32_t)(s / NS) & 1u, DERR_TIMEOUT_FULL)) {
          *abort_flag = 1u;
          return false;
        }
        tc_fence_after();
        const uint32_t bQ = smem_u32(ring + st * L::STAGE);
        const uint32_t bdO = bQ + L::T;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          tc_mma_f16(tmem + TM_S + sb * kStep, kmaj_desc(aK, kBig, ks), kmaj_desc(bQ, kStep, ks),
                     idT, ks > 0 ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          tc_mma_f16(tmem + TM_DP + sb * kStep, kmaj_desc(aV, kBig, ks),
                     kmaj_desc(bdO, kStep, ks), idT, ks > 0 ? 1u : 0u);
        tc_commit(&t_full[sb]);
        return true;
      };
      if (ok) ok = issue_T(0);
      for (int s = 0; s < nsteps && ok; ++s) {
        if (s + 1 < nsteps && !(ok = issue_T(s + 1))) break;
        if (*abort_flag || !mbar_wait(pd_full, (uint32_t)s & 1u, DERR_TIMEOUT_BFULL)) {
          *abort_flag = 1u;
          break;
        }
        tc_fence_after();
        const int st = s % NS;
        const uint32_t bQ = smem_u32(ring + st * L::STAGE);
        const uint32_t bdO = bQ + L::T;
        const uint32_t pb = smem_u32(sPD);
#pragma unroll
        for (int ks = 0; ks < kStep / 16; ++ks)
          tc_mma_f16(tmem + TM_DV, kmaj_desc(pb, kBig, ks), mn_desc(bdO, ks), idG,
                     (s > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < kStep / 16; ++ks)
          tc_mma_f16(tmem + TM_DV, kmaj_desc(pb + L::P, kBig, ks), mn_desc(bdO, ks), idG, 1u);
#pragma unroll
        for (int ks = 0; ks < kStep / 16; ++ks)
          tc_mma_f16(tmem + TM_DK, kmaj_desc(pb + 2 * L::P, kBig, ks), mn_desc(bQ, ks), idG,
                     (s > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < kStep / 16; ++ks)
          tc_mma_f16(tmem + TM_DK, kmaj_desc(pb + 3 * L::P, kBig, ks), mn_desc(bQ, ks), idG, 1u);
        tc_commit(&empty[st]);
        tc_commit(pd_empty);
      }
      tc_commit(acc_full);
      tc_commit(drain);
      mbar_wait(drain, 0u, DERR_TIMEOUT_DRAIN);
    }
  } else if (run) {
    // ---- thread <-> key row r of the tile; columns are this step's queries
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int kj = kt * kBig + r;         // local key index
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    const float sl2 = a.sl2;
    bool ok = true;
    for (int s = 0; s < nsteps; ++s) {
      const int sb = s & 1;
      const int qb = (i0 + s) * kStep;    // local index of this step's first query
      // this step's lse2 and D values: lane l holds columns l and 32 + l
      float lse_c[2], D_c[2];
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const int c = w * 32 + lane;
        const int64_t qrow = (int64_t)b * S + qb + c;
        const bool in = qb + c < S && qrow < a.M;
        lse_c[w] = in ? a.lse[(int64_t)h * a.M + qrow] * kLog2e : 0.0f;
        D_c[w] = in ? a.Dvec[(int64_t)h * a.M + qrow] : 0.0f;
      }
      if (!warp_all(!*abort_flag &&
                    mbar_wait(&t_full[sb], (uint32_t)(s >> 1) & 1u, DERR_TIMEOUT_ACC) &&
                    mbar_wait(pd_empty, ((uint32_t)s & 1u) ^ 1u, DERR_TIMEOUT_BEMPTY))) {
        *abort_flag = 1u;
        ok = false;
        break;
      }
      tc_fence_after();
      float st_[kStep], dp[kStep];
      tmem_row64(trow + TM_S + sb * kStep, st_);
      tmem_row64(trow + TM_DP + sb * kStep, dp);
      tc_fence_before();
#pragma unroll
      for (int c = 0; c < kStep; ++c) {
        const int qi = qb + c;
        const float l2 = __shfl_sync(0xffffffffu, lse_c[c >> 5], c & 31);
        const float Dq = __shfl_sync(0xffffffffu, D_c[c >> 5], c & 31);
        const float p = (kj > qi || qi >= S) ? 0.0f : ex2(st_[c] * sl2 - l2);
        st_[c] = p;
        dp[c] = p * (dp[c] - Dq);
      }
      put_row_hilo(sPD, sPD + L::P, r, st_);
      put_row_hilo(sPD + 2 * L::P, sPD + 3 * L::P, r, dp);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&t_empty[sb]);
        mbar_arrive(pd_full);
      }
    }
    if (warp_all(ok && mbar_wait_backoff(acc_full, 0u, DERR_TIMEOUT_ACC) && !*abort_flag)) {
      tc_fence_after();
      const int64_t row = krow0 + r;
      const bool valid = kj < S && row < a.M;
      float* dkp = a.dk_part + ((int64_t)h * a.M + row) * D;
      float* dvp = a.dv_part + ((int64_t)h * a.M + row) * D;
#pragma unroll
      for (int cc = 0; cc < D; cc += 32) {
        uint32_t av[32], ak[32];
        tmem_ld_32x32b_x32(trow + TM_DV + cc, av);
        tmem_ld_32x32b_x32(trow + TM_DK + cc, ak);
        tmem_ld_wait();
        if (!valid) continue;
        if ((reinterpret_cast<uintptr_t>(a.dk_part) & 31u) != 0u) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            *reinterpret_cast<float4*>(dvp + cc + e) =
                make_float4(__uint_as_float(av[e]), __uint_as_float(av[e + 1]),
                            __uint_as_float(av[e + 2]), __uint_as_float(av[e + 3]));
            *reinterpret_cast<float4*>(dkp + cc + e) = make_float4(
                a.scale * __uint_as_float(ak[e]), a.scale * __uint_as_float(ak[e + 1]),
                a.scale * __uint_as_float(ak[e + 2]), a.scale * __uint_as_float(ak[e + 3]));
          }
          continue;
        }
        // whole 32-byte sectors per store (rows of D fp32 values keep the
        // 32-byte alignment of the workspace)
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          st_global_v8(dvp + cc + e, av[e], av[e + 1], av[e + 2], av[e + 3], av[e + 4], av[e + 5],
                       av[e + 6], av[e + 7]);
          st_global_v8(dkp + cc + e, __float_as_uint(a.scale * __uint_as_float(ak[e])),
                       __float_as_uint(a.scale * __uint_as_float(ak[e + 1])),
                       __float_as_uint(a.scale * __uint_as_float(ak[e + 2])),
                       __float_as_uint(a.scale * __uint_as_float(ak[e + 3])),
                       __float_as_uint(a.scale * __uint_as_float(ak[e + 4])),
                       __float_as_uint(a.scale * __uint_as_float(ak[e + 5])),
                       __float_as_uint(a.scale * __uint_as_float(ak[e + 6])),
                       __float_as_uint(a.scale * __uint_as_float(ak[e + 7])));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TM_COLS);
}

// Both backward roles in one launch, so the two halves of the backward
// share the machine: head h = blockIdx.x (fastest), sequence blockIdx.z, and
// blockIdx.y = 2p + role: role 0 the dQ tile ntiles - 1 - p, role 1 the
// dK/dV tile p.  The longest tiles of both roles (the last queries, the
// first keys) come first.
struct AttnBwdArgs {
  AttnDqArgs dq;
  AttnDkvArgs dkv;
  int ntiles;
};

template <int D>
constexpr uint32_t bwd_smem_bytes() {
  return DqSmem<D>::BYTES > DkvSmem<D>::BYTES ? DqSmem<D>::BYTES : DkvSmem<D>::BYTES;
}

template <int D>
__global__ void __launch_bounds__(kAtThreads, 1) k_attn_bwd(const __grid_constant__ AttnBwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int y = (int)blockIdx.y, h = (int)blockIdx.x, b = (int)blockIdx.z;
  if ((y & 1) == 0)
    attn_dq_tile<D>(a.dq, smem, a.ntiles - 1 - (y >> 1), h, b);
  else
    attn_dkv_tile<D>(a.dkv, smem, y >> 1, h, b);
}

// Dvec[h, m] = dO[m, h*D ..] . o32[m, h*D ..] for every token and head, one
// warp per (token, head): lane l takes columns l, l + 32, ..., then a fixed
// butterfly sum.
__global__ void k_attn_dvec(const uint16_t* __restrict__ dO, const float* __restrict__ o32,
                            int64_t M, int nh, int D, float* __restrict__ Dvec) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  const int lane = (int)(threadIdx.x & 31);
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; w < M * nh;
       w += warps) {
    const int64_t m = w / nh;
    const int h = (int)(w % nh);
    const uint16_t* pd = dO + (m * nh + h) * D;
    const float* po = o32 + (m * nh + h) * D;
    float acc = 0.0f;
    for (int c = lane; c < D; c += 32) acc = fmaf(bf16_bits_to_f32(pd[c]), po[c], acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) Dvec[(int64_t)h * M + m] = acc;
  }
}

// dk[m, g*D + c] = bf16(sum over the rep query heads h of group g, in head
// order, of dk_part[h, m, c]); the same for dv.  4 columns per thread.
__global__ void k_attn_group_sum(const float* __restrict__ dk_part,
                                 const float* __restrict__ dv_part, int64_t M, int nkv, int rep,
                                 int D, uint16_t* __restrict__ dk, uint16_t* __restrict__ dv) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t n4 = M * nkv * D / 4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = i * 4;
    const int64_t m = e / ((int64_t)nkv * D);
    const int col = (int)(e % ((int64_t)nkv * D));
    const int g = col / D, c = col % D;
    float4 sk = make_float4(0.f, 0.f, 0.f, 0.f), sv = sk;
    for (int t = 0; t < rep; ++t) {
      const int64_t o = ((int64_t)(g * rep + t) * M + m) * D + c;
      const float4 k4 = *reinterpret_cast<const float4*>(dk_part + o);
      const float4 v4 = *reinterpret_cast<const float4*>(dv_part + o);
      sk = make_float4(sk.x + k4.x, sk.y + k4.y, sk.z + k4.z, sk.w + k4.w);
      sv = make_float4(sv.x + v4.x, sv.y + v4.y, sv.z + v4.z, sv.w + v4.w);
    }
    *reinterpret_cast<uint2*>(dk + e) = make_uint2(pack_bf16x2(sk.x, sk.y), pack_bf16x2(sk.z, sk.w));
    *reinterpret_cast<uint2*>(dv + e) = make_uint2(pack_bf16x2(sv.x, sv.y), pack_bf16x2(sv.z, sv.w));
  }
}

template <class F>
cudaError_t smem_attr_once(F* fn, uint32_t bytes) {
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

bool maps_for(CUtensorMap* m, const void* base, int64_t M, int64_t width, uint32_t rows) {
  return tmap_bf16_sw128(m, base, (uint64_t)width, (uint64_t)M, (uint64_t)width * 2, 64, rows);
}

}  // namespace

size_t attn_bwd_workspace_bytes(int64_t M, int nh, int head_dim) {
  // dk, dv partials [nh, M, D] fp32 each, then D [nh, M]
  return 2 * (size_t)nh * (size_t)M * (size_t)head_dim * 4 + (size_t)nh * (size_t)M * 4 + 256;
}

cudaError_t run_attn_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, int n_seq,
                         int S, int nh, int nkv, int hd, uint16_t* o, float* o32, float* lse,
                         cudaStream_t st) {
  const int64_t M = (int64_t)n_seq * S;
  AttnFwdArgs a;
  if (!maps_for(&a.tq, q, M, (int64_t)nh * hd, kBig) ||
      !maps_for(&a.tk, k, M, (int64_t)nkv * hd, kStep) ||
      !maps_for(&a.tv, v, M, (int64_t)nkv * hd, kStep))
    return cudaErrorInvalidValue;
  a.S = S;
  a.nh = nh;
  a.nkv = nkv;
  a.M = M;
  a.sl2 = kLog2e / sqrtf((float)hd);
  a.o = o;
  a.o32 = o32;
  a.lse = lse;
  const dim3 grid((unsigned)nh, (unsigned)((S + kBig - 1) / kBig), (unsigned)n_seq);
  note_launch();
  if (hd == 128) {
    static const cudaError_t e = smem_attr_once(k_attn_fwd<128>, FwdSmem<128>::BYTES);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_attn_fwd<128>, grid, dim3(kAtThreads), FwdSmem<128>::BYTES, st, a);
  }
  static const cudaError_t e = smem_attr_once(k_attn_fwd<64>, FwdSmem<64>::BYTES);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_attn_fwd<64>, grid, dim3(kAtThreads), FwdSmem<64>::BYTES, st, a);
}

cudaError_t run_attn_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const float* o32, const float* lse, const uint16_t* dO, int n_seq, int S,
                         int nh, int nkv, int hd, uint16_t* dq, uint16_t* dk, uint16_t* dv,
                         void* ws, cudaStream_t st) {
  const int64_t M = (int64_t)n_seq * S;
  float* dk_part = static_cast<float*>(ws);
  float* dv_part = dk_part + (size_t)nh * M * hd;
  float* Dvec = dv_part + (size_t)nh * M * hd;
  const float sl2 = kLog2e / sqrtf((float)hd);
  const float scale = 1.0f / sqrtf((float)hd);
  AttnDqArgs a;
  if (!maps_for(&a.tq, q, M, (int64_t)nh * hd, kBig) ||
      !maps_for(&a.tdo, dO, M, (int64_t)nh * hd, kBig) ||
      !maps_for(&a.tk, k, M, (int64_t)nkv * hd, kStep) ||
      !maps_for(&a.tv, v, M, (int64_t)nkv * hd, kStep))
    return cudaErrorInvalidValue;
  a.S = S;
  a.nh = nh;
  a.nkv = nkv;
  a.M = M;
  a.sl2 = sl2;
  a.scale = scale;
  a.lse = lse;
  a.Dvec = Dvec;
  a.dq = dq;
  AttnDkvArgs c;
  if (!maps_for(&c.tk, k, M, (int64_t)nkv * hd, kBig) ||
      !maps_for(&c.tv, v, M, (int64_t)nkv * hd, kBig) ||
      !maps_for(&c.tq, q, M, (int64_t)nh * hd, kStep) ||
      !maps_for(&c.tdo, dO, M, (int64_t)nh * hd, kStep))
    return cudaErrorInvalidValue;
  c.S = S;
  c.nh = nh;
  c.nkv = nkv;
  c.M = M;
  c.sl2 = sl2;
  c.scale = scale;
  c.lse = lse;
  c.Dvec = Dvec;
  c.dk_part = dk_part;
  c.dv_part = dv_part;
  const int ntiles = (S + kBig - 1) / kBig;
  AttnBwdArgs ab;
  ab.dq = a;
  ab.dkv = c;
  ab.ntiles = ntiles;
  cudaError_t e;
  {
    const int64_t pairs = M * nh;
    const unsigned blocks = (unsigned)std::min<int64_t>((pairs + 7) / 8, 8 * 152);
    note_launch();
    e = launch_pdl(k_attn_dvec, dim3(blocks), dim3(256), 0, st, dO, o32, M, nh, hd, Dvec);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid((unsigned)nh, (unsigned)(2 * ntiles), (unsigned)n_seq);
  note_launch();
  if (hd == 128) {
    static const cudaError_t e1 = smem_attr_once(k_attn_bwd<128>, bwd_smem_bytes<128>());
    if (e1 != cudaSuccess) return e1;
    e = launch_pdl(k_attn_bwd<128>, grid, dim3(kAtThreads), bwd_smem_bytes<128>(), st, ab);
  } else {
    static const cudaError_t e1 = smem_attr_once(k_attn_bwd<64>, bwd_smem_bytes<64>());
    if (e1 != cudaSuccess) return e1;
    e = launch_pdl(k_attn_bwd<64>, grid, dim3(kAtThreads), bwd_smem_bytes<64>(), st, ab);
  }
  if (e != cudaSuccess) return e;
  const int64_t n4 = M * nkv * hd / 4;
  const int threads = 256;
  const unsigned blocks = (unsigned)std::min<int64_t>((n4 + threads - 1) / threads, 4 * 152);
  note_launch();
  return launch_pdl(k_attn_group_sum, dim3(blocks), dim3(threads), 0, st,
                    (const float*)dk_part, (const float*)dv_part, M, nkv, nh / nkv, hd, dk, dv);
}

}  // namespace ws
