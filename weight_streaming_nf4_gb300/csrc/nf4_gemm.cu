// nf4_gemm.cu -- the NF4 dequant GEMM on the 5th-generation tensor cores.
//
// Forward (a2):  y[M,N]  = x[M,K] . W'[N,K]^T  (+ s U B^T as an extra step)
// Backward (a4): dX[M,K] = dY[M,N] . W'[N,K]   (+ s (G A) . mask)
//
// W' = bf16_RN(c[code] * absmax) is never materialised in global memory:
// packed 4-bit codes and the block absmax are staged into shared memory by
// TMA, dequantised by eight producer warps straight into the 128-byte
// swizzled operand layout the tensor cores read, and consumed by
// tcgen05.mma (bf16 x bf16 -> fp32 in TMEM) issued by one thread.
//
// Persistent CTA (one per SM) = 14 warps:
//   warp 0      TMA producer (activation tile + code tile + absmax tile)
//   warp 1      TMEM allocator and MMA issuer
//   warps 2-9   dequant producers
//   warps 10-13 epilogue (TMEM -> registers -> global), one TMEM lane
//               quarter per warp, overlapping the next tile's main loop
// Tile: 128*UM rows of activations (UM tensor-core atoms of M = 128 sharing
// one dequantised weight tile), BN output columns, 64-deep contraction steps.
//
// Schedule: the (tile, step) iterations of the whole problem are cut into
// gridDim.x equal contiguous ranges, one per CTA (stream-K).  A tile that a
// range boundary cuts is finished by a fixed-order fix-up kernel that adds
// the CTAs' fp32 partial tiles in step order; every other tile is written
// by its CTA's epilogue.  The cut points depend only on the shape and the
// grid size, so results are deterministic and identical run to run.  No
// atomics anywhere.
//
// The LoRA terms use the same tensor cores: the forward appends one 64-deep
// step whose A operand is [U_hi | U_lo | U_hi | 0] and whose B operand is
// [Bs_hi | Bs_hi | Bs_lo | 0] (Bs = s B, bf16 high/low splits), i.e.
// U Bs^T to about 16 significant bits.  The backward computes s G A the same
// way into a second TMEM accumulator and adds it under the dropout mask in
// the epilogue.
#define WS_GEMM_TU 1
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace ws {

cudaError_t read_and_clear_dev_error(uint32_t* flags) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(flags, g_dev_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  const uint32_t zero = 0;
  return cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(uint32_t));
}

__constant__ float c_nf4_levels[16] = {-1.0f,    -0.6962f, -0.5251f, -0.3949f,
                                       -0.2844f, -0.1848f, -0.0911f, 0.0f,
                                       0.0796f,  0.1609f,  0.2461f,  0.3379f,
                                       0.4407f,  0.5626f,  0.7230f,  1.0f};

namespace {

constexpr int kDqWarps = 8;
constexpr int kEpiWarps = 4;
constexpr int kThreads = (2 + kDqWarps + kEpiWarps) * 32;
constexpr int kDqThreads = kDqWarps * 32;

template <bool BWD, int UM, int BN>
struct Cfg {
  static constexpr int BM = 128 * UM;
  static constexpr uint32_t A_BYTES = BM * 128;   // BM rows x 64 bf16
  static constexpr uint32_t B_BYTES = BN * 128;   // BN x 64 bf16
  static constexpr uint32_t C_BYTES = BN * 32;    // codes: BN x 64 nibbles
  static constexpr uint32_t S_BYTES = BN * 4;     // absmax: BN floats
  static constexpr int BSTAGES = 2;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + C_BYTES + S_BYTES;
  static constexpr int STAGES_RAW =
      (int)((220u * 1024u - BSTAGES * B_BYTES - 1024u) / STAGE_BYTES);
  static constexpr int STAGES = STAGES_RAW > 4 ? 4 : STAGES_RAW;
  // one accumulator set: D (and for the backward the LoRA term D2)
  static constexpr uint32_t ACC_COLS = (BWD ? 2u : 1u) * UM * BN;
  // double-buffer the accumulator when TMEM has room, so the epilogue of
  // one tile overlaps the main loop of the next
  static constexpr int ACC_BUFS = 2 * ACC_COLS <= 512 ? 2 : 1;
  static constexpr uint32_t TMEM_COLS = ACC_COLS * ACC_BUFS;
  static constexpr int64_t TILE_FLOATS = (int64_t)BM * BN;
  // MN-major operand (backward): 64-element MN groups LBO apart, 8-row K
  // groups SBO apart.
  static constexpr uint32_t MN_LBO = 1024;
  static constexpr uint32_t MN_SBO = (BN / 64) * 1024;
  static constexpr uint32_t OFF_A = 0;
  static constexpr uint32_t OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr uint32_t OFF_C = OFF_B + BSTAGES * B_BYTES;
  static constexpr uint32_t OFF_S = OFF_C + STAGES * C_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_S + STAGES * S_BYTES;
  static constexpr uint32_t N_BARS = 2 * STAGES + 2 * BSTAGES + 2 * ACC_BUFS + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + N_BARS * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 1024;  // + alignment slack
  static_assert(STAGES >= 2, "pipeline needs two stages");
  static_assert(TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM columns");
  static_assert(SMEM_BYTES <= 227u * 1024u, "shared memory");
  static_assert(BN == 128 || BN == 256, "BN");
};

// CTA of the stream-K schedule that owns iteration i: ranges are
// [floor(g*I/G), floor((g+1)*I/G)), so g = ceil((i+1)*G/I) - 1.
__host__ __device__ inline int64_t sk_cta_of(int64_t i, int64_t I, int64_t G) {
  return ((i + 1) * G + I - 1) / I - 1;
}
__host__ __device__ inline int64_t sk_begin(int64_t g, int64_t I, int64_t G) { return g * I / G; }

WS_DEVINL void sts128(uint8_t* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4*>(p) = make_uint4(a, b, c, d);
}

// Dequantise 4 code bytes (8 consecutive weights along k) into a 16-byte
// chunk of bf16 values: element 2i from the high nibble of byte i, element
// 2i+1 from its low nibble.
// Two IEEE fp32 products (round to nearest) in one packed instruction.
WS_DEVINL void mul2_rn(float x0, float x1, float s, float& r0, float& r1) {
  asm("{\n .reg .b64 pa, pb, pd;\n mov.b64 pa, {%2, %3};\n mov.b64 pb, {%4, %4};\n"
      " mul.rn.f32x2 pd, pa, pb;\n mov.b64 {%0, %1}, pd;\n}"
      : "=f"(r0), "=f"(r1)
      : "f"(x0), "f"(x1), "f"(s));
}

WS_DEVINL uint4 dq8(uint32_t w, float a, const float* lv) {
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t byte = (w >> (8 * i)) & 0xFFu;
    float v0, v1;
    mul2_rn(lv[byte >> 4], lv[byte & 15u], a, v0, v1);
    o[i] = pack_bf16x2(v0, v1);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Forward weight tile, K-major 128B-swizzled: row j = output column n0 + j,
// 64 contraction elements; chunk cc of row j sits at (cc ^ (j & 7)) * 16.
template <int BN>
WS_DEVINL void dequant_fwd(const uint8_t* sC, const float* sS, uint8_t* sB, int t,
                           const float* lv) {
  if constexpr (BN == 256) {
    const int j = t;
    const uint4 c0 = *reinterpret_cast<const uint4*>(sC + j * 32);
    const uint4 c1 = *reinterpret_cast<const uint4*>(sC + j * 32 + 16);
    const float a = sS[j];
    const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    uint8_t* row = sB + j * 128;
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
      const uint4 v = dq8(words[cc], a, lv);
      sts128(row + ((cc ^ (j & 7)) << 4), v.x, v.y, v.z, v.w);
    }
  } else {
    const int j = t >> 1, half = t & 1;
    const uint4 c = *reinterpret_cast<const uint4*>(sC + j * 32 + half * 16);
    const float a = sS[j];
    const uint32_t words[4] = {c.x, c.y, c.z, c.w};
    uint8_t* row = sB + j * 128;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int cc = half * 4 + q;
      const uint4 v = dq8(words[q], a, lv);
      sts128(row + ((cc ^ (j & 7)) << 4), v.x, v.y, v.z, v.w);
    }
  }
}

// Backward weight tile, MN-major 128B-swizzled: the contraction runs over
// W's rows n (64 per step) and the output over W's columns k (BN per tile),
// so the tile keeps W's own orientation.  Element (k-col j, n-row c):
// group (c/8, j/64) at (c/8)*SBO + (j/64)*LBO, row c%8 inside the group,
// chunk ((j%64)/8) ^ (c%8).
template <int BN>
WS_DEVINL void dequant_bwd(const uint8_t* sC, const float* sS, uint8_t* sB, int t,
                           const float* lv) {
  using C = Cfg<true, 1, BN>;
  constexpr int SEGS = BN / 32;                  // 32-column segments per row
  constexpr int ITEMS = 64 * SEGS / kDqThreads;  // rows*segs per thread
#pragma unroll
  for (int it = 0; it < ITEMS; ++it) {
    const int item = t + it * kDqThreads;
    const int c = item / SEGS, seg = item % SEGS;
    const uint4 cw = *reinterpret_cast<const uint4*>(sC + c * (BN / 2) + seg * 16);
    const float a = sS[((seg * 32) / 64) * 64 + c];
    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
    const int mg = (seg * 32) / 64;
    uint8_t* grp = sB + (c >> 3) * C::MN_SBO + mg * C::MN_LBO + (c & 7) * 128;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int cc = ((seg * 32) % 64) / 8 + q;
      const uint4 v = dq8(words[q], a, lv);
      sts128(grp + ((cc ^ (c & 7)) << 4), v.x, v.y, v.z, v.w);
    }
  }
}

// The LoRA weight operand of the extra step, K-major like the forward
// tile: row j holds [Ws_hi(16) | Ws_hi(16) | Ws_lo(16) | 0(16)] with
// Ws = s * (row j of the LoRA factor).  Forward: factor row = B[n0+j, :];
// backward: factor row = A[:, n0+j] (column of A).
template <bool BWD, int BN>
WS_DEVINL void lora_tile(const float* F, int64_t rows_total, int64_t ld, int n0, float s,
                         uint8_t* sB, int t) {
  constexpr int TPR = kDqThreads / BN;  // threads per row: 1 (BN=256) or 2 (BN=128)
  const int j = t / TPR, part = t % TPR;
  const int64_t n = (int64_t)n0 + j;
  float v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float f = 0.0f;
    if (n < rows_total) f = BWD ? F[(int64_t)i * ld + n] : F[n * 16 + i];
    v[i] = s * f;
  }
  uint32_t hi[8], lo[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float h0 = bf16_lo(pack_bf16x2(v[2 * i], 0.0f));
    const float h1 = bf16_lo(pack_bf16x2(v[2 * i + 1], 0.0f));
    hi[i] = pack_bf16x2(h0, h1);
    lo[i] = pack_bf16x2(v[2 * i] - h0, v[2 * i + 1] - h1);
  }
  uint8_t* row = sB + j * 128;
#pragma unroll
  for (int q = 0; q < 8 / TPR; ++q) {
    const int cc = part * (8 / TPR) + q;
    uint4 val;
    if (cc == 0 || cc == 2) val = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    else if (cc == 1 || cc == 3) val = make_uint4(hi[4], hi[5], hi[6], hi[7]);
    else if (cc == 4) val = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    else if (cc == 5) val = make_uint4(lo[4], lo[5], lo[6], lo[7]);
    else val = make_uint4(0u, 0u, 0u, 0u);
    sts128(row + ((cc ^ (j & 7)) << 4), val.x, val.y, val.z, val.w);
  }
}

template <bool BWD, int UM, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    k_nf4_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmC,
               const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmL,
               const GemmArgs args) {
  using C = Cfg<BWD, UM, BN>;
  constexpr int STAGES = C::STAGES;
  constexpr int BSTAGES = C::BSTAGES;
  constexpr int NACC = C::ACC_BUFS;

  extern __shared__ uint8_t smem_raw[];
  __shared__ float s_lv[16];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + C::OFF_A;
  uint8_t* sB = smem + C::OFF_B;
  uint8_t* sC = smem + C::OFF_C;
  uint8_t* sS = smem + C::OFF_S;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = full + STAGES;
  uint64_t* bfull = empty + STAGES;
  uint64_t* bempty = bfull + BSTAGES;
  uint64_t* accfull = bempty + BSTAGES;
  uint64_t* accempty = accfull + NACC;
  uint64_t* drain = accempty + NACC;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  uint32_t* tmem_slot = misc;
  volatile uint32_t* abort_flag = misc + 1;
  volatile uint32_t* skip_flag = misc + 2;

  const int warp = (int)warp_id();
  const int lane = (int)lane_id();
  // ---- static stream-K schedule
  const int64_t S = (int64_t)args.nk_total + (args.has_lora ? 1 : 0);  // steps per tile
  const int64_t T = (int64_t)args.mtiles * args.ntiles;
  const int64_t I = T * S;
  const int64_t G = gridDim.x;
  const int64_t pb = sk_begin(blockIdx.x, I, G);
  const int64_t pe = sk_begin((int64_t)blockIdx.x + 1, I, G);

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    // an earlier kernel already gave up: do nothing rather than queue more work
    *skip_flag = (*(volatile uint32_t*)&g_dev_error != 0u || pe <= pb) ? 1u : 0u;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1 + kDqWarps);
    }
    for (int b = 0; b < BSTAGES; ++b) {
      mbar_init(&bfull[b], kDqWarps);
      mbar_init(&bempty[b], 1);
    }
    for (int a = 0; a < NACC; ++a) {
      mbar_init(&accfull[a], 1);
      mbar_init(&accempty[a], kEpiWarps);
    }
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (threadIdx.x < 16) s_lv[threadIdx.x] = c_nf4_levels[threadIdx.x];
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool skip = *skip_flag != 0u;

  if (!skip) {
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmC);
        tma_prefetch_desc(&tmS);
        if (args.has_lora) tma_prefetch_desc(&tmL);
        int64_t issued = 0;
        int s = 0;
        uint32_t ph = 0;
        int i = (int)(pb % S);
        int mt = (int)((pb / S) % args.mtiles);
        int nt = (int)((pb / S) / args.mtiles);
        for (int64_t q = 0; q < pe - pb; ++q) {
          if (*abort_flag || !mbar_wait(&empty[s], ph ^ 1u, DERR_TIMEOUT_EMPTY)) {
            *abort_flag = 1u;
            break;
          }
          const int m0 = mt * C::BM;
          const int n0 = nt * BN;
          if (!(args.has_lora && i == args.nk_total)) {
            const int c0 = i * 64;
            mbar_arrive_expect_tx(&full[s], C::A_BYTES + C::C_BYTES + C::S_BYTES);
            tma_load_2d(sA + s * C::A_BYTES, &tmA, &full[s], c0, m0);
            if (!BWD) {
              tma_load_2d(sC + s * C::C_BYTES, &tmC, &full[s], c0 / 2, n0);
              tma_load_2d(sS + s * C::S_BYTES, &tmS, &full[s], n0, c0 / 64);
            } else {
              tma_load_2d(sC + s * C::C_BYTES, &tmC, &full[s], n0 / 2, c0);
              tma_load_2d(sS + s * C::S_BYTES, &tmS, &full[s], c0, n0 / 64);
            }
          } else {
            mbar_arrive_expect_tx(&full[s], C::A_BYTES);
            tma_load_2d(sA + s * C::A_BYTES, &tmL, &full[s], 0, m0);
          }
          issued = q + 1;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
          if (++i == (int)S) {
            i = 0;
            if (++mt == args.mtiles) {
              mt = 0;
              ++nt;
            }
          }
        }
        if (*abort_flag) {
          // let every issued copy land before the CTA can exit
          for (int64_t q = (issued > STAGES ? issued - STAGES : 0); q < issued; ++q)
            mbar_wait(&full[q % STAGES], (uint32_t)(q / STAGES) & 1u, DERR_TIMEOUT_DRAIN);
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc_main = idesc_bf16_f32(128, BN, BWD ? 1u : 0u);
        constexpr uint32_t idesc_kmaj = idesc_bf16_f32(128, BN, 0u);
        int64_t q = 0;
        int64_t seg = 0;
        int ms_s = 0, ms_b = 0;
        uint32_t ms_ph = 0, ms_bph = 0;
        for (int64_t p = pb; p < pe && !*abort_flag; ++seg) {
          const int64_t t = p / S;
          const int64_t seg_end = min(pe, (t + 1) * S);
          const int a = (int)(seg % NACC);
          const uint32_t aph = (uint32_t)(seg / NACC) & 1u;
          if (!mbar_wait(&accempty[a], aph ^ 1u, DERR_TIMEOUT_ACC)) {
            *abort_flag = 1u;
            break;
          }
          tc_fence_after();
          const uint32_t dbase = tmem + (uint32_t)(a * C::ACC_COLS);
          int i = (int)(p % S);
          for (int64_t p2 = p; p2 < seg_end; ++p2, ++q, ++i) {
            const int s = ms_s, b = ms_b;
            const uint32_t ph = ms_ph, bph = ms_bph;
            if (++ms_s == STAGES) {
              ms_s = 0;
              ms_ph ^= 1u;
            }
            if (++ms_b == BSTAGES) {
              ms_b = 0;
              ms_bph ^= 1u;
            }
            if (*abort_flag || !mbar_wait(&full[s], ph, DERR_TIMEOUT_FULL) ||
                !mbar_wait(&bfull[b], bph, DERR_TIMEOUT_BFULL)) {
              *abort_flag = 1u;
              break;
            }
            tc_fence_after();
            const bool is_lora = args.has_lora && i == args.nk_total;
            const uint32_t a_base = smem_u32(sA + s * C::A_BYTES);
            const uint32_t b_base = smem_u32(sB + b * C::B_BYTES);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              uint64_t bdesc;
              if (!BWD || is_lora)
                bdesc = smem_desc_sw128(b_base + kk * 32, 16, 1024);
              else
                bdesc = smem_desc_sw128(b_base + kk * 2 * C::MN_SBO, C::MN_LBO, C::MN_SBO);
#pragma unroll
              for (int u = 0; u < UM; ++u) {
                const uint64_t adesc = smem_desc_sw128(a_base + u * 16384 + kk * 32, 16, 1024);
                uint32_t d = dbase + (uint32_t)(u * BN);
                uint32_t acc;
                if (BWD && is_lora) {
                  d += (uint32_t)(UM * BN);
                  acc = kk > 0 ? 1u : 0u;
                } else {
                  acc = (p2 > p || kk > 0) ? 1u : 0u;
                }
                tc_mma_f16(d, adesc, bdesc, is_lora ? idesc_kmaj : idesc_main, acc);
              }
            }
            tc_commit(&empty[s]);
            tc_commit(&bempty[b]);
          }
          tc_commit(&accfull[a]);
          p = seg_end;
        }
        // every MMA this thread issued has completed before TMEM is freed
        tc_commit(drain);
        mbar_wait(drain, 0u, DERR_TIMEOUT_DRAIN);
      }
    } else if (warp < 2 + kDqWarps) {
      // ------------------------------------------------------------ dequant producers
      const int t_idx = (int)threadIdx.x - 64;
      int s = 0, b = 0;
      uint32_t ph = 0, bph = 0;
      int i = (int)(pb % S);
      int mt = (int)((pb / S) % args.mtiles);
      int nt = (int)((pb / S) / args.mtiles);
      for (int64_t q = 0; q < pe - pb; ++q) {
        if (*abort_flag || !mbar_wait(&full[s], ph, DERR_TIMEOUT_FULL) ||
            !mbar_wait(&bempty[b], bph ^ 1u, DERR_TIMEOUT_BEMPTY)) {
          *abort_flag = 1u;
          break;
        }
        const int n0 = nt * BN;
        uint8_t* Bt = sB + b * C::B_BYTES;
        if (!(args.has_lora && i == args.nk_total)) {
          const uint8_t* cs = sC + s * C::C_BYTES;
          const float* ss = reinterpret_cast<const float*>(sS + s * C::S_BYTES);
          if (!BWD) dequant_fwd<BN>(cs, ss, Bt, t_idx, s_lv);
          else dequant_bwd<BN>(cs, ss, Bt, t_idx, s_lv);
        } else {
          lora_tile<BWD, BN>(args.lora_F, args.Nout, args.Nout, n0, args.lora_scale, Bt, t_idx);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bfull[b]);
          mbar_arrive(&empty[s]);
        }
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
        if (++b == BSTAGES) {
          b = 0;
          bph ^= 1u;
        }
        if (++i == (int)S) {
          i = 0;
          if (++mt == args.mtiles) {
            mt = 0;
            ++nt;
          }
        }
        (void)mt;
      }
    } else {
      // ------------------------------------------------------------ epilogue
      const int q4 = warp & 3;  // TMEM lane quarter this warp may read
      const int r = q4 * 32 + lane;
      int64_t seg = 0;
      for (int64_t p = pb; p < pe; ++seg) {
        const int64_t t = p / S;
        const int64_t i0 = p % S;
        const int64_t seg_end = min(pe, (t + 1) * S);
        const int64_t kb = seg_end - t * S;
        const int a = (int)(seg % NACC);
        const uint32_t aph = (uint32_t)(seg / NACC) & 1u;
        const bool ok = !*abort_flag && mbar_wait_backoff(&accfull[a], aph, DERR_TIMEOUT_ACC);
        tc_fence_after();
        const int64_t m0 = (t % args.mtiles) * C::BM;
        const int64_t n0 = (t / args.mtiles) * BN;
        const bool whole = (i0 == 0 && kb == S);
        const bool lora_in = args.has_lora && kb == S;
        // a backward segment made of the LoRA step alone never wrote D
        const bool main_in = !BWD || i0 < args.nk_total;
        const int slot = seg == 0 ? 0 : 1;
        float* part = args.partial + ((int64_t)blockIdx.x * 2 + slot) * C::TILE_FLOATS;
        const uint32_t dbase = tmem + (uint32_t)(a * C::ACC_COLS);
#pragma unroll 1
        for (int u = 0; u < UM; ++u) {
          const int row = u * 128 + r;
          const int64_t m = m0 + row;
          const bool row_ok = ok && m < args.M;
#pragma unroll 1
          for (int cc = 0; cc < BN; cc += 32) {
            const int64_t n = n0 + cc;
            if (n >= args.Nout) break;  // warp-uniform
            uint32_t acc[32];
            const uint32_t taddr = dbase + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(u * BN + cc);
            tmem_ld_32x32b_x32(taddr, acc);
            uint32_t lacc[32];
            if (BWD && lora_in) tmem_ld_32x32b_x32(taddr + (uint32_t)(UM * BN), lacc);
            tmem_ld_wait();
            if (!row_ok) continue;
            float v[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = main_in ? __uint_as_float(acc[e]) : 0.0f;
            if (BWD && lora_in) {
              const uint32_t bits = args.mask[(m * args.Nout + n) >> 5];
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if ((bits >> e) & 1u) v[e] += __uint_as_float(lacc[e]);
            }
            if (!whole) {
              float4* dst = reinterpret_cast<float4*>(part + (int64_t)row * BN + cc);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
            } else if (args.out_f32) {
              float4* dst =
                  reinterpret_cast<float4*>(static_cast<float*>(args.out) + m * args.Nout + n);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                float4 o = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                if (args.out_accum) {
                  const float4 pv = dst[e];
                  o.x = pv.x + o.x;
                  o.y = pv.y + o.y;
                  o.z = pv.z + o.z;
                  o.w = pv.w + o.w;
                }
                dst[e] = o;
              }
            } else {
              uint4* dst =
                  reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.out) + m * args.Nout + n);
#pragma unroll
              for (int e = 0; e < 4; ++e)
                dst[e] = make_uint4(pack_bf16x2(v[8 * e], v[8 * e + 1]),
                                    pack_bf16x2(v[8 * e + 2], v[8 * e + 3]),
                                    pack_bf16x2(v[8 * e + 4], v[8 * e + 5]),
                                    pack_bf16x2(v[8 * e + 6], v[8 * e + 7]));
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&accempty[a]);
        p = seg_end;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// Tiles cut by a stream-K range boundary: add the CTAs' partial tiles in
// step order (the CTA holding the tile's first steps first) and store.
// A partial of CTA g sits in slot 0 when the tile is g's first segment,
// slot 1 when it is g's last.
template <int BM, int BN>
__global__ void __launch_bounds__(256) k_streamk_fixup(const float* __restrict__ partial,
                                                       int64_t S, int mtiles, int ntiles, int64_t G,
                                                       int64_t M, int64_t Nout, void* out,
                                                       int out_f32, int out_accum) {
  constexpr int kMaxParts = 64;
  __shared__ const float* s_part[kMaxParts];
  __shared__ int s_nparts;
  const int64_t t = blockIdx.x;
  const int64_t I = (int64_t)mtiles * ntiles * S;
  const int64_t g1 = sk_cta_of(t * S, I, G);
  const int64_t g2 = sk_cta_of(t * S + S - 1, I, G);
  if (g1 == g2) return;
  if (threadIdx.x == 0) {
    int n = 0;
    for (int64_t g = g1; g <= g2 && n < kMaxParts; ++g, ++n) {
      const int slot = sk_begin(g, I, G) >= t * S ? 0 : 1;
      s_part[n] = partial + (g * 2 + slot) * (int64_t)BM * BN;
    }
    s_nparts = n;
  }
  __syncthreads();
  const int nparts = s_nparts;
  const int64_t m0 = (t % mtiles) * BM, n0 = (t / mtiles) * BN;
  const int rows = (int)((M - m0) < BM ? (M - m0) : BM);
  const int cols = (int)((Nout - n0) < BN ? (Nout - n0) : BN);
  for (int e4 = threadIdx.x; e4 < BM * BN / 4; e4 += 256) {
    const int row = (e4 * 4) / BN, col = (e4 * 4) % BN;
    if (row >= rows || col >= cols) continue;
    const int off = row * BN + col;
    float4 acc = *reinterpret_cast<const float4*>(s_part[0] + off);
    for (int k = 1; k < nparts; ++k) {
      const float4 v = *reinterpret_cast<const float4*>(s_part[k] + off);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const int64_t m = m0 + row, n = n0 + col;
    if (out_f32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + m * Nout + n);
      if (out_accum) {
        const float4 o = *dst;
        acc.x = o.x + acc.x;
        acc.y = o.y + acc.y;
        acc.z = o.z + acc.z;
        acc.w = o.w + acc.w;
      }
      *dst = acc;
    } else {
      uint2* dst = reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + m * Nout + n);
      *dst = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    }
  }
}

}  // namespace

// ---------------------------------------------------------------------------------- host
namespace {

PFN_encodeTiled g_encode = nullptr;

bool encode_fn() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return false;
  g_encode = reinterpret_cast<PFN_encodeTiled>(fn);
  return true;
}

// 2-D tensor map: inner dimension `inner` elements (contiguous), `outer` rows
// with a row pitch of `pitch_bytes`; box {box_inner, box_outer}.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
              uint64_t outer, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle sw) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {pitch_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Persistent grid: one CTA per SM, but at least kMinSteps (tile, step)
// iterations per CTA so tiny problems are not shredded into partials.
constexpr int64_t kMinSteps = 8;

template <bool BWD, int UM, int BN>
cudaError_t launch_cfg(const GemmPlan& p, const GemmArgs& a, const CUtensorMap& tA,
                       const CUtensorMap& tC, const CUtensorMap& tS, const CUtensorMap& tL,
                       cudaStream_t st) {
  using C = Cfg<BWD, UM, BN>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_nf4_gemm<BWD, UM, BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t S = (int64_t)p.nk + (a.has_lora ? 1 : 0);
  const int64_t I = (int64_t)p.mtiles * p.ntiles * S;
  const int64_t G = grid_ctas(p, a.has_lora != 0);
  note_launch();
  k_nf4_gemm<BWD, UM, BN><<<(unsigned)G, kThreads, C::SMEM_BYTES, st>>>(tA, tC, tS, tL, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || G == 1 || I % G == 0 && (I / G) % S == 0) return e;
  note_launch();
  k_streamk_fixup<C::BM, BN><<<(unsigned)(p.mtiles * p.ntiles), 256, 0, st>>>(
      a.partial, S, p.mtiles, p.ntiles, G, a.M, a.Nout, a.out, a.out_f32, a.out_accum);
  return cudaGetLastError();
}

}  // namespace

// ---------------------------------------------------------------- allocation-free scratch
// Split-contraction partials for ws_nf4_matmul_noalloc live in this
// file-scope device array rather than in a caller workspace.  Every device
// that loads the library holds it until the process exits; every call shares
// it.  Each split writes every element of its own partial slice before the
// reduce reads it, so nothing has to start at zero.
constexpr size_t kNoAllocScratchBytes = (size_t)WS_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

namespace {
std::mutex g_noalloc_mu;
constexpr int kMaxDevices = 64;
float* g_noalloc_ptr[kMaxDevices] = {};
}  // namespace

cudaError_t noalloc_scratch(float** ptr, size_t* bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    // host code cannot use the symbol itself: ask the runtime for this
    // device's address of the array (once per device)
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *ptr = g_noalloc_ptr[dev];
  *bytes = kNoAllocScratchBytes;
  return cudaSuccess;
}

int device_sm_count() {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  return sms;
}

int64_t grid_ctas(const GemmPlan& p, bool has_lora) {
  const int64_t S = (int64_t)p.nk + (has_lora ? 1 : 0);
  const int64_t I = (int64_t)p.mtiles * p.ntiles * S;
  // at least kMinSteps iterations per CTA, and few enough CTAs that one tile
  // is never cut into more pieces than the fix-up kernel gathers (64)
  int64_t min_steps = S / 48 + 2;
  if (min_steps < kMinSteps) min_steps = kMinSteps;
  int64_t G = (I + min_steps - 1) / min_steps;
  if (G > device_sm_count()) G = device_sm_count();
  return G < 1 ? 1 : G;
}

GemmPlan plan_gemm(bool bwd, int64_t M, int64_t Nout, int64_t Kc) {
  GemmPlan p{};
  p.bwd = bwd;
  p.um = M > 128 ? 2 : 1;
  p.bn = 128;
  p.mtiles = (int)((M + 128 * p.um - 1) / (128 * p.um));
  p.ntiles = (int)((Nout + p.bn - 1) / p.bn);
  p.nk = (int)(Kc / 64);
  return p;
}

size_t gemm_partial_bytes(const GemmPlan& p, int64_t M, int64_t Nout) {
  (void)M;
  (void)Nout;
  const int64_t G = grid_ctas(p, true);
  if (G <= 1) return 0;
  return (size_t)G * 2 * (size_t)(128 * p.um) * (size_t)p.bn * sizeof(float);
}

cudaError_t run_nf4_gemm(const GemmPlan& p, const NF4View& W, const uint16_t* act, int64_t M,
                         const uint16_t* lora_act, const float* lora_F, float lora_scale,
                         const uint32_t* mask, void* out, int out_f32, int out_accum,
                         float* partial, cudaStream_t st) {
  if (!encode_fn()) return cudaErrorNotSupported;
  const int64_t N = W.N, K = W.K;
  const int64_t Nout = p.bwd ? K : N;
  const int64_t Kc = p.bwd ? N : K;
  const int BM = 128 * p.um;
  CUtensorMap tA, tC, tS, tL;
  bool ok = make_map(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, act, (uint64_t)Kc, (uint64_t)M,
                     (uint64_t)Kc * 2, 64, (uint32_t)BM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!p.bwd) {
    ok = ok && make_map(&tC, CU_TENSOR_MAP_DATA_TYPE_UINT8, W.codes, (uint64_t)(K / 2),
                        (uint64_t)N, (uint64_t)(K / 2), 32, (uint32_t)p.bn,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
    ok = ok && make_map(&tS, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, W.absmax, (uint64_t)N,
                        (uint64_t)(K / 64), (uint64_t)N * 4, (uint32_t)p.bn, 1,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
  } else {
    ok = ok && make_map(&tC, CU_TENSOR_MAP_DATA_TYPE_UINT8, W.codes, (uint64_t)(K / 2),
                        (uint64_t)N, (uint64_t)(K / 2), (uint32_t)(p.bn / 2), 64,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
    ok = ok && make_map(&tS, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, W.absmax, (uint64_t)N,
                        (uint64_t)(K / 64), (uint64_t)N * 4, 64, (uint32_t)(p.bn / 64),
                        CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  const bool has_lora = lora_act != nullptr && lora_F != nullptr;
  if (has_lora)
    ok = ok && make_map(&tL, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, lora_act, 64, (uint64_t)M, 128, 64,
                        (uint32_t)BM, CU_TENSOR_MAP_SWIZZLE_128B);
  else
    tL = tA;
  if (!ok) return cudaErrorInvalidValue;

  GemmArgs a{};
  a.M = M;
  a.Nout = Nout;
  a.nk_total = p.nk;
  a.mtiles = p.mtiles;
  a.ntiles = p.ntiles;
  a.has_lora = has_lora ? 1 : 0;
  a.lora_F = lora_F;
  a.lora_scale = lora_scale;
  a.mask = mask;
  a.out = out;
  a.out_f32 = out_f32;
  a.out_accum = out_accum;
  a.partial = partial;

  if (partial == nullptr && grid_ctas(p, has_lora) > 1) return cudaErrorInvalidValue;
  if (!p.bwd) {
    if (p.um == 2) return launch_cfg<false, 2, 128>(p, a, tA, tC, tS, tL, st);
    return launch_cfg<false, 1, 128>(p, a, tA, tC, tS, tL, st);
  }
  if (p.um == 2) return launch_cfg<true, 2, 128>(p, a, tA, tC, tS, tL, st);
  return launch_cfg<true, 1, 128>(p, a, tA, tC, tS, tL, st);
}

}  // namespace ws
