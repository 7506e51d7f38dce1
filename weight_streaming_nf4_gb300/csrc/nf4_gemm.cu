// nf4_gemm.cu -- the NF4 dequant GEMM on the 5th-generation tensor cores.
//
// Forward:  y[M,N]  = x[M,K] . W'[N,K]^T  (+ s U B^T as an extra step)
// Backward: dX[M,K] = dY[M,N] . W'[N,K]   (+ s (G A) . mask)
//
// W' = bf16_RN(c[code] * absmax) is never materialised in global memory:
// packed 4-bit codes and the block absmax are staged into shared memory
// (cp.async), dequantised by eight producer warps straight into the 128-byte
// swizzled operand layout the tensor cores read, and consumed by
// tcgen05.mma (bf16 x bf16 -> fp32 in TMEM) issued by one thread.
//
// Persistent CTA (one per SM) = 18 warps:
//   warp 0      TMA producer (activation tiles)
//   warp 1      TMEM allocator and MMA issuer
//   warps 2-9   dequant producers (each stages its own codes and block
//               scales with cp.async)
//   warps 10-17 epilogue (TMEM -> registers -> global), two per TMEM lane
//               quarter, overlapping the next tile's main loop
// Tile: 128*UM rows of activations (UM tensor-core atoms of M = 128 sharing
// one dequantised weight tile), BN output columns, 64-deep contraction steps.
//
// Schedule: the (tile, step) iterations of the whole problem are cut into
// contiguous ranges, one per unit (a CTA, or a pair of CTAs), on a grid
// sized so that every CTA is resident at once (stream-K).  A tile cut by
// range boundaries is finished by the unit holding its first steps -- that
// is always the last segment of that unit's range, so it runs after the
// other pieces were made: it adds the later units' fp32 partial tiles to its
// own accumulator in step order (after waiting, with a time limit, for
// their completion flags) and stores the tile.  Every other tile is stored
// by its unit directly.  The cut points depend only on the shape and the
// grid size, so results are deterministic and identical run to run.  No
// atomics on data.
//
// Grouped forward: linears that read the same activation (q and k, gate and
// up) run as one launch over their concatenated output columns; each tile
// takes its weight, LoRA factor and output from its linear.
//
// The LoRA terms use the same tensor cores: the forward appends one 64-deep
// step whose A operand is [U_hi | U_lo | U_hi | 0] and whose B operand is
// [Bs_hi | Bs_hi | Bs_lo | 0] (Bs = s B, bf16 high/low splits), i.e.
// U Bs^T to about 16 significant bits.  The backward computes s G A the same
// way but as each tile's FIRST step: the epilogue warps then apply the
// dropout mask to the accumulator in TMEM (load, zero the dropped
// elements, store back) before the main steps accumulate on top, so one
// accumulator serves both terms.
#define WS_GEMM_TU 1
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace ws {

cudaError_t ring_clear();

cudaError_t read_and_clear_dev_error(uint32_t* flags) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(flags, g_dev_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  if (*flags != 0u) {
    // a kernel gave up part way: cross-CTA words may be left set
    e = ring_clear();
    if (e != cudaSuccess) return e;
  }
  const uint32_t zero = 0;
  e = cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  uint32_t attn = 0;
  e = attn_read_and_clear_dev_error(&attn);
  *flags |= attn;
  return e;
}


namespace {

// Pipeline depths: dequantised-operand buffers and activation-tile TMA
// stages (upper bound; the shared-memory budget may allow fewer).
#ifndef WS_GEMM_BSTAGES
#define WS_GEMM_BSTAGES 3
#endif
// One barrier and one commit per pipeline step on the pair MMA (0: an
// activation barrier and a weight-buffer barrier, each with its commit).
#ifndef WS_GEMM_MERGED_BARRIERS
#define WS_GEMM_MERGED_BARRIERS 1
#endif
constexpr bool kMergedBarriers = WS_GEMM_MERGED_BARRIERS != 0;
// Paired handovers per configuration, a bit mask: 1 forward 128-wide tiles,
// 2 forward 256-wide, 4 input gradient 128-wide, 8 input gradient 256-wide.
// On for all: the per-step handshake bounds the steps (32B step 73.6 -> 72.2
// ms against per-step handovers for the 256-wide tiles).
#ifndef WS_GEMM_PAIR_STEPS
#define WS_GEMM_PAIR_STEPS 15
#endif
constexpr int kPairSteps = WS_GEMM_PAIR_STEPS;

#ifndef WS_GEMM_STAGES_MAX
#define WS_GEMM_STAGES_MAX 6
#endif
// Forward dequant warps load their codes and block scales straight into
// registers, two steps ahead (1), instead of through a ring in shared memory
// (0).  The input gradient keeps the ring: its 8-byte code items, gathered
// from 64 weight rows per step, lose a fifth of the rate when loaded into
// registers.
#ifndef WS_GEMM_REG_CODES
#define WS_GEMM_REG_CODES 1
#endif
constexpr bool kRegCodes = WS_GEMM_REG_CODES != 0;
// Bytes (KB) of the dequant threads' code ring: each thread fetches its codes
// and block scales as many steps ahead as the ring holds (at least 4, at most
// 16), so a narrower tile (shorter steps) fetches more steps ahead.
#ifndef WS_GEMM_CODE_RING_KB
#define WS_GEMM_CODE_RING_KB 20
#endif
// Shared memory (KB) the pipeline stages may take (the rest holds the
// barriers and the alignment slack).
#ifndef WS_GEMM_SMEM_BUDGET_KB
#define WS_GEMM_SMEM_BUDGET_KB 220
#endif

constexpr int kDqWarps = 8;
constexpr int kEpiWarps = 8;
constexpr int kThreads = (2 + kDqWarps + kEpiWarps) * 32;
constexpr int kDqThreads = kDqWarps * 32;
constexpr int kFinRing = 8;  // finisher: partial-tile entries in flight per epilogue warp

// Dequant work of one thread per step.  A CTA fills the whole BN-wide
// weight tile itself, or -- as one CTA of a pair sharing the tile -- the half
// [rank * BN/2, (rank + 1) * BN/2) of it: PAIR = 1 writes that half into
// both CTAs' full-width buffers, PAIR = 2 keeps it in a half-width buffer of
// its own that the pair MMA reads from both CTAs.
//   forward: ROWS weight-tile rows (output columns) x 64 codes, TPR threads
//            per row, each with VB code bytes;
//   backward: 64 contraction rows x COLS output columns in items of
//            VB * 2 columns, one item per thread and vector.
template <bool BWD, int BN, int PAIR>
struct DqGeo {
  static constexpr int COLS = PAIR ? BN / 2 : BN;  // columns (bwd) / rows (fwd) this CTA fills
  static constexpr int TPR = BWD ? 0 : kDqThreads / COLS;
  // code bytes per vector and vectors per thread
  static constexpr int VB = BWD ? (PAIR ? 8 : 16) : (32 / (kDqThreads / COLS) >= 16 ? 16 : 8);
  static constexpr int NV = BWD ? (64 * COLS / (VB * 2)) / kDqThreads : (32 / TPR) / VB;
  // block scales per thread: one.  Backward items t*NV .. t*NV+NV-1 lie in
  // one row and, NV*2*VB columns wide and aligned to that width, in one
  // 64-column block, so they share one scale and one value table.
  static constexpr int NS = 1;
  static constexpr int SEGS = BWD ? COLS / (2 * VB) : 1;
  static_assert(!BWD || (SEGS % NV == 0 && 64 % (NV * 2 * VB) == 0), "backward items share a scale");
  static constexpr uint32_t SLOT_BYTES = NV * kDqThreads * VB + NS * kDqThreads * 4;
  static_assert(NV >= 1 && NV <= 2, "dequant geometry");
  static_assert(!BWD || (64 * COLS / (VB * 2)) % kDqThreads == 0, "dequant geometry");
  // Backward: item it of thread t is (contraction row c, segment seg).  A
  // thread's NV items are consecutive segments of one row (one 64-column
  // block: one scale); the eight lanes of each quarter warp take eight
  // consecutive rows of one segment group, so their 16-byte stores into the
  // swizzled tile land in eight different bank groups (lanes of one row in
  // the two 64-column halves hit the same banks).
  static constexpr int SG = BWD ? SEGS / NV : 1;  // segment groups per row
  static_assert(!BWD || (SEGS % NV == 0 && 32 % SG == 0), "backward item mapping");
  WS_DEVINL static void item(int t, int it, int& c, int& seg) {
    constexpr int RPW = 32 / SG;  // rows per warp
    const int l = t & 31;
    c = (t >> 5) * RPW + l % RPW;
    seg = (l / RPW) * NV + it;
  }
};

// WB: the weight is bf16 and its tiles are loaded by TMA (no dequantisation).
template <bool BWD, int UM, int BN, int PAIR, bool WB = false>
struct Cfg {
  static constexpr int BM = 128 * UM;
  static constexpr uint32_t A_BYTES = BM * 128;   // BM rows x 64 bf16
  static constexpr bool PM = PAIR == 2;            // one MMA across the pair
  static constexpr int BW = PM ? BN / 2 : BN;      // weight-tile width held by this CTA
  static constexpr uint32_t B_BYTES = BW * 128;    // BW x 64 bf16
#ifdef WS_GEMM_BSTAGES_PM
  static constexpr int BSTAGES = PM ? WS_GEMM_BSTAGES_PM : WS_GEMM_BSTAGES;
#else
  static constexpr int BSTAGES = PM ? WS_GEMM_BSTAGES + 1 : WS_GEMM_BSTAGES;
#endif
  // per-thread ring of fetched codes (cp.async), CSTAGES steps deep
  static constexpr bool REG_CODES = kRegCodes && !BWD;
  static constexpr uint32_t CODE_BYTES = (WB || REG_CODES) ? 0u : DqGeo<BWD, BN, PAIR>::SLOT_BYTES;
  static constexpr int CSTAGES_RAW =
      (int)((WS_GEMM_CODE_RING_KB * 1024u) / DqGeo<BWD, BN, PAIR>::SLOT_BYTES);
  static constexpr int CSTAGES = CSTAGES_RAW < 4 ? 4 : (CSTAGES_RAW > 16 ? 16 : CSTAGES_RAW);
  static constexpr int STAGES_RAW =
      (int)((WS_GEMM_SMEM_BUDGET_KB * 1024u - BSTAGES * B_BYTES - CSTAGES * CODE_BYTES - 1024u) /
            A_BYTES);
  static constexpr int STAGES_FREE = STAGES_RAW > WS_GEMM_STAGES_MAX ? WS_GEMM_STAGES_MAX : STAGES_RAW;
  // Pair MMA: an activation stage and a weight buffer are filled and freed
  // together (as many stages as buffers), so one barrier per stage says
  // "both operands ready" and one MMA commit frees both: one wait and one
  // commit per step for the MMA thread instead of two each.
  static constexpr bool MERGED = PM && kMergedBarriers;
  static constexpr int STAGES = MERGED ? BSTAGES : STAGES_FREE;
  // Merged NF4 stages are handed over in pairs: the dequant warps fill the
  // weight buffers of two consecutive steps, then make one arrival on the
  // even stage's barrier, which then stands for both buffers (the odd
  // stage's barrier counts only its activation copy).  One wait, one fence
  // and one arrival per two steps: the per-step handshake, not the decode,
  // bounds the producers' rate.
  static constexpr bool PAIRSTEP = MERGED && !WB && (BSTAGES % 2 == 0) &&
                                   ((kPairSteps >> ((BWD ? 2 : 0) + (BN == 256 ? 1 : 0))) & 1) != 0;
  // one accumulator set
  static constexpr uint32_t ACC_COLS = UM * BN;
  // double-buffer the accumulator when TMEM has room, so the epilogue of
  // one tile overlaps the main loop of the next
  static constexpr int ACC_BUFS = 2 * ACC_COLS <= 512 ? 2 : 1;
  static constexpr uint32_t TMEM_COLS = ACC_COLS * ACC_BUFS;
  static constexpr int64_t TILE_FLOATS = (int64_t)BM * BN;
  // MN-major operand (backward): 64-element MN groups LBO apart, 8-row K
  // groups SBO apart; MN_KK bytes per 16-deep slice.  The dequantiser
  // interleaves the MN groups inside each 8-row group; a bf16 tile arrives
  // as BW/64 TMA boxes of 64 rows x 64 columns, one 8 KB box per MN group.
  static constexpr uint32_t MN_LBO = WB ? 8192u : 1024u;
  static constexpr uint32_t MN_SBO = WB ? 1024u : (uint32_t)(BW / 64) * 1024u;
  static constexpr uint32_t MN_KK = 2 * MN_SBO;
  static constexpr uint32_t OFF_A = 0;
  static constexpr uint32_t OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr uint32_t OFF_CODE = OFF_B + BSTAGES * B_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_CODE + CSTAGES * CODE_BYTES;
  static constexpr uint32_t N_BARS = 2 * STAGES + 2 * BSTAGES + 2 * ACC_BUFS + 3;
  static constexpr uint32_t OFF_MISC = OFF_BAR + N_BARS * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 1024;  // + alignment slack
  static_assert(STAGES >= 2, "pipeline needs two stages");
  static_assert(!MERGED || STAGES_RAW >= BSTAGES, "merged stages fit the shared memory");
  static_assert(TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM columns");
  static_assert(SMEM_BYTES <= 227u * 1024u, "shared memory");
  static_assert(BN == 128 || BN == 256, "BN");
  static_assert(!PAIR || UM == 2, "a pair shares one weight tile between two 256-row halves");
  static_assert(!WB || PAIR != 1, "bf16 tiles are loaded by each CTA itself");
  static_assert(PAIR >= 0 && PAIR <= 2, "pair mode");
  static_assert(OFF_CODE >= (uint32_t)(kEpiWarps * kFinRing * 2048), "finisher ring fits the stages");
};

// CTA of the stream-K schedule that owns iteration i: ranges are
// [floor(g*I/G), floor((g+1)*I/G)), so g = ceil((i+1)*G/I) - 1.
__host__ __device__ inline int64_t sk_cta_of(int64_t i, int64_t I, int64_t G) {
  return ((i + 1) * G + I - 1) / I - 1;
}
__host__ __device__ inline int64_t sk_begin(int64_t g, int64_t I, int64_t G) { return g * I / G; }

// Two IEEE fp32 products (round to nearest) in one packed instruction.
WS_DEVINL void mul2_rn(float x0, float x1, float s, float& r0, float& r1) {
  asm("{\n .reg .b64 pa, pb, pd;\n mov.b64 pa, {%2, %3};\n mov.b64 pb, {%4, %4};\n"
      " mul.rn.f32x2 pd, pa, pb;\n mov.b64 {%0, %1}, pd;\n}"
      : "=f"(r0), "=f"(r1)
      : "f"(x0), "f"(x1), "f"(s));
}

// Byte permute: bytes of {b, a} (a = bytes 0-3, b = 4-7) picked by the four
// 4-bit fields of sel.
WS_DEVINL uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// The 16 dequantised values of one 64-weight block, T[i] = bf16_RN(c_i * a)
// (one fp32 product, one rounding), split into byte planes: lo[q] holds the
// low bytes of T[4q..4q+3], hi[q] their high bytes.  A 4-bit code then
// becomes a bf16 value with byte permutes in registers -- no shared-memory
// table lookup per weight.
struct Nf4Table {
  uint32_t lo[4], hi[4];
};
WS_DEVINL Nf4Table make_table(float a) {
  uint32_t R[8];
  float v0, v1;
  mul2_rn(-1.0f, -0.6962f, a, v0, v1);
  R[0] = pack_bf16x2(v0, v1);
  mul2_rn(-0.5251f, -0.3949f, a, v0, v1);
  R[1] = pack_bf16x2(v0, v1);
  mul2_rn(-0.2844f, -0.1848f, a, v0, v1);
  R[2] = pack_bf16x2(v0, v1);
  mul2_rn(-0.0911f, 0.0f, a, v0, v1);
  R[3] = pack_bf16x2(v0, v1);
  mul2_rn(0.0796f, 0.1609f, a, v0, v1);
  R[4] = pack_bf16x2(v0, v1);
  mul2_rn(0.2461f, 0.3379f, a, v0, v1);
  R[5] = pack_bf16x2(v0, v1);
  mul2_rn(0.4407f, 0.5626f, a, v0, v1);
  R[6] = pack_bf16x2(v0, v1);
  mul2_rn(0.7230f, 1.0f, a, v0, v1);
  R[7] = pack_bf16x2(v0, v1);
  Nf4Table t;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    t.lo[q] = prmt(R[2 * q], R[2 * q + 1], 0x6420u);
    t.hi[q] = prmt(R[2 * q], R[2 * q + 1], 0x7531u);
  }
  return t;
}

// 4 code bytes (8 consecutive weights along k: byte i holds k = 2i in its
// high nibble, 2i+1 in its low nibble) -> 8 bf16 values in k order.
// Nibble f of the word is the code of k = f ^ 1; the two interleaving
// permutes at the end put the pairs back in k order, so the codes need no
// nibble swap first.
WS_DEVINL uint4 dq8(uint32_t w, const Nf4Table& t) {
  const uint32_t s7 = w & 0x77777777u;                           // index within 8 entries
  const uint32_t s8 = ((w >> 1) & 0x44444444u) | 0x32103210u;    // which half (code >= 8)
  uint32_t o[4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t a7 = h ? (s7 >> 16) : s7;
    const uint32_t a8 = h ? (s8 >> 16) : s8;
    // byte p of lo / hi: low / high byte of the value of nibble 4h + p
    const uint32_t lo = prmt(prmt(t.lo[0], t.lo[1], a7), prmt(t.lo[2], t.lo[3], a7), a8);
    const uint32_t hi = prmt(prmt(t.hi[0], t.hi[1], a7), prmt(t.hi[2], t.hi[3], a7), a8);
    o[2 * h] = prmt(lo, hi, 0x4051u);      // k = 4h (nibble 4h+1), k = 4h+1 (nibble 4h)
    o[2 * h + 1] = prmt(lo, hi, 0x6273u);  // k = 4h+2 (nibble 4h+3), k = 4h+3 (nibble 4h+2)
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Code words and block scales of one dequant thread for one step.
struct Frag {
  uint32_t w[8];
  float a[1];
};

// Asynchronous 16- / 8- / 4-byte global -> shared copies; src_bytes = 0
// fills zeros without reading.
WS_DEVINL void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
WS_DEVINL void cp_async8(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
WS_DEVINL void cp_async4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
WS_DEVINL void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
WS_DEVINL void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
template <int VB>
WS_DEVINL void cp_async_v(uint32_t dst, const void* src, bool in) {
  if constexpr (VB == 16) cp_async16(dst, src, in ? 16u : 0u);
  else cp_async8(dst, src, in ? 8u : 0u);
}

// Each dequant thread stages its own codes and scales of a step in a ring
// slot of shared memory: code vectors at [v][t], scales after them at
// [v][t], so the reads back are conflict-free.
// Forward: thread t covers (part of) weight-tile row j, i.e. output column
// n0 + j.  Backward: item (c, seg) covers weight row i*64 + c (the
// contraction index) and 2*VB weight columns (the output index).
// Rows / columns past the weight's edge read as zero codes with scale 0.
template <bool BWD, int BN, int PAIR>
WS_DEVINL void fetch_codes(uint32_t slot, const uint8_t* codes, const float* absmax, int64_t wN,
                           int64_t wK, int i, int64_t n0, int rank, int t) {
  using D = DqGeo<BWD, BN, PAIR>;
  const int64_t kb = wK / 2;  // code bytes per weight row
  const int c0 = PAIR ? rank * D::COLS : 0;
  const uint32_t sc = slot + (uint32_t)(D::NV * kDqThreads * D::VB);
  if constexpr (!BWD) {
    const int j = c0 + t / D::TPR, part = t % D::TPR;
    const int64_t n = (int64_t)n0 + j;
    const bool in = n < wN;
    const int64_t nn = in ? n : 0;
    const uint8_t* src = codes + nn * kb + (int64_t)i * 32 + part * (32 / D::TPR);
#pragma unroll
    for (int v = 0; v < D::NV; ++v)
      cp_async_v<D::VB>(slot + (uint32_t)((v * kDqThreads + t) * D::VB), src + D::VB * v, in);
    cp_async4(sc + (uint32_t)(t * 4), absmax + (int64_t)i * wN + nn, in ? 4u : 0u);
  } else {
#pragma unroll
    for (int it = 0; it < D::NV; ++it) {
      int c, seg;
      D::item(t, it, c, seg);
      const int64_t r = (int64_t)i * 64 + c;
      const int64_t col = (int64_t)n0 + c0 + seg * 2 * D::VB;
      const bool in = r < wN && col < wK;
      const int64_t rr = in ? r : 0, cl = in ? col : 0;
      cp_async_v<D::VB>(slot + (uint32_t)((it * kDqThreads + t) * D::VB),
                        codes + rr * kb + cl / 2, in);
      if (it == 0)
        cp_async4(sc + (uint32_t)(t * 4), absmax + (cl / 64) * wN + rr, in ? 4u : 0u);
    }
  }
}

template <bool BWD, int BN, int PAIR>
WS_DEVINL void read_frag(Frag& f, const uint8_t* slot, int t) {
  using D = DqGeo<BWD, BN, PAIR>;
  const float* sc = reinterpret_cast<const float*>(slot + D::NV * kDqThreads * D::VB);
#pragma unroll
  for (int v = 0; v < D::NV; ++v) {
    if constexpr (D::VB == 16) {
      const uint4 x = *reinterpret_cast<const uint4*>(slot + (v * kDqThreads + t) * 16);
      f.w[4 * v] = x.x;
      f.w[4 * v + 1] = x.y;
      f.w[4 * v + 2] = x.z;
      f.w[4 * v + 3] = x.w;
    } else {
      const uint2 x = *reinterpret_cast<const uint2*>(slot + (v * kDqThreads + t) * 8);
      f.w[2 * v] = x.x;
      f.w[2 * v + 1] = x.y;
    }
  }
#pragma unroll
  for (int v = 0; v < D::NS; ++v) f.a[v] = sc[v * kDqThreads + t];
}

// The codes and scale fetch_codes + read_frag give a thread, loaded straight
// into registers on the read-only path (zero codes and scale past the edge).
template <bool BWD, int BN, int PAIR>
WS_DEVINL void load_frag(Frag& f, const uint8_t* codes, const float* absmax, int64_t wN,
                         int64_t wK, int i, int64_t n0, int rank, int t) {
  using D = DqGeo<BWD, BN, PAIR>;
  const int64_t kb = wK / 2;
  const int c0 = PAIR ? rank * D::COLS : 0;
  auto ld = [&](const uint8_t* p, bool in, int v) {
    if constexpr (D::VB == 16) {
      const uint4 x = in ? __ldg(reinterpret_cast<const uint4*>(p)) : make_uint4(0u, 0u, 0u, 0u);
      f.w[4 * v] = x.x;
      f.w[4 * v + 1] = x.y;
      f.w[4 * v + 2] = x.z;
      f.w[4 * v + 3] = x.w;
    } else {
      const uint2 x = in ? __ldg(reinterpret_cast<const uint2*>(p)) : make_uint2(0u, 0u);
      f.w[2 * v] = x.x;
      f.w[2 * v + 1] = x.y;
    }
  };
  if constexpr (!BWD) {
    const int j = c0 + t / D::TPR, part = t % D::TPR;
    const int64_t n = (int64_t)n0 + j;
    const bool in = n < wN;
    const int64_t nn = in ? n : 0;
    const uint8_t* src = codes + nn * kb + (int64_t)i * 32 + part * (32 / D::TPR);
#pragma unroll
    for (int v = 0; v < D::NV; ++v) ld(src + D::VB * v, in, v);
    f.a[0] = in ? __ldg(absmax + (int64_t)i * wN + nn) : 0.0f;
  } else {
#pragma unroll
    for (int it = 0; it < D::NV; ++it) {
      int c, seg;
      D::item(t, it, c, seg);
      const int64_t r = (int64_t)i * 64 + c;
      const int64_t col = (int64_t)n0 + c0 + seg * 2 * D::VB;
      const bool in = r < wN && col < wK;
      const int64_t rr = in ? r : 0, cl = in ? col : 0;
      ld(codes + rr * kb + cl / 2, in, it);
      if (it == 0) f.a[0] = in ? __ldg(absmax + (cl / 64) * wN + rr) : 0.0f;
    }
  }
}

// Forward weight tile, K-major 128B-swizzled: row j = output column n0 + j,
// 64 contraction elements; chunk cc of row j sits at (cc ^ (j & 7)) * 16.
template <int BN, int PAIR>
WS_DEVINL void dequant_fwd(const Frag& f, uint8_t* Bt, int rank, int t) {
  using D = DqGeo<false, BN, PAIR>;
  constexpr int WPT = 8 / D::TPR;  // code words per thread
  // row in this CTA's buffer
  const int j = (PAIR == 1 ? rank * D::COLS : 0) + t / D::TPR, part = t % D::TPR;
  const Nf4Table tb = make_table(f.a[0]);
#pragma unroll
  for (int q = 0; q < WPT; ++q) {
    const int cc = part * WPT + q;
    const uint4 v = dq8(f.w[q], tb);
    sts128(Bt + j * 128 + ((cc ^ (j & 7)) << 4), v.x, v.y, v.z, v.w);
  }
}

// Backward weight tile, MN-major 128B-swizzled: the contraction runs over
// W's rows n (64 per step) and the output over W's columns k (BN per tile),
// so the tile keeps W's own orientation.  Element (k-col j, n-row c):
// group (c/8, j/64) at (c/8)*SBO + (j/64)*LBO, row c%8 inside the group,
// chunk ((j%64)/8) ^ (c%8).
template <int BN, int PAIR>
WS_DEVINL void dequant_bwd(const Frag& f, uint8_t* Bt, int rank, int t) {
  using D = DqGeo<true, BN, PAIR>;
  constexpr uint32_t SBO = ((PAIR == 2 ? BN / 2 : BN) / 64) * 1024;  // this CTA's buffer width
  constexpr int WPI = D::VB / 4;  // code words per item: 8 weights each
  const Nf4Table tb = make_table(f.a[0]);  // the thread's items share one block scale
#pragma unroll
  for (int it = 0; it < D::NV; ++it) {
    int c, seg;
    D::item(t, it, c, seg);
    const int j0 = (PAIR == 1 ? rank * D::COLS : 0) + seg * 2 * D::VB;  // first buffer column
    const uint32_t grp = (uint32_t)((c >> 3) * SBO + (j0 / 64) * 1024 + (c & 7) * 128);
#pragma unroll
    for (int q = 0; q < WPI; ++q) {
      const int cc = (j0 % 64) / 8 + q;
      const uint4 v = dq8(f.w[it * WPI + q], tb);
      sts128(Bt + grp + ((cc ^ (c & 7)) << 4), v.x, v.y, v.z, v.w);
    }
  }
}

// The LoRA weight operand of the extra step, K-major like the forward
// tile: row j holds [Ws_hi(16) | Ws_hi(16) | Ws_lo(16) | 0(16)] with
// Ws = s * (row j of the LoRA factor).  Forward: factor row = B[n0+j, :];
// backward: factor row = A[:, n0+j] (column of A).  A CTA of a pair fills
// its half of the rows (PAIR = 2: into its own half-width buffer).
template <bool BWD, int BN, int PAIR>
WS_DEVINL void lora_tile(const float* F, int64_t rows_total, int64_t ld, int n0, float s,
                         uint8_t* Bt, int rank, int t) {
  constexpr int ROWS = PAIR ? BN / 2 : BN;
  constexpr int TPR = kDqThreads / ROWS;  // threads per row
  const int j = (PAIR == 1 ? rank * ROWS : 0) + t / TPR, part = t % TPR;  // buffer row
  const int64_t n = (int64_t)n0 + (PAIR ? rank * ROWS : 0) + t / TPR;
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
#pragma unroll
  for (int q = 0; q < 8 / TPR; ++q) {
    const int cc = part * (8 / TPR) + q;
    uint4 val;
    if (cc == 0 || cc == 2) val = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    else if (cc == 1 || cc == 3) val = make_uint4(hi[4], hi[5], hi[6], hi[7]);
    else if (cc == 4) val = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    else if (cc == 5) val = make_uint4(lo[4], lo[5], lo[6], lo[7]);
    else val = make_uint4(0u, 0u, 0u, 0u);
    sts128(Bt + j * 128 + ((cc ^ (j & 7)) << 4), val.x, val.y, val.z, val.w);
  }
}

// The linear a forward tile belongs to (grouped launches; see GemmArgs):
// selected with compares, so the parameter arrays are never indexed at run
// time.
struct TileGrp {
  const uint8_t* codes;
  const float* absmax;
  const float* lora_F;
  void* out;
  int64_t c0;     // first output column of the group
  int64_t width;  // its output columns (its weight's N; row pitch of its output)
  int g;
};
WS_DEVINL TileGrp tile_grp(const GemmArgs& a, int64_t n0) {
  TileGrp r;
  if (a.ngroups <= 1) {
    r.codes = a.codes;
    r.absmax = a.absmax;
    r.lora_F = a.lora_F;
    r.out = a.out;
    r.c0 = 0;
    r.width = a.Nout;
    r.g = 0;
    return r;
  }
  const bool g1 = n0 >= a.gcol[1];
  const bool g2 = a.ngroups > 2 && n0 >= a.gcol[2];
  r.g = g2 ? 2 : (g1 ? 1 : 0);
  r.codes = g2 ? a.gcodes[2] : (g1 ? a.gcodes[1] : a.gcodes[0]);
  r.absmax = g2 ? a.gabsmax[2] : (g1 ? a.gabsmax[1] : a.gabsmax[0]);
  r.lora_F = g2 ? a.glora_F[2] : (g1 ? a.glora_F[1] : a.glora_F[0]);
  r.out = g2 ? a.gout[2] : (g1 ? a.gout[1] : a.gout[0]);
  r.c0 = g2 ? a.gcol[2] : (g1 ? a.gcol[1] : 0);
  const int64_t c1 = g2 ? a.gcol[3] : (g1 ? a.gcol[2] : a.gcol[1]);
  r.width = c1 - r.c0;
  return r;
}

// Position of a (tile, step) iteration: step i of tile (mt, nt).
struct Pos {
  int i, mt, nt;
  WS_DEVINL void next(int S, int mtiles) {
    if (++i == S) {
      i = 0;
      if (++mt == mtiles) {
        mt = 0;
        ++nt;
      }
    }
  }
};

// PAIR != 0: the CTA is one of a cluster of two that share each weight
// tile.  The pair covers 2 * BM activation rows (rank r takes rows r * BM
// ...) and each CTA dequantises half of the tile's weight columns, so every
// weight is decoded once per 512 rows instead of once per 256.
//   PAIR = 1: each CTA copies its half into the other CTA's buffer as well
//     and issues its own MMAs; a buffer is refilled once the MMAs of both
//     CTAs that read it have completed (their commits arrive on both CTAs'
//     barriers).
//   PAIR = 2: the even CTA issues one M = 256 MMA for both CTAs
//     (cta_group::2): the tensor cores read each CTA's activation rows and
//     weight half where they lie, and each CTA's accumulator rows land in its
//     own tensor memory.  The odd CTA's activation copies, dequant warps and
//     epilogue warps signal the even CTA's barriers; the even CTA's commits
//     arrive on both CTAs' barriers.  Nothing is copied between the CTAs.
// The stream-K schedule runs over pairs; partial tiles and their flags stay
// per CTA.
// Tensor maps of bf16 weights (WB): the forward's group g uses m[g] (box 64
// x BW rows of W [N_g, K]); the backward uses m[0] (box 64 x 64).
struct WMaps {
  CUtensorMap m[kMaxGroups];
};

template <bool BWD, int UM, int BN, int PAIR, bool WB>
__global__ void __launch_bounds__(kThreads, 1)
    k_nf4_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmL,
               const GemmArgs args, const __grid_constant__ WMaps wm) {
  using C = Cfg<BWD, UM, BN, PAIR, WB>;
  constexpr int STAGES = C::STAGES;
  constexpr int BSTAGES = C::BSTAGES;
  constexpr int NACC = C::ACC_BUFS;
  constexpr bool PM = C::PM;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + C::OFF_A;
  uint8_t* sB = smem + C::OFF_B;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = full + STAGES;
  uint64_t* bfull = empty + STAGES;
  uint64_t* bempty = bfull + BSTAGES;
  uint64_t* accfull = bempty + BSTAGES;
  uint64_t* accempty = accfull + NACC;
  uint64_t* drain = accempty + NACC;
  uint64_t* lora_done = drain + 1;    // backward: the tile's LoRA step has completed
  uint64_t* lora_masked = drain + 2;  // backward: ... and the epilogue masked it
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  uint32_t* tmem_slot = misc;
  volatile uint32_t* abort_flag = misc + 1;
  volatile uint32_t* skip_flag = misc + 2;
  volatile uint32_t* fin_got = misc + 3;

  const int warp = (int)warp_id();
  const int lane = (int)lane_id();
  const int rank = PAIR ? (int)(cluster_ctarank() & 1u) : 0;
  // ---- static stream-K schedule over units (CTAs, or pairs of CTAs)
  const int S = args.nk_total + (args.has_lora ? 1 : 0);  // steps per tile
  // the LoRA step: last in the forward, first in the backward (where it is
  // masked before the main steps accumulate on top); kc = contraction step
  const bool lora_first = BWD && args.has_lora;
  auto is_lora_step = [&](int i) {
    return args.has_lora && (lora_first ? i == 0 : i == args.nk_total);
  };
  auto kstep = [&](int i) { return lora_first ? i - 1 : i; };
  const int64_t T = (int64_t)args.mtiles * args.ntiles;
  // ranges are cut over SV = S + epad iterations per tile; the last epad
  // carry no work (a range boundary inside them moves to the next tile)
  const int64_t SV = S + args.epad;
  const int64_t I = T * SV;
  const int64_t U = PAIR ? gridDim.x / 2 : gridDim.x;
  const int64_t unit = PAIR ? blockIdx.x / 2 : blockIdx.x;
  auto real_of = [&](int64_t v) -> int64_t {
    const int64_t t = v / SV, i = v % SV;
    return i >= S ? (t + 1) * S : t * S + i;
  };
  const int64_t pb = real_of(sk_begin(unit, I, U));
  const int64_t pe = real_of(sk_begin(unit + 1, I, U));
  const Pos pos0 = {(int)(pb % S), (int)((pb / S) % args.mtiles), (int)((pb / S) / args.mtiles)};
  constexpr int UROWS = PAIR ? 2 * C::BM : C::BM;  // activation rows per tile

  // a pair kernel launched without its two-CTA clusters has no partner to
  // share with: record the configuration error and do nothing
  const bool bad_cfg = PAIR && (cluster_nctarank() != 2u || (gridDim.x & 1u) != 0u);
  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    if (bad_cfg) atomicOr(&g_dev_error, DERR_BAD_CONFIG);
    // an earlier kernel already gave up: do nothing rather than queue more work
    *skip_flag = (bad_cfg || *(volatile uint32_t*)&g_dev_error != 0u || pe <= pb) ? 1u : 0u;
    for (int s = 0; s < STAGES; ++s) {
      // merged: the even CTA's full[s] also counts both CTAs' weight halves
      // (its own dequant warps and the odd CTA's forwarding thread)
      const bool dq_here = C::MERGED && rank == 0 && (!C::PAIRSTEP || (s & 1) == 0);
      mbar_init(&full[s], dq_here ? 1 + kDqWarps + 1 : 1);
      mbar_init(&empty[s], 1);
    }
    // PAIR = 2: the even CTA's full / bfull / accempty / lora_masked count
    // both CTAs' producers and epilogues: the odd CTA's dequant warps arrive
    // on its own bfull, and one forwarding thread passes each completed
    // phase on to the even CTA (one remote arrival per handover instead of
    // one per warp)
    for (int b = 0; b < BSTAGES; ++b) {
      mbar_init(&bfull[b], (PM && rank == 0) ? kDqWarps + 1 : kDqWarps);
      mbar_init(&bempty[b], PAIR == 1 ? 2 : 1);
    }
    for (int a = 0; a < NACC; ++a) {
      mbar_init(&accfull[a], 1);
      mbar_init(&accempty[a], PM ? 2 * kEpiWarps : kEpiWarps);
    }
    mbar_init(drain, 1);
    mbar_init(lora_done, 1);
    mbar_init(lora_masked, PM ? 2 * kEpiWarps : kEpiWarps);
    fence_barrier_init();
  }
  if (warp == 1) {
    if constexpr (PM) {
      // both CTAs of the pair allocate together; without a pair nothing runs
      if (!bad_cfg) {
        tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
        tmem_relinquish_pair();
      }
    } else {
      tmem_alloc(tmem_slot, C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  // both CTAs of a pair have their barriers set up before either arrives remotely
  if (PAIR && !bad_cfg) cluster_sync();
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool skip = *skip_flag != 0u;
  // setup done: from here on the earlier kernels' data is read and written
  pdl_wait();
  pdl_launch_dependents();

  if (!skip) {
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer (activations)
      if (lane == 0) {
        tma_prefetch_desc(&tmA);
        if (args.has_lora) tma_prefetch_desc(&tmL);
        int64_t issued = 0;
        int s = 0;
        uint32_t ph = 0;
        Pos ps = pos0;
        for (int64_t q = 0; q < pe - pb; ++q) {
          if (*abort_flag || !mbar_wait(&empty[s], ph ^ 1u, DERR_TIMEOUT_EMPTY)) {
            *abort_flag = 1u;
            break;
          }
          const int m0 = ps.mt * UROWS + rank * C::BM;
          const CUtensorMap* map = is_lora_step(ps.i) ? &tmL : &tmA;
          const int32_t x = is_lora_step(ps.i) ? 0 : kstep(ps.i) * 64;
          // a grouped forward's LoRA activation rows of group g start at g * M
          const int32_t y = m0 + ((!BWD && is_lora_step(ps.i)) ? (int32_t)(tile_grp(args, (int64_t)ps.nt * BN).g * args.M) : 0);
          if constexpr (PM) {
            // both CTAs' tiles complete on the even CTA's barrier
            if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * C::A_BYTES);
            tma_load_2d_pair(sA + s * C::A_BYTES, map, mapa_shared(smem_u32(&full[s]), 0u), x, y);
          } else {
            mbar_arrive_expect_tx(&full[s], C::A_BYTES);
            tma_load_2d(sA + s * C::A_BYTES, map, &full[s], x, y);
          }
          issued = q + 1;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
          ps.next(S, args.mtiles);
        }
        if (*abort_flag) {
          // let every issued copy land before the CTA can exit
          if ((!PM || rank == 0) && !C::MERGED) {
            for (int64_t q = (issued > STAGES ? issued - STAGES : 0); q < issued; ++q)
              mbar_wait(&full[q % STAGES], (uint32_t)(q / STAGES) & 1u, DERR_TIMEOUT_DRAIN);
          } else if (issued > 0) {
            // the odd CTA's copies complete on the even CTA's barriers: give
            // them time to land (a tile copy takes microseconds)
            const uint64_t t0 = globaltimer();
            while (globaltimer() - t0 < 200000ull) __nanosleep(1000);
          }
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // (PAIR = 2: the even CTA's thread issues for both CTAs)
      if (lane == 0 && (!PM || rank == 0)) {
        constexpr uint32_t MMA_M = PM ? 256 : 128;
        constexpr uint32_t idesc_main = idesc_bf16_f32(MMA_M, BN, BWD ? 1u : 0u);
        constexpr uint32_t idesc_kmaj = idesc_bf16_f32(MMA_M, BN, 0u);
        int64_t seg = 0;
        int ms_s = 0, ms_b = 0;
        uint32_t ms_ph = 0, ms_bph = 0;
        uint32_t lora_ph = 0;
        for (int64_t p = pb; p < pe && !*abort_flag; ++seg) {
          const int64_t t = p / S;
          const int64_t seg_end = min(pe, (t + 1) * S);
          const int a = (int)(seg % NACC);
          const uint32_t aph = (uint32_t)(seg / NACC) & 1u;
          const bool acc_ok = PM ? mbar_wait_cluster(&accempty[a], aph ^ 1u, DERR_TIMEOUT_ACC)
                                 : mbar_wait(&accempty[a], aph ^ 1u, DERR_TIMEOUT_ACC);
          if (!acc_ok) {
            *abort_flag = 1u;
            break;
          }
          tc_fence_after();
          const uint32_t dbase = tmem + (uint32_t)(a * C::ACC_COLS);
          int i = (int)(p % S);
          for (int64_t p2 = p; p2 < seg_end; ++p2, ++i) {
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
            bool ok = !*abort_flag;
            if constexpr (C::MERGED) {
              ok = ok && mbar_wait_cluster(&full[s], ph, DERR_TIMEOUT_FULL);
            } else {
              ok = ok && mbar_wait(&full[s], ph, DERR_TIMEOUT_FULL);
              if constexpr (PAIR != 0) ok = ok && mbar_wait_cluster(&bfull[b], bph, DERR_TIMEOUT_BFULL);
              else ok = ok && mbar_wait(&bfull[b], bph, DERR_TIMEOUT_BFULL);
            }
            if (!ok) {
              *abort_flag = 1u;
              break;
            }
            tc_fence_after();
            const bool is_lora = is_lora_step(i);
            // The descriptors of this step's operands are built once; each
            // 16-deep slice and 128-row atom is then a plain add to the
            // start-address field (address >> 4, which stays below 2^14 in
            // shared memory, so the adds never carry out of the field).
            const uint64_t adesc0 = smem_desc_sw128(smem_u32(sA + s * C::A_BYTES), 16, 1024);
            const bool kmaj = !BWD || is_lora;
            const uint64_t bdesc0 =
                kmaj ? smem_desc_sw128(smem_u32(sB + b * C::B_BYTES), 16, 1024)
                     : smem_desc_sw128(smem_u32(sB + b * C::B_BYTES), C::MN_LBO, C::MN_SBO);
            const uint64_t bstep = kmaj ? 2u : (uint64_t)(C::MN_KK >> 4);
            const uint32_t idesc = is_lora ? idesc_kmaj : idesc_main;
            const uint32_t first = p2 > p ? 1u : 0u;  // accumulate from the first slice on
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bdesc = bdesc0 + (uint64_t)kk * bstep;
#pragma unroll
              for (int u = 0; u < UM; ++u) {
                const uint64_t adesc = adesc0 + (uint64_t)(u * 1024 + kk * 2);
                const uint32_t d = dbase + (uint32_t)(u * BN);
                const uint32_t acc = kk > 0 ? 1u : first;
                if constexpr (PM) tc_mma_f16_pair(d, adesc, bdesc, idesc, acc);
                else tc_mma_f16(d, adesc, bdesc, idesc, acc);
              }
            }
            if constexpr (C::MERGED) {
              tc_commit_pair_multicast(&empty[s], (uint16_t)0x3);
            } else if constexpr (PM) {
              tc_commit_pair_multicast(&empty[s], (uint16_t)0x3);
              tc_commit_pair_multicast(&bempty[b], (uint16_t)0x3);
            } else {
              tc_commit(&empty[s]);
              if constexpr (PAIR == 1) tc_commit_multicast(&bempty[b], (uint16_t)0x3);
              else tc_commit(&bempty[b]);
            }
            if (BWD && is_lora) {
              // the epilogue masks s G A in TMEM before the main steps add on top
              if constexpr (PM) tc_commit_pair_multicast(lora_done, (uint16_t)0x3);
              else tc_commit(lora_done);
              const bool lm_ok = PM ? mbar_wait_cluster(lora_masked, lora_ph, DERR_TIMEOUT_ACC)
                                    : mbar_wait(lora_masked, lora_ph, DERR_TIMEOUT_ACC);
              if (!lm_ok) {
                *abort_flag = 1u;
                break;
              }
              lora_ph ^= 1u;
              tc_fence_after();
            }
          }
          if constexpr (PM) tc_commit_pair_multicast(&accfull[a], (uint16_t)0x3);
          else tc_commit(&accfull[a]);
          p = seg_end;
        }
        // every MMA this thread issued has completed before TMEM is freed
        if constexpr (PM) tc_commit_pair(drain);
        else tc_commit(drain);
        mbar_wait(drain, 0u, DERR_TIMEOUT_DRAIN);
      } else if (PM && lane == 0) {
        // odd CTA: forward each completed weight-buffer phase to the even CTA
        int b = 0;
        uint32_t bph = 0;
        constexpr int QS = C::PAIRSTEP ? 2 : 1;  // steps per handover
        for (int64_t q = 0; q < pe - pb; q += QS) {
          if (*abort_flag || !mbar_wait(&bfull[b], bph, DERR_TIMEOUT_BFULL)) {
            *abort_flag = 1u;
            break;
          }
          mbar_arrive_remote(mapa_shared(smem_u32(C::MERGED ? &full[b] : &bfull[b]), 0u));
          if ((b += QS) >= BSTAGES) {
            b -= BSTAGES;
            bph ^= 1u;
          }
        }
      }
    } else if (warp < 2 + kDqWarps) {
      // ------------------------------------------------------------ dequant producers
      // Codes and scales are copied from global memory into this thread's
      // ring slots CSTAGES - 1 steps ahead of their use; a weight buffer is
      // refilled once the MMAs that read it have completed.
      constexpr int CS = C::CSTAGES;
      const int t_idx = (int)threadIdx.x - 64;
      const int64_t n_it = pe - pb;
      uint8_t* ring = smem + C::OFF_CODE;
      const uint32_t peer = (uint32_t)(rank ^ 1);
      int b = 0;
      uint32_t bph = 0;
      Pos pc = pos0;  // position of the step being dequantised
      Pos pf = pos0;  // position of the next fetch
      int64_t fq = 0;
      auto fetch = [&]() {
        if (!WB && !C::REG_CODES && fq < n_it && !is_lora_step(pf.i)) {
          const uint32_t slot = smem_u32(ring + (fq % CS) * C::CODE_BYTES);
          const int64_t nb = (int64_t)pf.nt * BN;
          if constexpr (BWD) {
            fetch_codes<BWD, BN, PAIR>(slot, args.codes, args.absmax, args.wN, args.wK,
                                       kstep(pf.i), nb, rank, t_idx);
          } else {
            const TileGrp tg = tile_grp(args, nb);
            fetch_codes<BWD, BN, PAIR>(slot, tg.codes, tg.absmax, tg.width, args.wK, kstep(pf.i),
                                       nb - tg.c0, rank, t_idx);
          }
        }
        cp_async_commit();
        pf.next(S, args.mtiles);
        ++fq;
      };
      // register pipeline: f0, f1 hold the codes of the next two steps
      Frag f0{}, f1{};
      auto load_next = [&](Frag& f) {
        if (!WB && C::REG_CODES && fq < n_it && !is_lora_step(pf.i)) {
          const int64_t nb = (int64_t)pf.nt * BN;
          if constexpr (BWD) {
            load_frag<BWD, BN, PAIR>(f, args.codes, args.absmax, args.wN, args.wK, kstep(pf.i),
                                     nb, rank, t_idx);
          } else {
            const TileGrp tg = tile_grp(args, nb);
            load_frag<BWD, BN, PAIR>(f, tg.codes, tg.absmax, tg.width, args.wK, kstep(pf.i),
                                     nb - tg.c0, rank, t_idx);
          }
        }
        pf.next(S, args.mtiles);
        ++fq;
      };
      if constexpr (!WB && C::REG_CODES) {
        load_next(f0);
        load_next(f1);
      }
      // paired steps keep one ring slot more between a read and its refill
#pragma unroll 1
      for (int k = 0; k < CS - (C::PAIRSTEP ? 2 : 1); ++k)
        if constexpr (!WB && !C::REG_CODES) fetch();
      // Fill weight buffer bb for the step at position ps: decode the codes
      // in cur, build the LoRA factor tile, or (bf16 weights) have one
      // thread load the tile (this CTA's half of it in a pair) with TMA,
      // whose arrival carries the bytes.  Returns whether the tile came by TMA.
      auto fill = [&](const Frag& cur, int bb, const Pos& ps) -> bool {
        uint8_t* Bt = sB + bb * C::B_BYTES;
        const bool lora_step = is_lora_step(ps.i);
        const bool tma_step = WB && !lora_step;
        if (!lora_step) {
          if constexpr (WB) {
            if (warp == 2 && lane == 0) {
              const int64_t nb = (int64_t)ps.nt * BN;
              const int32_t kc = kstep(ps.i) * 64;
              const int32_t half0 = PM ? rank * C::BW : 0;
              // merged, even CTA: the stage barrier; else this CTA's buffer barrier
              uint64_t* wbar = (C::MERGED && rank == 0) ? &full[bb] : &bfull[bb];
              mbar_arrive_expect_tx(wbar, C::B_BYTES);
              if constexpr (!BWD) {
                const TileGrp tg = tile_grp(args, nb);
                const CUtensorMap* m = tg.g == 2 ? &wm.m[2] : (tg.g == 1 ? &wm.m[1] : &wm.m[0]);
                tma_load_2d(Bt, m, wbar, kc, (int32_t)(nb - tg.c0) + half0);
              } else {
#pragma unroll
                for (int j = 0; j < C::BW / 64; ++j)
                  tma_load_2d(Bt + j * 8192, &wm.m[0], wbar, (int32_t)nb + half0 + j * 64, kc);
              }
            }
          } else {
            if (!BWD) dequant_fwd<BN, PAIR>(cur, Bt, rank, t_idx);
            else dequant_bwd<BN, PAIR>(cur, Bt, rank, t_idx);
          }
        } else {
          const TileGrp tg = tile_grp(args, (int64_t)ps.nt * BN);
          lora_tile<BWD, BN, PAIR>(tg.lora_F, tg.width, tg.width, (int)((int64_t)ps.nt * BN - tg.c0),
                                   args.lora_scale, Bt, rank, t_idx);
        }
        return tma_step;
      };
      if constexpr (C::PAIRSTEP) {
        // Two steps per handover (merged pair MMA, NF4 codes): wait until the
        // later of the two buffers is free (the MMA commits complete in issue
        // order, so the earlier one is free too), fill both, then one fence
        // and one arrival on the even buffer's barrier (the odd CTA's on its
        // own buffer barrier, which its forwarding thread passes on).
        for (int64_t q = 0; q < n_it; q += 2) {
          const bool two = q + 1 < n_it;
          Frag c0, c1;
          if constexpr (C::REG_CODES) {
            c0 = f0;
            c1 = f1;
            load_next(f0);  // two steps ahead
            load_next(f1);
          } else {
            fetch();  // refill the slots read in the previous iteration
            fetch();
            cp_async_wait<CS - 2>();
            read_frag<BWD, BN, PAIR>(c0, ring + (q % CS) * C::CODE_BYTES, t_idx);
            read_frag<BWD, BN, PAIR>(c1, ring + ((q + 1) % CS) * C::CODE_BYTES, t_idx);
          }
          const int bw = two ? b + 1 : b;
          if (*abort_flag || !mbar_wait_cluster(&empty[bw], bph ^ 1u, DERR_TIMEOUT_BEMPTY)) {
            *abort_flag = 1u;
            break;
          }
          Pos p1 = pc;
          p1.next(S, args.mtiles);
          fill(c0, b, pc);
          if (two) fill(c1, b + 1, p1);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(rank == 0 ? &full[b] : &bfull[b]);
          pc = p1;
          pc.next(S, args.mtiles);
          if ((b += two ? 2 : 1) >= BSTAGES) {
            b -= BSTAGES;
            bph ^= 1u;
          }
        }
      } else {
        // One pipeline step; f holds its codes (register pipeline) and is
        // refilled with those of the step two ahead.  The loop below runs the
        // step twice per iteration, on f0 then f1, so a fragment is only
        // overwritten after its own use.
        auto dq_step = [&](int64_t q, Frag& f) -> bool {
          Frag cur;
          if constexpr (!WB && C::REG_CODES) {
            cur = f;
            load_next(f);  // the step after next
          } else if constexpr (!WB) {
            (void)f;
            fetch();  // refills the slot read in the previous iteration
            cp_async_wait<CS - 1>();
            read_frag<BWD, BN, PAIR>(cur, ring + (q % CS) * C::CODE_BYTES, t_idx);
          } else {
            (void)f;
          }
          bool ok = !*abort_flag;
          // merged: stage b's commit frees the buffer (b equals the stage index)
          uint64_t* freed = C::MERGED ? &empty[b] : &bempty[b];
          if constexpr (PAIR != 0) ok = ok && mbar_wait_cluster(freed, bph ^ 1u, DERR_TIMEOUT_BEMPTY);
          else ok = ok && mbar_wait(freed, bph ^ 1u, DERR_TIMEOUT_BEMPTY);
          if (!ok) {
            *abort_flag = 1u;
            return false;
          }
          const bool lora_step = is_lora_step(pc.i);
          const bool tma_step = fill(cur, b, pc);
          uint8_t* Bt = sB + b * C::B_BYTES;
          if (!tma_step) fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && !(tma_step && warp == 2)) {
            if constexpr (PM) {
              // the even CTA's MMA reads this half where it lies
              mbar_arrive((C::MERGED && rank == 0) ? &full[b] : &bfull[b]);
            } else if constexpr (PAIR == 1) {
              // this warp's share of the half tile is one contiguous block:
              // rows (K-major) or one 8-row contraction group (MN-major);
              // send it to the same place in the other CTA's buffer
              constexpr uint32_t kShare = C::B_BYTES / 16;
              const int dw = warp - 2;
              const uint32_t off =
                  (BWD && !lora_step)
                      ? (uint32_t)(dw * (int)C::MN_SBO + rank * (BN / 128) * 1024)
                      : (uint32_t)((rank * (BN / 2) + dw * (BN / 16)) * 128);
              mbar_arrive_expect_tx(&bfull[b], kShare);
              bulk_copy_to_peer(mapa_shared(smem_u32(Bt + off), peer), Bt + off, kShare,
                                mapa_shared(smem_u32(&bfull[b]), peer));
            } else {
              mbar_arrive(&bfull[b]);
            }
          }
          if (++b == BSTAGES) {
            b = 0;
            bph ^= 1u;
          }
          pc.next(S, args.mtiles);
          return true;
        };
        for (int64_t q = 0; q < n_it; q += 2) {
          if (!dq_step(q, f0)) break;
          if (q + 1 < n_it && !dq_step(q + 1, f1)) break;
        }
      }
      cp_async_wait<0>();  // no copy may land after the CTA is gone
      if (WB && *abort_flag && warp == 2 && lane == 0) {
        // weight tiles this thread loaded may still be in flight: give them
        // time to land (a tile copy takes microseconds)
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 200000ull) __nanosleep(1000);
      }
      if constexpr (PAIR != 0) {
        // the other CTA's MMA commits arrive on this CTA's buffer barriers:
        // wait for the last of them before the CTA can leave
        for (int k = 0; k < BSTAGES && !*abort_flag; ++k) {
          if (!mbar_wait_cluster(C::MERGED ? &empty[b] : &bempty[b], bph ^ 1u, DERR_TIMEOUT_DRAIN))
            break;
          if (++b == BSTAGES) {
            b = 0;
            bph ^= 1u;
          }
        }
      }
    } else {
      // ------------------------------------------------------------ epilogue
      // Eight warps: two per TMEM lane quarter, one for each half of the
      // tile's columns, 16 columns at a time.
      const int ew = warp - (2 + kDqWarps);
      const int q4 = warp & 3;  // TMEM lane quarter this warp may read
      const int half = ew >> 2;
      const int r = q4 * 32 + lane;
      // CTA holding this CTA's rows of the tile in unit u
      auto cta_of = [&](int64_t u) -> int64_t { return PAIR ? 2 * u + rank : u; };
      // A CTA's fp32 partial tile is stored as float4 [BN/4][BM]: element
      // (row, 4c..4c+3) at [c][row], so the 32 rows of a warp make one
      // contiguous 512-byte access per column group.
      auto part4 = [&](int64_t cta, int row, int cc) -> float4* {
        return reinterpret_cast<float4*>(args.partial + cta * C::TILE_FLOATS) +
               (int64_t)(cc / 4) * C::BM + row;
      };
      int64_t seg = 0;
      uint32_t lora_ph = 0;
      for (int64_t p = pb; p < pe; ++seg) {
        const int64_t t = p / S;
        const int64_t i0 = p % S;
        const int64_t seg_end = min(pe, (t + 1) * S);
        const int64_t kb = seg_end - t * S;
        const int a = (int)(seg % NACC);
        const uint32_t aph = (uint32_t)(seg / NACC) & 1u;
        if (lora_first && i0 == 0) {
          // the tile's first step was s G A: zero its dropped elements in
          // TMEM, then let the main steps accumulate on top
          const bool lok = !*abort_flag && mbar_wait_backoff(lora_done, lora_ph, DERR_TIMEOUT_ACC);
          lora_ph ^= 1u;
          tc_fence_after();
          const int64_t lm0 = (t % args.mtiles) * UROWS + rank * C::BM;
          const int64_t ln0 = (t / args.mtiles) * BN;
          const uint32_t lbase = tmem + (uint32_t)(a * C::ACC_COLS);
          // this thread's mask words (its row, this warp's columns), all
          // loaded at once: one memory round trip instead of one per chunk
          constexpr int MW = (BN / 2) / 32;
          uint32_t mw[UM * MW];
#pragma unroll
          for (int u = 0; u < UM; ++u) {
            const int64_t m = lm0 + u * 128 + r;
#pragma unroll
            for (int w = 0; w < MW; ++w) {
              const int64_t n = ln0 + half * (BN / 2) + 32 * w;
              mw[u * MW + w] = (lok && m < args.M && n < args.Nout) ? args.mask[(m * args.Nout + n) >> 5] : 0u;
            }
          }
#pragma unroll 1
          for (int u = 0; u < UM; ++u) {
#pragma unroll 1
            for (int cc = half * (BN / 2); cc < (half + 1) * (BN / 2); cc += 16) {
              const int64_t n = ln0 + cc;
              if (n >= args.Nout) break;  // warp-uniform
              const uint32_t taddr = lbase + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(u * BN + cc);
              uint32_t v[16];
              tmem_ld_32x32b_x16(taddr, v);
              // select word (u, (cc - half * BN/2) / 32) without indexing the array at run time
              const int wi = u * MW + (cc - half * (BN / 2)) / 32;
              uint32_t word = 0u;
#pragma unroll
              for (int w = 0; w < UM * MW; ++w) word = (w == wi) ? mw[w] : word;
              const uint32_t bits = word >> (cc & 31);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) v[e] = ((bits >> e) & 1u) ? v[e] : 0u;
              tmem_st_32x32b_x16(taddr, v);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (PM && rank == 1) mbar_arrive_remote(mapa_shared(smem_u32(lora_masked), 0u));
            else mbar_arrive(lora_masked);
          }
        }
        const bool ok = !*abort_flag && mbar_wait_backoff(&accfull[a], aph, DERR_TIMEOUT_ACC);
        tc_fence_after();
        const int64_t m0 = (t % args.mtiles) * UROWS + rank * C::BM;
        const int64_t n0 = (t / args.mtiles) * BN;
        const bool whole = (i0 == 0 && kb == S);
        // the tile's first steps with the rest held by later units: finish it here
        const bool finisher = (i0 == 0 && kb < S);
        const bool writer = !whole && !finisher;  // a later piece: hand it over
        (void)kb;
        int64_t u_last = unit;
        if (finisher) {
          u_last = sk_cta_of(t * SV + S - 1, I, U);  // unit holding the tile's last step
          // one thread waits for the later pieces (each CTA publishes at
          // most one); the barrier passes what it acquired to the others
          if (ew == 0 && lane == 0) {
            bool got = ok;
            for (int64_t u = unit + 1; u <= u_last && got; ++u)
              got = wait_flag_bounded(args.flags + cta_of(u), 1u, kWaitLimitNs, DERR_TIMEOUT_PEER);
            *fin_got = got ? 1u : 0u;
            // consumed: the flags go back to zero for the next launch using them
            if (got)
              for (int64_t u = unit + 1; u <= u_last; ++u) args.flags[cta_of(u)] = 0u;
          }
          named_bar_sync(2, kEpiWarps * 32);
          if (*fin_got == 0u) u_last = unit;  // timed out: store what is here, flagged as an error
        }
        const uint32_t dbase = tmem + (uint32_t)(a * C::ACC_COLS);
        // 16-column chunks of this warp's columns that lie inside the output
        // (of this tile's linear, for a grouped forward)
        const TileGrp og = tile_grp(args, n0);
        // 32-byte stores need 32-byte aligned rows of the output
        const bool v8_out = (reinterpret_cast<uintptr_t>(og.out) & 31u) == 0u &&
                            (og.width & (args.out_f32 ? 7 : 15)) == 0;
        constexpr int KCH = (BN / 2) / 16;
        const int64_t cols_left = og.width - (n0 - og.c0 + half * (BN / 2));
        const int kv = cols_left <= 0 ? 0 : (cols_left >= KCH * 16 ? KCH : (int)((cols_left + 15) / 16));
        // A finisher's segment is its unit's last, so the main loop's shared
        // memory is idle: the later pieces stream through a per-warp ring of
        // kFinRing cp.async entries there (entry = one piece's 32 rows x 16
        // columns), consumed chunk by chunk in step order.
        const int P = finisher ? (int)(u_last - unit) : 0;
        const uint32_t r_base = smem_u32(smem) + (uint32_t)(ew * kFinRing * 2048 + lane * 16);
        // Entries are issued in consumption order -- chunk k = (u, c) of this
        // warp, then piece 1 .. P -- with the position kept as counters (no
        // divisions in the loop).  Every call commits one group, so group g
        // always holds entry g (or nothing, past the last); an entry is
        // refilled right after it is consumed, so the slot to fill is always
        // the one just read.
        int ri_pp = 1, ri_k = 0, slot = 0;
        auto r_issue = [&](int into) {
          if (ri_k < UM * kv) {
            const int u = (UM == 2 && ri_k >= kv) ? 1 : 0;
            const float4* src = part4(cta_of(unit + ri_pp), u * 128 + r, half * (BN / 2) + (ri_k - u * kv) * 16);
            const uint32_t dst = r_base + (uint32_t)(into * 2048);
#pragma unroll
            for (int e = 0; e < 4; ++e) cp_async16(dst + (uint32_t)(e * 512), src + (int64_t)e * C::BM, 16u);
            if (++ri_pp > P) {
              ri_pp = 1;
              ++ri_k;
            }
          }
          cp_async_commit();
        };
        if (P > 0)
          for (int j = 0; j < kFinRing; ++j) r_issue(j);
#pragma unroll 1
        for (int u = 0; u < UM; ++u) {
          const int row = u * 128 + r;
          const int64_t m = m0 + row;
          const bool row_ok = ok && m < args.M;
#pragma unroll 1
          for (int c = 0; c < kv; ++c) {
            const int cc = half * (BN / 2) + c * 16;
            const int64_t n = n0 + cc;
            uint32_t acc[16];
            const uint32_t taddr = dbase + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(u * BN + cc);
            tmem_ld_32x32b_x16(taddr, acc);
            tmem_ld_wait();
            float v[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(acc[e]);
            if (writer) {
              if (!row_ok) continue;
              float4* dst = part4(blockIdx.x, row, cc);
#pragma unroll
              for (int e = 0; e < 4; ++e)
                dst[(int64_t)e * C::BM] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
              continue;
            }
            // finisher: add the later pieces in step order (every thread
            // consumes its ring entries, rows past M included)
            for (int pp = 0; pp < P; ++pp) {
              cp_async_wait<kFinRing - 1>();
              const float4* sl = reinterpret_cast<const float4*>(
                  smem + ew * kFinRing * 2048 + slot * 2048 + lane * 16);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float4 q = sl[e * 32];
                v[4 * e] += q.x;
                v[4 * e + 1] += q.y;
                v[4 * e + 2] += q.z;
                v[4 * e + 3] += q.w;
              }
              r_issue(slot);
              if (++slot == kFinRing) slot = 0;
            }
            if (!row_ok) continue;
            const int64_t o_off = m * og.width + (n - og.c0);
            if (v8_out) {
              // one 32-byte store per 8 fp32 or 16 bf16 values: whole
              // sectors (16-byte stores of the rows of a warp write half
              // sectors and held every accumulator drain back)
              if (args.out_f32) {
                float* dst = static_cast<float*>(og.out) + o_off;
                if (args.out_accum) {
                  uint32_t q[16];
                  ld_global_v8(dst, q);
                  ld_global_v8(dst + 8, q + 8);
#pragma unroll
                  for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(q[e]) + v[e];
                }
                st_global_v8(dst, __float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                             __float_as_uint(v[3]), __float_as_uint(v[4]), __float_as_uint(v[5]),
                             __float_as_uint(v[6]), __float_as_uint(v[7]));
                st_global_v8(dst + 8, __float_as_uint(v[8]), __float_as_uint(v[9]), __float_as_uint(v[10]),
                             __float_as_uint(v[11]), __float_as_uint(v[12]), __float_as_uint(v[13]),
                             __float_as_uint(v[14]), __float_as_uint(v[15]));
              } else {
                st_global_v8(static_cast<uint16_t*>(og.out) + o_off, pack_bf16x2(v[0], v[1]),
                             pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]),
                             pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]),
                             pack_bf16x2(v[12], v[13]), pack_bf16x2(v[14], v[15]));
              }
            } else if (args.out_f32) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(og.out) + o_off);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float4 o = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                if (args.out_accum) {
                  const float4 q = dst[e];
                  o.x = q.x + o.x;
                  o.y = q.y + o.y;
                  o.z = q.z + o.z;
                  o.w = q.w + o.w;
                }
                dst[e] = o;
              }
            } else {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(og.out) + o_off);
#pragma unroll
              for (int e = 0; e < 2; ++e)
                dst[e] = make_uint4(pack_bf16x2(v[8 * e], v[8 * e + 1]),
                                    pack_bf16x2(v[8 * e + 2], v[8 * e + 3]),
                                    pack_bf16x2(v[8 * e + 4], v[8 * e + 5]),
                                    pack_bf16x2(v[8 * e + 6], v[8 * e + 7]));
            }
          }
        }
        if (P > 0) cp_async_wait<0>();
        if (writer) {
          // publish the piece: every epilogue thread's stores, then one flag
          __threadfence();
          named_bar_sync(1, kEpiWarps * 32);
          if (ew == 0 && lane == 0) st_release_gpu(args.flags + blockIdx.x, 1u);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PM && rank == 1) mbar_arrive_remote(mapa_shared(smem_u32(&accempty[a]), 0u));
          else mbar_arrive(&accempty[a]);
        }
        p = seg_end;
      }
    }
  }

  tc_fence_before();
  // neither CTA of a pair leaves while the other may still write into it
  if (PAIR && !bad_cfg) cluster_sync();
  else __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    if constexpr (PM) {
      if (!bad_cfg) tmem_dealloc_pair(tmem, C::TMEM_COLS);
    } else {
      tmem_dealloc(tmem, C::TMEM_COLS);
    }
  }
}

// ------------------------------------------------------------------------ LoRA weight gradients
// out[c][j] = s * sum_m P[m][j] * Q~[m][c] (dB: P = U, Q = dY; dA: P = G,
// Q = x under the dropout mask) as a tensor-core GEMM D = P^T Q:
//   A = [P_hi^T ; P_lo^T ; 0] (128 rows x 64 tokens per step, bf16 high /
//       low parts of the fp32 P), built in shared memory by four warps,
//   B = Q tile (64 tokens x 128 columns, MN-major, two TMA boxes of 64
//       columns), masked in shared memory by the same warps for dA,
//   D = 128 x 128 fp32 in TMEM; rows j and 16+j add up to P^T Q.
// One CTA per 128 columns runs every token step, so the sum over tokens
// has one fixed order and the result is written straight out.
// Element g of a parameter array, chosen with compares (no run-time indexing).
template <class T>
WS_DEVINL T pick_group(const T (&a)[kMaxGroups], int g) {
  return g == 2 ? a[2] : (g == 1 ? a[1] : a[0]);
}

// Launch parameters of the weight-gradient kernel: group g = blockIdx.y
// (LoRA factors of linears with the same M and C in one launch).
struct WgArgs {
  CUtensorMap tmQ[kMaxGroups];
  const float* P[kMaxGroups];
  const uint32_t* mask[kMaxGroups];
  float* out[kMaxGroups];
  int64_t M, C;
  float s;
  int transpose_out;
  int accumulate;  // out = out + s P^T Q~ (gradient accumulation) instead of overwriting
};
constexpr int kWgThreads = 192;
constexpr int kWgStages = 4;
constexpr int kWgBN = 128;
constexpr uint32_t kWgA = 128 * 128;     // A stage bytes
constexpr uint32_t kWgB = 2 * 64 * 128;  // B stage bytes (2 boxes of 64 tokens x 128 B)
constexpr uint32_t kWgP = 64 * 16 * 4;   // P rows of one step, fp32
constexpr uint32_t kWgMw = 8 * 128 * 4;  // mask words of one step, 8 per builder thread
constexpr uint32_t kWgSmem =
    kWgStages * (kWgA + kWgB + kWgP + kWgMw) + (3 * kWgStages + 1) * 8 + 16 + 1024;

template <bool MASKED>
__global__ void __launch_bounds__(kWgThreads, 1)
    k_wgrad_tc(const __grid_constant__ WgArgs wa) {
  // group g = blockIdx.y: its own Q, P, mask and output (same M, C, s)
  const int grp = (int)blockIdx.y;
  const CUtensorMap* tmQ = grp == 2 ? &wa.tmQ[2] : (grp == 1 ? &wa.tmQ[1] : &wa.tmQ[0]);
  const float* __restrict__ P = pick_group(wa.P, grp);
  const uint32_t* __restrict__ mask = pick_group(wa.mask, grp);
  float* __restrict__ out = pick_group(wa.out, grp);
  const int64_t M = wa.M, C = wa.C;
  const float s = wa.s;
  const int transpose_out = wa.transpose_out;
  const bool accumulate = wa.accumulate != 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kWgStages * kWgA;
  uint8_t* sP = sB + kWgStages * kWgB;
  uint8_t* sMw = sP + kWgStages * kWgP;
  uint64_t* full = reinterpret_cast<uint64_t*>(sMw + kWgStages * kWgMw);
  uint64_t* ready = full + kWgStages;
  uint64_t* empty = ready + kWgStages;
  uint64_t* accfull = empty + kWgStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accfull + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* skip_flag = tmem_slot + 2;
  const int warp = (int)warp_id(), lane = (int)lane_id();
  const int64_t c0 = (int64_t)blockIdx.x * kWgBN;
  const int nsteps = (int)((M + 63) / 64);
  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    *skip_flag = (*(volatile uint32_t*)&g_dev_error != 0u || nsteps <= 0) ? 1u : 0u;
    for (int i = 0; i < kWgStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&ready[i], 4);
      mbar_init(&empty[i], 1);
    }
    mbar_init(accfull, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kWgBN);
    tmem_relinquish();
  }
  // rows 32..127 of every A stage stay zero
  for (uint32_t o = threadIdx.x * 16; o < kWgStages * kWgA; o += kWgThreads * 16)
    *reinterpret_cast<uint4*>(sA + o) = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_launch_dependents();
  if (*skip_flag == 0u) {
    if (warp == 0) {
      if (lane == 0) {
        int64_t issued = 0;
        for (int i = 0; i < nsteps; ++i) {
          const int st = i % kWgStages;
          const uint32_t ph = (uint32_t)(i / kWgStages) & 1u;
          if (*abort_flag || !mbar_wait(&empty[st], ph ^ 1u, DERR_TIMEOUT_EMPTY)) {
            *abort_flag = 1u;
            break;
          }
          const int t0 = i * 64;
          const int64_t rows = M - t0 < 64 ? M - t0 : 64;
          mbar_arrive_expect_tx(&full[st], kWgB + (uint32_t)rows * 64u);
          tma_load_2d(sB + st * kWgB, tmQ, &full[st], (int)c0, t0);
          tma_load_2d(sB + st * kWgB + 8192, tmQ, &full[st], (int)(c0 + 64), t0);
          bulk_load(sP + st * kWgP, P + (int64_t)t0 * 16, (uint32_t)rows * 64u, &full[st]);
          issued = i + 1;
        }
        if (*abort_flag)
          for (int64_t i = (issued > kWgStages ? issued - kWgStages : 0); i < issued; ++i)
            mbar_wait(&full[i % kWgStages], (uint32_t)(i / kWgStages) & 1u, DERR_TIMEOUT_DRAIN);
      }
    } else if (warp == 1) {
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_bf16_f32(128, kWgBN, 1u);
        for (int i = 0; i < nsteps; ++i) {
          const int st = i % kWgStages;
          const uint32_t ph = (uint32_t)(i / kWgStages) & 1u;
          if (*abort_flag || !mbar_wait(&ready[st], ph, DERR_TIMEOUT_FULL)) {
            *abort_flag = 1u;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + st * kWgA);
          const uint32_t b_base = smem_u32(sB + st * kWgB);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_f16(tmem, smem_desc_sw128(a_base + kk * 32, 16, 1024),
                       smem_desc_sw128(b_base + kk * 2048, 8192, 1024), idesc,
                       (i > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&empty[st]);
        }
        tc_commit(accfull);
      }
    } else {
      // ---- warps 2-5: build the A tile from P and (dA) mask the Q tile
      // P rows arrive with the Q tile; this thread's dropout-mask words are
      // copied into its own ring slots kWgStages - 1 steps ahead.
      const int t = (int)threadIdx.x - 64;  // 0..127
      const int jj = t & 15, tg = t >> 4;   // P column, 8-token group
      auto fetch_mask = [&](int i) {
        if (MASKED && i < nsteps) {
          const int64_t t0 = (int64_t)i * 64;
          const uint32_t slot = smem_u32(sMw + (i % kWgStages) * kWgMw);
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int ch = t + it * 128;  // 0..1023: token row r, 8-column chunk q
            const int r = ch >> 4, q = ch & 15;
            const int64_t m = t0 + r, c = c0 + q * 8;
            const bool in = m < M && c < C;
            cp_async4(slot + (uint32_t)((it * 128 + t) * 4), mask + (in ? (m * C + c) >> 5 : 0),
                      in ? 4u : 0u);
          }
        }
        cp_async_commit();
      };
#pragma unroll 1
      for (int k = 0; k < kWgStages - 1; ++k) fetch_mask(k);
      for (int i = 0; i < nsteps; ++i) {
        const int st = i % kWgStages;
        const uint32_t ph = (uint32_t)(i / kWgStages) & 1u;
        const int64_t t0 = (int64_t)i * 64;
        fetch_mask(i + kWgStages - 1);  // refills the slot read in the previous step
        if (*abort_flag || !mbar_wait(&full[st], ph, DERR_TIMEOUT_FULL)) {
          *abort_flag = 1u;
          break;
        }
        float pv[8];
        const float* sp = reinterpret_cast<const float*>(sP + st * kWgP);
#pragma unroll
        for (int e = 0; e < 8; ++e) pv[e] = (t0 + tg * 8 + e < M) ? sp[(tg * 8 + e) * 16 + jj] : 0.0f;
        uint32_t mw[8];
        if (MASKED) {
          cp_async_wait<kWgStages - 1>();
          const uint32_t* sm = reinterpret_cast<const uint32_t*>(sMw + st * kWgMw);
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int ch = t + it * 128;
            const int r = ch >> 4, q = ch & 15;
            mw[it] = (t0 + r < M && c0 + q * 8 < C) ? sm[it * 128 + t] : 0xFFFFFFFFu;
          }
        }
        // A rows jj (high parts) and 16 + jj (low parts), tokens 8 tg .. 8 tg + 7
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float h0 = bf16_lo(pack_bf16x2(pv[2 * e], 0.0f));
          const float h1 = bf16_lo(pack_bf16x2(pv[2 * e + 1], 0.0f));
          hi[e] = pack_bf16x2(h0, h1);
          lo[e] = pack_bf16x2(pv[2 * e] - h0, pv[2 * e + 1] - h1);
        }
        uint8_t* At = sA + st * kWgA;
        sts128(At + jj * 128 + ((tg ^ (jj & 7)) << 4), hi[0], hi[1], hi[2], hi[3]);
        sts128(At + (16 + jj) * 128 + ((tg ^ ((16 + jj) & 7)) << 4), lo[0], lo[1], lo[2], lo[3]);
        if (MASKED) {
          uint8_t* tile = sB + st * kWgB;
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int ch = t + it * 128;
            const int r = ch >> 4, q = ch & 15;
            const uint32_t bits = (mw[it] >> ((q & 3) * 8)) & 0xFFu;
            if (bits == 0xFFu) continue;
            const int b = q >> 3, q8 = q & 7;
            uint4* p4 = reinterpret_cast<uint4*>(tile + b * 8192 + r * 128 + ((q8 ^ (r & 7)) << 4));
            uint4 v = *p4;
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t keep = ((bits >> (2 * e)) & 1u ? 0x0000FFFFu : 0u) |
                                    ((bits >> (2 * e + 1)) & 1u ? 0xFFFF0000u : 0u);
              w[e] &= keep;
            }
            *p4 = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ready[st]);
      }
      cp_async_wait<0>();  // no copy may land after the CTA is gone
      if (warp == 4) {
        // rows 0..31 of D live in TMEM lanes 0..31 (lane quarter of warp 4)
        const bool ok = mbar_wait(accfull, 0u, DERR_TIMEOUT_ACC) && !*abort_flag;
        tc_fence_after();
        for (int cc = 0; cc < kWgBN; cc += 32) {
          uint32_t acc[32];
          tmem_ld_32x32b_x32(tmem + (uint32_t)cc, acc);
          tmem_ld_wait();
          const int64_t cb = c0 + cc;
          if (!ok || cb >= C) continue;  // warp-uniform
          float v[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float x = __uint_as_float(acc[e]);
            v[e] = s * (x + __shfl_xor_sync(0xffffffffu, x, 16));  // high row + low row
          }
          if (lane < 16) {
            const int ncol = (int)(C - cb < 32 ? C - cb : 32);
            if (transpose_out) {
              float* dst = out + (int64_t)lane * C + cb;
              if (ncol == 32 && ((C & 3) == 0)) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  float4 o = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                  if (accumulate) {
                    const float4 q = reinterpret_cast<const float4*>(dst)[e];
                    o = make_float4(q.x + o.x, q.y + o.y, q.z + o.z, q.w + o.w);
                  }
                  reinterpret_cast<float4*>(dst)[e] = o;
                }
              } else {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  if (e < ncol) dst[e] = accumulate ? dst[e] + v[e] : v[e];
              }
            } else {
              float* dst = out + cb * 16 + lane;
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (e < ncol) dst[(int64_t)e * 16] = accumulate ? dst[(int64_t)e * 16] + v[e] : v[e];
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kWgBN);
}

// ------------------------------------------------------------------------ LoRA skinny products
// out[m][j] = sum_k X~[m][k] * F[j][k] for the 16 LoRA columns j (U: X = x
// under the dropout mask, whose bits this kernel draws and stores, F = A;
// G: X = dY, F = B^T), on the tensor cores:
//   A operand = X tile (128 rows x 64 k, TMA, 128-byte swizzle), masked in
//       shared memory for U,
//   B operand = [F_hi ; F_mid ; F_lo] (48 rows x 64 k): the fp32 factor
//       split into three bf16 parts, built in shared memory,
//   D = 128 x 48 fp32 in TMEM; out = (D_hi + D_mid) + D_lo per column.
// CTA = one 128-row block x one chunk of k steps; each CTA stores its
// partial sums, and the last CTA of a row block (counted with an atomic)
// adds the chunks in index order and writes the result and its bf16 split.
constexpr int kSkThreads = 320;  // TMA, MMA, 8 builder warps
constexpr int kSkStages = 4;
constexpr uint32_t kSkX = 128 * 128;    // X stage bytes
constexpr uint32_t kSkF = 64 * 16 * 4;  // fp32 factor slice of one step
constexpr uint32_t kSkB = 64 * 128;     // B operand: 48 rows used of 64
constexpr uint32_t kSkSmem =
    kSkStages * (kSkX + kSkF + kSkB) + (3 * kSkStages + 1) * 8 + 16 + 1024;

// Launch parameters: group g = blockIdx.z has its own X, factor, dropout
// key and outputs (the LoRA products of several linears in one launch).
struct SkArgs {
  CUtensorMap tmX[kMaxGroups];  // X of each group (the same map for a forward group)
  CUtensorMap tmF[kMaxGroups];  // A factors [16][K] fp32 (F_KJ = false)
  const float* F[kMaxGroups];
  DropKey key[kMaxGroups];
  uint8_t* mask_bytes[kMaxGroups];
  float* partial[kMaxGroups];
  uint32_t* counters[kMaxGroups];
  float* out[kMaxGroups];
  uint16_t* ext[kMaxGroups];
  int64_t M, K;
  int steps_per_chunk;
};
// F_KJ: the factor is given as [K][16] (B), else as [16][K] (A).
template <bool MASKED, bool F_KJ>
__global__ void __launch_bounds__(kSkThreads, 1) k_skinny_tc(const __grid_constant__ SkArgs sa) {
  const int grp = (int)blockIdx.z;
  const CUtensorMap* tmX = grp == 2 ? &sa.tmX[2] : (grp == 1 ? &sa.tmX[1] : &sa.tmX[0]);
  const CUtensorMap* tmF = grp == 2 ? &sa.tmF[2] : (grp == 1 ? &sa.tmF[1] : &sa.tmF[0]);
  const float* __restrict__ F = pick_group(sa.F, grp);
  DropKey key = pick_group(sa.key, grp);
  uint8_t* __restrict__ mask_bytes = pick_group(sa.mask_bytes, grp);
  float* __restrict__ partial = pick_group(sa.partial, grp);
  uint32_t* __restrict__ counters = pick_group(sa.counters, grp);
  float* __restrict__ out = pick_group(sa.out, grp);
  uint16_t* __restrict__ ext = pick_group(sa.ext, grp);
  const int64_t M = sa.M, K = sa.K;
  const int steps_per_chunk = sa.steps_per_chunk;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sX = smem;
  uint8_t* sBop = sX + kSkStages * kSkX;
  uint8_t* sF = sBop + kSkStages * kSkB;
  uint64_t* full = reinterpret_cast<uint64_t*>(sF + kSkStages * kSkF);
  uint64_t* ready = full + kSkStages;
  uint64_t* empty = ready + kSkStages;
  uint64_t* accfull = empty + kSkStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accfull + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* flags = tmem_slot + 2;  // [0] skip, [1] this CTA finishes the row block
  const int warp = (int)warp_id(), lane = (int)lane_id();
  const int64_t m0 = (int64_t)blockIdx.x * 128;
  const int chunks = (int)gridDim.y;
  const int64_t nsteps_total = K / 64;
  const int64_t s_begin = (int64_t)blockIdx.y * steps_per_chunk;
  const int64_t s_end = min(nsteps_total, s_begin + steps_per_chunk);
  const int nsteps = (int)(s_end > s_begin ? s_end - s_begin : 0);
  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    flags[0] = (*(volatile uint32_t*)&g_dev_error != 0u) ? 1u : 0u;
    flags[1] = 0u;
    for (int i = 0; i < kSkStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&ready[i], 8);
      mbar_init(&empty[i], 1);
    }
    mbar_init(accfull, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 64);
    tmem_relinquish();
  }
  // rows 48..63 of every B-operand stage stay zero
  for (uint32_t o = threadIdx.x * 16; o < kSkStages * kSkB; o += kSkThreads * 16)
    *reinterpret_cast<uint4*>(sBop + o) = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool skip = flags[0] != 0u;
  pdl_wait();
  pdl_launch_dependents();
  if (MASKED) resolve_step(key);
  if (!skip) {
    if (warp == 0) {
      if (lane == 0 && nsteps > 0) {
        int64_t issued = 0;
        for (int i = 0; i < nsteps; ++i) {
          const int st = i % kSkStages;
          const uint32_t ph = (uint32_t)(i / kSkStages) & 1u;
          if (*abort_flag || !mbar_wait(&empty[st], ph ^ 1u, DERR_TIMEOUT_EMPTY)) {
            *abort_flag = 1u;
            break;
          }
          const int k0 = (int)((s_begin + i) * 64);
          mbar_arrive_expect_tx(&full[st], kSkX + kSkF);
          tma_load_2d(sX + st * kSkX, tmX, &full[st], k0, (int)m0);
          if (F_KJ) bulk_load(sF + st * kSkF, F + (int64_t)k0 * 16, kSkF, &full[st]);
          else {
            // two 32-column boxes, 128-byte swizzled (see the reads below)
            tma_load_2d(sF + st * kSkF, tmF, &full[st], k0, 0);
            tma_load_2d(sF + st * kSkF + kSkF / 2, tmF, &full[st], k0 + 32, 0);
          }
          issued = i + 1;
        }
        if (*abort_flag)
          for (int64_t i = (issued > kSkStages ? issued - kSkStages : 0); i < issued; ++i)
            mbar_wait(&full[i % kSkStages], (uint32_t)(i / kSkStages) & 1u, DERR_TIMEOUT_DRAIN);
      }
    } else if (warp == 1) {
      if (lane == 0 && nsteps > 0) {
        constexpr uint32_t idesc = idesc_bf16_f32(128, 48, 0u);
        for (int i = 0; i < nsteps; ++i) {
          const int st = i % kSkStages;
          const uint32_t ph = (uint32_t)(i / kSkStages) & 1u;
          if (*abort_flag || !mbar_wait(&ready[st], ph, DERR_TIMEOUT_FULL)) {
            *abort_flag = 1u;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sX + st * kSkX);
          const uint32_t b_base = smem_u32(sBop + st * kSkB);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_f16(tmem, smem_desc_sw128(a_base + kk * 32, 16, 1024),
                       smem_desc_sw128(b_base + kk * 32, 16, 1024), idesc,
                       (i > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&empty[st]);
        }
        tc_commit(accfull);
      }
    } else {
      // ---- warps 2-9: the split factor operand and (U) the dropout mask
      const int t = (int)threadIdx.x - 64;  // 0..255
      for (int i = 0; i < nsteps; ++i) {
        const int st = i % kSkStages;
        const uint32_t ph = (uint32_t)(i / kSkStages) & 1u;
        const int64_t k0 = (s_begin + i) * 64;
        // U: the dropout bits depend on the position only, so they are drawn
        // (and stored) before the tile is waited for, beside its copy
        uint32_t bits8[4];
        if (MASKED) {
#pragma unroll
          for (int it = 0; it < 4; ++it) {
            const int ch = t + it * 256;  // 0..1023: row r, 8-column chunk q
            const int64_t m = m0 + (ch >> 3);
            const uint64_t e0 = (uint64_t)m * (uint64_t)K + (uint64_t)(k0 + (ch & 7) * 8);
            bits8[it] = keep4(key, e0) | (keep4(key, e0 + 4) << 4);
            if (mask_bytes && m < M) mask_bytes[e0 >> 3] = (uint8_t)bits8[it];
          }
        }
        if (*abort_flag || !mbar_wait(&full[st], ph, DERR_TIMEOUT_FULL)) {
          *abort_flag = 1u;
          break;
        }
        if (t < 128) {
          // B rows jj, 16 + jj, 32 + jj: high, middle, low bf16 parts of
          // F[jj][k0 + 8 kc ...]
          const int jj = t & 15, kc = t >> 4;
          const float* fs = reinterpret_cast<const float*>(sF + st * kSkF);
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (F_KJ) f[e] = fs[(kc * 8 + e) * 16 + jj];
          }
          if (!F_KJ) {
            // row jj, columns 8 kc .. 8 kc + 7 of the [16][64] slice, held as
            // two [16][32] boxes whose 16-byte chunks are XOR-swizzled by the
            // row: the eight rows of a quarter warp read eight different
            // bank groups (unswizzled, the rows' 256-byte pitch put all
            // sixteen on the same banks)
            const uint8_t* half = sF + st * kSkF + (kc >> 2) * (kSkF / 2) + jj * 128;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const float4 v = *reinterpret_cast<const float4*>(half + ((((kc & 3) * 2 + q) ^ (jj & 7)) << 4));
              f[4 * q] = v.x;
              f[4 * q + 1] = v.y;
              f[4 * q + 2] = v.z;
              f[4 * q + 3] = v.w;
            }
          }
          uint32_t w[3][4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float a0 = f[2 * e], a1 = f[2 * e + 1];
#pragma unroll
            for (int part = 0; part < 3; ++part) {
              const uint32_t pk = pack_bf16x2(a0, a1);
              w[part][e] = pk;
              a0 -= bf16_lo(pk);
              a1 -= bf16_hi(pk);
            }
          }
          uint8_t* Bt = sBop + st * kSkB;
#pragma unroll
          for (int part = 0; part < 3; ++part) {
            const int row = part * 16 + jj;
            sts128(Bt + row * 128 + ((kc ^ (row & 7)) << 4), w[part][0], w[part][1], w[part][2],
                   w[part][3]);
          }
        }
        if (MASKED) {
          uint8_t* tile = sX + st * kSkX;
#pragma unroll
          for (int it = 0; it < 4; ++it) {
            const int ch = t + it * 256;  // 0..1023: row r, 8-column chunk q
            const int r = ch >> 3, q = ch & 7;
            const int64_t m = m0 + r;
            if (m >= M) continue;
            const uint32_t bits = bits8[it];
            if (bits == 0xFFu) continue;
            uint4* p4 = reinterpret_cast<uint4*>(tile + r * 128 + ((q ^ (r & 7)) << 4));
            uint4 v = *p4;
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t keep = ((bits >> (2 * e)) & 1u ? 0x0000FFFFu : 0u) |
                                    ((bits >> (2 * e + 1)) & 1u ? 0xFFFF0000u : 0u);
              w[e] &= keep;
            }
            *p4 = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ready[st]);
      }
      if (warp < 6) {
        // ---- epilogue, warps 2-5 (TMEM lane quarters 2, 3, 0, 1): this
        // chunk's partial sums of its rows
        const int q4 = warp & 3;
        const int64_t m = m0 + q4 * 32 + lane;
        const bool ok =
            nsteps == 0 || (mbar_wait(accfull, 0u, DERR_TIMEOUT_ACC) && !*abort_flag);
        tc_fence_after();
        float v[16];
        if (nsteps > 0) {
          uint32_t a[32], b[16];
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(q4 * 32) << 16), a);
          tmem_ld_32x32b_x16(tmem + ((uint32_t)(q4 * 32) << 16) + 32u, b);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            v[j] = (__uint_as_float(a[j]) + __uint_as_float(a[16 + j])) + __uint_as_float(b[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = 0.0f;
        }
        if (ok && m < M) {
          float* dst = partial + ((int64_t)blockIdx.y * M + m) * 16;
          if ((reinterpret_cast<uintptr_t>(partial) & 31u) == 0u) {
            // whole 32-byte sectors (a warp's lanes hold different rows)
            st_global_v8(dst, __float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                         __float_as_uint(v[3]), __float_as_uint(v[4]), __float_as_uint(v[5]),
                         __float_as_uint(v[6]), __float_as_uint(v[7]));
            st_global_v8(dst + 8, __float_as_uint(v[8]), __float_as_uint(v[9]), __float_as_uint(v[10]),
                         __float_as_uint(v[11]), __float_as_uint(v[12]), __float_as_uint(v[13]),
                         __float_as_uint(v[14]), __float_as_uint(v[15]));
          } else {
            float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              d4[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
          }
        }
        if (!ok) *abort_flag = 1u;
      }
      // The last chunk of this row block to finish sums them all, in chunk
      // order, with all eight warps: two threads per row, eight columns each
      // (each column's sum keeps its order), sixteen chunks in flight.
      __threadfence();
      named_bar_sync(1, 256);
      if (warp == 2 && lane == 0) {
        const uint32_t done = atomicAdd(counters + blockIdx.x, 1u);
        if (done >= (uint32_t)chunks) atomicOr(&g_dev_error, DERR_BAD_CONFIG);  // left over
        flags[1] = (done == (uint32_t)chunks - 1u) ? 1u : 0u;
      }
      named_bar_sync(1, 256);
      if (flags[1] != 0u) {
        __threadfence();
        const int h = t >> 7;  // column half
        const int64_t m = m0 + (t & 127);
        if (!*abort_flag && m < M) {
          float acc[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
          const float4* src = reinterpret_cast<const float4*>(partial + m * 16) + 2 * h;
          const int64_t cstride = M * 4;  // float4 per chunk
          int c = 0;
          for (; c + 16 <= chunks; c += 16) {
            float4 q[16][2];
#pragma unroll
            for (int u = 0; u < 16; ++u)
#pragma unroll
              for (int e = 0; e < 2; ++e) q[u][e] = __ldcg(src + (int64_t)(c + u) * cstride + e);
#pragma unroll
            for (int u = 0; u < 16; ++u)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                acc[4 * e] += q[u][e].x;
                acc[4 * e + 1] += q[u][e].y;
                acc[4 * e + 2] += q[u][e].z;
                acc[4 * e + 3] += q[u][e].w;
              }
          }
          for (; c < chunks; ++c) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float4 q = __ldcg(src + (int64_t)c * cstride + e);
              acc[4 * e] += q.x;
              acc[4 * e + 1] += q.y;
              acc[4 * e + 2] += q.z;
              acc[4 * e + 3] += q.w;
            }
          }
          float4* o = reinterpret_cast<float4*>(out + m * 16) + 2 * h;
          o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
          o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
          // [hi | lo | hi | 0] bf16 row for the tensor-core LoRA step; this
          // thread's eight columns of each part
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            hi[e] = pack_bf16x2(acc[2 * e], acc[2 * e + 1]);
            lo[e] = pack_bf16x2(acc[2 * e] - bf16_lo(hi[e]), acc[2 * e + 1] - bf16_hi(hi[e]));
          }
          uint4* x4 = reinterpret_cast<uint4*>(ext + m * 64);
          x4[h] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          x4[2 + h] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          x4[4 + h] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          x4[6 + h] = make_uint4(0u, 0u, 0u, 0u);
        }
        if (warp == 2 && lane == 0) counters[blockIdx.x] = 0u;  // ready for the next launch
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 64);
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

#ifndef WS_GEMM_EPAD
#define WS_GEMM_EPAD 10
#endif
constexpr int kEpadSteps = WS_GEMM_EPAD;

// 256-wide tiles when every unit's stream-K range covers at least this many
// (tile, step) iterations (a 256-wide pair MMA step costs about what a
// 128-wide one does; below ~20 steps per unit the finisher's partial tiles
// outweigh that: 32B q/o 44 against 41 us at 21 steps, 7B down 98 against
// 109 us at 55).
#ifndef WS_GEMM_BN256_MIN_STEPS
#define WS_GEMM_BN256_MIN_STEPS 32
#endif
constexpr int64_t kBn256MinSteps = WS_GEMM_BN256_MIN_STEPS;

// Persistent grid: one CTA per SM, but at least kMinSteps (tile, step)
// iterations per CTA so tiny problems are not shredded into partials.
constexpr int64_t kMinSteps = 8;

template <bool BWD, int UM, int BN, int PAIR, bool WB = false>
cudaError_t set_smem_attr() {
  static cudaError_t e = cudaFuncSetAttribute(k_nf4_gemm<BWD, UM, BN, PAIR, WB>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              (int)Cfg<BWD, UM, BN, PAIR, WB>::SMEM_BYTES);
  return e;
}

}  // namespace

bool tmap_bf16_sw128(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer) {
  return encode_fn() && make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, inner, outer,
                                 pitch_bytes, box_inner, box_outer,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("WS_NF4_PDL");
    return !(v && v[0] == '0');
  }();
  return on;
}

namespace {

// How a pair of CTAs shares a weight tile: 2 = one MMA across both CTAs
// (the default), 1 = each CTA issues its own MMAs on a full-width tile that
// both CTAs fill (WS_NF4_PAIR_MMA=0).
int pair_mode() {
  static const int m = [] {
    const char* v = getenv("WS_NF4_PAIR_MMA");
    return (v && v[0] == '0') ? 1 : 2;
  }();
  return m;
}

// Pairs of CTAs that can be resident at once (one CTA per SM).
template <bool BWD, int BN, int PAIR, bool WB = false>
int64_t pair_capacity_of() {
  static int64_t cap = -1;
  if (cap < 0) {
    cap = 0;
    if (set_smem_attr<BWD, 2, BN, PAIR, WB>() == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * (unsigned)(device_sm_count() / 2));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = Cfg<BWD, 2, BN, PAIR, WB>::SMEM_BYTES;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, k_nf4_gemm<BWD, 2, BN, PAIR, WB>, &cfg) == cudaSuccess)
        cap = n;
      else
        cudaGetLastError();
    } else {
      cudaGetLastError();
    }
  }
  return cap;
}

template <bool BWD, int UM, int BN, int PAIR, bool WB = false>
cudaError_t launch_cfg(const GemmPlan& p, const GemmArgs& a, const CUtensorMap& tA,
                       const CUtensorMap& tL, const WMaps& wm, cudaStream_t st) {
  using C = Cfg<BWD, UM, BN, PAIR, WB>;
  cudaError_t e = set_smem_attr<BWD, UM, BN, PAIR, WB>();
  if (e != cudaSuccess) return e;
  const int64_t G = grid_ctas(p, a.has_lora != 0);
  // the plan sizes pair grids by the NF4 kernel's residency; the bf16
  // variant (no code ring) must fit the same grid at once
  if (WB && PAIR != 0 && G / 2 > pair_capacity_of<BWD, BN, PAIR, WB>())
    return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  // The grid is sized to be resident at once, so a finisher's wait for a
  // later CTA's piece ends.  Cooperative launch guarantees it outright;
  // WS_NF4_COOP=0 drops that attribute (profilers that cannot launch
  // cooperative clusters need it).  With programmatic serialization the grid
  // may start while the previous kernel still holds SMs, which a cooperative
  // launch does not allow: CTAs the previous kernel delays start as its CTAs
  // leave (it never waits on this grid), so the bounded waits still end.
  static const bool coop = [] {
    const char* v = getenv("WS_NF4_COOP");
    return !(v && v[0] == '0');
  }();
  const bool pdl = pdl_enabled();
  cudaLaunchAttribute attr[3];
  int na = 0;
  if (coop && !pdl) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  }
  if (PAIR != 0) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 2;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  note_launch();
  return cudaLaunchKernelEx(&cfg, k_nf4_gemm<BWD, UM, BN, PAIR, WB>, tA, tL, a, wm);
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

int64_t pair_capacity(bool bwd, int bn) {
  if (pair_mode() == 2) {
    if (bwd) return bn == 256 ? pair_capacity_of<true, 256, 2>() : pair_capacity_of<true, 128, 2>();
    return bn == 256 ? pair_capacity_of<false, 256, 2>() : pair_capacity_of<false, 128, 2>();
  }
  if (bwd) return bn == 256 ? pair_capacity_of<true, 256, 1>() : pair_capacity_of<true, 128, 1>();
  return bn == 256 ? pair_capacity_of<false, 256, 1>() : pair_capacity_of<false, 128, 1>();
}

int64_t grid_units(const GemmPlan& p, bool has_lora) {
  const int64_t S = (int64_t)p.nk + (has_lora ? 1 : 0);
  const int64_t I = (int64_t)p.mtiles * p.ntiles * S;
  // at least kMinSteps iterations per unit, and at least a third of a short
  // tile, so a short tile is cut into at most about four pieces (the
  // finisher adds the pieces one after the other); long tiles fill the GPU
  int64_t min_steps = S / 3 + 2;
  if (min_steps > 64) min_steps = 64;
  if (min_steps < kMinSteps) min_steps = kMinSteps;
  int64_t G = (I + min_steps - 1) / min_steps;
  const int64_t cap = p.pair ? pair_capacity(p.bwd, p.bn) : device_sm_count();
  if (G > cap) G = cap;
  return G < 1 ? 1 : G;
}

int64_t grid_ctas(const GemmPlan& p, bool has_lora) {
  return grid_units(p, has_lora) * (p.pair ? 2 : 1);
}

GemmPlan plan_gemm(bool bwd, int64_t M, int64_t Nout, int64_t Kc) {
  GemmPlan p{};
  p.bwd = bwd;
  p.um = M > 128 ? 2 : 1;
  p.bn = 128;
  // Two CTAs of a cluster share each weight tile when there are rows for
  // both (one dequantisation per 512 activation rows).
  p.pair = M > 256 && pair_capacity(bwd, 128) > 0;
  const int64_t urows = 128 * p.um * (p.pair ? 2 : 1);
  if (p.um == 2 && (!bwd || p.pair)) {
    // A 256-wide tile reads less shared memory per flop (256-wide MMAs) but
    // has a single accumulator (no epilogue overlap): worth it when each
    // unit's stream-K range stays long enough (kBn256MinSteps).
    const int64_t units = p.pair ? pair_capacity(bwd, 256) : device_sm_count();
    const int64_t mt = (M + urows - 1) / urows, nt = (Nout + 255) / 256;
    if (units > 0 && mt * nt * (Kc / 64 + 1) >= kBn256MinSteps * units) p.bn = 256;
  }
  p.mtiles = (int)((M + urows - 1) / urows);
  p.ntiles = (int)((Nout + p.bn - 1) / p.bn);
  p.nk = (int)(Kc / 64);
  // A single accumulator (UM = 2, BN = 256) stalls the MMAs for the drain of
  // every tile a unit ends: charge it in the schedule when units end about
  // one tile each (with fewer tiles than units, ranges end mostly inside
  // tiles and the finisher's wait for the later pieces dominates).
  p.epad = 0;
  if (p.um == 2 && p.bn == 256) {
    const int64_t units = p.pair ? pair_capacity(bwd, 256) : device_sm_count();
    if (units > 0 && (int64_t)p.mtiles * p.ntiles >= units) p.epad = kEpadSteps;
  }
  return p;
}

// [G][BM][BN] fp32 partial tiles.
size_t gemm_partial_bytes(const GemmPlan& p, int64_t M, int64_t Nout) {
  (void)M;
  (void)Nout;
  const int64_t G = grid_ctas(p, true);
  if (grid_units(p, true) <= 1) return 0;
  return (size_t)G * (size_t)(128 * p.um) * (size_t)p.bn * sizeof(float);
}

namespace {
// The kernel instantiation of a plan.
cudaError_t dispatch_gemm(const GemmPlan& p, const GemmArgs& a, const CUtensorMap& tA,
                          const CUtensorMap& tL, const WMaps& wm, cudaStream_t st) {
  const bool pm = pair_mode() == 2;
  if (!p.bwd) {
    if (p.pair && pm) {
      if (p.bn == 256) return launch_cfg<false, 2, 256, 2>(p, a, tA, tL, wm, st);
      return launch_cfg<false, 2, 128, 2>(p, a, tA, tL, wm, st);
    }
    if (p.pair) {
      if (p.bn == 256) return launch_cfg<false, 2, 256, 1>(p, a, tA, tL, wm, st);
      return launch_cfg<false, 2, 128, 1>(p, a, tA, tL, wm, st);
    }
    if (p.um == 2 && p.bn == 256) return launch_cfg<false, 2, 256, 0>(p, a, tA, tL, wm, st);
    if (p.um == 2) return launch_cfg<false, 2, 128, 0>(p, a, tA, tL, wm, st);
    return launch_cfg<false, 1, 128, 0>(p, a, tA, tL, wm, st);
  }
  if (p.pair && pm) {
    if (p.bn == 256) return launch_cfg<true, 2, 256, 2>(p, a, tA, tL, wm, st);
    return launch_cfg<true, 2, 128, 2>(p, a, tA, tL, wm, st);
  }
  if (p.pair) {
    if (p.bn == 256) return launch_cfg<true, 2, 256, 1>(p, a, tA, tL, wm, st);
    return launch_cfg<true, 2, 128, 1>(p, a, tA, tL, wm, st);
  }
  if (p.um == 2) return launch_cfg<true, 2, 128, 0>(p, a, tA, tL, wm, st);
  return launch_cfg<true, 1, 128, 0>(p, a, tA, tL, wm, st);
}

// The same for a bf16 weight: pairs always share the tile through the pair MMA.
cudaError_t dispatch_gemm_wb(const GemmPlan& p, const GemmArgs& a, const CUtensorMap& tA,
                             const CUtensorMap& tL, const WMaps& wm, cudaStream_t st) {
  if (!p.bwd) {
    if (p.pair) {
      if (p.bn == 256) return launch_cfg<false, 2, 256, 2, true>(p, a, tA, tL, wm, st);
      return launch_cfg<false, 2, 128, 2, true>(p, a, tA, tL, wm, st);
    }
    if (p.um == 2 && p.bn == 256) return launch_cfg<false, 2, 256, 0, true>(p, a, tA, tL, wm, st);
    if (p.um == 2) return launch_cfg<false, 2, 128, 0, true>(p, a, tA, tL, wm, st);
    return launch_cfg<false, 1, 128, 0, true>(p, a, tA, tL, wm, st);
  }
  if (p.pair) {
    if (p.bn == 256) return launch_cfg<true, 2, 256, 2, true>(p, a, tA, tL, wm, st);
    return launch_cfg<true, 2, 128, 2, true>(p, a, tA, tL, wm, st);
  }
  if (p.um == 2) return launch_cfg<true, 2, 128, 0, true>(p, a, tA, tL, wm, st);
  return launch_cfg<true, 1, 128, 0, true>(p, a, tA, tL, wm, st);
}

// Tensor maps of bf16 weights for a plan: rows of W [N, K] in boxes of
// 64 x (this CTA's share of the tile's rows) for the forward, 64 x 64 for the
// backward (which reads BW / 64 column groups per contraction step).
bool make_wmap(CUtensorMap* m, const GemmPlan& p, const uint16_t* w, int64_t N, int64_t K) {
  const uint32_t bw = (uint32_t)(p.pair ? p.bn / 2 : p.bn);
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w, (uint64_t)K, (uint64_t)N,
                  (uint64_t)K * 2, 64, p.bwd ? 64u : bw, CU_TENSOR_MAP_SWIZZLE_128B);
}
}  // namespace

cudaError_t run_nf4_gemm(const GemmPlan& p, const NF4View& W, const uint16_t* act, int64_t M,
                         const uint16_t* lora_act, const float* lora_F, float lora_scale,
                         const uint32_t* mask, void* out, int out_f32, int out_accum,
                         float* partial, cudaStream_t st) {
  if (!encode_fn()) return cudaErrorNotSupported;
  const int64_t N = W.N, K = W.K;
  const int64_t Nout = p.bwd ? K : N;
  const int64_t Kc = p.bwd ? N : K;
  const int BM = 128 * p.um;
  CUtensorMap tA, tL;
  bool ok = make_map(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, act, (uint64_t)Kc, (uint64_t)M,
                     (uint64_t)Kc * 2, 64, (uint32_t)BM, CU_TENSOR_MAP_SWIZZLE_128B);
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
  a.codes = W.codes;
  a.absmax = W.absmax;
  a.wN = N;
  a.wK = K;
  a.epad = p.epad;
  a.flags = nullptr;
  if (grid_units(p, has_lora) > 1) {
    cudaError_t e = ring_slots((uint32_t)grid_ctas(p, has_lora), &a.flags);
    if (e != cudaSuccess) return e;
  }

  if (partial == nullptr && grid_units(p, has_lora) > 1) return cudaErrorInvalidValue;
  WMaps wm;
  memset(&wm, 0, sizeof(wm));
  if (W.wbf16) {
    if (!make_wmap(&wm.m[0], p, W.wbf16, N, K)) return cudaErrorInvalidValue;
    return dispatch_gemm_wb(p, a, tA, tL, wm, st);
  }
  return dispatch_gemm(p, a, tA, tL, wm, st);
}

cudaError_t run_nf4_gemm_group(const GemmPlan& p, int ng, const NF4View* W, const uint16_t* act,
                               int64_t M, const uint16_t* lora_act, const float* const* lora_F,
                               float lora_scale, uint16_t* const* out, float* partial,
                               cudaStream_t st) {
  if (!encode_fn()) return cudaErrorNotSupported;
  if (ng < 1 || ng > kMaxGroups || p.bwd || lora_act == nullptr) return cudaErrorInvalidValue;
  const int64_t K = W[0].K;
  WMaps wm;
  memset(&wm, 0, sizeof(wm));
  const bool wb = W[0].wbf16 != nullptr;
  for (int g = 0; g < ng; ++g) {
    if ((W[g].wbf16 != nullptr) != wb) return cudaErrorInvalidValue;
    if (wb && !make_wmap(&wm.m[g], p, W[g].wbf16, W[g].N, K)) return cudaErrorInvalidValue;
  }
  GemmArgs a{};
  a.ngroups = ng;
  a.gcol[0] = 0;
  for (int g = 0; g < ng; ++g) {
    if (W[g].K != K || W[g].N % p.bn != 0) return cudaErrorInvalidValue;
    a.gcol[g + 1] = a.gcol[g] + W[g].N;
    a.gcodes[g] = W[g].codes;
    a.gabsmax[g] = W[g].absmax;
    a.glora_F[g] = lora_F[g];
    a.gout[g] = out[g];
  }
  const int64_t Nsum = a.gcol[ng];
  // group 0 also fills the single-linear fields (ng = 1 reads those)
  a.codes = W[0].codes;
  a.absmax = W[0].absmax;
  a.lora_F = lora_F[0];
  a.out = out[0];
  a.wN = W[0].N;
  if (p.ntiles != (int)(Nsum / p.bn) || p.nk != (int)(K / 64)) return cudaErrorInvalidValue;
  const int BM = 128 * p.um;
  CUtensorMap tA, tL;
  bool ok = make_map(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, act, (uint64_t)K, (uint64_t)M,
                     (uint64_t)K * 2, 64, (uint32_t)BM, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&tL, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, lora_act, 64, (uint64_t)(ng * M), 128,
                      64, (uint32_t)BM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  a.M = M;
  a.Nout = Nsum;
  a.nk_total = p.nk;
  a.mtiles = p.mtiles;
  a.ntiles = p.ntiles;
  a.has_lora = 1;
  a.lora_scale = lora_scale;
  a.partial = partial;
  a.wK = K;
  a.epad = p.epad;
  a.flags = nullptr;
  if (grid_units(p, true) > 1) {
    cudaError_t e = ring_slots((uint32_t)grid_ctas(p, true), &a.flags);
    if (e != cudaSuccess) return e;
    if (partial == nullptr) return cudaErrorInvalidValue;
  }
  if (wb) return dispatch_gemm_wb(p, a, tA, tL, wm, st);
  return dispatch_gemm(p, a, tA, tL, wm, st);
}

// ------------------------------------------------------------------------ bounded-wait self-check
// One thread waits, through the finisher's bounded wait but with the given
// limit, for a ring word that nothing sets; it gives up, records the peer
// timeout bit and returns.
__global__ void k_wait_selfcheck(const uint32_t* word, uint64_t limit_ns) {
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0 && blockIdx.x == 0)
    (void)wait_flag_bounded(word, 1u, limit_ns, DERR_TIMEOUT_PEER);
}

cudaError_t run_wait_selfcheck(uint32_t limit_us, cudaStream_t st) {
  uint32_t* word = nullptr;
  cudaError_t e = ring_slots(1, &word);
  if (e != cudaSuccess) return e;
  note_launch();
  (void)launch_pdl(k_wait_selfcheck, dim3(1), dim3(32), 0, st, (const uint32_t*)word,
                   (uint64_t)limit_us * 1000ull);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------ skinny products (host)
// k-chunks per 128-row block: the whole launch (ng groups) fits one wave of
// one CTA per SM, so no CTA waits for another's slot.
int skinny_tc_chunks(int64_t M, int64_t K, int ng = 1) {
  const int64_t atoms = (M + 127) / 128;
  const int64_t steps = K / 64;
  int64_t ch = device_sm_count() / ((atoms > 0 ? atoms : 1) * (ng > 0 ? ng : 1));
  if (ch > steps) ch = steps;
  if (ch < 1) ch = 1;
  const int64_t spc = (steps + ch - 1) / ch;
  return (int)((steps + spc - 1) / spc);
}

// Chunks (CTAs per row block) of the unmasked products G = dY B at most.
constexpr int kSkChunksG = 10;

size_t skinny_partial_bytes(int64_t M, int64_t K) {
  return (size_t)skinny_tc_chunks(M, K) * (size_t)M * 16 * sizeof(float);
}

// Cross-CTA words of a launch (stream-K completion flags of the dequant
// GEMM, arrival counters of the skinny products' row blocks), taken
// round-robin from a library-owned array.  They start at zero and each
// launch leaves the words it used at zero again (a finisher clears the flags
// it consumed; the last CTA of a row block clears its counter), so no launch
// has to clear them first.  Launches in flight at the same time on different
// streams get different words unless more than kRingWords words are handed
// out in between.  ws_device_error clears the whole array after a kernel
// gave up.
constexpr uint32_t kRingWords = 1u << 20;
static __device__ uint32_t g_ring_words[kRingWords];
namespace {
std::mutex g_ring_mu;
uint32_t* g_ring_ptr[64] = {};
uint32_t g_ring_next = 0;
}  // namespace

static cudaError_t ring_base(uint32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!g_ring_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_ring_words);
    if (e != cudaSuccess) return e;
    g_ring_ptr[dev] = static_cast<uint32_t*>(p);
  }
  *out = g_ring_ptr[dev];
  return cudaSuccess;
}

cudaError_t ring_slots(uint32_t n, uint32_t** out) {
  if (n == 0 || n > 4096) return cudaErrorInvalidValue;
  std::lock_guard<std::mutex> lock(g_ring_mu);
  uint32_t* base = nullptr;
  cudaError_t e = ring_base(&base);
  if (e != cudaSuccess) return e;
  if (g_ring_next + n > kRingWords) g_ring_next = 0;
  *out = base + g_ring_next;
  g_ring_next += n;
  return cudaSuccess;
}

cudaError_t ring_clear() {
  std::lock_guard<std::mutex> lock(g_ring_mu);
  uint32_t* base = nullptr;
  cudaError_t e = ring_base(&base);
  if (e != cudaSuccess) return e;
  return cudaMemset(base, 0, (size_t)kRingWords * sizeof(uint32_t));
}

namespace {
cudaError_t skinny_launch(const uint16_t* const* X, int ng, const float* const* F, bool f_kj, int64_t M,
                          int64_t K, const DropKey* keys, uint8_t* const* mask_bytes,
                          float* const* partial, float* const* out, uint16_t* const* ext,
                          cudaStream_t st) {
  if (!encode_fn()) return cudaErrorNotSupported;
  if (K % 64 != 0 || M < 1 || ng < 1 || ng > kMaxGroups) return cudaErrorInvalidValue;
  const int64_t atoms = (M + 127) / 128;
  int chunks = skinny_tc_chunks(M, K, ng);
  const int64_t steps = K / 64;
  if (f_kj && chunks > kSkChunksG) {
    // G = dY B draws no dropout bits, so its steps are short: fewer, longer
    // chunks leave the last CTA of a row block fewer partial sums to add
    const int64_t sp = (steps + kSkChunksG - 1) / kSkChunksG;
    chunks = (int)((steps + sp - 1) / sp);
  }
  const int spc = (int)((steps + chunks - 1) / chunks);
  uint32_t* counters = nullptr;
  cudaError_t e = ring_slots((uint32_t)(atoms * ng), &counters);
  if (e != cudaSuccess) return e;
  SkArgs sa;
  memset(&sa, 0, sizeof(sa));
  for (int g = 0; g < ng; ++g) {
    if (g > 0 && X[g] == X[g - 1]) sa.tmX[g] = sa.tmX[g - 1];
    else if (!make_map(&sa.tmX[g], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X[g], (uint64_t)K, (uint64_t)M,
                       (uint64_t)K * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    // the factor slices are fetched with 16-byte copies
    if ((reinterpret_cast<uintptr_t>(F[g]) & 15u) != 0u) return cudaErrorInvalidValue;
    if (f_kj) sa.tmF[g] = sa.tmX[g];
    else if (!make_map(&sa.tmF[g], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, F[g], (uint64_t)K, 16,
                       (uint64_t)K * 4, 32, 16, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    sa.F[g] = F[g];
    if (keys) sa.key[g] = keys[g];
    sa.mask_bytes[g] = mask_bytes ? mask_bytes[g] : nullptr;
    sa.partial[g] = partial[g];
    sa.counters[g] = counters + g * atoms;
    sa.out[g] = out[g];
    sa.ext[g] = ext[g];
  }
  sa.M = M;
  sa.K = K;
  sa.steps_per_chunk = spc;
  static cudaError_t a0 = cudaFuncSetAttribute(
      k_skinny_tc<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSkSmem);
  static cudaError_t a1 = cudaFuncSetAttribute(
      k_skinny_tc<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSkSmem);
  static cudaError_t a2 = cudaFuncSetAttribute(
      k_skinny_tc<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSkSmem);
  if (a0 != cudaSuccess) return a0;
  if (a1 != cudaSuccess) return a1;
  if (a2 != cudaSuccess) return a2;
  const dim3 grid((unsigned)atoms, (unsigned)chunks, (unsigned)ng);
  note_launch();
  if (keys && !f_kj)
    (void)launch_pdl(k_skinny_tc<true, false>, grid, dim3(kSkThreads), kSkSmem, st, sa);
  else if (f_kj)
    (void)launch_pdl(k_skinny_tc<false, true>, grid, dim3(kSkThreads), kSkSmem, st, sa);
  else
    (void)launch_pdl(k_skinny_tc<false, false>, grid, dim3(kSkThreads), kSkSmem, st, sa);
  return cudaGetLastError();
}
}  // namespace

cudaError_t run_skinny_tc(const uint16_t* X, const float* F, bool f_kj, int64_t M, int64_t K,
                          const DropKey* key, uint8_t* mask_bytes, float* partial, float* out,
                          uint16_t* ext, cudaStream_t st) {
  return skinny_launch(&X, 1, &F, f_kj, M, K, key, &mask_bytes, &partial, &out, &ext, st);
}

cudaError_t run_skinny_tc_group(const uint16_t* X, int ng, const float* const* F, int64_t M,
                                int64_t K, const DropKey* keys, uint8_t* const* mask_bytes,
                                float* const* partial, float* const* out, uint16_t* const* ext,
                                cudaStream_t st) {
  const uint16_t* Xs[kMaxGroups];
  for (int g = 0; g < ng && g < kMaxGroups; ++g) Xs[g] = X;
  return skinny_launch(Xs, ng, F, false, M, K, keys, mask_bytes, partial, out, ext, st);
}

cudaError_t run_skinny_G_group(int ng, const uint16_t* const* dY, const float* const* B, int64_t M,
                               int64_t N, float* const* partial, float* const* G,
                               uint16_t* const* Gext, cudaStream_t st) {
  return skinny_launch(dY, ng, B, true, M, N, nullptr, nullptr, partial, G, Gext, st);
}

// ------------------------------------------------------------------------ weight gradients (host)
size_t wgrad_tc_bytes(int64_t M, int64_t C) {
  (void)M;
  (void)C;
  return 0;
}

cudaError_t run_wgrad_tc_group(int ng, const float* const* P, const uint16_t* const* Q,
                               const uint32_t* const* mask, int64_t M, int64_t C, float s,
                               float* const* out, int transpose_out, int accumulate,
                               cudaStream_t st) {
  if (!encode_fn()) return cudaErrorNotSupported;
  if (ng < 1 || ng > kMaxGroups) return cudaErrorInvalidValue;
  WgArgs wa;
  memset(&wa, 0, sizeof(wa));
  bool masked = false;
  for (int g = 0; g < ng; ++g) {
    // P rows are fetched with 16-byte bulk copies
    if ((reinterpret_cast<uintptr_t>(P[g]) & 15u) != 0u) return cudaErrorInvalidValue;
    if (g > 0 && Q[g] == Q[g - 1]) wa.tmQ[g] = wa.tmQ[g - 1];
    else if (!make_map(&wa.tmQ[g], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Q[g], (uint64_t)C, (uint64_t)M,
                       (uint64_t)C * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    wa.P[g] = P[g];
    wa.mask[g] = mask ? mask[g] : nullptr;
    wa.out[g] = out[g];
    masked = masked || wa.mask[g] != nullptr;
  }
  // one launch masks every group or none
  for (int g = 0; g < ng; ++g)
    if ((wa.mask[g] != nullptr) != masked) return cudaErrorInvalidValue;
  wa.M = M;
  wa.C = C;
  wa.s = s;
  wa.transpose_out = transpose_out;
  wa.accumulate = accumulate;
  static cudaError_t attr0 = cudaFuncSetAttribute(
      k_wgrad_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWgSmem);
  static cudaError_t attr1 = cudaFuncSetAttribute(
      k_wgrad_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWgSmem);
  if (attr0 != cudaSuccess) return attr0;
  if (attr1 != cudaSuccess) return attr1;
  const dim3 grid((unsigned)((C + kWgBN - 1) / kWgBN), (unsigned)ng);
  note_launch();
  if (masked)
    (void)launch_pdl(k_wgrad_tc<true>, grid, dim3(kWgThreads), kWgSmem, st, wa);
  else
    (void)launch_pdl(k_wgrad_tc<false>, grid, dim3(kWgThreads), kWgSmem, st, wa);
  return cudaGetLastError();
}

cudaError_t run_wgrad_tc(const float* P, const uint16_t* Q, const uint32_t* mask, int64_t M,
                         int64_t C, float s, float* out, int transpose_out, int accumulate,
                         void* ws, cudaStream_t st) {
  (void)ws;
  return run_wgrad_tc_group(1, &P, &Q, &mask, M, C, s, &out, transpose_out, accumulate, st);
}

}  // namespace ws
