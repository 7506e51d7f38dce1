// lora_small.cu -- the HBM-bound pieces of one NF4-LoRA linear and the
// orchestration of its forward and backward:
//   a0  NF4 quantisation of a bf16 weight
//   a1  dropout bits (Philox4x32-10) + LoRA down projection U = (m.x) A^T
//   a3  G = dY B and dB = s dY^T U
//   a5  dA = s G^T (m.x)
// Every reduction runs in a fixed order (per-lane sequential sums, a fixed
// butterfly across lanes, fixed-order sums across row chunks): no atomics.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace ws {

namespace {

__constant__ float c_levels_q[16] = {-1.0f,    -0.6962f, -0.5251f, -0.3949f, -0.2844f, -0.1848f,
                                     -0.0911f, 0.0f,     0.0796f,  0.1609f,  0.2461f,  0.3379f,
                                     0.4407f,  0.5626f,  0.7230f,  1.0f};

// ------------------------------------------------------------------------ a0: quantise
// One warp per 64-weight block; lane i handles weights 2i and 2i+1 and
// writes code byte i.  The block maximum is a max-reduction (exact in any
// order); v = w / absmax is an IEEE division; the code counts the midpoints
// below v.
__global__ void k_quantize_nf4(const uint16_t* __restrict__ W, int64_t N, int64_t K,
                               uint8_t* __restrict__ codes, float* __restrict__ absmax) {
  const int64_t nkb = K / 64;
  const int64_t blk = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x / 32);
  if (blk >= N * nkb) return;
  const int lane = threadIdx.x & 31;
  const int64_t n = blk / nkb, kb = blk % nkb;
  const uint32_t pair = *reinterpret_cast<const uint32_t*>(W + n * K + kb * 64 + 2 * lane);
  const float w0 = __uint_as_float(pair << 16);
  const float w1 = __uint_as_float(pair & 0xffff0000u);
  float amax = fmaxf(fabsf(w0), fabsf(w1));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  uint32_t c0 = 7, c1 = 7;
  if (amax != 0.0f) {
    const float v0 = __fdiv_rn(w0, amax);
    const float v1 = __fdiv_rn(w1, amax);
    c0 = 0;
    c1 = 0;
#pragma unroll
    for (int i = 0; i < 15; ++i) {
      const float mid = __fmul_rn(__fadd_rn(c_levels_q[i], c_levels_q[i + 1]), 0.5f);
      c0 += v0 > mid ? 1u : 0u;
      c1 += v1 > mid ? 1u : 0u;
    }
  }
  codes[n * (K / 2) + kb * 32 + lane] = (uint8_t)((c0 << 4) | c1);
  if (lane == 0) absmax[kb * N + n] = amax;
}

// ------------------------------------------------------------------------ a1: down + mask
// One warp per row, 8 rows per block; the block stages a 16 x 256 slice of
// A in shared memory; each lane covers 8 consecutive k per slice.
constexpr int kDownRows = 8;
constexpr int kSlice = 256;

WS_DEVINL void write_split_row(float (&acc)[16], int64_t m, float* __restrict__ U,
                               uint16_t* __restrict__ Uext) {
  // U fp32 and [hi | lo | hi | 0] bf16 split of the same row
  float4* u4 = reinterpret_cast<float4*>(U + m * 16);
  uint32_t hi[8], lo[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float h0 = bf16_lo(pack_bf16x2(acc[2 * i], 0.0f));
    const float h1 = bf16_lo(pack_bf16x2(acc[2 * i + 1], 0.0f));
    hi[i] = pack_bf16x2(h0, h1);
    lo[i] = pack_bf16x2(acc[2 * i] - h0, acc[2 * i + 1] - h1);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) u4[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
  uint4* e4 = reinterpret_cast<uint4*>(Uext + m * 64);
  e4[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  e4[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
  e4[2] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  e4[3] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
  e4[4] = e4[0];
  e4[5] = e4[1];
  e4[6] = make_uint4(0u, 0u, 0u, 0u);
  e4[7] = make_uint4(0u, 0u, 0u, 0u);
}

__global__ void __launch_bounds__(256) k_lora_down(const uint16_t* __restrict__ x,
                                                   const float* __restrict__ A, int64_t M,
                                                   int64_t K, DropKey key, float* __restrict__ U,
                                                   uint16_t* __restrict__ Uext,
                                                   uint8_t* __restrict__ mask_bytes) {
  __shared__ __align__(16) float sA[16][kSlice];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * kDownRows + warp;
  float acc[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
  for (int64_t k0 = 0; k0 < K; k0 += kSlice) {
    __syncthreads();
    for (int i = threadIdx.x; i < 16 * kSlice / 4; i += blockDim.x) {
      const int j = i / (kSlice / 4), c4 = (i % (kSlice / 4)) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (k0 + c4 < K) v = *reinterpret_cast<const float4*>(A + (int64_t)j * K + k0 + c4);
      *reinterpret_cast<float4*>(&sA[j][c4]) = v;
    }
    __syncthreads();
    const int64_t k = k0 + 8 * lane;
    if (m < M && k < K) {
      const uint64_t e0 = (uint64_t)(m * K + k);
      const uint32_t bits = keep4(key, e0) | (keep4(key, e0 + 4) << 4);
      if (mask_bytes) mask_bytes[e0 >> 3] = (uint8_t)bits;
      const uint4 xv = *reinterpret_cast<const uint4*>(x + m * K + k);
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
      float xm[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xm[2 * i] = ((bits >> (2 * i)) & 1u) ? bf16_lo(xw[i]) : 0.0f;
        xm[2 * i + 1] = ((bits >> (2 * i + 1)) & 1u) ? bf16_hi(xw[i]) : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float4 a0 = *reinterpret_cast<const float4*>(&sA[j][8 * lane]);
        const float4 a1 = *reinterpret_cast<const float4*>(&sA[j][8 * lane + 4]);
        float s = acc[j];
        s = fmaf(xm[0], a0.x, s);
        s = fmaf(xm[1], a0.y, s);
        s = fmaf(xm[2], a0.z, s);
        s = fmaf(xm[3], a0.w, s);
        s = fmaf(xm[4], a1.x, s);
        s = fmaf(xm[5], a1.y, s);
        s = fmaf(xm[6], a1.z, s);
        s = fmaf(xm[7], a1.w, s);
        acc[j] = s;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 16; ++j)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], o);
  if (m < M && lane == 0) write_split_row(acc, m, U, Uext);
}

// ------------------------------------------------------------------------ a3: G = dY B
__global__ void __launch_bounds__(256) k_lora_G(const uint16_t* __restrict__ dY,
                                                const float* __restrict__ B, int64_t M, int64_t N,
                                                float* __restrict__ G, uint16_t* __restrict__ Gext) {
  __shared__ __align__(16) float sBt[16][kSlice];  // B slice transposed: [j][n]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * kDownRows + warp;
  float acc[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
  for (int64_t n0 = 0; n0 < N; n0 += kSlice) {
    __syncthreads();
    for (int i = threadIdx.x; i < kSlice; i += blockDim.x) {
      const int64_t n = n0 + i;
#pragma unroll
      for (int j4 = 0; j4 < 4; ++j4) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (n < N) v = *reinterpret_cast<const float4*>(B + n * 16 + 4 * j4);
        sBt[4 * j4 + 0][i] = v.x;
        sBt[4 * j4 + 1][i] = v.y;
        sBt[4 * j4 + 2][i] = v.z;
        sBt[4 * j4 + 3][i] = v.w;
      }
    }
    __syncthreads();
    const int64_t n = n0 + 8 * lane;
    if (m < M && n < N) {
      const uint4 dv = *reinterpret_cast<const uint4*>(dY + m * N + n);
      const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
      float d[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        d[2 * i] = bf16_lo(dw[i]);
        d[2 * i + 1] = bf16_hi(dw[i]);
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float4 b0 = *reinterpret_cast<const float4*>(&sBt[j][8 * lane]);
        const float4 b1 = *reinterpret_cast<const float4*>(&sBt[j][8 * lane + 4]);
        float s = acc[j];
        s = fmaf(d[0], b0.x, s);
        s = fmaf(d[1], b0.y, s);
        s = fmaf(d[2], b0.z, s);
        s = fmaf(d[3], b0.w, s);
        s = fmaf(d[4], b1.x, s);
        s = fmaf(d[5], b1.y, s);
        s = fmaf(d[6], b1.z, s);
        s = fmaf(d[7], b1.w, s);
        acc[j] = s;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 16; ++j)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], o);
  if (m < M && lane == 0) write_split_row(acc, m, G, Gext);
}

// ------------------------------------------------------------------------ a3/a5: s P^T Q
// Thread = one column c; block = 256 columns x one chunk of rows; rows are
// summed sequentially; a second kernel sums the chunks in order.
constexpr int kWgradCols = 256;

__global__ void __launch_bounds__(256) k_wgrad_partial(const float* __restrict__ P,
                                                       const uint16_t* __restrict__ Q,
                                                       const uint32_t* __restrict__ mask,
                                                       int64_t M, int64_t C, int rows_per_chunk,
                                                       float* __restrict__ partial) {
  __shared__ __align__(16) float sP[64][16];
  const int64_t c = (int64_t)blockIdx.x * kWgradCols + threadIdx.x;
  const int64_t r0 = (int64_t)blockIdx.y * rows_per_chunk;
  const int64_t r1 = min(M, r0 + rows_per_chunk);
  float acc[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
  for (int64_t mb = r0; mb < r1; mb += 64) {
    const int rows = (int)((r1 - mb) < 64 ? (r1 - mb) : 64);
    __syncthreads();
    for (int i = threadIdx.x; i < rows * 4; i += blockDim.x)
      *reinterpret_cast<float4*>(&sP[i / 4][(i % 4) * 4]) =
          *reinterpret_cast<const float4*>(P + (mb + i / 4) * 16 + (i % 4) * 4);
    __syncthreads();
    if (c < C) {
      for (int rr = 0; rr < rows; ++rr) {
        const int64_t m = mb + rr;
        float q = bf16_bits_to_f32(Q[m * C + c]);
        if (mask && !((mask[(m * C + c) >> 5] >> (c & 31)) & 1u)) q = 0.0f;
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
          const float4 p = *reinterpret_cast<const float4*>(&sP[rr][4 * j4]);
          acc[4 * j4 + 0] = fmaf(p.x, q, acc[4 * j4 + 0]);
          acc[4 * j4 + 1] = fmaf(p.y, q, acc[4 * j4 + 1]);
          acc[4 * j4 + 2] = fmaf(p.z, q, acc[4 * j4 + 2]);
          acc[4 * j4 + 3] = fmaf(p.w, q, acc[4 * j4 + 3]);
        }
      }
    }
  }
  if (c < C) {
    float4* dst = reinterpret_cast<float4*>(partial + ((int64_t)blockIdx.y * C + c) * 16);
#pragma unroll
    for (int j4 = 0; j4 < 4; ++j4)
      dst[j4] = make_float4(acc[4 * j4], acc[4 * j4 + 1], acc[4 * j4 + 2], acc[4 * j4 + 3]);
  }
}

__global__ void k_wgrad_reduce(const float* __restrict__ partial, int chunks, int64_t C, float s,
                               float* __restrict__ out, int transpose_out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // (c, j) flat, j fastest
  if (i >= C * 16) return;
  float acc = partial[i];
  for (int ch = 1; ch < chunks; ++ch) acc += partial[(int64_t)ch * C * 16 + i];
  acc *= s;
  const int64_t c = i / 16, j = i % 16;
  if (transpose_out) out[j * C + c] = acc;
  else out[i] = acc;
}

int wgrad_chunks(int64_t M, int64_t C) {
  const int64_t cblocks = (C + kWgradCols - 1) / kWgradCols;
  int64_t want = (2 * device_sm_count() + cblocks - 1) / cblocks;
  const int64_t maxc = (M + 15) / 16;
  if (want > maxc) want = maxc;
  if (want < 1) want = 1;
  return (int)want;
}

// ------------------------------------------------------------------------ mask regeneration
__global__ void k_mask_gen(int64_t words, DropKey key, uint32_t* __restrict__ mask) {
  const int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (w >= words) return;
  const uint64_t e0 = (uint64_t)w * 32;
  uint32_t bits = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) bits |= keep4(key, e0 + 4 * i) << (4 * i);
  mask[w] = bits;
}

DropKey to_dev(const DropKeyHost& h) {
  DropKey k;
  k.k0 = h.k0;
  k.k1 = h.k1;
  k.c1 = h.c1;
  k.c2 = h.c2;
  k.c3 = h.c3;
  k.thresh = h.thresh;
  k.drop_all = h.drop_all;
  return k;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

DropKeyHost make_drop_key(const ws_dropout_key& k) {
  DropKeyHost h{};
  h.k0 = (uint32_t)k.seed;
  h.k1 = (uint32_t)(k.seed >> 32);
  h.c1 = k.linear | (k.microbatch << 8);
  h.c2 = k.layer;
  h.c3 = k.step;
  const double t = ceil(k.p * 4294967296.0);
  if (t >= 4294967296.0) {
    h.drop_all = 1;
    h.thresh = 0xffffffffu;
  } else {
    h.drop_all = 0;
    h.thresh = t <= 0.0 ? 0u : (uint32_t)t;
  }
  return h;
}

cudaError_t run_quantize_nf4(const uint16_t* W, int64_t N, int64_t K, uint8_t* codes,
                             float* absmax, cudaStream_t st) {
  const int64_t blocks = N * (K / 64);
  const int per = 8;  // warps per CTA
  note_launch();
  k_quantize_nf4<<<(unsigned)((blocks + per - 1) / per), 32 * per, 0, st>>>(W, N, K, codes, absmax);
  return cudaGetLastError();
}

cudaError_t run_lora_down(const uint16_t* x, const float* A, int64_t M, int64_t K,
                          const DropKeyHost& key, float* U, uint16_t* Uext, uint32_t* mask_out,
                          cudaStream_t st) {
  note_launch();
  k_lora_down<<<(unsigned)((M + kDownRows - 1) / kDownRows), 256, 0, st>>>(
      x, A, M, K, to_dev(key), U, Uext, reinterpret_cast<uint8_t*>(mask_out));
  return cudaGetLastError();
}

cudaError_t run_lora_G(const uint16_t* dY, const float* B, int64_t M, int64_t N, float* G,
                       uint16_t* Gext, cudaStream_t st) {
  note_launch();
  k_lora_G<<<(unsigned)((M + kDownRows - 1) / kDownRows), 256, 0, st>>>(dY, B, M, N, G, Gext);
  return cudaGetLastError();
}

size_t wgrad_partial_bytes(int64_t M, int64_t C) {
  return (size_t)wgrad_chunks(M, C) * (size_t)C * 16 * sizeof(float);
}

cudaError_t run_lora_wgrad(const float* P, const uint16_t* Q, const uint32_t* mask, int64_t M,
                           int64_t C, float s, float* out, int transpose_out, float* partial,
                           cudaStream_t st) {
  const int chunks = wgrad_chunks(M, C);
  const int rpc = (int)((M + chunks - 1) / chunks);
  dim3 grid((unsigned)((C + kWgradCols - 1) / kWgradCols), (unsigned)chunks);
  note_launch();
  k_wgrad_partial<<<grid, kWgradCols, 0, st>>>(P, Q, mask, M, C, rpc, partial);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t n = C * 16;
  note_launch();
  k_wgrad_reduce<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(partial, chunks, C, s, out,
                                                              transpose_out);
  return cudaGetLastError();
}

cudaError_t run_mask_gen(int64_t M, int64_t K, const DropKeyHost& key, uint32_t* mask,
                         cudaStream_t st) {
  const int64_t words = M * K / 32;
  note_launch();
  k_mask_gen<<<(unsigned)((words + 255) / 256), 256, 0, st>>>(words, to_dev(key), mask);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------ one linear
// Workspace layout (each piece 256-aligned):
//   ext     [M, 64] bf16       U or G split factor
//   G       [M, 16] fp32       backward only
//   mask    [M, K/32] u32      backward, when the caller kept no mask
//   wgrad   chunks x C x 16 fp32, C = max(N, K)
//   split   splits x M x Nout fp32, max over forward and backward plans
namespace {
struct LinWs {
  size_t ext, G, mask, wgrad, split, total;
};
LinWs lin_ws_layout(int64_t M, int64_t N, int64_t K) {
  LinWs w{};
  size_t off = 0;
  w.ext = off;
  off += align256((size_t)M * 64 * 2);
  w.G = off;
  off += align256((size_t)M * 16 * 4);
  w.mask = off;
  off += align256((size_t)M * (size_t)(K / 32) * 4);
  w.wgrad = off;
  const size_t wg = wgrad_partial_bytes(M, N) > wgrad_partial_bytes(M, K) ? wgrad_partial_bytes(M, N)
                                                                          : wgrad_partial_bytes(M, K);
  off += align256(wg);
  w.split = off;
  const GemmPlan pf = plan_gemm(false, M, N, K);
  const GemmPlan pb = plan_gemm(true, M, K, N);
  const size_t sf = gemm_partial_bytes(pf, M, N), sb = gemm_partial_bytes(pb, M, K);
  off += align256(sf > sb ? sf : sb);
  w.total = off;
  return w;
}
}  // namespace

size_t linear_workspace_bytes(int64_t M, int64_t N, int64_t K) { return lin_ws_layout(M, N, K).total; }

cudaError_t linear_fwd(const NF4View& W, const uint16_t* x, const float* A, const float* B,
                       int64_t M, float scale, const DropKeyHost& key, uint16_t* y, float* U,
                       uint32_t* mask, void* ws, cudaStream_t st) {
  const LinWs L = lin_ws_layout(M, W.N, W.K);
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint16_t* Uext = reinterpret_cast<uint16_t*>(w + L.ext);
  cudaError_t e = run_lora_down(x, A, M, W.K, key, U, Uext, mask, st);
  if (e != cudaSuccess) return e;
  const GemmPlan p = plan_gemm(false, M, W.N, W.K);
  return run_nf4_gemm(p, W, x, M, Uext, B, scale, nullptr, y, 0, 0,
                      reinterpret_cast<float*>(w + L.split), st);
}

cudaError_t linear_bwd(const NF4View& W, const uint16_t* x, const float* A, const float* B,
                       int64_t M, float scale, const DropKeyHost& key, const float* U,
                       const uint32_t* mask, const uint16_t* dY, void* dX, int dX_f32,
                       int dX_accum, float* dA, float* dB, void* ws, cudaStream_t st) {
  const LinWs L = lin_ws_layout(M, W.N, W.K);
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint16_t* Gext = reinterpret_cast<uint16_t*>(w + L.ext);
  float* G = reinterpret_cast<float*>(w + L.G);
  float* wg = reinterpret_cast<float*>(w + L.wgrad);
  cudaError_t e;
  if (mask == nullptr) {
    uint32_t* m = reinterpret_cast<uint32_t*>(w + L.mask);
    e = run_mask_gen(M, W.K, key, m, st);
    if (e != cudaSuccess) return e;
    mask = m;
  }
  e = run_lora_G(dY, B, M, W.N, G, Gext, st);
  if (e != cudaSuccess) return e;
  if (dB) {
    e = run_lora_wgrad(U, dY, nullptr, M, W.N, scale, dB, 0, wg, st);
    if (e != cudaSuccess) return e;
  }
  if (dA) {
    e = run_lora_wgrad(G, x, mask, M, W.K, scale, dA, 1, wg, st);
    if (e != cudaSuccess) return e;
  }
  if (dX) {
    const GemmPlan p = plan_gemm(true, M, W.K, W.N);
    e = run_nf4_gemm(p, W, dY, M, Gext, A, scale, mask, dX, dX_f32, dX_accum,
                     reinterpret_cast<float*>(w + L.split), st);
  }
  return e;
}

}  // namespace ws
