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

// ------------------------------------------------------------------------ a1/a3: skinny products
// partial[c][m][j] = sum_{k in chunk c} x~[m,k] * F[j,k] for the 16 LoRA
// columns j, where x~ is x (optionally under the dropout mask, whose bits the
// kernel also draws and stores) and F[j,k] is A[j,k] (down projection) or
// B[k,j] (G = dY B).  Block = 32 rows x 256 columns of one chunk; warp w
// owns rows 4w..4w+3, lane l owns columns 8l..8l+7.  The 16-wide slice of F
// is staged in shared memory once per block and reused by all 32 rows.  The
// 32 lanes' partial sums are combined by a fixed butterfly reduce-scatter
// (after it lane l holds entries 2l and 2l+1 of the warp's 4 x 16 block),
// and a second kernel sums the chunks in index order: the result depends
// only on the shapes, never on scheduling.
constexpr int kSkRows = 32;
constexpr int kSkCols = 256;

template <bool MASKED, bool F_ROWMAJOR_KJ>
__global__ void __launch_bounds__(256, 2) k_skinny_partial(const uint16_t* __restrict__ x,
                                                           const float* __restrict__ F, int64_t M,
                                                           int64_t K, int slices, DropKey key,
                                                           uint8_t* __restrict__ mask_bytes,
                                                           float* __restrict__ partial) {
  __shared__ __align__(16) float sF[16][kSkCols];
  if (MASKED) resolve_step(key);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m0 = (int64_t)blockIdx.x * kSkRows + warp * 4;
  float acc[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
  for (int sl = 0; sl < slices; ++sl) {
    const int64_t k0 = ((int64_t)blockIdx.y * slices + sl) * kSkCols;
    if (k0 >= K) break;  // block-uniform
    __syncthreads();
    // stage F[:, k0:k0+256]
    if (F_ROWMAJOR_KJ) {
      // F given as [K][16] (B): thread i loads row k0+i and scatters it
      const int i = threadIdx.x;
      const int64_t k = k0 + i;
#pragma unroll
      for (int j4 = 0; j4 < 4; ++j4) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < K) v = *reinterpret_cast<const float4*>(F + k * 16 + 4 * j4);
        sF[4 * j4 + 0][i] = v.x;
        sF[4 * j4 + 1][i] = v.y;
        sF[4 * j4 + 2][i] = v.z;
        sF[4 * j4 + 3][i] = v.w;
      }
    } else {
      // F given as [16][K] (A)
      for (int i = threadIdx.x; i < 16 * kSkCols / 4; i += 256) {
        const int j = i / (kSkCols / 4), c4 = (i % (kSkCols / 4)) * 4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k0 + c4 < K) v = *reinterpret_cast<const float4*>(F + (int64_t)j * K + k0 + c4);
        *reinterpret_cast<float4*>(&sF[j][c4]) = v;
      }
    }
    __syncthreads();
    const int64_t k = k0 + 8 * lane;
    // this lane's 4 rows x 8 columns of x~ (zero outside the matrix)
    float xm[4][8];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int64_t m = m0 + r;
#pragma unroll
      for (int e = 0; e < 8; ++e) xm[r][e] = 0.0f;
      if (m < M && k < K) {
        const uint4 xv = *reinterpret_cast<const uint4*>(x + m * K + k);
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
        uint32_t bits = 0xFFu;
        if (MASKED) {
          const uint64_t e0 = (uint64_t)(m * K + k);
          bits = keep4(key, e0) | (keep4(key, e0 + 4) << 4);
          if (mask_bytes) mask_bytes[e0 >> 3] = (uint8_t)bits;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          xm[r][2 * i] = ((bits >> (2 * i)) & 1u) ? bf16_lo(xw[i]) : 0.0f;
          xm[r][2 * i + 1] = ((bits >> (2 * i + 1)) & 1u) ? bf16_hi(xw[i]) : 0.0f;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float4 a0 = *reinterpret_cast<const float4*>(&sF[j][8 * lane]);
      const float4 a1 = *reinterpret_cast<const float4*>(&sF[j][8 * lane + 4]);
      const float f[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        float s = acc[r * 16 + j];
#pragma unroll
        for (int e = 0; e < 8; ++e) s = fmaf(xm[r][e], f[e], s);
        acc[r * 16 + j] = s;
      }
    }
  }
  // fixed butterfly reduce-scatter over the 32 lanes: 64 -> 2 values/lane
#pragma unroll
  for (int lvl = 0, width = 32; lvl < 5; ++lvl, width >>= 1) {
    const int off = 16 >> lvl;
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int v = 0; v < 32; ++v) {
      if (v < width) {
        const float keep = upper ? acc[v + width] : acc[v];
        const float send = upper ? acc[v] : acc[v + width];
        acc[v] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
  }
  const int64_t m = m0 + lane / 8;
  if (m < M) {
    float2* dst = reinterpret_cast<float2*>(partial + ((int64_t)blockIdx.y * M + m) * 16 +
                                            2 * (lane % 8));
    *dst = make_float2(acc[0], acc[1]);
  }
}

// out[m][:] = sum over chunks (index order) -> fp32 [M,16] and the bf16
// [hi | lo | hi | 0] split row [M,64] the tensor-core LoRA step consumes.
__global__ void k_skinny_finish(const float* __restrict__ partial, int chunks, int64_t M,
                                float* __restrict__ out, uint16_t* __restrict__ ext) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // (m, j)
  if (t >= M * 16) return;
  const int64_t m = t / 16;
  const int j = (int)(t % 16);
  const float* src = partial + t;
  const int64_t stride = M * 16;
  float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
  int c = 0;
  // four interleaved running sums, combined in a fixed order at the end
  for (; c + 4 <= chunks; c += 4) {
    a0 += __ldg(src + (int64_t)c * stride);
    a1 += __ldg(src + (int64_t)(c + 1) * stride);
    a2 += __ldg(src + (int64_t)(c + 2) * stride);
    a3 += __ldg(src + (int64_t)(c + 3) * stride);
  }
  for (; c < chunks; ++c) a0 += __ldg(src + (int64_t)c * stride);
  const float a = (a0 + a1) + (a2 + a3);
  out[t] = a;
  const uint16_t hi = f32_to_bf16_bits(a);
  const uint16_t lo = f32_to_bf16_bits(a - bf16_bits_to_f32(hi));
  uint16_t* e = ext + m * 64;
  e[j] = hi;
  e[16 + j] = lo;
  e[32 + j] = hi;
  e[48 + j] = 0;
}

// Column slices of 256 per block, chosen so the grid still covers about two
// blocks per SM; the chunk count (partials to sum) shrinks accordingly.
int skinny_slices(int64_t M, int64_t K) {
  const int64_t slices = (K + kSkCols - 1) / kSkCols;
  const int64_t mblocks = (M + kSkRows - 1) / kSkRows;
  int64_t per = slices * mblocks / (2 * device_sm_count());
  if (per < 1) per = 1;
  if (per > slices) per = slices;
  return (int)per;
}
int skinny_chunks(int64_t M, int64_t K) {
  const int64_t slices = (K + kSkCols - 1) / kSkCols;
  const int per = skinny_slices(M, K);
  return (int)((slices + per - 1) / per);
}

// ------------------------------------------------------------------------ a3/a5: s P^T Q
// out[c][j] = s * sum_m P[m][j] * Q~[m][c].  Thread = two adjacent columns;
// block = 512 columns x one chunk of rows (rows summed in order); a second
// kernel sums the chunks in index order.
constexpr int kWgradCols = 512;

__global__ void __launch_bounds__(256) k_wgrad_partial(const float* __restrict__ P,
                                                       const uint16_t* __restrict__ Q,
                                                       const uint32_t* __restrict__ mask,
                                                       int64_t M, int64_t C, int rows_per_chunk,
                                                       float* __restrict__ partial) {
  __shared__ __align__(16) float sP[64][16];
  const int64_t c = (int64_t)blockIdx.x * kWgradCols + 2 * threadIdx.x;
  const int64_t r0 = (int64_t)blockIdx.y * rows_per_chunk;
  const int64_t r1 = min(M, r0 + rows_per_chunk);
  const bool col_ok = c < C;
  float acc0[16], acc1[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    acc0[j] = 0.0f;
    acc1[j] = 0.0f;
  }
  for (int64_t mb = r0; mb < r1; mb += 64) {
    const int rows = (int)((r1 - mb) < 64 ? (r1 - mb) : 64);
    __syncthreads();
    for (int i = threadIdx.x; i < rows * 4; i += blockDim.x)
      *reinterpret_cast<float4*>(&sP[i / 4][(i % 4) * 4]) =
          *reinterpret_cast<const float4*>(P + (mb + i / 4) * 16 + (i % 4) * 4);
    __syncthreads();
    if (!col_ok) continue;
    // rows in groups of 8: issue the 8 independent loads first, then the FMAs
    for (int rg = 0; rg < rows; rg += 8) {
      float q0[8], q1[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        q0[u] = 0.0f;
        q1[u] = 0.0f;
        if (rg + u < rows) {
          const int64_t m = mb + rg + u;
          const uint32_t qq = __ldg(reinterpret_cast<const unsigned int*>(Q + m * C + c));
          q0[u] = bf16_lo(qq);
          q1[u] = bf16_hi(qq);
          if (mask) {
            const uint32_t w = __ldg(mask + ((m * C + c) >> 5));
            const int b = (int)(c & 31);
            if (!((w >> b) & 1u)) q0[u] = 0.0f;
            if (!((w >> (b + 1)) & 1u)) q1[u] = 0.0f;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (rg + u < rows) {
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            const float4 p = *reinterpret_cast<const float4*>(&sP[rg + u][4 * j4]);
            acc0[4 * j4 + 0] = fmaf(p.x, q0[u], acc0[4 * j4 + 0]);
            acc0[4 * j4 + 1] = fmaf(p.y, q0[u], acc0[4 * j4 + 1]);
            acc0[4 * j4 + 2] = fmaf(p.z, q0[u], acc0[4 * j4 + 2]);
            acc0[4 * j4 + 3] = fmaf(p.w, q0[u], acc0[4 * j4 + 3]);
            acc1[4 * j4 + 0] = fmaf(p.x, q1[u], acc1[4 * j4 + 0]);
            acc1[4 * j4 + 1] = fmaf(p.y, q1[u], acc1[4 * j4 + 1]);
            acc1[4 * j4 + 2] = fmaf(p.z, q1[u], acc1[4 * j4 + 2]);
            acc1[4 * j4 + 3] = fmaf(p.w, q1[u], acc1[4 * j4 + 3]);
          }
        }
      }
    }
  }
  if (col_ok) {
    float4* dst = reinterpret_cast<float4*>(partial + ((int64_t)blockIdx.y * C + c) * 16);
#pragma unroll
    for (int j4 = 0; j4 < 4; ++j4) {
      dst[j4] = make_float4(acc0[4 * j4], acc0[4 * j4 + 1], acc0[4 * j4 + 2], acc0[4 * j4 + 3]);
      dst[4 + j4] = make_float4(acc1[4 * j4], acc1[4 * j4 + 1], acc1[4 * j4 + 2], acc1[4 * j4 + 3]);
    }
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
  // at least 64 rows per chunk: below that the partials cost more traffic
  // than the rows they sum
  const int64_t maxc = (M + 63) / 64;
  if (want > maxc) want = maxc;
  if (want < 1) want = 1;
  return (int)want;
}

// ------------------------------------------------------------------------ mask regeneration
__global__ void k_mask_gen(int64_t words, DropKey key, uint32_t* __restrict__ mask) {
  const int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (w >= words) return;
  resolve_step(key);
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
  k.step_dev = h.step_dev;
  return k;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

DropKeyHost make_drop_key(const ws_dropout_key& k) {
  DropKeyHost h{};
  h.step_dev = nullptr;
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

size_t skinny_partial_bytes(int64_t M, int64_t K) {
  return (size_t)skinny_chunks(M, K) * (size_t)M * 16 * sizeof(float);
}

cudaError_t run_lora_down(const uint16_t* x, const float* A, int64_t M, int64_t K,
                          const DropKeyHost& key, float* U, uint16_t* Uext, uint32_t* mask_out,
                          float* partial, cudaStream_t st) {
  const int chunks = skinny_chunks(M, K);
  dim3 grid((unsigned)((M + kSkRows - 1) / kSkRows), (unsigned)chunks);
  note_launch();
  k_skinny_partial<true, false><<<grid, 256, 0, st>>>(x, A, M, K, skinny_slices(M, K), to_dev(key),
                                                      reinterpret_cast<uint8_t*>(mask_out), partial);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  note_launch();
  k_skinny_finish<<<(unsigned)((M * 16 + 255) / 256), 256, 0, st>>>(partial, chunks, M, U, Uext);
  return cudaGetLastError();
}

cudaError_t run_lora_G(const uint16_t* dY, const float* B, int64_t M, int64_t N, float* G,
                       uint16_t* Gext, float* partial, cudaStream_t st) {
  const int chunks = skinny_chunks(M, N);
  dim3 grid((unsigned)((M + kSkRows - 1) / kSkRows), (unsigned)chunks);
  DropKey none{};
  note_launch();
  k_skinny_partial<false, true><<<grid, 256, 0, st>>>(dY, B, M, N, skinny_slices(M, N), none, nullptr,
                                                      partial);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  note_launch();
  k_skinny_finish<<<(unsigned)((M * 16 + 255) / 256), 256, 0, st>>>(partial, chunks, M, G, Gext);
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
  k_wgrad_partial<<<grid, kWgradCols / 2, 0, st>>>(P, Q, mask, M, C, rpc, partial);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t n = C * 16;
  note_launch();
  k_wgrad_reduce<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(partial, chunks, C, s, out,
                                                              transpose_out);
  return cudaGetLastError();
}

cudaError_t run_wgrad_reduce(const float* partial, int chunks, int64_t C, float s, float* out,
                             int transpose_out, cudaStream_t st) {
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
  size_t ext, G, mask, wgrad, skinny, split, total;
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
  const size_t wg = wgrad_tc_bytes(M, N) > wgrad_tc_bytes(M, K) ? wgrad_tc_bytes(M, N)
                                                                : wgrad_tc_bytes(M, K);
  off += align256(wg);
  w.skinny = off;
  const size_t sk = skinny_partial_bytes(M, N) > skinny_partial_bytes(M, K) ? skinny_partial_bytes(M, N)
                                                                            : skinny_partial_bytes(M, K);
  off += align256(sk);
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
  cudaError_t e = run_lora_down(x, A, M, W.K, key, U, Uext, mask,
                                reinterpret_cast<float*>(w + L.skinny), st);
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
  e = run_lora_G(dY, B, M, W.N, G, Gext, reinterpret_cast<float*>(w + L.skinny), st);
  if (e != cudaSuccess) return e;
  if (dB) {
    e = run_wgrad_tc(U, dY, nullptr, M, W.N, scale, dB, 0, wg, st);
    if (e != cudaSuccess) return e;
  }
  if (dA) {
    e = run_wgrad_tc(G, x, mask, M, W.K, scale, dA, 1, wg, st);
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
