// stack.cu -- the synthetic transformer stack around the NF4-LoRA linears,
// the block forward / backward-with-recompute, and the streamed training
// step (pinned host -> 2-slot HBM window on a copy stream).
//
// Pointwise and row kernels are HBM-bound; each row reduction (RMSNorm,
// its backward, the loss) sums in a fixed order: per-thread strided sums, a
// fixed butterfly inside each warp, warps added in index order.
#include <math.h>
#include <string.h>

#include "common.cuh"
#include "kernels.h"

namespace ws {

namespace {

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

// ---------------------------------------------------------------------------- kernels
WS_DEVINL float block_sum_256(float v, float* red) {
  // blockDim.x == 256: butterfly inside each warp, then warp 0 adds the 8
  // warp totals in index order; every thread returns the same total.
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.0f;
  if (threadIdx.x == 0) {
    for (int w = 0; w < 8; ++w) t += red[w];
    red[8] = t;
  }
  __syncthreads();
  return red[8];
}

__global__ void __launch_bounds__(256) k_rmsnorm_fwd(const float* __restrict__ h, int64_t H,
                                                     float eps, uint16_t* __restrict__ out,
                                                     float* __restrict__ rstd) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float red[9];
  const int64_t m = blockIdx.x;
  const float4* row = reinterpret_cast<const float4*>(h + m * H);
  const int H4 = (int)(H / 4);
  float ss = 0.0f;
  for (int i = threadIdx.x; i < H4; i += 256) {
    const float4 v = row[i];
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
  }
  ss = block_sum_256(ss, red);
  const float rs = 1.0f / sqrtf(ss / (float)H + eps);
  if (threadIdx.x == 0) rstd[m] = rs;
  uint2* o = reinterpret_cast<uint2*>(out + m * H);
  for (int i = threadIdx.x; i < H4; i += 256) {
    const float4 v = row[i];
    o[i] = make_uint2(pack_bf16x2(v.x * rs, v.y * rs), pack_bf16x2(v.z * rs, v.w * rs));
  }
}

// dx_out = dx_in + (rstd*dy - rstd^3 * x * (dy . x) / H); dx_out may be dx_in
__global__ void __launch_bounds__(256) k_rmsnorm_bwd(const float* __restrict__ x,
                                                     const float* __restrict__ rstd,
                                                     const float* __restrict__ dy, int64_t H,
                                                     const float* dx_in, float* dx_out) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float red[9];
  const int64_t m = blockIdx.x;
  const float4* xr = reinterpret_cast<const float4*>(x + m * H);
  const float4* dr = reinterpret_cast<const float4*>(dy + m * H);
  const int H4 = (int)(H / 4);
  float dot = 0.0f;
  for (int i = threadIdx.x; i < H4; i += 256) {
    const float4 a = dr[i], b = xr[i];
    dot = fmaf(a.x, b.x, dot);
    dot = fmaf(a.y, b.y, dot);
    dot = fmaf(a.z, b.z, dot);
    dot = fmaf(a.w, b.w, dot);
  }
  dot = block_sum_256(dot, red);
  const float rs = rstd[m];
  const float coef = rs * rs * rs * dot / (float)H;
  const float4* in = reinterpret_cast<const float4*>(dx_in + m * H);
  float4* o = reinterpret_cast<float4*>(dx_out + m * H);
  for (int i = threadIdx.x; i < H4; i += 256) {
    const float4 a = dr[i], b = xr[i];
    float4 v = in[i];
    v.x += rs * a.x - coef * b.x;
    v.y += rs * a.y - coef * b.y;
    v.z += rs * a.z - coef * b.z;
    v.w += rs * a.w - coef * b.w;
    o[i] = v;
  }
}

WS_DEVINL float silu_sig(float g) { return 1.0f / (1.0f + expf(-g)); }

// 8 elements per thread (n % 8 == 0)
__global__ void k_silu_mul_fwd(const uint16_t* __restrict__ g, const uint16_t* __restrict__ u,
                               int64_t n, uint16_t* __restrict__ act) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t i8 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i8 * 8 >= n) return;
  const uint4 gv = reinterpret_cast<const uint4*>(g)[i8];
  const uint4 uv = reinterpret_cast<const uint4*>(u)[i8];
  const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float g0 = bf16_lo(gw[k]), g1 = bf16_hi(gw[k]);
    const float u0 = bf16_lo(uw[k]), u1 = bf16_hi(uw[k]);
    o[k] = pack_bf16x2(g0 * silu_sig(g0) * u0, g1 * silu_sig(g1) * u1);
  }
  reinterpret_cast<uint4*>(act)[i8] = make_uint4(o[0], o[1], o[2], o[3]);
}

__global__ void k_silu_mul_bwd(const float* __restrict__ dact, const uint16_t* __restrict__ g,
                               const uint16_t* __restrict__ u, int64_t n, uint16_t* __restrict__ dg,
                               uint16_t* __restrict__ du) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t i8 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i8 * 8 >= n) return;
  const uint4 gv = reinterpret_cast<const uint4*>(g)[i8];
  const uint4 uv = reinterpret_cast<const uint4*>(u)[i8];
  const float4 d0 = reinterpret_cast<const float4*>(dact)[2 * i8];
  const float4 d1 = reinterpret_cast<const float4*>(dact)[2 * i8 + 1];
  const float d[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
  const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
  uint32_t og[4], ou[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float g0 = bf16_lo(gw[k]), g1 = bf16_hi(gw[k]);
    const float u0 = bf16_lo(uw[k]), u1 = bf16_hi(uw[k]);
    const float s0 = silu_sig(g0), s1 = silu_sig(g1);
    ou[k] = pack_bf16x2(d[2 * k] * g0 * s0, d[2 * k + 1] * g1 * s1);
    og[k] = pack_bf16x2(d[2 * k] * u0 * s0 * (1.0f + g0 * (1.0f - s0)),
                        d[2 * k + 1] * u1 * s1 * (1.0f + g1 * (1.0f - s1)));
  }
  reinterpret_cast<uint4*>(dg)[i8] = make_uint4(og[0], og[1], og[2], og[3]);
  reinterpret_cast<uint4*>(du)[i8] = make_uint4(ou[0], ou[1], ou[2], ou[3]);
}

// vr[m, hh*hd + d] = v[m, (hh / rep)*hd + d]; 8 elements per thread
__global__ void k_repeat_fwd(const uint16_t* __restrict__ v, int M, int H, int KV, int hd,
                             uint16_t* __restrict__ vr) {
  pdl_wait();
  pdl_launch_dependents();
  const int i8 = blockIdx.x * blockDim.x + threadIdx.x;
  const int H8 = H / 8;
  if (i8 >= M * H8) return;
  const int m = i8 / H8, c = (i8 % H8) * 8;
  const int rep = H / KV;
  const int hh = c / hd, d = c % hd;
  reinterpret_cast<uint4*>(vr)[i8] =
      *reinterpret_cast<const uint4*>(v + (int64_t)m * KV + (hh / rep) * hd + d);
}

// dv[m, kh*hd + d] = bf16( sum_{t < rep} dvr[m, (kh*rep + t)*hd + d] ), t ascending;
// 4 elements per thread
__global__ void k_repeat_bwd(const float* __restrict__ dvr, int M, int H, int KV, int hd,
                             uint16_t* __restrict__ dv) {
  pdl_wait();
  pdl_launch_dependents();
  const int i4 = blockIdx.x * blockDim.x + threadIdx.x;
  const int KV4 = KV / 4;
  if (i4 >= M * KV4) return;
  const int m = i4 / KV4, c = (i4 % KV4) * 4;
  const int rep = H / KV;
  const int kh = c / hd, d = c % hd;
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int t = 0; t < rep; ++t) {
    const float4 x = *reinterpret_cast<const float4*>(dvr + (int64_t)m * H + (kh * rep + t) * hd + d);
    s.x += x.x;
    s.y += x.y;
    s.z += x.z;
    s.w += x.w;
  }
  reinterpret_cast<uint2*>(dv)[i4] = make_uint2(pack_bf16x2(s.x, s.y), pack_bf16x2(s.z, s.w));
}

// out = h + float(y); 8 elements per thread
__global__ void k_add_bf16(const float* __restrict__ h, const uint16_t* __restrict__ y, int64_t n,
                           float* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t i8 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i8 * 8 >= n) return;
  const uint4 yv = reinterpret_cast<const uint4*>(y)[i8];
  const float4 h0 = reinterpret_cast<const float4*>(h)[2 * i8];
  const float4 h1 = reinterpret_cast<const float4*>(h)[2 * i8 + 1];
  reinterpret_cast<float4*>(out)[2 * i8] =
      make_float4(h0.x + bf16_lo(yv.x), h0.y + bf16_hi(yv.x), h0.z + bf16_lo(yv.y), h0.w + bf16_hi(yv.y));
  reinterpret_cast<float4*>(out)[2 * i8 + 1] =
      make_float4(h1.x + bf16_lo(yv.z), h1.y + bf16_hi(yv.z), h1.z + bf16_lo(yv.w), h1.w + bf16_hi(yv.w));
}

__global__ void k_cast_bf16(const float* __restrict__ x, int64_t n, uint16_t* __restrict__ y) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t i8 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i8 * 8 >= n) return;
  const float4 a = reinterpret_cast<const float4*>(x)[2 * i8];
  const float4 b = reinterpret_cast<const float4*>(x)[2 * i8 + 1];
  reinterpret_cast<uint4*>(y)[i8] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w),
                                               pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
}

// loss = 0.5 * sum(h^2) / n in two fixed-order passes; dh = h / n.
constexpr int kLossBlocks = 256;
__global__ void __launch_bounds__(256) k_loss_partial(const float* __restrict__ h, int64_t n,
                                                      float* __restrict__ partial,
                                                      float* __restrict__ dh, float inv_n) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float red[9];
  const int64_t per = (n + kLossBlocks - 1) / kLossBlocks;
  const int64_t b0 = (int64_t)blockIdx.x * per, b1 = min(n, b0 + per);
  float s = 0.0f;
  for (int64_t i = b0 + threadIdx.x; i < b1; i += 256) {
    const float v = h[i];
    s = fmaf(v, v, s);
    dh[i] = v * inv_n;
  }
  s = block_sum_256(s, red);
  if (threadIdx.x == 0) partial[blockIdx.x] = s;
}
// accumulate != 0: add this micro-batch's share to the step loss (micro-batches in order)
__global__ void k_loss_final(const float* __restrict__ partial, float inv_n, int accumulate,
                             float* __restrict__ loss) {
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  float s = 0.0f;
  for (int i = 0; i < kLossBlocks; ++i) s += partial[i];
  const float l = 0.5f * s * inv_n;
  *loss = accumulate ? *loss + l : l;
}

// PyTorch-default Adam (no weight decay, bias-corrected); 4 parameters per
// thread.  The step t = *step_dev + 1 is read on the device so the same
// kernel serves eager calls and graph replays; the bias corrections are
// computed in double, once per block.
WS_DEVINL void adam1(float& p, float g, float& m, float& v, float beta1, float beta2, float eps,
                     float step_size, float bc2_sqrt) {
  m = beta1 * m + (1.0f - beta1) * g;
  v = beta2 * v + (1.0f - beta2) * g * g;
  const float denom = sqrtf(v) / bc2_sqrt + eps;
  p = p - step_size * (m / denom);
}
__global__ void k_adam(float* __restrict__ p, const float* __restrict__ g, float* __restrict__ m,
                       float* __restrict__ v, int64_t n, const uint32_t* __restrict__ step_dev,
                       float lr) {
  pdl_wait();
  pdl_launch_dependents();
  // bias corrections of this step, computed once by k_set_step
  const float step_size = lr * __uint_as_float(__ldg(step_dev + 2));
  const float bc2_sqrt = __uint_as_float(__ldg(step_dev + 3));
  const float beta1 = 0.9f, beta2 = 0.999f, eps = 1e-8f;
  const int64_t i4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i4 * 4 >= n) return;
  float4 pp = reinterpret_cast<float4*>(p)[i4];
  const float4 gg = reinterpret_cast<const float4*>(g)[i4];
  float4 mm = reinterpret_cast<float4*>(m)[i4];
  float4 vv = reinterpret_cast<float4*>(v)[i4];
  adam1(pp.x, gg.x, mm.x, vv.x, beta1, beta2, eps, step_size, bc2_sqrt);
  adam1(pp.y, gg.y, mm.y, vv.y, beta1, beta2, eps, step_size, bc2_sqrt);
  adam1(pp.z, gg.z, mm.z, vv.z, beta1, beta2, eps, step_size, bc2_sqrt);
  adam1(pp.w, gg.w, mm.w, vv.w, beta1, beta2, eps, step_size, bc2_sqrt);
  reinterpret_cast<float4*>(p)[i4] = pp;
  reinterpret_cast<float4*>(m)[i4] = mm;
  reinterpret_cast<float4*>(v)[i4] = vv;
}

// The step word and, after it, Adam's bias corrections for step t = step + 1:
// 1 / (1 - 0.9^t) and sqrt(1 - 0.999^t), computed in double, stored as fp32.
__global__ void k_set_step(uint32_t* step_dev, uint32_t step) {
  pdl_wait();
  pdl_launch_dependents();
  const double t = (double)step + 1.0;
  step_dev[0] = step;
  step_dev[2] = __float_as_uint((float)(1.0 / (1.0 - pow(0.9, t))));
  step_dev[3] = __float_as_uint((float)sqrt(1.0 - pow(0.999, t)));
}

unsigned nblk(int64_t n, int t = 256) { return (unsigned)((n + t - 1) / t); }

// ---------------------------------------------------------------------------- layouts
struct Shapes {
  int64_t N[WS_NLIN], K[WS_NLIN];
};
Shapes shapes_of(const ws_stack_cfg& c) {
  Shapes s;
  const int64_t H = c.H, KV = c.KV, I = c.I;
  const int64_t N[WS_NLIN] = {H, KV, KV, H, I, I, H};
  const int64_t K[WS_NLIN] = {H, H, H, H, H, H, I};
  for (int i = 0; i < WS_NLIN; ++i) {
    s.N[i] = N[i];
    s.K[i] = K[i];
  }
  return s;
}

struct SavedLayout {
  size_t h, a, rstd1, v, vr, h1, b, rstd2, g, u, act, U[WS_NLIN], mask[WS_NLIN];
  size_t q, k, o32, lse;  // attention core only (zero bytes with repeat(v))
  size_t total;
};
SavedLayout saved_layout(const ws_stack_cfg& c) {
  const Shapes s = shapes_of(c);
  const size_t M = (size_t)c.M, H = (size_t)c.H, KV = (size_t)c.KV, I = (size_t)c.I;
  SavedLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t r = o;
    o += al256(bytes);
    return r;
  };
  L.h = take(M * H * 4);
  L.a = take(M * H * 2);
  L.rstd1 = take(M * 4);
  L.v = take(M * KV * 2);
  L.vr = take(M * H * 2);
  L.h1 = take(M * H * 4);
  L.b = take(M * H * 2);
  L.rstd2 = take(M * 4);
  L.g = take(M * I * 2);
  L.u = take(M * I * 2);
  L.act = take(M * I * 2);
  for (int i = 0; i < WS_NLIN; ++i) L.U[i] = take(M * 16 * 4);
  for (int i = 0; i < WS_NLIN; ++i) L.mask[i] = take(M * (size_t)(s.K[i] / 32) * 4);
  const bool at = c.attn == WS_ATTN_CAUSAL;
  L.q = take(at ? M * H * 2 : 0);
  L.k = take(at ? M * KV * 2 : 0);
  L.o32 = take(at ? M * H * 4 : 0);
  L.lse = take(at ? (H / (size_t)c.head_dim) * M * 4 : 0);
  L.total = o;
  return L;
}

struct WeightLayout {
  size_t codes[WS_NLIN], absmax[WS_NLIN], layer_bytes;
};
// Per layer, the 7 linears in q,k,v,o,gate,up,down order, each piece
// 256-aligned: NF4 codes then block scales, or the bf16 weight alone.
WeightLayout weight_layout(const ws_stack_cfg& c) {
  const Shapes s = shapes_of(c);
  WeightLayout L{};
  size_t o = 0;
  for (int i = 0; i < WS_NLIN; ++i) {
    L.codes[i] = o;
    if (c.base == WS_BASE_BF16) {
      o += al256((size_t)s.N[i] * (size_t)s.K[i] * 2);
      L.absmax[i] = L.codes[i];
      continue;
    }
    o += al256((size_t)s.N[i] * (size_t)(s.K[i] / 2));
    L.absmax[i] = o;
    o += al256((size_t)(s.K[i] / 64) * (size_t)s.N[i] * 4);
  }
  L.layer_bytes = o;
  return L;
}

struct ParamLayout {
  int64_t A[WS_NLIN], B[WS_NLIN], layer_floats;
};
ParamLayout param_layout(const ws_stack_cfg& c) {
  const Shapes s = shapes_of(c);
  ParamLayout L{};
  int64_t o = 0;
  auto al = [](int64_t x) { return (x + 63) & ~int64_t(63); };
  for (int i = 0; i < WS_NLIN; ++i) {
    L.A[i] = o;
    o += al(16 * s.K[i]);
    L.B[i] = o;
    o += al(s.N[i] * 16);
  }
  L.layer_floats = o;
  return L;
}

struct WsLayout {
  size_t lin, blk, qout, kout, yout, y1, dact, dg, du, db, dh1, dvr, dv, da, lossp, stepw;
  size_t dob, dq, dk, attn;  // attention core only
  size_t total;
};
WsLayout ws_layout(const ws_stack_cfg& c, int block_layers) {
  const Shapes s = shapes_of(c);
  const size_t M = (size_t)c.M, H = (size_t)c.H, KV = (size_t)c.KV, I = (size_t)c.I;
  WsLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t r = o;
    o += al256(bytes);
    return r;
  };
  size_t lin = 0;
  for (int i = 0; i < WS_NLIN; ++i) {
    const size_t b = linear_workspace_bytes(c.M, s.N[i], s.K[i]);
    if (b > lin) lin = b;
  }
  // the forward runs q, k, v and gate, up as groups (one launch each)
  const int64_t nqkv[3] = {s.N[WS_LIN_Q], s.N[WS_LIN_K], s.N[WS_LIN_V]};
  const int64_t ngu[2] = {s.N[WS_LIN_GATE], s.N[WS_LIN_UP]};
  const size_t g3 = linear_group_workspace_bytes(c.M, 3, nqkv, s.K[WS_LIN_Q]);
  const size_t g2 = linear_group_workspace_bytes(c.M, 2, ngu, s.K[WS_LIN_GATE]);
  if (g3 > lin) lin = g3;
  if (g2 > lin) lin = g2;
  const size_t b2 = linear_bwd_group_workspace_bytes(c.M, 2, s.N[WS_LIN_GATE], s.K[WS_LIN_GATE]);
  if (b2 > lin) lin = b2;
  // the attention core's backward runs v and k as one group
  const size_t b3 = linear_bwd_group_workspace_bytes(c.M, 2, s.N[WS_LIN_K], s.K[WS_LIN_K]);
  if (b3 > lin) lin = b3;
  L.lin = take(lin);
  L.blk = take((size_t)block_layers * saved_layout(c).total);
  L.qout = take(M * H * 2);
  L.kout = take(M * KV * 2);
  L.yout = take(M * H * 2);
  L.y1 = take(M * H * 2);
  L.dact = take(M * I * 4);
  L.dg = take(M * I * 2);
  L.du = take(M * I * 2);
  L.db = take(M * H * 4);
  L.dh1 = take(M * H * 4);
  L.dvr = take(M * H * 4);
  L.dv = take(M * KV * 2);
  L.da = take(M * H * 4);
  L.lossp = take(kLossBlocks * 4);
  L.stepw = take(16);
  const bool at = c.attn == WS_ATTN_CAUSAL;
  L.dob = take(at ? M * H * 2 : 0);
  L.dq = take(at ? M * H * 2 : 0);
  L.dk = take(at ? M * KV * 2 : 0);
  L.attn = take(at ? attn_bwd_workspace_bytes(c.M, (int)(c.H / c.head_dim), (int)c.head_dim) : 0);
  L.total = o;
  return L;
}

template <class T>
T* at(const void* base, size_t off) {
  return reinterpret_cast<T*>(const_cast<uint8_t*>(static_cast<const uint8_t*>(base)) + off);
}

#define WS_TRY(x)                           \
  do {                                      \
    cudaError_t e_ = (x);                   \
    if (e_ != cudaSuccess) return e_;       \
  } while (0)

struct Ctx {
  ws_stack_cfg c;
  Shapes s;
  SavedLayout SL;
  WeightLayout WL;
  ParamLayout PL;
  WsLayout WSL;
  float scale;
  cudaStream_t st;
  void* ws;
  const uint32_t* step_dev;
};

NF4View wview(const Ctx& x, const void* block, int layer_in_block, int lin) {
  NF4View v;
  const uint8_t* base = static_cast<const uint8_t*>(block) + (size_t)layer_in_block * x.WL.layer_bytes;
  v.N = x.s.N[lin];
  v.K = x.s.K[lin];
  if (x.c.base == WS_BASE_BF16) {
    v.codes = nullptr;
    v.absmax = nullptr;
    v.wbf16 = reinterpret_cast<const uint16_t*>(base + x.WL.codes[lin]);
    return v;
  }
  v.codes = base + x.WL.codes[lin];
  v.absmax = reinterpret_cast<const float*>(base + x.WL.absmax[lin]);
  return v;
}

DropKeyHost key_of(const Ctx& x, uint32_t step, int layer, int lin, uint32_t mb) {
  ws_dropout_key k{};
  k.seed = x.c.seed;
  k.step = step;
  k.layer = (uint32_t)layer;
  k.linear = (uint32_t)lin;
  k.microbatch = mb;
  k.p = x.c.p;
  DropKeyHost h = make_drop_key(k);
  h.step_dev = x.step_dev;
  return h;
}

// Forward of one layer.  S: saved slot of this layer.  with_qk: compute the
// q and k projections (the first forward does; a recompute skips them since
// nothing downstream reads them).
cudaError_t layer_fwd(const Ctx& x, const void* block, int lib, int layer, const float* params,
                      uint32_t step, uint32_t mb, const float* h_in, float* h_out, uint8_t* S,
                      bool with_qk) {
  const int64_t M = x.c.M, H = x.c.H, KV = x.c.KV, I = x.c.I;
  const SavedLayout& L = x.SL;
  cudaStream_t st = x.st;
  uint8_t* ws = static_cast<uint8_t*>(x.ws);
  void* lws = ws + x.WSL.lin;
  const float* P = params + (int64_t)layer * x.PL.layer_floats;
  auto lin = [&](int li, const uint16_t* in, uint16_t* out) {
    return linear_fwd(wview(x, block, lib, li), in, P + x.PL.A[li], P + x.PL.B[li], M, x.scale,
                      key_of(x, step, layer, li, mb), out, at<float>(S, L.U[li]),
                      at<uint32_t>(S, L.mask[li]), lws, st);
  };
  // linears reading the same input: one LoRA-down launch and one GEMM
  auto lin_group = [&](int ng, int ng_gemm, const int* li, const uint16_t* in,
                       uint16_t* const* outs) {
    NF4View W[kMaxGroups];
    const float* A[kMaxGroups];
    const float* B[kMaxGroups];
    DropKeyHost keys[kMaxGroups];
    float* U[kMaxGroups];
    uint32_t* mk[kMaxGroups];
    for (int g = 0; g < ng; ++g) {
      W[g] = wview(x, block, lib, li[g]);
      A[g] = P + x.PL.A[li[g]];
      B[g] = P + x.PL.B[li[g]];
      keys[g] = key_of(x, step, layer, li[g], mb);
      U[g] = at<float>(S, L.U[li[g]]);
      mk[g] = at<uint32_t>(S, L.mask[li[g]]);
    }
    return linear_fwd_group(ng, ng_gemm, W, in, A, B, M, x.scale, keys, outs, U, mk, lws, st);
  };
  float* h = at<float>(S, L.h);
  if (h != h_in) WS_TRY(cudaMemcpyAsync(h, h_in, (size_t)M * H * 4, cudaMemcpyDeviceToDevice, st));
  note_launch();
  (void)launch_pdl(k_rmsnorm_fwd, dim3((unsigned)M), dim3(256), 0, st, h, H, x.c.eps, at<uint16_t>(S, L.a), at<float>(S, L.rstd1));
  WS_TRY(cudaGetLastError());
  const bool attn = x.c.attn == WS_ATTN_CAUSAL;
  {
    // q, k, v share one LoRA-down launch and q + k one GEMM; v gets a GEMM
    // of its own.  A recompute of the repeat(v) stack needs only v: it runs
    // the same LoRA-down launch (so v's U is the forward's bit for bit) and
    // v's GEMM alone.
    const bool qk = with_qk || attn;
    const int li[3] = {WS_LIN_Q, WS_LIN_K, WS_LIN_V};
    uint16_t* outs[3] = {qk ? (attn ? at<uint16_t>(S, L.q) : at<uint16_t>(ws, x.WSL.qout)) : nullptr,
                         qk ? (attn ? at<uint16_t>(S, L.k) : at<uint16_t>(ws, x.WSL.kout)) : nullptr,
                         at<uint16_t>(S, L.v)};
    WS_TRY(lin_group(3, 2, li, at<uint16_t>(S, L.a), outs));
  }
  if (attn) {
    // causal attention over the M tokens as one sequence
    const int hd = (int)x.c.head_dim;
    WS_TRY(run_attn_fwd(at<uint16_t>(S, L.q), at<uint16_t>(S, L.k), at<uint16_t>(S, L.v), 1,
                        (int)M, (int)(H / hd), (int)(KV / hd), hd, at<uint16_t>(S, L.vr),
                        at<float>(S, L.o32), at<float>(S, L.lse), st));
  } else {
    note_launch();
    (void)launch_pdl(k_repeat_fwd, dim3(nblk(M * H / 8)), dim3(256), 0, st, at<uint16_t>(S, L.v),
                     (int)M, (int)H, (int)KV, (int)x.c.head_dim, at<uint16_t>(S, L.vr));
    WS_TRY(cudaGetLastError());
  }
  uint16_t* y = at<uint16_t>(ws, x.WSL.yout);
  WS_TRY(lin(WS_LIN_O, at<uint16_t>(S, L.vr), y));
  note_launch();
  (void)launch_pdl(k_add_bf16, dim3(nblk(M * H / 8)), dim3(256), 0, st, h, y, M * H, at<float>(S, L.h1));
  WS_TRY(cudaGetLastError());
  note_launch();
  (void)launch_pdl(k_rmsnorm_fwd, dim3((unsigned)M), dim3(256), 0, st, at<float>(S, L.h1), H, x.c.eps, at<uint16_t>(S, L.b),
                                            at<float>(S, L.rstd2));
  WS_TRY(cudaGetLastError());
  {
    const int li[2] = {WS_LIN_GATE, WS_LIN_UP};
    uint16_t* outs[2] = {at<uint16_t>(S, L.g), at<uint16_t>(S, L.u)};
    WS_TRY(lin_group(2, 2, li, at<uint16_t>(S, L.b), outs));
  }
  note_launch();
  (void)launch_pdl(k_silu_mul_fwd, dim3(nblk(M * I / 8)), dim3(256), 0, st, at<uint16_t>(S, L.g), at<uint16_t>(S, L.u), M * I,
                                              at<uint16_t>(S, L.act));
  WS_TRY(cudaGetLastError());
  WS_TRY(lin(WS_LIN_DOWN, at<uint16_t>(S, L.act), y));
  note_launch();
  (void)launch_pdl(k_add_bf16, dim3(nblk(M * H / 8)), dim3(256), 0, st, at<float>(S, L.h1), y, M * H, h_out);
  return cudaGetLastError();
}

// Backward of one layer from its saved slot S; dh holds the gradient at
// the layer output on entry and at the layer input on exit.  gacc != 0 adds
// the adapter gradients into `grads` (gradient accumulation) instead of
// overwriting them.  Every intermediate gradient has a workspace buffer of
// its own, so after the call they all hold this layer's values.
cudaError_t layer_bwd(const Ctx& x, const void* block, int lib, int layer, const float* params,
                      uint32_t step, uint32_t mb, const uint8_t* S, float* dh, float* grads,
                      int gacc) {
  const int64_t M = x.c.M, H = x.c.H, KV = x.c.KV, I = x.c.I;
  const SavedLayout& L = x.SL;
  cudaStream_t st = x.st;
  uint8_t* ws = static_cast<uint8_t*>(x.ws);
  void* lws = ws + x.WSL.lin;
  const float* P = params + (int64_t)layer * x.PL.layer_floats;
  float* Gd = grads + (int64_t)layer * x.PL.layer_floats;
  auto lin = [&](int li, const uint16_t* in, const uint16_t* dY, float* dX, int accum) {
    return linear_bwd(wview(x, block, lib, li), in, P + x.PL.A[li], P + x.PL.B[li], M, x.scale,
                      key_of(x, step, layer, li, mb), at<const float>(S, L.U[li]),
                      at<const uint32_t>(S, L.mask[li]), dY, dX, 1, accum, Gd + x.PL.A[li],
                      Gd + x.PL.B[li], gacc, lws, st);
  };
  uint16_t* y1 = at<uint16_t>(ws, x.WSL.y1);
  float* dact = at<float>(ws, x.WSL.dact);
  uint16_t* dg = at<uint16_t>(ws, x.WSL.dg);
  uint16_t* du = at<uint16_t>(ws, x.WSL.du);
  float* db = at<float>(ws, x.WSL.db);
  float* dh1 = at<float>(ws, x.WSL.dh1);
  float* dvr = at<float>(ws, x.WSL.dvr);
  uint16_t* dv = at<uint16_t>(ws, x.WSL.dv);
  float* da = at<float>(ws, x.WSL.da);

  note_launch();
  (void)launch_pdl(k_cast_bf16, dim3(nblk(M * H / 8)), dim3(256), 0, st, dh, M * H, y1);
  WS_TRY(cudaGetLastError());
  WS_TRY(lin(WS_LIN_DOWN, at<const uint16_t>(S, L.act), y1, dact, 0));
  note_launch();
  (void)launch_pdl(k_silu_mul_bwd, dim3(nblk(M * I / 8)), dim3(256), 0, st, dact, at<const uint16_t>(S, L.g),
                                              at<const uint16_t>(S, L.u), M * I, dg, du);
  WS_TRY(cudaGetLastError());
  {
    // gate and up read the same input: their LoRA products share launches
    const int li[2] = {WS_LIN_GATE, WS_LIN_UP};
    NF4View W[2];
    const float* A[2];
    const float* B[2];
    DropKeyHost keys[2];
    const float* U[2];
    const uint32_t* mk[2];
    const uint16_t* dYs[2] = {dg, du};
    float* dAs[2];
    float* dBs[2];
    for (int g = 0; g < 2; ++g) {
      W[g] = wview(x, block, lib, li[g]);
      A[g] = P + x.PL.A[li[g]];
      B[g] = P + x.PL.B[li[g]];
      keys[g] = key_of(x, step, layer, li[g], mb);
      U[g] = at<const float>(S, L.U[li[g]]);
      mk[g] = at<const uint32_t>(S, L.mask[li[g]]);
      dAs[g] = Gd + x.PL.A[li[g]];
      dBs[g] = Gd + x.PL.B[li[g]];
    }
    WS_TRY(linear_bwd_group(2, W, at<const uint16_t>(S, L.b), A, B, M, x.scale, keys, U, mk, dYs,
                            db, 1, 0, dAs, dBs, gacc, lws, st));
  }
  // dh1 = dh + RMSNorm2 backward (the residual passes dh through)
  note_launch();
  (void)launch_pdl(k_rmsnorm_bwd, dim3((unsigned)M), dim3(256), 0, st, at<const float>(S, L.h1), at<const float>(S, L.rstd2),
                                             (const float*)db, H, (const float*)dh, dh1);
  WS_TRY(cudaGetLastError());
  note_launch();
  (void)launch_pdl(k_cast_bf16, dim3(nblk(M * H / 8)), dim3(256), 0, st, (const float*)dh1, M * H, y1);
  WS_TRY(cudaGetLastError());
  if (x.c.attn == WS_ATTN_CAUSAL) {
    // o projection's input gradient as bf16 dO, the attention backward, then
    // the v, k and q projections, their input gradients summed into da
    const int hd = (int)x.c.head_dim;
    uint16_t* dob = at<uint16_t>(ws, x.WSL.dob);
    uint16_t* dq = at<uint16_t>(ws, x.WSL.dq);
    uint16_t* dk = at<uint16_t>(ws, x.WSL.dk);
    WS_TRY(linear_bwd(wview(x, block, lib, WS_LIN_O), at<const uint16_t>(S, L.vr),
                      P + x.PL.A[WS_LIN_O], P + x.PL.B[WS_LIN_O], M, x.scale,
                      key_of(x, step, layer, WS_LIN_O, mb), at<const float>(S, L.U[WS_LIN_O]),
                      at<const uint32_t>(S, L.mask[WS_LIN_O]), y1, dob, 0, 0,
                      Gd + x.PL.A[WS_LIN_O], Gd + x.PL.B[WS_LIN_O], gacc, lws, st));
    WS_TRY(run_attn_bwd(at<const uint16_t>(S, L.q), at<const uint16_t>(S, L.k),
                        at<const uint16_t>(S, L.v), at<const float>(S, L.o32),
                        at<const float>(S, L.lse), dob, 1, (int)M, (int)(H / hd), (int)(KV / hd),
                        hd, dq, dk, dv, ws + x.WSL.attn, st));
    {
      // v and k have one shape and read the same input: their LoRA products
      // and weight gradients share launches; da = dX_v + dX_k, then + dX_q
      const int li[2] = {WS_LIN_V, WS_LIN_K};
      NF4View W[2];
      const float* A[2];
      const float* B[2];
      DropKeyHost keys[2];
      const float* U[2];
      const uint32_t* mk[2];
      const uint16_t* dYs[2] = {dv, dk};
      float* dAs[2];
      float* dBs[2];
      for (int g = 0; g < 2; ++g) {
        W[g] = wview(x, block, lib, li[g]);
        A[g] = P + x.PL.A[li[g]];
        B[g] = P + x.PL.B[li[g]];
        keys[g] = key_of(x, step, layer, li[g], mb);
        U[g] = at<const float>(S, L.U[li[g]]);
        mk[g] = at<const uint32_t>(S, L.mask[li[g]]);
        dAs[g] = Gd + x.PL.A[li[g]];
        dBs[g] = Gd + x.PL.B[li[g]];
      }
      WS_TRY(linear_bwd_group(2, W, at<const uint16_t>(S, L.a), A, B, M, x.scale, keys, U, mk, dYs,
                              da, 1, 0, dAs, dBs, gacc, lws, st));
    }
    WS_TRY(lin(WS_LIN_Q, at<const uint16_t>(S, L.a), dq, da, 1));
    note_launch();
    (void)launch_pdl(k_rmsnorm_bwd, dim3((unsigned)M), dim3(256), 0, st,
                     at<const float>(S, L.h), at<const float>(S, L.rstd1), (const float*)da, H,
                     (const float*)dh1, dh);
    return cudaGetLastError();
  }
  WS_TRY(lin(WS_LIN_O, at<const uint16_t>(S, L.vr), y1, dvr, 0));
  note_launch();
  (void)launch_pdl(k_repeat_bwd, dim3(nblk(M * KV / 4)), dim3(256), 0, st, dvr, (int)M, (int)H, (int)KV, (int)x.c.head_dim, dv);
  WS_TRY(cudaGetLastError());
  WS_TRY(lin(WS_LIN_V, at<const uint16_t>(S, L.a), dv, da, 0));
  // dh = dh1 + RMSNorm1 backward
  note_launch();
  (void)launch_pdl(k_rmsnorm_bwd, dim3((unsigned)M), dim3(256), 0, st, at<const float>(S, L.h), at<const float>(S, L.rstd1),
                                             (const float*)da, H, (const float*)dh1, dh);
  WS_TRY(cudaGetLastError());
  // q and k feed only the replaced attention core: exactly zero gradient
  // (already zero when accumulating)
  if (!gacc) {
    for (int li : {WS_LIN_Q, WS_LIN_K}) {
      WS_TRY(cudaMemsetAsync(Gd + x.PL.A[li], 0, sizeof(float) * 16 * (size_t)x.s.K[li], st));
      WS_TRY(cudaMemsetAsync(Gd + x.PL.B[li], 0, sizeof(float) * 16 * (size_t)x.s.N[li], st));
    }
  }
  return cudaSuccess;
}

Ctx make_ctx(const ws_stack_cfg& c, int block_layers, void* ws, cudaStream_t st,
             const uint32_t* step_dev) {
  Ctx x;
  x.c = c;
  x.s = shapes_of(c);
  x.SL = saved_layout(c);
  x.WL = weight_layout(c);
  x.PL = param_layout(c);
  x.WSL = ws_layout(c, block_layers);
  x.scale = (float)(((double)c.alpha / (double)c.r) / (1.0 - c.p));
  x.st = st;
  x.ws = ws;
  x.step_dev = step_dev;
  return x;
}

}  // namespace

// ---------------------------------------------------------------------------- host API
ws_status stack_check(const ws_stack_cfg* c) {
  if (!c) return WS_ERR_INVALID;
  if (c->M < 1 || c->H < 64 || c->KV < 64 || c->I < 64 || c->head_dim < 1 || c->n_layers < 1)
    return WS_ERR_SHAPE;
  if (c->H % 64 || c->KV % 64 || c->I % 64) return WS_ERR_SHAPE;
  if (c->H % c->KV || c->H % c->head_dim || c->KV % c->head_dim) return WS_ERR_SHAPE;
  if (c->r != 16) return WS_ERR_SHAPE;
  if (!(c->p >= 0.0 && c->p < 1.0)) return WS_ERR_INVALID;
  if (c->base != WS_BASE_NF4 && c->base != WS_BASE_BF16) return WS_ERR_INVALID;
  if (c->attn != WS_ATTN_REPEAT_V && c->attn != WS_ATTN_CAUSAL) return WS_ERR_INVALID;
  if (c->attn == WS_ATTN_CAUSAL && ((c->head_dim != 64 && c->head_dim != 128) || c->M >= (1ll << 31)))
    return WS_ERR_SHAPE;
  if ((double)c->M * (double)c->I >= 17179869184.0) return WS_ERR_SHAPE;
  return WS_OK;
}

size_t stack_block_bytes(const ws_stack_cfg& c, int bl) { return (size_t)bl * weight_layout(c).layer_bytes; }
int64_t stack_n_params(const ws_stack_cfg& c) { return (int64_t)c.n_layers * param_layout(c).layer_floats; }
size_t stack_saved_layer(const ws_stack_cfg& c) { return saved_layout(c).total; }
size_t stack_ws_bytes(const ws_stack_cfg& c, int bl) { return ws_layout(c, bl).total; }
uint32_t* stack_step_word(const ws_stack_cfg& c, int block_layers, void* ws) {
  return at<uint32_t>(ws, ws_layout(c, block_layers).stepw);
}
bool stack_ws_offset(const ws_stack_cfg& c, int block_layers, int field, size_t* off) {
  const WsLayout L = ws_layout(c, block_layers);
  const size_t f[] = {L.y1, L.dact, L.dg, L.du, L.db, L.dh1, L.dvr, L.dv, L.da, L.yout, L.dob,
                      L.dq, L.dk};
  if (field < 0 || field >= (int)(sizeof(f) / sizeof(f[0]))) return false;
  *off = f[field];
  return true;
}
void stack_weight_offset(const ws_stack_cfg& c, int lib, int lin, size_t* oc, size_t* oa) {
  const WeightLayout L = weight_layout(c);
  *oc = (size_t)lib * L.layer_bytes + L.codes[lin];
  *oa = (size_t)lib * L.layer_bytes + L.absmax[lin];
}
bool stack_saved_offset(const ws_stack_cfg& c, int field, int lin, size_t* off) {
  const SavedLayout L = saved_layout(c);
  const size_t f[] = {L.h, L.a, L.rstd1, L.v, L.vr, L.h1, L.b, L.rstd2, L.g, L.u, L.act};
  if (field >= 0 && field <= WS_SV_ACT) {
    *off = f[field];
    return true;
  }
  if (field >= WS_SV_Q && field <= WS_SV_LSE) {
    const size_t g[] = {L.q, L.k, L.o32, L.lse};
    *off = g[field - WS_SV_Q];
    return true;
  }
  if (lin < 0 || lin >= WS_NLIN) return false;
  if (field == WS_SV_LORA_U) *off = L.U[lin];
  else if (field == WS_SV_MASK) *off = L.mask[lin];
  else return false;
  return true;
}
void stack_param_offset(const ws_stack_cfg& c, int layer, int lin, int64_t* oA, int64_t* oB) {
  const ParamLayout L = param_layout(c);
  *oA = (int64_t)layer * L.layer_floats + L.A[lin];
  *oB = (int64_t)layer * L.layer_floats + L.B[lin];
}

cudaError_t block_forward(const ws_stack_cfg& c, int block_layers_ws, const void* block,
                          int first_layer, int n_layers, const float* params, uint32_t step,
                          uint32_t mb, const uint32_t* step_dev, const float* h_in, float* h_out,
                          void* saved, void* ws, cudaStream_t st) {
  const Ctx x = make_ctx(c, block_layers_ws, ws, st, step_dev);
  uint8_t* blk_area = static_cast<uint8_t*>(ws) + x.WSL.blk;
  // Layer i works in slot S_i: the caller's saved area (kept for the
  // backward) or, when nothing is kept, one reused workspace slot.  Layer i
  // reads its input from S_i.h and writes its output into S_{i+1}.h; with a
  // single reused slot that overwrite happens after the layer's last read of
  // its input.
  auto slot = [&](int i) {
    return saved ? static_cast<uint8_t*>(saved) + (size_t)i * x.SL.total : blk_area;
  };
  for (int i = 0; i < n_layers; ++i) {
    uint8_t* S = slot(i);
    const float* src = i == 0 ? h_in : at<float>(S, x.SL.h);
    float* dst = i == n_layers - 1 ? h_out : at<float>(slot(i + 1), x.SL.h);
    WS_TRY(layer_fwd(x, block, i, first_layer + i, params, step, mb, src, dst, S, true));
  }
  return cudaSuccess;
}

cudaError_t block_backward(const ws_stack_cfg& c, int block_layers_ws, const void* block,
                           int first_layer, int n_layers, const float* params, uint32_t step,
                           uint32_t mb, const uint32_t* step_dev, const float* h_in,
                           const void* saved, const float* dh_out, float* dh_in, float* grads,
                           int grad_accum, void* ws, cudaStream_t st) {
  const Ctx x = make_ctx(c, block_layers_ws, ws, st, step_dev);
  const int64_t MH = c.M * c.H;
  const uint8_t* area = static_cast<const uint8_t*>(saved);
  if (!saved) {
    // recompute the block forward from its boundary activation, keeping
    // every layer's intermediates in the workspace block area
    uint8_t* blk = static_cast<uint8_t*>(ws) + x.WSL.blk;
    for (int i = 0; i < n_layers; ++i) {
      uint8_t* S = blk + (size_t)i * x.SL.total;
      const float* src = i == 0 ? h_in : at<float>(S, x.SL.h);
      float* dst;
      if (i == n_layers - 1) dst = at<float>(static_cast<uint8_t*>(ws) + x.WSL.dvr, 0);  // unused output
      else dst = at<float>(blk + (size_t)(i + 1) * x.SL.total, x.SL.h);
      WS_TRY(layer_fwd(x, block, i, first_layer + i, params, step, mb, src, dst, S, false));
    }
    area = blk;
  }
  if (dh_in != dh_out)
    WS_TRY(cudaMemcpyAsync(dh_in, dh_out, (size_t)MH * 4, cudaMemcpyDeviceToDevice, st));
  for (int i = n_layers - 1; i >= 0; --i)
    WS_TRY(layer_bwd(x, block, i, first_layer + i, params, step, mb, area + (size_t)i * x.SL.total,
                     dh_in, grads, grad_accum));
  return cudaSuccess;
}

cudaError_t loss_and_grad(const ws_stack_cfg& c, int block_layers_ws, const float* h, float* dh,
                          float* loss, int n_micro, int accumulate, void* ws, cudaStream_t st) {
  const WsLayout L = ws_layout(c, block_layers_ws);
  const int64_t n = c.M * c.H;
  float* part = at<float>(ws, L.lossp);
  // the step loss is the mean over micro-batches: each one contributes
  // 0.5 sum(h^2) / (n * n_micro), and its gradient is h / (n * n_micro)
  const float inv_n = (float)(1.0 / ((double)n * (double)n_micro));
  note_launch();
  (void)launch_pdl(k_loss_partial, dim3(kLossBlocks), dim3(256), 0, st, h, n, part, dh, inv_n);
  WS_TRY(cudaGetLastError());
  note_launch();
  (void)launch_pdl(k_loss_final, dim3(1), dim3(32), 0, st, (const float*)part, inv_n, accumulate, loss);
  return cudaGetLastError();
}

cudaError_t adam_step(float* p, const float* g, float* m, float* v, int64_t n,
                      const uint32_t* step_dev, float lr, cudaStream_t st) {
  note_launch();
  (void)launch_pdl(k_adam, dim3(nblk(n / 4)), dim3(256), 0, st, p, g, m, v, n, step_dev, lr);
  return cudaGetLastError();
}

cudaError_t set_step(uint32_t* step_dev, uint32_t step, cudaStream_t st) {
  note_launch();
  (void)launch_pdl(k_set_step, dim3(1), dim3(1), 0, st, step_dev, step);
  return cudaGetLastError();
}

}  // namespace ws
