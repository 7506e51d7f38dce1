// lora_small.cu -- the smaller pieces of one NF4-LoRA linear and the
// orchestration of its forward and backward: NF4 quantisation of a bf16
// weight, dropout-mask regeneration, the workspace layout, and the order of
// the kernels (the tensor-core kernels live in nf4_gemm.cu).  Every
// reduction runs in a fixed order: no atomics on data.
#include <math.h>
#include <stdlib.h>

#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "kernels.h"

namespace ws {

namespace {

__constant__ float c_levels_q[16] = {-1.0f,    -0.6962f, -0.5251f, -0.3949f, -0.2844f, -0.1848f,
                                     -0.0911f, 0.0f,     0.0796f,  0.1609f,  0.2461f,  0.3379f,
                                     0.4407f,  0.5626f,  0.7230f,  1.0f};

// ------------------------------------------------------------------------ NF4 quantisation
// One warp per 64-weight block; lane i handles weights 2i and 2i+1 and
// writes code byte i.  The block maximum is a max-reduction (exact in any
// order); v = w / absmax is an IEEE division; the code counts the midpoints
// below v.
__global__ void k_quantize_nf4(const uint16_t* __restrict__ W, int64_t N, int64_t K,
                               uint8_t* __restrict__ codes, float* __restrict__ absmax) {
  pdl_wait();
  pdl_launch_dependents();
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

// ------------------------------------------------------------------------ mask regeneration
__global__ void k_mask_gen(int64_t words, DropKey key, uint32_t* __restrict__ mask) {
  pdl_wait();
  pdl_launch_dependents();
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
  (void)launch_pdl(k_quantize_nf4, dim3((unsigned)((blocks + per - 1) / per)), dim3(32 * per), 0, st, W, N, K, codes, absmax);
  return cudaGetLastError();
}

cudaError_t run_lora_down(const uint16_t* x, const float* A, int64_t M, int64_t K,
                          const DropKeyHost& key, float* U, uint16_t* Uext, uint32_t* mask_out,
                          float* partial, cudaStream_t st) {
  const DropKey k = to_dev(key);
  return run_skinny_tc(x, A, false, M, K, &k, reinterpret_cast<uint8_t*>(mask_out), partial, U,
                       Uext, st);
}
cudaError_t run_lora_G(const uint16_t* dY, const float* B, int64_t M, int64_t N, float* G,
                       uint16_t* Gext, float* partial, cudaStream_t st) {
  return run_skinny_tc(dY, B, true, M, N, nullptr, nullptr, partial, G, Gext, st);
}

cudaError_t run_mask_gen(int64_t M, int64_t K, const DropKeyHost& key, uint32_t* mask,
                         cudaStream_t st) {
  const int64_t words = M * K / 32;
  note_launch();
  (void)launch_pdl(k_mask_gen, dim3((unsigned)((words + 255) / 256)), dim3(256), 0, st, words, to_dev(key), mask);
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

// ------------------------------------------------------------------------ side stream
// A library-owned stream (and a fork / join event pair) per device and
// caller stream: work that depends only on inputs ready at the fork runs
// there beside the caller's stream and is joined back before anything that
// needs it.  Under stream capture the fork and join become graph edges.
// WS_NF4_SIDE=0 keeps everything on the caller's stream.
namespace {
struct Side {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, fork2 = nullptr;
};
std::mutex g_side_mu;
std::map<std::pair<int, cudaStream_t>, Side> g_side;

bool side_enabled() {
  static const bool on = [] {
    const char* v = getenv("WS_NF4_SIDE");
    return !(v && v[0] == '0');
  }();
  return on;
}
// dA joins dB on the side stream once G is ready, and both run beside the
// input gradient's GEMM (joined after it: the GEMM's persistent CTAs take the
// SMs the short weight-gradient launches leave; 5% off the 32B step).
// WS_NF4_SIDE=1 joins them before the GEMM instead.
bool side_late() {
  static const bool on = [] {
    const char* v = getenv("WS_NF4_SIDE");
    return !(v && v[0] == '1');
  }();
  return on;
}

cudaError_t side_of(cudaStream_t st, Side* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_side_mu);
  Side& sd = g_side[std::make_pair(dev, st)];
  if (sd.s == nullptr) {
    e = cudaStreamCreateWithFlags(&sd.s, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sd.fork2, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      g_side.erase(std::make_pair(dev, st));
      return e;
    }
  }
  *out = sd;
  return cudaSuccess;
}
}  // namespace

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

// ------------------------------------------------------------------------ linears sharing x
// Workspace of a group (each piece 256-aligned):
//   ext     [ng][M][64] bf16   U split factors, contiguous (one TMA map)
//   skinny  ng x skinny_partial_bytes(M, K)
//   split   max over the grouped plan and the one-launch-per-linear plans
namespace {
struct GrpWs {
  size_t ext, skinny, skinny_each, split, total;
};
GrpWs grp_ws_layout(int64_t M, int ng, const int64_t* N, int64_t K) {
  GrpWs w{};
  size_t off = 0;
  w.ext = off;
  off += align256((size_t)ng * (size_t)M * 64 * 2);
  w.skinny = off;
  w.skinny_each = align256(skinny_partial_bytes(M, K));
  off += (size_t)ng * w.skinny_each;
  w.split = off;
  int64_t Nsum = 0;
  size_t sp = 0;
  for (int g = 0; g < ng; ++g) {
    Nsum += N[g];
    const size_t b = gemm_partial_bytes(plan_gemm(false, M, N[g], K), M, N[g]);
    if (b > sp) sp = b;
  }
  (void)Nsum;
  int64_t Npre = N[0];
  for (int g = 1; g < ng; ++g) {
    Npre += N[g];
    const size_t b = gemm_partial_bytes(plan_gemm(false, M, Npre, K), M, Npre);
    if (b > sp) sp = b;
  }
  off += align256(sp);
  w.total = off;
  return w;
}
}  // namespace

size_t linear_group_workspace_bytes(int64_t M, int ng, const int64_t* N, int64_t K) {
  return grp_ws_layout(M, ng, N, K).total;
}

// One LoRA-down launch for all ng linears (ng dropout masks of the same x;
// the bits are those of each linear's own key, U is summed in k-chunks sized
// for the whole launch, so it can differ in the last bits from a launch of
// that linear alone), then one GEMM over the concatenated output columns of
// the first ng_gemm linears and one GEMM per remaining linear.  A width that
// is not a multiple of the grouped plan's tile width falls back to one GEMM
// per linear.  y[g] == NULL skips linear g's GEMM (its U and bits are still
// produced), so a pass that needs only some outputs of a group reproduces
// them bit for bit; the grouped GEMM runs only if all its y are given.
cudaError_t linear_fwd_group(int ng, int ng_gemm, const NF4View* W, const uint16_t* x, const float* const* A,
                             const float* const* B, int64_t M, float scale, const DropKeyHost* keys,
                             uint16_t* const* y, float* const* U, uint32_t* const* mask, void* ws,
                             cudaStream_t st) {
  if (ng < 1 || ng > kMaxGroups || ng_gemm < 0 || ng_gemm > ng) return cudaErrorInvalidValue;
  const int64_t K = W[0].K;
  int64_t N[kMaxGroups];
  int64_t Nsum = 0;
  for (int g = 0; g < ng; ++g) {
    if (W[g].K != K) return cudaErrorInvalidValue;
    N[g] = W[g].N;
    Nsum += N[g];
  }
  const GrpWs L = grp_ws_layout(M, ng, N, K);
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint16_t* ext = reinterpret_cast<uint16_t*>(w + L.ext);
  float* split = reinterpret_cast<float*>(w + L.split);
  DropKey dk[kMaxGroups];
  uint16_t* exts[kMaxGroups];
  float* parts[kMaxGroups];
  uint8_t* mb[kMaxGroups];
  for (int g = 0; g < ng; ++g) {
    dk[g] = to_dev(keys[g]);
    exts[g] = ext + (size_t)g * (size_t)M * 64;
    parts[g] = reinterpret_cast<float*>(w + L.skinny + (size_t)g * L.skinny_each);
    mb[g] = reinterpret_cast<uint8_t*>(mask[g]);
  }
  cudaError_t e = run_skinny_tc_group(x, ng, A, M, K, dk, mb, parts, U, exts, st);
  if (e != cudaSuccess) return e;
  int first_single = 0;
  bool all_y = true, no_y = true;
  for (int g = 0; g < ng_gemm; ++g) {
    all_y = all_y && y[g] != nullptr;
    no_y = no_y && y[g] == nullptr;
  }
  if (ng_gemm > 1 && !all_y && !no_y) return cudaErrorInvalidValue;
  if (ng_gemm > 1 && no_y) first_single = ng_gemm;
  if (ng_gemm > 1 && all_y) {
    int64_t Ng = 0;
    for (int g = 0; g < ng_gemm; ++g) Ng += N[g];
    const GemmPlan p = plan_gemm(false, M, Ng, K);
    bool fits = true;
    for (int g = 0; g < ng_gemm; ++g) fits = fits && (N[g] % p.bn == 0);
    if (fits) {
      e = run_nf4_gemm_group(p, ng_gemm, W, x, M, ext, B, scale, y, split, st);
      if (e != cudaSuccess) return e;
      first_single = ng_gemm;
    }
  }
  for (int g = first_single; g < ng && e == cudaSuccess; ++g)
    if (y[g])
      e = run_nf4_gemm(plan_gemm(false, M, N[g], K), W[g], x, M, exts[g], B[g], scale, nullptr,
                       y[g], 0, 0, split, st);
  return e;
}

cudaError_t linear_bwd(const NF4View& W, const uint16_t* x, const float* A, const float* B,
                       int64_t M, float scale, const DropKeyHost& key, const float* U,
                       const uint32_t* mask, const uint16_t* dY, void* dX, int dX_f32,
                       int dX_accum, float* dA, float* dB, int grad_accum, void* ws,
                       cudaStream_t st) {
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
  // dB needs only U and dY: on the side stream it runs beside G; dA follows
  // it there once G is ready, and both overlap the input gradient's GEMM
  Side side;
  const bool use_side = dB != nullptr && side_enabled() && side_of(st, &side) == cudaSuccess;
  const bool late = use_side && side_late() && dX != nullptr;
  if (use_side) {
    e = cudaEventRecord(side.fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side.s, side.fork, 0);
    if (e == cudaSuccess) e = run_wgrad_tc(U, dY, nullptr, M, W.N, scale, dB, 0, grad_accum, wg, side.s);
    if (e == cudaSuccess && !late) e = cudaEventRecord(side.join, side.s);
    if (e != cudaSuccess) return e;
  }
  e = run_lora_G(dY, B, M, W.N, G, Gext, reinterpret_cast<float*>(w + L.skinny), st);
  if (e == cudaSuccess && dB && !use_side)
    e = run_wgrad_tc(U, dY, nullptr, M, W.N, scale, dB, 0, grad_accum, wg, st);
  if (e == cudaSuccess && dA) {
    if (late) {
      // dA needs G: the side stream waits for it, then runs beside the GEMM
      e = cudaEventRecord(side.fork2, st);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(side.s, side.fork2, 0);
      if (e == cudaSuccess) e = run_wgrad_tc(G, x, mask, M, W.K, scale, dA, 1, grad_accum, wg, side.s);
    } else {
      e = run_wgrad_tc(G, x, mask, M, W.K, scale, dA, 1, grad_accum, wg, st);
    }
  }
  // join even after an error, so a capture is never left with an unjoined stream
  if (use_side && !late) {
    const cudaError_t ej = cudaStreamWaitEvent(st, side.join, 0);
    if (e == cudaSuccess) e = ej;
  }
  if (e == cudaSuccess && dX) {
    const GemmPlan p = plan_gemm(true, M, W.K, W.N);
    e = run_nf4_gemm(p, W, dY, M, Gext, A, scale, mask, dX, dX_f32, dX_accum,
                     reinterpret_cast<float*>(w + L.split), st);
  }
  if (late) {
    cudaError_t ej = cudaEventRecord(side.join, side.s);
    if (ej == cudaSuccess) ej = cudaStreamWaitEvent(st, side.join, 0);
    if (e == cudaSuccess) e = ej;
  }
  return e;
}

// ------------------------------------------------------------------------ linears sharing x (backward)
// Per linear: Gext [M,64] bf16, G [M,16] fp32, mask [M,K/32] (when the
// caller kept none), skinny partials; then the split partials of one
// input-gradient plan (all linears have the same shape).
namespace {
struct BwdGrpWs {
  size_t ext, G, mask, skinny, per, split, total;
};
BwdGrpWs bwd_grp_ws_layout(int64_t M, int ng, int64_t N, int64_t K) {
  BwdGrpWs w{};
  w.ext = 0;
  w.G = align256((size_t)M * 64 * 2);
  w.mask = w.G + align256((size_t)M * 16 * 4);
  w.skinny = w.mask + align256((size_t)M * (size_t)(K / 32) * 4);
  w.per = w.skinny + align256(skinny_partial_bytes(M, N));
  w.split = (size_t)ng * w.per;
  w.total = w.split + align256(gemm_partial_bytes(plan_gemm(true, M, K, N), M, K));
  return w;
}
}  // namespace

size_t linear_bwd_group_workspace_bytes(int64_t M, int ng, int64_t N, int64_t K) {
  return bwd_grp_ws_layout(M, ng, N, K).total;
}

// ng linears of the same shape reading the same x, each with its own dY:
// the G products in one launch, the dA weight gradients in one launch, the
// dB weight gradients in one launch on the side stream, then the input
// gradients one GEMM after the other into dX (the first one written, or
// added when dX_accum, the others added).  Each result equals the one-linear
// backward's bit for bit.
cudaError_t linear_bwd_group(int ng, const NF4View* W, const uint16_t* x, const float* const* A,
                             const float* const* B, int64_t M, float scale, const DropKeyHost* keys,
                             const float* const* U, const uint32_t* const* mask,
                             const uint16_t* const* dY, void* dX, int dX_f32, int dX_accum,
                             float* const* dA, float* const* dB, int grad_accum, void* ws,
                             cudaStream_t st) {
  if (ng < 1 || ng > kMaxGroups) return cudaErrorInvalidValue;
  const int64_t N = W[0].N, K = W[0].K;
  bool any_dA = false, any_dB = false;
  for (int g = 0; g < ng; ++g) {
    if (W[g].N != N || W[g].K != K) return cudaErrorInvalidValue;
    any_dA = any_dA || dA[g] != nullptr;
    any_dB = any_dB || dB[g] != nullptr;
  }
  for (int g = 0; g < ng; ++g)
    if ((dA[g] != nullptr) != any_dA || (dB[g] != nullptr) != any_dB) return cudaErrorInvalidValue;
  const BwdGrpWs L = bwd_grp_ws_layout(M, ng, N, K);
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint16_t* Gext[kMaxGroups];
  float* G[kMaxGroups];
  float* part[kMaxGroups];
  const uint32_t* mk[kMaxGroups];
  cudaError_t e = cudaSuccess;
  for (int g = 0; g < ng && e == cudaSuccess; ++g) {
    uint8_t* base = w + (size_t)g * L.per;
    Gext[g] = reinterpret_cast<uint16_t*>(base + L.ext);
    G[g] = reinterpret_cast<float*>(base + L.G);
    part[g] = reinterpret_cast<float*>(base + L.skinny);
    mk[g] = mask[g];
    if (mk[g] == nullptr) {
      uint32_t* m = reinterpret_cast<uint32_t*>(base + L.mask);
      e = run_mask_gen(M, K, keys[g], m, st);
      mk[g] = m;
    }
  }
  if (e != cudaSuccess) return e;
  Side side;
  const bool use_side = any_dB && side_enabled() && side_of(st, &side) == cudaSuccess;
  const bool late = use_side && side_late() && dX != nullptr;
  if (use_side) {
    e = cudaEventRecord(side.fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side.s, side.fork, 0);
    if (e == cudaSuccess) e = run_wgrad_tc_group(ng, U, dY, nullptr, M, N, scale, dB, 0, grad_accum, side.s);
    if (e == cudaSuccess && !late) e = cudaEventRecord(side.join, side.s);
    if (e != cudaSuccess) return e;
  }
  e = run_skinny_G_group(ng, dY, B, M, N, part, G, Gext, st);
  if (e == cudaSuccess && any_dB && !use_side)
    e = run_wgrad_tc_group(ng, U, dY, nullptr, M, N, scale, dB, 0, grad_accum, st);
  if (e == cudaSuccess && any_dA) {
    const float* Gc[kMaxGroups];
    const uint16_t* xs[kMaxGroups];
    for (int g = 0; g < ng; ++g) {
      Gc[g] = G[g];
      xs[g] = x;
    }
    if (late) {
      e = cudaEventRecord(side.fork2, st);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(side.s, side.fork2, 0);
      if (e == cudaSuccess) e = run_wgrad_tc_group(ng, Gc, xs, mk, M, K, scale, dA, 1, grad_accum, side.s);
    } else {
      e = run_wgrad_tc_group(ng, Gc, xs, mk, M, K, scale, dA, 1, grad_accum, st);
    }
  }
  if (use_side && !late) {
    const cudaError_t ej = cudaStreamWaitEvent(st, side.join, 0);
    if (e == cudaSuccess) e = ej;
  }
  if (e == cudaSuccess && dX != nullptr) {
    const GemmPlan p = plan_gemm(true, M, K, N);
    for (int g = 0; g < ng && e == cudaSuccess; ++g)
      e = run_nf4_gemm(p, W[g], dY[g], M, Gext[g], A[g], scale, mk[g], dX, dX_f32,
                       g > 0 ? 1 : dX_accum, reinterpret_cast<float*>(w + L.split), st);
  }
  if (late) {
    cudaError_t ej = cudaEventRecord(side.join, side.s);
    if (ej == cudaSuccess) ej = cudaStreamWaitEvent(st, side.join, 0);
    if (e == cudaSuccess) e = ej;
  }
  return e;
}

}  // namespace ws
