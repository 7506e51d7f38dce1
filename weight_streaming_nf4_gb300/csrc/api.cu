// api.cu -- the C ABI of libwsnf4.so (declared in include/wsnf4.h):
// argument validation, dispatch to the kernels, the pinned-host -> HBM block
// copy, and the host-side engine of one streamed or resident training step.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <new>

#include "common.cuh"
#include "kernels.h"

using namespace ws;

namespace {
std::atomic<uint64_t> g_launches{0};
}  // namespace

void ws::note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ws_status cuda_status(cudaError_t e) { return e == cudaSuccess ? WS_OK : WS_ERR_CUDA; }

ws_status check_linear(const ws_nf4* W, ws_lora_shape sh, const ws_dropout_key& key) {
  if (!W || !W->codes || !W->absmax) return WS_ERR_INVALID;
  if (sh.M < 1 || sh.N < 64 || sh.K < 64) return WS_ERR_SHAPE;
  if (sh.N % 64 || sh.K % 64) return WS_ERR_SHAPE;
  if (W->N != sh.N || W->K != sh.K) return WS_ERR_SHAPE;
  if (sh.r != 16) return WS_ERR_SHAPE;
  if ((double)sh.M * (double)sh.K >= 17179869184.0) return WS_ERR_SHAPE;  // 2^34
  if (sh.N > (int64_t)1 << 30 || sh.K > (int64_t)1 << 30 || sh.M > (int64_t)1 << 30)
    return WS_ERR_SHAPE;
  if (!(key.p >= 0.0 && key.p < 1.0)) return WS_ERR_INVALID;
  if (key.linear > 255u || key.microbatch > 0xFFFFFFu) return WS_ERR_INVALID;
  if (!aligned16(W->codes) || !aligned16(W->absmax)) return WS_ERR_ALIGN;
  return WS_OK;
}

NF4View view_of(const ws_nf4* W) {
  NF4View v;
  v.codes = W->codes;
  v.absmax = W->absmax;
  v.wbf16 = nullptr;
  v.N = W->N;
  v.K = W->K;
  return v;
}

float lora_scale(ws_lora_shape sh, double p) {
  return (float)(((double)sh.alpha / (double)sh.r) / (1.0 - p));
}

}  // namespace

extern "C" {

const char* ws_status_string(ws_status st) {
  switch (st) {
    case WS_OK: return "WS_OK";
    case WS_ERR_INVALID: return "WS_ERR_INVALID: invalid argument";
    case WS_ERR_SHAPE: return "WS_ERR_SHAPE: shape outside the supported contract";
    case WS_ERR_ALIGN: return "WS_ERR_ALIGN: pointer not 16-byte aligned";
    case WS_ERR_CUDA: return "WS_ERR_CUDA: CUDA call or kernel launch failed";
    case WS_ERR_TIMEOUT: return "WS_ERR_TIMEOUT: a bounded device wait gave up";
    case WS_ERR_OOM: return "WS_ERR_OOM: buffer or workspace too small";
    case WS_ERR_UNSUPPORTED: return "WS_ERR_UNSUPPORTED: configuration would break exactness";
    case WS_ERR_NOT_PINNED: return "WS_ERR_NOT_PINNED: host buffer is not page-locked";
    default: return "WS_ERR_UNKNOWN";
  }
}

uint64_t ws_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

ws_status ws_device_error(uint32_t* flags) {
  if (!flags) return WS_ERR_INVALID;
  *flags = 0;
  const cudaError_t e = read_and_clear_dev_error(flags);
  if (e != cudaSuccess) return WS_ERR_CUDA;
  return *flags ? WS_ERR_TIMEOUT : WS_OK;
}

ws_status ws_selfcheck_bounded_wait(uint32_t limit_us, ws_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000u) return WS_ERR_INVALID;
  return cuda_status(run_wait_selfcheck(limit_us, (cudaStream_t)stream));
}

ws_status ws_quantize_nf4(const uint16_t* W, int64_t N, int64_t K, uint8_t* codes, float* absmax,
                          ws_stream_t stream) {
  if (!W || !codes || !absmax) return WS_ERR_INVALID;
  if (N < 1 || K < 64 || K % 64) return WS_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(codes) || !aligned16(absmax)) return WS_ERR_ALIGN;
  return cuda_status(run_quantize_nf4(W, N, K, codes, absmax, (cudaStream_t)stream));
}

namespace {
ws_status attn_check(int32_t n_seq, int32_t seq_len, int32_t nh, int32_t nkv, int32_t hd) {
  if (n_seq < 1 || seq_len < 1 || nh < 1 || nkv < 1) return WS_ERR_SHAPE;
  if (hd != 64 && hd != 128) return WS_ERR_SHAPE;
  if (nh % nkv) return WS_ERR_SHAPE;
  if ((int64_t)n_seq * seq_len >= (1ll << 31)) return WS_ERR_SHAPE;
  return WS_OK;
}
}  // namespace

ws_status ws_attention_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           int32_t n_seq, int32_t seq_len, int32_t n_heads, int32_t n_kv_heads,
                           int32_t head_dim, uint16_t* o, float* o32, float* lse,
                           ws_stream_t stream) {
  if (!q || !k || !v || !o || !lse) return WS_ERR_INVALID;
  const ws_status c = attn_check(n_seq, seq_len, n_heads, n_kv_heads, head_dim);
  if (c != WS_OK) return c;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      (o32 && !aligned16(o32)))
    return WS_ERR_ALIGN;
  return cuda_status(run_attn_fwd(q, k, v, n_seq, seq_len, n_heads, n_kv_heads, head_dim, o, o32,
                                  lse, (cudaStream_t)stream));
}

ws_status ws_attention_workspace_size(int64_t M, int32_t n_heads, int32_t head_dim,
                                      size_t* bytes) {
  if (!bytes) return WS_ERR_INVALID;
  if (M < 1 || n_heads < 1 || (head_dim != 64 && head_dim != 128)) return WS_ERR_SHAPE;
  *bytes = attn_bwd_workspace_bytes(M, n_heads, head_dim);
  return WS_OK;
}

ws_status ws_attention_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           const float* o32, const float* lse, const uint16_t* dO,
                           int32_t n_seq, int32_t seq_len, int32_t n_heads, int32_t n_kv_heads,
                           int32_t head_dim, uint16_t* dq, uint16_t* dk, uint16_t* dv,
                           void* workspace, size_t workspace_bytes, ws_stream_t stream) {
  if (!q || !k || !v || !o32 || !lse || !dO || !dq || !dk || !dv || !workspace)
    return WS_ERR_INVALID;
  const ws_status c = attn_check(n_seq, seq_len, n_heads, n_kv_heads, head_dim);
  if (c != WS_OK) return c;
  const int64_t M = (int64_t)n_seq * seq_len;
  if (workspace_bytes < attn_bwd_workspace_bytes(M, n_heads, head_dim)) return WS_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o32) || !aligned16(lse) ||
      !aligned16(dO) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      !aligned16(workspace))
    return WS_ERR_ALIGN;
  return cuda_status(run_attn_bwd(q, k, v, o32, lse, dO, n_seq, seq_len, n_heads, n_kv_heads,
                                  head_dim, dq, dk, dv, workspace, (cudaStream_t)stream));
}

ws_status ws_lora_workspace_size(ws_lora_shape sh, size_t* bytes) {
  if (!bytes) return WS_ERR_INVALID;
  if (sh.M < 1 || sh.N < 64 || sh.K < 64 || sh.N % 64 || sh.K % 64 || sh.r != 16)
    return WS_ERR_SHAPE;
  *bytes = linear_workspace_bytes(sh.M, sh.N, sh.K);
  return WS_OK;
}

ws_status ws_lora_linear_fwd(const ws_nf4* W, const uint16_t* x, const float* A, const float* B,
                             ws_lora_shape sh, ws_dropout_key key, uint16_t* y, float* U_saved,
                             uint32_t* mask_saved, void* workspace, size_t ws_bytes,
                             ws_stream_t stream) {
  ws_status s = check_linear(W, sh, key);
  if (s != WS_OK) return s;
  if (!x || !A || !B || !y || !U_saved || !workspace) return WS_ERR_INVALID;
  if (!aligned16(x) || !aligned16(A) || !aligned16(B) || !aligned16(y) || !aligned16(U_saved) ||
      !aligned16(workspace) || (mask_saved && !aligned16(mask_saved)))
    return WS_ERR_ALIGN;
  if (ws_bytes < linear_workspace_bytes(sh.M, sh.N, sh.K)) return WS_ERR_OOM;
  return cuda_status(linear_fwd(view_of(W), x, A, B, sh.M, lora_scale(sh, key.p),
                                make_drop_key(key), y, U_saved, mask_saved, workspace,
                                (cudaStream_t)stream));
}

ws_status ws_lora_linear_bwd(const ws_nf4* W, const uint16_t* x, const float* A, const float* B,
                             ws_lora_shape sh, ws_dropout_key key, const float* U_saved,
                             const uint32_t* mask_saved, const uint16_t* dY, void* dX,
                             int32_t dX_dtype, int32_t accumulate, float* dA, float* dB,
                             void* workspace, size_t ws_bytes, ws_stream_t stream) {
  ws_status s = check_linear(W, sh, key);
  if (s != WS_OK) return s;
  if (!x || !A || !B || !U_saved || !dY || !dX || !dA || !dB || !workspace) return WS_ERR_INVALID;
  if (dX_dtype != WS_DTYPE_BF16 && dX_dtype != WS_DTYPE_F32) return WS_ERR_INVALID;
  if (accumulate & ~(WS_ACC_DX | WS_ACC_GRADS)) return WS_ERR_INVALID;
  const int dX_accumulate = (accumulate & WS_ACC_DX) ? 1 : 0;
  if (dX_accumulate && dX_dtype != WS_DTYPE_F32) return WS_ERR_INVALID;
  if (!aligned16(x) || !aligned16(A) || !aligned16(B) || !aligned16(U_saved) || !aligned16(dY) ||
      !aligned16(dX) || !aligned16(dA) || !aligned16(dB) || !aligned16(workspace) ||
      (mask_saved && !aligned16(mask_saved)))
    return WS_ERR_ALIGN;
  if (ws_bytes < linear_workspace_bytes(sh.M, sh.N, sh.K)) return WS_ERR_OOM;
  return cuda_status(linear_bwd(view_of(W), x, A, B, sh.M, lora_scale(sh, key.p),
                                make_drop_key(key), U_saved, mask_saved, dY, dX,
                                dX_dtype == WS_DTYPE_F32 ? 1 : 0, dX_accumulate, dA, dB,
                                (accumulate & WS_ACC_GRADS) ? 1 : 0, workspace,
                                (cudaStream_t)stream));
}

ws_status ws_lora_group_workspace_size(int32_t ng, const int64_t* N, int64_t M, int64_t K,
                                       size_t* bytes) {
  if (!bytes || !N) return WS_ERR_INVALID;
  if (ng < 1 || ng > kMaxGroups || M < 1 || K < 64 || K % 64) return WS_ERR_SHAPE;
  bool same = true;
  for (int g = 0; g < ng; ++g) {
    if (N[g] < 64 || N[g] % 64) return WS_ERR_SHAPE;
    same = same && N[g] == N[0];
  }
  size_t b = linear_group_workspace_bytes(M, ng, N, K);
  if (same) {
    const size_t bb = linear_bwd_group_workspace_bytes(M, ng, N[0], K);
    if (bb > b) b = bb;
  }
  *bytes = b;
  return WS_OK;
}

ws_status ws_lora_linear_fwd_group(int32_t ng, const ws_nf4* W, const uint16_t* x,
                                   const float* const* A, const float* const* B, ws_lora_shape sh,
                                   const ws_dropout_key* keys, uint16_t* const* y,
                                   float* const* U_saved, uint32_t* const* mask_saved,
                                   void* workspace, size_t ws_bytes, ws_stream_t stream) {
  if (ng < 1 || ng > kMaxGroups || !W || !A || !B || !keys || !y || !U_saved || !x || !workspace)
    return WS_ERR_INVALID;
  NF4View v[kMaxGroups];
  DropKeyHost k[kMaxGroups];
  int64_t N[kMaxGroups];
  uint32_t* mk[kMaxGroups];
  float scale = 0.0f;
  for (int g = 0; g < ng; ++g) {
    ws_lora_shape sg = sh;
    sg.N = W[g].N;
    const ws_status s = check_linear(&W[g], sg, keys[g]);
    if (s != WS_OK) return s;
    if (W[g].K != sh.K) return WS_ERR_SHAPE;
    if (keys[g].p != keys[0].p) return WS_ERR_INVALID;
    if (!A[g] || !B[g] || !y[g] || !U_saved[g]) return WS_ERR_INVALID;
    if (!aligned16(A[g]) || !aligned16(B[g]) || !aligned16(y[g]) || !aligned16(U_saved[g]) ||
        (mask_saved && mask_saved[g] && !aligned16(mask_saved[g])))
      return WS_ERR_ALIGN;
    v[g] = view_of(&W[g]);
    k[g] = make_drop_key(keys[g]);
    N[g] = W[g].N;
    mk[g] = mask_saved ? mask_saved[g] : nullptr;
    scale = lora_scale(sg, keys[g].p);
  }
  if (!aligned16(x) || !aligned16(workspace)) return WS_ERR_ALIGN;
  if (ws_bytes < linear_group_workspace_bytes(sh.M, ng, N, sh.K)) return WS_ERR_OOM;
  return cuda_status(linear_fwd_group(ng, ng, v, x, A, B, sh.M, scale, k, y, U_saved, mk,
                                      workspace, (cudaStream_t)stream));
}

ws_status ws_lora_linear_bwd_group(int32_t ng, const ws_nf4* W, const uint16_t* x,
                                   const float* const* A, const float* const* B, ws_lora_shape sh,
                                   const ws_dropout_key* keys, const float* const* U_saved,
                                   const uint32_t* const* mask_saved, const uint16_t* const* dY,
                                   void* dX, int32_t dX_dtype, int32_t accumulate,
                                   float* const* dA, float* const* dB, void* workspace,
                                   size_t ws_bytes, ws_stream_t stream) {
  if (ng < 1 || ng > kMaxGroups || !W || !A || !B || !keys || !U_saved || !dY || !dX || !dA ||
      !dB || !x || !workspace)
    return WS_ERR_INVALID;
  if (dX_dtype != WS_DTYPE_BF16 && dX_dtype != WS_DTYPE_F32) return WS_ERR_INVALID;
  if (accumulate & ~(WS_ACC_DX | WS_ACC_GRADS)) return WS_ERR_INVALID;
  const int dX_accumulate = (accumulate & WS_ACC_DX) ? 1 : 0;
  // the sum over linears is taken in fp32
  if ((dX_accumulate || ng > 1) && dX_dtype != WS_DTYPE_F32) return WS_ERR_INVALID;
  NF4View v[kMaxGroups];
  DropKeyHost k[kMaxGroups];
  const uint32_t* mk[kMaxGroups];
  float scale = 0.0f;
  for (int g = 0; g < ng; ++g) {
    ws_lora_shape sg = sh;
    sg.N = W[0].N;
    const ws_status s = check_linear(&W[g], sg, keys[g]);
    if (s != WS_OK) return s;
    if (W[g].K != sh.K) return WS_ERR_SHAPE;
    if (keys[g].p != keys[0].p) return WS_ERR_INVALID;
    if (!A[g] || !B[g] || !U_saved[g] || !dY[g] || !dA[g] || !dB[g]) return WS_ERR_INVALID;
    if (!aligned16(A[g]) || !aligned16(B[g]) || !aligned16(U_saved[g]) || !aligned16(dY[g]) ||
        !aligned16(dA[g]) || !aligned16(dB[g]) ||
        (mask_saved && mask_saved[g] && !aligned16(mask_saved[g])))
      return WS_ERR_ALIGN;
    v[g] = view_of(&W[g]);
    k[g] = make_drop_key(keys[g]);
    mk[g] = mask_saved ? mask_saved[g] : nullptr;
    scale = lora_scale(sg, keys[g].p);
  }
  if (!aligned16(x) || !aligned16(dX) || !aligned16(workspace)) return WS_ERR_ALIGN;
  if (ws_bytes < linear_bwd_group_workspace_bytes(sh.M, ng, W[0].N, sh.K)) return WS_ERR_OOM;
  return cuda_status(linear_bwd_group(ng, v, x, A, B, sh.M, scale, k, U_saved, mk, dY, dX,
                                      dX_dtype == WS_DTYPE_F32 ? 1 : 0, dX_accumulate, dA, dB,
                                      (accumulate & WS_ACC_GRADS) ? 1 : 0, workspace,
                                      (cudaStream_t)stream));
}

namespace {
ws_status check_bf16(const ws_bf16* W, ws_lora_shape sh, const ws_dropout_key& key, ws_nf4* as) {
  if (!W || !W->w) return WS_ERR_INVALID;
  // the shape and key checks of the NF4 path, with the bf16 pointer standing in
  *as = ws_nf4{reinterpret_cast<const uint8_t*>(W->w), reinterpret_cast<const float*>(W->w), W->N,
               W->K};
  return check_linear(as, sh, key);
}
NF4View view_of_bf16(const ws_bf16* W) {
  NF4View v;
  v.codes = nullptr;
  v.absmax = nullptr;
  v.wbf16 = W->w;
  v.N = W->N;
  v.K = W->K;
  return v;
}
}  // namespace

ws_status ws_lora_linear_fwd_bf16(const ws_bf16* W, const uint16_t* x, const float* A,
                                  const float* B, ws_lora_shape sh, ws_dropout_key key,
                                  uint16_t* y, float* U_saved, uint32_t* mask_saved,
                                  void* workspace, size_t ws_bytes, ws_stream_t stream) {
  ws_nf4 as;
  ws_status s = check_bf16(W, sh, key, &as);
  if (s != WS_OK) return s;
  if (!x || !A || !B || !y || !U_saved || !workspace) return WS_ERR_INVALID;
  if (!aligned16(x) || !aligned16(A) || !aligned16(B) || !aligned16(y) || !aligned16(U_saved) ||
      !aligned16(workspace) || (mask_saved && !aligned16(mask_saved)))
    return WS_ERR_ALIGN;
  if (ws_bytes < linear_workspace_bytes(sh.M, sh.N, sh.K)) return WS_ERR_OOM;
  return cuda_status(linear_fwd(view_of_bf16(W), x, A, B, sh.M, lora_scale(sh, key.p),
                                make_drop_key(key), y, U_saved, mask_saved, workspace,
                                (cudaStream_t)stream));
}

ws_status ws_lora_linear_bwd_bf16(const ws_bf16* W, const uint16_t* x, const float* A,
                                  const float* B, ws_lora_shape sh, ws_dropout_key key,
                                  const float* U_saved, const uint32_t* mask_saved,
                                  const uint16_t* dY, void* dX, int32_t dX_dtype,
                                  int32_t accumulate, float* dA, float* dB, void* workspace,
                                  size_t ws_bytes, ws_stream_t stream) {
  ws_nf4 as;
  ws_status s = check_bf16(W, sh, key, &as);
  if (s != WS_OK) return s;
  if (!x || !A || !B || !U_saved || !dY || !dX || !dA || !dB || !workspace) return WS_ERR_INVALID;
  if (dX_dtype != WS_DTYPE_BF16 && dX_dtype != WS_DTYPE_F32) return WS_ERR_INVALID;
  if (accumulate & ~(WS_ACC_DX | WS_ACC_GRADS)) return WS_ERR_INVALID;
  const int dX_accumulate = (accumulate & WS_ACC_DX) ? 1 : 0;
  if (dX_accumulate && dX_dtype != WS_DTYPE_F32) return WS_ERR_INVALID;
  if (!aligned16(x) || !aligned16(A) || !aligned16(B) || !aligned16(U_saved) || !aligned16(dY) ||
      !aligned16(dX) || !aligned16(dA) || !aligned16(dB) || !aligned16(workspace) ||
      (mask_saved && !aligned16(mask_saved)))
    return WS_ERR_ALIGN;
  if (ws_bytes < linear_workspace_bytes(sh.M, sh.N, sh.K)) return WS_ERR_OOM;
  return cuda_status(linear_bwd(view_of_bf16(W), x, A, B, sh.M, lora_scale(sh, key.p),
                                make_drop_key(key), U_saved, mask_saved, dY, dX,
                                dX_dtype == WS_DTYPE_F32 ? 1 : 0, dX_accumulate, dA, dB,
                                (accumulate & WS_ACC_GRADS) ? 1 : 0, workspace,
                                (cudaStream_t)stream));
}

ws_status ws_nf4_matmul_workspace_size(int64_t M, int64_t N, int64_t K, int32_t transpose_w,
                                       size_t* bytes) {
  if (!bytes) return WS_ERR_INVALID;
  if (M < 1 || N < 64 || K < 64 || N % 64 || K % 64) return WS_ERR_SHAPE;
  const GemmPlan p = transpose_w ? plan_gemm(true, M, K, N) : plan_gemm(false, M, N, K);
  *bytes = gemm_partial_bytes(p, M, transpose_w ? K : N);
  if (*bytes == 0) *bytes = 256;
  return WS_OK;
}

ws_status ws_nf4_matmul(const ws_nf4* W, const uint16_t* act, int64_t M, int32_t transpose_w,
                        void* out, int32_t out_dtype, void* workspace, size_t ws_bytes,
                        ws_stream_t stream) {
  if (!W || !W->codes || !W->absmax || !act || !out || !workspace) return WS_ERR_INVALID;
  if (out_dtype != WS_DTYPE_BF16 && out_dtype != WS_DTYPE_F32) return WS_ERR_INVALID;
  if (M < 1 || W->N < 64 || W->K < 64 || W->N % 64 || W->K % 64) return WS_ERR_SHAPE;
  if (M > (int64_t)1 << 30 || W->N > (int64_t)1 << 30 || W->K > (int64_t)1 << 30)
    return WS_ERR_SHAPE;
  if (!aligned16(W->codes) || !aligned16(W->absmax) || !aligned16(act) || !aligned16(out) ||
      !aligned16(workspace))
    return WS_ERR_ALIGN;
  size_t need = 0;
  ws_nf4_matmul_workspace_size(M, W->N, W->K, transpose_w, &need);
  if (ws_bytes < need) return WS_ERR_OOM;
  const bool bwd = transpose_w != 0;
  const GemmPlan p = bwd ? plan_gemm(true, M, W->K, W->N) : plan_gemm(false, M, W->N, W->K);
  return cuda_status(run_nf4_gemm(p, view_of(W), act, M, nullptr, nullptr, 0.0f, nullptr, out,
                                  out_dtype == WS_DTYPE_F32 ? 1 : 0, 0,
                                  static_cast<float*>(workspace), (cudaStream_t)stream));
}

ws_status ws_nf4_matmul_noalloc(const ws_nf4* W, const uint16_t* act, int64_t M,
                                int32_t transpose_w, void* out, int32_t out_dtype,
                                ws_stream_t stream) {
  if (!W || !W->codes || !W->absmax || !act || !out) return WS_ERR_INVALID;
  if (out_dtype != WS_DTYPE_BF16 && out_dtype != WS_DTYPE_F32) return WS_ERR_INVALID;
  if (M < 1 || W->N < 64 || W->K < 64 || W->N % 64 || W->K % 64) return WS_ERR_SHAPE;
  if (M > (int64_t)1 << 30 || W->N > (int64_t)1 << 30 || W->K > (int64_t)1 << 30)
    return WS_ERR_SHAPE;
  if (!aligned16(W->codes) || !aligned16(W->absmax) || !aligned16(act) || !aligned16(out))
    return WS_ERR_ALIGN;
  const bool bwd = transpose_w != 0;
  const GemmPlan p = bwd ? plan_gemm(true, M, W->K, W->N) : plan_gemm(false, M, W->N, W->K);
  const size_t need = gemm_partial_bytes(p, M, bwd ? W->K : W->N);
  float* scratch = nullptr;
  size_t have = 0;
  if (noalloc_scratch(&scratch, &have) != cudaSuccess) return WS_ERR_CUDA;
  if (need > have) return WS_ERR_OOM;
  return cuda_status(run_nf4_gemm(p, view_of(W), act, M, nullptr, nullptr, 0.0f, nullptr, out,
                                  out_dtype == WS_DTYPE_F32 ? 1 : 0, 0, scratch,
                                  (cudaStream_t)stream));
}

ws_status ws_stack_sizes(const ws_stack_cfg* cfg, int32_t block_layers, size_t* block_weight_bytes,
                         int64_t* n_params, size_t* saved_bytes_layer, size_t* workspace_bytes) {
  ws_status s = stack_check(cfg);
  if (s != WS_OK) return s;
  if (block_layers < 1 || block_layers > cfg->n_layers) return WS_ERR_SHAPE;
  if (block_weight_bytes) *block_weight_bytes = stack_block_bytes(*cfg, block_layers);
  if (n_params) *n_params = stack_n_params(*cfg);
  if (saved_bytes_layer) *saved_bytes_layer = stack_saved_layer(*cfg);
  if (workspace_bytes) *workspace_bytes = stack_ws_bytes(*cfg, block_layers);
  return WS_OK;
}

ws_status ws_stack_weight_offset(const ws_stack_cfg* cfg, int32_t layer_in_block, int32_t lin,
                                 size_t* off_codes, size_t* off_absmax) {
  ws_status s = stack_check(cfg);
  if (s != WS_OK) return s;
  if (!off_codes || !off_absmax || lin < 0 || lin >= WS_NLIN || layer_in_block < 0)
    return WS_ERR_INVALID;
  stack_weight_offset(*cfg, layer_in_block, lin, off_codes, off_absmax);
  return WS_OK;
}

ws_status ws_stack_saved_offset(const ws_stack_cfg* cfg, int32_t field, int32_t lin,
                                size_t* offset) {
  ws_status s = stack_check(cfg);
  if (s != WS_OK) return s;
  if (!offset) return WS_ERR_INVALID;
  return stack_saved_offset(*cfg, field, lin, offset) ? WS_OK : WS_ERR_INVALID;
}

ws_status ws_stack_loader_staging_bytes(const ws_stack_cfg* cfg, size_t* bytes) {
  ws_status s = stack_check(cfg);
  if (s != WS_OK) return s;
  if (!bytes) return WS_ERR_INVALID;
  const int64_t N[WS_NLIN] = {cfg->H, cfg->KV, cfg->KV, cfg->H, cfg->I, cfg->I, cfg->H};
  const int64_t K[WS_NLIN] = {cfg->H, cfg->H, cfg->H, cfg->H, cfg->H, cfg->H, cfg->I};
  size_t mx = 0;
  for (int i = 0; i < WS_NLIN; ++i) {
    // codes, then the block scales 256 bytes further on
    const size_t b = (((size_t)N[i] * (size_t)(K[i] / 2) + 255) & ~(size_t)255) +
                     (size_t)(K[i] / 64) * (size_t)N[i] * 4;
    if (b > mx) mx = b;
  }
  *bytes = mx;
  return WS_OK;
}

ws_status ws_stack_put_weight(const ws_stack_cfg* cfg, int32_t block_layers, int32_t layer,
                              int32_t lin, const uint16_t* W, int64_t N, int64_t K, void* image,
                              void* staging, size_t staging_bytes, ws_stream_t stream) {
  ws_status s = stack_check(cfg);
  if (s != WS_OK) return s;
  if (!W || !image) return WS_ERR_INVALID;
  if (block_layers < 1 || cfg->n_layers % block_layers) return WS_ERR_SHAPE;
  if (layer < 0 || layer >= cfg->n_layers || lin < 0 || lin >= WS_NLIN) return WS_ERR_INVALID;
  const int64_t Ns[WS_NLIN] = {cfg->H, cfg->KV, cfg->KV, cfg->H, cfg->I, cfg->I, cfg->H};
  const int64_t Ks[WS_NLIN] = {cfg->H, cfg->H, cfg->H, cfg->H, cfg->H, cfg->H, cfg->I};
  if (N != Ns[lin] || K != Ks[lin]) return WS_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(image)) return WS_ERR_ALIGN;
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, image) != cudaSuccess) {
    cudaGetLastError();
    return WS_ERR_NOT_PINNED;
  }
  const bool host = attr.type == cudaMemoryTypeHost;
  if (!host && attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
    return WS_ERR_NOT_PINNED;
  size_t oc = 0, oa = 0;
  const int blk = layer / block_layers, lib = layer % block_layers;
  stack_weight_offset(*cfg, lib, lin, &oc, &oa);
  const size_t base = (size_t)blk * stack_block_bytes(*cfg, block_layers);
  uint8_t* img = static_cast<uint8_t*>(image) + base;
  const cudaStream_t st = (cudaStream_t)stream;
  if (cfg->base == WS_BASE_BF16)
    return cuda_status(cudaMemcpyAsync(img + oc, W, (size_t)N * (size_t)K * 2, cudaMemcpyDefault, st));
  const size_t code_bytes = (size_t)N * (size_t)(K / 2);
  const size_t scale_bytes = (size_t)(K / 64) * (size_t)N * 4;
  if (!host)
    return cuda_status(run_quantize_nf4(W, N, K, img + oc, reinterpret_cast<float*>(img + oa), st));
  size_t need = 0;
  ws_stack_loader_staging_bytes(cfg, &need);
  if (!staging) return WS_ERR_INVALID;
  if (!aligned16(staging)) return WS_ERR_ALIGN;
  if (staging_bytes < need) return WS_ERR_OOM;
  uint8_t* sg = static_cast<uint8_t*>(staging);
  const size_t sa = (code_bytes + 255) & ~(size_t)255;
  cudaError_t e = run_quantize_nf4(W, N, K, sg, reinterpret_cast<float*>(sg + sa), st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(img + oc, sg, code_bytes, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(img + oa, sg + sa, scale_bytes, cudaMemcpyDeviceToHost, st);
  return cuda_status(e);
}

ws_status ws_stack_workspace_offset(const ws_stack_cfg* cfg, int32_t block_layers, int32_t field,
                                   size_t* offset) {
  ws_status s = stack_check(cfg);
  if (s != WS_OK) return s;
  if (!offset || block_layers < 1 || block_layers > cfg->n_layers) return WS_ERR_INVALID;
  return stack_ws_offset(*cfg, block_layers, field, offset) ? WS_OK : WS_ERR_INVALID;
}

ws_status ws_stack_param_offset(const ws_stack_cfg* cfg, int32_t layer, int32_t lin,
                                int64_t* off_A, int64_t* off_B) {
  ws_status s = stack_check(cfg);
  if (s != WS_OK) return s;
  if (!off_A || !off_B || lin < 0 || lin >= WS_NLIN || layer < 0 || layer >= cfg->n_layers)
    return WS_ERR_INVALID;
  stack_param_offset(*cfg, layer, lin, off_A, off_B);
  return WS_OK;
}

ws_status ws_block_forward(const ws_stack_cfg* cfg, const void* block_weights, int32_t first_layer,
                           int32_t n_layers, const float* params, uint32_t step, uint32_t microbatch,
                           const float* h_in, float* h_out, void* saved, void* workspace,
                           size_t ws_bytes, ws_stream_t stream) {
  ws_status s = stack_check(cfg);
  if (s != WS_OK) return s;
  if (!block_weights || !params || !h_in || !h_out || !workspace) return WS_ERR_INVALID;
  if (n_layers < 1 || first_layer < 0 || first_layer + n_layers > cfg->n_layers) return WS_ERR_SHAPE;
  if (h_in == h_out || microbatch > 0xFFFFFFu) return WS_ERR_INVALID;
  if (!aligned16(block_weights) || !aligned16(params) || !aligned16(h_in) || !aligned16(h_out) ||
      !aligned16(workspace) || (saved && !aligned16(saved)))
    return WS_ERR_ALIGN;
  if (ws_bytes < stack_ws_bytes(*cfg, n_layers)) return WS_ERR_OOM;
  return cuda_status(block_forward(*cfg, n_layers, block_weights, first_layer, n_layers, params,
                                   step, microbatch, nullptr, h_in, h_out, saved, workspace,
                                   (cudaStream_t)stream));
}

ws_status ws_block_backward_recompute(const ws_stack_cfg* cfg, const void* block_weights,
                                      int32_t first_layer, int32_t n_layers, const float* params,
                                      uint32_t step, uint32_t microbatch, const float* h_in,
                                      const void* saved, const float* dh_out, float* dh_in,
                                      float* grads, int32_t grad_accumulate, void* workspace,
                                      size_t ws_bytes, ws_stream_t stream) {
  ws_status s = stack_check(cfg);
  if (s != WS_OK) return s;
  if (!block_weights || !params || !dh_out || !dh_in || !grads || !workspace) return WS_ERR_INVALID;
  if (!saved && !h_in) return WS_ERR_INVALID;
  if (microbatch > 0xFFFFFFu) return WS_ERR_INVALID;
  if (n_layers < 1 || first_layer < 0 || first_layer + n_layers > cfg->n_layers) return WS_ERR_SHAPE;
  if (!aligned16(block_weights) || !aligned16(params) || !aligned16(dh_out) || !aligned16(dh_in) ||
      !aligned16(grads) || !aligned16(workspace) || (saved && !aligned16(saved)) ||
      (h_in && !aligned16(h_in)))
    return WS_ERR_ALIGN;
  if (ws_bytes < stack_ws_bytes(*cfg, n_layers)) return WS_ERR_OOM;
  return cuda_status(block_backward(*cfg, n_layers, block_weights, first_layer, n_layers, params,
                                    step, microbatch, nullptr, h_in, saved, dh_out, dh_in, grads,
                                    grad_accumulate ? 1 : 0, workspace, (cudaStream_t)stream));
}

ws_status ws_stream_block_h2d(const void* pinned_src, void* dev_dst, size_t bytes,
                              ws_stream_t copy_stream, ws_event_t wait_event,
                              ws_event_t done_event) {
  if (!pinned_src || !dev_dst) return WS_ERR_INVALID;
  if (bytes == 0) return WS_OK;
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, pinned_src) != cudaSuccess) {
    cudaGetLastError();
    return WS_ERR_NOT_PINNED;
  }
  if (attr.type != cudaMemoryTypeHost) return WS_ERR_NOT_PINNED;
  cudaStream_t st = (cudaStream_t)copy_stream;
  if (wait_event && cudaStreamWaitEvent(st, (cudaEvent_t)wait_event, 0) != cudaSuccess)
    return WS_ERR_CUDA;
  if (cudaMemcpyAsync(dev_dst, pinned_src, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return WS_ERR_CUDA;
  if (done_event && cudaEventRecord((cudaEvent_t)done_event, st) != cudaSuccess) return WS_ERR_CUDA;
  return WS_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------- training step
namespace {

// Events of one step: the window slots' loaded / freed events, the fork and
// join of the copy stream and, when copies are timed, one start / end pair
// per block copy (recorded as external events so they become nodes of a
// captured graph and carry the replay's timestamps).
struct StepEvents {
  cudaEvent_t loaded[2] = {nullptr, nullptr}, freed[2] = {nullptr, nullptr};
  cudaEvent_t fork = nullptr, join = nullptr;
  int n_timed = 0, cap_timed = 0;
  cudaEvent_t* t0 = nullptr;
  cudaEvent_t* t1 = nullptr;
  cudaError_t create(int copies_to_time) {
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
      e = cudaEventCreateWithFlags(&loaded[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&freed[i], cudaEventDisableTiming);
    }
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&join, cudaEventDisableTiming);
    if (e == cudaSuccess && copies_to_time > 0) {
      t0 = new (std::nothrow) cudaEvent_t[copies_to_time]();
      t1 = new (std::nothrow) cudaEvent_t[copies_to_time]();
      if (!t0 || !t1) return cudaErrorMemoryAllocation;
      for (int i = 0; i < copies_to_time && e == cudaSuccess; ++i) {
        e = cudaEventCreate(&t0[i]);
        if (e == cudaSuccess) e = cudaEventCreate(&t1[i]);
      }
      cap_timed = copies_to_time;
    }
    return e;
  }
  void destroy() {
    for (int i = 0; i < 2; ++i) {
      if (loaded[i]) cudaEventDestroy(loaded[i]);
      if (freed[i]) cudaEventDestroy(freed[i]);
      loaded[i] = freed[i] = nullptr;
    }
    if (fork) cudaEventDestroy(fork);
    if (join) cudaEventDestroy(join);
    fork = join = nullptr;
    for (int i = 0; i < cap_timed; ++i) {
      if (t0 && t0[i]) cudaEventDestroy(t0[i]);
      if (t1 && t1[i]) cudaEventDestroy(t1[i]);
    }
    delete[] t0;
    delete[] t1;
    t0 = t1 = nullptr;
    cap_timed = n_timed = 0;
  }
};

struct StepOpts {
  int n_micro = 1;
  int order = WS_GA_MICROBATCH_MAJOR;
  bool time_copies = false;
  size_t piece = 0;  // 0: one copy per block
};

ws_status read_opts(const ws_step_opts* o, StepOpts* out) {
  StepOpts r;
  if (o) {
    if (o->n_micro < 1 || o->n_micro > 0xFFFFFF) return WS_ERR_INVALID;
    if (o->order != WS_GA_MICROBATCH_MAJOR && o->order != WS_GA_BLOCK_MAJOR) return WS_ERR_INVALID;
    if (o->copy_piece_bytes < 0 || (o->copy_piece_bytes % 256) != 0 || o->reserved != 0)
      return WS_ERR_INVALID;
    r.n_micro = o->n_micro;
    r.order = o->order;
    r.time_copies = o->time_copies != 0;
    r.piece = (size_t)o->copy_piece_bytes;
  }
  *out = r;
  return WS_OK;
}

ws_status check_step(const ws_stack_cfg* cfg, int32_t block_layers, int32_t streamed,
                     const ws_stack_buffers* buf, const void* copy_stream) {
  ws_status s = stack_check(cfg);
  if (s != WS_OK) return s;
  if (!buf) return WS_ERR_INVALID;
  if (block_layers < 1 || cfg->n_layers % block_layers) return WS_ERR_SHAPE;
  if (!buf->params || !buf->grads || !buf->adam_m || !buf->adam_v || !buf->boundary || !buf->dh ||
      !buf->workspace || !buf->loss)
    return WS_ERR_INVALID;
  if (streamed) {
    if (!buf->host_weights || !buf->window || buf->saved || !copy_stream) return WS_ERR_INVALID;
  } else {
    if (!buf->dev_weights || !buf->saved) return WS_ERR_INVALID;
  }
  if (buf->workspace_bytes < stack_ws_bytes(*cfg, block_layers)) return WS_ERR_OOM;
  return WS_OK;
}

// Everything of one step after the step word and the micro-batches' block-0
// boundaries (= h0) are set.  Reads the step from the device word, so eager
// calls and graph replays run the same kernels with the same arguments.
//
// Streamed mode keeps a 2-slot window: slot s holds block b with s = b % 2.
// The copy of block b+1 is issued before block b's compute so it runs on the
// copy engine meanwhile; a copy into a slot waits for the compute stream's
// last use of that slot.  A block still resident in its slot (the last two at
// the forward/backward turnaround, or between micro-batches) is not copied
// again.  The copy stream is forked from and joined back into the compute
// stream, so the whole step can be captured as one graph.
// warm: the window already holds blocks 0 and 1 (slots 0 and 1), as the
// previous step's backward left it; their copies are skipped.
//
// Gradient accumulation over n_micro micro-batches (each with its own h0,
// boundary activations, output gradient and dropout keys): micro-batch-major
// runs the whole forward and backward of one micro-batch after the other;
// block-major (streamed) loads each block once per direction and runs every
// micro-batch through it.  Both add the micro-batches' adapter gradients in
// the same order (micro-batch 0 writes, the others add), so the two orders,
// and a resident run, give bitwise the same step.
ws_status step_body(const ws_stack_cfg& cfg, int block_layers, bool streamed, const StepOpts& o,
                    const ws_stack_buffers& buf, float lr, cudaStream_t cs, cudaStream_t ps,
                    StepEvents& ev, bool warm = false) {
  const int nb = cfg.n_layers / block_layers;
  const size_t bbytes = stack_block_bytes(cfg, block_layers);
  const size_t slayer = stack_saved_layer(cfg);
  const int64_t MH = cfg.M * cfg.H;
  const int64_t np = stack_n_params(cfg);
  const int nm = o.n_micro;
  const uint32_t* stepw = stack_step_word(cfg, block_layers, buf.workspace);
  int slot_block[2] = {-1, -1};
  bool slot_used[2] = {false, false};
  bool slot_copied[2] = {false, false};  // a copy into the slot was issued in this step
  if (streamed && warm && nb >= 2) {
    slot_block[0] = 0;
    slot_block[1] = 1;
  }
  const uint8_t* host = static_cast<const uint8_t*>(buf.host_weights);
  uint8_t* window = static_cast<uint8_t*>(buf.window);
  ev.n_timed = 0;
#define WS_STEP_TRY(x)                          \
  do {                                          \
    if ((x) != cudaSuccess) return WS_ERR_CUDA; \
  } while (0)
  auto ensure = [&](int blk) -> ws_status {
    if (blk < 0 || blk >= nb) return WS_OK;
    const int sl = blk % 2;
    if (slot_block[sl] == blk) return WS_OK;
    cudaStream_t st = ps;
    if (slot_used[sl] && cudaStreamWaitEvent(st, ev.freed[sl], 0) != cudaSuccess) return WS_ERR_CUDA;
    const bool timed = ev.n_timed < ev.cap_timed;
    if (timed && cudaEventRecordWithFlags(ev.t0[ev.n_timed], st, cudaEventRecordExternal) != cudaSuccess)
      return WS_ERR_CUDA;
    const size_t piece = (o.piece == 0 || o.piece > bbytes) ? bbytes : o.piece;
    for (size_t off = 0; off < bbytes; off += piece) {
      const size_t n = bbytes - off < piece ? bbytes - off : piece;
      ws_status r = ws_stream_block_h2d(host + (size_t)blk * bbytes + off,
                                        window + (size_t)sl * bbytes + off, n, (ws_stream_t)st,
                                        nullptr, off + n == bbytes ? (ws_event_t)ev.loaded[sl] : nullptr);
      if (r != WS_OK) return r;
    }
    if (timed) {
      if (cudaEventRecordWithFlags(ev.t1[ev.n_timed], st, cudaEventRecordExternal) != cudaSuccess)
        return WS_ERR_CUDA;
      ++ev.n_timed;
    }
    slot_block[sl] = blk;
    slot_copied[sl] = true;
    return WS_OK;
  };
  // the compute stream waits for a slot's copy only if one was issued in this step
  auto wait_loaded = [&](int blk) -> cudaError_t {
    const int sl = blk % 2;
    return slot_copied[sl] ? cudaStreamWaitEvent(cs, ev.loaded[sl], 0) : cudaSuccess;
  };
  auto block_ptr = [&](int blk) -> const void* {
    if (streamed) return window + (size_t)(blk % 2) * bbytes;
    return static_cast<const uint8_t*>(buf.dev_weights) + (size_t)blk * bbytes;
  };
  auto bnd = [&](int mb, int b) { return buf.boundary + ((size_t)mb * (nb + 1) + b) * MH; };
  auto dh = [&](int mb) { return buf.dh + (size_t)mb * MH; };
  auto saved = [&](int b) -> void* {
    return streamed ? nullptr : static_cast<uint8_t*>(buf.saved) + (size_t)b * block_layers * slayer;
  };
  auto release = [&](int b) -> cudaError_t {
    if (!streamed) return cudaSuccess;
    slot_used[b % 2] = true;
    return cudaEventRecord(ev.freed[b % 2], cs);
  };
  auto fwd = [&](int b, int mb) {
    return block_forward(cfg, block_layers, block_ptr(b), b * block_layers, block_layers,
                         buf.params, 0u, (uint32_t)mb, stepw, bnd(mb, b), bnd(mb, b + 1),
                         saved(b), buf.workspace, cs);
  };
  auto bwd = [&](int b, int mb) {
    return block_backward(cfg, block_layers, block_ptr(b), b * block_layers, block_layers,
                          buf.params, 0u, (uint32_t)mb, stepw, bnd(mb, b), saved(b), dh(mb),
                          dh(mb), buf.grads, mb > 0 ? 1 : 0, buf.workspace, cs);
  };
  auto loss = [&](int mb) {
    return loss_and_grad(cfg, block_layers, bnd(mb, nb), dh(mb), buf.loss, nm, mb > 0 ? 1 : 0,
                         buf.workspace, cs);
  };
  ws_status rc = WS_OK;
  if (streamed) {
    WS_STEP_TRY(cudaEventRecord(ev.fork, cs));
    WS_STEP_TRY(cudaStreamWaitEvent(ps, ev.fork, 0));
  }
  // Micro-batch-major in a resident run; block-major only changes the order
  // of a streamed run (a resident run loads nothing).
  const bool block_major = streamed && o.order == WS_GA_BLOCK_MAJOR;
  const int passes = block_major ? 1 : nm;
  for (int pass = 0; pass < passes; ++pass) {
    const int mb0 = block_major ? 0 : pass, mb1 = block_major ? nm : pass + 1;
    // ---- forward
    if (streamed && (rc = ensure(0)) != WS_OK) return rc;
    for (int b = 0; b < nb; ++b) {
      if (streamed && (rc = ensure(b + 1)) != WS_OK) return rc;
      if (streamed) WS_STEP_TRY(wait_loaded(b));
      for (int mb = mb0; mb < mb1; ++mb) WS_STEP_TRY(fwd(b, mb));
      WS_STEP_TRY(release(b));
    }
    // ---- loss
    for (int mb = mb0; mb < mb1; ++mb) WS_STEP_TRY(loss(mb));
    // ---- backward, blocks in reverse
    for (int b = nb - 1; b >= 0; --b) {
      if (streamed) {
        if ((rc = ensure(b)) != WS_OK) return rc;
        if ((rc = ensure(b - 1)) != WS_OK) return rc;
        WS_STEP_TRY(wait_loaded(b));
      }
      for (int mb = mb0; mb < mb1; ++mb) WS_STEP_TRY(bwd(b, mb));
      WS_STEP_TRY(release(b));
    }
  }
  // ---- optimizer
  WS_STEP_TRY(adam_step(buf.params, buf.grads, buf.adam_m, buf.adam_v, np, stepw, lr, cs));
  if (streamed) {
    WS_STEP_TRY(cudaEventRecord(ev.join, ps));
    WS_STEP_TRY(cudaStreamWaitEvent(cs, ev.join, 0));
  }
#undef WS_STEP_TRY
  return WS_OK;
}

// The block copies one step can issue at most (for timing events).
int max_copies(const ws_stack_cfg& cfg, int block_layers, const StepOpts& o) {
  const int nb = cfg.n_layers / block_layers;
  return 2 * nb * (o.order == WS_GA_BLOCK_MAJOR ? 1 : o.n_micro);
}

ws_status step_prologue(const ws_stack_cfg& cfg, int block_layers, const StepOpts& o,
                        const ws_stack_buffers& buf, uint32_t step, const float* h0,
                        cudaStream_t cs) {
  uint32_t* stepw = stack_step_word(cfg, block_layers, buf.workspace);
  if (set_step(stepw, step, cs) != cudaSuccess) return WS_ERR_CUDA;
  const int nb = cfg.n_layers / block_layers;
  const size_t MH = (size_t)(cfg.M * cfg.H);
  for (int mb = 0; mb < o.n_micro; ++mb)
    if (cudaMemcpyAsync(buf.boundary + (size_t)mb * (nb + 1) * MH, h0 + (size_t)mb * MH, MH * 4,
                        cudaMemcpyDeviceToDevice, cs) != cudaSuccess)
      return WS_ERR_CUDA;
  return WS_OK;
}

}  // namespace

// Two captures of the step: "cold" copies every block it needs; "warm"
// (streamed only) starts from the window the previous step left behind
// (blocks 0 and 1 in slots 0 and 1) and skips those two copies.  The first
// replay is cold, every later one warm.
struct ws_step_graph {
  ws_stack_cfg cfg;
  int32_t block_layers;
  StepOpts opts;
  ws_stack_buffers buf;
  StepEvents ev[2];
  cudaGraph_t graph[2] = {nullptr, nullptr};
  cudaGraphExec_t exec[2] = {nullptr, nullptr};
  bool warm_ok = false;   // a warm capture exists
  bool window_warm = false;
  int last = -1;          // capture replayed last
};

extern "C" {

ws_status ws_stack_train_step_ex(const ws_stack_cfg* cfg, int32_t block_layers, int32_t streamed,
                                 const ws_step_opts* opts, const ws_stack_buffers* buf,
                                 uint32_t step, const float* h0, float lr, ws_stream_t compute,
                                 ws_stream_t copy_stream) {
  ws_status s = check_step(cfg, block_layers, streamed, buf, copy_stream);
  if (s != WS_OK) return s;
  StepOpts o;
  if ((s = read_opts(opts, &o)) != WS_OK) return s;
  if (o.time_copies) return WS_ERR_INVALID;  // timed copies are read from a graph
  if (!h0) return WS_ERR_INVALID;
  const cudaStream_t cs = (cudaStream_t)compute;
  s = step_prologue(*cfg, block_layers, o, *buf, step, h0, cs);
  if (s != WS_OK) return s;
  StepEvents ev;
  if (streamed && ev.create(0) != cudaSuccess) {
    ev.destroy();
    return WS_ERR_CUDA;
  }
  s = step_body(*cfg, block_layers, streamed != 0, o, *buf, lr, cs, (cudaStream_t)copy_stream, ev);
  ev.destroy();
  return s;
}

ws_status ws_stack_train_step(const ws_stack_cfg* cfg, int32_t block_layers, int32_t streamed,
                              const ws_stack_buffers* buf, uint32_t step, const float* h0, float lr,
                              ws_stream_t compute, ws_stream_t copy_stream) {
  return ws_stack_train_step_ex(cfg, block_layers, streamed, nullptr, buf, step, h0, lr, compute,
                                copy_stream);
}

ws_status ws_stack_graph_create_ex(const ws_stack_cfg* cfg, int32_t block_layers, int32_t streamed,
                                   const ws_step_opts* opts, const ws_stack_buffers* buf, float lr,
                                   ws_stream_t compute, ws_stream_t copy_stream,
                                   ws_step_graph** out) {
  if (!out) return WS_ERR_INVALID;
  *out = nullptr;
  ws_status s = check_step(cfg, block_layers, streamed, buf, copy_stream);
  if (s != WS_OK) return s;
  StepOpts o;
  if ((s = read_opts(opts, &o)) != WS_OK) return s;
  if (o.time_copies && !streamed) return WS_ERR_INVALID;
  ws_step_graph* g = new (std::nothrow) ws_step_graph();
  if (!g) return WS_ERR_OOM;
  g->cfg = *cfg;
  g->block_layers = block_layers;
  g->opts = o;
  g->buf = *buf;
  const cudaStream_t cs = (cudaStream_t)compute;
  g->warm_ok = streamed != 0 && cfg->n_layers / block_layers >= 2;
  for (int v = 0; v < (g->warm_ok ? 2 : 1) && s == WS_OK; ++v) {
    if (g->ev[v].create(o.time_copies ? max_copies(*cfg, block_layers, o) : 0) != cudaSuccess) {
      s = WS_ERR_CUDA;
      break;
    }
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
      s = WS_ERR_CUDA;
      break;
    }
    s = step_body(*cfg, block_layers, streamed != 0, o, *buf, lr, cs, (cudaStream_t)copy_stream,
                  g->ev[v], v == 1);
    cudaGraph_t graph = nullptr;
    const cudaError_t ec = cudaStreamEndCapture(cs, &graph);
    g->graph[v] = graph;
    if (s == WS_OK && ec != cudaSuccess) s = WS_ERR_CUDA;
    if (s == WS_OK && cudaGraphInstantiate(&g->exec[v], graph, 0) != cudaSuccess) s = WS_ERR_CUDA;
  }
  if (s != WS_OK) {
    cudaGetLastError();
    ws_stack_graph_destroy(g);
    return s;
  }
  *out = g;
  return WS_OK;
}

ws_status ws_stack_graph_create(const ws_stack_cfg* cfg, int32_t block_layers, int32_t streamed,
                                const ws_stack_buffers* buf, float lr, ws_stream_t compute,
                                ws_stream_t copy_stream, ws_step_graph** out) {
  return ws_stack_graph_create_ex(cfg, block_layers, streamed, nullptr, buf, lr, compute,
                                  copy_stream, out);
}

ws_status ws_stack_graph_step(ws_step_graph* g, uint32_t step, const float* h0,
                              ws_stream_t compute) {
  if (!g || !h0) return WS_ERR_INVALID;
  const cudaStream_t cs = (cudaStream_t)compute;
  ws_status s = step_prologue(g->cfg, g->block_layers, g->opts, g->buf, step, h0, cs);
  if (s != WS_OK) return s;
  const int v = (g->warm_ok && g->window_warm) ? 1 : 0;
  if (cudaGraphLaunch(g->exec[v], cs) != cudaSuccess) return WS_ERR_CUDA;
  g->window_warm = g->warm_ok;
  g->last = v;
  return WS_OK;
}

ws_status ws_stack_graph_copy_times(ws_step_graph* g, float* ms, int32_t capacity, int32_t* n) {
  if (!g || !n || (capacity > 0 && !ms)) return WS_ERR_INVALID;
  *n = 0;
  if (g->last < 0 || g->ev[g->last].cap_timed == 0) return WS_ERR_INVALID;
  const StepEvents& ev = g->ev[g->last];
  if (cudaEventSynchronize(ev.t1[ev.n_timed > 0 ? ev.n_timed - 1 : 0]) != cudaSuccess)
    return WS_ERR_CUDA;
  for (int i = 0; i < ev.n_timed; ++i) {
    float t = 0.0f;
    if (cudaEventElapsedTime(&t, ev.t0[i], ev.t1[i]) != cudaSuccess) return WS_ERR_CUDA;
    if (i < capacity) ms[i] = t;
  }
  *n = ev.n_timed;
  return WS_OK;
}

ws_status ws_stack_graph_destroy(ws_step_graph* g) {
  if (!g) return WS_ERR_INVALID;
  for (int v = 0; v < 2; ++v) {
    if (g->exec[v]) cudaGraphExecDestroy(g->exec[v]);
    if (g->graph[v]) cudaGraphDestroy(g->graph[v]);
    g->ev[v].destroy();
  }
  delete g;
  return WS_OK;
}

}  // extern "C"
