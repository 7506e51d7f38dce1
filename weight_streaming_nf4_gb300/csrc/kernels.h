// kernels.h -- internal interfaces between the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "wsnf4.h"

namespace ws {

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// A frozen base weight [N, K]: NF4 (codes, absmax) or, when wbf16 is set,
// bf16 row-major (codes and absmax unused).
struct NF4View {
  const uint8_t* codes;  // [N, K/2]
  const float* absmax;   // [K/64, N]
  int64_t N, K;
  const uint16_t* wbf16 = nullptr;
};

// Linears of one grouped launch at most (q, k, v share the attention
// input; gate and up share the MLP input).
constexpr int kMaxGroups = 3;

// Arguments of one dequant-GEMM launch (see nf4_gemm.cu).
struct GemmArgs {
  int64_t M;            // activation rows
  int64_t Nout;         // output columns (forward: N, backward: K)
  int nk_total;         // 64-deep contraction steps per tile
  int mtiles, ntiles;   // output tiles (M-tiles vary fastest in the schedule)
  int has_lora;         // split 0 runs the extra LoRA step
  const float* lora_F;  // forward: B [N, 16]; backward: A [16, K]
  float lora_scale;     // s = (alpha / r) / (1 - p)
  const uint32_t* mask; // backward: dropout bits [M, K/32]
  void* out;            // [M, Nout] bf16 or fp32
  int out_f32, out_accum;
  float* partial;       // per CTA one fp32 partial tile (its cut first segment), stored as
                        // float4 [BN/4][BM]
  uint32_t* flags;      // [grid] set to 1 once that partial is complete (ring words, zero
                        // before and after the launch)
  const uint8_t* codes; // the weight's packed codes [N, K/2]
  const float* absmax;  // the weight's block scales [K/64, N]
  int64_t wN, wK;       // the weight's shape
  int epad;             // schedule-only steps charged per tile (see GemmPlan::epad)
  // Forward only: ngroups linears that read the same activation, side by
  // side along the output columns.  Group g owns output columns
  // [gcol[g], gcol[g+1]) (multiples of the tile width), with its own weight
  // (gcodes, gabsmax; wN = its width), LoRA factor glora_F, output gout
  // (row pitch = its width) and LoRA activation rows [g*M, (g+1)*M) of the
  // lora map.  ngroups = 1 uses codes / absmax / lora_F / out above.
  int ngroups;
  int64_t gcol[kMaxGroups + 1];
  const uint8_t* gcodes[kMaxGroups];
  const float* gabsmax[kMaxGroups];
  const float* glora_F[kMaxGroups];
  void* gout[kMaxGroups];
};

// Tile configuration: a pure function of the shape and the SM count, so a
// resident and a streamed run always pick the same kernels and split order.
struct GemmPlan {
  bool bwd;
  bool pair;  // two CTAs of a cluster share each weight tile
  int um, bn;
  int mtiles, ntiles, nk;
  // Stream-K ranges are cut over tiles of S + epad iterations, the last
  // epad of which carry no work: a unit whose range ends more tiles (one
  // accumulator drain each) gets fewer contraction steps.
  int epad;
};

int device_sm_count();
// CTAs of the persistent stream-K grid for a plan (with or without the extra
// LoRA step): min(SM count, iterations / 8), at least 1.
int64_t grid_ctas(const GemmPlan& p, bool has_lora);
int64_t grid_units(const GemmPlan& p, bool has_lora);
// This device's address and size of the built-in scratch array used by
// ws_nf4_matmul_noalloc (looked up once per device).
cudaError_t noalloc_scratch(float** ptr, size_t* bytes);
// Counts every kernel launch the library makes (reported by ws_kernel_launches).
void note_launch();
cudaError_t read_and_clear_dev_error(uint32_t* flags);
// One kernel that waits (bounded by limit_us) for a ring word nothing sets.
cudaError_t run_wait_selfcheck(uint32_t limit_us, cudaStream_t st);
// n zeroed cross-CTA words that the launch using them leaves zeroed again.
cudaError_t ring_slots(uint32_t n, uint32_t** out);
GemmPlan plan_gemm(bool bwd, int64_t M, int64_t Nout, int64_t Kc);
size_t gemm_partial_bytes(const GemmPlan& p, int64_t M, int64_t Nout);

// act: [M, Kc] bf16 (forward x, backward dY); lora_act: [M, 64] bf16 split
// factor (U or G hi/lo) or NULL; lora_F: the other LoRA factor (B or A).
cudaError_t run_nf4_gemm(const GemmPlan& p, const NF4View& W, const uint16_t* act, int64_t M,
                         const uint16_t* lora_act, const float* lora_F, float lora_scale,
                         const uint32_t* mask, void* out, int out_f32, int out_accum,
                         float* partial, cudaStream_t st);

// Forward of ng linears sharing the activation act [M, K] in one launch:
// out[g] = act . W[g]'^T + s * lora_act[g] . F[g]^T, lora_act [ng][M][64]
// contiguous.  p = plan_gemm(false, M, sum of widths, K); every width a
// multiple of p.bn (else cudaErrorInvalidValue).
cudaError_t run_nf4_gemm_group(const GemmPlan& p, int ng, const NF4View* W, const uint16_t* act,
                               int64_t M, const uint16_t* lora_act, const float* const* lora_F,
                               float lora_scale, uint16_t* const* out, float* partial,
                               cudaStream_t st);

// ---- small kernels (lora_small.cu) ----------------------------------------------------
struct DropKeyHost {
  uint32_t k0, k1, c1, c2, c3, thresh, drop_all;
  const uint32_t* step_dev;  // device step word (replaces c3) or NULL
};
DropKeyHost make_drop_key(const ws_dropout_key& k);

cudaError_t run_quantize_nf4(const uint16_t* W, int64_t N, int64_t K, uint8_t* codes,
                             float* absmax, cudaStream_t st);
// Scratch of run_skinny_tc / run_lora_down / run_lora_G (chunk partial sums
// and per-row-block counters).
size_t skinny_partial_bytes(int64_t M, int64_t K);
// out [M,16] = X~ F^T on the tensor cores (see nf4_gemm.cu); key != NULL:
// X under the dropout mask (bits stored to mask_bytes when not NULL).
cudaError_t run_skinny_tc(const uint16_t* X, const float* F, bool f_kj, int64_t M, int64_t K,
                          const DropKey* key, uint8_t* mask_bytes, float* partial, float* out,
                          uint16_t* ext, cudaStream_t st);
// The same for ng <= kMaxGroups factors F[g] ([16][K], A layout) applied to
// one X under ng dropout masks (keys[g]) in one launch: out[g], ext[g],
// mask_bytes[g] (entries may be NULL), partial[g] (skinny_partial_bytes each).
cudaError_t run_skinny_tc_group(const uint16_t* X, int ng, const float* const* F, int64_t M,
                                int64_t K, const DropKey* keys, uint8_t* const* mask_bytes,
                                float* const* partial, float* const* out, uint16_t* const* ext,
                                cudaStream_t st);
// G[g] = dY[g] B[g] for ng linears with the same M and N in one launch.
cudaError_t run_skinny_G_group(int ng, const uint16_t* const* dY, const float* const* B, int64_t M,
                               int64_t N, float* const* partial, float* const* G,
                               uint16_t* const* Gext, cudaStream_t st);
// U = (mask . x) A^T [M,16] fp32; Uext [M,64] bf16 hi/lo; mask bits (optional).
cudaError_t run_lora_down(const uint16_t* x, const float* A, int64_t M, int64_t K,
                          const DropKeyHost& key, float* U, uint16_t* Uext, uint32_t* mask_out,
                          float* partial, cudaStream_t st);
// G = dY B [M,16] fp32 and Gext [M,64] bf16 hi/lo.
cudaError_t run_lora_G(const uint16_t* dY, const float* B, int64_t M, int64_t N, float* G,
                       uint16_t* Gext, float* partial, cudaStream_t st);
// Dropout keep bits [M, K/32] of one linear, regenerated from the key.
cudaError_t run_mask_gen(int64_t M, int64_t K, const DropKeyHost& key, uint32_t* mask,
                         cudaStream_t st);
// Weight gradient of a LoRA factor on the tensor cores (nf4_gemm.cu):
// out = s * P^T Q~ with P [M,16] fp32, Q [M,C] bf16 (masked by `mask`
// [M, C/32] when not NULL).  out layout is [C,16] (dB) or, when
// transpose_out, [16,C] (dA).  accumulate != 0: out = out + s * P^T Q~
// (one fp32 add per element after the fixed-order sum).  No workspace.
size_t wgrad_tc_bytes(int64_t M, int64_t C);
// ng weight gradients with the same M, C and s in one launch (masks: all or none).
cudaError_t run_wgrad_tc_group(int ng, const float* const* P, const uint16_t* const* Q,
                               const uint32_t* const* mask, int64_t M, int64_t C, float s,
                               float* const* out, int transpose_out, int accumulate,
                               cudaStream_t st);
cudaError_t run_wgrad_tc(const float* P, const uint16_t* Q, const uint32_t* mask, int64_t M,
                         int64_t C, float s, float* out, int transpose_out, int accumulate,
                         void* ws, cudaStream_t st);

// 2-D bf16 tensor map with the 128-byte swizzle: `inner` contiguous elements,
// `outer` rows pitch_bytes apart, box {box_inner, box_outer} (nf4_gemm.cu).
bool tmap_bf16_sw128(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer);

// ---- attention core (attention.cu) ----------------------------------------------------
// Causal attention with grouped kv heads over n_seq sequences of S tokens:
// q [M, nh*hd], k, v [M, nkv*hd] bf16 (M = n_seq*S, hd 64 or 128).  Forward:
// o [M, nh*hd] bf16, o32 (optional) the same in fp32, lse [nh, M] natural
// log-sum-exp.  Backward from dO [M, nh*hd] bf16, the forward's o32 and lse:
// dq [M, nh*hd], dk, dv [M, nkv*hd] bf16; ws of attn_bwd_workspace_bytes.
cudaError_t attn_read_and_clear_dev_error(uint32_t* flags);
size_t attn_bwd_workspace_bytes(int64_t M, int nh, int head_dim);
cudaError_t run_attn_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, int n_seq,
                         int S, int nh, int nkv, int hd, uint16_t* o, float* o32, float* lse,
                         cudaStream_t st);
cudaError_t run_attn_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const float* o32, const float* lse, const uint16_t* dO, int n_seq, int S,
                         int nh, int nkv, int hd, uint16_t* dq, uint16_t* dk, uint16_t* dv,
                         void* ws, cudaStream_t st);

// ---- one LoRA linear (linear.cu) --------------------------------------------------------
size_t linear_workspace_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t linear_fwd(const NF4View& W, const uint16_t* x, const float* A, const float* B,
                       int64_t M, float scale, const DropKeyHost& key, uint16_t* y, float* U,
                       uint32_t* mask, void* ws, cudaStream_t st);
// ng linears reading the same x: one LoRA-down launch, one GEMM for the
// first ng_gemm of them and one GEMM for each of the others.
size_t linear_group_workspace_bytes(int64_t M, int ng, const int64_t* N, int64_t K);
cudaError_t linear_fwd_group(int ng, int ng_gemm, const NF4View* W, const uint16_t* x, const float* const* A,
                             const float* const* B, int64_t M, float scale, const DropKeyHost* keys,
                             uint16_t* const* y, float* const* U, uint32_t* const* mask, void* ws,
                             cudaStream_t st);
// ng linears of one shape reading the same x, each with its own dY; their
// input gradients summed into dX.
size_t linear_bwd_group_workspace_bytes(int64_t M, int ng, int64_t N, int64_t K);
// grad_accum != 0 adds dA, dB into the existing gradients (gradient
// accumulation over micro-batches) instead of overwriting them.
cudaError_t linear_bwd_group(int ng, const NF4View* W, const uint16_t* x, const float* const* A,
                             const float* const* B, int64_t M, float scale, const DropKeyHost* keys,
                             const float* const* U, const uint32_t* const* mask,
                             const uint16_t* const* dY, void* dX, int dX_f32, int dX_accum,
                             float* const* dA, float* const* dB, int grad_accum, void* ws,
                             cudaStream_t st);
cudaError_t linear_bwd(const NF4View& W, const uint16_t* x, const float* A, const float* B,
                       int64_t M, float scale, const DropKeyHost& key, const float* U,
                       const uint32_t* mask, const uint16_t* dY, void* dX, int dX_f32,
                       int dX_accum, float* dA, float* dB, int grad_accum, void* ws,
                       cudaStream_t st);

}  // namespace ws

namespace ws {
// ---- synthetic stack (stack.cu) -------------------------------------------------------
ws_status stack_check(const ws_stack_cfg* c);
size_t stack_block_bytes(const ws_stack_cfg& c, int block_layers);
int64_t stack_n_params(const ws_stack_cfg& c);
size_t stack_saved_layer(const ws_stack_cfg& c);
size_t stack_ws_bytes(const ws_stack_cfg& c, int block_layers);
void stack_weight_offset(const ws_stack_cfg& c, int layer_in_block, int lin, size_t* off_codes,
                         size_t* off_absmax);
void stack_param_offset(const ws_stack_cfg& c, int layer, int lin, int64_t* off_A, int64_t* off_B);
bool stack_saved_offset(const ws_stack_cfg& c, int field, int lin, size_t* off);
// step_dev: device step word for the dropout keys (NULL: use `step`);
// mb: micro-batch index of the dropout keys.
cudaError_t block_forward(const ws_stack_cfg& c, int block_layers_ws, const void* block,
                          int first_layer, int n_layers, const float* params, uint32_t step,
                          uint32_t mb, const uint32_t* step_dev, const float* h_in, float* h_out,
                          void* saved, void* ws, cudaStream_t st);
// grad_accum != 0: the block's adapter gradients are added to `grads`.
cudaError_t block_backward(const ws_stack_cfg& c, int block_layers_ws, const void* block,
                           int first_layer, int n_layers, const float* params, uint32_t step,
                           uint32_t mb, const uint32_t* step_dev, const float* h_in,
                           const void* saved, const float* dh_out, float* dh_in, float* grads,
                           int grad_accum, void* ws, cudaStream_t st);
// Device word reserved in the stack workspace for the step counter.
uint32_t* stack_step_word(const ws_stack_cfg& c, int block_layers, void* ws);
// Byte offset of a backward intermediate (WS_WK_*) in the stack workspace.
bool stack_ws_offset(const ws_stack_cfg& c, int block_layers, int field, size_t* off);
// Loss of one micro-batch's final activation h and its gradient dh, as its
// share of the step loss (mean over n_micro micro-batches); accumulate != 0
// adds the share to *loss.
cudaError_t loss_and_grad(const ws_stack_cfg& c, int block_layers_ws, const float* h, float* dh,
                          float* loss, int n_micro, int accumulate, void* ws, cudaStream_t st);
// Adam at step t = *step_dev + 1 (bias corrections computed on the device).
cudaError_t adam_step(float* p, const float* g, float* m, float* v, int64_t n,
                      const uint32_t* step_dev, float lr, cudaStream_t st);
cudaError_t set_step(uint32_t* step_dev, uint32_t step, cudaStream_t st);
}  // namespace ws
