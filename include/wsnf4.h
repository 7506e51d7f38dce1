/*
 * wsnf4.h -- C ABI of libwsnf4.so: the streamed frozen-NF4-base LoRA linear
 * on one GB300 (sm_103a).
 *
 * The method (Poros, blockwise residency for frozen-base QLoRA).  Citations
 * name the page and its section; the research page "Poros" has no section
 * headings, so its paragraphs are named by their subject.
 *  - The frozen base is stored as 4-bit NormalFloat (NF4), one fp32 absmax
 *    per 64 consecutive weights of a row; NF4 is the precision whose
 *    streamed run is held bit for bit to a resident run ("Limitations",
 *    section "What 0.00e+00 means").
 *  - Every linear computes y = x W'^T + (alpha/r) B A dropout(x); the
 *    backward produces gradients for the adapters and the block inputs
 *    only, never for the frozen weights ("Poros", training-step paragraph).
 *  - Frozen blocks pass through a small GPU window that is prefetched
 *    asynchronously; only block-boundary activations are kept; the backward
 *    visits the blocks in reverse, reloads each one, recomputes its forward
 *    and back-propagates ("Poros", streamed-residency and training-step
 *    paragraphs).
 *  - The recompute must draw the forward's dropout masks again ("Poros",
 *    dropout and RNG-capture paragraphs).  Here masks come from a
 *    counter-based Philox4x32-10 keyed by (seed, step, layer, linear,
 *    micro-batch), so nothing is snapshotted or restored.
 *
 * Conventions for every entry point:
 *  - Return value: ws_status (0 = WS_OK).  Argument and shape errors are
 *    reported synchronously before anything is enqueued; launch errors come
 *    back as WS_ERR_CUDA.  Nothing aborts the process; no C++ exception
 *    crosses the ABI.
 *  - Memory: the caller owns every buffer.  The library never allocates or
 *    frees device, pinned or host tensor memory; scratch is a caller-provided
 *    workspace whose size the *_workspace_size queries return.  Pointers
 *    documented as "device" must be device (or managed) memory of the current
 *    CUDA device; "pinned" means cudaHostAlloc'd / registered host memory.
 *  - Execution: all work is enqueued asynchronously on the given stream(s);
 *    no call synchronises the host except ws_device_error.  Kernels are
 *    launched with programmatic dependent launch (each waits for the
 *    previous kernel of its stream before touching data; WS_NF4_PDL=0 in
 *    the environment turns it off).  The LoRA backward forks part of its
 *    work onto a library-owned side stream and joins it back before the
 *    call's last kernel: the first such call for a (device, caller stream)
 *    pair creates that stream and two events, which live until the process
 *    exits (WS_NF4_SIDE=0 keeps everything on the caller's stream).  Under
 *    stream capture the fork and join become graph edges.
 *  - Alignment: every device pointer must be 16-byte aligned
 *    (WS_ERR_ALIGN otherwise).
 *  - Shapes: K % 64 == 0 and N % 64 == 0 for NF4 weights; M >= 1;
 *    r == 16; M*K < 2^34 for the dropout counter (WS_ERR_SHAPE otherwise).
 *  - bf16 tensors are passed as uint16_t bit patterns.
 *  - Determinism: every reduction runs in a fixed order that depends only on
 *    the shapes, so repeated calls, and a streamed versus a resident run,
 *    give bitwise identical results.
 *
 * Layouts (row-major unless stated):
 *   W (bf16)   [N, K]
 *   codes      uint8 [N, K/2]; byte j of row n holds k = 2j in the high
 *              nibble and k = 2j+1 in the low nibble
 *   absmax     fp32 [K/64, N]  (block-major: absmax[(k/64)*N + n])
 *   x, dX      [M, K];  y, dY [M, N]
 *   A          fp32 [r, K];  B fp32 [N, r]
 *   U          fp32 [M, r] = (mask . x) A^T  (saved by the forward)
 *   mask       uint32 [M, K/32]; bit (k % 32) of word (m*K + k)/32 is 1 when
 *              element (m, k) of the LoRA input is kept
 */
#ifndef WSNF4_H
#define WSNF4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ws_stream_t; /* identical to cudaStream_t */
typedef struct CUevent_st* ws_event_t;   /* identical to cudaEvent_t  */

typedef int32_t ws_status;
enum {
  WS_OK = 0,
  WS_ERR_INVALID = -1,     /* null pointer / bad enum / bad flag          */
  WS_ERR_SHAPE = -2,       /* shape outside the supported contract        */
  WS_ERR_ALIGN = -3,       /* pointer not 16-byte aligned                 */
  WS_ERR_CUDA = -4,        /* a CUDA runtime call or a launch failed      */
  WS_ERR_TIMEOUT = -5,     /* a bounded device wait gave up               */
  WS_ERR_OOM = -6,         /* caller-provided buffer or workspace too small */
  WS_ERR_UNSUPPORTED = -7, /* configuration that would break exactness    */
  WS_ERR_NOT_PINNED = -8   /* host pointer is not page-locked             */
};

enum { WS_DTYPE_BF16 = 0, WS_DTYPE_F32 = 1 };

/* Accumulation flags of ws_lora_linear_bwd. */
enum { WS_ACC_DX = 1,     /* add the input gradient into an fp32 dX          */
       WS_ACC_GRADS = 2   /* add dA and dB into the existing gradients        */
};

/* Linear ids inside a layer of the synthetic stack. */
enum { WS_LIN_Q = 0, WS_LIN_K = 1, WS_LIN_V = 2, WS_LIN_O = 3,
       WS_LIN_GATE = 4, WS_LIN_UP = 5, WS_LIN_DOWN = 6, WS_NLIN = 7 };

/* A frozen NF4 weight [N, K] (device pointers). */
typedef struct {
  const uint8_t* codes; /* [N, K/2] */
  const float* absmax;  /* [K/64, N] */
  int64_t N, K;
} ws_nf4;

/* A frozen bf16 weight [N, K], row-major (device pointer); the base of the
 * bf16 streaming mode ("Limitations", section "bf16 LoRA (EXPERIMENTAL)"). */
typedef struct {
  const uint16_t* w;
  int64_t N, K;
} ws_bf16;

/* Dropout key of one linear.  Element e = m*K + k of the LoRA input is kept
 * iff word (e & 3) of Philox4x32-10(counter = (e >> 2, linear | microbatch
 * << 8, layer, step), key = (seed_lo, seed_hi)) >= ceil(p * 2^32).
 * p in [0, 1); linear < 256, microbatch < 2^24. */
typedef struct {
  uint64_t seed;
  uint32_t step, layer, linear, microbatch;
  double p;
} ws_dropout_key;

/* Shape of one LoRA linear: x [M, K] -> y [M, N], rank r, scale alpha / r. */
typedef struct {
  int64_t M, N, K;
  int32_t r;
  float alpha;
} ws_lora_shape;

/* ---- status ------------------------------------------------------------- */

/* Human-readable name of a status code (static string, never NULL). */
const char* ws_status_string(ws_status st);

/* Reads (and clears) the library's device error word, which kernels set when
 * a bounded wait times out.  Synchronises the current device.  *flags = 0
 * means no kernel reported a problem.  Returns WS_ERR_TIMEOUT if a flag was
 * set, WS_OK otherwise.  Every wait in the library's kernels gives up after
 * one second of wall-clock time: the kernel then sets a bit below, lets its
 * copies in flight land, frees its tensor memory and returns; kernels that
 * start while the word is set skip their work, until the word is read and
 * cleared here (which also clears the library's cross-CTA words). */
enum { WS_DERR_PIPELINE_MASK = 0x3F, /* a pipeline barrier wait inside a kernel gave up  */
       WS_DERR_BAD_CONFIG = 0x40,    /* a kernel refused its launch configuration       */
       WS_DERR_TIMEOUT_PEER = 0x80   /* a wait for another CTA's published result gave up */
};
ws_status ws_device_error(uint32_t* flags);

/* Failure-detection self-check (no counterpart on the method's pages; it
 * exercises the bounded waits above).  Launches one small kernel on `stream`
 * that waits for a cross-CTA completion word that nothing sets, through the
 * same bounded wait the dequant GEMM's stream-K finisher uses, but giving up
 * after limit_us microseconds (1 .. 1000000) instead of one second.  The
 * wait gives up, sets WS_DERR_TIMEOUT_PEER and the kernel returns; the CUDA
 * context stays usable, and the next ws_device_error reports and clears it.
 * Nothing faults or traps. */
ws_status ws_selfcheck_bounded_wait(uint32_t limit_us, ws_stream_t stream);

/* Number of CUDA kernels this library has launched in the process so far
 * (host-side counter; copies are not counted). */
uint64_t ws_kernel_launches(void);

/* ---- NF4 quantisation ------------------------------------------------------ */
/* The frozen base's precision ("Limitations", section "What 0.00e+00 means";
 * the research page "Poros", block-streamed NF4 loader paragraphs, where
 * each tensor is quantised as it is loaded).
 * Quantises a bf16 weight W [N, K] (device) into NF4 codes [N, K/2] and
 * block-major absmax [K/64, N] (device, caller-allocated).
 * Per 64-block: absmax = max |w| (fp32); v = w / absmax as an IEEE fp32
 * division; code = number of the 15 midpoints mid_i = fp32(fp32(c_i +
 * c_{i+1}) * 0.5) that v exceeds (ties go to the lower level); an all-zero
 * block gives absmax 0 and code 7.  c_i are the 16 NF4 levels
 * {-1, -0.6962, -0.5251, -0.3949, -0.2844, -0.1848, -0.0911, 0, 0.0796,
 * 0.1609, 0.2461, 0.3379, 0.4407, 0.5626, 0.7230, 1} as fp32 literals.
 * Requires K % 64 == 0, N >= 1.  Dequantisation used by the GEMMs is
 * w' = bf16_RN(fp32(c[code]) * absmax), one rounding. */
ws_status ws_quantize_nf4(const uint16_t* W, int64_t N, int64_t K, uint8_t* codes,
                          float* absmax, ws_stream_t stream);

/* ---- LoRA linear forward ------------------------------------------------- */
/* Workspace (device bytes) needed by ws_lora_linear_fwd / _bwd for a shape. */
ws_status ws_lora_workspace_size(ws_lora_shape sh, size_t* bytes);

/* The forward of one NF4-LoRA linear ("Poros", training-step paragraph: the
 * frozen base is only read; the adapter sees dropout(x)).
 * y = x W'^T + s * U B^T with U = (mask . x) A^T and s = (alpha/r)/(1-p)
 * (inverted dropout folded into the scale).  W' is the NF4 weight
 * dequantised on the fly inside the tensor-core GEMM; nothing dequantised
 * is ever written to memory.
 *   x [M,K] bf16, A [r,K] fp32, B [N,r] fp32              (device, in)
 *   y [M,N] bf16                                            (device, out)
 *   U_saved [M,r] fp32                                      (device, out, required)
 *   mask_saved [M,K/32] uint32                              (device, out, may be NULL)
 *   workspace >= ws_lora_workspace_size(sh)                 (device scratch)
 * Accumulation: fp32 on the tensor cores (TMEM); the LoRA up projection is an
 * extra contraction step of the same GEMM with U and s*B split into bf16
 * high and low parts (about 16 significant bits per factor). */
ws_status ws_lora_linear_fwd(const ws_nf4* W, const uint16_t* x, const float* A,
                             const float* B, ws_lora_shape sh, ws_dropout_key key,
                             uint16_t* y, float* U_saved, uint32_t* mask_saved,
                             void* workspace, size_t ws_bytes, ws_stream_t stream);

/* The forward of ng (1..3) NF4-LoRA linears that read the same input x (a
 * layer's q, k, v, or its gate and up): the same computation per linear as
 * ws_lora_linear_fwd, in fewer, fuller launches: one LoRA-down launch draws
 * every linear's dropout mask and U, and one dequant GEMM covers their
 * concatenated outputs when every width is a multiple of the GEMM's tile
 * width (else one GEMM per linear).  Arrays are indexed by linear g < ng:
 * W[g] [N_g, K] (every K equal), A[g] [r, K], B[g] [N_g, r], keys[g],
 * y[g] [M, N_g] bf16, U_saved[g] [M, r] fp32, mask_saved[g] (entries may be
 * NULL).  sh gives M, K, r, alpha (its N is ignored).  U and y can differ in
 * the last bits from single-linear calls (the LoRA-down sums run in
 * k-chunks sized for the whole launch); a given grouping always gives the
 * same bits.  workspace >= ws_lora_group_workspace_size. */
ws_status ws_lora_group_workspace_size(int32_t ng, const int64_t* N, int64_t M, int64_t K,
                                       size_t* bytes);
ws_status ws_lora_linear_fwd_group(int32_t ng, const ws_nf4* W, const uint16_t* x,
                                   const float* const* A, const float* const* B, ws_lora_shape sh,
                                   const ws_dropout_key* keys, uint16_t* const* y,
                                   float* const* U_saved, uint32_t* const* mask_saved,
                                   void* workspace, size_t ws_bytes, ws_stream_t stream);
/* The backward of ng (1..3) linears of one shape [N, K] that read the same x
 * (a layer's k and v, or gate and up), each with its own dY[g]: G, dB and dA
 * of every linear as in ws_lora_linear_bwd, their input gradients summed into
 * one dX (linear 0 first), with the skinny products and weight gradients of
 * all ng in one launch each.  accumulate: WS_ACC_* as for ws_lora_linear_bwd;
 * dX is fp32 (WS_DTYPE_F32) whenever ng > 1.
 * workspace >= ws_lora_group_workspace_size with every N_g = N. */
ws_status ws_lora_linear_bwd_group(int32_t ng, const ws_nf4* W, const uint16_t* x,
                                   const float* const* A, const float* const* B, ws_lora_shape sh,
                                   const ws_dropout_key* keys, const float* const* U_saved,
                                   const uint32_t* const* mask_saved, const uint16_t* const* dY,
                                   void* dX, int32_t dX_dtype, int32_t accumulate,
                                   float* const* dA, float* const* dB, void* workspace,
                                   size_t ws_bytes, ws_stream_t stream);

/* ---- LoRA linear backward ------------------------------------------------ */
/* The backward of one linear: gradients for the adapters and the input only,
 * none for the frozen weight ("Poros", training-step paragraph).
 * Given dY [M,N] bf16 computes
 *   G  = dY B                              (fp32, internal)
 *   dB = s dY^T U_saved                    [N, r] fp32 (overwritten)
 *   dA = s G^T (mask . x)                  [r, K] fp32 (overwritten)
 *   dX = dY W' + s (G A) . mask            [M, K] bf16 or fp32
 * dX_dtype: WS_DTYPE_BF16 or WS_DTYPE_F32.  accumulate is a set of WS_ACC_*
 * flags: WS_ACC_DX adds into an existing fp32 dX, WS_ACC_GRADS adds dA and
 * dB into the existing gradients (gradient accumulation over micro-batches);
 * either way the new contribution is added to the old value once, in fp32,
 * after its own fixed-order sum.  mask_saved may be NULL: the masks are then
 * regenerated from `key` (bit-identical to the forward's).
 * No atomics: dA, dB and split contractions are reduced in a fixed order. */
ws_status ws_lora_linear_bwd(const ws_nf4* W, const uint16_t* x, const float* A,
                             const float* B, ws_lora_shape sh, ws_dropout_key key,
                             const float* U_saved, const uint32_t* mask_saved,
                             const uint16_t* dY, void* dX, int32_t dX_dtype,
                             int32_t accumulate, float* dA, float* dB,
                             void* workspace, size_t ws_bytes, ws_stream_t stream);

/* The same forward and backward with a bf16 base weight (the pages' bf16
 * streaming mode, "Limitations", section "bf16 LoRA (EXPERIMENTAL)"): the
 * weight tiles are loaded by TMA into the tensor-core operand layout instead
 * of being dequantised; everything else, the shapes, arguments, workspace
 * and errors, is that of ws_lora_linear_fwd / _bwd. */
ws_status ws_lora_linear_fwd_bf16(const ws_bf16* W, const uint16_t* x, const float* A,
                                  const float* B, ws_lora_shape sh, ws_dropout_key key,
                                  uint16_t* y, float* U_saved, uint32_t* mask_saved,
                                  void* workspace, size_t ws_bytes, ws_stream_t stream);
ws_status ws_lora_linear_bwd_bf16(const ws_bf16* W, const uint16_t* x, const float* A,
                                  const float* B, ws_lora_shape sh, ws_dropout_key key,
                                  const float* U_saved, const uint32_t* mask_saved,
                                  const uint16_t* dY, void* dX, int32_t dX_dtype,
                                  int32_t accumulate, float* dA, float* dB, void* workspace,
                                  size_t ws_bytes, ws_stream_t stream);

/* ---- the frozen NF4 product alone ---------------------------------------------- */
/* The dequant GEMM of the LoRA linear without adapter or dropout (a frozen NF4
 * linear; the base term of the training-step paragraph of "Poros"):
 *   transpose_w == 0:  out[M,N] = act[M,K] W'^T   (forward)
 *   transpose_w != 0:  out[M,K] = act[M,N] W'     (input gradient)
 * act bf16 (device); out bf16 or fp32 (out_dtype) (device); workspace >=
 * ws_nf4_matmul_workspace_size() (device scratch for contraction splits). */
ws_status ws_nf4_matmul_workspace_size(int64_t M, int64_t N, int64_t K, int32_t transpose_w,
                                       size_t* bytes);
ws_status ws_nf4_matmul(const ws_nf4* W, const uint16_t* act, int64_t M, int32_t transpose_w,
                        void* out, int32_t out_dtype, void* workspace, size_t ws_bytes,
                        ws_stream_t stream);

/* Allocation-free variant of ws_nf4_matmul (no counterpart on the method's
 * pages; an addition for callers that cannot allocate device memory).
 *
 * Some callers cannot call cudaMalloc or hand out a workspace: code that runs
 * under a host framework whose allocator owns all device memory, plugins
 * with no allocation hooks, or paths that must not allocate at all once
 * running.  This entry point takes only the inputs and the output; the
 * scratch it needs (fp32 partial tiles of a split contraction and their
 * completion flags) lives in a
 * file-scope device array of WS_NOALLOC_SCRATCH_BYTES (48 MiB) inside the
 * library, which every GPU that loads the library holds until the process
 * exits.  Only the partial tiles live in that array; the completion flags
 * of the split come from the library's shared ring of cross-CTA words,
 * which every launch of the library uses and leaves at zero.  Nothing is
 * allocated or freed by the call.
 *  - The first call on a device looks up that device's address of the
 *    array, and of the flag ring, with cudaGetSymbolAddress (once per
 *    device, with the device current); make that first call before any
 *    stream capture.
 *  - Every call shares the one array: calls that overlap on the GPU (other
 *    streams, other host threads) race on it and must be serialised by the
 *    caller.  Each call overwrites all scratch it reads, so no clearing is
 *    needed between calls.
 *  - A shape whose split partials would exceed the array returns
 *    WS_ERR_OOM before anything is enqueued (ws_nf4_matmul_workspace_size
 *    gives the bytes a shape needs).
 * Arguments, layouts and results are those of ws_nf4_matmul. */
#define WS_NOALLOC_SCRATCH_BYTES (48u << 20)
ws_status ws_nf4_matmul_noalloc(const ws_nf4* W, const uint16_t* act, int64_t M,
                                int32_t transpose_w, void* out, int32_t out_dtype,
                                ws_stream_t stream);

/* ---- attention core ---------------------------------------------------------- */
/* The attention of the trained model, which streaming leaves unchanged (the
 * research page "Poros", the paragraph saying the learning problem itself is
 * unchanged).  The pages print no formula; this is scaled dot-product
 * attention (Vaswani et al., 2017), causal, with grouped kv heads (Ainslie et
 * al., 2023): query head h reads kv head h / (n_heads / n_kv_heads).
 * Tokens are n_seq sequences of seq_len, token t = b*seq_len + i, M =
 * n_seq*seq_len.  All pointers are device memory, 16-byte aligned:
 *   q [M, n_heads*head_dim], k and v [M, n_kv_heads*head_dim]   bf16
 *   o [M, n_heads*head_dim] bf16 and, if o32 != NULL, the same in fp32
 *   lse [n_heads, M] fp32: ln sum_{j<=i} exp(q_i.k_j / sqrt(head_dim))
 *   o_i = sum_{j<=i} exp(q_i.k_j / sqrt(head_dim) - lse_i) v_j.
 * head_dim is 64 or 128; n_heads a multiple of n_kv_heads; seq_len >= 1.
 * The probabilities enter the tensor-core products as two bf16 parts (about
 * 16 significant bits); every sum has a fixed order, so results repeat bit
 * for bit.  WS_ERR_SHAPE / WS_ERR_ALIGN / WS_ERR_INVALID on bad arguments,
 * before anything is launched. */
ws_status ws_attention_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           int32_t n_seq, int32_t seq_len, int32_t n_heads, int32_t n_kv_heads,
                           int32_t head_dim, uint16_t* o, float* o32, float* lse,
                           ws_stream_t stream);
/* Workspace of ws_attention_bwd for M = n_seq*seq_len tokens. */
ws_status ws_attention_workspace_size(int64_t M, int32_t n_heads, int32_t head_dim, size_t* bytes);
/* Gradients for the upstream gradient dO [M, n_heads*head_dim] bf16, given the
 * forward's o32 and lse: dq [M, n_heads*head_dim], dk and dv [M,
 * n_kv_heads*head_dim], bf16 (overwritten).  With p the probabilities,
 * D_i = dO_i . o_i, ds_ij = p_ij (dO_i . v_j - D_i): dq_i = sum_j ds_ij k_j /
 * sqrt(head_dim), dk_j = sum_i ds_ij q_i / sqrt(head_dim), dv_j = sum_i p_ij
 * dO_i, dk and dv summed over the query heads sharing the kv head (in head
 * order).  workspace: device, ws_attention_workspace_size bytes. */
ws_status ws_attention_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           const float* o32, const float* lse, const uint16_t* dO,
                           int32_t n_seq, int32_t seq_len, int32_t n_heads, int32_t n_kv_heads,
                           int32_t head_dim, uint16_t* dq, uint16_t* dk, uint16_t* dv,
                           void* workspace, size_t workspace_bytes, ws_stream_t stream);

/* ---- the synthetic stack ----------------------------------------------------- */
/* The transformer layers the method trains ("Poros", learning-problem
 * paragraph: the layer computation is that of a resident run).  One layer:
 * h -> RMSNorm -> q,k,v (NF4-LoRA) -> attention -> o -> residual; -> RMSNorm
 * -> gate, up -> SiLU(gate)*up -> down -> residual.  The attention is
 *   attn = WS_ATTN_REPEAT_V: v repeated across the H/head_dim query heads
 *          (head h reads kv head h / (H/KV)) in place of the attention core;
 *          q and k then feed nothing, so their adapters receive exactly zero
 *          gradient;
 *   attn = WS_ATTN_CAUSAL: the causal attention core above (ws_attention_fwd)
 *          over the M tokens as one sequence, with H/head_dim query heads
 *          and KV/head_dim kv heads (head_dim 64 or 128).
 * RMSNorm has unit gain and eps `eps`, computed in fp32; the residual stream
 * is fp32; linear inputs and outputs are bf16; gradients that enter a linear
 * as dY are bf16 (with the attention core also the o projection's input
 * gradient dO, and dq, dk, dv), all other activation gradients are fp32.
 * loss = 0.5 mean(h_L^2). */
enum { WS_BASE_NF4 = 0, WS_BASE_BF16 = 1 };
enum { WS_ATTN_REPEAT_V = 0, WS_ATTN_CAUSAL = 1 };
typedef struct {
  int64_t M, H, KV, I, head_dim;
  int32_t n_layers;
  int32_t r;
  float alpha;
  double p;
  float eps;
  uint64_t seed;
  int32_t base;  /* the frozen base's format: WS_BASE_NF4, or WS_BASE_BF16
                    (the pages' bf16_bitwise mode: same engine and GEMM, the
                    weights stream as bf16, 2 bytes per weight) */
  int32_t attn;  /* WS_ATTN_REPEAT_V or WS_ATTN_CAUSAL */
} ws_stack_cfg;

/* Sizes of the stack's buffers for a given block size (layers per block):
 *   block_weight_bytes : base-weight bytes of one block (one window slot)
 *   n_params           : fp32 LoRA parameters of the whole stack (A then B
 *                        of every linear, see ws_stack_param_offset)
 *   saved_bytes_layer  : activations one layer keeps for its backward
 *   workspace_bytes    : scratch for block_forward / block_backward_recompute
 *                        (includes one block of recompute storage) */
ws_status ws_stack_sizes(const ws_stack_cfg* cfg, int32_t block_layers,
                         size_t* block_weight_bytes, int64_t* n_params,
                         size_t* saved_bytes_layer, size_t* workspace_bytes);

/* Offsets inside a block's image of layer `layer_in_block`, linear `lin`:
 * NF4 base: codes at byte *off_codes, absmax at byte *off_absmax (both
 * 256-aligned); bf16 base: the weight W [N, K] at *off_codes (256-aligned),
 * and *off_absmax = *off_codes. */
ws_status ws_stack_weight_offset(const ws_stack_cfg* cfg, int32_t layer_in_block, int32_t lin,
                                 size_t* off_codes, size_t* off_absmax);

/* Activations one layer keeps for its backward (the `saved` areas of
 * ws_block_forward / ws_stack_buffers, one slot of saved_bytes_layer per
 * layer): the layer input h [M,H] fp32, a = RMSNorm(h) [M,H] bf16, rstd1 [M]
 * fp32, v [M,KV] bf16, vr = the attention output (repeat(v), or the
 * attention core's o) [M,H] bf16, h1 = h + o [M,H] fp32, b = RMSNorm(h1)
 * [M,H] bf16, rstd2 [M] fp32, gate and up outputs [M,I] bf16, act =
 * SiLU(gate)*up [M,I] bf16, and per linear its U [M,16] fp32 and dropout
 * mask [M,K/32] uint32.  With the attention core also q [M,H] and k [M,KV]
 * bf16, the attention output in fp32 [M,H] and its log-sum-exp [H/head_dim,
 * M] fp32 (zero bytes otherwise). */
enum { WS_SV_H = 0, WS_SV_A = 1, WS_SV_RSTD1 = 2, WS_SV_V = 3, WS_SV_VR = 4, WS_SV_H1 = 5,
       WS_SV_B = 6, WS_SV_RSTD2 = 7, WS_SV_GATE = 8, WS_SV_UP = 9, WS_SV_ACT = 10,
       WS_SV_LORA_U = 11, WS_SV_MASK = 12, WS_SV_Q = 13, WS_SV_K = 14, WS_SV_O32 = 15,
       WS_SV_LSE = 16 };

/* Byte offset of field `field` (for WS_SV_LORA_U / WS_SV_MASK: of linear
 * `lin`) inside one layer's saved slot. */
ws_status ws_stack_saved_offset(const ws_stack_cfg* cfg, int32_t field, int32_t lin,
                                size_t* offset);

/* The streamed NF4 loader ("Poros", block-streamed NF4 loader paragraphs:
 * one tensor is staged at a time, quantised and evicted before the next, so
 * the whole base never sits on the GPU, and the result is byte-identical to a
 * standard load).  For an NF4 base, ws_stack_put_weight quantises one bf16 weight
 * W [N, K] (device; (N, K) must be linear `lin`'s shape) of layer `layer`
 * into its place in a stack image that holds all n_layers / block_layers
 * blocks back to back:
 *   image on the device: quantised straight into place;
 *   image in pinned host memory: quantised into `staging` (device, at least
 *   ws_stack_loader_staging_bytes) and copied from there with
 *   cudaMemcpyAsync on `stream` (the copy reads staging, so a later call on
 *   the same stream may reuse it; a call on another stream may not until
 *   this one's copy has completed).
 * The caller feeds the tensors one at a time (its own W buffer can be freed
 * or refilled after the call's work on `stream` is done), so the GPU holds
 * one bf16 tensor and one tensor's NF4 at a time.  Bytes between the
 * 256-aligned pieces of the image are not written: zero the image first for
 * a byte-comparable result.  Errors: WS_ERR_SHAPE for a wrong (N, K),
 * WS_ERR_OOM for a staging buffer too small, WS_ERR_INVALID for a layer or
 * linear out of range, WS_ERR_NOT_PINNED for a host image that is not
 * page-locked.  For a bf16 base the weight is copied into place as it is
 * (cudaMemcpyAsync; no staging is used, `staging` may be NULL). */
ws_status ws_stack_loader_staging_bytes(const ws_stack_cfg* cfg, size_t* bytes);
ws_status ws_stack_put_weight(const ws_stack_cfg* cfg, int32_t block_layers, int32_t layer,
                              int32_t lin, const uint16_t* W, int64_t N, int64_t K, void* image,
                              void* staging, size_t staging_bytes, ws_stream_t stream);

/* Offsets (in floats) of A [r, K] and B [N, r] of (layer, lin) in the
 * parameter arrays (params, grads and both Adam moments share the layout). */
ws_status ws_stack_param_offset(const ws_stack_cfg* cfg, int32_t layer, int32_t lin,
                                int64_t* off_A, int64_t* off_B);

/* Intermediate gradients of a layer's backward inside the stack workspace
 * (for inspection; after ws_block_backward_recompute they hold the values of
 * the block's first layer, the last one processed):
 *   WS_WK_Y1    bf16 [M,H]  bf16(dh1), the o projection's dY
 *   WS_WK_DACT  fp32 [M,I]  gradient at act (the down projection's dX)
 *   WS_WK_DG, WS_WK_DU  bf16 [M,I]  gradients at the gate and up outputs
 *   WS_WK_DB    fp32 [M,H]  gradient at b (sum of the gate and up dX)
 *   WS_WK_DH1   fp32 [M,H]  gradient at h1 (layer output gradient + RMSNorm2 backward)
 *   WS_WK_DVR   fp32 [M,H]  gradient at repeat(v) (the o projection's dX;
 *                           repeat(v) stack only)
 *   WS_WK_DV    bf16 [M,KV] gradient at v (sum over the query heads of each kv head)
 *   WS_WK_DA    fp32 [M,H]  gradient at a (the v projection's dX, plus the k and q
 *                           projections' with the attention core)
 *   WS_WK_YOUT  bf16 [M,H]  the last forward linear output (the down projection's y)
 *   WS_WK_DO    bf16 [M,H]  gradient at the attention output (the o projection's dX;
 *                           attention core only)
 *   WS_WK_DQ    bf16 [M,H]  gradient at q (attention core only)
 *   WS_WK_DK    bf16 [M,KV] gradient at k (attention core only) */
enum { WS_WK_Y1 = 0, WS_WK_DACT = 1, WS_WK_DG = 2, WS_WK_DU = 3, WS_WK_DB = 4, WS_WK_DH1 = 5,
       WS_WK_DVR = 6, WS_WK_DV = 7, WS_WK_DA = 8, WS_WK_YOUT = 9, WS_WK_DO = 10,
       WS_WK_DQ = 11, WS_WK_DK = 12 };
ws_status ws_stack_workspace_offset(const ws_stack_cfg* cfg, int32_t block_layers, int32_t field,
                                    size_t* offset);

/* The forward of one block ("Poros", streamed-residency paragraph: a block
 * is loaded, run forward, and only its boundary activation is kept).
 * Forward of layers [first_layer, first_layer + n_layers) whose NF4
 * weights are the block image at `block_weights` (device).  h_in / h_out
 * [M, H] fp32 (device; may not alias).  params: device LoRA parameters.
 * saved: device area of n_layers * saved_bytes_layer that receives every
 * activation the backward needs (resident mode), or NULL to keep nothing
 * (streamed mode: only h_out survives).  step and microbatch key the
 * dropout masks. */
ws_status ws_block_forward(const ws_stack_cfg* cfg, const void* block_weights,
                           int32_t first_layer, int32_t n_layers, const float* params,
                           uint32_t step, uint32_t microbatch, const float* h_in, float* h_out,
                           void* saved, void* workspace, size_t ws_bytes, ws_stream_t stream);

/* The backward of one block ("Poros", streamed-residency and RNG-capture
 * paragraphs: the block is reloaded, its forward recomputed with the same
 * dropout, then differentiated for the adapters and the block input).
 * Backward of the same layers.  If `saved` is NULL the block's forward is
 * first recomputed from the boundary activation h_in (same kernels, same
 * Philox keys, hence bit-identical intermediates) into the workspace; if
 * `saved` is the area ws_block_forward filled, it is used directly
 * (resident mode).  dh_out [M,H] fp32 is the gradient at the block output;
 * dh_in (may alias dh_out) receives the gradient at the block input.
 * grads: device LoRA gradients (same layout as params); the block's entries
 * are overwritten, or, with grad_accumulate != 0, added to (gradient
 * accumulation over micro-batches). */
ws_status ws_block_backward_recompute(const ws_stack_cfg* cfg, const void* block_weights,
                                      int32_t first_layer, int32_t n_layers,
                                      const float* params, uint32_t step, uint32_t microbatch,
                                      const float* h_in, const void* saved, const float* dh_out,
                                      float* dh_in, float* grads, int32_t grad_accumulate,
                                      void* workspace, size_t ws_bytes, ws_stream_t stream);

/* The window's prefetch ("Poros", training-step paragraph: frozen blocks pass
 * through a small GPU window, prefetched asynchronously on CUDA streams).
 * Copy one block (bytes) from pinned host memory to a device window slot
 * on `copy_stream`.  If wait_event is not NULL the copy first waits for it
 * (the slot's previous user is done); if done_event is not NULL it is
 * recorded after the copy.  A pageable source gives WS_ERR_NOT_PINNED. */
ws_status ws_stream_block_h2d(const void* pinned_src, void* dev_dst, size_t bytes,
                              ws_stream_t copy_stream, ws_event_t wait_event,
                              ws_event_t done_event);

/* ---- one training step ---------------------------------------------------------- */
typedef struct {
  const void* host_weights; /* pinned: all blocks back to back (streamed), else NULL */
  const void* dev_weights;  /* device: all blocks back to back (resident), else NULL */
  void* window;             /* device: 2 * block_weight_bytes (streamed)              */
  float* params;            /* device: n_params LoRA parameters                       */
  float* grads;             /* device: n_params                                        */
  float* adam_m;            /* device: n_params, first moment                          */
  float* adam_v;            /* device: n_params, second moment                         */
  float* boundary;          /* device: n_micro * (n_blocks + 1) * M * H fp32 block-boundary h */
  void* saved;              /* device: n_layers * saved_bytes_layer (resident), else NULL */
  float* dh;                /* device: max(2, n_micro) * M * H fp32 gradients            */
  void* workspace;          /* device: workspace_bytes                                  */
  size_t workspace_bytes;
  float* loss;              /* device: 1 float, receives the loss                      */
} ws_stack_buffers;

/* One training step ("Poros", training-step paragraph: streamed forward,
 * reverse-order reload-recompute-backward, then one optimizer step equal to
 * a resident run's).
 * One full training step of the stack: forward over the blocks, loss,
 * backward over the blocks in reverse, one Adam step (PyTorch defaults:
 * betas 0.9 / 0.999, eps 1e-8, bias-corrected, no weight decay) with
 * learning rate lr at Adam step t = step + 1.
 * streamed != 0: weights come from host_weights through the 2-slot window;
 *   block b+1's copy (copy_stream) overlaps block b's compute, the backward
 *   reloads blocks in reverse and recomputes each from its boundary
 *   activation (saved must be NULL).
 * streamed == 0: weights are read from dev_weights and every intermediate
 *   is kept in `saved` (no recompute).
 * Both modes run the same kernels in the same order on the same data, so
 * loss, gradients, parameters and Adam moments are bitwise identical.
 * h0 [M, H] fp32 (device) is the step's input.  Enqueued on `compute`;
 * returns without waiting for the GPU. */
ws_status ws_stack_train_step(const ws_stack_cfg* cfg, int32_t block_layers, int32_t streamed,
                              const ws_stack_buffers* buf, uint32_t step, const float* h0,
                              float lr, ws_stream_t compute, ws_stream_t copy_stream);

/* Gradient accumulation ("Poros", block-major and parity-gate paragraphs:
 * the pages run accumulation at 2 and 4 micro-batches and refuse the
 * block-major order with dropout, because their sequential RNG would be
 * consumed in another order).  Here every micro-batch has its own dropout
 * keys (the micro-batch index is in the Philox counter), so the order in
 * which micro-batches and blocks are visited changes nothing:
 *   WS_GA_MICROBATCH_MAJOR  forward and backward of micro-batch 0, then 1, ...;
 *   WS_GA_BLOCK_MAJOR       (streamed) each block is loaded once per
 *                           direction and every micro-batch runs through it.
 * The step loss is the mean of the micro-batch losses; adapter gradients are
 * summed in micro-batch order (micro-batch 0 writes, the others add), so
 * both orders and a resident run are bitwise identical.  A resident run
 * ignores `order`.  h0 holds n_micro inputs [n_micro, M, H]; the buffers
 * grow as ws_stack_buffers states.
 * time_copies != 0 (graphs of streamed steps only) records timing events
 * around every block copy; ws_stack_graph_copy_times reads them.
 * copy_piece_bytes > 0 issues each block copy as consecutive
 * cudaMemcpyAsync pieces of that size (a multiple of 256) instead of one
 * copy; results are the same. */
enum { WS_GA_MICROBATCH_MAJOR = 0, WS_GA_BLOCK_MAJOR = 1 };
typedef struct {
  int32_t n_micro;           /* micro-batches per step, >= 1 */
  int32_t order;             /* WS_GA_*                       */
  int32_t time_copies;       /* 0 or 1                        */
  int32_t reserved;          /* 0                             */
  int64_t copy_piece_bytes;  /* 0: one copy per block         */
} ws_step_opts;
/* opts == NULL: one micro-batch, no timing (ws_stack_train_step). */
ws_status ws_stack_train_step_ex(const ws_stack_cfg* cfg, int32_t block_layers, int32_t streamed,
                                 const ws_step_opts* opts, const ws_stack_buffers* buf,
                                 uint32_t step, const float* h0, float lr, ws_stream_t compute,
                                 ws_stream_t copy_stream);

/* ---- the same step as one CUDA graph ---------------------------------------------
 * ws_stack_graph_create captures everything ws_stack_train_step enqueues
 * after its first two operations (writing `step` into a device word inside
 * the workspace, copying h0 into boundary block 0) into one graph: every
 * block's kernels, the window copies on copy_stream (forked from and joined
 * back into `compute` inside the graph), the loss and the Adam step.
 * Streamed: a second capture starts from the window the previous step left
 * (blocks 0 and 1 in slots 0 and 1) and skips their two copies; the first
 * ws_stack_graph_step replays the full capture, every later one the second,
 * so the window must not be written between steps of one graph.
 * Kernels that depend on the step (dropout keys, Adam bias corrections) read
 * it from that device word, so replays with different steps need no
 * re-capture.  The graph keeps the pointers of *buf, the config, lr and the
 * copy stream; they must stay valid until ws_stack_graph_destroy.  `compute`
 * must not be capturing already and may not be the legacy default stream.
 * ws_stack_graph_step(g, step, h0, compute) enqueues the step-word write,
 * the h0 copy and the graph on `compute`; results are bitwise those of
 * ws_stack_train_step with the same arguments.  Errors: the checks of
 * ws_stack_train_step, WS_ERR_CUDA when capture or instantiation fails
 * (*out stays NULL). */
typedef struct ws_step_graph ws_step_graph;
ws_status ws_stack_graph_create(const ws_stack_cfg* cfg, int32_t block_layers, int32_t streamed,
                                const ws_stack_buffers* buf, float lr, ws_stream_t compute,
                                ws_stream_t copy_stream, ws_step_graph** out);
ws_status ws_stack_graph_create_ex(const ws_stack_cfg* cfg, int32_t block_layers, int32_t streamed,
                                   const ws_step_opts* opts, const ws_stack_buffers* buf, float lr,
                                   ws_stream_t compute, ws_stream_t copy_stream,
                                   ws_step_graph** out);
/* Durations (ms) of the block copies of the graph's last replay, in issue
 * order, from the timing events of a graph created with time_copies: *n
 * receives their number, the first `capacity` go to ms.  Waits for the
 * replay's last copy.  WS_ERR_INVALID if the graph times no copies or has
 * not been replayed. */
ws_status ws_stack_graph_copy_times(ws_step_graph* g, float* ms, int32_t capacity, int32_t* n);
ws_status ws_stack_graph_step(ws_step_graph* g, uint32_t step, const float* h0,
                              ws_stream_t compute);
ws_status ws_stack_graph_destroy(ws_step_graph* g);

#ifdef __cplusplus
}
#endif
#endif /* WSNF4_H */
