"""Thin ctypes binding of libwsnf4.so (C ABI in include/wsnf4.h).

Argument marshalling only: every function here forwards torch tensors'
device pointers and the current CUDA stream to the entry point of the same
name (without the ``ws_`` prefix) and raises ``WsError`` on a non-zero
status.  PyTorch provides device memory, pinned host memory and streams;
all arithmetic runs in the library's CUDA kernels.  Importing this module
loads the library and fails loudly if it has not been built -- there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import dataclasses
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libwsnf4.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`"
        " (nvcc, sm_103a); there is no non-CUDA fallback")
_lib = C.CDLL(LIB_PATH)

P = C.c_void_p
i32, i64, u32, u64 = C.c_int32, C.c_int64, C.c_uint32, C.c_uint64

WS_DTYPE_BF16, WS_DTYPE_F32 = 0, 1
WS_ACC_DX, WS_ACC_GRADS = 1, 2
GA_MICROBATCH_MAJOR, GA_BLOCK_MAJOR = 0, 1
LIN = dict(q=0, k=1, v=2, o=3, gate=4, up=5, down=6)
LIN_NAMES = ("q", "k", "v", "o", "gate", "up", "down")


class WsError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        msg = _lib.ws_status_string(status).decode()
        super().__init__(f"{fn}: {msg} ({status})")


class Nf4(C.Structure):
    _fields_ = [("codes", P), ("absmax", P), ("N", i64), ("K", i64)]


class DropoutKey(C.Structure):
    _fields_ = [("seed", u64), ("step", u32), ("layer", u32), ("linear", u32),
                ("microbatch", u32), ("p", C.c_double)]


class LoraShape(C.Structure):
    _fields_ = [("M", i64), ("N", i64), ("K", i64), ("r", i32), ("alpha", C.c_float)]


class Bf16W(C.Structure):
    _fields_ = [("w", P), ("N", i64), ("K", i64)]


BASE_NF4, BASE_BF16 = 0, 1
ATTN_REPEAT_V, ATTN_CAUSAL = 0, 1


class StackCfgC(C.Structure):
    _fields_ = [("M", i64), ("H", i64), ("KV", i64), ("I", i64), ("head_dim", i64),
                ("n_layers", i32), ("r", i32), ("alpha", C.c_float), ("p", C.c_double),
                ("eps", C.c_float), ("seed", u64), ("base", i32), ("attn", i32)]


class StepOptsC(C.Structure):
    _fields_ = [("n_micro", i32), ("order", i32), ("time_copies", i32), ("reserved", i32),
                ("copy_piece_bytes", i64)]


class StackBuffersC(C.Structure):
    _fields_ = [("host_weights", P), ("dev_weights", P), ("window", P), ("params", P),
                ("grads", P), ("adam_m", P), ("adam_v", P), ("boundary", P), ("saved", P),
                ("dh", P), ("workspace", P), ("workspace_bytes", C.c_size_t), ("loss", P)]


def _sig(name, args):
    f = getattr(_lib, name)
    f.restype = i32
    f.argtypes = args
    return f


_lib.ws_status_string.restype = C.c_char_p
_lib.ws_status_string.argtypes = [i32]
_sig("ws_device_error", [C.POINTER(u32)])
_sig("ws_selfcheck_bounded_wait", [u32, P])
_lib.ws_kernel_launches.restype = u64
_lib.ws_kernel_launches.argtypes = []
_sig("ws_quantize_nf4", [P, i64, i64, P, P, P])
_sig("ws_lora_workspace_size", [LoraShape, C.POINTER(C.c_size_t)])
_sig("ws_lora_linear_fwd", [C.POINTER(Nf4), P, P, P, LoraShape, DropoutKey, P, P, P, P,
                            C.c_size_t, P])
_sig("ws_lora_linear_bwd", [C.POINTER(Nf4), P, P, P, LoraShape, DropoutKey, P, P, P, P, i32,
                            i32, P, P, P, C.c_size_t, P])
_sig("ws_lora_linear_fwd_bf16", [C.POINTER(Bf16W), P, P, P, LoraShape, DropoutKey, P, P, P, P,
                                 C.c_size_t, P])
_sig("ws_lora_linear_bwd_bf16", [C.POINTER(Bf16W), P, P, P, LoraShape, DropoutKey, P, P, P, P, i32,
                                 i32, P, P, P, C.c_size_t, P])
_sig("ws_nf4_matmul_workspace_size", [i64, i64, i64, i32, C.POINTER(C.c_size_t)])
_sig("ws_nf4_matmul", [C.POINTER(Nf4), P, i64, i32, P, i32, P, C.c_size_t, P])
_sig("ws_nf4_matmul_noalloc", [C.POINTER(Nf4), P, i64, i32, P, i32, P])
_sig("ws_lora_group_workspace_size", [i32, P, i64, i64, C.POINTER(C.c_size_t)])
_sig("ws_lora_linear_fwd_group", [i32, P, P, P, P, LoraShape, P, P, P, P, P, C.c_size_t, P])
_sig("ws_lora_linear_bwd_group", [i32, P, P, P, P, LoraShape, P, P, P, P, P, i32, i32, P, P, P,
                                  C.c_size_t, P])
_sig("ws_attention_fwd", [P, P, P, i32, i32, i32, i32, i32, P, P, P, P])
_sig("ws_attention_workspace_size", [i64, i32, i32, C.POINTER(C.c_size_t)])
_sig("ws_attention_bwd", [P, P, P, P, P, P, i32, i32, i32, i32, i32, P, P, P, P, C.c_size_t, P])
_sig("ws_stack_sizes", [C.POINTER(StackCfgC), i32, C.POINTER(C.c_size_t), C.POINTER(i64),
                        C.POINTER(C.c_size_t), C.POINTER(C.c_size_t)])
_sig("ws_stack_weight_offset", [C.POINTER(StackCfgC), i32, i32, C.POINTER(C.c_size_t),
                                C.POINTER(C.c_size_t)])
_sig("ws_stack_param_offset", [C.POINTER(StackCfgC), i32, i32, C.POINTER(i64), C.POINTER(i64)])
_sig("ws_stack_saved_offset", [C.POINTER(StackCfgC), i32, i32, C.POINTER(C.c_size_t)])
_sig("ws_stack_workspace_offset", [C.POINTER(StackCfgC), i32, i32, C.POINTER(C.c_size_t)])
_sig("ws_stack_loader_staging_bytes", [C.POINTER(StackCfgC), C.POINTER(C.c_size_t)])
_sig("ws_stack_put_weight", [C.POINTER(StackCfgC), i32, i32, i32, P, i64, i64, P, P, C.c_size_t, P])
_sig("ws_block_forward", [C.POINTER(StackCfgC), P, i32, i32, P, u32, u32, P, P, P, P, C.c_size_t,
                          P])
_sig("ws_block_backward_recompute", [C.POINTER(StackCfgC), P, i32, i32, P, u32, u32, P, P, P, P,
                                     P, i32, P, C.c_size_t, P])
_sig("ws_stream_block_h2d", [P, P, C.c_size_t, P, P, P])
_sig("ws_stack_train_step", [C.POINTER(StackCfgC), i32, i32, C.POINTER(StackBuffersC), u32, P,
                             C.c_float, P, P])
_sig("ws_stack_graph_create", [C.POINTER(StackCfgC), i32, i32, C.POINTER(StackBuffersC), C.c_float,
                               P, P, C.POINTER(P)])
_sig("ws_stack_train_step_ex", [C.POINTER(StackCfgC), i32, i32, C.POINTER(StepOptsC),
                                C.POINTER(StackBuffersC), u32, P, C.c_float, P, P])
_sig("ws_stack_graph_create_ex", [C.POINTER(StackCfgC), i32, i32, C.POINTER(StepOptsC),
                                  C.POINTER(StackBuffersC), C.c_float, P, P, C.POINTER(P)])
_sig("ws_stack_graph_copy_times", [P, C.POINTER(C.c_float), i32, C.POINTER(i32)])
_sig("ws_stack_graph_step", [P, u32, P, P])
_sig("ws_stack_graph_destroy", [P])

EXPORTED = ("ws_status_string", "ws_device_error", "ws_selfcheck_bounded_wait", "ws_kernel_launches", "ws_quantize_nf4", "ws_lora_workspace_size",
            "ws_lora_linear_fwd", "ws_lora_linear_bwd", "ws_lora_linear_fwd_bf16",
            "ws_lora_linear_bwd_bf16", "ws_nf4_matmul_workspace_size",
            "ws_nf4_matmul", "ws_nf4_matmul_noalloc", "ws_lora_group_workspace_size",
            "ws_lora_linear_fwd_group", "ws_lora_linear_bwd_group", "ws_attention_fwd",
            "ws_attention_workspace_size", "ws_attention_bwd", "ws_stack_sizes",
            "ws_stack_weight_offset", "ws_stack_param_offset", "ws_stack_saved_offset",
            "ws_stack_workspace_offset", "ws_stack_loader_staging_bytes", "ws_stack_put_weight",
            "ws_block_forward", "ws_block_backward_recompute",
            "ws_stream_block_h2d", "ws_stack_train_step", "ws_stack_train_step_ex",
            "ws_stack_graph_create", "ws_stack_graph_create_ex", "ws_stack_graph_copy_times",
            "ws_stack_graph_step", "ws_stack_graph_destroy")


def _check(fn, st):
    if st != 0:
        raise WsError(fn, st)


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def status_string(st: int) -> str:
    return _lib.ws_status_string(st).decode()


def kernel_launches() -> int:
    """Kernels launched by the library in this process so far."""
    return int(_lib.ws_kernel_launches())


def device_error() -> int:
    """Reads and clears the device error word (0 = no kernel timed out)."""
    f = u32(0)
    st = _lib.ws_device_error(C.byref(f))
    if st not in (0, -5):
        raise WsError("ws_device_error", st)
    return int(f.value)


WS_DERR_PIPELINE_MASK, WS_DERR_BAD_CONFIG, WS_DERR_TIMEOUT_PEER = 0x3F, 0x40, 0x80


def selfcheck_bounded_wait(limit_us: int, stream=None):
    """Enqueue the bounded-wait self-check (a wait that gives up after limit_us)."""
    _check("ws_selfcheck_bounded_wait", _lib.ws_selfcheck_bounded_wait(limit_us, _stream(stream)))


# ------------------------------------------------------------------------------ a0
def quantize_nf4(W: torch.Tensor, codes: torch.Tensor = None, absmax: torch.Tensor = None,
                 stream=None):
    """W: bf16 [N, K] (device) -> (codes uint8 [N, K/2], absmax fp32 [K/64, N])."""
    N, K = W.shape
    if codes is None:
        codes = torch.empty((N, K // 2), dtype=torch.uint8, device=W.device)
    if absmax is None:
        absmax = torch.empty((K // 64, N), dtype=torch.float32, device=W.device)
    _check("ws_quantize_nf4", _lib.ws_quantize_nf4(_ptr(W), N, K, _ptr(codes), _ptr(absmax),
                                                   _stream(stream)))
    return codes, absmax


# ------------------------------------------------------------------------------ linear
@dataclasses.dataclass
class NF4Weight:
    codes: torch.Tensor   # uint8 [N, K/2]
    absmax: torch.Tensor  # fp32 [K/64, N]
    N: int
    K: int

    def c(self):
        return Nf4(self.codes.data_ptr(), self.absmax.data_ptr(), self.N, self.K)


@dataclasses.dataclass
class Bf16Weight:
    """A frozen bf16 base weight W [N, K] (device)."""
    w: torch.Tensor
    N: int
    K: int

    def c(self):
        return Bf16W(self.w.data_ptr(), self.N, self.K)


def dropout_key(seed=0, step=0, layer=0, linear=0, microbatch=0, p=0.1):
    return DropoutKey(seed, step, layer, linear, microbatch, float(p))


def lora_workspace_size(M, N, K, r=16) -> int:
    n = C.c_size_t(0)
    _check("ws_lora_workspace_size",
           _lib.ws_lora_workspace_size(LoraShape(M, N, K, r, 32.0), C.byref(n)))
    return int(n.value)


def lora_linear_fwd(W: NF4Weight, x, A, B, key: DropoutKey, alpha=32.0, y=None, U=None,
                    mask=None, workspace=None, stream=None, keep_mask=True):
    M, K = x.shape
    sh = LoraShape(M, W.N, W.K, A.shape[0], alpha)
    dev = x.device
    if y is None:
        y = torch.empty((M, W.N), dtype=torch.bfloat16, device=dev)
    if U is None:
        U = torch.empty((M, A.shape[0]), dtype=torch.float32, device=dev)
    if mask is None and keep_mask:
        mask = torch.empty((M, K // 32), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(lora_workspace_size(M, W.N, W.K), dtype=torch.uint8, device=dev)
    w = W.c()
    fn = "ws_lora_linear_fwd_bf16" if isinstance(W, Bf16Weight) else "ws_lora_linear_fwd"
    _check(fn, getattr(_lib, fn)(C.byref(w), _ptr(x), _ptr(A), _ptr(B), sh, key, _ptr(y), _ptr(U),
                                 _ptr(mask), _ptr(workspace), workspace.numel(), _stream(stream)))
    return y, U, mask


def lora_linear_bwd(W: NF4Weight, x, A, B, key: DropoutKey, U, mask, dY, alpha=32.0,
                    dX=None, dX_f32=False, accumulate=False, dA=None, dB=None, workspace=None,
                    stream=None, grad_accumulate=False):
    """accumulate: add the input gradient into the given fp32 dX;
    grad_accumulate: add dA, dB into the given gradients."""
    M, K = x.shape
    sh = LoraShape(M, W.N, W.K, A.shape[0], alpha)
    dev = x.device
    if dX is None:
        dX = torch.empty((M, K), dtype=torch.float32 if dX_f32 else torch.bfloat16, device=dev)
    if dA is None:
        dA = torch.empty_like(A)
    if dB is None:
        dB = torch.empty_like(B)
    if workspace is None:
        workspace = torch.empty(lora_workspace_size(M, W.N, W.K), dtype=torch.uint8, device=dev)
    w = W.c()
    dt = WS_DTYPE_F32 if dX.dtype == torch.float32 else WS_DTYPE_BF16
    fn = "ws_lora_linear_bwd_bf16" if isinstance(W, Bf16Weight) else "ws_lora_linear_bwd"
    _check(fn,
           getattr(_lib, fn)(C.byref(w), _ptr(x), _ptr(A), _ptr(B), sh, key, _ptr(U),
                                   _ptr(mask), _ptr(dY), _ptr(dX), dt,
                                   (WS_ACC_DX if accumulate else 0)
                                   | (WS_ACC_GRADS if grad_accumulate else 0),
                                   _ptr(dA), _ptr(dB), _ptr(workspace), workspace.numel(),
                                   _stream(stream)))
    return dX, dA, dB


def _ptrs(ts):
    """A C array of device pointers (None entries -> NULL; ts None -> a NULL array)."""
    if ts is None:
        return None
    return (C.c_void_p * len(ts))(*[None if t is None else t.data_ptr() for t in ts])


def lora_group_workspace_size(Ns, M, K) -> int:
    n = C.c_size_t(0)
    arr = (i64 * len(Ns))(*Ns)
    _check("ws_lora_group_workspace_size",
           _lib.ws_lora_group_workspace_size(len(Ns), arr, M, K, C.byref(n)))
    return int(n.value)


def lora_linear_fwd_group(Ws, x, As, Bs, keys, alpha=32.0, ys=None, Us=None, masks=None,
                          workspace=None, stream=None):
    """ws_lora_linear_fwd_group: ng linears reading the same x [M, K].  Returns
    (ys, Us, masks) lists."""
    ng = len(Ws)
    M, K = x.shape
    dev = x.device
    ys = ys or [torch.empty((M, W.N), dtype=torch.bfloat16, device=dev) for W in Ws]
    Us = Us or [torch.empty((M, A.shape[0]), dtype=torch.float32, device=dev) for A in As]
    masks = masks or [torch.empty((M, K // 32), dtype=torch.int32, device=dev) for _ in Ws]
    if workspace is None:
        workspace = torch.empty(lora_group_workspace_size([W.N for W in Ws], M, K),
                                dtype=torch.uint8, device=dev)
    ws_arr = (Nf4 * ng)(*[W.c() for W in Ws])
    key_arr = (DropoutKey * ng)(*keys)
    sh = LoraShape(M, Ws[0].N, K, As[0].shape[0], alpha)
    _check("ws_lora_linear_fwd_group",
           _lib.ws_lora_linear_fwd_group(ng, ws_arr, _ptr(x), _ptrs(As), _ptrs(Bs), sh, key_arr,
                                         _ptrs(ys), _ptrs(Us), _ptrs(masks), _ptr(workspace),
                                         workspace.numel(), _stream(stream)))
    return ys, Us, masks


def lora_linear_bwd_group(Ws, x, As, Bs, keys, Us, masks, dYs, alpha=32.0, dX=None,
                          accumulate=False, dAs=None, dBs=None, workspace=None, stream=None,
                          grad_accumulate=False):
    """ws_lora_linear_bwd_group: ng linears of one shape reading the same x,
    their input gradients summed into one fp32 dX.  Returns (dX, dAs, dBs)."""
    ng = len(Ws)
    M, K = x.shape
    dev = x.device
    if dX is None:
        dX = torch.empty((M, K), dtype=torch.float32, device=dev)
    dAs = dAs or [torch.empty_like(A) for A in As]
    dBs = dBs or [torch.empty_like(B) for B in Bs]
    if workspace is None:
        workspace = torch.empty(lora_group_workspace_size([W.N for W in Ws], M, K),
                                dtype=torch.uint8, device=dev)
    ws_arr = (Nf4 * ng)(*[W.c() for W in Ws])
    key_arr = (DropoutKey * ng)(*keys)
    sh = LoraShape(M, Ws[0].N, K, As[0].shape[0], alpha)
    dt = WS_DTYPE_F32 if dX.dtype == torch.float32 else WS_DTYPE_BF16
    _check("ws_lora_linear_bwd_group",
           _lib.ws_lora_linear_bwd_group(ng, ws_arr, _ptr(x), _ptrs(As), _ptrs(Bs), sh, key_arr,
                                         _ptrs(Us), _ptrs(masks), _ptrs(dYs), _ptr(dX), dt,
                                         (WS_ACC_DX if accumulate else 0)
                                         | (WS_ACC_GRADS if grad_accumulate else 0),
                                         _ptrs(dAs), _ptrs(dBs), _ptr(workspace),
                                         workspace.numel(), _stream(stream)))
    return dX, dAs, dBs


def nf4_matmul_workspace_size(M, N, K, transpose_w=False) -> int:
    n = C.c_size_t(0)
    _check("ws_nf4_matmul_workspace_size",
           _lib.ws_nf4_matmul_workspace_size(M, N, K, 1 if transpose_w else 0, C.byref(n)))
    return int(n.value)


def nf4_matmul(W: NF4Weight, act, transpose_w=False, out=None, out_f32=False, workspace=None,
               stream=None):
    """act [M, K] -> act W'^T [M, N]; with transpose_w, act [M, N] -> act W' [M, K]."""
    M = act.shape[0]
    cols = W.K if transpose_w else W.N
    if out is None:
        out = torch.empty((M, cols), dtype=torch.float32 if out_f32 else torch.bfloat16,
                          device=act.device)
    if workspace is None:
        workspace = torch.empty(nf4_matmul_workspace_size(M, W.N, W.K, transpose_w),
                                dtype=torch.uint8, device=act.device)
    w = W.c()
    dt = WS_DTYPE_F32 if out.dtype == torch.float32 else WS_DTYPE_BF16
    _check("ws_nf4_matmul", _lib.ws_nf4_matmul(C.byref(w), _ptr(act), M, 1 if transpose_w else 0,
                                               _ptr(out), dt, _ptr(workspace), workspace.numel(),
                                               _stream(stream)))
    return out


NOALLOC_SCRATCH_BYTES = 48 << 20


def nf4_matmul_noalloc(W: NF4Weight, act, transpose_w=False, out=None, out_f32=False,
                       stream=None):
    """ws_nf4_matmul without a workspace: the library's built-in scratch array
    holds the split partials (see include/wsnf4.h).  `out` must be given by
    callers that cannot allocate."""
    M = act.shape[0]
    cols = W.K if transpose_w else W.N
    if out is None:
        out = torch.empty((M, cols), dtype=torch.float32 if out_f32 else torch.bfloat16,
                          device=act.device)
    w = W.c()
    dt = WS_DTYPE_F32 if out.dtype == torch.float32 else WS_DTYPE_BF16
    _check("ws_nf4_matmul_noalloc",
           _lib.ws_nf4_matmul_noalloc(C.byref(w), _ptr(act), M, 1 if transpose_w else 0,
                                      _ptr(out), dt, _stream(stream)))
    return out


# ------------------------------------------------------------------------------ attention
def attention_fwd(q, k, v, n_seq: int, head_dim: int, o=None, o32=None, lse=None,
                  want_o32=True, stream=None):
    """Causal attention with grouped kv heads (ws_attention_fwd).  q [M, nh*hd],
    k/v [M, nkv*hd] bf16 (M = n_seq * seq_len).  Returns (o bf16, o32 fp32 or
    None, lse [nh, M])."""
    M = q.shape[0]
    nh, nkv = q.shape[1] // head_dim, k.shape[1] // head_dim
    assert M % n_seq == 0
    if o is None:
        o = torch.empty((M, nh * head_dim), dtype=torch.bfloat16, device=q.device)
    if o32 is None and want_o32:
        o32 = torch.empty((M, nh * head_dim), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((nh, M), dtype=torch.float32, device=q.device)
    _check("ws_attention_fwd",
           _lib.ws_attention_fwd(_ptr(q), _ptr(k), _ptr(v), n_seq, M // n_seq, nh, nkv, head_dim,
                                 _ptr(o), _ptr(o32), _ptr(lse), _stream(stream)))
    return o, o32, lse


def attention_workspace_size(M: int, n_heads: int, head_dim: int) -> int:
    n = C.c_size_t(0)
    _check("ws_attention_workspace_size",
           _lib.ws_attention_workspace_size(M, n_heads, head_dim, C.byref(n)))
    return int(n.value)


def attention_bwd(q, k, v, o32, lse, dO, n_seq: int, head_dim: int, dq=None, dk=None, dv=None,
                  workspace=None, stream=None):
    """Gradients (dq, dk, dv) bf16 of the causal attention (ws_attention_bwd)."""
    M = q.shape[0]
    nh, nkv = q.shape[1] // head_dim, k.shape[1] // head_dim
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(attention_workspace_size(M, nh, head_dim), dtype=torch.uint8,
                                device=q.device)
    _check("ws_attention_bwd",
           _lib.ws_attention_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o32), _ptr(lse), _ptr(dO), n_seq,
                                 M // n_seq, nh, nkv, head_dim, _ptr(dq), _ptr(dk), _ptr(dv),
                                 _ptr(workspace), workspace.numel(), _stream(stream)))
    return dq, dk, dv


# ------------------------------------------------------------------------------ stack
@dataclasses.dataclass
class StackCfg:
    M: int
    H: int
    KV: int
    I: int
    head_dim: int
    n_layers: int
    r: int = 16
    alpha: float = 32.0
    p: float = 0.1
    eps: float = 1e-6
    seed: int = 0
    base: int = BASE_NF4
    attn: int = ATTN_REPEAT_V

    def c(self):
        return StackCfgC(self.M, self.H, self.KV, self.I, self.head_dim, self.n_layers, self.r,
                         self.alpha, self.p, self.eps, self.seed, self.base, self.attn)

    def shapes(self):
        H, KV, I = self.H, self.KV, self.I
        return [(H, H), (KV, H), (KV, H), (H, H), (I, H), (I, H), (H, I)]


def stack_sizes(cfg: StackCfg, block_layers: int):
    bb, npar, sl, wsb = C.c_size_t(0), i64(0), C.c_size_t(0), C.c_size_t(0)
    c = cfg.c()
    _check("ws_stack_sizes", _lib.ws_stack_sizes(C.byref(c), block_layers, C.byref(bb),
                                                 C.byref(npar), C.byref(sl), C.byref(wsb)))
    return dict(block_bytes=int(bb.value), n_params=int(npar.value), saved_layer=int(sl.value),
                workspace=int(wsb.value))


def stack_weight_offset(cfg: StackCfg, layer_in_block: int, lin: int):
    oc, oa = C.c_size_t(0), C.c_size_t(0)
    c = cfg.c()
    _check("ws_stack_weight_offset",
           _lib.ws_stack_weight_offset(C.byref(c), layer_in_block, lin, C.byref(oc), C.byref(oa)))
    return int(oc.value), int(oa.value)


def stack_param_offset(cfg: StackCfg, layer: int, lin: int):
    oA, oB = i64(0), i64(0)
    c = cfg.c()
    _check("ws_stack_param_offset",
           _lib.ws_stack_param_offset(C.byref(c), layer, lin, C.byref(oA), C.byref(oB)))
    return int(oA.value), int(oB.value)


SAVED_FIELDS = dict(h=0, a=1, rstd1=2, v=3, vr=4, h1=5, b=6, rstd2=7, gate=8, up=9, act=10,
                    lora_u=11, mask=12, q=13, k=14, o32=15, lse=16)


def stack_saved_offset(cfg: StackCfg, field: str, lin: int = 0) -> int:
    off = C.c_size_t(0)
    c = cfg.c()
    _check("ws_stack_saved_offset",
           _lib.ws_stack_saved_offset(C.byref(c), SAVED_FIELDS[field], lin, C.byref(off)))
    return int(off.value)


def stack_loader_staging_bytes(cfg: StackCfg) -> int:
    n = C.c_size_t(0)
    c = cfg.c()
    _check("ws_stack_loader_staging_bytes", _lib.ws_stack_loader_staging_bytes(C.byref(c), C.byref(n)))
    return int(n.value)


def stack_put_weight(cfg: StackCfg, block_layers: int, layer: int, lin: int, W, image,
                         staging=None, stream=None):
    """Quantise one bf16 weight W [N, K] (device) into its place in a stack image
    (device, or pinned host through the device staging buffer)."""
    c = cfg.c()
    N, K = W.shape
    _check("ws_stack_put_weight",
           _lib.ws_stack_put_weight(C.byref(c), block_layers, layer, lin, _ptr(W), N, K,
                                        _ptr(image), _ptr(staging),
                                        0 if staging is None else staging.numel(), _stream(stream)))


WORKSPACE_FIELDS = dict(y1=0, dact=1, dg=2, du=3, db=4, dh1=5, dvr=6, dv=7, da=8, yout=9, do=10,
                        dq=11, dk=12)


def stack_workspace_offset(cfg: StackCfg, block_layers: int, field: str) -> int:
    off = C.c_size_t(0)
    c = cfg.c()
    _check("ws_stack_workspace_offset",
           _lib.ws_stack_workspace_offset(C.byref(c), block_layers, WORKSPACE_FIELDS[field],
                                          C.byref(off)))
    return int(off.value)


def block_forward(cfg: StackCfg, block_weights, first_layer, n_layers, params, step, h_in, h_out,
                  saved, workspace, stream=None, microbatch=0):
    c = cfg.c()
    _check("ws_block_forward",
           _lib.ws_block_forward(C.byref(c), _ptr(block_weights), first_layer, n_layers,
                                 _ptr(params), step, microbatch, _ptr(h_in), _ptr(h_out),
                                 _ptr(saved), _ptr(workspace), workspace.numel(), _stream(stream)))


def block_backward_recompute(cfg: StackCfg, block_weights, first_layer, n_layers, params, step,
                             h_in, saved, dh_out, dh_in, grads, workspace, stream=None,
                             microbatch=0, grad_accumulate=False):
    c = cfg.c()
    _check("ws_block_backward_recompute",
           _lib.ws_block_backward_recompute(C.byref(c), _ptr(block_weights), first_layer,
                                            n_layers, _ptr(params), step, microbatch, _ptr(h_in),
                                            _ptr(saved), _ptr(dh_out), _ptr(dh_in), _ptr(grads),
                                            1 if grad_accumulate else 0, _ptr(workspace),
                                            workspace.numel(), _stream(stream)))


def stream_block_h2d(pinned_src: torch.Tensor, dev_dst: torch.Tensor, nbytes: int = None,
                     copy_stream=None, wait_event=None, done_event=None):
    """Copies nbytes (default: all of pinned_src) host -> device on copy_stream.
    Events are raw cudaEvent_t handles (int) or None."""
    n = pinned_src.numel() * pinned_src.element_size() if nbytes is None else nbytes
    _check("ws_stream_block_h2d",
           _lib.ws_stream_block_h2d(_ptr(pinned_src), _ptr(dev_dst), n, _stream(copy_stream),
                                    C.c_void_p(wait_event) if wait_event else None,
                                    C.c_void_p(done_event) if done_event else None))


def step_opts(n_micro=1, order=GA_MICROBATCH_MAJOR, time_copies=False, copy_piece_bytes=0):
    return StepOptsC(n_micro, order, 1 if time_copies else 0, 0, copy_piece_bytes)


def stack_train_step(cfg: StackCfg, block_layers: int, streamed: bool, bufs: StackBuffersC,
                     step: int, h0, lr: float = 2e-4, stream=None, copy_stream=None, opts=None):
    """opts: StepOptsC (micro-batches and their order) or None for one micro-batch."""
    c = cfg.c()
    _check("ws_stack_train_step_ex",
           _lib.ws_stack_train_step_ex(C.byref(c), block_layers, 1 if streamed else 0,
                                       C.byref(opts) if opts is not None else None,
                                       C.byref(bufs), step, _ptr(h0), lr, _stream(stream),
                                       _stream(copy_stream) if copy_stream is not None else None))


class StepGraph:
    """One training step of the stack captured as a CUDA graph
    (ws_stack_graph_create_ex); ``step`` replays it for any step number."""

    def __init__(self, cfg: StackCfg, block_layers: int, streamed: bool, bufs: StackBuffersC,
                 lr: float, stream, copy_stream=None, opts=None):
        self._bufs = bufs  # the graph keeps these pointers
        self._opts = opts
        c = cfg.c()
        h = C.c_void_p()
        _check("ws_stack_graph_create_ex",
               _lib.ws_stack_graph_create_ex(C.byref(c), block_layers, 1 if streamed else 0,
                                             C.byref(opts) if opts is not None else None,
                                             C.byref(bufs), lr, _stream(stream),
                                             _stream(copy_stream) if copy_stream is not None
                                             else None, C.byref(h)))
        self._h = h

    def step(self, step: int, h0, stream=None):
        _check("ws_stack_graph_step", _lib.ws_stack_graph_step(self._h, step, _ptr(h0), _stream(stream)))

    def copy_times_ms(self):
        """Durations (ms) of the block copies of the last replay (graphs made with time_copies)."""
        n = i32(0)
        cap = 4096
        buf = (C.c_float * cap)()
        _check("ws_stack_graph_copy_times",
               _lib.ws_stack_graph_copy_times(self._h, buf, cap, C.byref(n)))
        return [float(buf[i]) for i in range(min(n.value, cap))]

    def close(self):
        if self._h is not None and self._h.value:
            _lib.ws_stack_graph_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
