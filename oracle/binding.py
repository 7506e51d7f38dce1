"""ctypes wrappers around the C oracle (test infrastructure only)."""
from __future__ import annotations

import ctypes as C
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

LIN_NAMES = ("q", "k", "v", "o", "gate", "up", "down")


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (OpenMP, no fp contraction)."""
    with _lock:
        if (not force and os.path.exists(_SO)
                and os.path.getmtime(_SO) >= max(os.path.getmtime(_SRC),
                                                 os.path.getmtime(os.path.join(_HERE, "oracle.h")))):
            return _SO
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", "-D_GNU_SOURCE",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
        return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_SO)
        P = C.c_void_p
        i64 = C.c_int64
        L.orc_f32_to_bf16.restype = C.c_uint16
        L.orc_f32_to_bf16.argtypes = [C.c_float]
        L.orc_bf16_to_f64.restype = C.c_double
        L.orc_bf16_to_f64.argtypes = [C.c_uint16]
        L.orc_f64_to_bf16.restype = C.c_uint16
        L.orc_f64_to_bf16.argtypes = [C.c_double]
        L.orc_quantize_nf4.argtypes = [P, i64, i64, P, P]
        L.orc_dequant_nf4.argtypes = [P, P, i64, i64, P]
        L.orc_philox4x32_10.argtypes = [P, P, P]
        L.orc_keep_threshold.restype = C.c_uint64
        L.orc_keep_threshold.argtypes = [C.c_double]
        L.orc_dropout_mask.argtypes = [C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint32,
                                       C.c_uint32, C.c_double, i64, i64, P]
        L.orc_lora_fwd_rows.argtypes = [i64, i64, i64, C.c_int, P, P, P, P, P,
                                        C.c_double, P, i64, P, P]
        L.orc_lora_bwd.argtypes = [i64, i64, i64, C.c_int, P, P, P, P, P, P,
                                   C.c_double, P, i64, P, P, P]
        L.orc_stack_fwd_bwd.argtypes = [P, C.c_uint32, P, P, P, P, P, P]
        L.orc_adam_step.argtypes = [i64, P, P, P, P, i64, C.c_double, C.c_double,
                                    C.c_double, C.c_double]
        L.orc_num_threads.restype = C.c_int
        L.orc_rmsnorm_bf16.argtypes = [i64, i64, C.c_double, P, P, P]
        L.orc_silu_mul_bf16.argtypes = [i64, P, P, P]
        L.orc_repeat_kv.argtypes = [i64, i64, i64, i64, P, P]
        L.orc_stack_fwd_bwd_mb.argtypes = [P, C.c_uint32, C.c_uint32, C.c_int, P, P, P, P, P, P]
        L.orc_silu_mul_f64.argtypes = [i64, P, P, P]
        L.orc_rmsnorm_f64.argtypes = [i64, i64, C.c_double, C.c_int, P, P, P]
        L.orc_rmsnorm_bwd_add.argtypes = [i64, i64, P, P, P, P]
        L.orc_silu_mul_bwd.argtypes = [i64, C.c_int, P, P, P, P, P]
        L.orc_repeat_kv_bwd.argtypes = [i64, i64, i64, i64, C.c_int, P, P]
        L.orc_attention_fwd.argtypes = [i64, i64, i64, i64, i64, P, P, P, P, P]
        L.orc_attention_bwd.argtypes = [i64, i64, i64, i64, i64, P, P, P, P, P, P, P]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def nf4_levels() -> np.ndarray:
    """The oracle's 16 NF4 levels (fp32)."""
    L = lib()
    arr = (C.c_float * 16).in_dll(L, "orc_nf4_levels")
    return np.array(list(arr), dtype=np.float32)


def num_threads() -> int:
    return int(lib().orc_num_threads())


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    L = lib()
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([L.orc_f32_to_bf16(float(v)) for v in x], dtype=np.uint16)


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    L = lib()
    b = np.asarray(b, dtype=np.uint16).ravel()
    return np.array([L.orc_bf16_to_f64(int(v)) for v in b], dtype=np.float64)


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    L = lib()
    x = np.asarray(x, dtype=np.float64).ravel()
    return np.array([L.orc_f64_to_bf16(float(v)) for v in x], dtype=np.uint16)


def quantize_nf4(W_bf16: np.ndarray):
    """W_bf16: uint16 [N, K] -> (codes uint8 [N, K/2], absmax f32 [K/64, N])."""
    W = _c(W_bf16, np.uint16)
    N, K = W.shape
    assert K % 64 == 0
    codes = np.empty((N, K // 2), np.uint8)
    absmax = np.empty((K // 64, N), np.float32)
    lib().orc_quantize_nf4(_p(W), N, K, _p(codes), _p(absmax))
    return codes, absmax


def dequant_nf4(codes: np.ndarray, absmax: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.uint8)
    absmax = _c(absmax, np.float32)
    N = codes.shape[0]
    K = codes.shape[1] * 2
    out = np.empty((N, K), np.uint16)
    lib().orc_dequant_nf4(_p(codes), _p(absmax), N, K, _p(out))
    return out


def philox4x32_10(ctr, key):
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    out = np.empty(4, np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def keep_threshold(p: float) -> int:
    return int(lib().orc_keep_threshold(float(p)))


def dropout_mask(seed, step, layer, linear, microbatch, p, M, K) -> np.ndarray:
    assert K % 32 == 0
    bits = np.empty((M, K // 32), np.uint32)
    lib().orc_dropout_mask(seed, step, layer, linear, microbatch, float(p), M, K, _p(bits))
    return bits


def lora_fwd(x, Wq, A, B, mask, scale, rows=None):
    """Returns (y [rows, N] f64, U [rows, r] f64)."""
    x = _c(x, np.uint16)
    Wq = _c(Wq, np.uint16)
    A = _c(A, np.float32)
    B = _c(B, np.float32)
    M, K = x.shape
    N = Wq.shape[0]
    r = A.shape[0]
    m = None if mask is None else _c(mask, np.uint32)
    if rows is None:
        rws = None
        nrows = M
    else:
        rws = _c(rows, np.int64)
        nrows = len(rws)
    y = np.empty((nrows, N), np.float64)
    U = np.empty((nrows, r), np.float64)
    lib().orc_lora_fwd_rows(M, N, K, r, _p(x), _p(Wq), _p(A), _p(B), _p(m), float(scale),
                            _p(rws), nrows, _p(y), _p(U))
    return y, U


def lora_bwd(x, Wq, A, B, mask, dY, scale, rows=None, want_dx=True):
    """Returns (dX [rows, K] f64 or None, dA [r, K] f64, dB [N, r] f64)."""
    x = _c(x, np.uint16)
    Wq = _c(Wq, np.uint16)
    A = _c(A, np.float32)
    B = _c(B, np.float32)
    dY = _c(dY, np.uint16)
    M, K = x.shape
    N = Wq.shape[0]
    r = A.shape[0]
    m = None if mask is None else _c(mask, np.uint32)
    if rows is None:
        rws = None
        nrows = M
    else:
        rws = _c(rows, np.int64)
        nrows = len(rws)
    dX = np.empty((nrows, K), np.float64) if want_dx else None
    dA = np.empty((r, K), np.float64)
    dB = np.empty((N, r), np.float64)
    lib().orc_lora_bwd(M, N, K, r, _p(x), _p(Wq), _p(A), _p(B), _p(m), _p(dY), float(scale),
                       _p(rws), nrows, _p(dX), _p(dA), _p(dB))
    return dX, dA, dB


class _StackCfgC(C.Structure):
    _fields_ = [("M", C.c_int64), ("H", C.c_int64), ("KV", C.c_int64), ("I", C.c_int64),
                ("head_dim", C.c_int64), ("n_layers", C.c_int), ("r", C.c_int),
                ("alpha", C.c_double), ("p", C.c_double), ("eps", C.c_double),
                ("seed", C.c_uint64), ("round_bf16", C.c_int), ("attn", C.c_int)]


class _StackParamsC(C.Structure):
    _fields_ = [("Wq", C.c_void_p), ("A", C.c_void_p), ("B", C.c_void_p)]


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
    round_bf16: bool = True
    attn: int = 0  # 0: repeat(v) in place of attention; 1: causal attention core

    def shapes(self):
        """(N, K) of each linear in a layer, in q,k,v,o,gate,up,down order."""
        H, KV, I = self.H, self.KV, self.I
        return [(H, H), (KV, H), (KV, H), (H, H), (I, H), (I, H), (H, I)]


def stack_fwd_bwd(cfg: StackCfg, step: int, Wq, A, B, h0, backward=True, microbatch=0,
                  n_micro=1):
    """Wq/A/B: lists indexed [layer*7 + linear].  Returns (loss, h_L, dA, dB).
    With gradient accumulation over n_micro micro-batches, one call covers
    micro-batch `microbatch` (its dropout keys) and returns its share of the
    step loss and gradients (see orc_stack_fwd_bwd_mb)."""
    L = lib()
    n = cfg.n_layers * 7
    assert len(Wq) == len(A) == len(B) == n
    Wq = [_c(w, np.uint16) for w in Wq]
    A = [_c(a, np.float32) for a in A]
    B = [_c(b, np.float32) for b in B]
    h0 = _c(h0, np.float64)
    arrW = (C.c_void_p * n)(*[w.ctypes.data for w in Wq])
    arrA = (C.c_void_p * n)(*[a.ctypes.data for a in A])
    arrB = (C.c_void_p * n)(*[b.ctypes.data for b in B])
    prm = _StackParamsC(C.cast(arrW, C.c_void_p), C.cast(arrA, C.c_void_p),
                        C.cast(arrB, C.c_void_p))
    cc = _StackCfgC(cfg.M, cfg.H, cfg.KV, cfg.I, cfg.head_dim, cfg.n_layers, cfg.r,
                    cfg.alpha, cfg.p, cfg.eps, cfg.seed, 1 if cfg.round_bf16 else 0,
                    int(cfg.attn))
    loss = C.c_double(0.0)
    h_out = np.empty((cfg.M, cfg.H), np.float64)
    if backward:
        dA = [np.zeros_like(a, dtype=np.float64) for a in A]
        dB = [np.zeros_like(b, dtype=np.float64) for b in B]
        arrdA = (C.c_void_p * n)(*[a.ctypes.data for a in dA])
        arrdB = (C.c_void_p * n)(*[b.ctypes.data for b in dB])
        pdA, pdB = C.cast(arrdA, C.c_void_p), C.cast(arrdB, C.c_void_p)
    else:
        dA = dB = None
        pdA = pdB = None
    L.orc_stack_fwd_bwd_mb(C.byref(cc), step, microbatch, n_micro, C.byref(prm), _p(h0),
                           C.byref(loss), _p(h_out), pdA, pdB)
    return loss.value, h_out, dA, dB


def attention_fwd(q, k, v, n_seq, head_dim, want_lse=False):
    """Causal attention with grouped kv heads.  q [M, nh*d], k/v [M, nkv*d]
    (float, M = n_seq * S) -> o [M, nh*d] (and lse [nh, M]), in double."""
    q, k, v = _c(q, np.float64), _c(k, np.float64), _c(v, np.float64)
    M = q.shape[0]
    nh, nkv = q.shape[1] // head_dim, k.shape[1] // head_dim
    assert M % n_seq == 0 and k.shape == v.shape and k.shape[0] == M
    o = np.empty_like(q)
    lse = np.empty((nh, M), np.float64)
    lib().orc_attention_fwd(n_seq, M // n_seq, nh, nkv, head_dim, _p(q), _p(k), _p(v), _p(o),
                            _p(lse))
    return (o, lse) if want_lse else o


def attention_bwd(q, k, v, dO, n_seq, head_dim):
    """Gradients (dq, dk, dv) of the causal attention for upstream dO, in double."""
    q, k, v, dO = (_c(a, np.float64) for a in (q, k, v, dO))
    M = q.shape[0]
    nh, nkv = q.shape[1] // head_dim, k.shape[1] // head_dim
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    lib().orc_attention_bwd(n_seq, M // n_seq, nh, nkv, head_dim, _p(q), _p(k), _p(v), _p(dO),
                            _p(dq), _p(dk), _p(dv))
    return dq, dk, dv


def rmsnorm_bf16(x, eps=1e-6):
    """x: [M, H] float -> (bf16 bits [M, H], rstd [M])."""
    x = _c(x, np.float64)
    M, H = x.shape
    y = np.empty((M, H), np.uint16)
    rstd = np.empty(M, np.float64)
    lib().orc_rmsnorm_bf16(M, H, eps, _p(x), _p(y), _p(rstd))
    return y, rstd


def silu_mul_bf16(g, u):
    g = _c(g, np.uint16)
    u = _c(u, np.uint16)
    act = np.empty_like(g)
    lib().orc_silu_mul_bf16(g.size, _p(g), _p(u), _p(act))
    return act


def repeat_kv(v, H, head_dim):
    v = _c(v, np.uint16)
    M, KV = v.shape
    vr = np.empty((M, H), np.uint16)
    lib().orc_repeat_kv(M, H, KV, head_dim, _p(v), _p(vr))
    return vr


def adam_step(p, g, m, v, t, lr=2e-4, beta1=0.9, beta2=0.999, eps=1e-8):
    """In-place Adam step on float64 arrays."""
    for a in (p, g, m, v):
        assert a.dtype == np.float64 and a.flags.c_contiguous
    lib().orc_adam_step(p.size, _p(p), _p(g), _p(m), _p(v), int(t), lr, beta1, beta2, eps)



def rmsnorm_f64(x, eps=1e-6, round_bf16=False):
    """x: [M, H] -> (y [M, H] double (bf16-valued when round_bf16), rstd [M])."""
    x = _c(x, np.float64)
    M, H = x.shape
    y = np.empty((M, H), np.float64)
    rstd = np.empty(M, np.float64)
    lib().orc_rmsnorm_f64(M, H, eps, 1 if round_bf16 else 0, _p(x), _p(y), _p(rstd))
    return y, rstd


def rmsnorm_bwd(x, rstd, dy, dx=None):
    """dx + (rstd dy - rstd^3 x (dy . x) / H) per row (dx = 0 when not given)."""
    x = _c(x, np.float64)
    M, H = x.shape
    out = np.zeros((M, H), np.float64) if dx is None else _c(dx, np.float64).copy()
    lib().orc_rmsnorm_bwd_add(M, H, _p(x), _p(_c(rstd, np.float64)), _p(_c(dy, np.float64)),
                              _p(out))
    return out


def silu_mul_f64(g, u):
    """act = SiLU(g) u in double, unrounded (g, u doubles)."""
    g = _c(g, np.float64)
    u = _c(u, np.float64)
    act = np.empty_like(g)
    lib().orc_silu_mul_f64(g.size, _p(g), _p(u), _p(act))
    return act


def silu_mul_bwd(dact, g, u, round_bf16=True):
    """Gradients (dg, du) of act = SiLU(g) u for upstream dact (doubles)."""
    dact = _c(dact, np.float64)
    g = _c(g, np.float64)
    u = _c(u, np.float64)
    dg = np.empty_like(dact)
    du = np.empty_like(dact)
    lib().orc_silu_mul_bwd(dact.size, 1 if round_bf16 else 0, _p(dact), _p(g), _p(u), _p(dg),
                           _p(du))
    return dg, du


def repeat_kv_bwd(dvr, KV, head_dim, round_bf16=True):
    """dvr [M, H] -> dv [M, KV]: the sum over the query heads sharing each kv head."""
    dvr = _c(dvr, np.float64)
    M, H = dvr.shape
    dv = np.empty((M, KV), np.float64)
    lib().orc_repeat_kv_bwd(M, H, KV, head_dim, 1 if round_bf16 else 0, _p(dvr), _p(dv))
    return dv
