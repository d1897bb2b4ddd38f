"""Python access to the oracle (oracle.c): plain double-precision CPU code.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
CPU-baseline leg of bench.py may import this package.  Nothing here imports
the CUDA path, and the CUDA path never imports this.

Besides thin ctypes wrappers this module holds the oracle's own conversion of
float32 values to bfloat16 values (round to nearest, ties to even), used to
give the oracle exactly the bf16 weights a bf16-mode step computes with.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        dp = C.POINTER(C.c_double)
        ip = C.POINTER(C.c_int)
        sz = C.c_size_t
        i = C.c_int
        d = C.c_double
        sig = {
            "or_num_params": (sz, [i, i, i, i, i]),
            "or_param_offset": (i, [i, i, i, i, i, i, i, C.POINTER(sz), C.POINTER(sz)]),
            "or_set_threads": (None, [i]),
            "or_get_threads": (i, []),
            "or_linear_fwd": (None, [dp, dp, dp, i, i, i, dp]),
            "or_linear_bwd": (None, [dp, dp, dp, i, i, i, dp, dp, dp]),
            "or_layernorm_fwd": (None, [dp, dp, dp, i, i, d, dp, dp, dp]),
            "or_layernorm_bwd": (None, [dp, dp, dp, dp, dp, i, i, dp, dp, dp]),
            "or_gelu_fwd": (None, [dp, sz, dp]),
            "or_gelu_bwd": (None, [dp, dp, sz, dp]),
            "or_attention_fwd": (None, [dp, i, i, i, i, dp, dp, dp]),
            "or_attention_bwd": (None, [dp, dp, dp, i, i, i, i, dp]),
            "or_xent": (d, [dp, ip, i, i, dp, dp, d]),
            "or_embed_fwd": (None, [dp, dp, ip, i, i, i, dp]),
            "or_embed_bwd": (None, [dp, ip, i, i, i, dp, dp]),
            "or_adamw": (None, [dp, dp, dp, dp, sz, d, d, d, d, d, i]),
            "or_gpt2_step": (d, [i, i, i, i, i, dp, ip, ip, i, i, dp, dp]),
            "or_gpt2_logits_last": (i, [i, i, i, i, i, dp, ip, i, i, dp]),
            "or_matmul": (None, [dp, dp, i, i, i, dp]),
            "or_matmul_bwd": (None, [dp, dp, dp, i, i, i, dp, dp]),
            "or_add_row": (None, [dp, dp, i, i, dp]),
            "or_add_row_bwd": (None, [dp, i, i, dp, dp]),
            "or_softmax_rows": (None, [dp, i, i, dp]),
            "or_softmax_rows_bwd": (None, [dp, dp, i, i, dp]),
            "or_xent_probs": (d, [dp, ip, i, i, dp, d]),
            "or_mlp_sgd": (None, [dp, ip, i, i, i, i, dp, dp, dp, dp, d, i, dp, dp]),
            "or_grad_norm": (d, [dp, sz, d, ip]),
            "or_clip_coef": (d, [d, d]),
            "or_adamw_ex": (i, [dp, dp, dp, dp, sz, d, d, d, d, d, i, d, d]),
            "or_loss_scale_update": (None, [dp, ip, i, i, d, d]),
            "or_val_reset": (None, []),
            "or_val_leaf": (i, [d]),
            "or_val_add": (i, [i, i]),
            "or_val_mul": (i, [i, i]),
            "or_val_pow": (i, [i, d]),
            "or_val_exp": (i, [i]),
            "or_val_log": (i, [i]),
            "or_val_data": (d, [i]),
            "or_val_grad": (d, [i]),
            "or_val_backward": (i, [i]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _d(a):
    """float64 C-contiguous pointer (None passes NULL)."""
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(C.POINTER(C.c_double))


def _i(a):
    assert a.dtype == np.int32 and a.flags.c_contiguous
    return a.ctypes.data_as(C.POINTER(C.c_int))


def f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def set_threads(n: int) -> None:
    lib().or_set_threads(int(n))


def get_threads() -> int:
    return int(lib().or_get_threads())


# ---------------------------------------------------------------- layout
def num_params(L, C_, H, V, maxT) -> int:
    return int(lib().or_num_params(L, C_, H, V, maxT))


def param_offset(L, C_, H, V, maxT, layer, which):
    off = C.c_size_t()
    n = C.c_size_t()
    rc = lib().or_param_offset(L, C_, H, V, maxT, layer, which, C.byref(off), C.byref(n))
    if rc != 0:
        raise ValueError("bad tensor index")
    return int(off.value), int(n.value)


# ---------------------------------------------------------------- bf16 values
def bf16_values(x) -> np.ndarray:
    """Nearest bfloat16 value of each float32 (ties to even), as float64: the
    16-bit parameter copy of the mixed-precision step (dl-scratch page, 3.4,
    which stores fp16; bf16 is the storage type this library reads it with on
    the tensor cores)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def f16_values(x) -> np.ndarray:
    """Nearest IEEE half value of each float32 (ties to even; beyond the
    largest half, 65504, the value becomes +-inf; below the smallest
    subnormal, 2^-24, it rounds to zero or 2^-24), as float64: the fp16
    parameter copy of the dl-scratch page's mixed precision (3.4)."""
    with np.errstate(over="ignore"):
        return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).astype(np.float64)


# ---------------------------------------------------------------- ops
def linear_fwd(x, W, b=None):
    x, W = f64(x), f64(W)
    M, K = x.shape
    N = W.shape[0]
    y = np.zeros((M, N))
    lib().or_linear_fwd(_d(x), _d(W), _d(None if b is None else f64(b)), M, K, N, _d(y))
    return y


def linear_bwd(x, W, dy, with_bias=True):
    x, W, dy = f64(x), f64(W), f64(dy)
    M, K = x.shape
    N = W.shape[0]
    dx, dW = np.zeros_like(x), np.zeros_like(W)
    db = np.zeros(N) if with_bias else None
    lib().or_linear_bwd(_d(x), _d(W), _d(dy), M, K, N, _d(dx), _d(dW), _d(db))
    return dx, dW, db


def layernorm_fwd(x, w, b, eps=1e-5):
    x, w, b = f64(x), f64(w), f64(b)
    M, Cc = x.shape
    y = np.zeros_like(x)
    mean, rstd = np.zeros(M), np.zeros(M)
    lib().or_layernorm_fwd(_d(x), _d(w), _d(b), M, Cc, eps, _d(y), _d(mean), _d(rstd))
    return y, mean, rstd


def layernorm_bwd(x, w, mean, rstd, dy):
    x, w, mean, rstd, dy = map(f64, (x, w, mean, rstd, dy))
    M, Cc = x.shape
    dx, dw, db = np.zeros_like(x), np.zeros(Cc), np.zeros(Cc)
    lib().or_layernorm_bwd(_d(x), _d(w), _d(mean), _d(rstd), _d(dy), M, Cc, _d(dx), _d(dw), _d(db))
    return dx, dw, db


def gelu_fwd(u):
    u = f64(u)
    g = np.zeros_like(u)
    lib().or_gelu_fwd(_d(u), u.size, _d(g))
    return g


def gelu_bwd(u, dg):
    u, dg = f64(u), f64(dg)
    du = np.zeros_like(u)
    lib().or_gelu_bwd(_d(u), _d(dg), u.size, _d(du))
    return du


def attention_fwd(qkv, B, T, C_, H, want_lse=False):
    """(y, P), or (y, P, lse) with lse [B, H, T] the log of each row's softmax
    denominator over the scaled scores."""
    qkv = f64(qkv)
    y = np.zeros((B * T, C_))
    P = np.zeros((B, H, T, T))
    lse = np.zeros((B, H, T)) if want_lse else None
    lib().or_attention_fwd(_d(qkv), B, T, C_, H, _d(y), _d(P), _d(lse) if want_lse else None)
    return (y, P, lse) if want_lse else (y, P)


def attention_bwd(qkv, P, dy, B, T, C_, H):
    qkv, P, dy = f64(qkv), f64(P), f64(dy)
    dqkv = np.zeros_like(qkv)
    lib().or_attention_bwd(_d(qkv), _d(P), _d(dy), B, T, C_, H, _d(dqkv))
    return dqkv


def xent(z, targets, want_grad=False):
    z = f64(z)
    t = np.ascontiguousarray(targets, dtype=np.int32)
    M, V = z.shape
    rl = np.zeros(M)
    dz = np.zeros_like(z) if want_grad else None
    loss = lib().or_xent(_d(z), _i(t), M, V, _d(rl), _d(dz), 1.0)
    return loss, rl, dz


def embed_fwd(wte, wpe, tok, B, T):
    wte, wpe = f64(wte), f64(wpe)
    tok = np.ascontiguousarray(tok, dtype=np.int32)
    Cc = wte.shape[1]
    x = np.zeros((B * T, Cc))
    lib().or_embed_fwd(_d(wte), _d(wpe), _i(tok), B, T, Cc, _d(x))
    return x


def embed_bwd(dx, tok, B, T, V, maxT):
    dx = f64(dx)
    tok = np.ascontiguousarray(tok, dtype=np.int32)
    Cc = dx.shape[1]
    dwte, dwpe = np.zeros((V, Cc)), np.zeros((maxT, Cc))
    lib().or_embed_bwd(_d(dx), _i(tok), B, T, Cc, _d(dwte), _d(dwpe))
    return dwte, dwpe


def adamw(p, g, m, v, lr, beta1, beta2, eps, weight_decay, t):
    """Updates copies of p, m, v and returns them."""
    p, g, m, v = (f64(a).copy() for a in (p, g, m, v))
    lib().or_adamw(_d(p), _d(g), _d(m), _d(v), p.size, lr, beta1, beta2, eps, weight_decay, int(t))
    return p, m, v


# ---------------------------------------------------------------- model
def gpt2_step(shape, params, tokens, targets, want_grads=True, want_row_loss=False):
    """One forward+backward of the GPT-2 step.

    shape: object with L, C, H, V, maxT.  params: flat (any float dtype; the
    values are taken exactly as float64).  tokens/targets: int [B, T].
    Returns (loss, grads or None, row_loss or None)."""
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    targets = np.ascontiguousarray(targets, dtype=np.int32)
    B, T = tokens.shape
    P = f64(params)
    n = num_params(shape.L, shape.C, shape.H, shape.V, shape.maxT)
    if P.size != n:
        raise ValueError(f"expected {n} parameters, got {P.size}")
    G = np.zeros(n) if want_grads else None
    rl = np.zeros(B * T) if want_row_loss else None
    loss = lib().or_gpt2_step(shape.L, shape.C, shape.H, shape.V, shape.maxT, _d(P),
                              _i(tokens), _i(targets), B, T, _d(G), _d(rl))
    return float(loss), G, rl


def gpt2_logits_last(shape, params, tokens):
    """Logits of each sequence's last position, float64 [B, V] (forward only)."""
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    B, T = tokens.shape
    P = f64(params)
    out = np.zeros((B, shape.V))
    rc = lib().or_gpt2_logits_last(shape.L, shape.C, shape.H, shape.V, shape.maxT, _d(P), _i(tokens),
                                   B, T, _d(out))
    if rc != 0:
        raise ValueError("bad arguments to or_gpt2_logits_last")
    return out


# ---------------------------------------------------------------- generic ops
def matmul(A, B):
    """C = A B with B [K, N]."""
    A, B = f64(A), f64(B)
    M, K = A.shape
    N = B.shape[1]
    out = np.zeros((M, N))
    lib().or_matmul(_d(A), _d(B), M, K, N, _d(out))
    return out


def matmul_bwd(A, B, dC):
    A, B, dC = f64(A), f64(B), f64(dC)
    M, K = A.shape
    N = B.shape[1]
    dA, dB = np.zeros_like(A), np.zeros_like(B)
    lib().or_matmul_bwd(_d(A), _d(B), _d(dC), M, K, N, _d(dA), _d(dB))
    return dA, dB


def add_row(A, b):
    A, b = f64(A), f64(b)
    R, Cc = A.shape
    out = np.zeros_like(A)
    lib().or_add_row(_d(A), _d(b), R, Cc, _d(out))
    return out


def add_row_bwd(dC):
    dC = f64(dC)
    R, Cc = dC.shape
    dA, db = np.zeros_like(dC), np.zeros(Cc)
    lib().or_add_row_bwd(_d(dC), R, Cc, _d(dA), _d(db))
    return dA, db


def softmax_rows(Z):
    Z = f64(Z)
    R, Cc = Z.shape
    P = np.zeros_like(Z)
    lib().or_softmax_rows(_d(Z), R, Cc, _d(P))
    return P


def softmax_rows_bwd(P, dP):
    P, dP = f64(P), f64(dP)
    R, Cc = P.shape
    dZ = np.zeros_like(P)
    lib().or_softmax_rows_bwd(_d(P), _d(dP), R, Cc, _d(dZ))
    return dZ


def xent_probs(P, y, dloss=1.0):
    """(loss, dP) of the cross entropy of probabilities P [R, C] at labels y."""
    P = f64(P)
    y = np.ascontiguousarray(y, dtype=np.int32)
    R, Cc = P.shape
    dP = np.zeros_like(P)
    loss = lib().or_xent_probs(_d(P), _i(y), R, Cc, _d(dP), float(dloss))
    return float(loss), dP


def mlp_sgd(x, y, W1, b1, W2, b2, lr, steps):
    """The small classifier trained by SGD on a fixed batch.  Returns
    (losses [steps], updated (W1, b1, W2, b2), gradients of the last step)."""
    x = f64(x)
    y = np.ascontiguousarray(y, dtype=np.int32)
    W1, b1, W2, b2 = (f64(a).copy() for a in (W1, b1, W2, b2))
    R, nin = x.shape
    nh, nout = W1.shape[1], W2.shape[1]
    losses = np.zeros(max(steps, 1))
    grads = np.zeros(W1.size + b1.size + W2.size + b2.size)
    lib().or_mlp_sgd(_d(x), _i(y), R, nin, nh, nout, _d(W1), _d(b1), _d(W2), _d(b2), float(lr), int(steps),
                     _d(losses), _d(grads))
    n1, n2 = W1.size, W2.size
    g = (grads[:n1].reshape(W1.shape), grads[n1:n1 + nh], grads[n1 + nh:n1 + nh + n2].reshape(W2.shape),
         grads[n1 + nh + n2:])
    return losses[:steps], (W1, b1, W2, b2), g


# ---------------------------------------------------------------- update-side variants
def grad_norm(g, scale=1.0):
    """(||g / scale||_2, nonfinite flag)."""
    g = f64(np.ravel(g))
    bad = C.c_int()
    n = lib().or_grad_norm(_d(g), g.size, float(scale), C.byref(bad))
    return float(n), int(bad.value)


def clip_coef(norm, max_norm):
    return float(lib().or_clip_coef(float(norm), float(max_norm)))


def adamw_ex(p, g, m, v, lr, beta1, beta2, eps, weight_decay, t, scale=1.0, max_norm=0.0):
    """Updates copies of p, m, v; returns (p, m, v, skipped)."""
    p, g, m, v = (f64(a).copy() for a in (p, g, m, v))
    skipped = lib().or_adamw_ex(_d(p), _d(g), _d(m), _d(v), p.size, lr, beta1, beta2, eps, weight_decay, int(t),
                                float(scale), float(max_norm))
    return p, m, v, bool(skipped)


def loss_scale_update(scale, clean, overflow, window=1000, growth=1.001, backoff=0.5):
    """One update of the dynamic loss scale; returns (scale, clean)."""
    s, c = C.c_double(scale), C.c_int(clean)
    lib().or_loss_scale_update(C.byref(s), C.byref(c), int(bool(overflow)), int(window), float(growth),
                               float(backoff))
    return float(s.value), int(c.value)


# ---------------------------------------------------------------- scalar tape
class Value:
    """A scalar node of the oracle's scalar tape (handle into its pool)."""

    def __init__(self, h: int):
        if h < 0:
            raise ValueError("invalid operand")
        self.h = h

    @staticmethod
    def leaf(x: float) -> "Value":
        return Value(lib().or_val_leaf(float(x)))

    def __add__(self, o):
        return Value(lib().or_val_add(self.h, o.h))

    def __mul__(self, o):
        return Value(lib().or_val_mul(self.h, o.h))

    def pow(self, e: float):
        return Value(lib().or_val_pow(self.h, float(e)))

    def exp(self):
        return Value(lib().or_val_exp(self.h))

    def log(self):
        return Value(lib().or_val_log(self.h))

    @property
    def data(self) -> float:
        return float(lib().or_val_data(self.h))

    @property
    def grad(self) -> float:
        return float(lib().or_val_grad(self.h))

    def backward(self) -> int:
        return int(lib().or_val_backward(self.h))


def value_reset() -> None:
    lib().or_val_reset()


def value_backward_raw(handle: int) -> int:
    return int(lib().or_val_backward(handle))
