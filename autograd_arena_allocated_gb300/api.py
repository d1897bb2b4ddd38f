"""Thin Python binding of the C ABI (argument marshalling only).

Tensors are passed as raw pointers: torch tensors by data_ptr(), numpy arrays
by their host address.  Every computation runs in libtt.so's CUDA kernels;
torch is used only for device memory and streams.
"""
from __future__ import annotations

import ctypes as C
from typing import Optional

from ._native import GPT2Config, OpProfile, TT_BF16, TT_FP16, TT_FP32, TTError, lib

DTYPES = {"fp32": TT_FP32, "bf16": TT_BF16, "fp16": TT_FP16}


def _ptr(x) -> Optional[int]:
    """Address of a torch tensor, numpy array or raw int (None passes NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        if not x.flags.c_contiguous:
            raise ValueError("array must be C-contiguous")
        return x.ctypes.data
    raise TypeError(f"cannot pass {type(x)!r} as a pointer")


def make_config(L, C_, H, V, maxT, dtype="bf16") -> GPT2Config:
    return GPT2Config(L, C_, H, V, maxT, DTYPES[dtype] if isinstance(dtype, str) else int(dtype))


def num_params(cfg: GPT2Config) -> int:
    return int(lib().tt_gpt2_num_params(C.byref(cfg)))


def param_offset(cfg: GPT2Config, layer: int, which: int):
    off, n = C.c_size_t(), C.c_size_t()
    rc = lib().tt_gpt2_param_offset(C.byref(cfg), layer, which, C.byref(off), C.byref(n))
    if rc != 0:
        raise TTError(rc, "bad tensor index")
    return int(off.value), int(n.value)


def generate_arena_bytes(cfg, B: int, T_prompt: int, n_new: int) -> int:
    """Exact arena bytes of tt_gpt2_generate."""
    return int(lib().tt_gpt2_generate_arena_bytes(C.byref(cfg), int(B), int(T_prompt), int(n_new)))


def arena_bytes(cfg: GPT2Config, B: int, T: int) -> int:
    return int(lib().tt_gpt2_arena_bytes(C.byref(cfg), B, T))


class Context:
    """One device arena + tape (tt_ctx).  Use as a context manager or close()."""

    def __init__(self, arena_bytes: int, stream=None):
        h = C.c_void_p()
        rc = lib().tt_ctx_create(int(arena_bytes), C.byref(h))
        if rc != 0:
            raise TTError(rc, "tt_ctx_create failed")
        self.h = h
        if stream is None:
            import torch
            if torch.cuda.is_available():
                stream = torch.cuda.current_stream().cuda_stream
        if stream is not None:
            self._check(lib().tt_ctx_set_stream(self.h, C.c_void_p(int(stream))))
        self.cfg: Optional[GPT2Config] = None

    # -------------------------------------------------------------- plumbing
    def _check(self, rc):
        if rc != 0:
            raise TTError(rc, lib().tt_last_error(self.h).decode())
        return rc

    def close(self):
        if self.h is not None and self.h.value:
            lib().tt_ctx_destroy(self.h)
        self.h = C.c_void_p()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -------------------------------------------------------------- context
    def set_stream(self, stream):
        self._check(lib().tt_ctx_set_stream(self.h, C.c_void_p(int(stream) if stream else 0)))

    def set_model(self, cfg: GPT2Config):
        self._check(lib().tt_ctx_set_model(self.h, C.byref(cfg)))
        self.cfg = cfg

    def set_gemm_backend(self, backend: int):
        """0 automatic, 1 SIMT only, 2 tensor cores without the two-CTA pair form."""
        self._check(lib().tt_ctx_set_gemm_backend(self.h, int(backend)))

    def set_wait_limit(self, cycles: int):
        """Limit of the device-side bounded waits in clock64 cycles (<= 0: the default)."""
        self._check(lib().tt_ctx_set_wait_limit(self.h, int(cycles)))

    def reset(self):
        self._check(lib().tt_ctx_reset(self.h))

    def sync(self):
        self._check(lib().tt_ctx_sync(self.h))

    @property
    def capacity(self) -> int:
        return int(lib().tt_ctx_arena_capacity(self.h))

    @property
    def used(self) -> int:
        return int(lib().tt_ctx_arena_used(self.h))

    @property
    def high_water(self) -> int:
        return int(lib().tt_ctx_arena_high_water(self.h))

    @property
    def launches(self) -> int:
        return int(lib().tt_ctx_launch_count(self.h))

    def set_profiling(self, on: bool):
        self._check(lib().tt_ctx_set_profiling(self.h, int(bool(on))))

    def profile(self):
        """{op kind: dict(calls, ms, flops, bytes)} since profiling was switched on."""
        rows = (OpProfile * 32)()
        n = lib().tt_ctx_profile_read(self.h, rows, 32)
        if n < 0:
            self._check(n)
        return {rows[i].name.decode(): dict(calls=int(rows[i].calls), ms=rows[i].ms,
                                            flops=rows[i].flops, bytes=rows[i].bytes)
                for i in range(n)}

    @property
    def last_error(self) -> str:
        return lib().tt_last_error(self.h).decode()

    # -------------------------------------------------------------- training
    def step(self, params, grads, tokens, targets, B: int, T: int, sync: bool = True):
        """tt_gpt2_step; returns the mean loss (sync=True) or None."""
        loss = C.c_float()
        self._check(lib().tt_gpt2_step(self.h, _ptr(params), _ptr(grads), _ptr(tokens),
                                       _ptr(targets), int(B), int(T),
                                       C.byref(loss) if sync else None))
        return float(loss.value) if sync else None

    def step_ex(self, params, grads, tokens, targets, B: int, T: int, accumulate: bool = False,
                loss_scale=None, sync: bool = True):
        """tt_gpt2_step_ex: accumulate adds into grads; loss_scale is a device
        float (torch tensor) that scales the backward."""
        loss = C.c_float()
        self._check(lib().tt_gpt2_step_ex(self.h, _ptr(params), _ptr(grads), _ptr(tokens), _ptr(targets),
                                          int(B), int(T), 1 if accumulate else 0, _ptr(loss_scale),
                                          C.byref(loss) if sync else None))
        return float(loss.value) if sync else None

    def grad_stats(self, grads, stats, loss_scale=None, n=None):
        """stats (device float[2]) = (||grads / scale||, not finite)."""
        n = grads.numel() if n is None else n
        self._check(lib().tt_grad_stats(self.h, _ptr(grads), int(n), _ptr(loss_scale), _ptr(stats)))

    def adamw_ex(self, master, lowp, grads, m, v, lr, beta1, beta2, eps, weight_decay, step, stats=None,
                 max_norm=0.0, loss_scale=None, n=None):
        """tt_adamw_ex; step is a device int32 tensor (updates taken so far)."""
        n = master.numel() if n is None else n
        self._check_lowp(lowp)
        self._check(lib().tt_adamw_ex(self.h, _ptr(master), _ptr(lowp), _ptr(grads), _ptr(m), _ptr(v), int(n),
                                      float(lr), float(beta1), float(beta2), float(eps), float(weight_decay),
                                      _ptr(step), _ptr(stats), float(max_norm), _ptr(loss_scale)))

    def loss_scale_update(self, loss_scale, clean_steps, stats, window=1000, growth=1.001, backoff=0.5):
        self._check(lib().tt_loss_scale_update(self.h, _ptr(loss_scale), _ptr(clean_steps), _ptr(stats),
                                               int(window), float(growth), float(backoff)))

    def eval(self, params, tokens, targets, B: int, T: int) -> float:
        """tt_gpt2_eval: forward and mean loss only (synchronizes)."""
        loss = C.c_float()
        self._check(lib().tt_gpt2_eval(self.h, _ptr(params), _ptr(tokens), _ptr(targets), int(B), int(T),
                                       C.byref(loss)))
        return float(loss.value)

    def generate(self, params, prompt, B: int, T_prompt: int, n_new: int, out):
        """tt_gpt2_generate: greedy tokens; out [B, T_prompt + n_new] int32 (host or device)."""
        self._check(lib().tt_gpt2_generate(self.h, _ptr(params), _ptr(prompt), int(B), int(T_prompt), int(n_new),
                                           _ptr(out)))
        return out

    def loss_device(self):
        """(mean_loss_ptr, row_losses_ptr) device addresses of the last step."""
        a, b = C.c_void_p(), C.c_void_p()
        self._check(lib().tt_ctx_loss_device(self.h, C.byref(a), C.byref(b)))
        return a.value, b.value

    def row_losses(self, out):
        """Copy the last step's per-position losses into `out` (host or device)."""
        self._check(lib().tt_ctx_copy_row_losses(self.h, _ptr(out), int(out.numel() if hasattr(out, "numel") else out.size)))
        return out

    def _check_lowp(self, lowp):
        """The 16-bit parameter copy's element type follows the model's dtype:
        half for a TT_FP16 model, bf16 otherwise (torch tensors are checked)."""
        import torch

        dt = getattr(lowp, "dtype", None)
        if not isinstance(dt, torch.dtype):
            return
        want = torch.float16 if (self.cfg is not None and self.cfg.dtype == TT_FP16) else torch.bfloat16
        if dt != want:
            raise ValueError(f"the 16-bit parameter copy is {dt}; this context's model writes {want}")

    def adamw(self, master, lowp, grads, m, v, lr, beta1, beta2, eps, weight_decay, step, n=None):
        n = master.numel() if n is None else n
        self._check_lowp(lowp)
        self._check(lib().tt_adamw(self.h, _ptr(master), _ptr(lowp), _ptr(grads), _ptr(m), _ptr(v),
                                   int(n), lr, beta1, beta2, eps, weight_decay, int(step)))

    def cast_bf16(self, src, dst, n=None):
        n = src.numel() if n is None else n
        self._check(lib().tt_cast_f32_to_bf16(self.h, _ptr(src), _ptr(dst), int(n)))

    def cast_f16(self, src, dst, n=None):
        n = src.numel() if n is None else n
        self._check(lib().tt_cast_f32_to_f16(self.h, _ptr(src), _ptr(dst), int(n)))

    # -------------------------------------------------------------- ops
    def linear_fwd(self, dtype, x, W, b, residual, y, pre, M, K, N, gelu=False):
        self._check(lib().tt_op_linear_fwd(self.h, DTYPES[dtype], _ptr(x), _ptr(W), _ptr(b),
                                           _ptr(residual), _ptr(y), _ptr(pre), M, K, N, int(gelu)))

    def linear_bwd_dx(self, dtype, dy, W, pre, dx, M, K, N, accumulate=False):
        self._check(lib().tt_op_linear_bwd_dx(self.h, DTYPES[dtype], _ptr(dy), _ptr(W), _ptr(pre),
                                              _ptr(dx), M, K, N, int(accumulate)))

    def linear_bwd_dw(self, dtype, dy, x, dW, db, M, K, N):
        self._check(lib().tt_op_linear_bwd_dw(self.h, DTYPES[dtype], _ptr(dy), _ptr(x), _ptr(dW),
                                              _ptr(db), M, K, N))

    def attention_fwd(self, dtype, qkv, y, lse, B, T, C_, H):
        self._check(lib().tt_op_attention_fwd(self.h, DTYPES[dtype], _ptr(qkv), _ptr(y), _ptr(lse),
                                              B, T, C_, H))

    def attention_bwd(self, dtype, qkv, y, lse, dy, dqkv, B, T, C_, H):
        self._check(lib().tt_op_attention_bwd(self.h, DTYPES[dtype], _ptr(qkv), _ptr(y), _ptr(lse),
                                              _ptr(dy), _ptr(dqkv), B, T, C_, H))

    def layernorm_fwd(self, dtype, x, w, b, y, mean, rstd, M, C_):
        self._check(lib().tt_op_layernorm_fwd(self.h, DTYPES[dtype], _ptr(x), _ptr(w), _ptr(b),
                                              _ptr(y), _ptr(mean), _ptr(rstd), M, C_))

    def layernorm_bwd(self, dtype, x, w, mean, rstd, dy, dx, dw, db, M, C_, accumulate=False):
        self._check(lib().tt_op_layernorm_bwd(self.h, DTYPES[dtype], _ptr(x), _ptr(w), _ptr(mean),
                                              _ptr(rstd), _ptr(dy), _ptr(dx), _ptr(dw), _ptr(db),
                                              M, C_, int(accumulate)))

    def xent(self, dtype, logits, targets, row_loss, mean_loss, M, V, ld, dscale):
        self._check(lib().tt_op_xent(self.h, DTYPES[dtype], _ptr(logits), _ptr(targets),
                                     _ptr(row_loss), _ptr(mean_loss), M, V, ld, float(dscale)))

    def embed_fwd(self, dtype, wte, wpe, tokens, x, B, T, C_, V):
        self._check(lib().tt_op_embed_fwd(self.h, DTYPES[dtype], _ptr(wte), _ptr(wpe), _ptr(tokens),
                                          _ptr(x), B, T, C_, V))

    def embed_bwd(self, dtype, dx, tokens, dwte, dwpe, B, T, C_, V, maxT):
        self._check(lib().tt_op_embed_bwd(self.h, DTYPES[dtype], _ptr(dx), _ptr(tokens), _ptr(dwte),
                                          _ptr(dwpe), B, T, C_, V, maxT))

    # -------------------------------------------------------------- generic graph (tt_graph.h)
    def _node(self, h: int) -> int:
        if h < 0:
            raise TTError(h, lib().tt_last_error(self.h).decode())
        return h

    def tensor(self, *shape, dtype: str = "f32") -> "Node":
        """A new leaf of the given shape (values zero); dtype "f32" or "i32"."""
        n = len(shape)
        arr = (C.c_int * max(n, 1))(*[int(d) for d in shape])
        return Node(self, self._node(lib().tt_node_new(self.h, n, arr, NODE_I32 if dtype == "i32" else NODE_F32)))

    def sgd(self, params, lr: float):
        """p -= lr * grad on the device for each node of params."""
        hs = (C.c_int * max(len(params), 1))(*[p.h for p in params])
        self._check(lib().tt_node_sgd(self.h, hs, len(params), float(lr)))

    def capture_begin(self):
        self._check(lib().tt_capture_begin(self.h))

    def capture_end(self):
        self._check(lib().tt_capture_end(self.h))

    def replay(self, times: int = 1):
        self._check(lib().tt_replay(self.h, int(times)))

    def record(self, fn):
        """Record the graph calls fn() makes (run nothing); replay() runs them."""
        self.capture_begin()
        try:
            fn()
        except BaseException:
            try:
                self.capture_end()
            except TTError:
                pass
            raise
        self.capture_end()


# ---------------------------------------------------------------- generic tensor graph
NODE_F32, NODE_I32 = 0, 1


class Node:
    """A tensor of a context's generic graph (tt_graph.h).  Operators build
    new nodes; forward / zero_grad / backward / fill / numpy run on the
    device through the C ABI."""

    def __init__(self, ctx: "Context", h: int):
        self.ctx = ctx
        self.h = int(h)

    def _made(self, h):
        return Node(self.ctx, self.ctx._node(h))

    def matmul(self, other: "Node") -> "Node":
        return self._made(lib().tt_node_matmul(self.ctx.h, self.h, other.h))

    __matmul__ = matmul

    def __add__(self, other: "Node") -> "Node":
        return self._made(lib().tt_node_add(self.ctx.h, self.h, other.h))

    def __mul__(self, other: "Node") -> "Node":
        return self._made(lib().tt_node_mul(self.ctx.h, self.h, other.h))

    def gelu(self) -> "Node":
        return self._made(lib().tt_node_gelu(self.ctx.h, self.h))

    def softmax(self) -> "Node":
        return self._made(lib().tt_node_softmax(self.ctx.h, self.h))

    def cross_entropy(self, labels: "Node") -> "Node":
        return self._made(lib().tt_node_cross_entropy(self.ctx.h, self.h, labels.h))

    def forward(self):
        self.ctx._check(lib().tt_node_forward(self.ctx.h, self.h))

    def zero_grad(self):
        self.ctx._check(lib().tt_node_zero_grad(self.ctx.h, self.h))

    def backward(self):
        self.ctx._check(lib().tt_node_backward(self.ctx.h, self.h))

    def info(self):
        nd, shp = C.c_int(), (C.c_int * 4)()
        data, grad = C.c_void_p(), C.c_void_p()
        self.ctx._check(lib().tt_node_info(self.ctx.h, self.h, C.byref(nd), shp, C.byref(data), C.byref(grad)))
        return tuple(shp[:nd.value]), data.value, grad.value

    @property
    def shape(self):
        return self.info()[0]

    def fill(self, values):
        """values: numpy array (host) or torch tensor (device) of the node's size."""
        import numpy as np
        if hasattr(values, "data_ptr"):
            src, n = values, values.numel()
        else:
            src = np.ascontiguousarray(values)
            n = src.size
        self.ctx._check(lib().tt_node_fill(self.ctx.h, self.h, C.c_void_p(_ptr(src)), n))
        return self

    def numpy(self, grad: bool = False):
        import math

        import numpy as np
        shp, _, g = self.info()
        if grad and g is None:
            raise ValueError("an int32 node has no gradient")
        out = np.zeros(shp, dtype=np.float32 if (grad or g is not None) else np.int32)
        self.ctx._check(lib().tt_node_read(self.ctx.h, self.h, 1 if grad else 0, C.c_void_p(out.ctypes.data),
                                           math.prod(shp)))
        return out

    def grad(self):
        return self.numpy(grad=True)


