"""ctypes declarations of the C ABI in include/tt.h, include/tt_ops.h and
include/tt_graph.h.

The shared library libtt.so is built in-tree by build.py.  There is no
fallback: if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtt.so")

TT_OK = 0
STATUS_NAMES = {
    0: "TT_OK", -1: "TT_ERR", -2: "TT_ERR_ARG", -3: "TT_ERR_ARENA_OOM", -4: "TT_ERR_CUDA",
    -5: "TT_ERR_TIMEOUT", -6: "TT_ERR_NONFINITE", -7: "TT_ERR_STALE", -8: "TT_ERR_STATE",
}
TT_FP32, TT_BF16, TT_FP16 = 0, 1, 2


class GPT2Config(C.Structure):
    _fields_ = [("L", C.c_int), ("C", C.c_int), ("H", C.c_int), ("V", C.c_int),
                ("maxT", C.c_int), ("dtype", C.c_int)]


class OpProfile(C.Structure):
    _fields_ = [("name", C.c_char * 24), ("calls", C.c_uint64), ("ms", C.c_double),
                ("flops", C.c_double), ("bytes", C.c_double)]


_vp = C.c_void_p
_i = C.c_int
_sz = C.c_size_t
_f = C.c_float
_st = C.c_int  # tt_status

SIGNATURES = {
    # tt.h
    "tt_ctx_create": (_st, [_sz, C.POINTER(_vp)]),
    "tt_ctx_destroy": (None, [_vp]),
    "tt_ctx_set_stream": (_st, [_vp, _vp]),
    "tt_ctx_set_model": (_st, [_vp, C.POINTER(GPT2Config)]),
    "tt_ctx_reset": (_st, [_vp]),
    "tt_ctx_sync": (_st, [_vp]),
    "tt_ctx_arena_capacity": (_sz, [_vp]),
    "tt_ctx_arena_used": (_sz, [_vp]),
    "tt_ctx_arena_high_water": (_sz, [_vp]),
    "tt_ctx_launch_count": (C.c_uint64, [_vp]),
    "tt_last_error": (C.c_char_p, [_vp]),
    "tt_ctx_set_profiling": (_st, [_vp, _i]),
    "tt_ctx_profile_read": (_i, [_vp, C.POINTER(OpProfile), _i]),
    "tt_gpt2_num_params": (_sz, [C.POINTER(GPT2Config)]),
    "tt_gpt2_param_offset": (_st, [C.POINTER(GPT2Config), _i, _i, C.POINTER(_sz), C.POINTER(_sz)]),
    "tt_gpt2_arena_bytes": (_sz, [C.POINTER(GPT2Config), _i, _i]),
    "tt_gpt2_step": (_st, [_vp, _vp, _vp, _vp, _vp, _i, _i, C.POINTER(_f)]),
    "tt_ctx_loss_device": (_st, [_vp, C.POINTER(_vp), C.POINTER(_vp)]),
    "tt_ctx_copy_row_losses": (_st, [_vp, _vp, _sz]),
    "tt_adamw": (_st, [_vp, _vp, _vp, _vp, _vp, _vp, _sz, _f, _f, _f, _f, _f, _i]),
    "tt_cast_f32_to_bf16": (_st, [_vp, _vp, _vp, _sz]),
    "tt_cast_f32_to_f16": (_st, [_vp, _vp, _vp, _sz]),
    "tt_gpt2_eval": (_st, [_vp, _vp, _vp, _vp, _i, _i, C.POINTER(C.c_float)]),
    "tt_gpt2_step_ex": (_st, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _vp, C.POINTER(_f)]),
    "tt_grad_stats": (_st, [_vp, _vp, _sz, _vp, _vp]),
    "tt_adamw_ex": (_st, [_vp, _vp, _vp, _vp, _vp, _vp, _sz, _f, _f, _f, _f, _f, _vp, _vp, _f, _vp]),
    "tt_loss_scale_update": (_st, [_vp, _vp, _vp, _vp, _i, _f, _f]),
    "tt_gpt2_generate_arena_bytes": (_sz, [_vp, _i, _i, _i]),
    "tt_gpt2_generate": (_st, [_vp, _vp, _vp, _i, _i, _i, _vp]),
    # tt_ops.h
    "tt_ctx_set_gemm_backend": (_st, [_vp, _i]),
    "tt_ctx_set_wait_limit": (_st, [_vp, C.c_longlong]),
    "tt_op_linear_fwd": (_st, [_vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i]),
    "tt_op_linear_bwd_dx": (_st, [_vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i]),
    "tt_op_linear_bwd_dw": (_st, [_vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i]),
    "tt_op_attention_fwd": (_st, [_vp, _i, _vp, _vp, _vp, _i, _i, _i, _i]),
    "tt_op_attention_bwd": (_st, [_vp, _i, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i]),
    "tt_op_layernorm_fwd": (_st, [_vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i]),
    "tt_op_layernorm_bwd": (_st, [_vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i]),
    "tt_op_xent": (_st, [_vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _f]),
    "tt_op_embed_fwd": (_st, [_vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i]),
    "tt_op_embed_bwd": (_st, [_vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i]),
    "tt_linear_bwd_dw_noalloc": (_st, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i]),
    # tt_graph.h (node handles are int32; negative = tt_status)
    "tt_node_new": (_i, [_vp, _i, C.POINTER(_i), _i]),
    "tt_node_matmul": (_i, [_vp, _i, _i]),
    "tt_node_add": (_i, [_vp, _i, _i]),
    "tt_node_mul": (_i, [_vp, _i, _i]),
    "tt_node_gelu": (_i, [_vp, _i]),
    "tt_node_softmax": (_i, [_vp, _i]),
    "tt_node_cross_entropy": (_i, [_vp, _i, _i]),
    "tt_node_forward": (_st, [_vp, _i]),
    "tt_node_zero_grad": (_st, [_vp, _i]),
    "tt_node_backward": (_st, [_vp, _i]),
    "tt_node_fill": (_st, [_vp, _i, _vp, _sz]),
    "tt_node_read": (_st, [_vp, _i, _i, _vp, _sz]),
    "tt_node_info": (_st, [_vp, _i, C.POINTER(_i), C.POINTER(_i), C.POINTER(_vp), C.POINTER(_vp)]),
    "tt_node_sgd": (_st, [_vp, C.POINTER(_i), _i, _f]),
    "tt_capture_begin": (_st, [_vp]),
    "tt_capture_end": (_st, [_vp]),
    "tt_replay": (_st, [_vp, _i]),
}

_lib = None


def lib():
    """Load libtt.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "autograd_arena_allocated_gb300.build.build() (there is no CPU fallback)")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


class TTError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
