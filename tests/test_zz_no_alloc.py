"""tt_linear_bwd_dw_noalloc: the weight-gradient GEMM for callers that cannot
allocate device memory (their GPU memory belongs to another allocator, so a
library must not call cudaMalloc for them, and they cannot create a tt_ctx,
whose arena is one cudaMalloc).  The call keeps its scratch in a fixed array
inside libtt.so and takes a stream instead of a context.

Checked through the C ABI against the existing entry point,
tt_op_linear_bwd_dw, on two calls in a row (the shared scratch keeps the
first call's contents when the second runs), with the tolerance the other
weight-gradient tests use.  This file is named to be collected last."""
import ctypes as C

import numpy as np
import pytest
import torch

from autograd_arena_allocated_gb300 import _native, api, synth
from autograd_arena_allocated_gb300 import build as native_build

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rnd(seed, *shape):
    n = int(np.prod(shape))
    return torch.from_numpy(synth.normals(seed, 0, n).astype(np.float32).reshape(shape)).to(DEV)


def _close(got, ref, rtol=2e-5, atol_frac=1e-5):
    got = got.double().cpu().numpy()
    ref = ref.double().cpu().numpy()
    scale = np.sqrt(np.mean(ref ** 2)) + 1e-30
    assert np.all(np.abs(got - ref) <= rtol * np.abs(ref) + atol_frac * scale)


def test_noalloc_weight_gradient_matches_context_entry_point():
    native_build.build()
    lib = _native.lib()
    stream = torch.cuda.current_stream()
    shapes = [(4096, 768, 768), (3000, 256, 2304)]  # (M tokens, K in, N out)
    with api.Context(1 << 28) as ctx:
        for i, (M, K, N) in enumerate(shapes):
            dy = _rnd(900 + i, M, N).to(torch.bfloat16)
            x = _rnd(950 + i, M, K).to(torch.bfloat16)
            ref_w = torch.empty(N, K, device=DEV)
            ref_b = torch.empty(N, device=DEV)
            ctx.reset()
            ctx.linear_bwd_dw("bf16", dy, x, ref_w, ref_b, M, K, N)
            got_w = torch.full((N, K), float("nan"), device=DEV)
            got_b = torch.full((N,), float("nan"), device=DEV)
            rc = lib.tt_linear_bwd_dw_noalloc(C.c_void_p(stream.cuda_stream), dy.data_ptr(),
                                              x.data_ptr(), got_w.data_ptr(), got_b.data_ptr(),
                                              M, K, N)
            assert rc == 0
            torch.cuda.synchronize()
            _close(got_w, ref_w)
            _close(got_b, ref_b)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    native_build.build()
    lib = _native.lib()
    # bias partial sums: ceil(M/256) * N floats must fit TT_NOALLOC_BIAS_FLOATS;
    # the buffers are full size, so even a wrong answer would stay in bounds
    M, N, K = 32768, 16392, 8
    dy = torch.zeros(M, N, device=DEV, dtype=torch.bfloat16)
    x = torch.zeros(M, K, device=DEV, dtype=torch.bfloat16)
    w = torch.zeros(N, K, device=DEV)
    b = torch.zeros(N, device=DEV)
    rc = lib.tt_linear_bwd_dw_noalloc(None, dy.data_ptr(), x.data_ptr(), w.data_ptr(),
                                      b.data_ptr(), M, K, N)
    assert rc == -2  # TT_ERR_ARG, before anything is launched
    assert lib.tt_linear_bwd_dw_noalloc(None, None, x.data_ptr(), w.data_ptr(), None, M, K, N) == -2
    # without the bias the same shape is accepted
    assert lib.tt_linear_bwd_dw_noalloc(None, dy.data_ptr(), x.data_ptr(), w.data_ptr(), None,
                                        M, K, N) == 0
    torch.cuda.synchronize()
    assert torch.all(w == 0)
