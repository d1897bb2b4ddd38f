"""Failure detection on the device without a fault: a bounded wait that runs
out.  With the context's wait limit at one cycle, the first device-side wait
that is not already complete when it starts gives up.  The kernel records the
timeout and a code naming the wait, lets its issued copies and MMAs finish,
frees its tensor memory and returns; tt_ctx_sync reports TT_ERR_TIMEOUT;
after tt_ctx_reset, with the default limit again, the same context computes
the right result.  (The microcrad page's boundary reports failure through a
status code; this is the device-side wait's status.)"""
import numpy as np
import pytest
import torch

from autograd_arena_allocated_gb300 import api, synth
from autograd_arena_allocated_gb300 import build as native_build

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ctx():
    native_build.build()
    c = api.Context(1 << 30)
    yield c
    c.close()


def rnd(seed, *shape, scale=1.0):
    n = int(np.prod(shape))
    return (synth.normals(seed, 0, n) * scale).astype(np.float32).reshape(shape)


def bf(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV).to(torch.bfloat16)


def test_gemm_wait_runs_out_and_context_recovers(ctx, oracle):
    """Single-CTA tensor-core GEMM (no pair form) with a long main loop
    (K = 16384): the epilogue's first wait, for an accumulator that needs the
    whole main loop, cannot be complete when it starts."""
    M, K, N = 256, 16384, 256
    x, W = rnd(11, M, K), rnd(12, N, K, scale=0.02)
    xd, Wd = bf(x), bf(W)
    y = torch.empty(M, N, device=DEV, dtype=torch.bfloat16)
    ctx.set_gemm_backend(2)
    try:
        ctx.reset()
        ctx.set_wait_limit(1)  # one cycle: a wait not complete at its start runs out
        ctx.linear_fwd("bf16", xd, Wd, None, None, y, None, M, K, N)
        with pytest.raises(api.TTError, match="TT_ERR_TIMEOUT") as ei:
            ctx.sync()
        assert "site 0x4" in str(ei.value), str(ei.value)  # a wait of the GEMM kernel
        print(f"[gemm timeout] {ei.value}")
        # the context recovers: reset clears the flag
        ctx.set_wait_limit(-1)
        ctx.reset()
        ctx.linear_fwd("bf16", xd, Wd, None, None, y, None, M, K, N)
        ctx.sync()
    finally:
        ctx.set_wait_limit(-1)
        ctx.set_gemm_backend(0)
    ref = oracle.linear_fwd(oracle.bf16_values(x).reshape(M, K), oracle.bf16_values(W).reshape(N, K), None)
    got = y.float().cpu().numpy().astype(np.float64)
    # bf16 output rounding plus fp32 accumulation over K = 16384
    assert np.all(np.abs(got - ref) <= 2 ** -8 * np.abs(ref) + 1e-3 * np.sqrt(np.mean(ref ** 2)))


def test_attention_wait_runs_out_and_context_recovers(ctx, oracle):
    """The tensor-core attention forward (B=1, T=1024, two heads of 64): its
    row warps wait for every block's scores, which cannot all be ready when
    the waits start."""
    B, T, C_, H = 1, 1024, 128, 2
    qkv = rnd(21, B * T, 3 * C_)
    qd = bf(qkv)
    y = torch.empty(B * T, C_, device=DEV, dtype=torch.bfloat16)
    lse = torch.empty(B, H, T, device=DEV)
    try:
        ctx.reset()
        ctx.set_wait_limit(1)  # one cycle: a wait not complete at its start runs out
        ctx.attention_fwd("bf16", qd, y, lse, B, T, C_, H)
        with pytest.raises(api.TTError, match="TT_ERR_TIMEOUT") as ei:
            ctx.sync()
        assert "site 0x1" in str(ei.value), str(ei.value)  # a wait of the attention forward
        print(f"[attention timeout] {ei.value}")
        ctx.set_wait_limit(-1)
        ctx.reset()
        ctx.attention_fwd("bf16", qd, y, lse, B, T, C_, H)
        ctx.sync()
    finally:
        ctx.set_wait_limit(-1)
    ry, _, rlse = oracle.attention_fwd(oracle.bf16_values(qkv).reshape(B * T, 3 * C_), B, T, C_, H,
                                       want_lse=True)
    got = y.float().cpu().numpy().astype(np.float64)
    assert np.linalg.norm(got - ry) / np.linalg.norm(ry) < 5e-3
    assert np.max(np.abs(lse.cpu().numpy() - rlse)) < 1e-4


def test_wait_limit_and_backend_arguments(ctx):
    with pytest.raises(api.TTError, match="TT_ERR_ARG"):
        ctx.set_gemm_backend(3)
    ctx.set_wait_limit(123456789)
    ctx.set_wait_limit(-5)  # <= 0: the default again
    ctx.set_gemm_backend(0)
