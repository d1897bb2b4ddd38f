"""Per-kernel parity: each op of the C ABI (include/tt_ops.h) against the
oracle on the same seeded inputs, at sizes that span several tiles with
ragged tails.  Tolerances: fp32 mode ~1e-5 relative (fp32 accumulation);
bf16 mode bounded by bf16 output rounding (2^-9 relative) plus fp32
accumulation error, written per test."""
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


_seed = [100]


def rnd(*shape, scale=1.0):
    _seed[0] += 1
    n = int(np.prod(shape))
    return (synth.normals(_seed[0], 0, n) * scale).astype(np.float32).reshape(shape)


def to_dev(a, dt):
    t = torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    return t.to(torch.bfloat16) if dt == "bf16" else t.float()


def ovals(a, dt, oracle):
    return oracle.bf16_values(a).reshape(a.shape) if dt == "bf16" else a.astype(np.float64)


def host(t):
    return t.float().cpu().numpy().astype(np.float64)


def assert_close(got, ref, rtol, atol_frac, what=""):
    """|got - ref| <= rtol*|ref| + atol_frac*rms(ref), element-wise."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), what
    scale = np.sqrt(np.mean(ref ** 2)) + 1e-30
    err = np.abs(got - ref)
    bound = rtol * np.abs(ref) + atol_frac * scale
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} / {err.size} outside tolerance; worst at {i}: "
                             f"got {got[i]} ref {ref[i]} (rms {scale})")


TOL = {"fp32": (2e-5, 1e-5), "bf16": (8e-3, 4e-3)}


# ----------------------------------------------------------------- linear
@pytest.mark.parametrize("dt,backend", [("fp32", 1), ("bf16", 1), ("bf16", 0)])
@pytest.mark.parametrize("M,K,N", [(200, 64, 96), (300, 192, 520), (512, 768, 2304), (129, 3072, 768)])
@pytest.mark.parametrize("variant", ["plain", "bias_res", "gelu"])
def test_linear_fwd(ctx, oracle, dt, backend, M, K, N, variant):
    ctx.set_gemm_backend(backend)
    x, W, b, r = rnd(M, K), rnd(N, K, scale=0.05), rnd(N, scale=0.1), rnd(M, N)
    xd, Wd, bd, rd = (to_dev(a, dt) for a in (x, W, b, r))
    y = torch.empty(M, N, device=DEV, dtype=xd.dtype)
    pre = torch.empty_like(y) if variant == "gelu" else None
    ctx.linear_fwd(dt, xd, Wd, bd if variant != "plain" else None,
                   rd if variant == "bias_res" else None, y, pre, M, K, N, gelu=variant == "gelu")
    torch.cuda.synchronize()
    u = oracle.linear_fwd(ovals(x, dt, oracle), ovals(W, dt, oracle),
                          ovals(b, dt, oracle) if variant != "plain" else None)
    rtol, atol = TOL[dt]
    if variant == "gelu":
        assert_close(host(pre), u, rtol, atol, "pre-activation")
        ref = oracle.gelu_fwd(u)
    elif variant == "bias_res":
        ref = u + ovals(r, dt, oracle)
    else:
        ref = u
    assert_close(host(y), ref, rtol, atol, f"linear fwd {variant}")
    ctx.set_gemm_backend(0)


@pytest.mark.parametrize("dt,backend", [("fp32", 1), ("bf16", 1), ("bf16", 0)])
@pytest.mark.parametrize("M,K,N", [(200, 64, 96), (300, 520, 192), (256, 768, 3072), (130, 3072, 768)])
@pytest.mark.parametrize("variant", ["plain", "dgelu", "accumulate"])
def test_linear_bwd_dx(ctx, oracle, dt, backend, M, K, N, variant):
    ctx.set_gemm_backend(backend)
    dy, W, pre, dx0 = rnd(M, N), rnd(N, K, scale=0.05), rnd(M, K), rnd(M, K)
    dyd, Wd, pred = (to_dev(a, dt) for a in (dy, W, pre))
    dx = to_dev(dx0, dt) if variant == "accumulate" else torch.empty(M, K, device=DEV, dtype=dyd.dtype)
    ctx.linear_bwd_dx(dt, dyd, Wd, pred if variant == "dgelu" else None, dx, M, K, N,
                      accumulate=variant == "accumulate")
    torch.cuda.synchronize()
    ref, _, _ = oracle.linear_bwd(np.zeros((M, K)), ovals(W, dt, oracle), ovals(dy, dt, oracle),
                                  with_bias=False)
    if variant == "dgelu":
        ref = oracle.gelu_bwd(ovals(pre, dt, oracle), ref)
    if variant == "accumulate":
        ref = ref + ovals(dx0, dt, oracle)
    rtol, atol = TOL[dt]
    assert_close(host(dx), ref, rtol, atol, f"linear dx {variant}")
    ctx.set_gemm_backend(0)


@pytest.mark.parametrize("dt,backend", [("fp32", 1), ("bf16", 1), ("bf16", 0)])
@pytest.mark.parametrize("M,K,N", [(200, 64, 96), (4096, 256, 192), (1000, 768, 2304), (2048, 3072, 768),
                                   (600, 512, 384)])  # 3 row tiles of dW: the pair form's odd count
def test_linear_bwd_dw(ctx, oracle, dt, backend, M, K, N):
    ctx.set_gemm_backend(backend)
    dy, x = rnd(M, N), rnd(M, K)
    dyd, xd = to_dev(dy, dt), to_dev(x, dt)
    dW = torch.empty(N, K, device=DEV)
    db = torch.empty(N, device=DEV)
    ctx.linear_bwd_dw(dt, dyd, xd, dW, db, M, K, N)
    torch.cuda.synchronize()
    _, rW, rb = oracle.linear_bwd(ovals(x, dt, oracle), np.zeros((N, K)), ovals(dy, dt, oracle))
    # fp32 outputs: only accumulation-order error (sums of M products)
    assert_close(host(dW), rW, 2e-5, 1e-5, "dW")
    assert_close(host(db), rb, 2e-5, 1e-5, "db")
    # deterministic: a second call gives the same bits
    dW2 = torch.empty_like(dW)
    ctx.linear_bwd_dw(dt, dyd, xd, dW2, None, M, K, N)
    torch.cuda.synchronize()
    assert torch.equal(dW, dW2)
    ctx.set_gemm_backend(0)


# ----------------------------------------------------------------- attention
SUM_ROUNDINGS = 12.0  # random-walk part of the bound: 12 x 2^-9 x root-sum-square


def _attention_sum_scales(qkv, dy, P, y, B, T, C_, H):
    """Error scales, in units of the bf16 unit roundoff u = 2^-9, of each
    element of y and of dqkv in bf16 mode (the oracle's exact P, y as inputs).

    * Random-walk part: one factor of every product the kernels add up carries
      one bf16 rounding (P in P.V and P^T.dO; dS in dS.K and dS^T.Q) and the
      sums run in fp32, so an element's error is a sum of independent terms of
      relative size <= u: SUM_ROUNDINGS x the root-sum-square of the products
      (|dS| bounded by P (|dP| + |D|)).
    * Coherent part (dQ, dK): D = rowsum(dO o y) is formed from the kernel's
      own bf16 y, whose error is within u |y| + SUM_ROUNDINGS u rss(y); that
      error e_q of D_q enters every dS[q, k] as -P[q, k] e_q, so it is bounded
      by sum_k P |e_q| |K| (and sum_q P |e_q| |Q| for dK).
    Returns (scale_y, scale_dqkv): the bound is u |ref| + u x scale."""
    hd = C_ // H
    sc = 1.0 / np.sqrt(hd)
    sy = np.zeros((B * T, C_))
    sd = np.zeros((B * T, 3 * C_))
    for b in range(B):
        rows = slice(b * T, (b + 1) * T)
        for h in range(H):
            cq, ck, cv = (slice(j * C_ + h * hd, j * C_ + (h + 1) * hd) for j in range(3))
            q, k, v = qkv[rows, cq], qkv[rows, ck], qkv[rows, cv]
            do = dy[rows, h * hd:(h + 1) * hd]
            yh = y[rows, h * hd:(h + 1) * hd]
            p = P[b, h]
            dp = do @ v.T
            a = p * (np.abs(dp) + np.abs(np.sum(p * dp, axis=1))[:, None])
            rss_y = np.sqrt((p ** 2) @ (v ** 2))
            e = np.sum(np.abs(do) * (np.abs(yh) + SUM_ROUNDINGS * rss_y), axis=1)  # |D_q error| / u
            pe = p * e[:, None]
            sy[rows, h * hd:(h + 1) * hd] = SUM_ROUNDINGS * rss_y
            sd[rows, cq] = SUM_ROUNDINGS * np.sqrt((a ** 2) @ (k ** 2)) * sc + (pe @ np.abs(k)) * sc
            sd[rows, ck] = SUM_ROUNDINGS * np.sqrt((a ** 2).T @ (q ** 2)) * sc + (pe.T @ np.abs(q)) * sc
            sd[rows, cv] = SUM_ROUNDINGS * np.sqrt((p ** 2).T @ (do ** 2))
    return sy, sd


def _check_attention(dt, got_y, got_lse, got_dqkv, ry, rlse, rd, scales=None):
    """y, the saved log-sum-exp and dqkv against the oracle, element by element.
    fp32 mode: fp32-level relative tolerances.  bf16 mode: each element within
    its output's bf16 rounding (2^-9 relative) plus 2^-9 x its error scale
    from the arithmetic (_attention_sum_scales), which covers long rows (1024
    keys) as well as short ones.  The log-sum-exp
    is accumulated in fp32 from the exact products of the same 16-bit q and k,
    so it is held to fp32-level error."""
    err = np.abs(got_lse - rlse)
    assert np.all(err <= 2e-5 * np.abs(rlse) + 1e-4), f"lse: worst abs err {np.max(err):.3e}"
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    worst = 0.0
    if dt == "fp32":
        rtol, atol = TOL[dt]
        assert_close(got_y, ry, rtol, atol, "attention y")
        assert_close(got_dqkv, rd, 4 * rtol, 2 * atol, "attention dqkv")
    else:
        sy, sd = scales
        u = 2.0 ** -9
        for what, got, ref, sc in (("y", got_y, ry, sy), ("dqkv", got_dqkv, rd, sd)):
            e = np.abs(got - ref)
            floor = 1e-6 * np.sqrt(np.mean(ref ** 2))
            bound = u * np.abs(ref) + u * sc + floor
            bad = e > bound
            if bad.any():
                i = np.unravel_index(np.argmax(e - bound), e.shape)
                raise AssertionError(f"attention {what}: {bad.sum()} / {e.size} outside the bound; worst at "
                                     f"{i}: got {got[i]} ref {ref[i]} bound {bound[i]:.3e}")
            # the largest error as a fraction of its bound (printed)
            worst = max(worst, float(np.max(e / bound)))
        assert rel(got_y, ry) < 5e-3
        assert rel(got_dqkv, rd) < 1e-2
    return rel(got_y, ry), float(np.max(err)), rel(got_dqkv, rd), worst


# (6, 256, 768, 12): 72 (batch, head) pairs, i.e. two bands of 64 pairs with
# the second band's 56 unused slots; (1, 1024, 128, 2): the benchmark's
# sequence length, every key tile of a 1024-long row.
@pytest.mark.parametrize("dt,B,T,C_,H", [("fp32", 2, 37, 64, 4), ("fp32", 1, 70, 64, 2),
                                         ("bf16", 2, 100, 128, 2), ("bf16", 1, 257, 384, 6),
                                         ("bf16", 3, 1, 128, 2), ("bf16", 6, 256, 768, 12),
                                         ("bf16", 1, 1024, 128, 2), ("fp32", 5, 70, 960, 15)])
def test_attention(ctx, oracle, dt, B, T, C_, H):
    qkv, dy = rnd(B * T, 3 * C_), rnd(B * T, C_)
    qd, dyd = to_dev(qkv, dt), to_dev(dy, dt)
    y = torch.empty(B * T, C_, device=DEV, dtype=qd.dtype)
    lse = torch.empty(B, H, T, device=DEV)
    ctx.attention_fwd(dt, qd, y, lse, B, T, C_, H)
    dqkv = torch.empty_like(qd)
    ctx.attention_bwd(dt, qd, y, lse, dyd, dqkv, B, T, C_, H)
    torch.cuda.synchronize()
    q64, dy64 = ovals(qkv, dt, oracle), ovals(dy, dt, oracle)
    ry, P, rlse = oracle.attention_fwd(q64, B, T, C_, H, want_lse=True)
    rd = oracle.attention_bwd(q64, P, dy64, B, T, C_, H)
    scales = _attention_sum_scales(q64, dy64, P, ry, B, T, C_, H) if dt == "bf16" else None
    e = _check_attention(dt, host(y), host(lse), host(dqkv), ry, rlse, rd, scales)
    print(f"[attention {dt} B={B} T={T} H={H}] y rel-L2 {e[0]:.2e}, lse max abs err {e[1]:.2e}, "
          f"dqkv rel-L2 {e[2]:.2e}, worst error {e[3]:.2f} of its bound")


def test_attention_benchmark_shape_sampled(ctx, oracle):
    """The step's own attention call at the benchmark's size (B=32, T=1024,
    C=768, H=12: 384 (batch, head) pairs in six bands), in the launch
    configuration the step uses.  (batch, head) pairs are independent, so
    sampled pairs -- the first and last of a band, either side of a band edge,
    and the last pair -- are each checked against the oracle run on that
    pair's head alone."""
    B, T, C_, H = 32, 1024, 768, 12
    D = C_ // H
    qkv, dy = rnd(B * T, 3 * C_), rnd(B * T, C_)
    qd, dyd = to_dev(qkv, "bf16"), to_dev(dy, "bf16")
    with api.Context(4 << 30) as big:
        y = torch.empty(B * T, C_, device=DEV, dtype=qd.dtype)
        lse = torch.empty(B, H, T, device=DEV)
        big.attention_fwd("bf16", qd, y, lse, B, T, C_, H)
        dqkv = torch.empty_like(qd)
        big.attention_bwd("bf16", qd, y, lse, dyd, dqkv, B, T, C_, H)
        torch.cuda.synchronize()
    q16 = ovals(qkv, "bf16", oracle)
    dy16 = ovals(dy, "bf16", oracle)
    y_h, lse_h, dqkv_h = host(y), host(lse), host(dqkv)
    for pair in (0, 63, 64, 200, 383):
        b, h = divmod(pair, H)
        rows = slice(b * T, (b + 1) * T)
        cols = [slice(j * C_ + h * D, j * C_ + (h + 1) * D) for j in range(3)]
        one = np.ascontiguousarray(np.concatenate([q16[rows, c] for c in cols], axis=1))
        ry, P, rlse = oracle.attention_fwd(one, 1, T, D, 1, want_lse=True)
        rd = oracle.attention_bwd(one, P, np.ascontiguousarray(dy16[rows, h * D:(h + 1) * D]), 1, T, D, 1)
        got_d = np.concatenate([dqkv_h[rows, c] for c in cols], axis=1)
        dy_one = np.ascontiguousarray(dy16[rows, h * D:(h + 1) * D])
        e = _check_attention("bf16", y_h[rows, h * D:(h + 1) * D], lse_h[b, h][None, None, :], got_d,
                             ry, rlse, rd, _attention_sum_scales(one, dy_one, P, ry, 1, T, D, 1))
        print(f"[attention B=32 T=1024 pair {pair}] y rel-L2 {e[0]:.2e}, lse max abs err {e[1]:.2e}, "
              f"dqkv rel-L2 {e[2]:.2e}, worst error {e[3]:.2f} of its bound")


@pytest.mark.parametrize("T", [384, 1000])
def test_attention_growing_max(ctx, oracle, T):
    """Score rows whose maximum keeps rising along the keys (odd rows) beside
    rows whose maximum is the first key (even rows), so that the online
    softmax's running maximum is raised many times for some rows of a warp and
    never for their neighbours; the scores span ~30 in log2 units."""
    B, C_, H = 1, 128, 2
    D = C_ // H
    qkv = rnd(B * T, 3 * C_, scale=0.5)
    sign = np.where(np.arange(T) % 2 == 1, 1.0, -1.0).astype(np.float32)
    ramp = (24.0 * np.arange(T) / T).astype(np.float32)
    for h in range(H):
        qkv[:, h * D] = 6.0 * sign                # q . e0
        qkv[:, C_ + h * D] = ramp                 # k . e0 grows with the key position
    dy = rnd(B * T, C_)
    qd, dyd = to_dev(qkv, "bf16"), to_dev(dy, "bf16")
    y = torch.empty(B * T, C_, device=DEV, dtype=qd.dtype)
    lse = torch.empty(B, H, T, device=DEV)
    ctx.attention_fwd("bf16", qd, y, lse, B, T, C_, H)
    dqkv = torch.empty_like(qd)
    ctx.attention_bwd("bf16", qd, y, lse, dyd, dqkv, B, T, C_, H)
    torch.cuda.synchronize()
    q64, dy64 = ovals(qkv, "bf16", oracle), ovals(dy, "bf16", oracle)
    ry, P, rlse = oracle.attention_fwd(q64, B, T, C_, H, want_lse=True)
    rd = oracle.attention_bwd(q64, P, dy64, B, T, C_, H)
    e = _check_attention("bf16", host(y), host(lse), host(dqkv), ry, rlse, rd,
                         _attention_sum_scales(q64, dy64, P, ry, B, T, C_, H))
    print(f"[attention growing max T={T}] y rel-L2 {e[0]:.2e}, dqkv rel-L2 {e[2]:.2e}, "
          f"worst error {e[3]:.2f} of its bound")


# ----------------------------------------------------------------- layernorm
@pytest.mark.parametrize("dt", ["fp32", "bf16"])
@pytest.mark.parametrize("M,C_", [(300, 64), (130, 384), (257, 768), (64, 1024)])
def test_layernorm(ctx, oracle, dt, M, C_):
    x = rnd(M, C_) * 2 + 0.5
    w, b, dy, dx0 = rnd(C_) * 0.2 + 1, rnd(C_, scale=0.1), rnd(M, C_), rnd(M, C_)
    xd, wd, bd, dyd = (to_dev(a, dt) for a in (x, w, b, dy))
    y = torch.empty_like(xd)
    mean = torch.empty(M, device=DEV)
    rstd = torch.empty(M, device=DEV)
    ctx.layernorm_fwd(dt, xd, wd, bd, y, mean, rstd, M, C_)
    dx = to_dev(dx0, dt)
    dw = torch.empty(C_, device=DEV)
    db = torch.empty(C_, device=DEV)
    ctx.layernorm_bwd(dt, xd, wd, mean, rstd, dyd, dx, dw, db, M, C_, accumulate=True)
    torch.cuda.synchronize()
    x64, w64, b64, dy64 = (ovals(a, dt, oracle) for a in (x, w, b, dy))
    ry, rmean, rrstd = oracle.layernorm_fwd(x64, w64, b64)
    rtol, atol = TOL[dt]
    assert_close(host(y), ry, rtol, atol, "ln y")
    assert_close(host(mean), rmean, 1e-5, 1e-6, "ln mean")
    assert_close(host(rstd), rrstd, 1e-5, 1e-6, "ln rstd")
    rdx, rdw, rdb = oracle.layernorm_bwd(x64, w64, rmean, rrstd, dy64)
    assert_close(host(dx), rdx + ovals(dx0, dt, oracle), rtol, atol, "ln dx (accumulated)")
    assert_close(host(dw), rdw, 1e-4, 1e-5, "ln dw")
    assert_close(host(db), rdb, 1e-4, 1e-5, "ln db")


# ----------------------------------------------------------------- cross entropy
@pytest.mark.parametrize("dt,M,V,ld", [("fp32", 37, 65, 128), ("bf16", 37, 65, 128),
                                       ("fp32", 5, 256, 256), ("bf16", 9, 50257, 50304)])
def test_xent(ctx, oracle, dt, M, V, ld):
    z = rnd(M, ld, scale=3.0)
    tgt = synth.token_stream(1, M, V, "zipf", seed=7)[0].reshape(M)
    zd = to_dev(z, dt)
    td = torch.from_numpy(tgt).to(DEV)
    rl = torch.empty(M, device=DEV)
    ml = torch.empty(1, device=DEV)
    ctx.xent(dt, zd, td, rl, ml, M, V, ld, 1.0 / M)
    torch.cuda.synchronize()
    z64 = ovals(z, dt, oracle)[:, :V].copy()
    loss, rrl, rdz = oracle.xent(z64, tgt, want_grad=True)
    assert_close(host(rl), rrl, 2e-6, 1e-6, "row loss")
    assert abs(ml.item() - loss) <= 2e-6 * abs(loss)
    g = host(zd)
    rtol, atol = TOL[dt]
    assert_close(g[:, :V], rdz, rtol, atol, "dlogits")
    assert np.all(g[:, V:] == 0.0)


def test_xent_uniform_logits_is_log_v(ctx):
    import math
    M, V, ld = 4, 50257, 50304
    z = torch.zeros(M, ld, device=DEV, dtype=torch.bfloat16)
    td = torch.tensor([0, 1, V - 1, 77], dtype=torch.int32, device=DEV)
    rl = torch.empty(M, device=DEV)
    ml = torch.empty(1, device=DEV)
    ctx.xent("bf16", z, td, rl, ml, M, V, ld, 1.0 / M)
    torch.cuda.synchronize()
    assert abs(ml.item() - math.log(V)) < 2e-6 * math.log(V)


# ----------------------------------------------------------------- embedding
@pytest.mark.parametrize("dt,B,T,C_,V,maxT", [("fp32", 3, 50, 64, 100, 64),
                                              ("bf16", 4, 128, 768, 50257, 1024),
                                              ("bf16", 2, 33, 384, 65, 256),
                                              # several sort tiles and a ragged tail
                                              ("bf16", 5, 1000, 64, 50257, 1024),
                                              # ids of 17 bits: three radix passes
                                              ("fp32", 3, 777, 32, 70000, 1024),
                                              # the full token count of the benchmark
                                              ("bf16", 32, 1024, 64, 50257, 1024)])
def test_embedding(ctx, oracle, dt, B, T, C_, V, maxT):
    wte, wpe = rnd(V, C_, scale=0.02), rnd(maxT, C_, scale=0.02)
    tok = synth.token_stream(B, T, V, "zipf", seed=3)[0]
    dx = rnd(B * T, C_)
    base = rnd(V, C_)  # dwte is accumulated into
    wted, wped, dxd = to_dev(wte, dt), to_dev(wpe, dt), to_dev(dx, dt)
    td = torch.from_numpy(tok).to(DEV)
    x = torch.empty(B * T, C_, device=DEV, dtype=wted.dtype)
    ctx.embed_fwd(dt, wted, wped, td, x, B, T, C_, V)
    dwte = torch.from_numpy(base).to(DEV)
    dwpe = torch.full((maxT, C_), 7.0, device=DEV)
    ctx.embed_bwd(dt, dxd, td, dwte, dwpe, B, T, C_, V, maxT)
    torch.cuda.synchronize()
    rx = oracle.embed_fwd(ovals(wte, dt, oracle), ovals(wpe, dt, oracle), tok, B, T)
    rtol, atol = TOL[dt]
    assert_close(host(x), rx, rtol, atol, "embedding x")
    dx64 = ovals(dx, dt, oracle)
    rwte, rwpe = oracle.embed_bwd(dx64, tok, B, T, V, maxT)
    # fp32 sums of n terms in any order: |error| <= (n + 2) u sum|terms|,
    # u = 2^-24 (recursive summation bound); the base row counts as a term
    flat = tok.reshape(-1)
    n_v = np.bincount(flat, minlength=V).astype(np.float64)[:, None]
    abs_v = np.abs(base).astype(np.float64)
    np.add.at(abs_v, flat, np.abs(dx64))
    err = np.abs(host(dwte) - (rwte + base))
    bound = (n_v + 3) * 2.0 ** -24 * abs_v + 1e-12
    assert np.all(err <= bound), f"dwte: {(err > bound).sum()} elements above the summation bound"
    # and overall at rounding level (one row missed or doubled would be ~1/sqrt(M))
    assert np.linalg.norm(err) <= 1e-5 * np.linalg.norm(rwte + base)
    assert_close(host(dwpe), rwpe, 1e-5, 1e-6, "dwpe")
    # deterministic
    dwte2 = torch.from_numpy(base).to(DEV)
    ctx.embed_bwd(dt, dxd, td, dwte2, dwpe, B, T, C_, V, maxT)
    torch.cuda.synchronize()
    assert torch.equal(dwte, dwte2)


def test_embedding_bad_token_sets_flag(ctx):
    ctx.reset()
    wte = torch.zeros(10, 64, device=DEV)
    wpe = torch.zeros(4, 64, device=DEV)
    tok = torch.tensor([1, 2, 10, 3], dtype=torch.int32, device=DEV)
    x = torch.empty(4, 64, device=DEV)
    ctx.embed_fwd("fp32", wte, wpe, tok, x, 1, 4, 64, 10)
    with pytest.raises(api.TTError, match="TT_ERR_ARG"):
        ctx.sync()
    ctx.reset()
    ctx.sync()


# ----------------------------------------------------------------- adamw / cast
@pytest.mark.parametrize("n", [1, 7, 1001, 1 << 16])
def test_adamw_and_cast(ctx, oracle, n):
    p0, g, m0, v0 = rnd(n), rnd(n), rnd(n, scale=0.1), np.abs(rnd(n, scale=0.1))
    P, G, Mm, Vv = (torch.from_numpy(a.copy()).to(DEV) for a in (p0, g, m0, v0))
    low = torch.empty(n, device=DEV, dtype=torch.bfloat16)
    args = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    ctx.adamw(P, low, G, Mm, Vv, step=3, **args)
    torch.cuda.synchronize()
    rp, rm, rv = oracle.adamw(p0, g, m0, v0, args["lr"], args["beta1"], args["beta2"], args["eps"],
                              args["weight_decay"], 3)
    # fp32 arithmetic on fp32 inputs: a few ulps of the operands' scale.  The
    # moments are sums of two terms that can cancel, so their bound is taken
    # from the terms (b1|m| + (1-b1)|g|, b2 v + (1-b2) g^2), not from the result.
    assert_close(host(P), rp, 1e-6, 1e-6, "master")
    b1, b2 = args["beta1"], args["beta2"]
    m_scale = b1 * np.abs(m0.astype(np.float64)) + (1 - b1) * np.abs(g.astype(np.float64))
    v_scale = b2 * np.abs(v0.astype(np.float64)) + (1 - b2) * g.astype(np.float64) ** 2
    for got, ref, sc, what in [(host(Mm), rm, m_scale, "m"), (host(Vv), rv, v_scale, "v")]:
        err = np.abs(got - ref)
        assert np.all(err <= 1e-6 * np.abs(ref) + 8 * 2.0 ** -24 * sc), (what, float(np.max(err / (sc + 1e-30))))
    # the bf16 copy is the nearest bf16 of the updated fp32 master
    assert np.array_equal(host(low), oracle.bf16_values(P.cpu().numpy()))
    cast = torch.empty(n, device=DEV, dtype=torch.bfloat16)
    ctx.cast_bf16(G, cast)
    torch.cuda.synchronize()
    assert np.array_equal(host(cast), oracle.bf16_values(g))
