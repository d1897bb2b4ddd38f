"""Seeded synthetic inputs for the GPT-2 training step.

This module generates inputs only: token streams and initial weights.  It
holds none of the step's arithmetic and is shared by the CUDA path, the
oracle tests and the benchmark, so that both sides see bit-identical inputs.

Random numbers come from one counter-based generator, written out here from
its published definition (SplitMix64, Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014):

    x_i = mix(seed + (i + 1) * 0x9E3779B97F4A7C15)
    mix(z): z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
            z = (z ^ (z >> 27)) * 0x94D049BB133111EB
            z =  z ^ (z >> 31)
    u_i = (x_i >> 11) * 2**-53                      in [0, 1)

Normals use the Box-Muller transform on consecutive pairs:
    n_j = sqrt(-2 ln(1 - u_{2j})) * cos(2 pi u_{2j+1}).

Token streams: a B x (T+1) stream s is drawn, tokens = s[:, :T] and
targets = s[:, 1:] (next-token prediction).  Ids are either uniform over the
vocabulary or Zipf(s=1.1) with P(id = k) proportional to (k+1)^-1.1, sampled
by inverse CDF (binary search of a float64 CDF with u_i).

Weights: every matrix and both embedding tables ~ N(0, 0.02); the two
residual projections (attention proj_w and MLP fcproj_w) ~ N(0, 0.02/sqrt(2L));
biases 0; LayerNorm gamma 1, beta 0 (the init the tinytorch page's
RandomNorm() stands for, with GPT-2's residual scaling).  Normal j of the
parameter stream belongs to flat parameter index j.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

PARAM_SEED = 1337
TOKEN_SEED = 42


@dataclass(frozen=True)
class GPT2Shape:
    """Architecture of a GPT-2-style model (vocabulary V is unpadded)."""
    L: int
    C: int
    H: int
    V: int
    maxT: int


@dataclass(frozen=True)
class Workload:
    """One training-step workload: model shape, batch and input recipe."""
    name: str
    shape: GPT2Shape
    B: int
    T: int
    dtype: str          # "fp32" or "bf16"
    tokens: str         # "uniform" or "zipf"
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1


GPT2_124M = GPT2Shape(L=12, C=768, H=12, V=50257, maxT=1024)
GPT2_350M = GPT2Shape(L=24, C=1024, H=16, V=50257, maxT=1024)

WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", GPT2Shape(2, 64, 4, 256, 32), 4, 32, "fp32", "uniform"),
    "char_bf16": Workload("char_bf16", GPT2Shape(6, 384, 6, 65, 256), 64, 256, "bf16", "zipf"),
    "gpt2_124m_b8": Workload("gpt2_124m_b8", GPT2_124M, 8, 1024, "bf16", "zipf"),
    "gpt2_124m_b32": Workload("gpt2_124m_b32", GPT2_124M, 32, 1024, "bf16", "zipf"),
    "gpt2_350m_b8": Workload("gpt2_350m_b8", GPT2_350M, 8, 1024, "bf16", "zipf"),
}


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def uniforms(seed: int, start: int, count: int) -> np.ndarray:
    """u_i for i in [start, start+count) of the stream `seed` (float64)."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + idx * GOLDEN_GAMMA
        x = _mix(z)
    return (x >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normals(seed: int, start: int, count: int) -> np.ndarray:
    """n_j for j in [start, start+count) (float64), Box-Muller on pairs."""
    u = uniforms(seed, 2 * start, 2 * count)
    u1, u2 = u[0::2], u[1::2]
    return np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * math.pi * u2)


def zipf_cdf(V: int, s: float = 1.1) -> np.ndarray:
    w = (np.arange(1, V + 1, dtype=np.float64)) ** (-s)
    c = np.cumsum(w)
    return c / c[-1]


def token_stream(B: int, T: int, V: int, kind: str, seed: int = TOKEN_SEED):
    """Returns (tokens, targets), each int32 [B, T]."""
    u = uniforms(seed, 0, B * (T + 1))
    if kind == "uniform":
        ids = np.minimum((u * V).astype(np.int64), V - 1)
    elif kind == "zipf":
        ids = np.searchsorted(zipf_cdf(V), u, side="right")
        ids = np.minimum(ids, V - 1)
    else:
        raise ValueError(f"unknown token distribution {kind!r}")
    s = ids.reshape(B, T + 1).astype(np.int32)
    return np.ascontiguousarray(s[:, :T]), np.ascontiguousarray(s[:, 1:])


def param_table(sh: GPT2Shape):
    """(name, numel, init) for every tensor of the flat parameter vector, in
    the fixed order of the C-ABI: wte, wpe, per layer {ln1_w, ln1_b, qkv_w,
    qkv_b, proj_w, proj_b, ln2_w, ln2_b, fc_w, fc_b, fcproj_w, fcproj_b},
    lnf_w, lnf_b.  init is "normal", "resid" (scaled normal), "zeros" or "ones"."""
    C = sh.C
    t = [("wte", sh.V * C, "normal"), ("wpe", sh.maxT * C, "normal")]
    for l in range(sh.L):
        t += [
            (f"h{l}.ln1_w", C, "ones"), (f"h{l}.ln1_b", C, "zeros"),
            (f"h{l}.qkv_w", 3 * C * C, "normal"), (f"h{l}.qkv_b", 3 * C, "zeros"),
            (f"h{l}.proj_w", C * C, "resid"), (f"h{l}.proj_b", C, "zeros"),
            (f"h{l}.ln2_w", C, "ones"), (f"h{l}.ln2_b", C, "zeros"),
            (f"h{l}.fc_w", 4 * C * C, "normal"), (f"h{l}.fc_b", 4 * C, "zeros"),
            (f"h{l}.fcproj_w", 4 * C * C, "resid"), (f"h{l}.fcproj_b", C, "zeros"),
        ]
    t += [("lnf_w", C, "ones"), ("lnf_b", C, "zeros")]
    return t


def init_params(sh: GPT2Shape, seed: int = PARAM_SEED, std: float = 0.02,
                jitter: float = 0.0, chunk: int = 1 << 24) -> np.ndarray:
    """Flat float32 parameter vector with the init described above.

    jitter > 0 gives test inputs in which no tensor is constant: biases and
    LayerNorm beta ~ N(0, jitter), LayerNorm gamma ~ 1 + N(0, jitter)."""
    table = param_table(sh)
    total = sum(n for _, n, _ in table)
    out = np.empty(total, dtype=np.float32)
    resid_std = std / math.sqrt(2 * sh.L) if sh.L > 0 else std
    at = 0
    for _, n, kind in table:
        if kind in ("ones", "zeros") and jitter > 0:
            noise = normals(seed, at, n) * jitter
            out[at:at + n] = ((1.0 if kind == "ones" else 0.0) + noise).astype(np.float32)
        elif kind == "ones":
            out[at:at + n] = 1.0
        elif kind == "zeros":
            out[at:at + n] = 0.0
        else:
            sd = std if kind == "normal" else resid_std
            for c0 in range(0, n, chunk):
                c1 = min(n, c0 + chunk)
                out[at + c0:at + c1] = (normals(seed, at + c0, c1 - c0) * sd).astype(np.float32)
        at += n
    return out



# ---------------------------------------------------------------- the small classifier
# The tinytorch page's example (八.1 and 八.5): three features (colour, size,
# weight) in [0, 1], a hidden layer of 32, three classes.  Sample r draws its
# label y_r = floor(3 u_{4r}) and its features around the class centre,
# x_r = centre[y_r] + 0.3 (u_{4r+1..4r+3} - 0.5).  Parameters are N(0, std)
# in the flat order W1 [3, 32], b1 [32], W2 [32, 3], b2 [3] (RandomNorm).
FRUIT_SEED = 2024
FRUIT_SHAPE = (3, 32, 3)
FRUIT_CENTRES = np.array([[0.8, 0.5, 0.4], [0.5, 0.3, 0.8], [0.3, 0.7, 0.3]])


def fruit_batch(R: int, seed: int = FRUIT_SEED):
    """x float32 [R, 3] and labels int32 [R]."""
    u = uniforms(seed, 0, 4 * R).reshape(R, 4)
    y = np.minimum((u[:, 0] * 3).astype(np.int32), 2)
    x = FRUIT_CENTRES[y] + 0.3 * (u[:, 1:] - 0.5)
    return x.astype(np.float32), y


def mlp_init(nin: int, nh: int, nout: int, seed: int = PARAM_SEED, std: float = 1.0):
    """(W1 [nin, nh], b1 [nh], W2 [nh, nout], b2 [nout]) as float32."""
    sizes = [nin * nh, nh, nh * nout, nout]
    flat = (std * normals(seed, 0, sum(sizes))).astype(np.float32)
    out, o = [], 0
    for n, shp in zip(sizes, [(nin, nh), (nh,), (nh, nout), (nout,)]):
        out.append(flat[o:o + n].reshape(shp))
        o += n
    return tuple(out)
