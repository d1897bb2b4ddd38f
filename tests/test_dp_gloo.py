"""Data-parallel gradient exchange (autograd_arena_allocated_gb300.dp) on two
gloo ranks over CPU tensors.  Each rank takes half of the batch and its
gradient from the oracle; after the exchange, the all-reduce form must give
every rank the oracle's full-batch gradient, and the sharded form
(reduce-scatter, AdamW on a slice, all-gather) the oracle's full-batch AdamW
update.  The update here is the oracle's AdamW applied to the slices, standing
in for the native kernel (no GPU in these tests)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from autograd_arena_allocated_gb300 import api, dp, synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _tensor_starts(sh):
    """Start offsets of the flat vector's parameter tensors, from the oracle's
    layout (the fixed order)."""
    import oracle

    off = lambda layer, which: oracle.param_offset(sh.L, sh.C, sh.H, sh.V, sh.maxT, layer, which)[0]
    starts = [off(0, 0), off(0, 1)]
    for l in range(sh.L):
        starts += [off(l, 2 + j) for j in range(12)]
    return starts + [off(0, 14), off(0, 15)]


def _oracle_update(master, lowp, grads, m, v, h, step):
    import oracle

    p2, m2, v2 = oracle.adamw(master.numpy().astype(np.float64), grads.numpy().astype(np.float64),
                              m.numpy().astype(np.float64), v.numpy().astype(np.float64),
                              h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, step)
    master.copy_(torch.from_numpy(p2))
    m.copy_(torch.from_numpy(m2))
    v.copy_(torch.from_numpy(v2))
    lowp.copy_(master)  # the "16-bit copy" of this CPU test is fp32


def _rank_main(rank, world, port, out):
    import oracle

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.WORKLOADS["tiny_fp32"]
        sh = w.shape
        p = synth.init_params(sh, jitter=0.05)
        tok, tgt = synth.token_stream(w.B, w.T, sh.V, w.tokens)
        per = w.B // world
        mine = slice(rank * per, (rank + 1) * per)
        _, g, _ = oracle.gpt2_step(sh, p.astype(np.float64), tok[mine], tgt[mine])
        n = p.size
        ex = dp.DataParallel(dist, n, boundaries=_tensor_starts(sh), bucket_elems=20000)
        h = dp.Hyper(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)

        def padded(a):
            t = torch.zeros(ex.n_pad, dtype=torch.float32)
            t[:n] = torch.from_numpy(np.asarray(a, dtype=np.float32))
            return t

        # all-reduce form
        grads = padded(g)
        master, lowp = padded(p), padded(p)
        m, v = torch.zeros(ex.n_pad), torch.zeros(ex.n_pad)
        ex.step_allreduce(_oracle_update, master, lowp, grads, m, v, h, 1)
        res = dict(n_pad=ex.n_pad, lo=ex.lo, hi=ex.hi, buckets=ex.buckets,
                   mean_grad=grads[:n].numpy().copy(), ar_master=master[:n].numpy().copy(),
                   ar_pad=float(grads[n:].abs().sum()))
        # sharded form
        grads = padded(g)
        lowp = padded(p)
        master_s = padded(p)[ex.lo:ex.hi].clone()
        gs = torch.empty(ex.hi - ex.lo)
        ms, vs = torch.zeros(ex.hi - ex.lo), torch.zeros(ex.hi - ex.lo)
        ex.step_sharded(_oracle_update, master_s, lowp, grads, gs, ms, vs, h, 1)
        res.update(sh_lowp=lowp[:n].numpy().copy(), sh_master=master_s.numpy().copy())
        out[rank] = res
    finally:
        dist.destroy_process_group()


def test_two_rank_exchange_matches_full_batch(oracle):
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    w = synth.WORKLOADS["tiny_fp32"]
    sh = w.shape
    p = synth.init_params(sh, jitter=0.05).astype(np.float64)
    tok, tgt = synth.token_stream(w.B, w.T, sh.V, w.tokens)
    _, g_full, _ = oracle.gpt2_step(sh, p, tok, tgt)
    p_full, _, _ = oracle.adamw(p, g_full, np.zeros_like(p), np.zeros_like(p), w.lr, w.beta1, w.beta2,
                                w.eps, w.weight_decay, 1)
    rel = lambda a, b: float(np.linalg.norm(a - b) / np.linalg.norm(b))
    n = p.size
    for r in range(world):
        # the mean of the two half-batch gradients is the full batch's (fp32 rounding)
        assert rel(res[r]["mean_grad"], g_full) < 1e-6
        assert res[r]["ar_pad"] == 0.0
        assert rel(res[r]["ar_master"], p_full) < 1e-6
        # sharded: every rank holds the full updated copy, and its own master slice
        assert rel(res[r]["sh_lowp"], p_full) < 1e-6
        lo, hi = res[r]["lo"], res[r]["hi"]
        assert rel(res[r]["sh_master"][:max(0, min(hi, n) - lo)], p_full[lo:min(hi, n)]) < 1e-6
    # both ranks ran the same update: bit-identical results
    assert np.array_equal(res[0]["ar_master"], res[1]["ar_master"])
    assert np.array_equal(res[0]["sh_lowp"], res[1]["sh_lowp"])
    assert res[0]["hi"] == res[1]["lo"] and res[1]["hi"] == res[0]["n_pad"]
    # buckets tile the padded vector from its end to its start
    b = res[0]["buckets"]
    assert b[0][1] == res[0]["n_pad"] and b[-1][0] == 0
    assert all(b[i][0] == b[i + 1][1] for i in range(len(b) - 1))


def test_padding_slices_and_buckets():
    assert dp.padded_length(100, 2) == 112 and dp.padded_length(112, 2) == 112
    assert dp.padded_length(124_439_808, 8) % 64 == 0
    n_pad = dp.padded_length(1001, 3)
    ranges = [dp.shard_range(n_pad, 3, r) for r in range(3)]
    assert ranges[0][0] == 0 and ranges[-1][1] == n_pad
    assert all(hi - lo == n_pad // 3 and lo % dp.ALIGN == 0 for lo, hi in ranges)
    with pytest.raises(ValueError):
        dp.shard_range(1001, 3, 0)
    # tensors of 10, 30, 5, 50 elements (starts 0, 10, 40, 45; padded end 96)
    assert dp.tensor_buckets([0, 10, 40, 45], 96, 55) == [(45, 96), (0, 45)]
    assert dp.tensor_buckets([0, 10, 40, 45], 96, 20) == [(45, 96), (40, 45), (10, 40), (0, 10)]
    assert dp.tensor_buckets([0], 96, 10) == [(0, 96)]
    with pytest.raises(ValueError):
        dp.tensor_buckets([5, 10], 96, 10)


def test_tensor_starts_match_oracle_layout():
    """The buckets' tensor boundaries, read from the library's C ABI, are the
    oracle's flat layout."""
    sh = synth.WORKLOADS["char_bf16"].shape
    cfg = api.make_config(sh.L, sh.C, sh.H, sh.V, sh.maxT, "bf16")
    assert dp.tensor_starts(cfg) == _tensor_starts(sh)
