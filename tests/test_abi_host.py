"""Host-side checks of the C ABI that need no GPU: the library loads and
exports every function include/*.h declares; the flat parameter layout agrees
with the oracle's own layout and with the input generator's table (three
independent implementations); the exact arena plan behaves; calls fail
cleanly without a device and on NULL handles."""
import ctypes as C
import os
import re

import pytest

from autograd_arena_allocated_gb300 import api, synth
from autograd_arena_allocated_gb300 import _native
from autograd_arena_allocated_gb300 import build as native_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    native_build.build()
    return _native.lib()


def _declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if not f.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(tt_[a-z0-9_]+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 25
    for n in sorted(names):
        assert hasattr(lib, n), n
    # and the binding declares exactly these
    assert names == set(_native.SIGNATURES), names ^ set(_native.SIGNATURES)


CONFIGS = [
    (2, 64, 4, 256, 32, "fp32"),
    (6, 384, 6, 65, 256, "bf16"),
    (12, 768, 12, 50257, 1024, "bf16"),
    (24, 1024, 16, 50257, 1024, "bf16"),
]


@pytest.mark.parametrize("L,C_,H,V,maxT,dt", CONFIGS)
def test_layout_matches_oracle_and_generator(lib, oracle, L, C_, H, V, maxT, dt):
    cfg = api.make_config(L, C_, H, V, maxT, dt)
    n = api.num_params(cfg)
    assert n == oracle.num_params(L, C_, H, V, maxT)
    table = synth.param_table(synth.GPT2Shape(L, C_, H, V, maxT))
    assert n == sum(t[1] for t in table)
    at = 0
    idx = [(0, 0), (0, 1)] + [(l, w) for l in range(L) for w in range(2, 14)] + [(0, 14), (0, 15)]
    for (layer, which), (name, numel, _) in zip(idx, table):
        assert api.param_offset(cfg, layer, which) == (at, numel), name
        assert oracle.param_offset(L, C_, H, V, maxT, layer, which) == (at, numel), name
        at += numel
    assert at == n


def test_bad_configs_rejected(lib):
    for bad in [(2, 64, 3, 256, 32, "fp32"),    # C % H
                (2, 96, 4, 256, 32, "fp32"),    # C % 64
                (2, 64, 4, 256, 32, "bf16"),    # bf16 needs head dim 64
                (2, 64, 4, 256, 0, "fp32")]:    # maxT
        cfg = api.make_config(*bad)
        assert api.num_params(cfg) == 0
        assert api.arena_bytes(cfg, 1, 1) == 0
    cfg = api.make_config(2, 64, 4, 256, 32, "fp32")
    assert api.arena_bytes(cfg, 1, 33) == 0   # T > maxT
    assert api.arena_bytes(cfg, 0, 8) == 0
    off, n = C.c_size_t(), C.c_size_t()
    assert lib.tt_gpt2_param_offset(C.byref(cfg), 2, 5, C.byref(off), C.byref(n)) == -2  # layer >= L
    assert lib.tt_gpt2_param_offset(C.byref(cfg), 0, 16, C.byref(off), C.byref(n)) == -2


def test_arena_plan_grows_with_batch(lib):
    cfg = api.make_config(12, 768, 12, 50257, 1024, "bf16")
    a1 = api.arena_bytes(cfg, 1, 1024)
    a8 = api.arena_bytes(cfg, 8, 1024)
    a32 = api.arena_bytes(cfg, 32, 1024)
    assert 0 < a1 < a8 < a32
    # the logits alone are B*T*Vp bf16 values
    assert a32 > 32 * 1024 * 50304 * 2
    # the whole B=32 step fits comfortably in one GB300's HBM
    assert a32 < 64 * 2 ** 30
    cfg32 = api.make_config(2, 64, 4, 256, 32, "fp32")
    assert api.arena_bytes(cfg32, 4, 32) > 4 * 32 * 256 * 4


def test_null_and_missing_device(lib):
    assert lib.tt_ctx_reset(None) == -2
    assert lib.tt_ctx_sync(None) == -2
    assert lib.tt_gpt2_step(None, None, None, None, None, 1, 1, None) == -2
    assert lib.tt_last_error(None) == b"NULL context"
    lib.tt_ctx_destroy(None)  # NULL-safe
    assert lib.tt_ctx_arena_used(None) == 0
    h = C.c_void_p()
    assert lib.tt_ctx_create(0, C.byref(h)) == -2
    assert lib.tt_ctx_create(1 << 20, None) == -2
    import torch
    if not torch.cuda.is_available():
        assert lib.tt_ctx_create(1 << 20, C.byref(h)) == -4  # TT_ERR_CUDA, no device
        assert not h.value


def test_no_cpu_fallback_when_library_missing(monkeypatch, tmp_path):
    """The binding raises instead of computing anything on the CPU."""
    monkeypatch.setattr(_native, "_lib", None)
    monkeypatch.setattr(_native, "LIB_PATH", str(tmp_path / "libtt.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _native.lib()


def test_fp16_configs(lib):
    """IEEE half storage: any head dim the SIMT kernels take, the same
    parameter layout, 16-bit activations (a smaller arena than fp32), and no
    generation plan."""
    tiny16 = api.make_config(2, 64, 4, 256, 32, "fp16")  # head dim 16
    tiny32 = api.make_config(2, 64, 4, 256, 32, "fp32")
    assert api.num_params(tiny16) == api.num_params(tiny32) > 0
    assert 0 < api.arena_bytes(tiny16, 4, 32) < api.arena_bytes(tiny32, 4, 32)
    m16 = api.make_config(12, 768, 12, 50257, 1024, "fp16")
    mbf = api.make_config(12, 768, 12, 50257, 1024, "bf16")
    for layer, which in [(0, 0), (0, 1), (5, 8), (11, 13), (0, 15)]:
        assert api.param_offset(m16, layer, which) == api.param_offset(mbf, layer, which)
    assert api.generate_arena_bytes(m16, 8, 64, 16) == 0
    assert api.generate_arena_bytes(mbf, 8, 64, 16) > 0


def test_binding_checks_the_16bit_copy_type():
    """tt_adamw writes half for a TT_FP16 model and bf16 otherwise; the
    binding refuses a torch tensor of the other type before any call."""
    import torch

    c = object.__new__(api.Context)  # no device context needed for the check
    c.cfg = None
    c._check_lowp(None)
    c._check_lowp(torch.empty(2, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        c._check_lowp(torch.empty(2, dtype=torch.float16))
    c.cfg = api.make_config(2, 64, 4, 256, 32, "fp16")
    c._check_lowp(torch.empty(2, dtype=torch.float16))
    with pytest.raises(ValueError):
        c._check_lowp(torch.empty(2, dtype=torch.bfloat16))
