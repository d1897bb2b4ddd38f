"""GPT-2 training step on one GB300 (sm_103a): forward, reverse-mode tape
backward and AdamW over tensors bump-allocated from one device arena.

The compute path is the native library libtt.so (C ABI: include/tt.h,
include/tt_ops.h).  Importing this package does not load it; the first call
into `api` does, and raises if it has not been built (no CPU fallback).
"""
__all__ = ["api", "synth", "build"]
