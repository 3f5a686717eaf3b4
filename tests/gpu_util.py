"""Helpers shared by the GPU parity tests (inputs, tolerances, comparisons)."""

from __future__ import annotations

import dataclasses
from types import SimpleNamespace

import numpy as np
import torch

from cross_layer_kv_pool_b300 import build, synth, wm

# Tolerances, max|gpu - ref| / max|ref| per tensor: 1e-4 in fp32 mode; in bf16
# mode 2e-2 on logits and caches after whole passes, 1e-2 on the mixed
# channels and on a single attention call given identical inputs.
TOL = {"f32": dict(logits=1e-4, cache=1e-4, mixed=1e-4, coeff=1e-4, attn=1e-4),
       "bf16": dict(logits=2e-2, cache=2e-2, mixed=1e-2, coeff=2e-2, attn=1e-2)}


def ensure_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    return wm.lib()


def relerr(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.max(np.abs(b))
    return float(np.max(np.abs(a - b)) / den) if den > 0 else float(np.max(np.abs(a)))


def host(t) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def model(shape, seed=0, jitter=0.1, static=None, flags=0):
    W = synth.make_weights(shape, seed=seed, device="cuda", gain_jitter=jitter)
    return wm.Model(shape, W, static_coeff=static, flags=flags), synth.to_numpy_weights(W)


def ocfg(shape):
    """The oracle's view of a model: bf16 workloads use its bf16-storage mode
    (activations rounded where a bf16 pipeline stores them), fp32 workloads
    the plain fp64 arithmetic."""
    ns = SimpleNamespace(**dataclasses.asdict(shape))
    ns.nR = shape.nR
    if shape.dtype == "bf16":
        ns.storage = "bf16"
    return ns


def small_shape(dtype="f32", **kw):
    base = dict(L=4, D=128, k=2, p=2, Hq=4, Hkv=2, d=64, F=256, V=512, dtype=dtype)
    base.update(kw)
    return synth.ModelShape(**base)
