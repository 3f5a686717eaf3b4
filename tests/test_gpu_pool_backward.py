"""Backward pass of the pool through the C ABI against the CPU oracle's
pool_backward (itself pinned by finite differences) on seeded inputs."""

import numpy as np
import pytest
import torch

import oracle.whitematter as O
from cross_layer_kv_pool_b300 import synth, wm
from tests.gpu_util import ensure_lib, host, model, relerr, small_shape

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


KEYS = ("dstates", "dWr", "dWk", "dWv", "dsrc_norm", "dchan_norm", "dk_norm")


def _run(s, seed, N, static=None, calls=1):
    m, Wn = model(s, seed=seed, jitter=0.2, static=None if static is None else torch.tensor(static))
    dt = s.torch_dtype
    states = synth.make_normal((N, s.L, s.D), seed + 1, "cuda", 1.0, dt)
    pos_h = np.random.default_rng(seed + 2).integers(0, 4000, N)
    pos = torch.tensor(pos_h, dtype=torch.int32, device="cuda")
    dK = synth.make_normal((N, s.k, s.Hkv, s.d), seed + 3, "cuda", 1.0, dt)
    dV = synth.make_normal((N, s.k, s.Hkv, s.d), seed + 4, "cuda", 1.0, dt)
    dstates = torch.empty((N, s.L, s.D), dtype=torch.float32, device="cuda")
    g = wm.pool_grads(m, router=static is None)
    for _ in range(calls):
        wm.wm_pool_backward(m, states, pos, dK, dV, dstates, g)
    torch.cuda.synchronize()
    got = {"dstates": host(dstates), **{k: host(v) for k, v in g.items() if v is not None}}
    ref = O.pool_backward(s, Wn, host(states), pos_h, host(dK), host(dV), static)
    return got, ref


@pytest.mark.parametrize("shape_kw", [dict(L=4, k=2, p=2, Hq=4, Hkv=2),
                                      dict(L=6, k=3, p=2, p_offset=1, D=256, Hq=2, Hkv=1, d=128)])
def test_pool_backward_fp32(shape_kw):
    s = small_shape("f32", **shape_kw)
    got, ref = _run(s, 61, 37)
    for k in KEYS:
        assert relerr(got[k], ref[k]) <= 1e-4, k


def test_pool_backward_static_fp32():
    s = small_shape("f32", L=4, k=3, Hq=4, Hkv=2)
    static = np.random.default_rng(62).standard_normal((2, s.k, s.L))
    got, ref = _run(s, 63, 29, static=static)
    assert "dWr" not in got
    for k in KEYS[:1] + KEYS[2:]:
        assert relerr(got[k], ref[k]) <= 1e-4, k


def test_pool_backward_accumulates():
    """Parameter gradients add up over calls; dstates is overwritten."""
    s = small_shape("f32", L=4, k=2, Hq=4, Hkv=2)
    got, ref = _run(s, 64, 21, calls=2)
    assert relerr(got["dstates"], ref["dstates"]) <= 1e-4
    for k in KEYS[1:]:
        assert relerr(got[k], 2.0 * ref[k]) <= 1e-4, k


def test_pool_backward_bf16_storage_1p3b_widths():
    """bf16 inputs at the 1.3B widths (fp32 arithmetic inside)."""
    s = synth.HALF_1P3B.replace(L=8, k=8, V=1000)
    got, ref = _run(s, 65, 48)
    for k in KEYS:
        assert relerr(got[k], ref[k]) <= 1e-3, k
