"""wm_pool_mix_static: the pool for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: a plug-in host that owns
all device memory and passes only input and output pointers, or a loop that
must not call cudaMalloc because it synchronises the device. The static entry
point keeps its scratch in a fixed device array inside the library instead.
These tests check, through the C ABI, that consecutive calls of it give what
wm_pool_mix (with a caller workspace) gives on the same inputs: with and
without the optional coefficient and channel outputs (the latter leaves them
in the internal array), with static mixing weights, and after a larger call
has left its data in the shared array. A warm call changes neither the
device's free memory nor PyTorch's allocations. The file is named to be
collected last, so a run that stops at the first failure has run every other
test before this one."""

import numpy as np
import pytest
import torch

from cross_layer_kv_pool_b300 import synth, wm
from tests.gpu_util import TOL, ensure_lib, host, model, relerr

pytestmark = pytest.mark.gpu


def _inputs(s, N, B, Tmax, seed):
    rng = np.random.default_rng(seed)
    flat = rng.choice(B * Tmax, size=N, replace=False)
    states = synth.make_normal((N, s.L, s.D), 100 + seed, "cuda", 1.0, s.torch_dtype)
    seq = torch.tensor(flat // Tmax, dtype=torch.int32, device="cuda")
    pos = torch.tensor(flat % Tmax, dtype=torch.int32, device="cuda")
    return states, seq, pos


def _caches_match(ck, cv, ref_k, ref_v, tol, call):
    for got, ref in ((host(ck), host(ref_k)), (host(cv), host(ref_v))):
        assert np.array_equal(np.isnan(got), np.isnan(ref)), call
        w = ~np.isnan(ref)
        assert relerr(got[w], ref[w]) <= tol["cache"], call


def _one_call(m, N, B, Tmax, seed, outputs, tol, call):
    """wm_pool_mix with a workspace, then wm_pool_mix_static, same inputs."""
    s = m.shape
    states, seq, pos = _inputs(s, N, B, Tmax, seed)
    ref_k, ref_v = m.new_cache(B, Tmax, fill=float("nan"))
    ref_c = torch.empty((N, 2, s.k, s.L), dtype=torch.float32, device="cuda")
    ref_m = torch.empty((2, s.k, N, s.D), dtype=s.torch_dtype, device="cuda")
    ws = m.workspace(N, Tmax)
    wm.wm_pool_mix(m, states, seq, pos, ref_k, ref_v, ws, coeff_out=ref_c, mixed_out=ref_m)
    ck, cv = m.new_cache(B, Tmax, fill=float("nan"))
    co = torch.empty_like(ref_c) if outputs else None
    mx = torch.empty_like(ref_m) if outputs else None
    wm.wm_pool_mix_static(m, states, seq, pos, ck, cv, coeff_out=co, mixed_out=mx)
    torch.cuda.synchronize()
    assert wm.wm_check_flags(ws) == 0
    assert wm.wm_check_static_flags() == 0
    if outputs:
        assert relerr(host(co), host(ref_c)) <= tol["coeff"], call
        assert relerr(host(mx), host(ref_m)) <= tol["mixed"], call
    _caches_match(ck, cv, ref_k, ref_v, tol, call)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_pool_mix_static_matches_workspace_entry(dtype):
    ensure_lib()
    s = synth.HALF_SMALL.replace(V=1000, dtype=dtype)
    m, _ = model(s, seed=11, jitter=0.2)
    B, Tmax = 4, 300
    tol = TOL[dtype]
    # two calls in a row, the second smaller, then two that keep the
    # coefficients and channels in the internal array
    for call, (N, seed, outputs) in enumerate(((200, 1, True), (96, 2, True),
                                               (150, 3, False), (64, 4, False))):
        _one_call(m, N, B, Tmax, seed, outputs, tol, call)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_pool_mix_static_with_static_coefficients(dtype):
    """Router-free mixing (constant weights, different per branch)."""
    ensure_lib()
    s = synth.HALF_SMALL.replace(V=1000, k=4, dtype=dtype)
    st = np.random.default_rng(8).standard_normal((2, s.k, s.L))
    st[1] *= -0.7
    m, _ = model(s, seed=12, jitter=0.2, static=torch.tensor(st))
    tol = TOL[dtype]
    for call, (N, seed, outputs) in enumerate(((120, 5, True), (80, 6, False))):
        _one_call(m, N, 3, 200, seed, outputs, tol, call)


def test_pool_mix_static_allocates_nothing():
    """A warm call leaves the device's free memory and PyTorch's allocations
    unchanged (the first call on a device may load the library's kernels)."""
    ensure_lib()
    s = synth.HALF_SMALL.replace(V=1000)
    m, _ = model(s, seed=13)
    B, Tmax, N = 2, 256, 128
    states, seq, pos = _inputs(s, N, B, Tmax, 9)
    ck, cv = m.new_cache(B, Tmax)
    co = torch.empty((N, 2, s.k, s.L), dtype=torch.float32, device="cuda")
    mx = torch.empty((2, s.k, N, s.D), dtype=s.torch_dtype, device="cuda")
    wm.wm_pool_mix_static(m, states, seq, pos, ck, cv, coeff_out=co, mixed_out=mx)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(3):
        wm.wm_pool_mix_static(m, states, seq, pos, ck, cv, coeff_out=co, mixed_out=mx)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_allocated() == alloc0
    assert wm.wm_check_static_flags() == 0


def test_pool_mix_static_rejects_rows_beyond_its_scratch():
    ensure_lib()
    s = synth.HALF_1P3B.replace(L=4, k=2, V=1000)
    m, _ = model(s, seed=3)
    N, B, Tmax = 4096, 2, 2048       # about 120 MiB of pool scratch: too large
    states = torch.zeros((N, s.L, s.D), dtype=s.torch_dtype, device="cuda")
    idx = torch.arange(N, dtype=torch.int32, device="cuda")
    ck, cv = m.new_cache(B, Tmax)
    with pytest.raises(wm.WMError) as e:
        wm.wm_pool_mix_static(m, states, idx % B, idx // B, ck, cv)
    assert e.value.status == wm.WM_ERR_WORKSPACE
