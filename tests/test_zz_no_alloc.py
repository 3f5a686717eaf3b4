"""wm_pool_mix_static: the pool for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: a plug-in host that owns
all device memory and passes only input and output pointers, or a loop that
must not call cudaMalloc because it synchronises the device. The static entry
point keeps its scratch in a fixed device array inside the library instead.
This test checks, through the C ABI, that two consecutive calls of it give
what wm_pool_mix (with a caller workspace) gives on the same inputs. The
file is named to be collected last, so a run that stops at the first failure
has run every other test before this one."""

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


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_pool_mix_static_matches_workspace_entry(dtype):
    ensure_lib()
    s = synth.HALF_SMALL.replace(V=1000, dtype=dtype)
    m, _ = model(s, seed=11, jitter=0.2)
    B, Tmax, N = 4, 300, 96
    tol = TOL[dtype]
    for call, seed in enumerate((1, 2)):       # two calls in a row
        states, seq, pos = _inputs(s, N, B, Tmax, seed)
        ref_k, ref_v = m.new_cache(B, Tmax, fill=float("nan"))
        ref_c = torch.empty((N, 2, s.k, s.L), dtype=torch.float32, device="cuda")
        ref_m = torch.empty((2, s.k, N, s.D), dtype=s.torch_dtype, device="cuda")
        ws = m.workspace(N, Tmax)
        wm.wm_pool_mix(m, states, seq, pos, ref_k, ref_v, ws, coeff_out=ref_c, mixed_out=ref_m)
        ck, cv = m.new_cache(B, Tmax, fill=float("nan"))
        co = torch.empty_like(ref_c)
        mx = torch.empty_like(ref_m)
        wm.wm_pool_mix_static(m, states, seq, pos, ck, cv, coeff_out=co, mixed_out=mx)
        torch.cuda.synchronize()
        assert wm.wm_check_flags(ws) == 0
        assert relerr(host(co), host(ref_c)) <= tol["coeff"], call
        assert relerr(host(mx), host(ref_m)) <= tol["mixed"], call
        K, Kr = host(ck), host(ref_k)
        assert np.array_equal(np.isnan(K), np.isnan(Kr)), call
        w = ~np.isnan(Kr)
        assert relerr(K[w], Kr[w]) <= tol["cache"], call
        Vv, Vr = host(cv), host(ref_v)
        assert np.array_equal(np.isnan(Vv), np.isnan(Vr)), call
        assert relerr(Vv[~np.isnan(Vr)], Vr[~np.isnan(Vr)]) <= tol["cache"], call


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
