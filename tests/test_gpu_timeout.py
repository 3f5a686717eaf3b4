"""The timeout path of the bounded device-side waits, without a GPU fault.

WM_FLAG_WAIT_PROBE makes every CTA of the tensor-core GEMM engine wait, before
its first product, on a barrier that nothing completes, for at most 2 ms. The
wait runs out: the kernel raises the timeout bit, drains its copies and
returns. Every later kernel of the call that holds bounded waits (GEMM,
attention, mixer) reads the bit at entry and returns without work, so the
whole call ends in a few milliseconds however many launches it has. The host
learns of it through wm_check_flags (WM_ERR_TIMEOUT), and the next call on the
same workspace computes normally.
"""

import time

import numpy as np
import pytest
import torch

from cross_layer_kv_pool_b300 import synth, wm
from tests.gpu_util import ensure_lib, host, model, relerr, small_shape

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _expect_timeout(ws):
    with pytest.raises(wm.WMError) as e:
        wm.wm_check_flags(ws)
    assert e.value.status == wm.WM_ERR_TIMEOUT


def test_prefill_timeout_surfaces_in_bounded_time():
    s = small_shape("bf16", D=256, Hq=4, Hkv=2, d=64, F=512, L=4, k=2)
    m, _ = model(s, seed=31)
    probe = wm.Model(s, m.W, flags=wm.WM_FLAG_WAIT_PROBE)
    B, T, g = 4, 64, 16          # 16 groups: ~400 GEMM launches in the call
    tok = synth.make_tokens(s, B, T, seed=5, device="cuda")
    ws = m.workspace(wm.rows_for_pass(B, T, g), T)
    lg_ref = torch.zeros((B, s.V), dtype=torch.float32, device="cuda")
    ck_ref, cv_ref = m.new_cache(B, T)
    wm.wm_cyclic_pass(m, tok, g, ck_ref, cv_ref, ws, logits=lg_ref, logits_mode="last")
    torch.cuda.synchronize()
    assert wm.wm_check_flags(ws) == 0

    # the probe: every GEMM launch would wait 2 ms if the timeout bit did not
    # stop the later kernels of the call at entry (>= 0.8 s in all)
    ck, cv = m.new_cache(B, T)
    lg = torch.zeros_like(lg_ref)
    t0 = time.perf_counter()
    wm.wm_cyclic_pass(probe, tok, g, ck, cv, ws, logits=lg, logits_mode="last")
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    _expect_timeout(ws)
    assert elapsed < 0.4, elapsed

    # the flag word was cleared by the check; the next call computes normally
    ck2, cv2 = m.new_cache(B, T)
    lg2 = torch.zeros_like(lg_ref)
    wm.wm_cyclic_pass(m, tok, g, ck2, cv2, ws, logits=lg2, logits_mode="last")
    torch.cuda.synchronize()
    assert wm.wm_check_flags(ws) == 0
    assert relerr(host(lg2), host(lg_ref)) <= 2e-2
    assert relerr(host(ck2), host(ck_ref)) <= 2e-2
    assert np.isfinite(host(lg2)).all()


def test_decode_timeout_cluster_products():
    """Decode-sized products split K over a thread-block cluster; every CTA of
    a cluster times out alike and still meets its peers at the cluster
    barriers before leaving."""
    s = synth.HALF_1P3B.replace(L=2, k=2, V=1000)
    m, _ = model(s, seed=7)
    probe = wm.Model(s, m.W, flags=wm.WM_FLAG_WAIT_PROBE)
    B, Tmax = 8, 64
    ck, cv = m.new_cache(B, Tmax)
    ws = m.workspace(B, Tmax)
    tok = torch.randint(0, s.V, (B,), dtype=torch.int32, device="cuda")
    lg = torch.zeros((B, s.V), dtype=torch.float32, device="cuda")
    wm.wm_decode_step(probe, tok, 3, ck, cv, lg, ws)
    torch.cuda.synchronize()
    _expect_timeout(ws)
    wm.wm_decode_step(m, tok, 3, ck, cv, lg, ws)
    torch.cuda.synchronize()
    assert wm.wm_check_flags(ws) == 0
    assert np.isfinite(host(lg)).all()
