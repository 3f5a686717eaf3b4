"""The feedback-free variant (k = L, one exact pass) through the C ABI
against the CPU oracle on seeded inputs."""

import numpy as np
import pytest
import torch

import oracle.whitematter as O
from cross_layer_kv_pool_b300 import wm
from tests.gpu_util import (SPREAD_EPS, TOL, ensure_lib, host, model, ocfg, perturbed, relerr,
                            small_shape, within)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _gpu(m, tokens_h, logits_mode="all", Tmax=None, ws_rows=None, steps=False):
    """One feedback-free pass (or, with ``steps``, T single-token calls)."""
    s = m.shape
    B, T = tokens_h.shape
    Tmax = Tmax or T
    tok = torch.tensor(tokens_h, dtype=torch.int32, device="cuda")
    ck, cv = m.new_cache(B, Tmax)
    ws = m.workspace(ws_rows or B * T, Tmax)
    if steps:
        lg = torch.zeros((B, T, s.V), dtype=torch.float32, device="cuda")
        step = torch.zeros((B, s.V), dtype=torch.float32, device="cuda")
        for t in range(T):
            wm.wm_feedforward_pass(m, tok[:, t:t + 1].contiguous(), ck, cv, ws, pos0=t, logits=step,
                                   logits_mode="last")
            lg[:, t] = step
    else:
        shp = (B, T, s.V) if logits_mode == "all" else (B, s.V)
        lg = torch.zeros(shp, dtype=torch.float32, device="cuda")
        wm.wm_feedforward_pass(m, tok, ck, cv, ws, logits=lg, logits_mode=logits_mode)
    torch.cuda.synchronize()
    assert wm.wm_check_flags(ws) == 0
    return host(lg), host(ck), host(cv)


def _oracle(s, Wn, tokens_h, logits="all", Tmax=None, static=None):
    B, T = tokens_h.shape
    oc = ocfg(s)
    ck, cv = O.new_cache(oc, B, Tmax or T)
    lg = O.feedback_free_pass(oc, Wn, tokens_h, ck, cv, logits=logits, static_coeff=static)
    return lg, ck, cv


@pytest.mark.parametrize("mode", ["all", "last"])
@pytest.mark.parametrize("p_offset", [0, 1])
def test_feedback_free_fp32_end_to_end(mode, p_offset):
    s = small_shape("f32", L=4, k=4, p_offset=p_offset, Hq=4, Hkv=2)
    m, Wn = model(s, seed=21, jitter=0.2)
    tokens = np.random.default_rng(22).integers(0, s.V, size=(2, 24))
    lg, ck, cv = _gpu(m, tokens, mode, Tmax=27)
    rlg, rck, rcv = _oracle(s, Wn, tokens, mode, Tmax=27)
    assert relerr(lg, rlg) <= TOL["f32"]["logits"]
    assert relerr(ck, rck) <= TOL["f32"]["cache"] and relerr(cv, rcv) <= TOL["f32"]["cache"]


def test_feedback_free_fp32_static_one_hot():
    """Constant mixtures: channel l from the state of layer src[l] <= l."""
    s = small_shape("f32", L=4, k=4, Hq=4, Hkv=2)
    src = [0, 0, 1, 3]
    static = np.zeros((2, s.k, s.L))
    for l in range(s.L):
        static[:, l, src[l]] = 1.0
    m, Wn = model(s, seed=23, jitter=0.2, static=torch.tensor(static))
    tokens = np.random.default_rng(24).integers(0, s.V, size=(2, 20))
    lg, ck, cv = _gpu(m, tokens)
    rlg, rck, rcv = _oracle(s, Wn, tokens, static=static)
    assert relerr(lg, rlg) <= TOL["f32"]["logits"]
    assert relerr(ck, rck) <= TOL["f32"]["cache"] and relerr(cv, rcv) <= TOL["f32"]["cache"]


def test_feedback_free_one_pass_equals_token_steps_fp32():
    """No iteration: one pass = T single-token calls at positions 0..T-1."""
    s = small_shape("f32", L=4, k=4, Hq=4, Hkv=2)
    m, _ = model(s, seed=25, jitter=0.2)
    tokens = np.random.default_rng(26).integers(0, s.V, size=(3, 16))
    lg1, ck1, cv1 = _gpu(m, tokens)
    lg2, ck2, cv2 = _gpu(m, tokens, steps=True)
    assert relerr(lg2, lg1) <= TOL["f32"]["logits"]
    assert relerr(ck2, ck1) <= TOL["f32"]["cache"] and relerr(cv2, cv1) <= TOL["f32"]["cache"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_feedback_free_chunked_workspace(dtype):
    """A workspace for one sequence: the call walks the batch in chunks."""
    s = small_shape(dtype, L=4, k=4, Hq=4, Hkv=2)
    m, _ = model(s, seed=27, jitter=0.2)
    tokens = np.random.default_rng(28).integers(0, s.V, size=(3, 40))
    lg1, ck1, cv1 = _gpu(m, tokens)
    lg2, ck2, cv2 = _gpu(m, tokens, ws_rows=40)
    tol = 1e-5 if dtype == "f32" else 1e-2
    assert relerr(lg2, lg1) <= tol
    assert relerr(ck2, ck1) <= tol and relerr(cv2, cv1) <= tol


@pytest.mark.parametrize("shape_kw", [dict(L=4, k=4, D=256, Hq=4, Hkv=2, d=64),
                                      dict(L=6, k=6, D=512, p=2, p_offset=1, Hq=8, Hkv=2, d=128)])
def test_feedback_free_bf16_vs_oracle(shape_kw):
    """bf16 against the oracle's bf16-storage mode on short sequences; the
    tolerance admits 2.5x the oracle's own spread under 1e-5 weight noise."""
    s = small_shape("bf16", **shape_kw)
    m, Wn = model(s, seed=29, jitter=0.2)
    tokens = np.random.default_rng(30).integers(0, s.V, size=(2, 12))
    lg, ck, cv = _gpu(m, tokens)
    rlg, rck, rcv = _oracle(s, Wn, tokens)
    plg, pck, pcv = _oracle(s, perturbed(Wn, SPREAD_EPS), tokens)
    spread_c = max(relerr(pck, rck), relerr(pcv, rcv))
    assert within(relerr(lg, rlg), TOL["bf16"]["logits"], relerr(plg, rlg), "logits")
    assert within(max(relerr(ck, rck), relerr(cv, rcv)), TOL["bf16"]["cache"], spread_c, "cache")
