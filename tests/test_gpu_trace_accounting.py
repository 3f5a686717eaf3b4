"""The work the library reports to its measurement hook (the numerators and
denominators of bench.py's roofline lines) checked against the tensors of
the call: the pool mixer's bytes, the products' FLOPs and the channel
attention's causal FLOPs, counted from the model's weights and the call's
inputs rather than from the library's formulas."""

import pytest
import torch

from cross_layer_kv_pool_b300 import synth, wm
from tests.gpu_util import ensure_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


SHAPE = synth.HALF_1P3B.replace(L=6, D=256, k=3, Hq=4, Hkv=2, d=64, F=512, V=700)


def _traced(m, kind, call):
    tr = wm.Tracer(kind, 512)
    tr.attach(m)
    try:
        call()
    finally:
        wm.Tracer.detach(m)
    torch.cuda.synchronize()
    return tr.results()


def test_mixer_reports_the_bytes_of_the_pool_tensors():
    """One traced wm_pool_mix launch: the layer states read once, the
    coefficients and inverse RMS read once, the mixed channels written once."""
    s = SHAPE
    m = wm.Model(s, synth.make_weights(s, seed=3, device="cuda"))
    N, B, Tmax = 301, 3, 128
    states = synth.make_normal((N, s.L, s.D), 4, "cuda", 1.0, torch.bfloat16)
    g = torch.Generator().manual_seed(5)
    seq = torch.randint(0, B, (N,), generator=g, dtype=torch.int32).cuda()
    pos = torch.randint(0, Tmax, (N,), generator=g, dtype=torch.int32).cuda()
    ck, cv = m.new_cache(B, Tmax)
    ws = m.workspace(N, Tmax)
    res = _traced(m, wm.WM_TRACE_MIX, lambda: wm.wm_pool_mix(m, states, seq, pos, ck, cv, ws))
    assert len(res) == 1
    coeff = torch.empty((N, 2, s.k, s.L), dtype=torch.float32)
    inv = torch.empty((N, s.L), dtype=torch.float32)
    mixed = torch.empty((N, 2, s.k, s.D), dtype=torch.bfloat16)
    assert res[0][1] == states.nbytes + coeff.nbytes + inv.nbytes + mixed.nbytes


def test_decode_step_reports_the_flops_of_its_weights_and_keys():
    """A decode step of B sequences at position t multiplies B rows by every
    weight matrix once (2 FLOP per multiply-add) and, per layer, attends
    over t visible keys per row (QK^T and PV: 4 Hq d FLOP per key)."""
    s = SHAPE
    W = synth.make_weights(s, seed=6, device="cuda")
    m = wm.Model(s, W)
    B, Tmax, t = 5, 96, 37
    ck, cv = m.new_cache(B, Tmax)
    ck.copy_(synth.make_normal(tuple(ck.shape), 7, "cuda", 1.0, torch.bfloat16))
    cv.copy_(synth.make_normal(tuple(cv.shape), 8, "cuda", 1.0, torch.bfloat16))
    tok = synth.make_tokens(s, B, 1, seed=9, device="cuda")[:, 0].contiguous()
    lg = torch.empty((B, s.V), dtype=torch.float32, device="cuda")
    ws = m.workspace(B, Tmax)

    def step():
        wm.wm_decode_step(m, tok, t, ck, cv, lg, ws)

    matrices = ("Wq", "Wo", "Wgate", "Wup", "Wdown", "lm_head", "Wr", "Wk", "Wv")
    gemm = _traced(m, wm.WM_TRACE_GEMM, step)
    assert sum(w for _, w in gemm) == 2 * B * sum(W[n].numel() for n in matrices)
    attn = _traced(m, wm.WM_TRACE_ATTN, step)
    assert len(attn) == s.L
    assert sum(w for _, w in attn) == s.L * 4 * s.Hq * s.d * B * t
    assert wm.wm_check_flags(ws) == 0
