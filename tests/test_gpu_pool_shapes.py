"""Pool parity at the shapes the benchmark runs and at the edges of the pool's
design space, through the C ABI against the CPU oracle:

- the 1.3B model's pool (L = 28 states of D = 1792, k = 14 channels, router
  stride 2): 1,024 rows, a ragged 1,000, rows with strongly correlated layer
  states (the residual stream's shape, where signed mixing cancels), and a
  full 8,192-row group in the benchmark's launch configuration, sampled;
- pool ranks k = 1 (the 16x compression point of the rank sweep, which takes
  the one-channel mixer) and k = 12 ([PL 5 ANALYSIS, "Pool rank"]; [OD
  "Assumptions and limits"]: k swept over 1, 2, 4, 8, 12, 16), in the pool
  alone and in whole cyclic passes;
- static mixing ([PL 5 ANALYSIS, "Dynamic routing"]) with k < L and signed
  constant weights that differ between the K and V branches, so that a
  transposed [2][k][L] read or a branch swap shows.

Bounds (max|gpu - ref| / max|ref| per tensor, bf16 with fp32 accumulation):
coefficients 2e-2, mixed channels 1e-2, K/V 2e-2, logits 2e-2; fp32 1e-4.
bf16 pool results are compared with both placements of the oracle's rounding
of the stored channel (reading R17): "gained" rounds u = tau (.) m as the
kernel stores it, "normed" rounds the normalised channel c, the plain reading.
"""

import copy

import numpy as np
import pytest
import torch

import oracle.whitematter as O
from cross_layer_kv_pool_b300 import synth, wm
from tests.gpu_util import (TOL, ensure_lib, host, isolated_passes, model, normerr, ocfg,
                            record, relerr, small_shape, within)

pytestmark = pytest.mark.gpu

# The 1.3B model's pool; F, Hq and V do not enter the pool and are kept small
# so that the unused stack weights stay small.
POOL_1P3B = synth.HALF_1P3B.replace(F=64, Hq=2, V=64)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _placements(s):
    out = {"gained": ocfg(s)}
    if s.dtype == "bf16":
        normed = copy.copy(out["gained"])
        normed.mixed_storage = "normed"
        out["normed"] = normed
    return out


def _states(s, N, seed, correlated):
    x = synth.make_normal((N, s.L, s.D), seed, "cuda", 1.0, torch.float32)
    if correlated:
        # h^l = h^0 + small increments: the layer states of a residual stream,
        # whose signed mixtures cancel
        x = x[:, :1, :] + 0.05 * torch.cumsum(x, dim=1)
    return x.to(s.torch_dtype).contiguous()


def _pool_call(m, states, seq_h, pos_h, B, Tmax, want_mixed=True):
    s = m.shape
    N = states.shape[0]
    seq = torch.tensor(seq_h, dtype=torch.int32, device="cuda")
    pos = torch.tensor(pos_h, dtype=torch.int32, device="cuda")
    ck, cv = m.new_cache(B, Tmax, fill=float("nan"))
    coeff = torch.empty((N, 2, s.k, s.L), dtype=torch.float32, device="cuda")
    mixed = torch.empty((2, s.k, N, s.D), dtype=s.torch_dtype, device="cuda") if want_mixed else None
    ws = m.workspace(N, Tmax)
    wm.wm_pool_mix(m, states, seq, pos, ck, cv, ws, coeff_out=coeff, mixed_out=mixed)
    torch.cuda.synchronize()
    assert wm.wm_check_flags(ws) == 0
    return ck, cv, coeff, mixed


def _compare(name, s, Wn, states_h, seq_h, pos_h, rows, ck, cv, coeff, mixed, static=None):
    """Oracle on ``rows`` (rows of a pool call do not interact) under each
    rounding placement; asserts the bounds and records the errors."""
    tol = TOL[s.dtype]
    K = ck[seq_h[rows], :, :, pos_h[rows], :]
    Vv = cv[seq_h[rows], :, :, pos_h[rows], :]
    gK, gV = host(K), host(Vv)
    gc = host(coeff[rows])
    gm = host(mixed[:, :, rows, :]).transpose(2, 0, 1, 3)
    for place, oc in _placements(s).items():
        ref = O.pool(oc, Wn, states_h, pos_h[rows], static_coeff=static)
        e = dict(coeff=relerr(gc, ref["coeff"]), mixed=relerr(gm, ref["mixed"]),
                 K=relerr(gK, ref["K"]), V=relerr(gV, ref["V"]),
                 mixed_norm=normerr(gm, ref["mixed"]), K_norm=normerr(gK, ref["K"]))
        record(name, placement=place, rows=len(rows), **e)
        assert e["coeff"] <= tol["coeff"], (place, e)
        assert e["mixed"] <= tol["mixed"], (place, e)
        assert e["K"] <= tol["cache"] and e["V"] <= tol["cache"], (place, e)


def _written_exactly(ck, cv, seq_h, pos_h, B, Tmax):
    """Exactly the rows' (seq, pos) slots became finite (bit-exact indexing)."""
    want = torch.zeros((B, Tmax), dtype=torch.bool, device="cuda")
    want[torch.as_tensor(seq_h, device="cuda"), torch.as_tensor(pos_h, device="cuda")] = True
    for c in (ck, cv):
        fin = ~torch.isnan(c).any(dim=4).any(dim=2).any(dim=1)
        assert torch.equal(fin, want)


@pytest.mark.parametrize("N,correlated", [(1024, False), (1000, False), (1024, True)])
def test_pool_mix_1p3b_shape(N, correlated):
    s = POOL_1P3B
    m, Wn = model(s, seed=41, jitter=0.1)
    B, Tmax = 8, 2048
    rng = np.random.default_rng(N)
    flat = rng.choice(B * Tmax, size=N, replace=False)
    seq_h, pos_h = flat // Tmax, flat % Tmax
    states = _states(s, N, 43, correlated)
    ck, cv, coeff, mixed = _pool_call(m, states, seq_h, pos_h, B, Tmax)
    _written_exactly(ck, cv, seq_h, pos_h, B, Tmax)
    rows = np.arange(N)
    _compare(f"pool_1p3b[N={N},corr={int(correlated)}]", s, Wn, host(states), seq_h, pos_h, rows,
             ck, cv, coeff, mixed)


def test_pool_mix_1p3b_full_group_sampled():
    """One 8,192-row group of the benchmark (64 sequences, group q = 15 of
    g = 16 over T = 2048): every written slot checked bit-exactly, 192
    sampled rows (both ends and the middle) against the oracle."""
    s = POOL_1P3B
    m, Wn = model(s, seed=42, jitter=0.1)
    B, T, g, q = 64, 2048, 16, 15
    P = np.arange(q, T, g)
    seq_h = np.repeat(np.arange(B), len(P))
    pos_h = np.tile(P, B)
    N = len(seq_h)
    assert N == 8192
    states = _states(s, N, 44, True)
    ck, cv, coeff, mixed = _pool_call(m, states, seq_h, pos_h, B, T)
    _written_exactly(ck, cv, seq_h, pos_h, B, T)
    rng = np.random.default_rng(3)
    rows = np.unique(np.r_[0:32, N - 32:N, rng.choice(N, 128, replace=False)])
    _compare("pool_1p3b_group8192", s, Wn, host(states[torch.as_tensor(rows, device="cuda")]),
             seq_h, pos_h, rows, ck, cv, coeff, mixed)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("k", [1, 12])
def test_pool_mix_rank(dtype, k):
    s = synth.HALF_SMALL.replace(k=k, V=64, dtype=dtype)
    m, Wn = model(s, seed=50 + k, jitter=0.2)
    B, Tmax, N = 4, 512, 300
    rng = np.random.default_rng(k)
    flat = rng.choice(B * Tmax, size=N, replace=False)
    seq_h, pos_h = flat // Tmax, flat % Tmax
    states = _states(s, N, 60 + k, False)
    ck, cv, coeff, mixed = _pool_call(m, states, seq_h, pos_h, B, Tmax)
    _written_exactly(ck, cv, seq_h, pos_h, B, Tmax)
    _compare(f"pool_rank[k={k},{dtype}]", s, Wn, host(states), seq_h, pos_h, np.arange(N),
             ck, cv, coeff, mixed)


@pytest.mark.parametrize("k", [1, 12])
def test_cyclic_pass_rank_fp32(k):
    """fp32 end to end: 3 cyclic passes (g = 4) at pool rank k."""
    s = small_shape("f32", L=12, k=k, D=128, Hq=4, Hkv=2, F=256, V=256)
    m, Wn = model(s, seed=70 + k, jitter=0.1)
    B, T, g = 2, 24, 4
    tokens = np.random.default_rng(k).integers(0, s.V, size=(B, T))
    tok = torch.tensor(tokens, dtype=torch.int32, device="cuda")
    ck, cv = m.new_cache(B, T)
    ws = m.workspace(wm.rows_for_pass(B, T, g), T)
    lg = torch.zeros((B, T, s.V), dtype=torch.float32, device="cuda")
    rck, rcv = O.new_cache(s, B, T)
    for n in range(3):
        last = n == 2
        wm.wm_cyclic_pass(m, tok, g, ck, cv, ws, logits=lg if last else None,
                          logits_mode="all" if last else "none")
        rl = O.cyclic_pass(ocfg(s), Wn, tokens, g, rck, rcv, logits="all" if last else None)
    torch.cuda.synchronize()
    assert wm.wm_check_flags(ws) == 0
    e = dict(logits=relerr(host(lg), rl), K=relerr(host(ck), rck), V=relerr(host(cv), rcv))
    record(f"cyclic_rank_fp32[k={k}]", **e)
    assert max(e.values()) <= 1e-4, e


@pytest.mark.parametrize("k", [1, 12])
def test_cyclic_pass_rank_bf16_isolated(k):
    """bf16 cyclic passes of the half-small model's widths at pool rank k,
    every group compared with the oracle from the GPU's cache snapshot."""
    s = synth.HALF_SMALL.replace(k=k, V=1000)
    m, Wn = model(s, seed=80 + k, jitter=0.1)
    B, T, g = 2, 32, 8
    tokens = np.random.default_rng(80 + k).integers(0, s.V, size=(B, T))
    w = isolated_passes(m, Wn, tokens, g, 2, logits_mode="last", spread=True)
    assert w["checked"] == 16
    assert within(w["logits"], TOL["bf16"]["logits"], w["spread_logits"], "logits"), w
    assert within(w["cache"], TOL["bf16"]["cache_step"], w["spread_cache"], "cache"), w


def _static(k, L, seed):
    rng = np.random.default_rng(seed)
    st = rng.standard_normal((2, k, L))
    st[1] = -0.5 * st[1][::-1]          # the V branch differs from the K branch
    return st


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_static_mixing_pool_asymmetric(dtype):
    s = small_shape(dtype, L=6, k=3, D=256, Hq=4, Hkv=2, d=64)
    st = _static(s.k, s.L, 5)
    m, Wn = model(s, seed=90, jitter=0.2, static=torch.tensor(st))
    B, Tmax, N = 3, 64, 61
    rng = np.random.default_rng(9)
    flat = rng.choice(B * Tmax, size=N, replace=False)
    seq_h, pos_h = flat // Tmax, flat % Tmax
    states = _states(s, N, 91, False)
    ck, cv, coeff, mixed = _pool_call(m, states, seq_h, pos_h, B, Tmax)
    _written_exactly(ck, cv, seq_h, pos_h, B, Tmax)
    # the coefficients are the constants themselves, for every row, bit-exactly
    assert np.array_equal(host(coeff), np.broadcast_to(st.astype(np.float32), (N, 2, s.k, s.L)))
    _compare(f"static_pool[{dtype}]", s, Wn, host(states), seq_h, pos_h, np.arange(N),
             ck, cv, coeff, mixed, static=st)


def test_static_mixing_cyclic_fp32():
    """fp32 end to end: cyclic passes with asymmetric static mixing, k < L."""
    s = small_shape("f32", L=6, k=3, D=128, Hq=4, Hkv=2, F=256, V=256)
    st = _static(s.k, s.L, 6)
    m, Wn = model(s, seed=92, jitter=0.1, static=torch.tensor(st))
    B, T, g = 2, 20, 4
    tokens = np.random.default_rng(92).integers(0, s.V, size=(B, T))
    tok = torch.tensor(tokens, dtype=torch.int32, device="cuda")
    ck, cv = m.new_cache(B, T)
    ws = m.workspace(wm.rows_for_pass(B, T, g), T)
    lg = torch.zeros((B, s.V), dtype=torch.float32, device="cuda")
    rck, rcv = O.new_cache(s, B, T)
    for n in range(3):
        last = n == 2
        wm.wm_cyclic_pass(m, tok, g, ck, cv, ws, logits=lg if last else None,
                          logits_mode="last" if last else "none")
        rl = O.cyclic_pass(ocfg(s), Wn, tokens, g, rck, rcv, logits="last" if last else None,
                           static_coeff=st)
    torch.cuda.synchronize()
    assert wm.wm_check_flags(ws) == 0
    e = dict(logits=relerr(host(lg), rl), K=relerr(host(ck), rck), V=relerr(host(cv), rcv))
    record("static_cyclic_fp32", **e)
    assert max(e.values()) <= 1e-4, e


def test_static_mixing_cyclic_bf16_isolated():
    s = small_shape("bf16", L=6, k=3, D=256, Hq=4, Hkv=2, F=256, V=512)
    st = _static(s.k, s.L, 7)
    m, Wn = model(s, seed=93, jitter=0.1, static=torch.tensor(st))
    B, T, g = 2, 24, 6
    tokens = np.random.default_rng(93).integers(0, s.V, size=(B, T))
    w = isolated_passes(m, Wn, tokens, g, 2, logits_mode="last", static=st)
    record("static_cyclic_bf16", **w)
    assert w["checked"] == 12
    assert w["logits"] <= TOL["bf16"]["logits"], w
    assert w["cache"] <= TOL["bf16"]["cache"], w
