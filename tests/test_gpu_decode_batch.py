"""wm_decode_batch (per-sequence positions read on the device) through the C
ABI: against the CPU oracle's decode_batch on ragged positions, against
wm_decode_step at a shared position, replayed from a CUDA graph, and with an
out-of-range position."""

import numpy as np
import pytest
import torch

import oracle.whitematter as O
from cross_layer_kv_pool_b300 import synth, wm
from tests.gpu_util import (SPREAD_EPS, TOL, ensure_lib, host, model, ocfg, perturbed, relerr,
                            small_shape, within)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _random_cache(s, B, Tmax, seed):
    ck = synth.make_normal((B, s.k, s.Hkv, Tmax, s.d), seed, "cuda", 1.0, s.torch_dtype)
    cv = synth.make_normal((B, s.k, s.Hkv, Tmax, s.d), seed + 1, "cuda", 1.0, s.torch_dtype)
    return ck, cv


def _i32(a):
    return torch.tensor(np.asarray(a), dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape_kw", [dict(), dict(d=128, Hq=14, Hkv=2, D=256, L=3, k=3)])
def test_decode_batch_ragged_positions(dtype, shape_kw):
    """Sequences at positions 0, 7, 23 and Tmax - 1 in one call, over a random
    prefix: each row against the oracle from the same cache snapshot."""
    s = small_shape(dtype, **shape_kw)
    m, Wn = model(s, seed=31)
    B, Tmax = 4, 40
    ck, cv = _random_cache(s, B, Tmax, 32)
    pos_h = np.array([0, 7, 23, Tmax - 1])
    tok_h = np.random.default_rng(33).integers(0, s.V, size=B)
    sk, sv = host(ck), host(cv)
    ws = m.workspace(B, Tmax)
    lg = torch.zeros((B, s.V), dtype=torch.float32, device="cuda")
    wm.wm_decode_batch(m, _i32(tok_h), _i32(pos_h), ck, cv, lg, ws)
    torch.cuda.synchronize()
    assert wm.wm_check_flags(ws) == 0
    oc = ocfg(s)
    rk, rv = sk.copy(), sv.copy()
    rl = O.decode_batch(oc, Wn, tok_h, pos_h, rk, rv)
    gk, gv = host(ck), host(cv)
    rows = np.arange(B)
    got_kv = np.stack([gk[rows, :, :, pos_h], gv[rows, :, :, pos_h]])
    ref_kv = np.stack([rk[rows, :, :, pos_h], rv[rows, :, :, pos_h]])
    tol = TOL[dtype]
    if dtype == "f32":
        assert relerr(host(lg), rl) <= tol["logits"]
        assert relerr(got_kv, ref_kv) <= tol["cache"]
    else:
        pk, pv = sk.copy(), sv.copy()
        pl = O.decode_batch(oc, perturbed(Wn, SPREAD_EPS), tok_h, pos_h, pk, pv)
        spread_kv = relerr(np.stack([pk[rows, :, :, pos_h], pv[rows, :, :, pos_h]]), ref_kv)
        assert within(relerr(host(lg), rl), tol["logits"], relerr(pl, rl), "logits")
        assert within(relerr(got_kv, ref_kv), tol["cache"], spread_kv, "cache")
    # nothing but the rows' own positions changed
    mask = np.ones(Tmax, dtype=bool)
    for b in range(B):
        mask[:] = True
        mask[pos_h[b]] = False
        assert np.array_equal(gk[b][:, :, mask], sk[b][:, :, mask])
        assert np.array_equal(gv[b][:, :, mask], sv[b][:, :, mask])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_batch_shared_position_equals_decode_step(dtype):
    s = small_shape(dtype, d=128, Hq=14, Hkv=2, D=256, L=3, k=3)
    m, _ = model(s, seed=34)
    B, Tmax, t = 3, 300, 250
    tok = synth.make_tokens(s, B, 1, seed=35, device="cuda")[:, 0].contiguous()
    out = []
    for batched in (False, True):
        ck, cv = _random_cache(s, B, Tmax, 36)
        ws = m.workspace(B, Tmax)
        lg = torch.zeros((B, s.V), dtype=torch.float32, device="cuda")
        if batched:
            wm.wm_decode_batch(m, tok, _i32(np.full(B, t)), ck, cv, lg, ws)
        else:
            wm.wm_decode_step(m, tok, t, ck, cv, lg, ws)
        torch.cuda.synchronize()
        out.append((host(lg), host(ck)[:, :, :, t], host(cv)[:, :, :, t]))
    tol = 1e-5 if dtype == "f32" else 1e-2
    for a, b in zip(out[0], out[1]):
        assert relerr(b, a) <= tol


def test_decode_batch_graph_replay():
    """One call recorded in a CUDA graph, replayed for 6 steps with the token
    and position buffers updated in place, equals 6 direct calls."""
    s = small_shape("bf16", d=128, Hq=14, Hkv=2, D=256, L=3, k=3)
    m, _ = model(s, seed=37)
    B, Tmax, T = 4, 64, 6
    pos0 = np.array([3, 10, 0, 20])
    toks = synth.make_tokens(s, B, T, seed=38, device="cuda")
    res = []
    for use_graph in (False, True):
        ck, cv = _random_cache(s, B, Tmax, 39)
        ws = m.workspace(B, Tmax)
        lg = torch.zeros((B, s.V), dtype=torch.float32, device="cuda")
        tok_buf = torch.zeros(B, dtype=torch.int32, device="cuda")
        pos_buf = _i32(pos0)
        logits = []
        if use_graph:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):  # first call outside capture (lazy set-up)
                wm.wm_decode_batch(m, tok_buf, pos_buf, ck, cv, lg, ws)
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            ck.copy_(_random_cache(s, B, Tmax, 39)[0])
            cv.copy_(_random_cache(s, B, Tmax, 39)[1])
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                wm.wm_decode_batch(m, tok_buf, pos_buf, ck, cv, lg, ws)
            for t in range(T):
                tok_buf.copy_(toks[:, t])
                g.replay()
                logits.append(lg.clone())
                pos_buf += 1
        else:
            for t in range(T):
                tok_buf.copy_(toks[:, t])
                wm.wm_decode_batch(m, tok_buf, pos_buf, ck, cv, lg, ws)
                logits.append(lg.clone())
                pos_buf += 1
        torch.cuda.synchronize()
        assert wm.wm_check_flags(ws) == 0
        res.append((host(torch.stack(logits)), host(ck), host(cv)))
    for a, b in zip(res[0], res[1]):
        assert relerr(b, a) <= 1e-6


def test_decode_batch_out_of_range_position_flags():
    """A position at Tmax is reported through the flag word; the other rows
    still match the oracle and that sequence's cache is untouched."""
    s = small_shape("f32")
    m, Wn = model(s, seed=40)
    B, Tmax = 3, 16
    ck, cv = _random_cache(s, B, Tmax, 41)
    pos_h = np.array([5, Tmax, 9])
    tok_h = np.random.default_rng(42).integers(0, s.V, size=B)
    sk, sv = host(ck), host(cv)
    ws = m.workspace(B, Tmax)
    lg = torch.zeros((B, s.V), dtype=torch.float32, device="cuda")
    wm.wm_decode_batch(m, _i32(tok_h), _i32(pos_h), ck, cv, lg, ws)
    torch.cuda.synchronize()
    with pytest.raises(wm.WMError):
        wm.wm_check_flags(ws)
    ok = np.array([0, 2])
    rk, rv = sk[ok].copy(), sv[ok].copy()
    rl = O.decode_batch(ocfg(s), Wn, tok_h[ok], pos_h[ok], rk, rv)
    assert relerr(host(lg)[ok], rl) <= TOL["f32"]["logits"]
    assert np.array_equal(host(ck)[1], sk[1]) and np.array_equal(host(cv)[1], sv[1])


def test_decode_batch_1p3b_widths_ragged():
    """The 1.3B model's widths (8 layers, 8 channels), 8 sequences spread over
    positions 1..299: cluster split-K products and the split-key attention
    with sequences of different lengths, against the oracle."""
    s = synth.HALF_1P3B.replace(L=8, k=8, V=2000)
    m, Wn = model(s, seed=43, jitter=0.1)
    B, Tmax = 8, 300
    ck, cv = _random_cache(s, B, Tmax, 44)
    pos_h = np.array([1, 17, 64, 129, 200, 255, 298, 299])
    tok_h = np.random.default_rng(45).integers(0, s.V, size=B)
    sk, sv = host(ck), host(cv)
    ws = m.workspace(B, Tmax)
    lg = torch.zeros((B, s.V), dtype=torch.float32, device="cuda")
    wm.wm_decode_batch(m, _i32(tok_h), _i32(pos_h), ck, cv, lg, ws)
    torch.cuda.synchronize()
    assert wm.wm_check_flags(ws) == 0
    oc = ocfg(s)
    rk, rv = sk.copy(), sv.copy()
    rl = O.decode_batch(oc, Wn, tok_h, pos_h, rk, rv)
    pk, pv = sk.copy(), sv.copy()
    pl = O.decode_batch(oc, perturbed(Wn, SPREAD_EPS), tok_h, pos_h, pk, pv)
    rows = np.arange(B)
    gk, gv = host(ck), host(cv)
    got_kv = np.stack([gk[rows, :, :, pos_h], gv[rows, :, :, pos_h]])
    ref_kv = np.stack([rk[rows, :, :, pos_h], rv[rows, :, :, pos_h]])
    spread_kv = relerr(np.stack([pk[rows, :, :, pos_h], pv[rows, :, :, pos_h]]), ref_kv)
    tol = TOL["bf16"]
    assert within(relerr(host(lg), rl), tol["logits"], relerr(pl, rl), "logits")
    assert within(relerr(got_kv, ref_kv), tol["cache"], spread_kv, "cache")


def test_decode_batch_split_k_fallback_matches_cluster():
    """The few-row products' other split-K path (global fp32 atomics and a
    finalize kernel, taken where a cluster does not fit) gives what the
    cluster path gives, at the 1.3B widths."""
    s = synth.HALF_1P3B.replace(L=4, k=4, V=2000)
    out = []
    for flags in (0, wm.WM_FLAG_NO_CLUSTER):
        W = synth.make_weights(s, seed=46, device="cuda", gain_jitter=0.1)
        m = wm.Model(s, W, flags=flags)
        B, Tmax = 8, 96
        ck, cv = _random_cache(s, B, Tmax, 47)
        pos_h = np.array([3, 10, 20, 33, 47, 60, 80, 95])
        tok_h = np.random.default_rng(48).integers(0, s.V, size=B)
        ws = m.workspace(B, Tmax)
        lg = torch.zeros((B, s.V), dtype=torch.float32, device="cuda")
        wm.wm_decode_batch(m, _i32(tok_h), _i32(pos_h), ck, cv, lg, ws)
        torch.cuda.synchronize()
        assert wm.wm_check_flags(ws) == 0
        rows = np.arange(B)
        out.append((host(lg), host(ck)[rows, :, :, pos_h], host(cv)[rows, :, :, pos_h]))
    for a, b in zip(out[0], out[1]):
        assert relerr(b, a) <= 1e-2


def test_decode_batch_cluster_path_is_repeatable():
    """Without global atomics (the cluster split-K products, the one-wave
    decode attention) a decode step is a fixed sequence of fixed-order sums:
    two calls on the same inputs give bit-identical logits and cache rows."""
    s = synth.HALF_1P3B.replace(L=4, k=4, V=2000)
    W = synth.make_weights(s, seed=49, device="cuda", gain_jitter=0.1)
    m = wm.Model(s, W)
    B, Tmax = 8, 300
    pos_h = np.array([3, 40, 77, 120, 161, 200, 250, 299])
    tok_h = np.random.default_rng(50).integers(0, s.V, size=B)
    rows = np.arange(B)
    outs = []
    for _ in range(2):
        ck, cv = _random_cache(s, B, Tmax, 51)
        ws = m.workspace(B, Tmax)
        lg = torch.zeros((B, s.V), dtype=torch.float32, device="cuda")
        wm.wm_decode_batch(m, _i32(tok_h), _i32(pos_h), ck, cv, lg, ws)
        torch.cuda.synchronize()
        assert wm.wm_check_flags(ws) == 0
        outs.append((host(lg), host(ck)[rows, :, :, pos_h], host(cv)[rows, :, :, pos_h]))
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a, b)
