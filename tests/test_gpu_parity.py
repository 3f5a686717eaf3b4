"""GPU path (through the C ABI) against the CPU oracle on seeded inputs."""

import numpy as np
import pytest
import torch

import oracle.whitematter as O
from cross_layer_kv_pool_b300 import synth, wm
from tests.gpu_util import (TOL, ensure_lib, host, isolated_decode, isolated_passes, model, ocfg,
                            record, relerr, small_shape, within)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


# ---------------------------------------------------------------------------
# Channel attention
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("rps", [0, 200, 1])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d,Hq,Hkv", [(64, 4, 2), (128, 14, 2), (64, 8, 8)])
def test_attention_uniform_closed_form(dtype, d, Hq, Hkv, rps):
    """Zero keys: the output is the mean of the visible values, which encode
    channel, sequence, position and KV head; checked exactly."""
    s = small_shape(dtype, d=d, Hq=Hq, Hkv=Hkv, k=3)
    cfg = wm.make_config(s)
    B, Tmax = 2, 200
    ck = torch.zeros((B, s.k, Hkv, Tmax, d), dtype=s.torch_dtype, device="cuda")
    cv = torch.zeros_like(ck)
    for c in range(s.k):
        cv[:, c, :, :, 0] = c
    cv[:, :, :, :, 1] = torch.arange(B, device="cuda").view(B, 1, 1, 1).to(s.torch_dtype)
    cv[:, :, :, :, 2] = torch.arange(Tmax, device="cuda").view(1, 1, 1, Tmax).to(s.torch_dtype)
    cv[:, :, :, :, 3] = torch.arange(Hkv, device="cuda").view(1, 1, Hkv, 1).to(s.torch_dtype)
    seq = torch.arange(B, device="cuda", dtype=torch.int32).repeat_interleave(Tmax)
    pos = torch.arange(Tmax, device="cuda", dtype=torch.int32).repeat(B)
    N = B * Tmax
    q = synth.make_normal((N, Hq, d), seed=3, device="cuda", dtype=s.torch_dtype)
    out = torch.empty((N, Hq * d), dtype=s.torch_dtype, device="cuda")
    ws = torch.zeros(wm.workspace_size(cfg, N, Tmax), dtype=torch.uint8, device="cuda")
    for c in range(s.k):
        wm.wm_channel_attn(cfg, q, seq, pos, c, ck, cv, out, ws, rows_per_seq=rps)
        torch.cuda.synchronize()
        o = host(out).reshape(N, Hq, d)
        P = host(pos)
        Sq = host(seq)
        z = P == 0
        assert np.all(o[z] == 0.0)
        nz = ~z
        assert np.all(o[nz, :, 0] == c)
        assert np.all(o[nz, :, 1] == Sq[nz, None])
        assert np.all(o[nz, :, 3] == (np.arange(Hq) * Hkv // Hq)[None, :])
        mean_pos = (P[nz] - 1) / 2.0
        if dtype == "bf16":
            assert np.all(o[nz, :, 2] == mean_pos[:, None])
        else:
            assert np.max(np.abs(o[nz, :, 2] - mean_pos[:, None])) <= 1e-5 * Tmax
    assert wm.wm_check_flags(ws) == 0


@pytest.mark.parametrize("rps", [0, 1])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d,Hq,Hkv,Tmax", [(64, 4, 2, 300), (128, 14, 2, 257), (64, 8, 8, 130),
                                           (128, 14, 2, 2304), (64, 16, 2, 520), (128, 16, 1, 700),
                                           (64, 12, 4, 333), (64, 16, 1, 450), (128, 12, 1, 610)])
def test_attention_vs_oracle(dtype, d, Hq, Hkv, Tmax, rps):
    """Random rows; rows_per_seq = 1 takes the decode engine (key splits)."""
    s = small_shape(dtype, d=d, Hq=Hq, Hkv=Hkv, k=2)
    cfg = wm.make_config(s)
    B = 2
    ck = synth.make_normal((B, s.k, Hkv, Tmax, d), 11, "cuda", 2.0, s.torch_dtype)
    cv = synth.make_normal((B, s.k, Hkv, Tmax, d), 12, "cuda", 1.0, s.torch_dtype)
    rng = np.random.default_rng(0)
    N = 97
    pos_h = rng.integers(0, Tmax, size=N)
    pos_h[:3] = [0, 1, Tmax - 1]
    seq_h = rng.integers(0, B, size=N)
    seq = torch.tensor(seq_h, dtype=torch.int32, device="cuda")
    pos = torch.tensor(pos_h, dtype=torch.int32, device="cuda")
    q = synth.make_normal((N, Hq, d), 13, "cuda", 1.0, s.torch_dtype)
    out = torch.empty((N, Hq * d), dtype=s.torch_dtype, device="cuda")
    ws = torch.zeros(wm.workspace_size(cfg, N, Tmax), dtype=torch.uint8, device="cuda")
    for c in range(s.k):
        wm.wm_channel_attn(cfg, q, seq, pos, c, ck, cv, out, ws, rows_per_seq=rps)
        torch.cuda.synchronize()
        K, Vv, Q = host(ck), host(cv), host(q)
        ref = np.stack([O.channel_attention(Q[r], K[seq_h[r], c], Vv[seq_h[r], c], pos_h[r], Hq, Hkv)
                        for r in range(N)])
        err = relerr(host(out).reshape(N, Hq, d), ref)
        record(f"attention_vs_oracle[{dtype},d={d},Hq={Hq},Hkv={Hkv},Tmax={Tmax},rps={rps}]",
               channel=c, attn=err)
        assert err <= TOL[dtype]["attn"], err


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d,Hq,Hkv,Tmax,g", [(128, 14, 2, 2304, 16), (64, 8, 8, 700, 4),
                                             (128, 4, 1, 300, 7)])
def test_attention_group_rows_vs_oracle(dtype, d, Hq, Hkv, Tmax, g):
    """Rows shaped like a cyclic group (per sequence, positions q + u*g), the
    tensor-core path, including key blocks past Tmax and a ragged last tile."""
    s = small_shape(dtype, d=d, Hq=Hq, Hkv=Hkv, k=3)
    cfg = wm.make_config(s)
    B, q = 3, g - 1
    P = np.arange(q, Tmax, g)
    nq = len(P)
    ck = synth.make_normal((B, s.k, Hkv, Tmax, d), 21, "cuda", 2.0, s.torch_dtype)
    cv = synth.make_normal((B, s.k, Hkv, Tmax, d), 22, "cuda", 1.0, s.torch_dtype)
    seq_h = np.repeat(np.arange(B), nq)
    pos_h = np.tile(P, B)
    N = B * nq
    seq = torch.tensor(seq_h, dtype=torch.int32, device="cuda")
    pos = torch.tensor(pos_h, dtype=torch.int32, device="cuda")
    qt = synth.make_normal((N, Hq, d), 23, "cuda", 1.0, s.torch_dtype)
    out = torch.empty((N, Hq * d), dtype=s.torch_dtype, device="cuda")
    ws = torch.zeros(wm.workspace_size(cfg, N, Tmax), dtype=torch.uint8, device="cuda")
    c = 2
    wm.wm_channel_attn(cfg, qt, seq, pos, c, ck, cv, out, ws, rows_per_seq=nq)
    torch.cuda.synchronize()
    assert wm.wm_check_flags(ws) == 0
    K, Vv, Q = host(ck), host(cv), host(qt)
    rows = np.r_[0:8, nq - 8:nq + 8, N - 8:N]
    ref = np.stack([O.channel_attention(Q[r], K[seq_h[r], c], Vv[seq_h[r], c], pos_h[r], Hq, Hkv)
                    for r in rows])
    err = relerr(host(out).reshape(N, Hq, d)[rows], ref)
    record(f"attention_group_rows[{dtype},d={d},Tmax={Tmax},g={g}]", attn=err)
    assert err <= TOL[dtype]["attn"], err


@pytest.mark.parametrize("d,Hq,Hkv,Tmax,nq", [(128, 14, 2, 900, 61), (64, 8, 2, 520, 37),
                                              (128, 2, 2, 300, 300), (64, 16, 1, 260, 9)])
def test_attention_tile_pairs_all_rows(d, Hq, Hkv, Tmax, nq):
    """Every row of structured calls on the tensor-core path (two query tiles
    per CTA sharing each key block): positions in any order within a
    sequence, a first tile whose rows all sit at position 0 (no visible key)
    beside a second that sees keys, a ragged last tile, and a sequence id
    out of range (its rows read no key and come out zero, with the flag)."""
    s = small_shape("bf16", d=d, Hq=Hq, Hkv=Hkv, k=2)
    cfg = wm.make_config(s)
    B = 3
    G = Hq // Hkv
    ck = synth.make_normal((B, s.k, Hkv, Tmax, d), 31, "cuda", 2.0, s.torch_dtype)
    cv = synth.make_normal((B, s.k, Hkv, Tmax, d), 32, "cuda", 1.0, s.torch_dtype)
    rng = np.random.default_rng(nq)
    nseq = 4
    seq_h = np.repeat(np.array([0, 2, 1, B]), nq)        # the last sequence id is invalid
    pos_h = rng.integers(0, Tmax, size=nseq * nq)
    cap = 128 // G
    tiles = -(-nq // cap)
    tiles += tiles & 1
    rpt = -(-nq // tiles)
    pos_h[nq:nq + min(rpt, nq)] = 0                       # sequence 1: its first tile sees nothing
    pos_h[0] = Tmax - 1
    N = nseq * nq
    seq = torch.tensor(seq_h, dtype=torch.int32, device="cuda")
    pos = torch.tensor(pos_h, dtype=torch.int32, device="cuda")
    qt = synth.make_normal((N, Hq, d), 33, "cuda", 1.0, s.torch_dtype)
    out = torch.full((N, Hq * d), float("nan"), dtype=s.torch_dtype, device="cuda")
    ws = torch.zeros(wm.workspace_size(cfg, N, Tmax), dtype=torch.uint8, device="cuda")
    c = 1
    wm.wm_channel_attn(cfg, qt, seq, pos, c, ck, cv, out, ws, rows_per_seq=nq)
    torch.cuda.synchronize()
    with pytest.raises(wm.WMError) as e:
        wm.wm_check_flags(ws)
    assert e.value.status == wm.WM_ERR_DEVICE_BOUNDS
    got = host(out).reshape(N, Hq, d)
    K, Vv, Q = host(ck), host(cv), host(qt)
    ok_rows = np.arange(3 * nq)
    ref = np.stack([O.channel_attention(Q[r], K[seq_h[r], c], Vv[seq_h[r], c], pos_h[r], Hq, Hkv)
                    for r in ok_rows])
    err = relerr(got[ok_rows], ref)
    record(f"attention_tile_pairs[d={d},Hq={Hq},Hkv={Hkv},Tmax={Tmax},nq={nq}]", attn=err)
    assert err <= TOL["bf16"]["attn"], err
    assert np.all(got[:3 * nq][pos_h[:3 * nq] == 0] == 0)
    assert np.all(got[3 * nq:] == 0)


# ---------------------------------------------------------------------------
# Pool
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape_kw", [dict(), dict(L=6, k=3, p=2, p_offset=1, d=128, Hq=2, Hkv=1, D=256),
                                      dict(L=5, k=5, p=3, Hkv=4, Hq=4)])
def test_pool_mix_vs_oracle(dtype, shape_kw):
    s = small_shape(dtype, **shape_kw)
    m, Wn = model(s, seed=5, jitter=0.2)
    B, Tmax, N = 3, 40, 37
    rng = np.random.default_rng(1)
    flat = rng.choice(B * Tmax, size=N, replace=False)
    seq_h, pos_h = flat // Tmax, flat % Tmax
    states = synth.make_normal((N, s.L, s.D), 21, "cuda", 1.0, s.torch_dtype)
    seq = torch.tensor(seq_h, dtype=torch.int32, device="cuda")
    pos = torch.tensor(pos_h, dtype=torch.int32, device="cuda")
    ck, cv = m.new_cache(B, Tmax, fill=float("nan"))
    coeff = torch.empty((N, 2, s.k, s.L), dtype=torch.float32, device="cuda")
    mixed = torch.empty((2, s.k, N, s.D), dtype=s.torch_dtype, device="cuda")
    ws = m.workspace(N, Tmax)
    wm.wm_pool_mix(m, states, seq, pos, ck, cv, ws, coeff_out=coeff, mixed_out=mixed)
    torch.cuda.synchronize()
    assert wm.wm_check_flags(ws) == 0
    ref = O.pool(ocfg(s), Wn, host(states), pos_h)
    tol = TOL[dtype]
    record(f"pool_mix_vs_oracle[{dtype},{shape_kw}]", coeff=relerr(host(coeff), ref["coeff"]),
           mixed=relerr(host(mixed).transpose(2, 0, 1, 3), ref["mixed"]),
           K=relerr(host(ck)[seq_h, :, :, pos_h, :], ref["K"]),
           V=relerr(host(cv)[seq_h, :, :, pos_h, :], ref["V"]))
    assert relerr(host(coeff), ref["coeff"]) <= tol["coeff"]
    assert relerr(host(mixed).transpose(2, 0, 1, 3), ref["mixed"]) <= tol["mixed"]
    K, Vv = host(ck), host(cv)
    written = np.zeros((B, Tmax), dtype=bool)
    written[seq_h, pos_h] = True
    assert np.array_equal(~np.isnan(K).any(axis=(1, 2, 4)), written)
    assert np.array_equal(~np.isnan(Vv).any(axis=(1, 2, 4)), written)
    gk = K[seq_h, :, :, pos_h, :]
    gv = Vv[seq_h, :, :, pos_h, :]
    assert relerr(gk, ref["K"]) <= tol["cache"]
    assert relerr(gv, ref["V"]) <= tol["cache"]


# ---------------------------------------------------------------------------
# Whole passes and decode
# ---------------------------------------------------------------------------

def _gpu_passes(m, tokens_h, g, passes, Tmax=None, logits_mode="all", static=None):
    s = m.shape
    B, T = tokens_h.shape
    Tmax = Tmax or T
    tok = torch.tensor(tokens_h, dtype=torch.int32, device="cuda")
    ck, cv = m.new_cache(B, Tmax)
    ws = m.workspace(wm.rows_for_pass(B, T, g), Tmax)
    shp = (B, T, s.V) if logits_mode == "all" else (B, s.V)
    lg = torch.zeros(shp, dtype=torch.float32, device="cuda")
    for n in range(passes):
        last = n == passes - 1
        wm.wm_cyclic_pass(m, tok, g, ck, cv, ws, logits=lg if last else None,
                          logits_mode=logits_mode if last else "none")
    torch.cuda.synchronize()
    assert wm.wm_check_flags(ws) == 0
    return host(lg), host(ck), host(cv)


def _oracle_passes(s, Wn, tokens_h, g, passes, Tmax=None, logits="all", static=None):
    B, T = tokens_h.shape
    s = ocfg(s)
    ck, cv = O.new_cache(s, B, Tmax or T)
    lg = None
    for n in range(passes):
        lg = O.cyclic_pass(s, Wn, tokens_h, g, ck, cv, logits=logits if n == passes - 1 else None,
                           static_coeff=static)
    return lg, ck, cv


def test_tiny_fp32_cyclic_and_jacobi():
    """The tiny fp32 workload: cyclic g=4 for 3 passes and Jacobi for 64."""
    wl = synth.WORKLOADS["tiny_fp32"]
    s = wl["shape"]
    m, Wn = model(s, seed=0, jitter=0.1)
    tokens = host(synth.make_tokens(s, wl["B"], wl["T"], seed=1)).astype(np.int64)
    for g, passes in ((4, 3), (1, 64)):
        lg, ck, cv = _gpu_passes(m, tokens, g, passes)
        rlg, rck, rcv = _oracle_passes(s, Wn, tokens, g, passes)
        assert relerr(lg, rlg) <= 1e-4, (g, relerr(lg, rlg))
        assert relerr(ck, rck) <= 1e-4
        assert relerr(cv, rcv) <= 1e-4


def test_decode_steps_fp32_end_to_end():
    """fp32: T decode steps from a zero cache equal the oracle's exact
    autoregressive evaluation, and so does one cyclic pass with g = T."""
    s = small_shape("f32")
    m, Wn = model(s, seed=2)
    B, T = 2, 12
    tokens = np.random.default_rng(3).integers(0, s.V, size=(B, T))
    ck, cv = m.new_cache(B, T)
    ws = m.workspace(B, T)
    lg = torch.zeros((B, s.V), dtype=torch.float32, device="cuda")
    tok = torch.tensor(tokens, dtype=torch.int32, device="cuda")
    out = []
    for t in range(T):
        wm.wm_decode_step(m, tok[:, t].contiguous(), t, ck, cv, lg, ws)
        out.append(host(lg))
    torch.cuda.synchronize()
    dec = np.stack(out, axis=1)
    rck, rcv = O.new_cache(s, B, T)
    ref = O.autoregressive(ocfg(s), Wn, tokens, rck, rcv)
    assert relerr(dec, ref) <= 1e-4
    assert relerr(host(ck), rck) <= 1e-4
    lg2, ck2, _ = _gpu_passes(m, tokens, T, 1)
    assert relerr(lg2, dec) <= 1e-4
    assert relerr(ck2, host(ck)) <= 1e-4


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape_kw", [dict(), dict(d=128, Hq=14, Hkv=2, D=256, L=3, k=3)])
def test_decode_steps_isolated(dtype, shape_kw):
    s = small_shape(dtype, **shape_kw)
    m, Wn = model(s, seed=2)
    B, T = 3, 10
    tokens = np.random.default_rng(3).integers(0, s.V, size=(B, T))
    w = isolated_decode(m, Wn, tokens, Tmax=T + 5, spread=dtype == "bf16")
    tol = TOL[dtype]
    assert within(w["logits"], tol["logits"], w["spread_logits"], "logits"), w
    assert within(w["cache"], tol["cache"], w["spread_cache"], "cache"), w


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape_kw", [dict(d=128, Hq=14, Hkv=2, D=256, L=3, k=3),
                                      dict(L=4, k=2, Hq=8, Hkv=8)])
def test_decode_long_context_isolated(dtype, shape_kw):
    """Decode steps at positions near 700 and 2000 over a random prefix: the
    decode engine splits the keys across CTAs and merges the splits."""
    s = small_shape(dtype, **shape_kw)
    m, Wn = model(s, seed=12)
    B, Tmax = 3, 2100
    for start in (700, 2001):
        ck = synth.make_normal((B, s.k, s.Hkv, Tmax, s.d), 40 + start, "cuda", 1.0, s.torch_dtype)
        cv = synth.make_normal((B, s.k, s.Hkv, Tmax, s.d), 41 + start, "cuda", 1.0, s.torch_dtype)
        tokens = np.random.default_rng(start).integers(0, s.V, size=(B, 3))
        w = isolated_decode(m, Wn, tokens, Tmax, start_cache=(ck, cv), start_pos=start,
                            spread=dtype == "bf16")
        tol = TOL[dtype]
        assert within(w["logits"], tol["logits"], w["spread_logits"], "logits"), (start, w)
        assert within(w["cache"], tol["cache"], w["spread_cache"], "cache"), (start, w)


def test_decode_1p3b_widths_isolated():
    """Decode steps with the 1.3B model's widths (D 1792, 14 query heads of 128,
    2 KV heads, F 4608), 8 layers and 8 channels: tcgen05 products with K
    split over a thread-block cluster (the SwiGLU projection included) and the
    split-key decode attention."""
    s = synth.HALF_1P3B.replace(L=8, k=8, V=2000)
    m, Wn = model(s, seed=21, jitter=0.1)
    B, Tmax, start = 8, 300, 250
    ck = synth.make_normal((B, s.k, s.Hkv, Tmax, s.d), 51, "cuda", 1.0, s.torch_dtype)
    cv = synth.make_normal((B, s.k, s.Hkv, Tmax, s.d), 52, "cuda", 1.0, s.torch_dtype)
    tokens = np.random.default_rng(5).integers(0, s.V, size=(B, 3))
    w = isolated_decode(m, Wn, tokens, Tmax, start_cache=(ck, cv), start_pos=start, spread=True)
    tol = TOL["bf16"]
    assert within(w["logits"], tol["logits"], w["spread_logits"], "logits"), w
    assert within(w["cache"], tol["cache"], w["spread_cache"], "cache"), w


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_partial_pass_writes_exact_positions(dtype):
    s = small_shape(dtype)
    m, _ = model(s, seed=4)
    B, T, g = 2, 23, 5
    tok = synth.make_tokens(s, B, T, seed=9, device="cuda")
    ws = m.workspace(wm.rows_for_pass(B, T, g), T)
    for qb, qe in ((0, 2), (1, 5), (4, 5), (2, 2)):
        ck, cv = m.new_cache(B, T, fill=1000.0)
        wm.wm_cyclic_pass(m, tok, g, ck, cv, ws, q_begin=qb, q_end=qe)
        torch.cuda.synchronize()
        K, Vv = host(ck), host(cv)
        changed = (K != 1000.0).any(axis=(1, 2, 4)) | (Vv != 1000.0).any(axis=(1, 2, 4))
        expect = np.array([[qb <= i % g < qe for i in range(T)]] * B)
        assert np.array_equal(changed, expect), (qb, qe)


def test_uneven_groups_fp32_end_to_end():
    s = small_shape("f32", Hkv=4, Hq=4)
    m, Wn = model(s, seed=6, jitter=0.2)
    B, T, g = 2, 29, 6
    tokens = np.random.default_rng(7).integers(0, s.V, size=(B, T))
    for mode in ("last", "all"):
        lg, ck, cv = _gpu_passes(m, tokens, g, 3, Tmax=T + 3, logits_mode=mode)
        rlg, rck, rcv = _oracle_passes(s, Wn, tokens, g, 3, Tmax=T + 3, logits=mode)
        assert relerr(lg, rlg) <= 1e-4
        assert relerr(ck, rck) <= 1e-4 and relerr(cv, rcv) <= 1e-4


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", ["last", "all"])
def test_uneven_groups_isolated(dtype, mode):
    s = small_shape(dtype, Hkv=4, Hq=4)
    m, Wn = model(s, seed=6, jitter=0.2)
    B, T, g = 2, 29, 6
    tokens = np.random.default_rng(7).integers(0, s.V, size=(B, T))
    w = isolated_passes(m, Wn, tokens, g, 3, Tmax=T + 3, logits_mode=mode, spread=dtype == "bf16")
    tol = TOL[dtype]
    assert w["checked"] == 18
    assert within(w["logits"], tol["logits"], w["spread_logits"], "logits"), w
    assert within(w["cache"], tol["cache"], w["spread_cache"], "cache"), w


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_identity_router_full_cache(dtype):
    """k = L with the forced identity mixture (static weights)."""
    s = small_shape(dtype, L=4, k=4)
    static = np.zeros((2, s.k, s.L))
    static[0] = static[1] = np.eye(s.L)
    m, Wn = model(s, seed=8, static=torch.tensor(static))
    B, T = 1, 16
    tokens = np.random.default_rng(8).integers(0, s.V, size=(B, T))
    if dtype == "f32":
        lg, ck, _ = _gpu_passes(m, tokens, 4, 4, static=static)
        rlg, rck, _ = _oracle_passes(s, Wn, tokens, 4, 4, static=static)
        assert relerr(lg, rlg) <= 1e-4 and relerr(ck, rck) <= 1e-4
    else:
        import oracle.whitematter as Om
        orig = Om.cyclic_pass

        def with_static(*a, **k):
            k["static_coeff"] = static
            return orig(*a, **k)
        Om.cyclic_pass = with_static
        try:
            w = isolated_passes(m, Wn, tokens, 4, 4, logits_mode="all")
        finally:
            Om.cyclic_pass = orig
        record("identity_router_bf16", **w)
        assert w["logits"] <= 2e-2 and w["cache"] <= 2e-2, w


def test_half_small_bf16_isolated_groups():
    """The half-cache small model (L16 D512 k8, vocab 151936) in bf16: three
    cyclic passes with g = 16, every group compared from the GPU snapshot."""
    s = synth.HALF_SMALL
    m, Wn = model(s, seed=0, jitter=0.1)
    B, T, g = 2, 96, 16
    tokens = host(synth.make_tokens(s, B, T, seed=1)).astype(np.int64)
    w = isolated_passes(m, Wn, tokens, g, 3, logits_mode="last", spread=True)
    tol = TOL["bf16"]
    assert w["checked"] == 48
    assert within(w["logits"], tol["logits"], w["spread_logits"], "logits"), w
    assert within(w["cache"], tol["cache_step"], w["spread_cache"], "cache"), w
    assert within(w["cache_norm"], tol["cache_step_norm"], w["spread_cache_norm"], "cache_norm"), w


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_multi_tile_groups_isolated(dtype):
    """Groups of 320 rows (three 128-row tiles and a ragged tail), with the
    full-cache small model's channel count."""
    s = synth.FULL_SMALL.replace(V=1000, dtype=dtype)
    m, Wn = model(s, seed=3, jitter=0.1)
    B, T, g = 8, 160, 4
    tokens = np.random.default_rng(4).integers(0, s.V, size=(B, T))
    w = isolated_passes(m, Wn, tokens, g, 2, logits_mode="last",
                        check=lambda n, q: (n, q) in ((0, 0), (1, 2), (1, 3)),
                        spread=dtype == "bf16")
    tol = TOL[dtype]
    assert w["checked"] == 3
    assert within(w["logits"], tol["logits"], w["spread_logits"], "logits"), w
    assert within(w["cache"], tol["cache_step"], w["spread_cache"], "cache"), w
    assert within(w["cache_norm"], tol["cache_step_norm"], w["spread_cache_norm"], "cache_norm"), w


def test_large_groups_fp32_isolated():
    """Groups of 1,024 rows (the row norms switch to one warp per row from
    there), one pass, every group against the oracle from the GPU snapshot."""
    s = small_shape("f32", L=2, k=2)
    m, Wn = model(s, seed=6, jitter=0.1)
    B, T, g = 16, 128, 2
    tokens = np.random.default_rng(7).integers(0, s.V, size=(B, T))
    w = isolated_passes(m, Wn, tokens, g, 1, logits_mode="last")
    tol = TOL["f32"]
    assert w["checked"] == 2
    assert w["logits"] <= tol["logits"] and w["cache"] <= tol["cache"], w


@pytest.mark.parametrize("N", [300, 1000, 1500])
def test_pool_mix_multi_tile_bf16(N):
    s = synth.HALF_SMALL.replace(V=1000)
    m, Wn = model(s, seed=9, jitter=0.2)
    B, Tmax = 4, 512
    rng = np.random.default_rng(2)
    flat = rng.choice(B * Tmax, size=N, replace=False)
    seq_h, pos_h = flat // Tmax, flat % Tmax
    states = synth.make_normal((N, s.L, s.D), 31, "cuda", 1.0, s.torch_dtype)
    seq = torch.tensor(seq_h, dtype=torch.int32, device="cuda")
    pos = torch.tensor(pos_h, dtype=torch.int32, device="cuda")
    ck, cv = m.new_cache(B, Tmax, fill=float("nan"))
    coeff = torch.empty((N, 2, s.k, s.L), dtype=torch.float32, device="cuda")
    mixed = torch.empty((2, s.k, N, s.D), dtype=s.torch_dtype, device="cuda")
    ws = m.workspace(N, Tmax)
    wm.wm_pool_mix(m, states, seq, pos, ck, cv, ws, coeff_out=coeff, mixed_out=mixed)
    torch.cuda.synchronize()
    ref = O.pool(ocfg(s), Wn, host(states), pos_h)
    record(f"pool_mix_multi_tile_bf16[N={N}]", coeff=relerr(host(coeff), ref["coeff"]),
           mixed=relerr(host(mixed).transpose(2, 0, 1, 3), ref["mixed"]),
           K=relerr(host(ck)[seq_h, :, :, pos_h, :], ref["K"]),
           V=relerr(host(cv)[seq_h, :, :, pos_h, :], ref["V"]))
    assert relerr(host(coeff), ref["coeff"]) <= 2e-2
    assert relerr(host(mixed).transpose(2, 0, 1, 3), ref["mixed"]) <= 1e-2
    K = host(ck)
    assert np.array_equal(~np.isnan(K).any(axis=(1, 2, 4)),
                          np.isin(np.arange(B * Tmax), flat).reshape(B, Tmax))
    assert relerr(K[seq_h, :, :, pos_h, :], ref["K"]) <= 2e-2
    assert relerr(host(cv)[seq_h, :, :, pos_h, :], ref["V"]) <= 2e-2
