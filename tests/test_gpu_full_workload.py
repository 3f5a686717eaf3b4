"""The prefill workload at its full size and in the launch configuration the
benchmark times: the 1.3B model (L = 28, D = 1792, k = 14, Hq = 14, Hkv = 2,
d = 128, F = 4608, V = 151936), 64 sequences of 2,048 tokens, g = 16, one
group of 8,192 rows through wm_cyclic_pass from a random cache.

The oracle cannot run 8,192 rows of a 28-layer stack in a test, but rows of
one group do not interact: each reads the cache as it stood before the group
("WhiteMatter: All-to-All Cross-Layer Connections via KV Mixing", 3 METHOD,
"How it differs"). So sampled rows are computed one by one by the oracle from
the same snapshot, and every other row is held to properties that hold at any
size (exactly the group's positions written, all of them finite)."""

import numpy as np
import pytest
import torch

import oracle.whitematter as O
from cross_layer_kv_pool_b300 import synth, wm
from tests.gpu_util import (SPREAD_EPS, TOL, ensure_lib, host, normerr, ocfg, relerr, within)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _oracle_weights(W, toks, vocab_rows, eps=0.0, seed=12345):
    """fp32 host copies (exact for bf16 values) with the embedding cut to the
    sampled tokens' rows (token r of the sample becomes id r) and the LM head
    to ``vocab_rows``. With eps > 0 every weight gets an independent relative
    perturbation of that size (the oracle's own conditioning)."""
    rng = np.random.default_rng(seed)
    out = {}
    for n, t in W.items():
        if n == "embed":
            t = t[torch.as_tensor(toks, device=t.device)]
        elif n == "lm_head":
            t = t[torch.as_tensor(vocab_rows, device=t.device)]
        v = t.float().cpu().numpy()
        if eps:
            v = (v * (1.0 + eps * rng.standard_normal(v.shape, dtype=np.float32))).astype(np.float32)
        out[n] = v
    return out


def _random_cache(m, B, Tmax, seed):
    ck, cv = m.new_cache(B, Tmax)
    ck.copy_(synth.make_normal(tuple(ck.shape), seed, "cuda", 1.0, torch.bfloat16))
    cv.copy_(synth.make_normal(tuple(cv.shape), seed + 1, "cuda", 1.0, torch.bfloat16))
    return ck, cv


def test_full_prefill_group_sampled_rows():
    s = synth.HALF_1P3B
    W = synth.make_weights(s, seed=0, device="cuda", gain_jitter=0.1)
    m = wm.Model(s, W)
    B, T, g, q = 64, 2048, 16, 15
    tok = synth.make_tokens(s, B, T, seed=1, device="cuda")
    ck, cv = _random_cache(m, B, T, 4)
    samples = [(0, 15), (29, 1039), (41, 1535), (63, 2047)]  # positions of group q
    seqs = [b for b, _ in samples]
    pos = np.array([p for _, p in samples])
    assert all(p % g == q for p in pos)
    snap_k, snap_v = host(ck[seqs]), host(cv[seqs])
    ws = m.workspace(wm.rows_for_pass(B, T, g), T)
    lg = torch.zeros((B, s.V), dtype=torch.float32, device="cuda")
    wm.wm_cyclic_pass(m, tok, g, ck, cv, ws, q_begin=q, q_end=q + 1, logits=lg, logits_mode="last")
    torch.cuda.synchronize()
    assert wm.wm_check_flags(ws) == 0

    # every row: exactly the group's positions written, all finite
    k0, v0 = _random_cache(m, B, T, 4)
    P = torch.arange(q, T, g, device="cuda")
    other = torch.ones(T, dtype=torch.bool, device="cuda")
    other[P] = False
    assert torch.equal(ck[:, :, :, other], k0[:, :, :, other])
    assert torch.equal(cv[:, :, :, other], v0[:, :, :, other])
    assert not torch.equal(ck[:, :, :, P], k0[:, :, :, P])
    assert torch.isfinite(ck[:, :, :, P].float()).all() and torch.isfinite(cv[:, :, :, P].float()).all()
    assert torch.isfinite(lg).all()
    del k0, v0

    # sampled rows against the oracle from the same snapshot
    toks_h = host(tok).astype(np.int64)
    row_toks = [int(toks_h[b, p]) for b, p in samples]
    vocab = np.arange(0, s.V, 37)
    oc = ocfg(s)
    rows = np.arange(len(samples))
    res, lo, _ = O.run_rows(oc, _oracle_weights(W, row_toks, vocab), rows, rows, pos, snap_k, snap_v,
                            want_logits=True)
    rp, lp, _ = O.run_rows(oc, _oracle_weights(W, row_toks, vocab, eps=SPREAD_EPS), rows, rows, pos,
                           snap_k, snap_v, want_logits=True)
    gk, gv = host(ck[seqs]), host(cv[seqs])
    got = np.stack([gk[rows, :, :, pos], gv[rows, :, :, pos]])
    ref = np.stack([res["K"], res["V"]])
    per = np.stack([rp["K"], rp["V"]])
    tol = TOL["bf16"]
    assert within(relerr(got, ref), tol["cache_step"], relerr(per, ref), "cache"), (relerr(got, ref), relerr(per, ref))
    assert within(normerr(got, ref), tol["cache_step_norm"], normerr(per, ref), "cache_norm"), \
        (normerr(got, ref), normerr(per, ref))
    last = pos == T - 1
    got_l = host(lg)[np.array(seqs)[last]][:, vocab]
    assert within(relerr(got_l, lo[last]), tol["logits"], relerr(lp[last], lo[last]), "logits"), \
        (relerr(got_l, lo[last]), relerr(lp[last], lo[last]))

