"""Helpers shared by the GPU parity tests (inputs, tolerances, comparisons)."""

from __future__ import annotations

import dataclasses
from types import SimpleNamespace

import numpy as np
import torch

from cross_layer_kv_pool_b300 import build, synth, wm

# Tolerances, max|gpu - ref| / max|ref| per tensor: 1e-4 in fp32 mode; in bf16
# mode 2e-2 on logits, 1e-2 on the mixed channels and on a single attention
# call, 2e-2 on K/V written from identical states. Cache entries written by a
# whole bf16 group step of a deep stack (8+ layers) use ``cache_step``: the
# oracle in bf16-storage mode, run against itself with weights perturbed by
# 1e-7..1e-5 (the scale of fp32-vs-fp64 arithmetic), already differs by
# 2.5-3.8% max-element and 1.0-1.6% in norm on those entries, because single
# bf16 rounding flips are amplified by the signed mixing. Whole bf16 group
# steps are therefore also allowed SPREAD_FACTOR times the oracle's own spread
# on the same instance (``within``), measured in the test itself.
TOL = {"f32": dict(logits=1e-4, cache=1e-4, mixed=1e-4, coeff=1e-4, attn=1e-4,
                   cache_step=1e-4, cache_step_norm=1e-4),
       "bf16": dict(logits=2e-2, cache=2e-2, mixed=1e-2, coeff=2e-2, attn=1e-2,
                    cache_step=1e-1, cache_step_norm=3e-2)}


def record(test: str, **vals):
    """Print the measured errors of one parity check and, when the
    environment variable WM_PARITY_LOG names a file, append them to it as one
    JSON line (the record of what each bf16 comparison achieved)."""
    import json
    import os
    line = json.dumps({"test": test, **{k: (float(v) if isinstance(v, (float, np.floating)) else v)
                                        for k, v in vals.items()}})
    print("parity", line)
    path = os.environ.get("WM_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(line + "\n")


def normerr(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def ensure_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    return wm.lib()


def relerr(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.max(np.abs(b))
    return float(np.max(np.abs(a - b)) / den) if den > 0 else float(np.max(np.abs(a)))


def host(t) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def model(shape, seed=0, jitter=0.1, static=None, flags=0):
    W = synth.make_weights(shape, seed=seed, device="cuda", gain_jitter=jitter)
    return wm.Model(shape, W, static_coeff=static, flags=flags), synth.to_numpy_weights(W)


def ocfg(shape):
    """The oracle's view of a model: bf16 workloads use its bf16-storage mode
    (activations rounded where a bf16 pipeline stores them), fp32 workloads
    the plain fp64 arithmetic. The bf16 pipeline's mixer stores the gained
    channel tau (.) m and leaves the norm factor to the K/V projection, so the
    oracle rounds at that tensor too (reading R17; every bf16 test shape is
    inside that mixer's envelope: k <= 16, L <= 64, D/32 divisible into
    slices of at most 14 warps)."""
    ns = SimpleNamespace(**dataclasses.asdict(shape))
    ns.nR = shape.nR
    if shape.dtype == "bf16":
        ns.storage = "bf16"
        ns.mixed_storage = "gained"
    return ns


def small_shape(dtype="f32", **kw):
    base = dict(L=4, D=128, k=2, p=2, Hq=4, Hkv=2, d=64, F=256, V=512, dtype=dtype)
    base.update(kw)
    return synth.ModelShape(**base)


def perturbed(Wn, eps, seed=12345):
    """Weights with independent relative perturbations of size eps: the
    oracle run on them measures how far the instance itself moves under
    arithmetic-level differences (its conditioning)."""
    rng = np.random.default_rng(seed)
    return {k: v * (1.0 + eps * rng.standard_normal(v.shape)) for k, v in Wn.items()}


SPREAD_EPS = 1e-5     # relative size of fp32-vs-fp64 differences in long reductions
SPREAD_FACTOR = 2.5   # a widened check allows this many times the oracle's own spread

# Whole-step bf16 comparisons for which the fixed bound is not attainable: the
# oracle against itself, with its weights perturbed by SPREAD_EPS, already
# moves the quantity by about the bound or more (random-weight models amplify
# single bf16 rounding flips through the signed mixing and the depth of the
# stack). Only these (test, quantity) pairs may use max(bound, SPREAD_FACTOR x
# spread); every other comparison is held to its fixed bound. The recorded
# numbers (max-element error / oracle spread, B300) that justify each entry:
WIDENED = {
    ("test_full_prefill_group_sampled_rows", "logits"): "3.70e-2 / 3.84e-2",
    ("test_full_prefill_group_sampled_rows", "cache_norm"): "3.71e-2 / 3.58e-2 (norm)",
    ("test_multi_tile_groups_isolated", "logits"): "2.57e-2 / 2.69e-2",
    ("test_decode_batch_1p3b_widths_ragged", "cache"): "2.73e-2 / 4.75e-2",
    ("test_decode_1p3b_widths_isolated", "cache"): "3.29e-2 / 4.13e-2",
    ("test_decode_long_context_isolated", "cache"): "2.17e-2 / 4.55e-2",
    ("test_uneven_groups_isolated", "cache"): "2.02e-2 / 3.23e-2",
    ("test_cyclic_pass_rank_bf16_isolated", "logits"): "2.00e-2 / (spread first recorded here)",
}


def within(err, base, spread, what=""):
    """The fixed bound ``base``, or, for the (test, quantity) pairs listed in
    WIDENED only, max(base, SPREAD_FACTOR x the oracle's measured spread).
    Records the error, the spread and whether the fixed bound alone held."""
    import os
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    name = test.split("::")[-1].split("[")[0]
    widened = (name, what) in WIDENED
    record(test, what=what, err=err, base=base, spread=spread, fixed_ok=bool(err <= base),
           widened=widened)
    return err <= (max(base, SPREAD_FACTOR * spread) if widened else base)


def isolated_passes(m, Wn, tokens_h, g, passes, Tmax=None, logits_mode="last", check=None,
                    spread=False, static=None, oc=None):
    """Run ``passes`` cyclic passes on the GPU one group at a time. Before each
    checked group (``check(n, q)``), copy the GPU cache to the host, run the
    oracle's same group from that snapshot, and compare what the group wrote
    (its cache positions and logits). Returns the worst relative errors.

    Comparing step by step gives both sides identical inputs at every group,
    which whole-sequence comparison cannot: the random-weight models amplify
    any bf16-level difference along the sequence (see the design notes)."""
    import oracle.whitematter as O
    s = m.shape
    oc = oc or ocfg(s)
    B, T = tokens_h.shape
    Tmax = Tmax or T
    tok = torch.tensor(tokens_h, dtype=torch.int32, device="cuda")
    ck, cv = m.new_cache(B, Tmax)
    ws = m.workspace(wm.rows_for_pass(B, T, g), Tmax)
    lg = torch.zeros((B, T, s.V) if logits_mode == "all" else (B, s.V), dtype=torch.float32,
                     device="cuda")
    worst = {"cache": 0.0, "cache_norm": 0.0, "logits": 0.0, "checked": 0,
             "spread_cache": 0.0, "spread_cache_norm": 0.0, "spread_logits": 0.0}
    Wp = perturbed(Wn, SPREAD_EPS) if spread else None
    for n in range(passes):
        mode = logits_mode if n == passes - 1 else "none"
        for q in range(g):
            do = check is None or check(n, q)
            if do:
                torch.cuda.synchronize()
                sk, sv = host(ck), host(cv)
                pk, pv = sk.copy(), sv.copy()
            wm.wm_cyclic_pass(m, tok, g, ck, cv, ws, q_begin=q, q_end=q + 1,
                              logits=None if mode == "none" else lg, logits_mode=mode)
            if not do:
                continue
            torch.cuda.synchronize()
            rl = O.cyclic_pass(oc, Wn, tokens_h, g, sk, sv, q_begin=q, q_end=q + 1,
                               logits=None if mode == "none" else mode, static_coeff=static)
            P = np.arange(q, T, g)
            gk, gv = host(ck), host(cv)
            if spread:
                pl = O.cyclic_pass(oc, Wp, tokens_h, g, pk, pv, q_begin=q, q_end=q + 1,
                                   logits=None if mode == "none" else mode, static_coeff=static)
                worst["spread_cache"] = max(worst["spread_cache"],
                                            relerr(pk[:, :, :, P], sk[:, :, :, P]),
                                            relerr(pv[:, :, :, P], sv[:, :, :, P]))
                worst["spread_cache_norm"] = max(worst["spread_cache_norm"],
                                                 normerr(pk[:, :, :, P], sk[:, :, :, P]),
                                                 normerr(pv[:, :, :, P], sv[:, :, :, P]))
                if mode == "all":
                    worst["spread_logits"] = max(worst["spread_logits"], relerr(pl[:, P], rl[:, P]))
                elif mode == "last" and (T - 1) % g == q:
                    worst["spread_logits"] = max(worst["spread_logits"], relerr(pl, rl))
            worst["cache"] = max(worst["cache"], relerr(gk[:, :, :, P], sk[:, :, :, P]),
                                 relerr(gv[:, :, :, P], sv[:, :, :, P]))
            worst["cache_norm"] = max(worst["cache_norm"], normerr(gk[:, :, :, P], sk[:, :, :, P]),
                                      normerr(gv[:, :, :, P], sv[:, :, :, P]))
            if mode == "all":
                worst["logits"] = max(worst["logits"], relerr(host(lg)[:, P], rl[:, P]))
            elif mode == "last" and (T - 1) % g == q:
                worst["logits"] = max(worst["logits"], relerr(host(lg), rl))
            worst["checked"] += 1
    assert wm.wm_check_flags(ws) == 0
    return worst


def isolated_decode(m, Wn, tokens_h, Tmax, start_cache=None, start_pos=0, spread=False):
    """Decode steps t = 0..T-1 on the GPU; each step is compared with the
    oracle's step from the GPU's cache snapshot. Returns worst errors."""
    import oracle.whitematter as O
    s = m.shape
    oc = ocfg(s)
    B, T = tokens_h.shape
    ck, cv = m.new_cache(B, Tmax) if start_cache is None else start_cache
    ws = m.workspace(B, Tmax)
    lg = torch.zeros((B, s.V), dtype=torch.float32, device="cuda")
    tok = torch.tensor(tokens_h, dtype=torch.int32, device="cuda")
    worst = {"cache": 0.0, "logits": 0.0, "spread_cache": 0.0, "spread_logits": 0.0}
    Wp = perturbed(Wn, SPREAD_EPS) if spread else None
    for i in range(T):
        t = start_pos + i
        torch.cuda.synchronize()
        sk, sv = host(ck), host(cv)
        wm.wm_decode_step(m, tok[:, i].contiguous(), t, ck, cv, lg, ws)
        torch.cuda.synchronize()
        if spread:
            pk, pv = sk.copy(), sv.copy()
        rl = O.decode_step(oc, Wn, tokens_h[:, i], t, sk, sv)
        if spread:
            pl = O.decode_step(oc, Wp, tokens_h[:, i], t, pk, pv)
            worst["spread_logits"] = max(worst["spread_logits"], relerr(pl, rl))
            worst["spread_cache"] = max(worst["spread_cache"], relerr(pk[:, :, :, t], sk[:, :, :, t]),
                                        relerr(pv[:, :, :, t], sv[:, :, :, t]))
        worst["logits"] = max(worst["logits"], relerr(host(lg), rl))
        worst["cache"] = max(worst["cache"], relerr(host(ck)[:, :, :, t], sk[:, :, :, t]),
                             relerr(host(cv)[:, :, :, t], sv[:, :, :, t]))
    assert wm.wm_check_flags(ws) == 0
    return worst
