"""Plant plausible mistakes in the CPU oracle and check that the pins catch
each one. A mutant replaces one oracle function by a copy of its source with
one edit (a dropped term, a wrong sign, index or order); the pin suite must
then fail somewhere. This is how the pins are shown to be strong enough."""

import inspect

import numpy as np
import pytest

import oracle.whitematter as O
from tests import oracle_pins

MUTANTS = [
    # (id, function, old text, new text)
    ("rope_sign", "rope", "x1 * c - x2 * s", "x1 * c + x2 * s"),
    ("rope_theta", "rope", "-2.0 * np.arange", "-1.0 * np.arange"),
    ("rope_pairing", "rope", "half = d // 2", "half = d // 2 - 1 if d > 2 else 1"),
    ("rmsnorm_eps", "rmsnorm", "np.sqrt(ms + eps)", "(np.sqrt(ms) + eps)"),
    ("rmsnorm_sum", "rmsnorm", "np.mean(x * x, axis=-1", "np.sum(x * x, axis=-1"),
    ("silu_sigmoid", "silu", "return x / (1.0 + np.exp(-x))", "return 1.0 / (1.0 + np.exp(-x))"),
    ("router_offset", "router_sources", "l % cfg.p == cfg.p_offset", "l % cfg.p == (cfg.p_offset + 1) % cfg.p"),
    ("channel_shift", "channel_of_layer", "return l % cfg.k", "return (l + 1) % cfg.k"),
    ("groups_contiguous", "group_positions", "np.arange(q, T, g, dtype=np.int64)",
     "np.arange(q * -(-T // g), min(T, (q + 1) * -(-T // g)), dtype=np.int64)"),
    ("attn_self_visible", "channel_attention", "    if n_keys <= 0:\n        return out",
     "    n_keys = n_keys + 1\n    if n_keys <= 0:\n        return out"),
    ("attn_gqa_modulo", "channel_attention", "hk = (h * Hkv) // Hq", "hk = h % Hkv"),
    ("attn_no_scale", "channel_attention", "z = keys @ q[h] / math.sqrt(d)", "z = keys @ q[h]"),
    ("layer_no_attn_residual", "consumer_layer", "_st(cfg, h + o.reshape", "_st(cfg, 0.0 * h + o.reshape"),
    ("layer_swap_gate_up", "consumer_layer", "silu(gate) * up", "silu(up) * gate"),
    ("layer_no_qnorm", "consumer_layer", 'q = rmsnorm(q, W["q_norm"][l], cfg.eps)', 'q = q * _f64(W["q_norm"][l])'),
    ("layer_no_q_rope", "consumer_layer", "q = _st(cfg, rope(q, _f64(pos)[:, None], cfg.rope_base))", "q = _st(cfg, q)"),
    ("pool_coeff_transposed", "pool", "reshape(N, k, L)", "reshape(N, L, k).transpose(0, 2, 1)"),
    ("pool_router_raw_states", "pool", "x = _st(cfg, n[:, R, :]", "x = _st(cfg, states[:, R, :]"),
    ("pool_mix_raw_states", "pool", 'np.einsum("njl,nld->njd", a, n)', 'np.einsum("njl,nld->njd", a, states)'),
    ("pool_no_channel_norm", "pool", 'mixed[:, beta] = _st(cfg, rmsnorm(m, W["chan_norm"][beta], cfg.eps))',
     'mixed[:, beta] = _st(cfg, m * _f64(W["chan_norm"][beta]))'),
    ("pool_knorm_after_rope", "pool",
     'kt = rmsnorm(kt, W["k_norm"][j], cfg.eps)\n        K[:, j] = _st(cfg, rope(kt, _f64(pos)[:, None], cfg.rope_base))',
     'kt = rope(kt, _f64(pos)[:, None], cfg.rope_base)\n        K[:, j] = _st(cfg, rmsnorm(kt, W["k_norm"][j], cfg.eps))'),
    ("pool_v_uses_wk", "pool", 'W["Wv"][j]', 'W["Wk"][j]'),
    ("pool_gained_scale_no_eps", "pool", "np.mean(m * m, axis=-1) + cfg.eps)", "np.mean(m * m, axis=-1))"),
    ("pool_gained_scale_sum", "pool", "np.mean(m * m, axis=-1)", "np.sum(m * m, axis=-1)"),
    ("pool_gained_no_tau", "pool", 'stored[:, beta] = _st(cfg, m * _f64(W["chan_norm"][beta]))',
     'stored[:, beta] = _st(cfg, m)'),
    ("pool_gained_scale_branch", "pool", "* scale[:, 1, j, None]", "* scale[:, 0, j, None]"),
    ("bwd_rms_no_cross_term", "rmsnorm_backward", "dx = g / r - x * np.sum(g * x, axis=-1, keepdims=True) / (n * r ** 3)",
     "dx = g / r"),
    ("bwd_rope_forward_rotation", "pool_backward", "rope(dK[:, j], -_f64(pos)[:, None]", "rope(dK[:, j], _f64(pos)[:, None]"),
    ("bwd_no_router_to_states", "pool_backward", "dn[:, R, :] += (daf @", "dn[:, R, :] -= 0 * (daf @"),
    ("bwd_mix_transposed", "pool_backward", 'dn = np.einsum("njl,njd->nld", a, dm)', 'dn = np.einsum("njl,njd->nld", a[:, ::-1], dm)'),
    ("bwd_branch_grads_overwrite", "pool_backward", 'g["dstates"] += dh', 'g["dstates"] = dh'),
    ("batch_shared_position", "decode_batch", "pos = np.asarray(pos, dtype=np.int64)",
     "pos = np.full(len(pos), int(np.max(pos)), dtype=np.int64)"),
    ("batch_sequences_swapped", "decode_batch", "seq = np.arange(B)", "seq = np.arange(B)[::-1].copy()"),
    ("ff_router_rows_shifted", "feedback_free_channel", "[l * L: l * L + l + 1, : len(Rl) * D]",
     "[l * L + 1: l * L + l + 2, : len(Rl) * D]"),
    ("ff_router_all_rows_of_channel", "feedback_free_channel", "Rl = [s for s in router_sources(cfg) if s <= l]",
     "Rl = [s for s in router_sources(cfg) if s <= max(l, 1)]"),
    ("ff_static_transposed", "feedback_free_channel", "static_coeff)[beta, l, : l + 1]",
     "static_coeff)[beta, : l + 1, l]"),
    ("ff_cache_after_layer", "feedback_free_pass",
     """        K, V, _ = feedback_free_channel(cfg, W, states[:, : l + 1], pos, l, static_coeff)
        for r in range(B * T):
            cache_k[seq[r], l, :, pos[r], :] = K[r]
            cache_v[seq[r], l, :, pos[r], :] = V[r]
        h = consumer_layer(cfg, W, l, h, seq, pos, cache_k, cache_v)""",
     """        K, V, _ = feedback_free_channel(cfg, W, states[:, : l + 1], pos, l, static_coeff)
        h = consumer_layer(cfg, W, l, h, seq, pos, cache_k, cache_v)
        for r in range(B * T):
            cache_k[seq[r], l, :, pos[r], :] = K[r]
            cache_v[seq[r], l, :, pos[r], :] = V[r]"""),
    ("ff_no_prefix_states", "feedback_free_pass", "states[:, : l + 1], pos, l, static_coeff)",
     "states[:, : max(l, 1)], pos, max(l - 1, 0), static_coeff)"),
    ("pool_router_one_branch", "pool", '(x @ _f64(W["Wr"][beta]).T).reshape(N, k, L)',
     '(x @ _f64(W["Wr"][0]).T).reshape(N, k, L)'),
    ("pool_channels_share_wk", "pool", '(stored[:, 0, j] @ _f64(W["Wk"][j]).T)',
     '(stored[:, 0, j] @ _f64(W["Wk"][0]).T)'),
    ("residual_key_branch_only", "kv_residual",
     "num = np.sum((_f64(cur_k) - _f64(prev_k)) ** 2) + np.sum((_f64(cur_v) - _f64(prev_v)) ** 2)",
     "num = np.sum((_f64(cur_k) - _f64(prev_k)) ** 2)"),
    ("pool_shared_src_norm", "pool", 'n = rmsnorm(states, W["src_norm"][beta], cfg.eps)',
     'n = rmsnorm(states, W["src_norm"][0], cfg.eps)'),
    ("states_are_outputs", "run_rows", "        states[:, l] = h\n        h = consumer_layer(cfg, W, l, h, seq, pos, cache_k, cache_v)",
     "        h = consumer_layer(cfg, W, l, h, seq, pos, cache_k, cache_v)\n        states[:, l] = h"),
    ("write_shifted", "_write", "cache_k[int(seq[r]), :, :, int(pos[r]), :] = K[r]",
     "cache_k[int(seq[r]), :, :, (int(pos[r]) + 1) % cache_k.shape[3], :] = K[r]"),
    ("groups_reversed", "cyclic_pass", "for q in range(q_begin, q_end):", "for q in reversed(range(q_begin, q_end)):"),
    ("bf16_truncates", "round_bf16", "u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000", "u = u & 0xFFFF0000"),
    ("bf16_ties_away", "round_bf16", "u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000", "u = (u + 0x8000) & 0xFFFF0000"),
    ("storage_ignored", "_st", 'if getattr(cfg, "storage", None) == "bf16":', "if False:"),
    ("decode_sees_self", "decode_step", "pos = np.full(B, t, dtype=np.int64)", "pos = np.full(B, t + 1, dtype=np.int64)"),
]


def _no_snapshot_cyclic_pass(cfg, W, tokens, g, cache_k, cache_v, q_begin=0, q_end=None,
                             logits=None, static_coeff=None):
    """Mutant: rows of a group are run one at a time and written immediately,
    so later rows of the same group see earlier rows' updates."""
    tokens = np.asarray(tokens, dtype=np.int64)
    B, T = tokens.shape
    q_end = g if q_end is None else q_end
    out = np.zeros((B, T, cfg.V)) if logits == "all" else (np.zeros((B, cfg.V)) if logits == "last" else None)
    for q in range(q_begin, q_end):
        for i in O.group_positions(T, g, q):
            for b in range(B):
                res, lg, _ = O.run_rows(cfg, W, tokens[b:b + 1, i], [b], [i], cache_k, cache_v,
                                        logits is not None, static_coeff)
                O._write(cache_k, cache_v, [b], [i], res["K"], res["V"])
                if logits == "all":
                    out[b, i] = lg[0]
                elif logits == "last" and i == T - 1:
                    out[b] = lg[0]
    return out


def _mutant(fname, old, new):
    src = inspect.getsource(getattr(O, fname))
    assert old in src, f"mutation text not found in {fname}"
    ns = {}
    exec(compile(src.replace(old, new, 1), f"<mutant of {fname}>", "exec"), O.__dict__, ns)
    return ns[fname]


def _caught():
    for check in oracle_pins.ALL_CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(O)
        except Exception:          # AssertionError, or the mutant crashing
            return check.__name__
    return None


@pytest.mark.parametrize("mut", MUTANTS, ids=lambda m: m[0])
def test_mutant_is_caught(mut, monkeypatch):
    _, fname, old, new = mut
    monkeypatch.setattr(O, fname, _mutant(fname, old, new))
    assert _caught() is not None, f"no pin caught mutant {mut[0]}"


def test_snapshot_violation_is_caught(monkeypatch):
    monkeypatch.setattr(O, "cyclic_pass", _no_snapshot_cyclic_pass)
    assert _caught() is not None
