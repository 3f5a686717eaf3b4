"""WhiteMatter cross-layer KV pool: plain, slow CPU oracle in fp64 NumPy.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run this module. It shares no
code with the CUDA implementation and imports nothing from it.

What is computed, and where the pages say so. The sources are public pages
about arXiv 2608.18486 ("WhiteMatter: All-to-All Cross-Layer Connections via
KV Mixing", Zhang & Ren); they are cited by tag and section:

  [PL]  paperlayer.ai summary, "WhiteMatter: All-to-All Cross-Layer
        Connections via KV Mixing"; sections "3 METHOD", "5 ANALYSIS".
  [OD]  onedev.kr review, "WhiteMatter가 모든 층의 KV 재사용으로 캐시를 절반으로
        줄인다"; sections "How it works" (어떻게 동작하나), "How it differs"
        (무엇과 다른가), "How it is used" (어떻게 쓰나).

  * Each consumer layer has no K/V projection of its own; K/V come from a
    cross-layer pool of k <= L channels ([PL 3 METHOD, opening paragraph];
    [OD How it works]).
  * Pool, per token and per branch beta in {K, V} with separate parameters
    ([OD How it works]; [PL 3 METHOD, "Cross-layer KV pool"]):
      n^{b,l} = RMSNorm(h^l; sigma^b_l)                 for l < L
      a^b     = W_R^b . concat_{l in R} n^{b,l}, viewed [k, L]  (signed, no
                softmax; R = every p-th source state)
      m^b_j   = sum_l a^b_{j,l} n^{b,l}
      c^b_j   = RMSNorm(m^b_j; tau^b_j)
      K_j     = RoPE_i(RMSNorm_d(W_K^j c^K_j per head; kappa_j)),  V_j = W_V^j c^V_j
  * Consumer layer l reads channel l mod k ([PL 3 METHOD, "Per-layer channel
    selection"]); attention is strictly causal, token i sees s < i, and a
    token's channels are appended only after its whole layer stack
    ([OD How it differs]; [PL 3 METHOD, "Execution schedules"]).
  * Prefill solves KV = Model(X; KV). Cyclic Gauss-Seidel: groups
    G_q = {i : i mod g = q} in order q = 0..g-1, parallel inside a group, the
    cache updated after each group ([OD How it differs]). Jacobi is g = 1.
  * Decoder layers are Qwen3-style ([OD How it is used]).

Readings where the pages are silent (each listed again in the design notes):
  R1  R = {l < L : l mod p == p_offset}, p_offset = 0 by default.
  R2  The L source states are the residual-stream INPUTS of layers 0..L-1;
      h^0 is the token embedding; h^L feeds only the final norm + LM head.
  R3  The router is one bias-free linear map per branch, |R|*D -> k*L,
      output index j*L + l.
  R4  The router reads the branch's own source-normed states n^{b,l}.
  R5  Source-norm gains are separate per (branch, source layer).
  R6  Queries: Qwen3-style per-head q-norm (gain [d] per layer) then RoPE.
  R7  Query head h reads KV head floor(h*Hkv/Hq); scale 1/sqrt(d).
  R8  K-norm: RMSNorm over d per KV head with gain kappa_j [d] per channel,
      before RoPE. Values are stored raw.
  R9  A token with no visible keys (i = 0) gets attention output 0.
  R10 The cache starts at zero; unwritten positions are read as zeros.
  R11 Groups run q = 0..g-1 every pass; any 1 <= g <= T is allowed.
  R13 RMSNorm eps = 1e-6; RoPE rotate-half, theta_t = base^(-2t/d).
  R14 bf16 storage. The pages run the 1.3B model in BF16 ([OD "Assumptions
      and limits" (전제와 한계): RTX A6000, BF16]). With ``cfg.storage ==
      "bf16"`` the oracle rounds (to nearest even) every tensor that a bf16
      pipeline stores between operations: normalised GEMM inputs, queries,
      attention outputs, residual-stream states, the SwiGLU activation, the
      router input, the mixed channels and the cached K/V. Arithmetic between
      those points stays fp64; router coefficients and logits stay unrounded.
      Without ``storage`` (the default) nothing is rounded.
  R17 Where the mixed channel is stored. c = RMSNorm(m; tau) feeds only the
      linear K/V projection, so W c = s * W (tau (.) m) with the scalar
      s = rsqrt(mean(m^2) + eps). ``cfg.mixed_storage == "gained"`` models a
      pipeline that stores u = tau (.) m and applies s to the projection
      output; the default "normed" stores c. In exact arithmetic the two are
      the same function (pinned); they differ only in which tensor bf16
      storage rounds, and ``mixed`` is then bf16(s * u).
  R18 The feedback-free variant ([PL 5 ANALYSIS, "Deep-to-shallow feedback":
      a 16-channel cache for 16 layers, costs like vanilla, no iteration) has
      k = L and builds channel l from the token's states h^0..h^l only: the
      router reads the sources of R inside 0..l (its other inputs unused)
      through rows l*L + 0..l of W_R (or static_coeff[b][l][0..l]); the
      channel is cached before layer l runs; layer l still attends to s < i.
  R19 Decode with sequences at different positions (continuous batching):
      the pages decode every sequence at the same step; a batch in which
      sequence b sits at pos[b] is read as the per-sequence decode step at
      t = pos[b] for each b, with no interaction between sequences.

Parity pins for every function below live in tests/test_oracle_pins.py and
tests/test_oracle_mutants.py (closed forms, special cases, brute force and an
independently written vanilla strict-causal Transformer).
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "round_bf16", "rmsnorm", "rope", "silu", "router_sources", "channel_of_layer",
    "group_positions", "channel_attention", "consumer_layer", "pool",
    "run_rows", "new_cache", "cyclic_pass", "decode_step",
    "autoregressive", "kv_residual", "feedback_free_channel", "feedback_free_pass",
    "rmsnorm_backward", "pool_backward",
]


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def round_bf16(x):
    """Round to the nearest bfloat16 (ties to even), returned as fp64: first
    to fp32 (nearest), then the low 16 bits of the fp32 pattern are rounded."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def _st(cfg, x):
    """A stored activation: rounded to bf16 in bf16-storage mode (R14)."""
    if getattr(cfg, "storage", None) == "bf16":
        return round_bf16(x)
    return _f64(x)


# ----------------------------------------------------------------------------
# Elementwise building blocks
# ----------------------------------------------------------------------------

def rmsnorm(x, w, eps):
    """RMSNorm over the last axis: w * x / sqrt(mean(x^2) + eps).

    Used for every norm in the model: layer input/post norms (Qwen3 style,
    [OD How it is used]), the per-source norm and the per-channel norm of the
    pool ([OD How it works]), the q-norm (R6) and the K-norm (R8).
    """
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return _f64(w) * (x / np.sqrt(ms + eps))


def rope(x, pos, base):
    """Rotary embedding, rotate-half convention (R13).

    Pairs (t, t + d/2) for t < d/2 are rotated by angle pos * base^(-2t/d).
    ``pos`` broadcasts against ``x.shape[:-1]``. Keys are stored rotated
    ([PL 3 METHOD, "Cross-layer KV pool": stored keys are rotated]).
    """
    x = _f64(x)
    d = x.shape[-1]
    half = d // 2
    theta = float(base) ** (-2.0 * np.arange(half, dtype=np.float64) / d)
    ang = _f64(pos)[..., None] * theta
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x):
    """x * sigmoid(x), the SwiGLU gate activation of a Qwen3-style FFN."""
    x = _f64(x)
    return x / (1.0 + np.exp(-x))


# ----------------------------------------------------------------------------
# Indexing rules
# ----------------------------------------------------------------------------

def router_sources(cfg):
    """Source layers the router reads: every p-th state ([OD How it works];
    [PL 3 METHOD, "Cross-layer KV pool": the router may read every pth source
    layer]). Reading R1: l = p_offset, p_offset + p, ..."""
    return [l for l in range(cfg.L) if l % cfg.p == cfg.p_offset]


def channel_of_layer(cfg, l):
    """Consumer layer l reads channel l mod k ([PL 3 METHOD, "Per-layer channel
    selection"]; [OD How it works])."""
    return l % cfg.k


def group_positions(T, g, q):
    """G_q = {i : i mod g = q}, 0 <= i < T ([OD How it differs])."""
    return np.arange(q, T, g, dtype=np.int64)


# ----------------------------------------------------------------------------
# Channel attention
# ----------------------------------------------------------------------------

def channel_attention(q, K, V, n_keys, Hq, Hkv):
    """Strictly causal attention of one token to one cache channel.

    q: [Hq, d] (already q-normed and rotated); K, V: [Hkv, S, d] for the
    token's sequence and the layer's channel; the token at position i sees
    keys s < i, i.e. ``n_keys = i`` ([OD How it differs]). Query head h reads
    KV head floor(h*Hkv/Hq) (R7). With no visible key the output is 0 (R9).
    Returns [Hq, d].
    """
    q = _f64(q)
    d = q.shape[-1]
    out = np.zeros((Hq, d), dtype=np.float64)
    if n_keys <= 0:
        return out
    for h in range(Hq):
        hk = (h * Hkv) // Hq
        keys = _f64(K[hk, :n_keys, :])
        vals = _f64(V[hk, :n_keys, :])
        z = keys @ q[h] / math.sqrt(d)
        z = z - np.max(z)
        w = np.exp(z)
        w = w / np.sum(w)
        out[h] = w @ vals
    return out


# ----------------------------------------------------------------------------
# One consumer layer (Qwen3-style decoder layer without its own K/V)
# ----------------------------------------------------------------------------

def consumer_layer(cfg, W, l, h, seq, pos, cache_k, cache_v):
    """h^{l+1} = Layer_l(h^l) for a set of rows that all read one cache snapshot.

    h: [N, D] layer input; seq, pos: [N] batch row and absolute position of
    each row; cache_k/v: [B, k, Hkv, Tmax, d]. Structure (Qwen3-style,
    [OD How it is used]; reading R6/R7): pre-norm, Q projection, per-head
    q-norm, RoPE, attention to channel l mod k over s < pos, O projection and
    residual, post-norm, SwiGLU FFN and residual.
    """
    N = h.shape[0]
    Hq, Hkv, d = cfg.Hq, cfg.Hkv, cfg.d
    h = _f64(h)
    a = _st(cfg, rmsnorm(h, W["in_norm"][l], cfg.eps))
    q = (a @ _f64(W["Wq"][l]).T).reshape(N, Hq, d)
    q = rmsnorm(q, W["q_norm"][l], cfg.eps)
    q = _st(cfg, rope(q, _f64(pos)[:, None], cfg.rope_base))
    c = channel_of_layer(cfg, l)
    o = np.zeros((N, Hq, d), dtype=np.float64)
    for r in range(N):
        b = int(seq[r])
        o[r] = channel_attention(q[r], cache_k[b, c], cache_v[b, c], int(pos[r]), Hq, Hkv)
    o = _st(cfg, o)
    h2 = _st(cfg, h + o.reshape(N, Hq * d) @ _f64(W["Wo"][l]).T)
    f = _st(cfg, rmsnorm(h2, W["post_norm"][l], cfg.eps))
    gate = f @ _f64(W["Wgate"][l]).T
    up = f @ _f64(W["Wup"][l]).T
    act = _st(cfg, silu(gate) * up)
    return _st(cfg, h2 + act @ _f64(W["Wdown"][l]).T)


# ----------------------------------------------------------------------------
# The cross-layer KV pool
# ----------------------------------------------------------------------------

def pool(cfg, W, states, pos, static_coeff=None):
    """Mix one token's L layer states into k K/V channels.

    states: [N, L, D] (the inputs h^0..h^{L-1} of each row's layers, R2);
    pos: [N] absolute positions (for the key RoPE).
    Per branch beta (0 = K, 1 = V), following [OD How it works] and
    [PL 3 METHOD, "Cross-layer KV pool"]:
      n      = RMSNorm(states; sigma^beta)       per (row, source layer)
      a      = W_R^beta . concat_{l in R} n_l    -> [N, k, L]      (R3/R4)
      m_j    = sum_l a_{j,l} n_l                  -> [N, k, D]
      c_j    = RMSNorm(m_j; tau^beta_j)
    then K_j = RoPE(RMSNorm_d(W_K^j c^K_j per head; kappa_j)), V_j = W_V^j c^V_j.
    ``static_coeff`` ([2, k, L]) replaces the router output for every token:
    the static-mixing variant ([PL 5 ANALYSIS, "Dynamic routing"]) and the
    forced identity router of the k = L special case.
    Returns a dict with K, V [N, k, Hkv, d], coeff [N, 2, k, L] and
    mixed [N, 2, k, D] (the channel-normed c).
    """
    states = _f64(states)
    N, L, D = states.shape
    k, Hkv, d = cfg.k, cfg.Hkv, cfg.d
    R = router_sources(cfg)
    coeff = np.zeros((N, 2, k, L), dtype=np.float64)
    mixed = np.zeros((N, 2, k, D), dtype=np.float64)
    stored = np.zeros((N, 2, k, D), dtype=np.float64)  # projection input (R17)
    scale = np.ones((N, 2, k), dtype=np.float64)        # applied to its output
    for beta in range(2):
        n = rmsnorm(states, W["src_norm"][beta], cfg.eps)          # [N, L, D]
        if static_coeff is None:
            x = _st(cfg, n[:, R, :].reshape(N, len(R) * D))
            a = (x @ _f64(W["Wr"][beta]).T).reshape(N, k, L)
        else:
            a = np.broadcast_to(_f64(static_coeff)[beta], (N, k, L))
        m = np.einsum("njl,nld->njd", a, n)
        coeff[:, beta] = a
        mixed[:, beta] = _st(cfg, rmsnorm(m, W["chan_norm"][beta], cfg.eps))
        stored[:, beta] = mixed[:, beta]
        if getattr(cfg, "mixed_storage", "normed") == "gained":
            scale[:, beta] = 1.0 / np.sqrt(np.mean(m * m, axis=-1) + cfg.eps)
            stored[:, beta] = _st(cfg, m * _f64(W["chan_norm"][beta]))
            mixed[:, beta] = _st(cfg, stored[:, beta] * scale[:, beta, :, None])
    K = np.zeros((N, k, Hkv, d), dtype=np.float64)
    V = np.zeros((N, k, Hkv, d), dtype=np.float64)
    for j in range(k):
        kt = ((stored[:, 0, j] @ _f64(W["Wk"][j]).T) * scale[:, 0, j, None]).reshape(N, Hkv, d)
        kt = rmsnorm(kt, W["k_norm"][j], cfg.eps)
        K[:, j] = _st(cfg, rope(kt, _f64(pos)[:, None], cfg.rope_base))
        V[:, j] = _st(cfg, ((stored[:, 1, j] @ _f64(W["Wv"][j]).T) * scale[:, 1, j, None]).reshape(N, Hkv, d))
    return {"K": K, "V": V, "coeff": coeff, "mixed": mixed}


# ----------------------------------------------------------------------------
# Layer stack + pool for a set of rows sharing one cache snapshot
# ----------------------------------------------------------------------------

def run_rows(cfg, W, tokens, seq, pos, cache_k, cache_v, want_logits=False,
             static_coeff=None):
    """Run the layer stack, then the pool, for rows that read one snapshot.

    tokens/seq/pos: [N]. The cache is only read here; the caller writes the
    returned K/V afterwards, so every row sees the snapshot taken before the
    group ([OD How it differs]: a token's channels are added after its layer
    stack). Returns (pool dict, logits [N, V] or None, states [N, L, D]).
    """
    N = len(tokens)
    h = _f64(W["embed"])[np.asarray(tokens, dtype=np.int64)]
    states = np.zeros((N, cfg.L, cfg.D), dtype=np.float64)
    for l in range(cfg.L):
        states[:, l] = h
        h = consumer_layer(cfg, W, l, h, seq, pos, cache_k, cache_v)
    logits = None
    if want_logits:
        logits = _st(cfg, rmsnorm(h, W["final_norm"], cfg.eps)) @ _f64(W["lm_head"]).T
    return pool(cfg, W, states, pos, static_coeff), logits, states


def new_cache(cfg, B, Tmax):
    """A zero K/V cache, [B, k, Hkv, Tmax, d] each (R10)."""
    shape = (B, cfg.k, cfg.Hkv, Tmax, cfg.d)
    return np.zeros(shape, dtype=np.float64), np.zeros(shape, dtype=np.float64)


def _write(cache_k, cache_v, seq, pos, K, V):
    for r in range(len(seq)):
        cache_k[int(seq[r]), :, :, int(pos[r]), :] = K[r]
        cache_v[int(seq[r]), :, :, int(pos[r]), :] = V[r]


def cyclic_pass(cfg, W, tokens, g, cache_k, cache_v, q_begin=0, q_end=None,
                logits=None, static_coeff=None):
    """One cyclic Gauss-Seidel pass over tokens [B, T] ([OD How it differs]).

    Groups q = q_begin..q_end-1 run in order; each group's rows read the cache
    as it stood before the group and write their channels after it, so later
    groups of the same pass see earlier groups' updates. g = 1 is a Jacobi
    pass; g = T is token-by-token autoregressive evaluation.
    ``logits``: None, "last" (position T-1 of every sequence, -> [B, V]) or
    "all" (-> [B, T, V]); each is computed inside its group's stack.
    The cache arrays are updated in place.
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    B, T = tokens.shape
    if q_end is None:
        q_end = g
    out = None
    if logits == "last":
        out = np.zeros((B, cfg.V), dtype=np.float64)
    elif logits == "all":
        out = np.zeros((B, T, cfg.V), dtype=np.float64)
    for q in range(q_begin, q_end):
        P = group_positions(T, g, q)
        if len(P) == 0:
            continue
        seq = np.repeat(np.arange(B), len(P))
        pos = np.tile(P, B)
        toks = tokens[seq, pos]
        want = logits == "all" or (logits == "last" and (T - 1) in set(P.tolist()))
        res, lg, _ = run_rows(cfg, W, toks, seq, pos, cache_k, cache_v, want, static_coeff)
        _write(cache_k, cache_v, seq, pos, res["K"], res["V"])
        if logits == "all":
            out[seq, pos] = lg
        elif want:
            sel = pos == T - 1
            out[seq[sel]] = lg[sel]
    return out


def decode_step(cfg, W, tokens, t, cache_k, cache_v, static_coeff=None):
    """Autoregressive step at position t for tokens [B] ([PL 3 METHOD,
    "Execution schedules"]): run the stack against keys s < t, then append the
    token's pooled channels at t. Returns logits [B, V]."""
    tokens = np.asarray(tokens, dtype=np.int64)
    B = len(tokens)
    seq = np.arange(B)
    pos = np.full(B, t, dtype=np.int64)
    res, lg, _ = run_rows(cfg, W, tokens, seq, pos, cache_k, cache_v, True, static_coeff)
    _write(cache_k, cache_v, seq, pos, res["K"], res["V"])
    return lg


def decode_batch(cfg, W, tokens, pos, cache_k, cache_v, static_coeff=None):
    """A decode step in which sequence b sits at its own position pos[b]
    (R19): it is decode_step with t = pos[b] for each sequence at once, as in
    [PL 3 METHOD, "Execution schedules"] -- sequence b attends to its keys
    s < pos[b], then its pooled channels are appended at pos[b]. Sequences do
    not interact. Returns logits [B, V]."""
    tokens = np.asarray(tokens, dtype=np.int64)
    pos = np.asarray(pos, dtype=np.int64)
    B = len(tokens)
    seq = np.arange(B)
    res, lg, _ = run_rows(cfg, W, tokens, seq, pos, cache_k, cache_v, True, static_coeff)
    _write(cache_k, cache_v, seq, pos, res["K"], res["V"])
    return lg


def autoregressive(cfg, W, tokens, cache_k, cache_v, static_coeff=None):
    """Exact token-by-token evaluation: T decode steps from the given cache.
    Returns logits [B, T, V]."""
    tokens = np.asarray(tokens, dtype=np.int64)
    B, T = tokens.shape
    out = np.zeros((B, T, cfg.V), dtype=np.float64)
    for t in range(T):
        out[:, t] = decode_step(cfg, W, tokens[:, t], t, cache_k, cache_v, static_coeff)
    return out


def kv_residual(prev_k, prev_v, cur_k, cur_v):
    """Relative fixed-point residual ||KV_n - KV_{n-1}||_F / ||KV_n||_F between
    two caches (the convergence measure of a prefill schedule)."""
    num = np.sum((_f64(cur_k) - _f64(prev_k)) ** 2) + np.sum((_f64(cur_v) - _f64(prev_v)) ** 2)
    den = np.sum(_f64(cur_k) ** 2) + np.sum(_f64(cur_v) ** 2)
    return math.sqrt(num / den) if den > 0 else 0.0


# ----------------------------------------------------------------------------
# Feedback-free variant (R18)
# ----------------------------------------------------------------------------

def feedback_free_channel(cfg, W, states, pos, l, static_coeff=None):
    """Channel l of the feedback-free variant ([PL 5 ANALYSIS, "Deep-to-shallow
    feedback"]; reading R18): the pool of :func:`pool` with k = L, restricted
    to the sources 0..l of each row. states: [N, l + 1, D] (h^0..h^l); pos: [N].
    The router reads the sources of R inside 0..l, a prefix of its input, and
    gives a^b_{l, 0..l} through rows l*L + 0..l of W_R^b; static_coeff gives
    static_coeff[b][l][0..l] instead. Storage rounding as in :func:`pool` (R14,
    R17). Returns K, V [N, Hkv, d] and coeff [N, 2, l + 1].
    """
    states = _f64(states)
    N, D, L = states.shape[0], cfg.D, cfg.L
    Hkv, d = cfg.Hkv, cfg.d
    Rl = [s for s in router_sources(cfg) if s <= l]
    gained = getattr(cfg, "mixed_storage", "normed") == "gained"
    coeff = np.zeros((N, 2, l + 1), dtype=np.float64)
    out = []
    for beta in range(2):
        n = rmsnorm(states, _f64(W["src_norm"][beta])[: l + 1], cfg.eps)   # [N, l+1, D]
        if static_coeff is not None:
            a = np.broadcast_to(_f64(static_coeff)[beta, l, : l + 1], (N, l + 1))
        elif Rl:
            x = _st(cfg, n[:, Rl, :].reshape(N, len(Rl) * D))
            Wr = _f64(W["Wr"][beta])[l * L: l * L + l + 1, : len(Rl) * D]
            a = x @ Wr.T
        else:
            a = np.zeros((N, l + 1))
        coeff[:, beta] = a
        m = np.einsum("nl,nld->nd", a, n)
        tau = _f64(W["chan_norm"][beta][l])
        if gained:
            stored = _st(cfg, m * tau)
            scale = 1.0 / np.sqrt(np.mean(m * m, axis=-1) + cfg.eps)
        else:
            stored = _st(cfg, rmsnorm(m, tau, cfg.eps))
            scale = np.ones(N)
        Wp = _f64(W["Wk"][l] if beta == 0 else W["Wv"][l])
        out.append(((stored @ Wp.T) * scale[:, None]).reshape(N, Hkv, d))
    kt = rmsnorm(out[0], W["k_norm"][l], cfg.eps)
    K = _st(cfg, rope(kt, _f64(pos)[:, None], cfg.rope_base))
    V = _st(cfg, out[1])
    return K, V, coeff


def feedback_free_pass(cfg, W, tokens, cache_k, cache_v, pos0=0, logits=None,
                       static_coeff=None):
    """Tokens [B, T] at positions pos0..pos0+T-1 through the feedback-free
    variant in one layer-by-layer pass ([PL 5 ANALYSIS, "Deep-to-shallow
    feedback"]: no iteration). For l = 0..L-1: every token's channel l is
    pooled from its states 0..l and written to cache channel l at its
    position, then layer l runs for every token and attends to channel l at
    s < pos (keys of earlier calls included). k must equal L. ``logits``:
    None, "last" (-> [B, V] at the last position) or "all" (-> [B, T, V]).
    The cache arrays are updated in place.
    """
    assert cfg.k == cfg.L, "the feedback-free variant has one channel per layer"
    tokens = np.asarray(tokens, dtype=np.int64)
    B, T = tokens.shape
    seq = np.repeat(np.arange(B), T)
    pos = pos0 + np.tile(np.arange(T), B)
    h = _f64(W["embed"])[tokens.reshape(-1)]
    states = np.zeros((B * T, cfg.L, cfg.D), dtype=np.float64)
    for l in range(cfg.L):
        states[:, l] = h
        K, V, _ = feedback_free_channel(cfg, W, states[:, : l + 1], pos, l, static_coeff)
        for r in range(B * T):
            cache_k[seq[r], l, :, pos[r], :] = K[r]
            cache_v[seq[r], l, :, pos[r], :] = V[r]
        h = consumer_layer(cfg, W, l, h, seq, pos, cache_k, cache_v)
    if logits is None:
        return None
    lg = _st(cfg, rmsnorm(h, W["final_norm"], cfg.eps)) @ _f64(W["lm_head"]).T
    lg = lg.reshape(B, T, cfg.V)
    return lg[:, -1] if logits == "last" else lg


# ----------------------------------------------------------------------------
# Backward pass of the pool (gradients for training schedules)
# ----------------------------------------------------------------------------

def rmsnorm_backward(x, w, eps, dy):
    """Gradients of y = w * x / sqrt(mean(x^2) + eps) over the last axis.
    Returns (dx, xdy): with r = sqrt(mean(x^2) + eps) and g = w * dy,
    dx = g / r - x * sum(g * x) / (n * r^3); xdy = (x / r) * dy, whose sum
    over the axes that share a gain is that gain's gradient."""
    x, dy = _f64(x), _f64(dy)
    n = x.shape[-1]
    r = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    g = _f64(w) * dy
    dx = g / r - x * np.sum(g * x, axis=-1, keepdims=True) / (n * r ** 3)
    return dx, (x / r) * dy


def pool_backward(cfg, W, states, pos, dK, dV, static_coeff=None):
    """Reverse-mode gradients of :func:`pool` (exact arithmetic, no storage
    rounding) for upstream gradients dK, dV [N, k, Hkv, d] of its outputs K, V.
    The steps of :func:`pool` are undone in reverse: RoPE (a rotation, whose
    transpose rotates by -pos), the K-norm, the channel projections, the channel
    norm, the mix m_j = sum_l a_{j,l} n_l, the router a = W_R x (skipped with
    ``static_coeff``) and the per-source norms; the two branches' state
    gradients add up. Returns a dict of fp64 arrays: dstates [N, L, D], dWr
    [2, k*L, nR*D] (zeros with static_coeff), dWk, dWv [k, Hkv*d, D],
    dsrc_norm [2, L, D], dchan_norm [2, k, D], dk_norm [k, d].
    """
    states = _f64(states)
    N, L, D = states.shape
    k, Hkv, d = cfg.k, cfg.Hkv, cfg.d
    R = router_sources(cfg)
    dK, dV = _f64(dK), _f64(dV)
    g = {"dstates": np.zeros((N, L, D)), "dWr": np.zeros((2, k * L, len(R) * D)),
         "dWk": np.zeros((k, Hkv * d, D)), "dWv": np.zeros((k, Hkv * d, D)),
         "dsrc_norm": np.zeros((2, L, D)), "dchan_norm": np.zeros((2, k, D)),
         "dk_norm": np.zeros((k, d))}
    for beta in range(2):
        sig = _f64(W["src_norm"][beta])
        n = rmsnorm(states, sig, cfg.eps)                              # [N, L, D]
        x = n[:, R, :].reshape(N, len(R) * D)
        if static_coeff is None:
            a = (x @ _f64(W["Wr"][beta]).T).reshape(N, k, L)
        else:
            a = np.broadcast_to(_f64(static_coeff)[beta], (N, k, L))
        m = np.einsum("njl,nld->njd", a, n)                           # [N, k, D]
        tau = _f64(W["chan_norm"][beta])
        c = rmsnorm(m, tau, cfg.eps)
        dc = np.zeros((N, k, D))
        for j in range(k):
            if beta == 0:
                Wp = _f64(W["Wk"][j])
                kt = (c[:, j] @ Wp.T).reshape(N, Hkv, d)
                dkn = rope(dK[:, j], -_f64(pos)[:, None], cfg.rope_base)
                dkt, kdy = rmsnorm_backward(kt, W["k_norm"][j], cfg.eps, dkn)
                g["dk_norm"][j] += kdy.reshape(-1, d).sum(axis=0)
                dy = dkt.reshape(N, Hkv * d)
                g["dWk"][j] += dy.T @ c[:, j]
            else:
                Wp = _f64(W["Wv"][j])
                dy = dV[:, j].reshape(N, Hkv * d)
                g["dWv"][j] += dy.T @ c[:, j]
            dc[:, j] = dy @ Wp
        dm, mdy = rmsnorm_backward(m, tau, cfg.eps, dc)
        g["dchan_norm"][beta] += mdy.sum(axis=0)
        da = np.einsum("njd,nld->njl", dm, n)                         # [N, k, L]
        dn = np.einsum("njl,njd->nld", a, dm)                         # [N, L, D]
        if static_coeff is None:
            daf = da.reshape(N, k * L)
            g["dWr"][beta] += daf.T @ x
            dn[:, R, :] += (daf @ _f64(W["Wr"][beta])).reshape(N, len(R), D)
        dh, hdy = rmsnorm_backward(states, sig, cfg.eps, dn)
        g["dstates"] += dh
        g["dsrc_norm"][beta] += hdy.sum(axis=0)
    return g
