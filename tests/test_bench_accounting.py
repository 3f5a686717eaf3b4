"""The bytes per decode step that bench.py divides by (its HBM fraction),
checked on CPU against the model's own tensors rather than against the
bench's formula."""

import importlib.util
import os

import torch

from cross_layer_kv_pool_b300 import synth


def _bench():
    path = os.path.join(os.path.dirname(__file__), "..", "bench.py")
    spec = importlib.util.spec_from_file_location("bench_under_test", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


# Tensors a decode step reads in full: the layer stack's matrices and gains,
# the LM head and final norm, the router and the channel projections. The
# embedding table is read at the B token rows only; the pool's own gains
# (source, channel and key norms) are below a thousandth of the total and are
# not counted.
READ_IN_FULL = ("lm_head", "final_norm", "in_norm", "post_norm", "q_norm", "Wq", "Wo", "Wgate",
                "Wup", "Wdown", "Wr", "Wk", "Wv")

SHAPES = [synth.ModelShape(L=4, D=128, k=2, p=2, Hq=4, Hkv=2, d=64, F=256, V=300),
          synth.ModelShape(L=6, D=256, k=3, p=3, p_offset=1, Hq=6, Hkv=3, d=32, F=512, V=97)]


def test_decode_bytes_at_position_zero_are_the_weights_read():
    b = _bench()
    for s in SHAPES:
        W = synth.make_weights(s, seed=0)
        for B in (1, 5):
            # weights read in full, B embedding rows, and each sequence's new
            # K and V entries of all k channels (bf16: 2 bytes an element)
            elems = sum(W[n].numel() for n in READ_IN_FULL) + B * s.D + 2 * B * s.k * s.Hkv * s.d
            assert b.decode_step_bytes(s, B, 0) == 2 * elems


def test_decode_bytes_grow_by_one_cache_position_per_layer():
    """Each visible position adds, for every layer, the K and V entries of
    that layer's channel for every sequence."""
    b = _bench()
    for s in SHAPES:
        for B in (1, 3):
            cache = torch.empty((B, s.k, s.Hkv, 1, s.d), dtype=torch.bfloat16)
            per_position = s.L * 2 * cache[:, 0].numel() * cache.element_size()
            for pos in (0, 7, 100):
                assert b.decode_step_bytes(s, B, pos + 1) - b.decode_step_bytes(s, B, pos) == per_position
