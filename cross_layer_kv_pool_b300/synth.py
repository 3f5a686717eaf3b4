"""Seeded synthetic inputs: model shapes, weights and token ids.

This module holds shapes and random draws only, none of the method's
arithmetic, so that both the CUDA path and the CPU oracle can be fed the same
inputs without sharing any computation.

Weights follow one recipe for every workload: every matrix is N(0, 0.02);
every RMSNorm gain is 1 (optionally 1 + N(0, gain_jitter), which the parity
tests use so that a gain applied to the wrong element shows up). Tensors are
drawn in ``WEIGHT_ORDER`` from one torch generator seeded with ``seed``, in
fp32, then rounded to the workload's storage type (bf16: round to nearest
even). Token ids are uniform over the vocabulary from their own seed.
"""

from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import torch

# Order in which weight tensors are drawn; it is also the field order of the
# C ABI's weight struct.
WEIGHT_ORDER = (
    "embed", "lm_head", "final_norm",
    "in_norm", "post_norm", "q_norm",
    "Wq", "Wo", "Wgate", "Wup", "Wdown",
    "src_norm", "Wr", "chan_norm", "Wk", "Wv", "k_norm",
)

GAIN_NAMES = frozenset({"final_norm", "in_norm", "post_norm", "q_norm",
                        "src_norm", "chan_norm", "k_norm"})


@dataclass(frozen=True)
class ModelShape:
    """Shape of a WhiteMatter decoder: L layers of width D, k pool channels,
    router stride p (reading layers l with l % p == p_offset), Hq query heads
    and Hkv KV heads of size d, SwiGLU width F, vocabulary V."""
    L: int
    D: int
    k: int
    p: int
    Hq: int
    Hkv: int
    d: int
    F: int
    V: int
    p_offset: int = 0
    eps: float = 1e-6
    rope_base: float = 1e6
    dtype: str = "bf16"          # "f32" or "bf16" storage / compute type

    @property
    def nR(self) -> int:
        return len([l for l in range(self.L) if l % self.p == self.p_offset])

    def replace(self, **kw) -> "ModelShape":
        return dataclasses.replace(self, **kw)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


def weight_shapes(s: ModelShape) -> dict:
    L, D, k, d = s.L, s.D, s.k, s.d
    return {
        "embed": (s.V, D), "lm_head": (s.V, D), "final_norm": (D,),
        "in_norm": (L, D), "post_norm": (L, D), "q_norm": (L, d),
        "Wq": (L, s.Hq * d, D), "Wo": (L, D, s.Hq * d),
        "Wgate": (L, s.F, D), "Wup": (L, s.F, D), "Wdown": (L, D, s.F),
        "src_norm": (2, L, D), "Wr": (2, k * L, s.nR * D),
        "chan_norm": (2, k, D), "Wk": (k, s.Hkv * d, D), "Wv": (k, s.Hkv * d, D),
        "k_norm": (k, d),
    }


def make_weights(s: ModelShape, seed: int = 0, device="cpu", gain_jitter: float = 0.0,
                 std: float = 0.02) -> dict:
    """Draw every weight tensor in WEIGHT_ORDER from one seeded generator."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    shapes = weight_shapes(s)
    out = {}
    for name in WEIGHT_ORDER:
        shp = shapes[name]
        if name in GAIN_NAMES:
            t = torch.ones(shp, dtype=torch.float32, device=device)
            if gain_jitter:
                t += gain_jitter * torch.randn(shp, generator=g, dtype=torch.float32, device=device)
        else:
            t = std * torch.randn(shp, generator=g, dtype=torch.float32, device=device)
        out[name] = t.to(s.torch_dtype).contiguous()
    return out


def make_tokens(s: ModelShape, B: int, T: int, seed: int = 1, device="cpu") -> torch.Tensor:
    """Token ids uniform over [0, V), int32 [B, T]."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randint(0, s.V, (B, T), generator=g, device=device, dtype=torch.int64).to(torch.int32)


def make_normal(shape, seed: int, device="cpu", std: float = 1.0, dtype=torch.float32):
    """Generic seeded N(0, std^2) tensor (states, queries, cache contents)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return (std * torch.randn(shape, generator=g, dtype=torch.float32, device=device)).to(dtype)


def to_numpy_weights(W: dict) -> dict:
    """Host float64 copies for the oracle (exact: bf16 and fp32 embed in fp64)."""
    return {n: t.detach().to("cpu", torch.float64).numpy() for n, t in W.items()}


# --------------------------------------------------------------------------
# Workloads: model shapes and batch sizes of the pages' models.
# --------------------------------------------------------------------------

TINY_FP32 = ModelShape(L=4, D=128, k=2, p=2, Hq=2, Hkv=2, d=64, F=512, V=1024, dtype="f32")
HALF_SMALL = ModelShape(L=16, D=512, k=8, p=2, Hq=8, Hkv=8, d=64, F=1536, V=151936)
FULL_SMALL = HALF_SMALL.replace(k=16)
HALF_1P3B = ModelShape(L=28, D=1792, k=14, p=2, Hq=14, Hkv=2, d=128, F=4608, V=151936)

WORKLOADS = {
    "tiny_fp32": dict(shape=TINY_FP32, B=1, T=64, g=4, passes=3),
    "half_small": dict(shape=HALF_SMALL, B=8, T=2048, g=16, passes=3),
    "full_small": dict(shape=FULL_SMALL, B=8, T=2048, g=16, passes=3),
    "prefill_1p3b": dict(shape=HALF_1P3B, B=64, T=2048, g=16, passes=3),
    "decode_1p3b": dict(shape=HALF_1P3B, B=64, T=2048, g=16, passes=3,
                        decode_steps=256, Tmax=2304),
}
