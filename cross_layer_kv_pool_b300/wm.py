"""ctypes binding of libwm (include/wm.h). Argument marshalling only.

Tensors are torch tensors in device memory (PyTorch supplies allocation and
streams); every computation happens in the library's CUDA kernels. The
library must have been built (``python -m cross_layer_kv_pool_b300.build``):
there is no other implementation to fall back to, and ``lib()`` raises if it
is missing.
"""

from __future__ import annotations

import ctypes
import os

import torch

from .synth import WEIGHT_ORDER, ModelShape

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libwm.so")

WM_OK, WM_ERR_INVALID_ARG, WM_ERR_UNSUPPORTED, WM_ERR_WORKSPACE, WM_ERR_CUDA, \
    WM_ERR_TIMEOUT, WM_ERR_DEVICE_BOUNDS = range(7)
WM_F32, WM_BF16 = 0, 1
LOGITS = {"none": 0, None: 0, "last": 1, "all": 2}
WM_FLAG_SIMT_GEMM = 1
WM_FLAG_NO_CLUSTER = 2
WM_FLAG_WAIT_PROBE = 4

EXPORTED = ("wm_workspace_size", "wm_pool_mix", "wm_channel_attn", "wm_cyclic_pass",
            "wm_decode_step", "wm_decode_batch", "wm_check_flags", "wm_status_string", "wm_abi_version",
            "wm_pool_mix_static", "wm_feedforward_pass", "wm_pool_backward",
            "wm_pool_backward_workspace_size")


class WMError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


WM_TRACE_GEMM, WM_TRACE_MIX, WM_TRACE_ATTN = 0, 1, 2


class WMTrace(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("capacity", ctypes.c_int32),
                ("count", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("begin", ctypes.POINTER(ctypes.c_void_p)), ("end", ctypes.POINTER(ctypes.c_void_p)),
                ("work", ctypes.POINTER(ctypes.c_double)), ("launches", ctypes.c_int64)]


class WMConfig(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int32), ("D", ctypes.c_int32), ("k", ctypes.c_int32),
                ("p", ctypes.c_int32), ("p_offset", ctypes.c_int32), ("Hq", ctypes.c_int32),
                ("Hkv", ctypes.c_int32), ("d", ctypes.c_int32), ("F", ctypes.c_int32),
                ("V", ctypes.c_int32), ("eps", ctypes.c_float), ("rope_base", ctypes.c_float),
                ("dtype", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("trace", ctypes.POINTER(WMTrace))]


class Tracer:
    """Event pairs for the measurement hook: ``attach(model)`` makes the
    library bracket each launch of ``kind`` with these torch CUDA events."""

    def __init__(self, kind: int, capacity: int):
        self.events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(capacity)]
        for b, e in self.events:       # create the driver handles
            b.record()
            e.record()
        torch.cuda.synchronize()
        n = capacity
        self._b = (ctypes.c_void_p * n)(*[b.cuda_event for b, _ in self.events])
        self._e = (ctypes.c_void_p * n)(*[e.cuda_event for _, e in self.events])
        self._w = (ctypes.c_double * n)()
        self.t = WMTrace(kind, n, 0, 0, ctypes.cast(self._b, ctypes.POINTER(ctypes.c_void_p)),
                         ctypes.cast(self._e, ctypes.POINTER(ctypes.c_void_p)),
                         ctypes.cast(self._w, ctypes.POINTER(ctypes.c_double)), 0)

    def attach(self, model: "Model"):
        model.cfg.trace = ctypes.pointer(self.t)

    @staticmethod
    def detach(model: "Model"):
        model.cfg.trace = ctypes.POINTER(WMTrace)()

    def reset(self):
        self.t.count = 0
        self.t.launches = 0

    def results(self):
        """[(milliseconds, work)] of the traced launches (after a sync)."""
        return [(self.events[i][0].elapsed_time(self.events[i][1]), self._w[i])
                for i in range(self.t.count)]


class WMPoolGrads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("dWr", "dWk", "dWv", "dsrc_norm", "dchan_norm", "dk_norm")]


class WMWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_ORDER] + [("static_coeff", ctypes.c_void_p)]


_lib = None


def lib():
    """Load libwm.so (once). Raises FileNotFoundError if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise FileNotFoundError(f"{LIB_PATH} is missing: build it with "
                                    "`python -m cross_layer_kv_pool_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        cfgp, wp = ctypes.POINTER(WMConfig), ctypes.POINTER(WMWeights)
        L.wm_workspace_size.restype = sz
        L.wm_workspace_size.argtypes = [cfgp, i32, i32]
        L.wm_pool_mix.restype = ctypes.c_int
        L.wm_pool_mix.argtypes = [cfgp, wp, vp, i32, vp, vp, vp, vp, i32, i32, vp, vp, vp, sz, vp]
        L.wm_channel_attn.restype = ctypes.c_int
        L.wm_channel_attn.argtypes = [cfgp, vp, i32, vp, vp, i32, vp, vp, i32, i32, vp, i32, vp, sz,
                                      vp]
        L.wm_cyclic_pass.restype = ctypes.c_int
        L.wm_cyclic_pass.argtypes = [cfgp, wp, vp, i32, i32, i32, i32, i32, vp, vp, i32, vp, i32,
                                     vp, sz, vp]
        L.wm_feedforward_pass.restype = ctypes.c_int
        L.wm_feedforward_pass.argtypes = [cfgp, wp, vp, i32, i32, i32, vp, vp, i32, vp, i32, vp,
                                          sz, vp]
        L.wm_pool_backward_workspace_size.restype = sz
        L.wm_pool_backward_workspace_size.argtypes = [cfgp, i32]
        L.wm_pool_backward.restype = ctypes.c_int
        L.wm_pool_backward.argtypes = [cfgp, wp, vp, i32, vp, vp, vp, vp,
                                       ctypes.POINTER(WMPoolGrads), vp, sz, vp]
        L.wm_decode_step.restype = ctypes.c_int
        L.wm_decode_step.argtypes = [cfgp, wp, vp, i32, i32, vp, vp, i32, vp, vp, sz, vp]
        L.wm_decode_batch.restype = ctypes.c_int
        L.wm_decode_batch.argtypes = [cfgp, wp, vp, vp, i32, vp, vp, i32, vp, vp, sz, vp]
        L.wm_pool_mix_static.restype = ctypes.c_int
        L.wm_pool_mix_static.argtypes = [cfgp, wp, vp, i32, vp, vp, vp, vp, i32, i32, vp, vp, vp]
        L.wm_check_flags.restype = ctypes.c_int
        L.wm_check_flags.argtypes = [vp, sz, ctypes.POINTER(ctypes.c_uint32), vp]
        L.wm_status_string.restype = ctypes.c_char_p
        L.wm_status_string.argtypes = [ctypes.c_int]
        L.wm_abi_version.restype = i32
        L.wm_abi_version.argtypes = []
        _lib = L
    return _lib


def status_string(s: int) -> str:
    return lib().wm_status_string(int(s)).decode()


def _check(status, where):
    if status != WM_OK:
        raise WMError(status, where)


def make_config(shape: ModelShape, flags: int = 0) -> WMConfig:
    return WMConfig(shape.L, shape.D, shape.k, shape.p, shape.p_offset, shape.Hq, shape.Hkv,
                    shape.d, shape.F, shape.V, shape.eps, shape.rope_base,
                    WM_F32 if shape.dtype == "f32" else WM_BF16, flags, None)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_weights_struct(W: dict, static_coeff: torch.Tensor | None = None) -> WMWeights:
    """Pointer struct for device weight tensors (kept alive by the caller)."""
    s = WMWeights()
    for n in WEIGHT_ORDER:
        setattr(s, n, W[n].data_ptr())
    s.static_coeff = None if static_coeff is None else static_coeff.data_ptr()
    return s


class Model:
    """Device weights of one model plus the C structs that describe them."""

    def __init__(self, shape: ModelShape, weights: dict, static_coeff=None, flags: int = 0):
        self.shape = shape
        self.W = weights
        self.static_coeff = None if static_coeff is None else \
            static_coeff.to(device=weights["embed"].device, dtype=torch.float32).contiguous()
        self.cfg = make_config(shape, flags)
        self.wstruct = make_weights_struct(weights, self.static_coeff)

    def new_cache(self, B: int, Tmax: int, fill: float = 0.0):
        s = self.shape
        shp = (B, s.k, s.Hkv, Tmax, s.d)
        dev = self.W["embed"].device
        ck = torch.full(shp, fill, dtype=s.torch_dtype, device=dev)
        cv = torch.full(shp, fill, dtype=s.torch_dtype, device=dev)
        return ck, cv

    def workspace(self, max_rows: int, Tmax: int):
        n = workspace_size(self.cfg, max_rows, Tmax)
        return torch.zeros(n, dtype=torch.uint8, device=self.W["embed"].device)


def workspace_size(cfg: WMConfig, max_rows: int, Tmax: int) -> int:
    n = lib().wm_workspace_size(ctypes.byref(cfg), int(max_rows), int(Tmax))
    if n == 0:
        raise WMError(WM_ERR_INVALID_ARG, "wm_workspace_size")
    return n


def wm_pool_mix(m: Model, states, seq, pos, cache_k, cache_v, ws, coeff_out=None,
                mixed_out=None, stream=None):
    B, Tmax = cache_k.shape[0], cache_k.shape[3]
    st = lib().wm_pool_mix(ctypes.byref(m.cfg), ctypes.byref(m.wstruct), _ptr(states),
                           states.shape[0], _ptr(seq), _ptr(pos), _ptr(cache_k), _ptr(cache_v),
                           B, Tmax, _ptr(coeff_out), _ptr(mixed_out), _ptr(ws), ws.numel(),
                           _stream(stream))
    _check(st, "wm_pool_mix")


def wm_pool_mix_static(m: Model, states, seq, pos, cache_k, cache_v, coeff_out=None,
                       mixed_out=None, stream=None):
    """wm_pool_mix with the library's fixed internal scratch instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    B, Tmax = cache_k.shape[0], cache_k.shape[3]
    st = lib().wm_pool_mix_static(ctypes.byref(m.cfg), ctypes.byref(m.wstruct), _ptr(states),
                                  states.shape[0], _ptr(seq), _ptr(pos), _ptr(cache_k),
                                  _ptr(cache_v), B, Tmax, _ptr(coeff_out), _ptr(mixed_out),
                                  _stream(stream))
    _check(st, "wm_pool_mix_static")


def wm_channel_attn(cfg: WMConfig, q, seq, pos, channel: int, cache_k, cache_v, out, ws,
                    rows_per_seq: int = 0, stream=None):
    B, Tmax = cache_k.shape[0], cache_k.shape[3]
    st = lib().wm_channel_attn(ctypes.byref(cfg), _ptr(q), q.shape[0], _ptr(seq), _ptr(pos),
                               int(channel), _ptr(cache_k), _ptr(cache_v), B, Tmax, _ptr(out),
                               int(rows_per_seq), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "wm_channel_attn")


def wm_cyclic_pass(m: Model, tokens, g: int, cache_k, cache_v, ws, q_begin: int = 0,
                   q_end: int | None = None, logits=None, logits_mode="none", stream=None):
    B, T = tokens.shape
    Tmax = cache_k.shape[3]
    q_end = g if q_end is None else q_end
    st = lib().wm_cyclic_pass(ctypes.byref(m.cfg), ctypes.byref(m.wstruct), _ptr(tokens), B, T,
                              int(g), int(q_begin), int(q_end), _ptr(cache_k), _ptr(cache_v),
                              Tmax, _ptr(logits), LOGITS[logits_mode], _ptr(ws), ws.numel(),
                              _stream(stream))
    _check(st, "wm_cyclic_pass")


def wm_feedforward_pass(m: Model, tokens, cache_k, cache_v, ws, pos0: int = 0, logits=None,
                        logits_mode="none", stream=None):
    """Feedback-free variant (k = L): tokens [B][T] at positions pos0.. in
    one exact pass; the workspace may hold fewer than B*T rows (at least T)."""
    B, T = tokens.shape
    Tmax = cache_k.shape[3]
    st = lib().wm_feedforward_pass(ctypes.byref(m.cfg), ctypes.byref(m.wstruct), _ptr(tokens), B,
                                   T, int(pos0), _ptr(cache_k), _ptr(cache_v), Tmax, _ptr(logits),
                                   LOGITS[logits_mode], _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "wm_feedforward_pass")


def pool_grads(m: Model, router: bool = True) -> dict:
    """Zeroed fp32 gradient accumulators for wm_pool_backward."""
    s = m.shape
    dev = m.W["embed"].device
    z = lambda *shape: torch.zeros(shape, dtype=torch.float32, device=dev)  # noqa: E731
    g = {"dWk": z(s.k, s.Hkv * s.d, s.D), "dWv": z(s.k, s.Hkv * s.d, s.D),
         "dsrc_norm": z(2, s.L, s.D), "dchan_norm": z(2, s.k, s.D), "dk_norm": z(s.k, s.d)}
    g["dWr"] = z(2, s.k * s.L, s.nR * s.D) if router else None
    return g


def wm_pool_backward(m: Model, states, pos, dK, dV, dstates, grads: dict, ws=None, stream=None):
    """Backward pass of the pool for N rows: writes dstates, adds to grads."""
    N = states.shape[0]
    if ws is None:
        n = lib().wm_pool_backward_workspace_size(ctypes.byref(m.cfg), N)
        ws = torch.zeros(n, dtype=torch.uint8, device=states.device)
    gs = WMPoolGrads(*[_ptr(grads.get(k)) for k in
                       ("dWr", "dWk", "dWv", "dsrc_norm", "dchan_norm", "dk_norm")])
    st = lib().wm_pool_backward(ctypes.byref(m.cfg), ctypes.byref(m.wstruct), _ptr(states), N,
                                _ptr(pos), _ptr(dK), _ptr(dV), _ptr(dstates), ctypes.byref(gs),
                                _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "wm_pool_backward")
    return ws


def wm_decode_step(m: Model, tokens, pos: int, cache_k, cache_v, logits, ws, stream=None):
    B = tokens.shape[0]
    Tmax = cache_k.shape[3]
    st = lib().wm_decode_step(ctypes.byref(m.cfg), ctypes.byref(m.wstruct), _ptr(tokens), B,
                              int(pos), _ptr(cache_k), _ptr(cache_v), Tmax, _ptr(logits),
                              _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "wm_decode_step")


def wm_decode_batch(m: Model, tokens, pos, cache_k, cache_v, logits, ws, stream=None):
    """One decode step with per-sequence positions ``pos`` (int32 device [B]).
    Nothing on the host depends on the values of ``tokens`` or ``pos``, so the
    call can be captured once in a CUDA graph and replayed."""
    B = tokens.shape[0]
    Tmax = cache_k.shape[3]
    st = lib().wm_decode_batch(ctypes.byref(m.cfg), ctypes.byref(m.wstruct), _ptr(tokens), _ptr(pos),
                               B, _ptr(cache_k), _ptr(cache_v), Tmax, _ptr(logits), _ptr(ws),
                               ws.numel(), _stream(stream))
    _check(st, "wm_decode_batch")


def wm_check_flags(ws, stream=None) -> int:
    """Reads and clears the device-side flag word; raises on a set check bit."""
    f = ctypes.c_uint32(0)
    st = lib().wm_check_flags(_ptr(ws), ws.numel(), ctypes.byref(f), _stream(stream))
    if st not in (WM_OK,):
        raise WMError(st, f"wm_check_flags (flags=0x{f.value:x})")
    return f.value


def wm_check_static_flags(stream=None) -> int:
    """wm_check_flags on the flag word of wm_pool_mix_static's internal scratch."""
    f = ctypes.c_uint32(0)
    st = lib().wm_check_flags(None, 0, ctypes.byref(f), _stream(stream))
    if st not in (WM_OK,):
        raise WMError(st, f"wm_check_flags (static scratch, flags=0x{f.value:x})")
    return f.value


def rows_for_pass(B: int, T: int, g: int) -> int:
    """Rows of the largest group of a cyclic pass: B * ceil(T / g)."""
    return B * (-(-T // g))
