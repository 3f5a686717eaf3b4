"""Host-side tests of the C ABI: the library loads, exports every function
that include/wm.h declares, and rejects bad arguments before launching
anything (these calls never reach the GPU, so they run on CPU-only hosts)."""

import ctypes
import os
import re

import pytest

from cross_layer_kv_pool_b300 import build, synth, wm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return wm.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "wm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(wm_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert "wm_cyclic_pass" in names and "wm_pool_mix" in names
    for n in names:
        assert hasattr(L, n), n
    assert set(wm.EXPORTED) <= set(names)


def test_version_and_status_strings(L):
    assert L.wm_abi_version() == 1
    for s in range(7):
        assert wm.status_string(s)
    assert wm.status_string(99) == "unknown status"


def _cfg(**kw):
    return wm.make_config(synth.TINY_FP32.replace(**kw))


def test_workspace_size(L):
    c = _cfg()
    n1 = wm.workspace_size(c, 16, 64)
    n2 = wm.workspace_size(c, 32, 64)
    assert 0 < n1 < n2
    assert n1 % 256 == 0
    bad = _cfg(d=96)
    assert L.wm_workspace_size(ctypes.byref(bad), 16, 64) == 0
    assert L.wm_workspace_size(ctypes.byref(c), 0, 64) == 0


FAKE = 1 << 20   # an aligned non-null address; never dereferenced by these calls


def _weights_struct(**override):
    s = wm.WMWeights()
    for i, n in enumerate(synth.WEIGHT_ORDER):
        setattr(s, n, FAKE + 4096 * i)
    for n, v in override.items():
        setattr(s, n, v)
    return s


def _pass(L, cfg, w, tokens=FAKE, B=1, T=64, g=4, qb=0, qe=4, ck=FAKE, cv=FAKE, Tmax=64,
          logits=None, mode=0, ws=FAKE, ws_bytes=1 << 40):
    return L.wm_cyclic_pass(ctypes.byref(cfg), ctypes.byref(w), tokens, B, T, g, qb, qe, ck, cv,
                            Tmax, logits, mode, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(L=0), wm.WM_ERR_INVALID_ARG),
    (dict(D=100), wm.WM_ERR_INVALID_ARG),
    (dict(k=5), wm.WM_ERR_INVALID_ARG),
    (dict(p=0), wm.WM_ERR_INVALID_ARG),
    (dict(p_offset=2), wm.WM_ERR_INVALID_ARG),
    (dict(Hq=3), wm.WM_ERR_INVALID_ARG),
    (dict(d=96), wm.WM_ERR_UNSUPPORTED),
    (dict(F=100), wm.WM_ERR_INVALID_ARG),
])
def test_bad_config_rejected(L, kw, status):
    assert _pass(L, _cfg(**kw), _weights_struct()) == status


@pytest.mark.parametrize("kw", [
    dict(tokens=None), dict(B=0), dict(T=0), dict(g=0), dict(g=65), dict(T=65),
    dict(qb=3, qe=2), dict(qe=5), dict(ck=None), dict(ck=FAKE + 2), dict(mode=1),
    dict(mode=3),
])
def test_bad_pass_args_rejected(L, kw):
    assert _pass(L, _cfg(), _weights_struct(), **kw) == wm.WM_ERR_INVALID_ARG


def test_bad_weights_and_workspace_rejected(L):
    c = _cfg()
    assert _pass(L, c, _weights_struct(Wr=None)) == wm.WM_ERR_INVALID_ARG
    assert _pass(L, c, _weights_struct(Wk=FAKE + 8)) == wm.WM_ERR_INVALID_ARG
    assert _pass(L, c, _weights_struct(), ws=None) == wm.WM_ERR_WORKSPACE
    assert _pass(L, c, _weights_struct(), ws=FAKE + 16) == wm.WM_ERR_WORKSPACE
    need = wm.workspace_size(c, 16, 64)
    assert _pass(L, c, _weights_struct(), ws_bytes=need - 1) == wm.WM_ERR_WORKSPACE


def test_other_entry_points_validate(L):
    c = _cfg()
    w = _weights_struct()
    vp = FAKE
    # decode: pos out of range, null logits
    assert L.wm_decode_step(ctypes.byref(c), ctypes.byref(w), vp, 1, 64, vp, vp, 64, vp, vp,
                            1 << 40, None) == wm.WM_ERR_INVALID_ARG
    assert L.wm_decode_step(ctypes.byref(c), ctypes.byref(w), vp, 1, 3, vp, vp, 64, None, vp,
                            1 << 40, None) == wm.WM_ERR_INVALID_ARG
    # batched decode: null positions, B = 0, null tokens
    assert L.wm_decode_batch(ctypes.byref(c), ctypes.byref(w), vp, None, 1, vp, vp, 64, vp, vp,
                             1 << 40, None) == wm.WM_ERR_INVALID_ARG
    assert L.wm_decode_batch(ctypes.byref(c), ctypes.byref(w), vp, vp, 0, vp, vp, 64, vp, vp,
                             1 << 40, None) == wm.WM_ERR_INVALID_ARG
    assert L.wm_decode_batch(ctypes.byref(c), ctypes.byref(w), None, vp, 1, vp, vp, 64, vp, vp,
                             1 << 40, None) == wm.WM_ERR_INVALID_ARG
    # attention: channel out of range
    assert L.wm_channel_attn(ctypes.byref(c), vp, 4, vp, vp, 2, vp, vp, 1, 64, vp, 0, vp, 1 << 40,
                             None) == wm.WM_ERR_INVALID_ARG
    # rows_per_seq must divide N
    assert L.wm_channel_attn(ctypes.byref(c), vp, 6, vp, vp, 0, vp, vp, 1, 64, vp, 4, vp, 1 << 40,
                             None) == wm.WM_ERR_INVALID_ARG
    # pool: N = 0, misaligned states
    assert L.wm_pool_mix(ctypes.byref(c), ctypes.byref(w), vp, 0, vp, vp, vp, vp, 1, 64, None,
                         None, vp, 1 << 40, None) == wm.WM_ERR_INVALID_ARG
    assert L.wm_pool_mix(ctypes.byref(c), ctypes.byref(w), vp + 4, 4, vp, vp, vp, vp, 1, 64,
                         None, None, vp, 1 << 40, None) == wm.WM_ERR_INVALID_ARG
    # flags: null workspace
    f = ctypes.c_uint32()
    assert L.wm_check_flags(None, 256, ctypes.byref(f), None) == wm.WM_ERR_INVALID_ARG


def test_feedforward_pass_validates(L):
    """The feedback-free pass needs k = L and the usual argument checks."""
    vp = FAKE
    c = _cfg()                      # k = 2 < L = 4
    w = _weights_struct()
    assert L.wm_feedforward_pass(ctypes.byref(c), ctypes.byref(w), vp, 1, 8, 0, vp, vp, 16, None, 0,
                                 vp, 1 << 40, None) == wm.WM_ERR_INVALID_ARG
    c4 = _cfg(k=4)
    assert L.wm_feedforward_pass(ctypes.byref(c4), ctypes.byref(w), vp, 1, 8, 9, vp, vp, 16, None,
                                 0, vp, 1 << 40, None) == wm.WM_ERR_INVALID_ARG   # pos0 + T > Tmax
    assert L.wm_feedforward_pass(ctypes.byref(c4), ctypes.byref(w), vp, 1, 8, 0, vp, vp, 16, None,
                                 1, vp, 1 << 40, None) == wm.WM_ERR_INVALID_ARG   # LAST, no logits
    assert L.wm_feedforward_pass(ctypes.byref(c4), ctypes.byref(w), vp, 1, 8, 0, vp, vp, 16, None,
                                 0, None, 1 << 40, None) == wm.WM_ERR_WORKSPACE
