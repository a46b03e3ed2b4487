"""The C ABI library builds, loads and exports every symbol of include/lat.h,
and its host-side argument checks answer without a GPU."""
import ctypes
import os
import re

import pytest

from latency_transformer_block_gb300 import build, lat

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return lat.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "lat.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lat_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("lat_create", "lat_prefill_kv", "lat_block_forward", "lat_denoise_chunk", "lat_destroy",
              "lat_set_schedule", "lat_sync", "lat_status_str", "lat_debug_indices"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in declared_functions():
        assert hasattr(L, n), f"{n} declared in lat.h but not exported by liblat.so"


def test_status_strings(L):
    for code, name in enumerate(lat.STATUS):
        assert L.lat_status_str(code).decode() == name


def test_host_validation_without_gpu(L):
    h = ctypes.c_void_p()
    assert L.lat_create(None, None, ctypes.byref(h)) == 1            # NULL desc -> ARG
    d = lat.ModelDesc()
    d.kind = 5
    assert L.lat_create(ctypes.byref(d), None, ctypes.byref(h)) == 8  # unknown kind
    d.kind = lat.LAT_PI0_ACTION_EXPERT
    d.D, d.Hq, d.Hkv, d.dh, d.F, d.L, d.S, d.T_q, d.act_dim = 200, 4, 1, 64, 1024, 1, 2, 64, 32
    d.rope_base, d.eps = 10000.0, 1e-6
    assert L.lat_create(ctypes.byref(d), None, ctypes.byref(h)) == 2  # D not a multiple of 128
    d.D = 256
    d.dh = 48
    assert L.lat_create(ctypes.byref(d), None, ctypes.byref(h)) == 2  # unsupported head dim
    d.dh, d.T_q = 64, 65
    assert L.lat_create(ctypes.byref(d), None, ctypes.byref(h)) == 2  # too many query tokens
    assert b"T_q" in L.lat_last_error()
    assert L.lat_sync(None) == 1
    assert L.lat_debug_wait_skew(None, 1, 1) == 1                     # NULL ctx -> ARG
    L.lat_destroy(None)


def _dit_desc(**kw):
    d = lat.ModelDesc()
    d.kind = 2   # LAT_DIT
    d.D, d.Hq, d.Hkv, d.dh, d.F, d.L, d.S, d.T_q = 256, 2, 2, 128, 512, 1, 4, 100
    d.n_hist, d.t_dim, d.max_batch, d.n_streams = 4, 64, 4, 1
    d.rope_base, d.eps = 10000.0, 1e-6
    for k, v in kw.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("kw,words", [
    (dict(dh=64), b"dh must be 128 or 256"),
    (dict(Hkv=1), b"Hq == Hkv"),
    (dict(n_hist=5), b"n_hist"),
    (dict(max_batch=17), b"max_batch"),
    (dict(grid_h=5), b"grid_h and grid_w"),                  # one of the two set
    (dict(grid_h=3, grid_w=7), b"whole frames"),            # 100 tokens are not whole 3 x 7 frames
    (dict(text_len=401), b"text_len"),                      # more than max_batch * T_q
    (dict(text_len=-1), b"text_len"),
    (dict(page_tokens=501), b"page_tokens"),                # larger than a ring of 5 x 100 tokens
])
def test_dit_descriptor_checks_without_gpu(L, kw, words):
    """The DiT options' descriptor checks run on the host before any CUDA call:
    LAT_ERR_SHAPE with the reason in lat_last_error."""
    h = ctypes.c_void_p()
    d = _dit_desc(**kw)
    assert L.lat_create(ctypes.byref(d), None, ctypes.byref(h)) == 2
    assert words in L.lat_last_error()
