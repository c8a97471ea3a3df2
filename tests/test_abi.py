"""CPU-only checks of the C ABI: the library builds and loads, exports every
function include/cb.h declares, and rejects bad arguments and inconsistent
metadata on the host before launching anything (no GPU needed: validation
returns before the first CUDA call)."""
import ctypes
import os
import re

import numpy as np
import pytest

import paged_kv_attention_cb_gb300 as cb
from paged_kv_attention_cb_gb300 import build as cbbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cbbuild.build()
    return cb.lib()


def declared_functions():
    names = []
    for fname in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fname.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fname)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(cb_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("cb_write_kv", "cb_paged_attention", "cb_workspace_size",
                     "cb_status_string", "cb_last_cuda_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_exports_are_plain_c_symbols(lib):
    nm = os.popen(f"nm -D --defined-only {cbbuild.LIB_PATH}").read()
    for n in declared_functions():
        assert re.search(rf"\bT {n}$", nm, flags=re.M), n


def test_status_strings_and_version(lib):
    assert lib.cb_abi_version() == 1
    for s in range(7):
        assert lib.cb_status_string(s)
    assert lib.cb_status_string(99) == b"unknown status"


def test_workspace_size_is_monotone(lib):
    a = lib.cb_workspace_size(4, 10, 4, 2, 64)
    b = lib.cb_workspace_size(64, 64, 32, 8, 128)
    c = lib.cb_workspace_size(128, 64, 32, 8, 128)
    assert 256 <= a < b < c


FAKE = 0x100000  # 16-byte aligned, never dereferenced: validation fails first


def call_attention(lib, qsl, seq, *, T=None, R=None, NB=40, BS=16, Hq=4, Hkv=2, D=64, dtype=0,
                   stride=None, ws_bytes=None, scale=0.0, window=0, workspace=FAKE, out=FAKE,
                   hq_ptr=True):
    qsl = np.ascontiguousarray(qsl, dtype=np.int32)
    seq = np.ascontiguousarray(seq, dtype=np.int32)
    R = len(seq) if R is None else R
    T = int(qsl[-1]) if T is None else T
    if stride is None:
        stride = max(1, int(max((seq + BS - 1) // BS))) if len(seq) else 1
    if ws_bytes is None:
        ws_bytes = lib.cb_workspace_size(R, T, Hq, Hkv, D)
    hq = qsl.ctypes.data_as(ctypes.c_void_p) if hq_ptr else None
    return lib.cb_paged_attention(out, FAKE, FAKE, FAKE, None, None, None, FAKE, FAKE, FAKE, stride,
                                  hq, seq.ctypes.data_as(ctypes.c_void_p), R, T, NB, BS, Hq, Hkv, D,
                                  scale, window, dtype, 0, workspace, ws_bytes, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(qsl=[1, 2], seq=[3]), 2),                    # query_start_loc[0] != 0
    (dict(qsl=[0, 3, 2], seq=[5, 5]), 2),              # decreasing
    (dict(qsl=[0, 4], seq=[3]), 2),                    # q_len > seq_len
    (dict(qsl=[0, 2], seq=[40], stride=2), 2),         # stride < ceil(40/16)
    (dict(qsl=[0, 2], seq=[4], T=3), 2),               # qsl[R] != T
    (dict(qsl=[0, 2], seq=[4], D=96), 3),              # head_dim
    (dict(qsl=[0, 2], seq=[4], Hq=6, Hkv=2), 3),       # G = 3
    (dict(qsl=[0, 2], seq=[4], Hq=5, Hkv=2), 1),       # Hq % Hkv
    (dict(qsl=[0, 2], seq=[4], BS=12), 3),             # block size not a power of two
    (dict(qsl=[0, 2], seq=[4], dtype=7), 1),           # dtype
    (dict(qsl=[0, 2], seq=[4], ws_bytes=16), 4),       # workspace too small
    (dict(qsl=[0, 2], seq=[4], workspace=None), 4),    # no workspace
    (dict(qsl=[0, 2], seq=[4], hq_ptr=False), 1),      # host mirror missing
    (dict(qsl=[0, 2], seq=[4], out=None), 1),          # null out
    (dict(qsl=[0, 2], seq=[4], NB=0), 1),              # empty pool
])
def test_host_validation_rejects(lib, kwargs, status):
    assert call_attention(lib, **kwargs) == status
    assert lib.cb_last_error_message()


def test_empty_step_is_a_no_op(lib):
    # T = 0: validated, nothing launched, OK without a GPU.
    assert call_attention(lib, qsl=[0, 0], seq=[7]) == 0
    assert call_attention(lib, qsl=[0], seq=[], R=0, stride=1) == 0


def test_write_kv_validation(lib):
    st = lib.cb_write_kv(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 10, 16, 1, 60, 1, None, None)
    assert st == 3  # 1 * 60 * 2 bytes is not a multiple of 16
    st = lib.cb_write_kv(None, FAKE, FAKE, FAKE, FAKE, 4, 10, 16, 2, 64, 1, None, None)
    assert st == 1
    st = lib.cb_write_kv(FAKE + 8, FAKE, FAKE, FAKE, FAKE, 4, 10, 16, 2, 64, 1, None, None)
    assert st == 1
    assert lib.cb_write_kv(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 10, 16, 2, 64, 1, None, None) == 0


def test_binding_raises_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(cb, "_LIB", None)
    monkeypatch.setenv("CB_LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        cb.lib()


def call_ring(lib, qsl, seq, ring, *, window=64, BS=16, stride=None, NB=40, Hq=4, Hkv=2, D=64):
    qsl = np.ascontiguousarray(qsl, dtype=np.int32)
    seq = np.ascontiguousarray(seq, dtype=np.int32)
    R, T = len(seq), int(qsl[-1])
    stride = ring if stride is None else stride
    return lib.cb_paged_attention_ring(
        FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE, FAKE, FAKE, stride, ring,
        qsl.ctypes.data_as(ctypes.c_void_p), seq.ctypes.data_as(ctypes.c_void_p), R, T, NB, BS,
        Hq, Hkv, D, 0.0, window, 0, 0, FAKE, lib.cb_workspace_size(R, T, Hq, Hkv, D), None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(qsl=[0, 1], seq=[1000], ring=0), 1),                  # no ring
    (dict(qsl=[0, 1], seq=[1000], ring=5, window=0), 1),        # a ring needs a window
    (dict(qsl=[0, 1], seq=[1000], ring=5, stride=4), 2),        # row shorter than the ring
    (dict(qsl=[0, 1], seq=[1000], ring=4, window=64), 2),       # window 64 spans 5 blocks here
    (dict(qsl=[0, 40], seq=[1000], ring=6, window=64), 2),      # + 40 new tokens: 7 blocks
    (dict(qsl=[0, 0], seq=[1000], ring=4, window=64), 2),       # checked even with T = 0
])
def test_ring_validation_rejects(lib, kwargs, status):
    assert call_ring(lib, **kwargs) == status
    assert lib.cb_last_error_message()


def test_ring_validation_accepts_exact_fit(lib):
    # T = 0 (nothing to launch): a request at 1000 positions, window 64, reads blocks
    # 58..62, so a ring of 5 pages fits; 40 new tokens after 960 positions span 56..62
    assert call_ring(lib, qsl=[0, 0], seq=[1000], ring=5, window=64) == 0
    assert call_ring(lib, qsl=[0, 0], seq=[1000], ring=7, window=104) == 0


# ------------------------------------------------------------------ CUDA-graph cache (host side)


def test_graph_cache_lifecycle(lib):
    h = ctypes.c_void_p()
    assert lib.cb_graph_cache_create(64, 0, ctypes.byref(h)) == 0 and h.value
    g, c, r = ctypes.c_int64(-1), ctypes.c_int64(-1), ctypes.c_int64(-1)
    assert lib.cb_graph_cache_stats(h, ctypes.byref(g), ctypes.byref(c), ctypes.byref(r)) == 0
    assert (g.value, c.value, r.value) == (0, 0, 0)
    lib.cb_graph_cache_destroy(h)
    bad = ctypes.c_void_p()
    assert lib.cb_graph_cache_create(0, 0, ctypes.byref(bad)) == 1 and not bad.value
    assert lib.cb_graph_cache_create(8, -1, ctypes.byref(bad)) == 1


def call_graphed(lib, cache, qsl, seq, T, stream=FAKE, Hq=4, Hkv=2, D=64, BS=16):
    qsl = np.ascontiguousarray(qsl, dtype=np.int32)
    seq = np.ascontiguousarray(seq, dtype=np.int32)
    R = len(seq)
    stride = max(1, int(max((seq + BS - 1) // BS)))
    return lib.cb_paged_attention_graphed(
        cache, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE, FAKE, FAKE, stride,
        qsl.ctypes.data_as(ctypes.c_void_p), seq.ctypes.data_as(ctypes.c_void_p), R, T, 40, BS,
        Hq, Hkv, D, 0.0, 0, 1, 0, FAKE, lib.cb_workspace_size(R, T, Hq, Hkv, D), stream)


def test_graphed_validation_rejects_before_any_launch(lib):
    h = ctypes.c_void_p()
    assert lib.cb_graph_cache_create(4, 0, ctypes.byref(h)) == 0
    try:
        assert call_graphed(lib, None, [0, 1, 2, 2, 2], [5, 9, 0, 0], T=4) == 1   # no cache
        assert call_graphed(lib, h, [0, 1, 2, 2], [5, 9, 0], T=4) == 1            # R not padded
        assert call_graphed(lib, h, [0, 1, 2, 2, 2], [5, 9, 0, 0], T=6) == 1      # T not padded
        assert call_graphed(lib, h, [0, 1, 5, 5, 5], [5, 9, 0, 0], T=4) == 2      # qsl[R] > T
        assert call_graphed(lib, h, [0, 1, 2, 2, 2], [5, 9, 0, 0], T=4, stream=None) == 1
        g = ctypes.c_int64(-1)
        assert lib.cb_graph_cache_stats(h, ctypes.byref(g), None, None) == 0 and g.value == 0
    finally:
        lib.cb_graph_cache_destroy(h)
