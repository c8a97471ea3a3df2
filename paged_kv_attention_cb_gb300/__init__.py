"""Python binding of libcb (C ABI in include/cb.h): argument marshalling only.

Every step of the attention path runs in the library's CUDA kernels; this
module only turns torch tensors into device pointers and sizes, passes the
caller's current CUDA stream, and raises ``CbError`` on a non-OK status. If
libcb.so has not been built, every call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import LIB_PATH

CB_F32 = 0
CB_BF16 = 1
CB_FLAG_PORTABLE_ONLY = 0x1
CB_FLAG_TEST_WAIT_EXPIRY = 0x2  # tests of the failure path only (see include/cb.h)
CB_DEVERR_BLOCK_ID = 0x1
CB_DEVERR_SLOT = 0x2
CB_DEVERR_TIMEOUT = 0x4

STATUS = {0: "CB_OK", 1: "CB_ERR_INVALID_ARG", 2: "CB_ERR_METADATA", 3: "CB_ERR_UNSUPPORTED",
          4: "CB_ERR_WORKSPACE", 5: "CB_ERR_CUDA", 6: "CB_ERR_DEVICE_CHECK"}


class CbError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_LIB = None

_i32 = ctypes.c_int32
_vp = ctypes.c_void_p
_SIGNATURES = {
    "cb_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "cb_last_error_message": (ctypes.c_char_p, []),
    "cb_last_cuda_error": (ctypes.c_int, []),
    "cb_abi_version": (ctypes.c_int, []),
    "cb_write_kv": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                   _vp, _vp]),
    "cb_copy_blocks": (ctypes.c_int, [_vp, _vp, _vp, _vp, ctypes.c_int64, ctypes.c_int64, _vp,
                                      _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp]),
    "cb_workspace_size": (ctypes.c_size_t, [_i32, _i32, _i32, _i32, _i32]),
    "cb_workspace_init": (ctypes.c_int, [_vp, ctypes.c_size_t, _vp]),
    "cb_paged_attention": (ctypes.c_int, [
        _vp, _vp, _vp, _vp,            # out, q, k_cache, v_cache
        _vp, _vp, _vp,                 # k_new, v_new, slot_mapping
        _vp, _vp, _vp, _i32,           # query_start_loc, seq_lens, block_table, stride
        _vp, _vp,                      # host mirrors
        _i32, _i32, _i32, _i32,        # R, T, num_blocks, block_size
        _i32, _i32, _i32,              # Hq, Hkv, D
        ctypes.c_float, _i32, _i32,    # scale, sliding_window, dtype
        ctypes.c_uint32, _vp, ctypes.c_size_t, _vp]),  # flags, workspace, bytes, stream
    "cb_paged_attention_ring": (ctypes.c_int, [
        _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32,  # ... stride, ring_blocks
        _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
        ctypes.c_float, _i32, _i32, ctypes.c_uint32, _vp, ctypes.c_size_t, _vp]),
    "cb_graph_cache_create": (ctypes.c_int, [_i32, _i32, ctypes.POINTER(ctypes.c_void_p)]),
    "cb_graph_cache_destroy": (None, [_vp]),
    "cb_graph_cache_stats": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_int64),
                                            ctypes.POINTER(ctypes.c_int64),
                                            ctypes.POINTER(ctypes.c_int64)]),
    "cb_paged_attention_graphed": (ctypes.c_int, [_vp] + [
        _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp,
        _i32, _i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_float, _i32, _i32, ctypes.c_uint32,
        _vp, ctypes.c_size_t, _vp]),
    "cb_read_error_word": (ctypes.c_int, [_vp, _vp, _vp]),
    "cb_no_alloc_read_error_word": (ctypes.c_int, [_vp, _vp]),
    "cb_paged_attention_no_alloc": (ctypes.c_int, [
        _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp,
        _i32, _i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_float, _i32, _i32, ctypes.c_uint32,
        _vp]),
    "cb_launch_count": (ctypes.c_longlong, [ctypes.c_int]),
    "cb_num_kernels": (ctypes.c_int, []),
    "cb_kernel_name": (ctypes.c_char_p, [ctypes.c_int]),
    "cb_kernel_timing": (ctypes.c_int, [ctypes.c_int]),
    "cb_kernel_timing_collect": (ctypes.c_int, [_vp, _vp, ctypes.c_int]),
}


def lib_path() -> str:
    return os.environ.get("CB_LIB", LIB_PATH)


def lib() -> ctypes.CDLL:
    """The loaded libcb.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libcb.so not built at {path}: run paged_kv_attention_cb_gb300.build")
        handle = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB


def _check(status: int):
    if status != 0:
        msg = lib().cb_last_error_message().decode()
        raise CbError(status, msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch

        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.float32:
        return CB_F32
    if t.dtype == torch.bfloat16:
        return CB_BF16
    raise CbError(1, f"unsupported dtype {t.dtype}")


def _host_i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def write_kv(k_new, v_new, k_cache, v_cache, slot_mapping, error_word=None, stream=None):
    """Scatter k_new/v_new [T, Hkv, D] into the caches [NB, BS, Hkv, D] at slot_mapping [T]."""
    T, Hkv, D = k_new.shape
    NB, BS = k_cache.shape[0], k_cache.shape[1]
    _check(lib().cb_write_kv(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                             _ptr(slot_mapping), T, NB, BS, Hkv, D, _dtype_code(k_new),
                             _ptr(error_word), _stream(stream)))


def copy_blocks(k_src, v_src, k_dst, v_dst, src_ids, dst_ids, error_word=None, stream=None):
    """Block dst_ids[i] of k_dst/v_dst [NBd, BS, Hkv, D] = block src_ids[i] of k_src/v_src."""
    NBs, BS, Hkv, D = k_src.shape
    n = int(src_ids.numel())
    if int(dst_ids.numel()) != n or tuple(k_dst.shape[1:]) != (BS, Hkv, D):
        raise ValueError("copy_blocks: id counts or block shapes differ")
    _check(lib().cb_copy_blocks(_ptr(k_src), _ptr(v_src), _ptr(k_dst), _ptr(v_dst), NBs,
                                k_dst.shape[0], _ptr(src_ids), _ptr(dst_ids), n, BS, Hkv, D,
                                _dtype_code(k_src), _ptr(error_word), _stream(stream)))


def workspace_size(num_requests, num_tokens, num_q_heads, num_kv_heads, head_dim) -> int:
    return int(lib().cb_workspace_size(num_requests, num_tokens, num_q_heads, num_kv_heads,
                                       head_dim))


def workspace_init(workspace, stream=None):
    _check(lib().cb_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _stream(stream)))


def read_error_word(workspace, stream=None) -> int:
    """Synchronise, return and clear the device error word (0 = no error recorded)."""
    word = ctypes.c_int32(0)
    status = lib().cb_read_error_word(_ptr(workspace), ctypes.byref(word), _stream(stream))
    if status not in (0, 6):
        _check(status)
    return int(word.value)


def paged_attention(out, q, k_cache, v_cache, query_start_loc, seq_lens, block_table,
                    h_query_start_loc, h_seq_lens, workspace, *, scale=0.0, sliding_window=0,
                    k_new=None, v_new=None, slot_mapping=None, flags=0, stream=None,
                    ring_blocks=0):
    """One ragged paged-attention step (see cb_paged_attention in include/cb.h).

    out, q: [T, Hq, D]; caches [NB, BS, Hkv, D]; device metadata int32 (slot_mapping
    int64); h_query_start_loc / h_seq_lens: host copies of the same metadata.
    ring_blocks > 0: a sliding-window layer whose pages are recycled in a ring
    (cb_paged_attention_ring): logical block b at block_table[r, b % ring_blocks].
    """
    T, Hq, D = q.shape
    NB, BS, Hkv, _ = k_cache.shape
    R = int(seq_lens.shape[0])
    hq = _host_i32(h_query_start_loc)
    hs = _host_i32(h_seq_lens)
    if hq.shape[0] != R + 1 or hs.shape[0] != R:
        raise CbError(2, "host mirrors must have R+1 and R entries")
    stride = int(block_table.shape[1]) if block_table.dim() == 2 else 0
    head = (_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
            _ptr(slot_mapping), _ptr(query_start_loc), _ptr(seq_lens), _ptr(block_table), stride)
    tail = (hq.ctypes.data_as(ctypes.c_void_p), hs.ctypes.data_as(ctypes.c_void_p),
            R, T, NB, BS, Hq, Hkv, D, float(scale), int(sliding_window), _dtype_code(q),
            int(flags), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream(stream))
    if ring_blocks:
        _check(lib().cb_paged_attention_ring(*head, int(ring_blocks), *tail))
    else:
        _check(lib().cb_paged_attention(*head, *tail))
    return out


class GraphCache:
    """CUDA graphs of the step, one per padded shape (cb_graph_cache in include/cb.h)."""

    def __init__(self, q_interval=64, kv_interval=0):
        h = ctypes.c_void_p()
        _check(lib().cb_graph_cache_create(int(q_interval), int(kv_interval), ctypes.byref(h)))
        self._h = h
        self.q_interval = int(q_interval)

    def close(self):
        if self._h:
            lib().cb_graph_cache_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def stats(self):
        g, c, r = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(lib().cb_graph_cache_stats(self._h, ctypes.byref(g), ctypes.byref(c),
                                          ctypes.byref(r)))
        return {"graphs": g.value, "captures": c.value, "replays": r.value}


def paged_attention_graphed(cache, out, q, k_cache, v_cache, query_start_loc, seq_lens,
                            block_table, h_query_start_loc, h_seq_lens, workspace, *, scale=0.0,
                            sliding_window=0, k_new=None, v_new=None, slot_mapping=None, flags=0,
                            stream=None):
    """paged_attention through a GraphCache: the buffers hold the padded shape (R and T
    multiples of the cache's q_interval; padding requests q_len 0 / seq_len 0, padding
    tokens past query_start_loc[R] with slot -1)."""
    T, Hq, D = q.shape
    NB, BS, Hkv, _ = k_cache.shape
    R = int(seq_lens.shape[0])
    hq = _host_i32(h_query_start_loc)
    hs = _host_i32(h_seq_lens)
    if hq.shape[0] != R + 1 or hs.shape[0] != R:
        raise CbError(2, "host mirrors must have R+1 and R entries")
    stride = int(block_table.shape[1]) if block_table.dim() == 2 else 0
    _check(lib().cb_paged_attention_graphed(
        cache._h, _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
        _ptr(slot_mapping), _ptr(query_start_loc), _ptr(seq_lens), _ptr(block_table), stride,
        hq.ctypes.data_as(ctypes.c_void_p), hs.ctypes.data_as(ctypes.c_void_p),
        R, T, NB, BS, Hq, Hkv, D, float(scale), int(sliding_window), _dtype_code(q), int(flags),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


class PreparedGraphStep:
    """paged_attention_graphed with the argument marshalling done once.

    For a serving loop over persistent buffers: the caller writes each step's inputs
    into the same device tensors and the same host-mirror arrays (numpy int32,
    updated in place), then calls the object; each call is one C call (a replay, or a
    capture for a new padded shape). The padded counts R and T are fixed by the
    tensors' shapes.
    """

    def __init__(self, cache, out, q, k_cache, v_cache, query_start_loc, seq_lens, block_table,
                 h_query_start_loc, h_seq_lens, workspace, *, scale=0.0, sliding_window=0,
                 k_new=None, v_new=None, slot_mapping=None, flags=0, stream=None):
        import numpy as np

        T, Hq, D = q.shape
        NB, BS, Hkv, _ = k_cache.shape
        R = int(seq_lens.shape[0])
        for h, n in ((h_query_start_loc, R + 1), (h_seq_lens, R)):
            if not (isinstance(h, np.ndarray) and h.dtype == np.int32 and h.flags.c_contiguous
                    and h.shape == (n,)):
                raise ValueError("host mirrors must be contiguous int32 numpy arrays of R+1 / R")
        self._keep = (cache, out, q, k_cache, v_cache, query_start_loc, seq_lens, block_table,
                      h_query_start_loc, h_seq_lens, workspace, k_new, v_new, slot_mapping)
        stride = int(block_table.shape[1]) if block_table.dim() == 2 else 0
        self._fn = lib().cb_paged_attention_graphed
        self._args = (
            cache._h, _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
            _ptr(slot_mapping), _ptr(query_start_loc), _ptr(seq_lens), _ptr(block_table), stride,
            h_query_start_loc.ctypes.data_as(ctypes.c_void_p),
            h_seq_lens.ctypes.data_as(ctypes.c_void_p), R, T, NB, BS, Hq, Hkv, D, float(scale),
            int(sliding_window), _dtype_code(q), int(flags), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream))

    def __call__(self):
        status = self._fn(*self._args)
        if status != 0:
            _check(status)


NO_ALLOC_SCRATCH_BYTES = 8 << 20


def paged_attention_no_alloc(out, q, k_cache, v_cache, query_start_loc, seq_lens, block_table,
                             h_query_start_loc, h_seq_lens, *, scale=0.0, sliding_window=0,
                             k_new=None, v_new=None, slot_mapping=None, flags=0, stream=None):
    """paged_attention without a workspace, for callers that may not allocate device memory
    at call time (see cb_paged_attention_no_alloc in include/cb.h)."""
    T, Hq, D = q.shape
    NB, BS, Hkv, _ = k_cache.shape
    R = int(seq_lens.shape[0])
    hq = _host_i32(h_query_start_loc)
    hs = _host_i32(h_seq_lens)
    if hq.shape[0] != R + 1 or hs.shape[0] != R:
        raise CbError(2, "host mirrors must have R+1 and R entries")
    stride = int(block_table.shape[1]) if block_table.dim() == 2 else 0
    _check(lib().cb_paged_attention_no_alloc(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
        _ptr(slot_mapping), _ptr(query_start_loc), _ptr(seq_lens), _ptr(block_table), stride,
        hq.ctypes.data_as(ctypes.c_void_p), hs.ctypes.data_as(ctypes.c_void_p),
        R, T, NB, BS, Hq, Hkv, D, float(scale), int(sliding_window), _dtype_code(q), int(flags),
        _stream(stream)))
    return out


def no_alloc_read_error_word(stream=None) -> int:
    """Synchronise, return and clear the error word of paged_attention_no_alloc on the
    current device (0 = no error recorded)."""
    word = ctypes.c_int32(0)
    status = lib().cb_no_alloc_read_error_word(ctypes.byref(word), _stream(stream))
    if status not in (0, 6):
        _check(status)
    return int(word.value)


def launch_count(kernel: int = -1) -> int:
    """Kernels launched by libcb in this process (all kernels when kernel < 0)."""
    return int(lib().cb_launch_count(kernel))


def kernel_names():
    n = lib().cb_num_kernels()
    return [lib().cb_kernel_name(k).decode() for k in range(n)]


def kernel_timing(enable: bool):
    _check(lib().cb_kernel_timing(1 if enable else 0))


def kernel_timing_collect():
    """{kernel name: (total ms, launches)} since the previous collect (synchronises)."""
    n = lib().cb_num_kernels()
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_longlong * n)()
    _check(lib().cb_kernel_timing_collect(ms, cnt, n))
    names = kernel_names()
    return {names[k]: (float(ms[k]), int(cnt[k])) for k in range(n) if cnt[k]}


def alloc_workspace(num_requests, num_tokens, num_q_heads, num_kv_heads, head_dim, device="cuda"):
    """Allocate (with torch) and zero a workspace of cb_workspace_size bytes."""
    import torch

    n = workspace_size(num_requests, num_tokens, num_q_heads, num_kv_heads, head_dim)
    return torch.zeros((n + 15) // 16 * 16, dtype=torch.uint8, device=device)
