"""CPU oracle for one continuous-batching attention step over a paged KV cache.

TEST INFRASTRUCTURE ONLY. Only the tests, the package's smoke check and the
bench's CPU-baseline leg may import this module. The product path (the C-ABI
library and its Python binding) never calls it, and it shares no code with
the CUDA kernels.

Everything here is plain and slow on purpose: a per-request loop that gathers
each request's KV positions through its block table, then, for every query
row and KV head, a masked softmax over the allowed positions in float64. It
follows these passages:

* "Continuous Batching" (languisher.top), section "Attention Mask
  construction": a token attends only to earlier tokens of its own request
  (block-diagonal causal mask).
* same page, section "Optimisation: the mask as offsets": with request start
  ``start`` and in-request position ``local_pos`` the attended range is
  ``[start, start + local_pos]`` -- nothing is materialised.
* same page, section "Extension: the vLLM v1 implementation": ``q_len =
  query_start_loc[r+1] - query_start_loc[r]``, ``context_len = seq_len -
  q_len``, ``max_kv_pos = context_len + local_q``, every ``kv_pos <=
  max_kv_pos`` is read from ``k_cache[block_table[r][kv_pos // BLOCK_SIZE]]
  [kv_pos % BLOCK_SIZE]``.
* The scheduler-built ``slot_mapping`` is where this step's new K/V go
  (same section). The scatter runs before the attention, because the
  attended range reaches this step's own tokens.

Readings where the pages leave a step open:
an explicit softmax ``scale``; grouped-query heads map to KV head
``h // (Hq // Hkv)``; an optional sliding window keeps the ``W`` most recent
positions up to and including the query's own; a slot below zero is skipped.

Parity pins: the worked example, a dense masked brute force, the causal SDPA
special case, invariants and closed forms, in tests/test_oracle_pins.py. The
value of the softmax scale is a free argument that the pages do not fix
("parity unpinned" for the scale's *value*; its use is pinned by the SDPA
special case).
"""
from __future__ import annotations

import numpy as np


# ------------------------------------------------------------------ scatter


def scatter_kv(k_cache, v_cache, k_new, v_new, slot_mapping):
    """Write token t's new K/V row into flat slot ``slot_mapping[t]`` (in place).

    ``k_cache``/``v_cache`` are ``[num_blocks, block_size, Hkv, D]`` arrays of
    any dtype (bit patterns are copied as they are); a slot below zero is
    skipped. Tokens are written in token order.
    """
    nb, bs, hkv, d = k_cache.shape
    kflat = k_cache.reshape(nb * bs, hkv, d)
    vflat = v_cache.reshape(nb * bs, hkv, d)
    for t in range(slot_mapping.shape[0]):
        s = int(slot_mapping[t])
        if s < 0:
            continue
        kflat[s] = k_new[t]
        vflat[s] = v_new[t]


# ----------------------------------------------------------- index mapping


def copy_blocks(k_dst, v_dst, k_src, v_src, src_ids, dst_ids):
    """Block ``dst_ids[i]`` of the destination caches becomes block ``src_ids[i]`` of the
    source caches (in place, pair by pair in order): the copy behind swapping a
    request's blocks out to CPU memory and back ("Continuous batching mechanics",
    d9bl.com, section "Running out of KV cache memory"; "Continuous batching
    architecture", section "Offloading")."""
    for s, d in zip(np.asarray(src_ids).tolist(), np.asarray(dst_ids).tolist()):
        k_dst[int(d)] = k_src[int(s)]
        v_dst[int(d)] = v_src[int(s)]


def resolve(block_table_row, kv_pos, block_size, ring_blocks=0):
    """Logical position -> (physical block, offset in block).

    With ``ring_blocks > 0`` the row is a ring of recycled pages of a sliding-window
    layer ("Continuous batching architecture", section "Memory management": sliding
    layers keep a fixed window of recent tokens by reusing a few pages): logical
    block b lives in entry ``b % ring_blocks``."""
    b = kv_pos // block_size
    if ring_blocks > 0:
        b %= ring_blocks
    return int(block_table_row[b]), kv_pos % block_size


def kv_range(context_len, local_q, sliding_window):
    """Inclusive range [lo, hi] of logical KV positions that query ``local_q`` attends."""
    hi = context_len + local_q  # max_kv_pos
    lo = 0 if sliding_window <= 0 else max(0, hi - sliding_window + 1)
    return lo, hi


def gather_request_kv(cache, block_table_row, seq_len, block_size, ring_blocks=0):
    """The request's KV in logical order, ``[seq_len, Hkv, D]`` float64, one position at a time.
    (With a ring, positions older than the ring hold whatever recycled them; the window
    never reaches them.)"""
    _, _, hkv, d = cache.shape
    out = np.empty((seq_len, hkv, d), dtype=np.float64)
    for p in range(seq_len):
        blk, off = resolve(block_table_row, p, block_size, ring_blocks)
        out[p] = cache[blk, off]
    return out


# ---------------------------------------------------------------- attention


def softmax_attend(q_heads, K, V, scale):
    """out[h] = sum_j softmax_j(scale * q_h . K_j) * V_j  for each row h of ``q_heads``."""
    s = scale * (q_heads @ K.T)  # [G, n]
    s = s - s.max(axis=1, keepdims=True)
    w = np.exp(s)
    w = w / w.sum(axis=1, keepdims=True)
    return w @ V


def paged_attention(q, k_cache, v_cache, query_start_loc, seq_lens, block_table, block_size,
                    scale, sliding_window=0, rows=None, ring_blocks=0):
    """Attention of every packed query row (or of ``rows`` only) over its request's paged KV.

    q: ``[T, Hq, D]``; caches ``[num_blocks, block_size, Hkv, D]`` (already
    holding this step's new K/V); query_start_loc ``[R+1]``; seq_lens ``[R]``;
    block_table ``[R, stride]``. Returns float64 ``[T, Hq, D]`` (rows not
    requested stay zero).
    """
    q = np.asarray(q, dtype=np.float64)
    T, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    G = Hq // Hkv
    out = np.zeros((T, Hq, D), dtype=np.float64)
    wanted = None if rows is None else set(int(t) for t in rows)
    R = len(seq_lens)
    for r in range(R):
        q_start = int(query_start_loc[r])
        q_end = int(query_start_loc[r + 1])
        q_len = q_end - q_start
        if q_len == 0:
            continue
        my_rows = [t for t in range(q_start, q_end) if wanted is None or t in wanted]
        if not my_rows:
            continue
        seq_len = int(seq_lens[r])
        context_len = seq_len - q_len
        K = gather_request_kv(k_cache, block_table[r], seq_len, block_size, ring_blocks)
        V = gather_request_kv(v_cache, block_table[r], seq_len, block_size, ring_blocks)
        for t in my_rows:
            local_q = t - q_start
            lo, hi = kv_range(context_len, local_q, sliding_window)
            for g in range(Hkv):
                heads = slice(g * G, (g + 1) * G)
                out[t, heads] = softmax_attend(q[t, heads], K[lo:hi + 1, g], V[lo:hi + 1, g], scale)
    return out


def step(q, k_cache, v_cache, k_new, v_new, slot_mapping, query_start_loc, seq_lens, block_table,
         block_size, scale, sliding_window=0, rows=None, ring_blocks=0):
    """One step: scatter the new K/V (on copies of the caches), then attend.

    Returns (out float64 [T, Hq, D], k_cache', v_cache').
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    scatter_kv(kc, vc, k_new, v_new, slot_mapping)
    out = paged_attention(q, kc, vc, query_start_loc, seq_lens, block_table, block_size, scale,
                          sliding_window, rows, ring_blocks)
    return out, kc, vc
