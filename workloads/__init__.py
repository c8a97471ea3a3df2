"""Seeded synthetic inputs for one continuous-batching attention step.

This module is shared by the tests, the bench and the oracle's checks, and it
holds no part of the attention arithmetic. It draws random tensors and builds
the per-step metadata the way a scheduler hands it to the attention backend
("Continuous Batching", languisher.top, section "Extension: the vLLM v1
implementation": the scheduler builds query_start_loc, seq_lens, slot_mapping
and block_table before the kernel runs).

Conventions (readings of what the pages leave open; the cache layout and the query_start_loc
length follow the same section of "Continuous Batching"):

* q is ``[T, Hq, D]``, k_new/v_new are ``[T, Hkv, D]``, the caches are
  ``[num_blocks, block_size, Hkv, D]`` (K and V in separate tensors).
* query_start_loc has R+1 entries, the last one equal to T.
* seq_lens[r] is the KV length of request r *including* this step's tokens,
  so its context is ``seq_lens[r] - q_len[r]``.
* Pages 0 and 1 are reserved for padding and never appear in a block table
  ("Continuous batching architecture", section "Memory management").
* Unused block-table tail entries hold 0.
* Every page of the pool, reserved or not, starts out N(0, 1): the KV of a
  request's context is simply whatever its block-table pages hold.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

RESERVED_PAGES = 2


@dataclasses.dataclass
class StepSpec:
    """Metadata of one step (host, numpy) plus the recipe for its tensors."""

    name: str
    dtype: str  # "f32" or "bf16"
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    q_lens: np.ndarray  # int32 [R]
    ctx_lens: np.ndarray  # int32 [R]
    query_start_loc: np.ndarray  # int32 [R+1]
    seq_lens: np.ndarray  # int32 [R]
    block_table: np.ndarray  # int32 [R, bt_stride]
    slot_mapping: np.ndarray  # int64 [T]
    scale: float
    sliding_window: int = 0
    seed: int = 0
    q_std: float = 1.0  # Q ~ N(0, q_std^2); K, V ~ N(0, 1)
    ring_blocks: int = 0  # > 0: sliding layer, logical block b at block_table[r, b % ring_blocks]

    @property
    def R(self) -> int:
        return int(self.q_lens.shape[0])

    @property
    def T(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def bt_stride(self) -> int:
        return int(self.block_table.shape[1])

    def kv_tokens_attended(self) -> int:
        """Number of distinct KV positions the step's queries read, per request once."""
        total = 0
        for r in range(self.R):
            ql = int(self.q_lens[r])
            if ql == 0:
                continue
            ctx = int(self.ctx_lens[r])
            hi = ctx + ql - 1
            lo = 0 if self.sliding_window <= 0 else max(0, ctx - self.sliding_window + 1)
            total += hi - lo + 1
        return total

    def elt_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


def build_metadata(q_lens, ctx_lens, block_size, rng, pool_factor=1.2, num_blocks=None):
    """Assign pages to requests and derive query_start_loc / seq_lens / block_table / slot_mapping.

    Pages are handed out from a seeded permutation of the free pool in request
    order, so logical neighbours are scattered across HBM. The pool holds
    ``pool_factor`` times the pages needed (free holes) plus the reserved pages.
    """
    q_lens = np.asarray(q_lens, dtype=np.int32)
    ctx_lens = np.asarray(ctx_lens, dtype=np.int32)
    R = q_lens.shape[0]
    seq_lens = (ctx_lens + q_lens).astype(np.int32)
    pages_per_req = [(int(s) + block_size - 1) // block_size for s in seq_lens]
    needed = sum(pages_per_req)
    if num_blocks is None:
        num_blocks = RESERVED_PAGES + int(math.ceil(pool_factor * needed))
    free = np.arange(RESERVED_PAGES, num_blocks, dtype=np.int64)
    if needed > free.shape[0]:
        raise ValueError("pool too small")
    perm = rng.permutation(free)
    bt_stride = max(1, max(pages_per_req) if R else 1)
    block_table = np.zeros((R, bt_stride), dtype=np.int32)
    cursor = 0
    for r in range(R):
        n = pages_per_req[r]
        block_table[r, :n] = perm[cursor:cursor + n]
        cursor += n
    qsl = np.zeros(R + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(q_lens)
    T = int(qsl[-1])
    slot_mapping = np.empty(T, dtype=np.int64)
    for r in range(R):
        for i in range(int(q_lens[r])):
            pos = int(ctx_lens[r]) + i
            slot_mapping[qsl[r] + i] = (int(block_table[r, pos // block_size]) * block_size
                                        + pos % block_size)
    return qsl, seq_lens, block_table, slot_mapping, int(num_blocks)


def custom(q_lens, ctx_lens, *, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
           dtype="bf16", seed=0, scale=None, sliding_window=0, pool_factor=1.2, q_std=1.0,
           num_blocks=None, name="custom") -> StepSpec:
    rng = np.random.default_rng(seed)
    qsl, seq_lens, bt, slots, nb = build_metadata(q_lens, ctx_lens, block_size, rng,
                                                  pool_factor=pool_factor, num_blocks=num_blocks)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return StepSpec(name=name, dtype=dtype, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                    head_dim=head_dim, block_size=block_size, num_blocks=nb,
                    q_lens=np.asarray(q_lens, np.int32), ctx_lens=np.asarray(ctx_lens, np.int32),
                    query_start_loc=qsl, seq_lens=seq_lens, block_table=bt, slot_mapping=slots,
                    scale=float(scale), sliding_window=int(sliding_window), seed=seed, q_std=q_std)


def share_prefix_pages(spec: StepSpec, donor: int, recipient: int, n_pages: int) -> StepSpec:
    """The same step with request ``recipient``'s first ``n_pages`` block-table entries
    pointing at request ``donor``'s first pages: a shared prompt prefix held once in the
    pool ("Continuous batching architecture", section "Prefix caching": full blocks
    shared between requests with the same prefix). Only full context blocks of both
    requests may be shared, so no new token of the step is written into a shared page."""
    bs = spec.block_size
    if n_pages * bs > min(int(spec.ctx_lens[donor]), int(spec.ctx_lens[recipient])):
        raise ValueError("only full context blocks can be shared")
    bt = spec.block_table.copy()
    bt[recipient, :n_pages] = bt[donor, :n_pages]
    return StepSpec(**{**spec.__dict__, "block_table": bt,
                       "name": f"{spec.name}_shared{donor}to{recipient}x{n_pages}"})


def ring_step(q_lens, ctx_lens, window, *, ring_blocks=None, num_q_heads=32, num_kv_heads=8,
              head_dim=128, block_size=16, dtype="bf16", seed=0, scale=None, pool_factor=1.2,
              q_std=1.0, name="ring") -> StepSpec:
    """A step of a sliding-window layer whose pages are recycled in a ring per request
    ("Continuous batching architecture", section "Memory management": sliding layers
    keep a fixed window of recent tokens by reusing a small number of pages).

    Each request owns ``ring_blocks`` pages (default: the fewest that hold every
    position the step reads or writes, from the first query's window start to the
    last new token); logical block b lives in ring entry b % ring_blocks, and the
    step's new tokens are scattered through the same mapping. Pages come from a
    seeded permutation of the pool."""
    q_lens = np.asarray(q_lens, dtype=np.int32)
    ctx_lens = np.asarray(ctx_lens, dtype=np.int32)
    R = q_lens.shape[0]
    seq = (ctx_lens + q_lens).astype(np.int32)
    lo = np.maximum(0, ctx_lens - window + 1)
    span = [int((seq[r] - 1) // block_size - lo[r] // block_size + 1) for r in range(R)]
    ring = int(ring_blocks or max(span))
    if ring < max(span):
        raise ValueError("ring too small for the window and the step's tokens")
    rng = np.random.default_rng(seed)
    num_blocks = RESERVED_PAGES + int(math.ceil(pool_factor * R * ring))
    perm = rng.permutation(np.arange(RESERVED_PAGES, num_blocks))
    bt = perm[:R * ring].reshape(R, ring).astype(np.int32)
    qsl = np.zeros(R + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(q_lens)
    slots = np.empty(int(qsl[-1]), dtype=np.int64)
    for r in range(R):
        for i in range(int(q_lens[r])):
            p = int(ctx_lens[r]) + i
            slots[qsl[r] + i] = int(bt[r, (p // block_size) % ring]) * block_size + p % block_size
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return StepSpec(name=name, dtype=dtype, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                    head_dim=head_dim, block_size=block_size, num_blocks=num_blocks,
                    q_lens=q_lens, ctx_lens=ctx_lens, query_start_loc=qsl, seq_lens=seq,
                    block_table=bt, slot_mapping=slots, scale=float(scale),
                    sliding_window=int(window), seed=seed, q_std=q_std, ring_blocks=ring)


def long_decode_ring(seed: int = 3, window: int = 4096) -> StepSpec:
    """long_decode_window on a sliding layer with ring-recycled pages: 16 requests at
    seq_len 32768, window 4096 (positions 28672..32767): 256 pages of 16 tokens per request
    instead of 2048."""
    return ring_step(np.ones(16, np.int32), np.full(16, 32767, np.int32), window, num_q_heads=64,
                     num_kv_heads=8, seed=seed, name=f"long_decode_16x32768_window{window}_ring")


def tiny_mixed(seed: int = 0) -> StepSpec:
    """Tiny mixed step, fp32: prefill (4,0), prefill (2,0), chunk (3, ctx 5), decode (1, ctx 8).

    Heads 4 Q / 2 KV, head_dim 64, block_size 2, a 40-page pool with pages
    0-1 reserved; the 12 pages needed come from a seeded permutation of pages
    2..39, handed out in request order.
    """
    return custom([4, 2, 3, 1], [0, 0, 5, 8], num_q_heads=4, num_kv_heads=2, head_dim=64,
                  block_size=2, dtype="f32", seed=seed, num_blocks=40, name="tiny_mixed_f32")


def decode_step(seed: int = 1, R: int = 64, lo: int = 128, hi: int = 2048) -> StepSpec:
    """Pure decode: R requests, q_len 1, seq_len ~ U{lo..hi}; 32 Q / 8 KV heads, D 128, BS 16.

    Q ~ N(0,1)/sqrt(128) with scale 1.0 (the 1/sqrt(D) factor is already in Q).
    """
    rng = np.random.default_rng(seed)
    seq = rng.integers(lo, hi, endpoint=True, size=R)
    return custom(np.ones(R, np.int32), (seq - 1).astype(np.int32), seed=seed, scale=1.0,
                  q_std=1.0 / math.sqrt(128.0), name=f"decode_{R}x[{lo},{hi}]_bf16")


def mixed_step(seed: int = 2) -> StepSpec:
    """Mixed step under max_batch_tokens=2048: 128 decodes (ctx ~ U{256..4096}),
    then a 960-token chunk at ctx 0, then a 960-token chunk at ctx 3072."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(256, 4096, endpoint=True, size=128)
    q_lens = np.concatenate([np.ones(128, np.int32), [960, 960]]).astype(np.int32)
    ctx_lens = np.concatenate([ctx, [0, 3072]]).astype(np.int32)
    return custom(q_lens, ctx_lens, seed=seed, name="mixed_128dec+2x960_bf16")


def long_decode(seed: int = 3, window: int = 0) -> StepSpec:
    """Long-context decode: 16 requests at seq_len 32768, 64 Q / 8 KV heads, D 128, BS 16,
    with 20% free holes in a globally shuffled pool; optional sliding window."""
    name = "long_decode_16x32768_bf16" + (f"_window{window}" if window > 0 else "")
    return custom(np.ones(16, np.int32), np.full(16, 32767, np.int32), num_q_heads=64,
                  num_kv_heads=8, seed=seed, sliding_window=window, name=name)


# ---------------------------------------------------------------- tensors


def draw_tensors(spec: StepSpec, device="cpu"):
    """Draw q, k_new, v_new and the whole K/V pool with a seeded torch generator.

    Returns a dict of torch tensors in the step's dtype on ``device``.
    """
    import torch

    tdt = torch.float32 if spec.dtype == "f32" else torch.bfloat16
    g = torch.Generator(device=device)
    g.manual_seed(int(spec.seed) * 1000003 + 12345)
    T, Hq, Hkv, D = spec.T, spec.num_q_heads, spec.num_kv_heads, spec.head_dim

    def randn(shape, std=1.0):
        out = torch.empty(shape, dtype=tdt, device=device)
        flat = out.view(-1)
        n = flat.numel()
        chunk = 1 << 26
        for s in range(0, n, chunk):
            e = min(n, s + chunk)
            x = torch.randn(e - s, generator=g, device=device, dtype=torch.float32)
            if std != 1.0:
                x.mul_(std)
            flat[s:e].copy_(x)
        return out

    q = randn((T, Hq, D), spec.q_std)
    k_new = randn((T, Hkv, D))
    v_new = randn((T, Hkv, D))
    cache_shape = (spec.num_blocks, spec.block_size, Hkv, D)
    k_cache = randn(cache_shape)
    v_cache = randn(cache_shape)
    return dict(q=q, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache)


def metadata_tensors(spec: StepSpec, device="cpu"):
    """Metadata as torch tensors (int32 except slot_mapping int64)."""
    import torch

    return dict(
        query_start_loc=torch.from_numpy(spec.query_start_loc.copy()).to(device),
        seq_lens=torch.from_numpy(spec.seq_lens.copy()).to(device),
        block_table=torch.from_numpy(spec.block_table.copy()).to(device),
        slot_mapping=torch.from_numpy(spec.slot_mapping.copy()).to(device),
    )


def to_f64(t) -> np.ndarray:
    """Exact widening of an fp32/bf16 torch tensor to a float64 numpy array."""
    import torch

    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


CONFIGS = {
    "tiny_mixed": tiny_mixed,
    "decode": decode_step,
    "mixed": mixed_step,
    "long_decode": long_decode,
    "long_decode_window": lambda seed=3: long_decode(seed, window=4096),
    "long_decode_ring": long_decode_ring,
}


def by_name(name: str, seed: Optional[int] = None) -> StepSpec:
    fn = CONFIGS[name]
    return fn() if seed is None else fn(seed)
