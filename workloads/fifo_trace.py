"""FIFO continuous-batching step trace: the host side that feeds the hot path.

A small scheduler and page allocator, outside the hot path, that turns a seeded
request stream into the per-step metadata the attention step consumes
(query_start_loc, seq_lens, block_table, slot_mapping). It follows
"Continuous batching architecture" (Transformers docs):

* request lifecycle PENDING -> PREFILLING -> DECODING -> FINISHED (section
  "Request lifecycle"); the step that completes a prompt yields the request's
  first output token, so an output of L tokens costs L - 1 decode steps;
* FIFO priority: active decodes first, then active (chunked) prefills, then
  waiting requests in arrival order (section "FIFO");
* budgets: at most ``max_batch_tokens`` query tokens and
  ``max_requests_per_batch`` requests per step; a prompt that does not fit the
  remaining token budget is split into chunks (section "Chunked prefill");
* admission: a waiting request is admitted only while the free share of the
  page pool is at least ``safety_margin`` and its first chunk's pages can be
  allocated, otherwise nothing is allocated (section "Admission");
* when an active request cannot get the page it needs, the newest other active
  request is soft-reset: its generated tokens are appended to its prompt, its
  pages are freed and it goes back to the front of the waiting queue; the last
  active request is never reset (sections "Soft reset", "Offloading");
* finished requests free their pages at once; pages 0-1 are reserved.
* prefix caching, when enabled (``prefix_groups > 0``): requests of a group
  start with the group's shared prompt prefix; every full block of that
  prefix, once its K/V are in the cache, is registered under a key, and a
  later request with the same prefix takes the same physical page into its
  block table (refcounted) and starts its prefill after the shared blocks.
  A page whose last user frees it keeps its key and content until an
  allocation finds no uninitialized page and demotes the most recently freed
  such page (sections "Prefix caching", "Eviction").

The second policy, prefill-first (section "PrefillFirst"), finishes chunked
prefills before it resumes decoding: active prefills first, then waiting
requests, then decodes with the budget that is left; its safety margin
defaults to 0 (section "Admission").

Readings (the pages leave them open): arrivals are drawn per step; a soft-reset
request re-enters at the head of the waiting queue; prefill-first still gives
decodes whatever token and request budget the prefills leave; a block's
content key is (prefix group, block index), only blocks that lie wholly in the
shared prefix are shared, and at least the prompt's last token is always
computed.
"""
from __future__ import annotations

import dataclasses
import math
from collections import OrderedDict, deque
from typing import List, Optional

import numpy as np

from . import RESERVED_PAGES, StepSpec


@dataclasses.dataclass
class TraceConfig:
    num_requests: int = 512
    prompt_median: float = 512.0
    prompt_sigma: float = 1.0
    prompt_max: int = 8192
    output_mean: float = 256.0
    arrivals_per_step: float = 40.0
    max_batch_tokens: int = 4096
    max_requests_per_batch: int = 256
    block_size: int = 16
    num_pages: int = 65536
    safety_margin: float = 0.15
    num_q_heads: int = 32
    num_kv_heads: int = 8
    head_dim: int = 128
    dtype: str = "bf16"
    seed: int = 4
    policy: str = "fifo"        # "fifo" or "prefill_first"
    prefix_groups: int = 0      # shared prompt prefixes (0: no prefix caching)
    prefix_share: float = 0.75  # fraction of requests that start with a group prefix
    prefix_len_min: int = 64
    prefix_len_max: int = 1024


def prefill_first_config(**kw) -> TraceConfig:
    """The prefill-first trace: same request stream, safety margin 0."""
    kw.setdefault("safety_margin", 0.0)
    return TraceConfig(policy="prefill_first", **kw)


@dataclasses.dataclass
class Request:
    rid: int
    prompt_len: int
    output_len: int
    arrival_step: int
    state: str = "PENDING"
    prefilled: int = 0          # prompt tokens already in the cache
    generated: int = 0          # output tokens produced so far
    pages: List[int] = dataclasses.field(default_factory=list)
    finish_step: Optional[int] = None
    resets: int = 0
    group: int = -1             # shared prompt prefix group (-1: none)
    prefix_len: int = 0         # tokens of the group prefix at the start of the prompt
    registered: int = 0         # prefix blocks of this request registered in the pool
    reused_tokens: int = 0      # prompt tokens taken from cached blocks at admission

    @property
    def kv_len(self) -> int:
        """Tokens whose K/V are in the cache."""
        if self.state == "DECODING":
            return self.prompt_len + self.generated - 1
        return self.prefilled


class PagePool:
    """Refcounted pages. A page holding a full block of a shared prefix carries that
    block's key; when its last user frees it, it stays as an initialized page that a
    later request with the same prefix can take back, until an allocation finds no
    uninitialized page and demotes the most recently freed initialized one."""

    def __init__(self, num_pages: int):
        self.num_pages = num_pages
        self.free = deque(range(RESERVED_PAGES, num_pages))  # uninitialized
        self.cached: "OrderedDict[tuple, int]" = OrderedDict()  # key -> page, refcount 0
        self.key_of = {}   # page -> key
        self.page_of = {}  # key -> page (in use or cached)
        self.ref = [0] * num_pages

    @property
    def capacity(self) -> int:
        return self.num_pages - RESERVED_PAGES

    def available(self) -> int:
        return len(self.free) + len(self.cached)

    def take(self, n: int) -> List[int]:
        out = []
        for _ in range(n):
            if self.free:
                p = self.free.popleft()
            else:  # demote the most recently freed initialized page
                key, p = self.cached.popitem(last=True)
                del self.key_of[p]
                del self.page_of[key]
            self.ref[p] = 1
            out.append(p)
        return out

    def give(self, pages: List[int]):
        for p in pages:
            self.ref[p] -= 1
            if self.ref[p] == 0:
                key = self.key_of.get(p)
                if key is None:
                    self.free.append(p)
                else:
                    self.cached[key] = p

    def cached_page(self, key) -> Optional[int]:
        return self.page_of.get(key)

    def share(self, key) -> int:
        """Take one more reference to the page that holds `key` (it must exist)."""
        p = self.page_of[key]
        if self.ref[p] == 0:
            del self.cached[key]
        self.ref[p] += 1
        return p

    def register(self, page: int, key):
        if key not in self.page_of and page not in self.key_of:
            self.page_of[key] = page
            self.key_of[page] = key


def draw_requests(cfg: TraceConfig, rng) -> List[Request]:
    """Lognormal prompts (median, sigma, clipped), geometric outputs (mean), Poisson arrivals."""
    prompts = np.clip(np.rint(rng.lognormal(math.log(cfg.prompt_median), cfg.prompt_sigma,
                                            size=cfg.num_requests)), 1, cfg.prompt_max)
    outputs = rng.geometric(1.0 / cfg.output_mean, size=cfg.num_requests)
    reqs, step, i = [], 0, 0
    while i < cfg.num_requests:
        n = int(rng.poisson(cfg.arrivals_per_step))
        for _ in range(min(n, cfg.num_requests - i)):
            reqs.append(Request(i, int(prompts[i]), int(outputs[i]), step))
            i += 1
        step += 1
    if cfg.prefix_groups > 0:
        # group prefixes from a stream of their own: the trace without them is unchanged
        prng = np.random.default_rng(cfg.seed + 7919)
        plens = prng.integers(cfg.prefix_len_min, cfg.prefix_len_max, endpoint=True,
                              size=cfg.prefix_groups)
        for req in reqs:
            if prng.random() < cfg.prefix_share:
                req.group = int(prng.integers(cfg.prefix_groups))
                req.prefix_len = int(plens[req.group])
                req.prompt_len += req.prefix_len  # the request's own text follows the prefix
    return reqs


@dataclasses.dataclass
class ScheduledStep:
    index: int
    entries: List[tuple]   # (request, ctx, q_len) in batch order
    spec: StepSpec


class FifoScheduler:
    def __init__(self, cfg: TraceConfig, requests: List[Request]):
        self.cfg = cfg
        self.pool = PagePool(cfg.num_pages)
        self.pending = deque(sorted(requests, key=lambda r: (r.arrival_step, r.rid)))
        self.waiting: deque = deque()
        self.active: List[Request] = []   # PREFILLING or DECODING, in admission order
        self.finished: List[Request] = []
        self.step_index = 0

    # ---------------------------------------------------------------- pages
    def _pages_needed(self, req: Request, new_len: int) -> int:
        return max(0, -(-new_len // self.cfg.block_size) - len(req.pages))

    def _grow(self, req: Request, new_len: int) -> bool:
        need = self._pages_needed(req, new_len)
        if need > self.pool.available():
            return False
        req.pages.extend(self.pool.take(need))
        return True

    def _soft_reset(self, req: Request):
        """Generated tokens join the prompt; pages freed; back to the head of the queue."""
        if req.state == "DECODING":
            req.prompt_len = req.prompt_len + req.generated
            req.output_len -= req.generated
        req.generated = 0
        req.prefilled = 0
        req.registered = 0
        req.state = "PENDING"
        self.pool.give(req.pages)
        req.pages = []
        req.resets += 1
        self.active.remove(req)
        self.waiting.appendleft(req)

    # ---------------------------------------------------------------- one step
    def schedule(self) -> Optional[List[tuple]]:
        cfg = self.cfg
        while self.pending and self.pending[0].arrival_step <= self.step_index:
            self.waiting.append(self.pending.popleft())
        batch = []
        tokens = 0

        def fit(req, ctx, q_len):
            nonlocal tokens
            while not self._grow(req, ctx + q_len):
                # stalled: reset the newest other active request, never the last one
                victims = [v for v in self.active if v is not req and v not in
                           [e[0] for e in batch]]
                if not victims or len(self.active) <= 1:
                    return False
                self._soft_reset(victims[-1])
            batch.append((req, ctx, q_len))
            tokens += q_len
            return True

        def active_of(kind):
            # FIFO over the active set
            for req in list(self.active):
                if req.state != kind or req not in self.active:
                    continue
                if len(batch) >= cfg.max_requests_per_batch or tokens >= cfg.max_batch_tokens:
                    break
                if kind == "DECODING":
                    fit(req, req.kv_len, 1)
                else:
                    n = min(req.prompt_len - req.prefilled, cfg.max_batch_tokens - tokens)
                    fit(req, req.prefilled, n)

        def admit():
            # waiting requests in arrival order, while the pool keeps its safety margin
            while (self.waiting and len(batch) < cfg.max_requests_per_batch
                   and tokens < cfg.max_batch_tokens):
                if self.pool.available() < cfg.safety_margin * self.pool.capacity:
                    break
                req = self.waiting[0]
                keys = self._cached_prefix(req)
                ctx = len(keys) * cfg.block_size
                n = min(req.prompt_len - ctx, cfg.max_batch_tokens - tokens)
                revived = sum(1 for k in keys if self.pool.ref[self.pool.page_of[k]] == 0)
                fresh = -(-(ctx + n) // cfg.block_size) - len(keys)
                if fresh > self.pool.available() - revived:
                    break  # admission needs every page of the first chunk
                self.waiting.popleft()
                req.pages = [self.pool.share(k) for k in keys]
                req.prefilled = ctx
                req.reused_tokens = ctx
                req.state = "PREFILLING"
                self.active.append(req)
                fit(req, ctx, n)

        if cfg.policy == "prefill_first":
            active_of("PREFILLING")
            admit()
            active_of("DECODING")
        else:
            active_of("DECODING")
            active_of("PREFILLING")
            admit()
        return batch

    def _cached_prefix(self, req: Request) -> List[tuple]:
        """Keys of the request's leading prefix blocks already in the pool (at least the
        prompt's last token stays to compute)."""
        if req.group < 0:
            return []
        bs = self.cfg.block_size
        keys = []
        for k in range(min(req.prefix_len, req.prompt_len - 1) // bs):
            if self.pool.cached_page((req.group, k)) is None:
                break
            keys.append((req.group, k))
        return keys

    def _register_prefix(self, req: Request):
        """Full prefix blocks whose K/V are now in the cache become shareable."""
        if req.group < 0:
            return
        full = min(req.prefilled, req.prefix_len) // self.cfg.block_size
        for k in range(req.registered, full):
            self.pool.register(req.pages[k], (req.group, k))
        req.registered = max(req.registered, full)

    def complete(self, batch):
        """Advance every scheduled request past this step's forward pass."""
        for req, ctx, q_len in batch:
            if req.state == "PREFILLING":
                req.prefilled += q_len
                self._register_prefix(req)
                if req.prefilled == req.prompt_len:
                    req.generated = 1  # the last chunk yields the first output token
                    req.state = "DECODING"
            else:
                req.generated += 1
            if req.state == "DECODING" and req.generated >= req.output_len:
                req.state = "FINISHED"
                req.finish_step = self.step_index
                self.pool.give(req.pages)
                req.pages = []
                self.active.remove(req)
                self.finished.append(req)
        self.step_index += 1

    def done(self) -> bool:
        return not (self.pending or self.waiting or self.active)


def to_spec(cfg: TraceConfig, batch, index: int) -> StepSpec:
    """The step's metadata in batch order (decodes first, then prefill chunks)."""
    q_lens = np.array([q for _, _, q in batch], dtype=np.int32)
    ctx_lens = np.array([c for _, c, _ in batch], dtype=np.int32)
    R = len(batch)
    qsl = np.zeros(R + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(q_lens)
    seq_lens = (ctx_lens + q_lens).astype(np.int32)
    stride = max([len(req.pages) for req, _, _ in batch] + [1])
    bt = np.zeros((R, stride), dtype=np.int32)
    for i, (req, _, _) in enumerate(batch):
        bt[i, :len(req.pages)] = req.pages
    BS = cfg.block_size
    slots = np.empty(int(qsl[-1]), dtype=np.int64)
    for i, (req, ctx, q_len) in enumerate(batch):
        for k in range(q_len):
            p = ctx + k
            slots[qsl[i] + k] = int(bt[i, p // BS]) * BS + p % BS
    return StepSpec(name=f"fifo_trace_step{index}", dtype=cfg.dtype, num_q_heads=cfg.num_q_heads,
                    num_kv_heads=cfg.num_kv_heads, head_dim=cfg.head_dim, block_size=BS,
                    num_blocks=cfg.num_pages, q_lens=q_lens, ctx_lens=ctx_lens,
                    query_start_loc=qsl, seq_lens=seq_lens, block_table=bt, slot_mapping=slots,
                    scale=1.0 / math.sqrt(cfg.head_dim), seed=cfg.seed + index)


def fifo_trace(cfg: Optional[TraceConfig] = None, max_steps: Optional[int] = None):
    """Yield (ScheduledStep) for every step of the trace until all requests finish."""
    cfg = cfg or TraceConfig()
    rng = np.random.default_rng(cfg.seed)
    sched = FifoScheduler(cfg, draw_requests(cfg, rng))
    while not sched.done() and (max_steps is None or sched.step_index < max_steps):
        batch = sched.schedule()
        if batch:
            yield ScheduledStep(sched.step_index, list(batch), to_spec(cfg, batch, sched.step_index))
        sched.complete(batch)
