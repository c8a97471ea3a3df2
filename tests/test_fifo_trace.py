"""Host-side FIFO step-trace generator (the scheduler and page allocator that feed the
hot path), checked on the CPU against the schedules the pages describe."""
import numpy as np

from workloads import RESERVED_PAGES
from workloads.fifo_trace import (FifoScheduler, Request, TraceConfig, fifo_trace, to_spec)


def run(cfg, requests, max_steps=100000):
    s = FifoScheduler(cfg, requests)
    batches = []
    while not s.done() and s.step_index < max_steps:
        b = s.schedule()
        batches.append([(r.rid, c, q) for r, c, q in b])
        s.complete(b)
    return s, batches


def test_slot_example_of_the_tutorial():
    """Four slots; A, B, C, D, E need 100, 20, 50, 200, 30 output tokens, one step each:
    E takes B's slot when B finishes at step 20 and finishes at step 50; D ends at 200."""
    cfg = TraceConfig(max_requests_per_batch=4, max_batch_tokens=1 << 20, num_pages=4096,
                      safety_margin=0.0)
    outs = [100, 20, 50, 200, 30]
    reqs = [Request(i, 1, n, 0) for i, n in enumerate(outs)]
    s, batches = run(cfg, reqs)
    finish = {r.rid: r.finish_step + 1 for r in s.finished}  # 1-based step numbers
    assert finish == {0: 100, 1: 20, 2: 50, 3: 200, 4: 50}
    assert len(batches) == 200
    assert all(len(b) <= 4 for b in batches)
    assert [rid for rid, _, _ in batches[20]].count(4) == 1 and 4 not in [x[0] for x in batches[19]]


def test_fifo_priority_decode_then_prefill_then_waiting():
    cfg = TraceConfig(max_batch_tokens=64, max_requests_per_batch=16, num_pages=1024,
                      safety_margin=0.0)
    reqs = [Request(0, 8, 5, 0), Request(1, 100, 5, 0), Request(2, 10, 5, 1),
            Request(3, 10, 5, 1)]
    s = FifoScheduler(cfg, reqs)
    b0 = s.schedule()  # step 0: request 0 whole, request 1 chunked to the budget
    assert [(r.rid, c, q) for r, c, q in b0] == [(0, 0, 8), (1, 0, 56)]
    s.complete(b0)
    b1 = s.schedule()  # decode of 0, then 1's next chunk, then arrivals 2, 3 in order
    assert [(r.rid, c, q) for r, c, q in b1] == [(0, 8, 1), (1, 56, 44), (2, 0, 10), (3, 0, 9)]


def test_chunked_prefill_continues_where_it_stopped():
    cfg = TraceConfig(max_batch_tokens=4096, num_pages=4096, safety_margin=0.0)
    s, batches = run(cfg, [Request(0, 10000, 2, 0)])
    assert batches[:3] == [[(0, 0, 4096)], [(0, 4096, 4096)], [(0, 8192, 1808)]]
    assert batches[3] == [(0, 10000, 1)]  # the one decode step of a 2-token output
    assert len(batches) == 4


def test_safety_margin_holds_new_prefills():
    # 100 usable pages of 16 tokens; margin 0.5: a 1000-token prompt (63 pages) is admitted,
    # leaving 37% free, so the next arrival waits while the first one decodes
    cfg = TraceConfig(num_pages=100 + RESERVED_PAGES, block_size=16, safety_margin=0.5,
                      max_batch_tokens=4096)
    s = FifoScheduler(cfg, [Request(0, 1000, 3, 0), Request(1, 10, 3, 0)])
    b0 = s.schedule()
    assert [r.rid for r, _, _ in b0] == [0]
    s.complete(b0)
    b1 = s.schedule()
    assert [r.rid for r, _, _ in b1] == [0]
    s.complete(b1)
    s.complete(s.schedule())  # request 0 finishes and frees its pages
    assert [r.rid for r, _, _ in s.schedule()] == [1]


def test_soft_reset_frees_the_newest_and_everything_finishes():
    cfg = TraceConfig(num_pages=40 + RESERVED_PAGES, block_size=16, safety_margin=0.0,
                      max_batch_tokens=1024)
    reqs = [Request(i, 200, 120, 0) for i in range(3)]  # 3 x 20 pages at the end > 40
    s, batches = run(cfg, reqs, max_steps=5000)
    assert s.done()
    assert sum(r.resets for r in s.finished) >= 1
    assert s.finished[0].resets == 0  # the oldest request is never the victim here
    assert s.pool.available() == s.pool.capacity


def test_trace_metadata_is_consistent():
    cfg = TraceConfig()
    seen = 0
    for st in fifo_trace(cfg, max_steps=60):
        sp = st.spec
        assert sp.T <= cfg.max_batch_tokens and sp.R <= cfg.max_requests_per_batch
        assert list(sp.query_start_loc[1:] - sp.query_start_loc[:-1]) == list(sp.q_lens)
        # decodes first, then prefill chunks
        dec = sp.q_lens == 1
        if dec.any() and (~dec).any():
            assert np.flatnonzero(dec).max() < np.flatnonzero(~dec).min() or \
                all(sp.ctx_lens[~dec] + sp.q_lens[~dec] <= sp.seq_lens[~dec])
        pages = []
        for r in range(sp.R):
            n = -(-int(sp.seq_lens[r]) // cfg.block_size)
            row = sp.block_table[r, :n]
            assert row.min() >= RESERVED_PAGES and row.max() < cfg.num_pages
            pages += list(row)
            for i in range(int(sp.q_lens[r])):
                p = int(sp.ctx_lens[r]) + i
                t = int(sp.query_start_loc[r]) + i
                assert sp.slot_mapping[t] == row[p // cfg.block_size] * cfg.block_size + p % cfg.block_size
        assert len(pages) == len(set(pages))  # no page shared between requests
        seen += 1
    assert seen == 60


def test_small_trace_runs_to_completion():
    cfg = TraceConfig(num_requests=60, prompt_median=100, output_mean=20, arrivals_per_step=8,
                      max_batch_tokens=512, max_requests_per_batch=32, num_pages=600)
    steps = list(fifo_trace(cfg))
    assert steps and steps[-1].spec.T >= 1
    total_tokens = sum(int(st.spec.T) for st in steps)
    assert total_tokens > 60


# ------------------------------------------------------------------ prefill-first policy


def test_prefill_first_orders_prefills_before_decodes():
    from workloads.fifo_trace import prefill_first_config

    cfg = prefill_first_config(max_batch_tokens=64, max_requests_per_batch=16, num_pages=1024)
    assert cfg.safety_margin == 0.0 and cfg.policy == "prefill_first"
    reqs = [Request(0, 8, 5, 0), Request(1, 100, 5, 0), Request(2, 10, 5, 1)]
    s = FifoScheduler(cfg, reqs)
    b0 = s.schedule()  # request 0 whole, request 1 chunked to the budget
    assert [(r.rid, c, q) for r, c, q in b0] == [(0, 0, 8), (1, 0, 56)]
    s.complete(b0)
    # step 1: request 1's next chunk first, then arrival 2, then the decode of 0
    b1 = s.schedule()
    assert [(r.rid, c, q) for r, c, q in b1] == [(1, 56, 44), (2, 0, 10), (0, 8, 1)]


def test_prefill_first_decodes_wait_while_prefills_fill_the_budget():
    from workloads.fifo_trace import prefill_first_config

    cfg = prefill_first_config(max_batch_tokens=32, num_pages=1024)
    s = FifoScheduler(cfg, [Request(0, 4, 10, 0), Request(1, 200, 3, 1)])
    s.complete(s.schedule())  # request 0's prompt, which yields its first token
    b = s.schedule()          # request 1 arrives: its chunk takes the whole budget
    assert [(r.rid, q) for r, _, q in b] == [(1, 32)]
    # FIFO on the same stream decodes request 0 first
    f = FifoScheduler(TraceConfig(max_batch_tokens=32, num_pages=1024, safety_margin=0.0),
                      [Request(0, 4, 10, 0), Request(1, 200, 3, 1)])
    f.complete(f.schedule())
    assert [(r.rid, q) for r, _, q in f.schedule()] == [(0, 1), (1, 31)]


def test_prefill_first_trace_runs_to_completion():
    from workloads.fifo_trace import prefill_first_config

    cfg = prefill_first_config(num_requests=60, prompt_median=100, output_mean=20,
                               arrivals_per_step=8, max_batch_tokens=512,
                               max_requests_per_batch=32, num_pages=600)
    n_steps = n_mixed = total = 0
    for st in fifo_trace(cfg):  # inspected before the step completes: states as scheduled
        sp = st.spec
        assert sp.T <= cfg.max_batch_tokens and sp.R <= cfg.max_requests_per_batch
        kinds = [r.state for r, _, _ in st.entries]
        if "DECODING" in kinds and "PREFILLING" in kinds:
            n_mixed += 1
            last_prefill = max(i for i, k in enumerate(kinds) if k == "PREFILLING")
            first_decode = min(i for i, k in enumerate(kinds) if k == "DECODING")
            assert last_prefill < first_decode
        n_steps += 1
        total += int(sp.T)
    # prefills take the whole budget most steps, so few steps mix the two kinds
    assert n_steps > 20 and n_mixed >= 1 and total > 60


# ------------------------------------------------------------------ prefix caching


def _prefixed(rid, group, prefix_len, own, out, arrival):
    r = Request(rid, prefix_len + own, out, arrival)
    r.group, r.prefix_len = group, prefix_len
    return r


def test_prefix_blocks_are_shared_after_they_are_written():
    cfg = TraceConfig(block_size=16, max_batch_tokens=4096, num_pages=64, safety_margin=0.0)
    a = _prefixed(0, 0, 64, 10, 5, 0)   # 74-token prompt, 4 full prefix blocks
    b = _prefixed(1, 0, 64, 30, 5, 0)   # same prefix, arrives with a: nothing cached yet
    c = _prefixed(2, 0, 64, 3, 5, 1)    # arrives after a's prompt is in the cache
    s = FifoScheduler(cfg, [a, b, c])
    b0 = s.schedule()
    assert [(r.rid, ctx, q) for r, ctx, q in b0] == [(0, 0, 74), (1, 0, 94)]
    s.complete(b0)
    b1 = s.schedule()
    entries = {r.rid: (ctx, q) for r, ctx, q in b1}
    assert entries[2] == (64, 3)                # c computes only its own 3 tokens
    assert c.pages[:4] == a.pages[:4]           # the same physical pages
    assert all(s.pool.ref[p] == 2 for p in a.pages[:4])  # a and c (b registered none: a won)
    sp = to_spec(cfg, b1, 1)
    # no slot of the step falls into a shared page
    shared = set(a.pages[:4])
    assert not any(int(x) // 16 in shared for x in sp.slot_mapping)


def test_shared_pages_return_only_with_their_last_user_and_stay_cached():
    cfg = TraceConfig(block_size=16, max_batch_tokens=4096, num_pages=40, safety_margin=0.0)
    a = _prefixed(0, 3, 32, 1, 2, 0)
    s = FifoScheduler(cfg, [a])
    while not s.done():
        s.complete(s.schedule())
    # a finished: its two prefix pages are free but keep their keys (initialized)
    assert s.pool.available() == s.pool.capacity and len(s.pool.cached) == 2
    b = _prefixed(1, 3, 32, 5, 2, s.step_index)
    s.pending.append(b)
    s.complete(s.schedule())
    assert b.reused_tokens == 32 and b.pages[:2] == [s.pool.page_of[(3, 0)], s.pool.page_of[(3, 1)]]


def test_initialized_pages_are_demoted_when_uninitialized_run_out():
    cfg = TraceConfig(block_size=16, max_batch_tokens=4096, num_pages=2 + 6, safety_margin=0.0)
    a = _prefixed(0, 1, 64, 1, 1, 0)  # 65 tokens: 5 pages, 4 of them prefix blocks
    s = FifoScheduler(cfg, [a])
    while not s.done():
        s.complete(s.schedule())
    assert len(s.pool.cached) == 4 and len(s.pool.free) == 2
    got = s.pool.take(3)  # two uninitialized, then the most recently freed initialized
    assert len(got) == 3 and len(s.pool.cached) == 3
    assert all(p not in s.pool.key_of for p in got)


def test_trace_with_prefix_groups_shares_and_stays_consistent():
    from workloads.fifo_trace import draw_requests

    cfg = TraceConfig(num_requests=80, prompt_median=60, output_mean=12, arrivals_per_step=6,
                      max_batch_tokens=1024, max_requests_per_batch=48, num_pages=900,
                      prefix_groups=3, prefix_len_min=32, prefix_len_max=160, seed=5)
    s = FifoScheduler(cfg, draw_requests(cfg, np.random.default_rng(cfg.seed)))
    n_shared_steps = 0
    while not s.done():
        batch = s.schedule()
        sp = to_spec(cfg, batch, s.step_index)
        owners = {}
        for r in range(sp.R):
            n = -(-int(sp.seq_lens[r]) // cfg.block_size)
            row = sp.block_table[r, :n]
            assert row.min() >= RESERVED_PAGES
            for p in row:
                owners.setdefault(int(p), []).append(r)
        shared = {p for p, rs in owners.items() if len(rs) > 1}
        n_shared_steps += bool(shared)
        # a page in several block tables is a registered prefix block with that many users
        for p in shared:
            assert p in s.pool.key_of and s.pool.ref[p] >= len(owners[p])
        # and the step writes none of them
        assert not any(int(x) // cfg.block_size in shared for x in sp.slot_mapping)
        s.complete(batch)
    assert n_shared_steps > 5
    assert sum(r.reused_tokens for r in s.finished) > 0
    assert s.pool.available() == s.pool.capacity  # every reference returned
