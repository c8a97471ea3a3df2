"""GPU parity over a FIFO step trace: every step's scatter + attention through the C ABI,
with the cache carried from step to step, against the oracle carrying its own cache."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_cb_gb300 as cb
from stepcheck import BF16_MAX_ABS, BF16_MEAN_ABS
from workloads.fifo_trace import TraceConfig, fifo_trace, prefill_first_config

pytestmark = pytest.mark.gpu


def draw_step(spec, device="cuda"):
    g = torch.Generator(device=device)
    g.manual_seed(int(spec.seed) * 7919 + 17)
    T, Hq, Hkv, D = spec.T, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    f = lambda *shape: torch.randn(*shape, generator=g, device=device).to(torch.bfloat16)
    return f(T, Hq, D), f(T, Hkv, D), f(T, Hkv, D)


@pytest.mark.parametrize("policy", ["fifo", "prefill_first", "fifo_prefix_cache"])
def test_reduced_trace_all_steps(policy):
    # the trace's structure (chunked prefills next to decodes, admission under a safety
    # margin, soft resets when the pool runs out) at a size the oracle follows step by step
    kw = dict(num_requests=48, prompt_median=160, prompt_max=1500, output_mean=24,
              arrivals_per_step=6, max_batch_tokens=512, max_requests_per_batch=24,
              num_pages=420, num_q_heads=8, num_kv_heads=2, head_dim=64, seed=4)
    if policy == "fifo_prefix_cache":
        # three shared prompt prefixes: later requests alias the cached prefix pages
        kw.update(prefix_groups=3, prefix_len_min=32, prefix_len_max=200)
    cfg = prefill_first_config(**kw) if policy == "prefill_first" else TraceConfig(**kw)
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    shape = (cfg.num_pages, cfg.block_size, cfg.num_kv_heads, cfg.head_dim)
    k_cache = torch.randn(*shape, generator=g, device="cuda").to(torch.bfloat16)
    v_cache = torch.randn(*shape, generator=g, device="cuda").to(torch.bfloat16)
    hk = k_cache.float().cpu().numpy()
    hv = v_cache.float().cpu().numpy()
    ws = cb.alloc_workspace(cfg.max_requests_per_batch, cfg.max_batch_tokens, cfg.num_q_heads,
                            cfg.num_kv_heads, cfg.head_dim)
    n_steps = n_mixed = n_aliased = 0
    worst = 0.0
    for st in fifo_trace(cfg):
        sp = st.spec
        q, k_new, v_new = draw_step(sp)
        md = {k: torch.from_numpy(getattr(sp, k).copy()).cuda()
              for k in ("query_start_loc", "seq_lens", "block_table", "slot_mapping")}
        out = torch.full_like(q, float("nan"))
        cb.paged_attention(out, q, k_cache, v_cache, md["query_start_loc"], md["seq_lens"],
                           md["block_table"], sp.query_start_loc, sp.seq_lens, ws, scale=sp.scale,
                           k_new=k_new, v_new=v_new, slot_mapping=md["slot_mapping"])
        # oracle: its own cache, its own scatter, then attention
        kn = k_new.float().cpu().numpy()
        vn = v_new.float().cpu().numpy()
        oracle.scatter_kv(hk, hv, kn, vn, sp.slot_mapping)
        ref = oracle.paged_attention(q.float().cpu().numpy(), hk, hv, sp.query_start_loc,
                                     sp.seq_lens, sp.block_table, sp.block_size, sp.scale)
        got = out.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all(), st.index
        err = np.abs(got - ref)
        assert err.max() <= BF16_MAX_ABS and err.mean() <= BF16_MEAN_ABS, (st.index, err.max())
        worst = max(worst, float(err.max()))
        n_steps += 1
        n_mixed += int((sp.q_lens == 1).any() and (sp.q_lens > 1).any())
        rows = [sp.block_table[r, :-(-int(sp.seq_lens[r]) // sp.block_size)] for r in range(sp.R)]
        n_aliased += int(len(np.concatenate(rows)) > len(np.unique(np.concatenate(rows))))
    assert cb.read_error_word(ws) == 0
    # the GPU cache after the whole trace equals the oracle's, bit for bit (pages >= 2)
    assert np.array_equal(k_cache.float().cpu().numpy()[2:], hk[2:])
    assert n_steps > 20 and n_mixed >= (1 if policy == "prefill_first" else 5)
    if policy == "fifo_prefix_cache":
        assert n_aliased > 5


def test_full_size_fifo_trace_sampled_rows():
    """The whole FIFO trace (512 requests, 2157 steps, 65536 pages) through the C ABI with
    the cache carried; the oracle follows with its own host cache and scatter and checks
    sampled rows of 12 spread-out steps, then the whole cache bit for bit."""
    cfg = TraceConfig()
    steps = list(fifo_trace(cfg))
    n = len(steps)
    check_at = {int(k * (n - 1) / 11) for k in range(12)}
    g = torch.Generator(device="cuda")
    g.manual_seed(cfg.seed)
    shape = (cfg.num_pages, cfg.block_size, cfg.num_kv_heads, cfg.head_dim)
    k_cache = torch.randn(*shape, generator=g, device="cuda").to(torch.bfloat16)
    v_cache = torch.randn(*shape, generator=g, device="cuda").to(torch.bfloat16)
    hk = k_cache.cpu().float().numpy()
    hv = v_cache.cpu().float().numpy()
    ws = cb.alloc_workspace(cfg.max_requests_per_batch, cfg.max_batch_tokens, cfg.num_q_heads,
                            cfg.num_kv_heads, cfg.head_dim)
    checked = 0
    for i, st in enumerate(steps):
        sp = st.spec
        q, k_new, v_new = draw_step(sp)
        md = {k: torch.from_numpy(getattr(sp, k).copy()).cuda()
              for k in ("query_start_loc", "seq_lens", "block_table", "slot_mapping")}
        out = torch.full_like(q, float("nan"))
        cb.paged_attention(out, q, k_cache, v_cache, md["query_start_loc"], md["seq_lens"],
                           md["block_table"], sp.query_start_loc, sp.seq_lens, ws, scale=sp.scale,
                           k_new=k_new, v_new=v_new, slot_mapping=md["slot_mapping"])
        oracle.scatter_kv(hk, hv, k_new.cpu().float().numpy(), v_new.cpu().float().numpy(),
                          sp.slot_mapping)
        if i in check_at:
            rows = sorted(set(np.random.default_rng(i).integers(0, sp.T, size=24).tolist()))
            ref = oracle.paged_attention(q.cpu().float().numpy(), hk, hv, sp.query_start_loc,
                                         sp.seq_lens, sp.block_table, sp.block_size, sp.scale,
                                         rows=rows)
            got = out.cpu().float().numpy().astype(np.float64)
            err = np.abs(got[rows] - ref[rows])
            assert np.isfinite(got[rows]).all(), i
            assert err.max() <= BF16_MAX_ABS and err.mean() <= BF16_MEAN_ABS, (i, err.max())
            checked += 1
    assert cb.read_error_word(ws) == 0
    assert checked == len(check_at)
    assert np.array_equal(k_cache.cpu().float().numpy()[2:], hk[2:])
    assert np.array_equal(v_cache.cpu().float().numpy()[2:], hv[2:])
