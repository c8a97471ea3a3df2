"""GPU: the step through CUDA graphs cached per padded shape (cb_paged_attention_graphed),
replayed over a FIFO trace with persistent padded buffers, against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_cb_gb300 as cb
from stepcheck import BF16_MAX_ABS, BF16_MEAN_ABS
from test_gpu_trace import draw_step
from workloads.fifo_trace import TraceConfig, fifo_trace

pytestmark = pytest.mark.gpu


def _pad(n, k):
    return -(-n // k) * k


def test_graph_replay_over_a_trace():
    Q = 64  # query padding interval
    cfg = TraceConfig(num_requests=40, prompt_median=120, prompt_max=900, output_mean=20,
                      arrivals_per_step=6, max_batch_tokens=448, max_requests_per_batch=24,
                      num_pages=400, num_q_heads=8, num_kv_heads=2, head_dim=128, seed=6)
    dev = "cuda"
    g = torch.Generator(device=dev)
    g.manual_seed(6)
    shape = (cfg.num_pages, cfg.block_size, cfg.num_kv_heads, cfg.head_dim)
    k_cache = torch.randn(*shape, generator=g, device=dev).to(torch.bfloat16)
    v_cache = torch.randn(*shape, generator=g, device=dev).to(torch.bfloat16)
    hk, hv = k_cache.float().cpu().numpy(), v_cache.float().cpu().numpy()
    R_max, T_max = _pad(cfg.max_requests_per_batch, Q), _pad(cfg.max_batch_tokens, Q)
    stride = cfg.num_pages
    # persistent buffers the graphs name, sized for the largest padded shape
    q_buf = torch.zeros(T_max, cfg.num_q_heads, cfg.head_dim, dtype=torch.bfloat16, device=dev)
    out_buf = torch.zeros_like(q_buf)
    kn_buf = torch.zeros(T_max, cfg.num_kv_heads, cfg.head_dim, dtype=torch.bfloat16, device=dev)
    vn_buf = torch.zeros_like(kn_buf)
    qsl_buf = torch.zeros(R_max + 1, dtype=torch.int32, device=dev)
    seq_buf = torch.zeros(R_max, dtype=torch.int32, device=dev)
    bt_buf = torch.zeros(R_max, stride, dtype=torch.int32, device=dev)
    slot_buf = torch.full((T_max,), -1, dtype=torch.int64, device=dev)
    ws = cb.alloc_workspace(R_max, T_max, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim)
    cache = cb.GraphCache(q_interval=Q)
    stream = torch.cuda.Stream()
    shapes = set()
    n_steps = n_mixed = 0
    with torch.cuda.stream(stream):
        for st in fifo_trace(cfg):
            sp = st.spec
            R, T = sp.R, sp.T
            Rp, Tp = _pad(max(R, 1), Q), _pad(T, Q)
            # a graph per padded shape and per kinds of rows present
            shapes.add((Rp, Tp, bool((sp.q_lens == 1).any()), bool((sp.q_lens > 1).any())))
            q, kn, vn = draw_step(sp)
            # the step's inputs into the persistent buffers, padded
            q_buf[:T].copy_(q)
            kn_buf[:T].copy_(kn)
            vn_buf[:T].copy_(vn)
            qsl = np.full(Rp + 1, T, dtype=np.int32)
            qsl[:R + 1] = sp.query_start_loc
            seq = np.zeros(Rp, dtype=np.int32)
            seq[:R] = sp.seq_lens
            bt = np.zeros((Rp, stride), dtype=np.int32)
            bt[:R, :sp.bt_stride] = sp.block_table
            slots = np.full(Tp, -1, dtype=np.int64)
            slots[:T] = sp.slot_mapping
            qsl_buf[:Rp + 1].copy_(torch.from_numpy(qsl))
            seq_buf[:Rp].copy_(torch.from_numpy(seq))
            bt_buf[:Rp].copy_(torch.from_numpy(bt))
            slot_buf[:Tp].copy_(torch.from_numpy(slots))
            out_buf.fill_(float("nan"))
            cb.paged_attention_graphed(cache, out_buf[:Tp], q_buf[:Tp], k_cache, v_cache,
                                       qsl_buf[:Rp + 1], seq_buf[:Rp], bt_buf[:Rp], qsl, seq, ws,
                                       scale=sp.scale, k_new=kn_buf[:Tp], v_new=vn_buf[:Tp],
                                       slot_mapping=slot_buf[:Tp], stream=stream)
            got = out_buf[:T].float().cpu().numpy().astype(np.float64)
            # the oracle keeps its own cache
            oracle.scatter_kv(hk, hv, kn.float().cpu().numpy(), vn.float().cpu().numpy(),
                              sp.slot_mapping)
            ref = oracle.paged_attention(q.float().cpu().numpy(), hk, hv, sp.query_start_loc,
                                         sp.seq_lens, sp.block_table, sp.block_size, sp.scale)
            assert np.isfinite(got).all(), st.index
            err = np.abs(got - ref)
            assert err.max() <= BF16_MAX_ABS and err.mean() <= BF16_MEAN_ABS, (st.index, err.max())
            # padding rows are never written
            assert torch.isnan(out_buf[T:Tp].float()).all()
            n_steps += 1
            n_mixed += int((sp.q_lens == 1).any() and (sp.q_lens > 1).any())
    assert cb.read_error_word(ws) == 0
    stats = cache.stats()
    assert stats["captures"] == len(shapes) == stats["graphs"]
    assert stats["replays"] == n_steps - len(shapes) and stats["replays"] > n_steps // 2
    assert np.array_equal(k_cache.float().cpu().numpy()[2:], hk[2:])
    assert n_steps > 20 and n_mixed > 3
    cache.close()
