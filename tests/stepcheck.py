"""Test-side helpers: run one step through the C ABI on the GPU and compare it
with the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_attention_cb_gb300 as cb
import workloads

BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
F32_MAX_ABS = 1e-4


class GpuStep:
    """Seeded inputs of a StepSpec on cuda:0 plus host copies of the pre-step state."""

    def __init__(self, spec: workloads.StepSpec, device="cuda"):
        self.spec = spec
        self.device = device
        self.x = workloads.draw_tensors(spec, device)
        self.md = workloads.metadata_tensors(spec, device)
        self.ws = cb.alloc_workspace(spec.R, spec.T, spec.num_q_heads, spec.num_kv_heads,
                                     spec.head_dim, device)

    def host_inputs(self):
        """Pre-step inputs as numpy (float32 holds bf16 exactly; the oracle widens to fp64)."""
        f = lambda t: t.detach().float().cpu().numpy()
        return {k: f(v) for k, v in self.x.items()}

    def run(self, flags=0, scatter=True, out=None, scale=None):
        s = self.spec
        if out is None:
            out = torch.full_like(self.x["q"], float("nan"))
        cb.paged_attention(out, self.x["q"], self.x["k_cache"], self.x["v_cache"],
                           self.md["query_start_loc"], self.md["seq_lens"], self.md["block_table"],
                           s.query_start_loc, s.seq_lens, self.ws,
                           scale=s.scale if scale is None else scale,
                           sliding_window=s.sliding_window,
                           k_new=self.x["k_new"] if scatter else None,
                           v_new=self.x["v_new"] if scatter else None,
                           slot_mapping=self.md["slot_mapping"] if scatter else None, flags=flags,
                           ring_blocks=s.ring_blocks)
        return out


def oracle_step(spec, h, rows=None, scale=None):
    """Scatter (in place on the host copies) then attend, float64."""
    oracle.scatter_kv(h["k_cache"], h["v_cache"], h["k_new"], h["v_new"], spec.slot_mapping)
    return oracle.paged_attention(h["q"], h["k_cache"], h["v_cache"], spec.query_start_loc,
                                  spec.seq_lens, spec.block_table, spec.block_size,
                                  spec.scale if scale is None else scale, spec.sliding_window,
                                  rows=rows, ring_blocks=spec.ring_blocks)


def compare(spec, got, ref, rows=None, max_abs=None, mean_abs=None):
    """Max-abs / mean-abs check of GPU rows against oracle rows; returns (max, mean)."""
    got = got.detach().float().cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[rows]
        ref = ref[rows]
    assert np.all(np.isfinite(got)), "non-finite output"
    err = np.abs(got - ref)
    mx, mn = float(err.max()), float(err.mean())
    if spec.dtype == "f32":
        max_abs = F32_MAX_ABS if max_abs is None else max_abs
        assert mx <= max_abs, (mx, mn)
    else:
        max_abs = BF16_MAX_ABS if max_abs is None else max_abs
        mean_abs = BF16_MEAN_ABS if mean_abs is None else mean_abs
        assert mx <= max_abs and mn <= mean_abs, (mx, mn)
    return mx, mn


def sample_rows(spec, n, seed=0):
    """Rows to check one by one at full size: every request's first and last row plus random."""
    rng = np.random.default_rng(seed)
    rows = set()
    qsl = spec.query_start_loc
    for r in range(spec.R):
        if qsl[r + 1] > qsl[r]:
            rows.add(int(qsl[r]))
            rows.add(int(qsl[r + 1] - 1))
    rows |= set(int(t) for t in rng.integers(0, spec.T, size=n))
    return sorted(rows)


def cache_bits(t):
    """Bit pattern of a cache tensor as a numpy integer array."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy()
    return t.view(torch.int32).cpu().numpy()


def oracle_cache_bits(spec, t_before, k_new, slots):
    """Oracle scatter on bit patterns: exact copy of each new row into its slot."""
    kb = cache_bits(t_before)
    nb = cache_bits(k_new)
    dummy = np.zeros_like(kb)
    oracle.scatter_kv(kb, dummy, nb, np.zeros_like(nb), slots)
    return kb
