"""The allocation-free entry point against the workspace entry point.

cb_paged_attention_no_alloc serves callers that may not allocate device memory
when they call the library (a plugin whose host program owns the device memory
pool, or a latency-critical caller that cannot pay cudaMalloc's implicit
synchronisation): its scratch is a fixed device array inside the library. These
tests call it through the C ABI twice in a row and check each result against
cb_paged_attention with a caller-allocated workspace, within the parity
tolerances of the other GPU tests. This file sorts last so that a run stopping
at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_cb_gb300 as cb
import workloads
from stepcheck import BF16_MAX_ABS, BF16_MEAN_ABS, F32_MAX_ABS, GpuStep

pytestmark = pytest.mark.gpu


def run_no_alloc(st, out):
    s = st.spec
    cb.paged_attention_no_alloc(out, st.x["q"], st.x["k_cache"], st.x["v_cache"],
                                st.md["query_start_loc"], st.md["seq_lens"], st.md["block_table"],
                                s.query_start_loc, s.seq_lens, scale=s.scale,
                                sliding_window=s.sliding_window, k_new=st.x["k_new"],
                                v_new=st.x["v_new"], slot_mapping=st.md["slot_mapping"])
    return out


def close(spec, got, ref):
    err = (got.float() - ref.float()).abs()
    if spec.dtype == "f32":
        return float(err.max()) <= F32_MAX_ABS
    return float(err.max()) <= BF16_MAX_ABS and float(err.mean()) <= BF16_MEAN_ABS


CASES = {
    # 64 decode requests over all SMs: most requests are split, so the partials
    # and arrival counters in the scratch array are exercised
    "decode_64": lambda: workloads.decode_step(),
    # a few long requests, each merged from many partials, plus prefill rows
    "long_split_mixed": lambda: workloads.custom([1, 1, 7, 1], [20000, 9000, 300, 5],
                                                 num_q_heads=16, num_kv_heads=4, seed=21),
    "tiny_fp32": lambda: workloads.tiny_mixed(),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_no_alloc_matches_workspace_entry_point_twice(name):
    spec = CASES[name]()
    st = GpuStep(spec)
    ref = st.run()  # cb_paged_attention with a torch-allocated workspace
    torch.cuda.synchronize()
    assert cb.read_error_word(st.ws) == 0
    for _ in range(2):
        got = run_no_alloc(st, torch.full_like(ref, float("nan")))
        torch.cuda.synchronize()
        assert torch.isfinite(got.float()).all()
        assert close(spec, got, ref), name


def test_no_alloc_rejects_a_step_larger_than_its_scratch():
    # 4096 decode requests with 64 query heads need far more than the fixed array
    R = 4096
    spec = workloads.custom([1] * R, [15] * R, num_q_heads=64, num_kv_heads=8, seed=3)
    st = GpuStep(spec)
    out = torch.zeros_like(st.x["q"])
    with pytest.raises(cb.CbError) as err:
        run_no_alloc(st, out)
    assert err.value.status == 4
    torch.cuda.synchronize()
    assert float(out.abs().max()) == 0.0  # nothing was launched
