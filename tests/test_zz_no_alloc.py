"""The allocation-free entry point against the workspace entry point.

cb_paged_attention_no_alloc serves callers that may not allocate device memory
when they call the library (a plugin whose host program owns the device memory
pool, or a latency-critical caller that cannot pay cudaMalloc's implicit
synchronisation): its scratch is a fixed device array inside the library. These
tests call it through the C ABI twice in a row and check each result against
cb_paged_attention with a caller-allocated workspace and against the fp64 CPU
oracle, within the parity tolerances of the other GPU tests. This file sorts
last so that a run stopping at the first failure has already run every other
test.
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_cb_gb300 as cb
import workloads
from stepcheck import BF16_MAX_ABS, BF16_MEAN_ABS, F32_MAX_ABS, GpuStep, compare, oracle_step

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
    # 64 decode requests over all SMs: most requests are split, so the split-KV
    # partials in the scratch array are exercised
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
    want = oracle_step(spec, st.host_inputs())  # fp64 CPU oracle on the pre-step inputs
    ref = st.run()  # cb_paged_attention with a torch-allocated workspace
    torch.cuda.synchronize()
    assert cb.read_error_word(st.ws) == 0
    compare(spec, ref, want)
    for _ in range(2):
        # the step's scatter writes the same rows again: the inputs stay those of the oracle
        got = run_no_alloc(st, torch.full_like(ref, float("nan")))
        torch.cuda.synchronize()
        assert cb.no_alloc_read_error_word() == 0
        assert torch.isfinite(got.float()).all()
        assert close(spec, got, ref), name
        compare(spec, got, want)


def test_no_alloc_error_word_is_readable_and_cleared():
    """A block-table entry past the pool is recorded (not faulted) in the scratch array's
    error word, which cb_no_alloc_read_error_word returns once and clears."""
    spec = workloads.custom([1, 1, 5], [300, 2000, 40], num_q_heads=16, num_kv_heads=4, seed=8)
    st = GpuStep(spec)
    bt = spec.block_table.copy()
    bt[1, 3] = spec.num_blocks + 7
    st.md["block_table"] = torch.from_numpy(bt).cuda()
    run_no_alloc(st, torch.zeros_like(st.x["q"]))
    assert cb.no_alloc_read_error_word() & cb.CB_DEVERR_BLOCK_ID
    assert cb.no_alloc_read_error_word() == 0
    # the next call starts from a clear word
    st.md["block_table"] = torch.from_numpy(spec.block_table).cuda()
    run_no_alloc(st, torch.zeros_like(st.x["q"]))
    assert cb.no_alloc_read_error_word() == 0


def test_no_alloc_rejects_a_zero_block_size_before_planning():
    spec = workloads.custom([1, 6], [100, 0], num_q_heads=8, num_kv_heads=2, seed=4)
    st = GpuStep(spec)
    s = spec
    out = torch.zeros_like(st.x["q"])
    hq = np.ascontiguousarray(s.query_start_loc, dtype=np.int32)  # kept alive over the call
    hs = np.ascontiguousarray(s.seq_lens, dtype=np.int32)
    status = cb.lib().cb_paged_attention_no_alloc(
        out.data_ptr(), st.x["q"].data_ptr(), st.x["k_cache"].data_ptr(),
        st.x["v_cache"].data_ptr(), None, None, None, st.md["query_start_loc"].data_ptr(),
        st.md["seq_lens"].data_ptr(), st.md["block_table"].data_ptr(),
        int(s.block_table.shape[1]),
        hq.ctypes.data, hs.ctypes.data,
        s.R, s.T, s.num_blocks, 0, s.num_q_heads, s.num_kv_heads, s.head_dim,
        0.0, 0, 1, 0, None)
    assert status == 1  # CB_ERR_INVALID_ARG


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
