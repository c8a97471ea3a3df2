"""The bounded-wait failure path of the tensor-core kernels, exercised without a fault.

Every pipeline wait in the decode and prefill kernels is bounded: when one gives up,
the kernel records CB_DEVERR_TIMEOUT in the error word, the kernel's other warps stop
waiting, the copies and tensor-core products already in flight are waited for, the
tensor memory is freed and the kernel returns, so the context stays usable.
CB_FLAG_TEST_WAIT_EXPIRY makes one consumer-side wait of each kernel run out after a
few polls (it waits on a barrier nothing arrives at). These tests check that the call
returns, that the timeout is recorded, and that the next step on the same buffers,
after cb_workspace_init, matches the oracle.
"""
import pytest
import torch

import paged_kv_attention_cb_gb300 as cb
import workloads
from stepcheck import GpuStep, compare, oracle_step

pytestmark = pytest.mark.gpu

CASES = {
    # decode rows only: the decode kernel (and its fused scatter) alone
    "decode": lambda: workloads.custom([1] * 6, [40, 700, 3, 1500, 90, 20000], num_q_heads=16,
                                       num_kv_heads=4, seed=31),
    # prefill rows only: the tile kernel, one and two query tiles per CTA
    "prefill": lambda: workloads.custom([37, 130, 300], [64, 0, 1000], num_q_heads=32,
                                        num_kv_heads=8, seed=32),
    # both kinds in one step
    "mixed": lambda: workloads.custom([1, 200, 1, 9], [3000, 100, 17, 0], num_q_heads=32,
                                      num_kv_heads=8, seed=33),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_expired_wait_is_recorded_and_the_next_step_is_exact(name):
    spec = CASES[name]()
    st = GpuStep(spec)
    h = st.host_inputs()
    st.run(flags=cb.CB_FLAG_TEST_WAIT_EXPIRY)
    torch.cuda.synchronize()  # the kernels returned
    word = cb.read_error_word(st.ws)
    assert word & cb.CB_DEVERR_TIMEOUT, word
    # the context is usable and the workspace reusable after re-initialisation
    cb.workspace_init(st.ws)
    out = st.run()
    torch.cuda.synchronize()
    assert cb.read_error_word(st.ws) == 0
    compare(spec, out, oracle_step(spec, h))


def test_repeated_expiry_then_normal_steps():
    """Several aborted steps in a row leave nothing behind that a later step sees."""
    spec = CASES["mixed"]()
    st = GpuStep(spec)
    h = st.host_inputs()
    for _ in range(3):
        st.run(flags=cb.CB_FLAG_TEST_WAIT_EXPIRY)
    torch.cuda.synchronize()
    assert cb.read_error_word(st.ws) & cb.CB_DEVERR_TIMEOUT
    cb.workspace_init(st.ws)
    ref = oracle_step(spec, h)
    for _ in range(2):
        out = st.run()
        torch.cuda.synchronize()
        assert cb.read_error_word(st.ws) == 0
        compare(spec, out, ref)
