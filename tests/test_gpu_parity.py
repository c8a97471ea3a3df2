"""GPU parity: the C-ABI path on cuda:0 against the CPU oracle on the same seeded inputs.

Scatter: bit-exact on the whole pool except the reserved pages 0-1.
Attention: bf16 within max-abs 2e-2 and mean-abs 2e-3; fp32 within max-abs 1e-4.
The mixed step is checked whole at full size; the other full-size steps on sampled rows
the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_cb_gb300 as cb
import workloads
from stepcheck import (GpuStep, cache_bits, compare, oracle_cache_bits, oracle_step, sample_rows)

pytestmark = pytest.mark.gpu

PATHS = {"fast": 0, "portable": cb.CB_FLAG_PORTABLE_ONLY}


def check_scatter(st, k_before, v_before):
    """K and V caches after the step: bit-exact against the oracle's scatter, outside the
    reserved pages 0-1 (where padding rows may land)."""
    spec = st.spec
    for name, before in (("k", k_before), ("v", v_before)):
        want = oracle_cache_bits(spec, before, st.x[name + "_new"], spec.slot_mapping)
        got = cache_bits(st.x[name + "_cache"])
        assert np.array_equal(got[2:], want[2:]), name


def full_check(spec, flags=0, scale=None, max_abs=None, mean_abs=None):
    st = GpuStep(spec)
    h = st.host_inputs()
    k_before, v_before = st.x["k_cache"].clone(), st.x["v_cache"].clone()
    out = st.run(flags=flags, scale=scale)
    torch.cuda.synchronize()
    assert cb.read_error_word(st.ws) == 0
    ref = oracle_step(spec, h, scale=scale)
    mx, mn = compare(spec, out, ref, max_abs=max_abs, mean_abs=mean_abs)
    check_scatter(st, k_before, v_before)
    return mx, mn


# ------------------------------------------------------------------ tiny fp32 step


@pytest.mark.parametrize("path", sorted(PATHS))
def test_tiny_mixed_fp32(path):
    full_check(workloads.tiny_mixed(), flags=PATHS[path])


# ------------------------------------------------------------------ randomised small cases

SMALL = []
for q_len in (1, 2, 17, 128, 129):
    for ctx in (0, 1, 15, 16, 17, 1000):
        SMALL.append((q_len, ctx))


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("BS", [2, 16])
@pytest.mark.parametrize("path", sorted(PATHS))
def test_small_ragged_bf16(G, BS, path):
    # all (q_len, ctx) combinations as one ragged step, plus an empty request
    q_lens = [q for q, _ in SMALL] + [0]
    ctx = [c for _, c in SMALL] + [5]
    Hkv = 2
    spec = workloads.custom(q_lens, ctx, num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=128,
                            block_size=BS, seed=100 + G * 10 + BS)
    full_check(spec, flags=PATHS[path])


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_head_dims_and_dtypes(D, dtype):
    spec = workloads.custom([1, 5, 1, 33], [40, 0, 7, 100], num_q_heads=8, num_kv_heads=2,
                            head_dim=D, block_size=16, dtype=dtype, seed=7 + D)
    full_check(spec)


@pytest.mark.parametrize("window", [1, 7, 16, 100])
def test_sliding_window(window):
    spec = workloads.custom([1, 20, 1, 64], [300, 50, 16, 0], num_q_heads=16, num_kv_heads=4,
                            block_size=16, seed=window, sliding_window=window)
    full_check(spec)


def test_sharp_softmax():
    """Scale x8 makes the softmax peaked so the tolerance bites on the largest weights."""
    spec = workloads.custom([1, 1, 40, 1], [500, 33, 64, 2000], num_q_heads=32, num_kv_heads=8,
                            seed=9)
    full_check(spec, scale=8.0 / np.sqrt(128.0))


# ------------------------------------------------------------------ full-size steps


def sampled_check(spec, n_rows=64, flags=0):
    st = GpuStep(spec)
    h = st.host_inputs()
    k_before, v_before = st.x["k_cache"].clone(), st.x["v_cache"].clone()
    out = st.run(flags=flags)
    torch.cuda.synchronize()
    assert cb.read_error_word(st.ws) == 0
    rows = sample_rows(spec, n_rows)
    ref = oracle_step(spec, h, rows=rows)
    check_scatter(st, k_before, v_before)
    return compare(spec, out, ref, rows=rows)


def test_decode_64_full_size():
    sampled_check(workloads.decode_step(), n_rows=64)


def test_mixed_2048_full_size():
    """The whole mixed step (128 decode rows and two 960-token chunks, 2048 rows x 32 heads)
    against the oracle: max-abs and mean-abs over every output element."""
    full_check(workloads.mixed_step())


@pytest.mark.parametrize("window", [0, 4096])
def test_long_decode_full_size(window):
    sampled_check(workloads.long_decode(window=window), n_rows=16)


# ------------------------------------------------------------------ invariants on the GPU


def test_physical_page_permutation_is_bitwise_invariant():
    spec = workloads.custom([1, 9, 1, 30], [77, 0, 500, 40], num_q_heads=32, num_kv_heads=8,
                            seed=3)
    st = GpuStep(spec)
    out1 = st.run(scatter=True).clone()
    # relabel pages: new_cache[perm[p]] = cache[p]; tables and slots follow
    rng = np.random.default_rng(1)
    nb = spec.num_blocks
    perm = np.arange(nb)
    perm[2:] = 2 + rng.permutation(nb - 2)
    pt = torch.from_numpy(perm).cuda()
    st2 = GpuStep(spec)
    kc = torch.empty_like(st2.x["k_cache"])
    vc = torch.empty_like(st2.x["v_cache"])
    kc[pt] = st2.x["k_cache"]
    vc[pt] = st2.x["v_cache"]
    st2.x["k_cache"], st2.x["v_cache"] = kc, vc
    bt = perm[spec.block_table].astype(np.int32)
    slots = perm[spec.slot_mapping // spec.block_size] * spec.block_size \
        + spec.slot_mapping % spec.block_size
    st2.md["block_table"] = torch.from_numpy(bt).cuda()
    st2.md["slot_mapping"] = torch.from_numpy(slots).cuda()
    out2 = st2.run(scatter=True)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)


def test_request_alone_equals_request_in_batch():
    spec = workloads.custom([1, 37, 1], [900, 300, 64], num_q_heads=32, num_kv_heads=8, seed=4)
    st = GpuStep(spec)
    out = st.run()
    # request 1 alone, same pages and values
    r = 1
    t0, t1 = int(spec.query_start_loc[r]), int(spec.query_start_loc[r + 1])
    alone = workloads.StepSpec(**{**spec.__dict__})
    alone.q_lens = spec.q_lens[r:r + 1]
    alone.ctx_lens = spec.ctx_lens[r:r + 1]
    alone.query_start_loc = np.array([0, t1 - t0], np.int32)
    alone.seq_lens = spec.seq_lens[r:r + 1]
    alone.block_table = spec.block_table[r:r + 1]
    alone.slot_mapping = spec.slot_mapping[t0:t1]
    st2 = GpuStep(alone)
    st2.x["k_cache"].copy_(st.x["k_cache"])  # already holds the scattered tokens
    st2.x["v_cache"].copy_(st.x["v_cache"])
    st2.x["q"] = st.x["q"][t0:t1].contiguous()
    out2 = st2.run(scatter=False)
    torch.cuda.synchronize()
    assert torch.equal(out[t0:t1], out2)


def test_out_of_range_block_id_is_recorded_not_faulted():
    spec = workloads.custom([1, 3], [40, 10], num_q_heads=8, num_kv_heads=2, seed=5)
    st = GpuStep(spec)
    bt = spec.block_table.copy()
    bt[0, 1] = spec.num_blocks + 5  # past the pool
    st.md["block_table"] = torch.from_numpy(bt).cuda()
    st.run(scatter=False)
    torch.cuda.synchronize()
    assert cb.read_error_word(st.ws) & 0x1
    assert cb.read_error_word(st.ws) == 0  # cleared by the read


def test_out_of_range_slot_is_recorded_and_skipped():
    spec = workloads.custom([2], [3], num_q_heads=8, num_kv_heads=2, seed=6)
    st = GpuStep(spec)
    slots = spec.slot_mapping.copy()
    slots[0] = spec.num_blocks * spec.block_size + 3
    slots[1] = -1
    before = st.x["k_cache"].clone()
    cb.write_kv(st.x["k_new"], st.x["v_new"], st.x["k_cache"], st.x["v_cache"],
                torch.from_numpy(slots).cuda(), error_word=st.ws.view(torch.int32)[:1])
    torch.cuda.synchronize()
    assert torch.equal(before, st.x["k_cache"])
    assert cb.read_error_word(st.ws) & 0x2


def test_decode_step_scatter_skips_negative_and_records_out_of_range_slots():
    """A step of decode rows only writes its rows from the decode kernel itself: a slot
    below zero is skipped, one past the pool is recorded (0x2) and skipped, the rest land
    bit-exactly and the rows whose slot was written attend to their new K/V."""
    spec = workloads.custom([1] * 5, [40, 700, 3, 1500, 90], num_q_heads=16, num_kv_heads=4,
                            seed=21)
    st = GpuStep(spec)
    slots = spec.slot_mapping.copy()
    slots[1] = -1
    slots[3] = spec.num_blocks * spec.block_size + 5
    st.md["slot_mapping"] = torch.from_numpy(slots).cuda()
    h = st.host_inputs()
    k_before, v_before = st.x["k_cache"].clone(), st.x["v_cache"].clone()
    out = st.run()
    torch.cuda.synchronize()
    assert cb.read_error_word(st.ws) & 0x2
    kept = slots.copy()
    kept[3] = -1  # what the kernel did with the slot past the pool: nothing
    for name, before in (("k", k_before), ("v", v_before)):
        want = oracle_cache_bits(spec, before, st.x[name + "_new"], kept)
        assert np.array_equal(cache_bits(st.x[name + "_cache"])[2:], want[2:]), name
    # rows 0, 2, 4 attend to their new K/V; rows 1 and 3 to what the cache held
    oracle.scatter_kv(h["k_cache"], h["v_cache"], h["k_new"], h["v_new"], kept)
    ref = oracle.paged_attention(h["q"], h["k_cache"], h["v_cache"], spec.query_start_loc,
                                 spec.seq_lens, spec.block_table, spec.block_size, spec.scale)
    compare(spec, out, ref)


def test_mixed_step_scatter_skips_negative_and_records_out_of_range_slots():
    """In a step with prefill rows the tile kernel reads the step's own positions from
    k_new / v_new where their slot is their own, and from the cache otherwise: a
    prefill row with slot -1 (or past the pool: recorded, skipped) leaves its cache
    position as it was, and the rows attending to it see that old value, as the
    oracle's scatter-then-attend has it. Context lengths off the page boundary make
    pages that straddle the context end."""
    spec = workloads.custom([1, 40, 1, 19], [300, 21, 1000, 7], num_q_heads=32, num_kv_heads=8,
                            seed=27)
    st = GpuStep(spec)
    slots = spec.slot_mapping.copy()
    q0 = int(spec.query_start_loc[1])  # the 40-token chunk
    slots[q0 + 3] = -1
    slots[q0 + 17] = spec.num_blocks * spec.block_size + 9
    slots[int(spec.query_start_loc[3]) + 5] = -1  # inside the 19-token prompt
    st.md["slot_mapping"] = torch.from_numpy(slots).cuda()
    h = st.host_inputs()
    k_before, v_before = st.x["k_cache"].clone(), st.x["v_cache"].clone()
    out = st.run()
    torch.cuda.synchronize()
    assert cb.read_error_word(st.ws) & 0x2
    kept = slots.copy()
    kept[q0 + 17] = -1
    for name, before in (("k", k_before), ("v", v_before)):
        want = oracle_cache_bits(spec, before, st.x[name + "_new"], kept)
        assert np.array_equal(cache_bits(st.x[name + "_cache"])[2:], want[2:]), name
    oracle.scatter_kv(h["k_cache"], h["v_cache"], h["k_new"], h["v_new"], kept)
    ref = oracle.paged_attention(h["q"], h["k_cache"], h["v_cache"], spec.query_start_loc,
                                 spec.seq_lens, spec.block_table, spec.block_size, spec.scale)
    compare(spec, out, ref)


def test_bf16_steps_launch_no_separate_scatter():
    """Steps whose rows all run on the tensor-core kernels write their new K/V from
    those kernels: decode-only, prefill-only and mixed steps launch no scatter kernel."""
    names = cb.kernel_names()
    wk = names.index("write_kv")
    for q_lens, ctx in (([1, 1, 1], [100, 2000, 5]), ([30, 200], [0, 64]),
                        ([1, 30, 1], [700, 16, 9])):
        spec = workloads.custom(q_lens, ctx, num_q_heads=32, num_kv_heads=8, seed=len(ctx))
        st = GpuStep(spec)
        h = st.host_inputs()
        before = cb.launch_count(wk)
        out = st.run()
        torch.cuda.synchronize()
        assert cb.launch_count(wk) == before, (q_lens, ctx)
        assert cb.read_error_word(st.ws) == 0
        compare(spec, out, oracle_step(spec, h))


@pytest.mark.parametrize("case", ["long_context_chunks", "window", "g1_d64", "g16"])
def test_prefill_long_context_chunks(case):
    """Chunks over long contexts, each (tile pair, KV head) CTA walking many key tiles,
    with windows, G 1 with head_dim 64, and G 16."""
    if case == "long_context_chunks":
        spec = workloads.custom([100, 300, 1], [20000, 5000, 700], num_q_heads=32,
                                num_kv_heads=8, seed=41)
    elif case == "window":
        spec = workloads.custom([200, 64], [12000, 3000], num_q_heads=32, num_kv_heads=8,
                                seed=42, sliding_window=2500)
    elif case == "g1_d64":
        spec = workloads.custom([150, 40], [9000, 16000], num_q_heads=4, num_kv_heads=4,
                                head_dim=64, seed=43)
    else:
        spec = workloads.custom([90, 33], [7000, 4000], num_q_heads=32, num_kv_heads=2,
                                seed=44)
    full_check(spec)


# ------------------------------------------------------------------ decode kernel coverage


@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (4, 4), (16, 8), (32, 16), (64, 8), (16, 1), (64, 4)])
@pytest.mark.parametrize("BS", [8, 16, 32, 256])
def test_decode_heads_and_block_sizes(Hq, Hkv, BS):
    rng = np.random.default_rng(Hq * 100 + Hkv + BS)
    ctx = [int(c) for c in rng.integers(0, 3000, size=12)] + [0, 15, 16, 31]
    spec = workloads.custom([1] * len(ctx), ctx, num_q_heads=Hq, num_kv_heads=Hkv,
                            block_size=BS, seed=BS + Hkv)
    full_check(spec)


def test_bf16_decode_shapes_run_on_the_tensor_core_kernels():
    """G = 16 decode (two 8-head column blocks per KV head) and 8-key pages (two page
    boxes per 16-key block) run on the split-KV kernel, not the CUDA-core one."""
    names = cb.kernel_names()
    split, portable = names.index("decode_split"), names.index("portable_attention")
    for Hq, Hkv, BS in ((16, 1, 16), (64, 4, 16), (32, 8, 8), (16, 1, 8)):
        spec = workloads.custom([1] * 6, [0, 15, 700, 2100, 40, 3000], num_q_heads=Hq,
                                num_kv_heads=Hkv, block_size=BS, seed=Hq + Hkv + BS)
        st = GpuStep(spec)
        h = st.host_inputs()
        s0, p0 = cb.launch_count(split), cb.launch_count(portable)
        out = st.run()
        torch.cuda.synchronize()
        assert cb.launch_count(split) > s0 and cb.launch_count(portable) == p0, (Hq, Hkv, BS)
        assert cb.read_error_word(st.ws) == 0
        compare(spec, out, oracle_step(spec, h))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("window", [0, 1, 33, 1000])
def test_decode_split_across_ctas(D, window):
    """Few long requests: each spans many CTAs, so the combine merges many partials."""
    spec = workloads.custom([1, 1, 1], [20000, 9000, 300], num_q_heads=16, num_kv_heads=4,
                            head_dim=D, seed=D + window, sliding_window=window)
    full_check(spec)


def test_split_requests_repeat_bitwise_on_one_workspace():
    """Requests split over several CTAs and merged by the combine kernel: repeated steps on
    one workspace agree bitwise (no partial of one step leaks into the next)."""
    spec = workloads.custom([1] * 6, [30000, 5, 17000, 64, 9000, 2048], num_q_heads=64,
                            num_kv_heads=8, seed=12)
    st = GpuStep(spec)
    first = st.run().clone()
    for _ in range(3):
        again = st.run()
        torch.cuda.synchronize()
        assert torch.equal(first, again)
    assert cb.read_error_word(st.ws) == 0


# ------------------------------------------------------------------ prefill tile kernel coverage


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("BS", [8, 32, 256])
def test_prefill_groups_and_block_sizes(G, BS):
    Hkv = 2
    spec = workloads.custom([2, 37, 130, 300], [0, 200, 5, 1000], num_q_heads=G * Hkv,
                            num_kv_heads=Hkv, block_size=BS, seed=G * 7 + BS)
    full_check(spec)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("window", [0, 50, 300])
def test_prefill_chunks_with_context(D, window):
    """A prompt continued in chunks: context in the cache, own tokens through slot_mapping."""
    spec = workloads.custom([129, 256, 64], [3000, 0, 700], num_q_heads=16, num_kv_heads=4,
                            head_dim=D, seed=D + window, sliding_window=window)
    full_check(spec)


def test_prefill_requests_over_several_launches_repeat_bitwise():
    """More prompt requests than one prefill launch lists: the launches of a step claim
    their units from one counter in the workspace header, which each launch's last CTA
    sets back to zero, so a second run of the step on the same workspace is bitwise equal."""
    rng = np.random.default_rng(23)
    n = 300
    q_lens = [int(x) for x in rng.integers(2, 10, n)]
    ctx = [int(x) for x in rng.integers(0, 300, n)]
    spec = workloads.custom(q_lens, ctx, num_q_heads=8, num_kv_heads=2, block_size=16, seed=23)
    full_check(spec)
    st = GpuStep(spec)
    first = st.run().clone()
    again = st.run()
    torch.cuda.synchronize()
    assert cb.read_error_word(st.ws) == 0
    assert torch.equal(first, again)


def test_prefill_fast_equals_portable_path():
    spec = workloads.custom([1, 70, 1, 200], [90, 400, 3, 0], num_q_heads=32, num_kv_heads=8,
                            seed=17)
    st = GpuStep(spec)
    fast = st.run().float()
    port = st.run(flags=cb.CB_FLAG_PORTABLE_ONLY).float()
    torch.cuda.synchronize()
    err = (fast - port).abs()
    assert float(err.max()) <= 2e-2 and float(err.mean()) <= 2e-3


@pytest.mark.parametrize("D,G", [(128, 4), (64, 8), (128, 1), (128, 16)])
def test_prefill_output_at_a_16_byte_offset_equals_aligned(D, G):
    """The prefill kernel writes O in 32-byte pieces where `out` is 32-byte aligned and in
    16-byte ones otherwise (the boundary asks for 16-byte alignment only): both give the
    same bits, every row of every request is written (the buffers start as NaN) and nothing
    past the last request's last token (a ragged tile) or before the output."""
    spec = workloads.custom([37, 300, 5, 129], [0, 200, 90, 7], num_q_heads=2 * G,
                            num_kv_heads=2, head_dim=D, seed=23)
    st = GpuStep(spec)
    h = st.host_inputs()
    aligned = st.run()
    assert aligned.data_ptr() % 32 == 0
    n, guard = aligned.numel(), 4096
    buf = torch.full((8 + n + guard,), float("nan"), dtype=aligned.dtype, device=aligned.device)
    shifted = buf[8:8 + n].view(aligned.shape)
    assert shifted.data_ptr() % 32 == 16
    st.run(out=shifted)
    torch.cuda.synchronize()
    assert cb.read_error_word(st.ws) == 0
    assert not torch.isnan(aligned.float()).any()
    assert torch.equal(aligned.view(torch.int16), shifted.view(torch.int16))
    assert torch.isnan(buf[:8].float()).all() and torch.isnan(buf[8 + n:].float()).all()
    compare(spec, aligned, oracle_step(spec, h))


# ------------------------------------------------------------------ ring-recycled sliding pages


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("D", [64, 128])
def test_ring_recycled_sliding_pages(path, D):
    """Sliding-window layer on rings of recycled pages: decodes, a chunk whose queries
    span several windows, a prompt start; the step's tokens scattered through the ring."""
    spec = workloads.ring_step([1, 1, 200, 1, 37, 64], [3000, 129, 500, 0, 2000, 0], window=300,
                               num_q_heads=16, num_kv_heads=4, head_dim=D, seed=D + 5)
    assert spec.ring_blocks < spec.seq_lens.max() // spec.block_size
    full_check(spec, flags=PATHS[path])


@pytest.mark.parametrize("BS", [8, 16, 64])
def test_ring_with_spare_entries(BS):
    base = workloads.ring_step([1, 130, 1], [777, 300, 64], window=96, block_size=BS, seed=BS)
    spec = workloads.ring_step([1, 130, 1], [777, 300, 64], window=96, block_size=BS, seed=BS,
                               ring_blocks=base.ring_blocks + 3)
    full_check(spec)


def test_long_decode_ring_full_size():
    spec = workloads.long_decode_ring()
    assert spec.ring_blocks == 256 and spec.block_table.shape[1] == 256  # window 4096 from 28672
    sampled_check(spec, n_rows=16)


# ------------------------------------------------------------------ workspace reuse


def test_workspace_reused_across_growing_request_counts():
    """One workspace for a 40-request step with many split requests, then a 256-request
    step: the larger step's split-merge counters must read zero, not where the smaller
    step left partial results (the workspace layout follows its size, not the step)."""
    ws = cb.alloc_workspace(256, 256, 32, 8, 128)
    small = GpuStep(workloads.decode_step(seed=22, R=40, lo=4096, hi=8192))
    small.ws = ws
    small.run()
    torch.cuda.synchronize()
    big_spec = workloads.decode_step(seed=21, R=256, lo=1024, hi=6000)
    big = GpuStep(big_spec)
    big.ws = ws
    h = big.host_inputs()
    out = big.run()
    torch.cuda.synchronize()
    assert cb.read_error_word(ws) == 0
    assert torch.isfinite(out.float()).all()
    rows = sample_rows(big_spec, 16)
    ref = oracle_step(big_spec, h, rows=rows)
    compare(big_spec, out, ref, rows=rows)
    # and back down: a small step after the large one on the same workspace
    again = small.run()
    torch.cuda.synchronize()
    assert torch.isfinite(again.float()).all()
