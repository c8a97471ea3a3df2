"""GPU: the batched block copy (swap-out / swap-in data movement) and attention over
block tables that share prefix pages, against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_cb_gb300 as cb
import workloads
from stepcheck import GpuStep, compare, oracle_step
from test_gpu_parity import full_check

pytestmark = pytest.mark.gpu


def _pool(nb, bs, hkv, d, dtype, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(nb, bs, hkv, d, generator=g, device="cuda").to(dtype),
            torch.randn(nb, bs, hkv, d, generator=g, device="cuda").to(dtype))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape", [(16, 8, 128), (2, 2, 64), (256, 1, 64)])
def test_copy_within_pool_bit_exact(dtype, shape):
    bs, hkv, d = shape
    nb = 300
    k, v = _pool(nb, bs, hkv, d, dtype, seed=bs + hkv)
    rng = np.random.default_rng(bs)
    perm = rng.permutation(nb)
    src, dst = perm[:120].astype(np.int32), perm[120:240].astype(np.int32)  # disjoint sets
    hk, hv = k.float().cpu().numpy(), v.float().cpu().numpy()
    cb.copy_blocks(k, v, k, v, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda())
    oracle.copy_blocks(hk, hv, hk, hv, src, dst)
    assert np.array_equal(k.float().cpu().numpy(), hk)
    assert np.array_equal(v.float().cpu().numpy(), hv)


def test_bad_ids_are_skipped_and_recorded():
    k, v = _pool(40, 16, 2, 64, torch.bfloat16, seed=3)
    k0, v0 = k.clone(), v.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    src = torch.tensor([5, 41, 7, -1], dtype=torch.int32, device="cuda")
    dst = torch.tensor([20, 21, 40, 23], dtype=torch.int32, device="cuda")
    cb.copy_blocks(k, v, k, v, src, dst, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == cb.CB_DEVERR_BLOCK_ID
    assert torch.equal(k[20], k0[5]) and torch.equal(v[20], v0[5])
    untouched = [b for b in range(40) if b != 20]
    assert torch.equal(k[untouched], k0[untouched]) and torch.equal(v[untouched], v0[untouched])
    # n = 0 launches nothing
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    cb.copy_blocks(k, v, k, v, e, e)


def test_swap_out_and_in_keeps_the_step_bitwise():
    """Swap two requests' context pages out through pinned host memory, let other data
    overwrite them, swap them into other free pages, rewrite the block table: the step
    (decode and prefill rows, through the fast kernels) gives the same bits as before."""
    spec = workloads.custom([1, 1, 300, 1], [700, 2000, 400, 33], seed=77, pool_factor=2.0)
    st = GpuStep(spec)
    k_keep, v_keep = st.x["k_cache"].clone(), st.x["v_cache"].clone()
    out0 = st.run(scatter=False)
    torch.cuda.synchronize()
    moved = [1, 2]
    pages = np.concatenate([spec.block_table[r, :-(-int(spec.ctx_lens[r]) // spec.block_size)]
                            for r in moved]).astype(np.int32)
    n = len(pages)
    kc, vc = st.x["k_cache"], st.x["v_cache"]
    stage_k = torch.empty((n,) + tuple(kc.shape[1:]), dtype=kc.dtype, device="cuda")
    stage_v = torch.empty_like(stage_k)
    ids = torch.arange(n, dtype=torch.int32, device="cuda")
    cb.copy_blocks(kc, vc, stage_k, stage_v, torch.from_numpy(pages).cuda(), ids)  # gather
    host_k = torch.empty(stage_k.shape, dtype=kc.dtype, pin_memory=True)
    host_v = torch.empty_like(host_k, pin_memory=True)
    host_k.copy_(stage_k, non_blocking=True)
    host_v.copy_(stage_v, non_blocking=True)
    torch.cuda.synchronize()
    kc[torch.from_numpy(pages).long().cuda()] = 0.5       # the pages serve other requests now
    vc[torch.from_numpy(pages).long().cuda()] = -0.5
    used = {int(p) for r in range(spec.R)
            for p in spec.block_table[r, :-(-int(spec.seq_lens[r]) // spec.block_size)]}
    free = np.array([p for p in range(workloads.RESERVED_PAGES, spec.num_blocks)
                     if p not in used][:n], dtype=np.int32)
    assert len(free) == n
    stage_k.copy_(host_k, non_blocking=True)
    stage_v.copy_(host_v, non_blocking=True)
    cb.copy_blocks(stage_k, stage_v, kc, vc, ids, torch.from_numpy(free).cuda())  # scatter back
    bt = spec.block_table.copy()
    off = 0
    for r in moved:
        m = -(-int(spec.ctx_lens[r]) // spec.block_size)
        bt[r, :m] = free[off:off + m]
        off += m
    spec2 = workloads.StepSpec(**{**spec.__dict__, "block_table": bt})
    st.spec = spec2
    st.md = workloads.metadata_tensors(spec2, "cuda")
    out1 = st.run(scatter=False)
    torch.cuda.synchronize()
    assert cb.read_error_word(st.ws) == 0
    assert torch.equal(out0, out1)
    # and the pool pages the requests never used are untouched
    keep = [p for p in range(spec.num_blocks) if p not in set(pages.tolist()) | set(free.tolist())]
    assert torch.equal(kc[keep], k_keep[keep]) and torch.equal(vc[keep], v_keep[keep])


@pytest.mark.parametrize("path", ["fast", "portable"])
def test_prefix_shared_pages_parity(path):
    """Requests whose block tables share prefix pages: decodes and a chunked prefill
    read the same physical pages; the step's new tokens go to private pages."""
    base = workloads.custom([1, 1, 200, 1, 64], [512, 600, 1040, 47, 520], seed=12)
    spec = workloads.share_prefix_pages(base, 0, 1, 32)   # 512 tokens shared
    spec = workloads.share_prefix_pages(spec, 0, 2, 32)
    spec = workloads.share_prefix_pages(spec, 0, 4, 30)
    assert (spec.block_table[1, :32] == spec.block_table[2, :32]).all()
    full_check(spec, flags=0 if path == "fast" else cb.CB_FLAG_PORTABLE_ONLY)
