"""Pins for the CPU oracle: values and facts that come from the pages or from mathematics,
not from the oracle itself.

* the worked example of "Continuous Batching" (languisher.top), sections
  "Optimisation: the mask as offsets" and "Extension: the vLLM v1
  implementation" (tests/golden/worked_example.json);
* a dense brute force with an explicit block-diagonal causal mask over the
  packed stream (section "Attention Mask construction"), written here without
  any of the oracle's helpers;
* the library special case: one request with no context equals causal
  scaled-dot-product attention (torch, float64, CPU);
* invariants: physical page placement, decode vs last prefill row, chunked vs
  one-shot prefill, a request alone vs inside a batch;
* closed forms: one KV token, Q = 0, window 1, window >= seq_len;
* planted mistakes: each plausible bug in the oracle's steps makes one of the
  pins above fail.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import oracle.paged_kv as opa
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")


# ------------------------------------------------------------ helpers (test-side)


def place_logical(cache, block_table_row, values, block_size):
    """Write a request's logical rows into its pages (test-side, flat-slot formulation)."""
    nb, bs, hkv, d = cache.shape
    flat = cache.reshape(nb * bs, hkv, d)
    n = values.shape[0]
    slots = np.array([block_table_row[p // block_size] * block_size + p % block_size for p in range(n)],
                     dtype=np.int64)
    flat[slots] = values


def make_case(q_lens, ctx_lens, Hq, Hkv, D, BS, seed, scale=None, window=0, q_scale=1.0,
              num_blocks=None):
    """Random step with per-request logical KV kept aside for the brute force."""
    spec = workloads.custom(q_lens, ctx_lens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                            block_size=BS, dtype="f32", seed=seed, scale=scale,
                            sliding_window=window, num_blocks=num_blocks)
    rng = np.random.default_rng(seed + 99)
    T = spec.T
    q = rng.standard_normal((T, Hq, D)) * q_scale
    k_new = rng.standard_normal((T, Hkv, D))
    v_new = rng.standard_normal((T, Hkv, D))
    k_cache = rng.standard_normal((spec.num_blocks, BS, Hkv, D))
    v_cache = rng.standard_normal((spec.num_blocks, BS, Hkv, D))
    logical_k, logical_v = [], []
    for r in range(spec.R):
        ctx = int(ctx_lens[r])
        ck = rng.standard_normal((ctx, Hkv, D))
        cv = rng.standard_normal((ctx, Hkv, D))
        place_logical(k_cache, spec.block_table[r], ck, BS)
        place_logical(v_cache, spec.block_table[r], cv, BS)
        t0 = int(spec.query_start_loc[r])
        t1 = int(spec.query_start_loc[r + 1])
        logical_k.append(np.concatenate([ck, k_new[t0:t1]], axis=0))
        logical_v.append(np.concatenate([cv, v_new[t0:t1]], axis=0))
    return spec, dict(q=q, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache,
                      logical_k=logical_k, logical_v=logical_v)


def run_oracle(spec, x, rows=None):
    out, kc, vc = oracle.step(x["q"], x["k_cache"], x["v_cache"], x["k_new"], x["v_new"],
                              spec.slot_mapping, spec.query_start_loc, spec.seq_lens,
                              spec.block_table, spec.block_size, spec.scale, spec.sliding_window,
                              rows)
    return out, kc, vc


def dense_brute_force(spec, x):
    """Explicit [T, N] block-diagonal causal mask over the packed logical KV stream."""
    q = x["q"]
    T, Hq, D = q.shape
    Hkv = spec.num_kv_heads
    G = Hq // Hkv
    kv_k = np.concatenate(x["logical_k"], axis=0)
    kv_v = np.concatenate(x["logical_v"], axis=0)
    kv_req = np.concatenate([np.full(k.shape[0], r) for r, k in enumerate(x["logical_k"])])
    kv_pos = np.concatenate([np.arange(k.shape[0]) for k in x["logical_k"]])
    q_req = np.concatenate([np.full(int(n), r) for r, n in enumerate(spec.q_lens)])
    q_pos = np.concatenate([int(c) + np.arange(int(n)) for c, n in zip(spec.ctx_lens, spec.q_lens)])
    mask = (kv_req[None, :] == q_req[:, None]) & (kv_pos[None, :] <= q_pos[:, None])
    if spec.sliding_window > 0:
        mask &= kv_pos[None, :] > (q_pos[:, None] - spec.sliding_window)
    out = np.zeros_like(q)
    for h in range(Hq):
        S = spec.scale * q[:, h, :] @ kv_k[:, h // G, :].T
        S = np.where(mask, S, -np.inf)
        S = S - S.max(axis=1, keepdims=True)
        P = np.exp(S)
        P /= P.sum(axis=1, keepdims=True)
        out[:, h, :] = P @ kv_v[:, h // G, :]
    return out


CASES = [
    # (q_lens, ctx_lens, Hq, Hkv, D, BS, window)
    ([4, 2, 3, 1], [0, 0, 5, 8], 4, 2, 8, 2, 0),
    ([1, 7, 1, 5], [12, 0, 3, 9], 8, 2, 16, 4, 0),
    ([3, 1, 6], [0, 20, 11], 4, 4, 8, 8, 5),
    ([2, 9, 1, 1], [17, 1, 0, 30], 8, 1, 4, 2, 3),
]


# ------------------------------------------------------------ worked example


def test_worked_example_index_mapping_and_ranges():
    with open(GOLDEN) as f:
        g = json.load(f)
    pr = g["printed"]
    rd = g["readings"]
    BS = pr["BLOCK_SIZE"]
    qsl = np.array(rd["query_start_loc"], dtype=np.int32)
    # the printed seq_start_loc is the first R entries of the reading
    assert list(qsl[:-1]) == pr["seq_start_loc"]
    assert list(np.diff(qsl)) == pr["seq_len"]
    # the printed lookup: kv_pos 1 of C -> logical block 0, offset 1, physical 7
    lk = pr["lookup"]
    blk, off = oracle.resolve(pr["block_table_C"], lk["kv_pos"], BS)
    assert (lk["kv_pos"] // BS, off, blk) == (lk["logical_block"], lk["block_offset"],
                                              lk["physical_block"])

    # Build the step: every token has a one-hot id row as V and K; Q = 0.
    tokens = pr["tokens"]
    n = len(tokens)
    D = 16
    Hq = Hkv = 1
    seq_lens = np.array(pr["seq_len"], dtype=np.int32)  # ctx = 0 for all three
    bt = np.zeros((3, 2), dtype=np.int32)
    bt[0, :2] = rd["block_table_A"]
    bt[1, :1] = rd["block_table_B"]
    bt[2, :2] = pr["block_table_C"]
    slots = []
    for r in range(3):
        for i in range(int(seq_lens[r])):
            slots.append(bt[r][i // BS] * BS + i % BS)
    slots = np.array(slots, dtype=np.int64)
    ids = np.eye(n, D)
    k_new = ids[:, None, :].copy()
    v_new = ids[:, None, :].copy()
    k_cache = np.full((20, BS, Hkv, D), 7.0)
    v_cache = np.full((20, BS, Hkv, D), 7.0)
    q = np.zeros((n, Hq, D))
    out, kc, vc = oracle.step(q, k_cache, v_cache, k_new, v_new, slots, qsl, seq_lens, bt, BS,
                              scale=1.0)
    # after the scatter, physical block 7 offset 1 holds c1
    c1 = tokens.index(lk["token"])
    assert np.array_equal(vc[7, 1, 0], ids[c1])
    # Q = 0: each row is the mean of exactly the ids in [start, start + local_pos]
    for t in range(n):
        r = int(np.searchsorted(qsl, t, side="right") - 1)
        start = int(qsl[r])
        local = t - start
        expect = np.zeros(D)
        expect[start:start + local + 1] = 1.0 / (local + 1)
        assert np.allclose(out[t, 0], expect, atol=1e-15, rtol=0), t
    # a sharp query for c2 that matches c1's key returns c1's id
    c2 = tokens.index("c2")
    q2 = np.zeros((n, Hq, D))
    q2[c2, 0, c1] = 60.0
    out2, _, _ = oracle.step(q2, k_cache, v_cache, k_new, v_new, slots, qsl, seq_lens, bt, BS,
                             scale=1.0)
    assert int(np.argmax(out2[c2, 0])) == c1
    assert out2[c2, 0, c1] > 1 - 1e-12


# ------------------------------------------------------------ brute force / SDPA


@pytest.mark.parametrize("case", CASES)
def test_dense_brute_force(case):
    q_lens, ctx_lens, Hq, Hkv, D, BS, W = case
    spec, x = make_case(q_lens, ctx_lens, Hq, Hkv, D, BS, seed=len(q_lens) * 7 + D, window=W,
                        q_scale=2.0)
    out, _, _ = run_oracle(spec, x)
    ref = dense_brute_force(spec, x)
    assert np.max(np.abs(out - ref)) <= 1e-12


@pytest.mark.parametrize("G", [1, 2, 4])
def test_single_request_equals_causal_sdpa(G):
    n, Hkv, D, BS = 13, 2, 16, 4
    Hq = G * Hkv
    spec, x = make_case([n], [0], Hq, Hkv, D, BS, seed=5 + G, q_scale=1.5)
    out, _, _ = run_oracle(spec, x)
    qt = torch.from_numpy(x["q"]).permute(1, 0, 2)[None]  # [1, Hq, n, D]
    kt = torch.from_numpy(x["k_new"]).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    vt = torch.from_numpy(x["v_new"]).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True,
                                                           scale=spec.scale)
    ref = ref[0].permute(1, 0, 2).numpy()
    assert np.max(np.abs(out - ref)) <= 1e-12


def test_scale_argument_is_applied():
    spec, x = make_case([6], [0], 4, 2, 8, 2, seed=3, scale=0.37)
    out, _, _ = run_oracle(spec, x)
    qt = torch.from_numpy(x["q"]).permute(1, 0, 2)[None]
    kt = torch.from_numpy(x["k_new"]).permute(1, 0, 2).repeat_interleave(2, dim=0)[None]
    vt = torch.from_numpy(x["v_new"]).permute(1, 0, 2).repeat_interleave(2, dim=0)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=0.37)
    assert np.max(np.abs(out - ref[0].permute(1, 0, 2).numpy())) <= 1e-12


# ------------------------------------------------------------ invariants


def test_physical_page_permutation_is_bitwise_invariant():
    spec, x = make_case([3, 1, 5, 2], [6, 10, 0, 4], 8, 2, 8, 4, seed=11)
    out, _, _ = run_oracle(spec, x)
    rng = np.random.default_rng(0)
    nb = spec.num_blocks
    perm = np.arange(nb)
    perm[2:] = 2 + rng.permutation(nb - 2)  # reserved pages stay put
    kc = np.empty_like(x["k_cache"])
    vc = np.empty_like(x["v_cache"])
    kc[perm] = x["k_cache"]
    vc[perm] = x["v_cache"]
    bt = perm[spec.block_table].astype(np.int32)
    slots = perm[spec.slot_mapping // spec.block_size] * spec.block_size \
        + spec.slot_mapping % spec.block_size
    out2, _, _ = oracle.step(x["q"], kc, vc, x["k_new"], x["v_new"], slots,
                             spec.query_start_loc, spec.seq_lens, bt, spec.block_size, spec.scale)
    assert np.array_equal(out, out2)


def test_decode_equals_last_row_of_prefill():
    n = 11
    spec, x = make_case([n], [0], 4, 2, 8, 4, seed=21)
    out, kc, vc = run_oracle(spec, x)
    # decode of the last token over the (now written) cache: ctx = n-1, q_len = 1
    qsl = np.array([0, 1], np.int32)
    seq = np.array([n], np.int32)
    dec = oracle.paged_attention(x["q"][n - 1:n], kc, vc, qsl, seq, spec.block_table,
                                 spec.block_size, spec.scale)
    assert np.array_equal(dec[0], out[n - 1])


def test_chunked_prefill_equals_one_shot():
    n, c1 = 14, 5
    spec, x = make_case([n], [0], 4, 2, 8, 2, seed=31)
    full, _, _ = run_oracle(spec, x)
    bt = spec.block_table
    BS = spec.block_size
    kc = x["k_cache"].copy()
    vc = x["v_cache"].copy()
    outs = []
    for lo, hi in ((0, c1), (c1, n)):
        qsl = np.array([0, hi - lo], np.int32)
        seq = np.array([hi], np.int32)
        slots = spec.slot_mapping[lo:hi]
        o, kc, vc = oracle.step(x["q"][lo:hi], kc, vc, x["k_new"][lo:hi], x["v_new"][lo:hi], slots,
                                qsl, seq, bt, BS, spec.scale)
        outs.append(o)
    assert np.array_equal(np.concatenate(outs), full)


def test_request_alone_equals_request_in_batch():
    spec, x = make_case([2, 5, 1, 3], [4, 0, 9, 2], 4, 2, 8, 2, seed=41)
    out, _, _ = run_oracle(spec, x)
    r = 1
    t0, t1 = int(spec.query_start_loc[r]), int(spec.query_start_loc[r + 1])
    qsl = np.array([0, t1 - t0], np.int32)
    alone, _, _ = oracle.step(x["q"][t0:t1], x["k_cache"], x["v_cache"], x["k_new"][t0:t1],
                              x["v_new"][t0:t1], spec.slot_mapping[t0:t1], qsl,
                              spec.seq_lens[r:r + 1], spec.block_table[r:r + 1],
                              spec.block_size, spec.scale)
    assert np.array_equal(alone, out[t0:t1])


# ------------------------------------------------------------ closed forms


def test_single_kv_token_returns_v():
    spec, x = make_case([1], [0], 4, 2, 8, 2, seed=51)
    out, _, _ = run_oracle(spec, x)
    G = 2
    for h in range(4):
        assert np.array_equal(out[0, h], x["v_new"][0, h // G])


def test_zero_query_gives_mean_of_attended_v():
    spec, x = make_case([3, 1], [4, 6], 4, 2, 8, 2, seed=61, window=0)
    x["q"][:] = 0.0
    out, _, _ = run_oracle(spec, x)
    for r in range(2):
        for i in range(int(spec.q_lens[r])):
            t = int(spec.query_start_loc[r]) + i
            upto = int(spec.ctx_lens[r]) + i
            for h in range(4):
                mean = x["logical_v"][r][:upto + 1, h // 2].mean(axis=0)
                assert np.allclose(out[t, h], mean, atol=1e-14, rtol=0)


def test_window_one_returns_own_v():
    spec, x = make_case([3, 1], [4, 6], 4, 2, 8, 2, seed=71, window=1)
    out, _, _ = run_oracle(spec, x)
    for t in range(spec.T):
        for h in range(4):
            assert np.array_equal(out[t, h], x["v_new"][t, h // 2])


def test_window_at_least_seq_len_equals_full():
    spec, x = make_case([3, 2], [5, 1], 4, 2, 8, 2, seed=81, window=0)
    full, _, _ = run_oracle(spec, x)
    spec.sliding_window = 8
    win, _, _ = run_oracle(spec, x)
    assert np.array_equal(full, win)


def test_scatter_roundtrip_and_untouched_pages():
    spec, x = make_case([3, 4], [5, 0], 4, 2, 8, 4, seed=91)
    kc = x["k_cache"].copy()
    vc = x["v_cache"].copy()
    oracle.scatter_kv(kc, vc, x["k_new"], x["v_new"], spec.slot_mapping)
    used = set()
    for r in range(spec.R):
        t0 = int(spec.query_start_loc[r])
        for i in range(int(spec.q_lens[r])):
            p = int(spec.ctx_lens[r]) + i
            blk = int(spec.block_table[r][p // spec.block_size])
            off = p % spec.block_size
            assert np.array_equal(kc[blk, off], x["k_new"][t0 + i])
            assert np.array_equal(vc[blk, off], x["v_new"][t0 + i])
            used.add((blk, off))
    for b in range(spec.num_blocks):
        for o in range(spec.block_size):
            if (b, o) not in used:
                assert np.array_equal(kc[b, o], x["k_cache"][b, o])


def test_scatter_skips_negative_slots():
    kc = np.zeros((4, 2, 1, 2))
    vc = np.zeros((4, 2, 1, 2))
    k_new = np.ones((3, 1, 2))
    v_new = 2 * np.ones((3, 1, 2))
    oracle.scatter_kv(kc, vc, k_new, v_new, np.array([5, -1, 0]))
    assert kc.reshape(8, 1, 2)[5, 0, 0] == 1 and vc.reshape(8, 1, 2)[0, 0, 0] == 2
    assert np.count_nonzero(kc) == 4


# ------------------------------------------------------------ planted mistakes


MUTANTS = {
    "causal bound excludes self": ("kv_range", lambda c, i, w: (0 if w <= 0 else max(0, c + i - w + 1), c + i - 1 if c + i > 0 else 0)),
    "causal bound one too far": ("kv_range", lambda c, i, w: (0 if w <= 0 else max(0, c + i - w + 1), c + i + 1)),
    "window off by one": ("kv_range", lambda c, i, w: (0 if w <= 0 else max(0, c + i - w), c + i)),
    "context dropped": ("kv_range", lambda c, i, w: (c if w <= 0 else max(c, c + i - w + 1), c + i)),
    "block index uses offset": ("resolve", lambda row, p, bs, ring=0: (int(row[p % bs]), p // bs)),
    "offset ignores block": ("resolve", lambda row, p, bs, ring=0: (int(row[0]), p % bs)),
    "no scale": ("softmax_attend", lambda qh, K, V, s: _attend(qh, K, V, 1.0)),
    "scale squared": ("softmax_attend", lambda qh, K, V, s: _attend(qh, K, V, s * s)),
    "softmax over heads": ("softmax_attend", lambda qh, K, V, s: _attend_wrong_axis(qh, K, V, s)),
    "V rows reversed": ("softmax_attend", lambda qh, K, V, s: _attend(qh, K, V[::-1], s)),
}


def _attend(qh, K, V, s):
    S = s * (qh @ K.T)
    S = S - S.max(axis=1, keepdims=True)
    w = np.exp(S)
    return (w / w.sum(axis=1, keepdims=True)) @ V


def _attend_wrong_axis(qh, K, V, s):
    S = s * (qh @ K.T)
    w = np.exp(S - S.max(axis=0, keepdims=True))
    return (w / w.sum(axis=0, keepdims=True)) @ V


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(opa, attr, fn)
    caught = False
    for case in CASES:
        q_lens, ctx_lens, Hq, Hkv, D, BS, W = case
        spec, x = make_case(q_lens, ctx_lens, Hq, Hkv, D, BS, seed=len(q_lens) * 7 + D, window=W,
                            q_scale=2.0)
        try:
            out, _, _ = run_oracle(spec, x)
        except (IndexError, ValueError):
            caught = True
            break
        ref = dense_brute_force(spec, x)
        if not np.all(np.isfinite(out)) or np.max(np.abs(out - ref)) > 1e-9:
            caught = True
            break
    assert caught, name


def test_gqa_mapping_is_pinned_by_brute_force():
    """Interleaved head grouping (h % Hkv) instead of contiguous groups would differ."""
    q_lens, ctx_lens, Hq, Hkv, D, BS, W = CASES[1]
    spec, x = make_case(q_lens, ctx_lens, Hq, Hkv, D, BS, seed=3, q_scale=2.0)
    out, _, _ = run_oracle(spec, x)
    # permute q heads so that head h uses kv head h % Hkv under the contiguous rule
    G = Hq // Hkv
    perm = np.array([(h % Hkv) * G + h // Hkv for h in range(Hq)])
    x2 = dict(x)
    x2["q"] = x["q"][:, perm]
    ref = dense_brute_force(spec, x)
    alt = dense_brute_force(spec, x2)[:, np.argsort(perm)]
    assert np.max(np.abs(out - ref)) < 1e-12
    assert np.max(np.abs(out - alt)) > 1e-3


def test_generators_are_seeded_and_consistent():
    a = workloads.tiny_mixed()
    b = workloads.tiny_mixed()
    assert np.array_equal(a.block_table, b.block_table)
    assert list(a.seq_lens) == [4, 2, 8, 9] and a.T == 10
    assert a.block_table.max() < a.num_blocks and a.block_table[a.block_table > 0].min() >= 2
    # pages of different requests are disjoint
    used = [p for r in range(a.R) for p in a.block_table[r][:math.ceil(a.seq_lens[r] / 2)]]
    assert len(used) == len(set(used)) == 12
    d = workloads.decode_step()
    assert d.R == 64 and d.T == 64 and 128 <= d.seq_lens.min() and d.seq_lens.max() <= 2048
    m = workloads.mixed_step()
    assert m.T == 2048 and list(m.q_lens[-2:]) == [960, 960] and list(m.ctx_lens[-2:]) == [0, 3072]


# ------------------------------------------------------------------ block copy and aliasing


def _free_pages(spec):
    used = {int(p) for r in range(spec.R)
            for p in spec.block_table[r, :-(-int(spec.seq_lens[r]) // spec.block_size)]}
    return [p for p in range(workloads.RESERVED_PAGES, spec.num_blocks) if p not in used]


def test_copy_blocks_swap_roundtrip_restores_the_request():
    """Swap a request's context pages out to a staging buffer, clobber them, swap them in
    to other free pages: its KV read through the new block table is the old KV bit for
    bit, and the step's output is unchanged."""
    spec, x = make_case([1, 4, 1], [9, 6, 13], 4, 2, 8, 2, seed=123, num_blocks=48)
    out0, _, _ = run_oracle(spec, x)
    r = 2
    n = -(-int(spec.ctx_lens[r]) // spec.block_size)  # pages that hold context
    pages = spec.block_table[r, :n].copy()
    kc, vc = x["k_cache"].copy(), x["v_cache"].copy()
    before_k = opa.gather_request_kv(kc, spec.block_table[r], int(spec.ctx_lens[r]), spec.block_size)
    before_v = opa.gather_request_kv(vc, spec.block_table[r], int(spec.ctx_lens[r]), spec.block_size)
    sk = np.zeros((n,) + kc.shape[1:])
    sv = np.zeros_like(sk)
    oracle.copy_blocks(sk, sv, kc, vc, pages, np.arange(n))          # swap out
    rng = np.random.default_rng(5)
    kc[pages] = rng.standard_normal(kc[pages].shape)                 # pages reused by others
    vc[pages] = rng.standard_normal(vc[pages].shape)
    new_pages = np.array(_free_pages(spec)[:n], dtype=np.int32)
    assert len(new_pages) == n
    oracle.copy_blocks(kc, vc, sk, sv, np.arange(n), new_pages)      # swap in elsewhere
    bt = spec.block_table.copy()
    bt[r, :n] = new_pages
    after_k = opa.gather_request_kv(kc, bt[r], int(spec.ctx_lens[r]), spec.block_size)
    after_v = opa.gather_request_kv(vc, bt[r], int(spec.ctx_lens[r]), spec.block_size)
    assert np.array_equal(after_k, before_k) and np.array_equal(after_v, before_v)
    # the step's own tokens land where the new table says
    slots = spec.slot_mapping.copy()
    t0 = int(spec.query_start_loc[r])
    for i in range(int(spec.q_lens[r])):
        p = int(spec.ctx_lens[r]) + i
        slots[t0 + i] = int(bt[r, p // spec.block_size]) * spec.block_size + p % spec.block_size
    out1, _, _ = oracle.step(x["q"], kc, vc, x["k_new"], x["v_new"], slots, spec.query_start_loc,
                             spec.seq_lens, bt, spec.block_size, spec.scale)
    assert np.array_equal(out0, out1)


def test_copy_blocks_moves_k_and_v_and_nothing_else():
    rng = np.random.default_rng(8)
    k = rng.standard_normal((12, 2, 1, 4))
    v = rng.standard_normal((12, 2, 1, 4))
    k0, v0 = k.copy(), v.copy()
    src, dst = np.array([3, 7, 5]), np.array([9, 2, 11])
    oracle.copy_blocks(k, v, k, v, src, dst)
    for s, d in zip(src, dst):
        assert np.array_equal(k[d], k0[s]) and np.array_equal(v[d], v0[s])
    keep = [b for b in range(12) if b not in set(dst.tolist())]
    assert np.array_equal(k[keep], k0[keep]) and np.array_equal(v[keep], v0[keep])


def test_shared_prefix_pages_equal_private_copies():
    """Two requests whose block tables name the same physical prefix pages get exactly
    the output they get when each owns a private copy of those pages."""
    spec, x = make_case([1, 3], [8, 8], 4, 2, 8, 4, seed=31)
    shared = 2  # the first two pages (8 tokens) of request 0 serve request 1's prefix too
    kc, vc = x["k_cache"].copy(), x["v_cache"].copy()
    bt_private = spec.block_table.copy()
    # private layout: request 1's prefix pages hold a copy of request 0's
    oracle.copy_blocks(kc, vc, kc, vc, bt_private[0, :shared], bt_private[1, :shared])
    out_private, _, _ = oracle.step(x["q"], kc, vc, x["k_new"], x["v_new"], spec.slot_mapping,
                                    spec.query_start_loc, spec.seq_lens, bt_private,
                                    spec.block_size, spec.scale)
    bt_shared = spec.block_table.copy()
    bt_shared[1, :shared] = bt_shared[0, :shared]
    out_shared, _, _ = oracle.step(x["q"], kc, vc, x["k_new"], x["v_new"], spec.slot_mapping,
                                   spec.query_start_loc, spec.seq_lens, bt_shared,
                                   spec.block_size, spec.scale)
    assert np.array_equal(out_private, out_shared)
    # and the shared prefix really is what request 1 attends: against a wrong prefix it differs
    kc[bt_private[1, 0]] += 1.0
    out_wrong, _, _ = oracle.step(x["q"], kc, vc, x["k_new"], x["v_new"], spec.slot_mapping,
                                  spec.query_start_loc, spec.seq_lens, bt_private,
                                  spec.block_size, spec.scale)
    t1 = int(spec.query_start_loc[1])
    assert not np.array_equal(out_wrong[t1:], out_shared[t1:])


# ------------------------------------------------------------------ ring-recycled sliding pages


def _ring_layout(spec, x, ring, rng):
    """The plain case's logical K/V laid out in rings of `ring` pages per request: the
    window's positions hold their values; older positions of the ring hold garbage."""
    bs, R = spec.block_size, spec.R
    nb = workloads.RESERVED_PAGES + R * ring
    shape = (nb, bs) + x["k_cache"].shape[2:]
    kc = rng.standard_normal(shape) * 1e3  # garbage everywhere first
    vc = rng.standard_normal(shape) * 1e3
    pages = workloads.RESERVED_PAGES + rng.permutation(R * ring)
    bt = pages.reshape(R, ring).astype(np.int32)
    slots = spec.slot_mapping.copy()
    for r in range(R):
        ctx, seq = int(spec.ctx_lens[r]), int(spec.seq_lens[r])
        lo = max(0, ctx - spec.sliding_window + 1)
        for p in range((lo // bs) * bs, ctx):  # context positions the step can read
            e = (p // bs) % ring
            kc[bt[r, e], p % bs] = x["logical_k"][r][p]
            vc[bt[r, e], p % bs] = x["logical_v"][r][p]
        t0 = int(spec.query_start_loc[r])
        for i in range(seq - ctx):  # the step's new tokens go through the ring too
            p = ctx + i
            slots[t0 + i] = int(bt[r, (p // bs) % ring]) * bs + p % bs
    return kc, vc, bt, slots


def test_ring_covering_every_block_equals_the_plain_table():
    spec, x = make_case([3, 1, 6], [20, 37, 9], 8, 2, 8, 4, seed=61, window=11)
    out, _, _ = run_oracle(spec, x)
    out_r, _, _ = oracle.step(x["q"], x["k_cache"], x["v_cache"], x["k_new"], x["v_new"],
                              spec.slot_mapping, spec.query_start_loc, spec.seq_lens,
                              spec.block_table, spec.block_size, spec.scale, spec.sliding_window,
                              ring_blocks=spec.block_table.shape[1])
    assert np.array_equal(out, out_r)


@pytest.mark.parametrize("window,extra", [(11, 0), (7, 2), (1, 0)])
def test_ring_layout_equals_plain_layout(window, extra):
    spec, x = make_case([3, 1, 6, 2], [20, 37, 9, 0], 8, 2, 8, 4, seed=62, window=window)
    out, _, _ = run_oracle(spec, x)
    bs = spec.block_size
    need = max((int(spec.seq_lens[r]) - 1) // bs
               - max(0, int(spec.ctx_lens[r]) - window + 1) // bs + 1 for r in range(spec.R))
    ring = need + extra
    kc, vc, bt, slots = _ring_layout(spec, x, ring, np.random.default_rng(3))
    out_r, _, _ = oracle.step(x["q"], kc, vc, x["k_new"], x["v_new"], slots, spec.query_start_loc,
                              spec.seq_lens, bt, bs, spec.scale, window, ring_blocks=ring)
    assert np.array_equal(out, out_r)
    # a ring index off by one reads the garbage and the output moves
    if ring > 1:
        bad = np.roll(bt, 1, axis=1)
        out_b, _, _ = oracle.step(x["q"], kc, vc, x["k_new"], x["v_new"], slots,
                                  spec.query_start_loc, spec.seq_lens, bad, bs, spec.scale, window,
                                  ring_blocks=ring)
        assert not np.allclose(out, out_b)
