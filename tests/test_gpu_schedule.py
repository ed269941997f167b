"""The decode's work split against the float64 oracle.

With fewer (token, head group) units than the GPU has SMs, a first kernel
compacts each token's list, the decode cuts every list into pieces of at most C
present entries (C chosen so that all pieces fit in one wave of CTAs, so a long
list gets more pieces than a short one) and a third kernel merges each token's
partials; with more units, one CTA takes one unit whole. The lists here are built to reach the corners of
both: tokens with no present entry, one entry, 31 / 32 / 33 entries (a block
boundary), full lists, present entries scattered among -1 or packed at the
front, and head counts that leave a short last head group.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_mla_kv_gb300 import mlasparse as M

from _parity import check_decode, dev

pytestmark = pytest.mark.gpu

NUM_SLOTS = 16384


def _cache(seed, nope=False):
    g = torch.Generator().manual_seed(seed)
    n = NUM_SLOTS - 1
    slots = torch.arange(1, NUM_SLOTS, dtype=torch.int64)
    lat = torch.randn((n, 512), generator=g).to(torch.bfloat16)
    rope = None if nope else torch.randn((n, 64), generator=g).to(torch.bfloat16)
    gc = torch.zeros((NUM_SLOTS, 656), dtype=torch.uint8, device=dev())
    M.mla_kv_write(gc, slots.to(dev()), lat.to(dev()), None if rope is None else rope.to(dev()))
    cc = np.zeros((NUM_SLOTS, 656), np.uint8)
    oracle.kv_write(cc, slots.numpy(), lat, rope)
    torch.cuda.synchronize()
    return gc, cc


def _topk(counts, W, seed):
    g = torch.Generator().manual_seed(seed)
    rows = []
    for t, cnt in enumerate(counts):
        row = torch.full((W,), -1, dtype=torch.int32)
        pick = (torch.randperm(NUM_SLOTS - 1, generator=g)[:cnt] + 1).to(torch.int32)
        if t % 2:
            row[torch.randperm(W, generator=g)[:cnt]] = pick       # scattered among -1
        else:
            row[:cnt] = pick                                        # packed at the front
        rows.append(row)
    return torch.stack(rows)


def _run(counts, H, W, seed, d_qk=576, tokens=None):
    gc, cc = _cache(seed, nope=(d_qk == 512))
    T = len(counts)
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn((T, H, d_qk), generator=g).to(torch.bfloat16)
    topk = _topk(counts, W, seed + 2)
    sm = 1.0 / d_qk ** 0.5
    out, lse = M.mla_sparse_decode(q.to(dev()), gc, topk.to(dev()), sm)
    torch.cuda.synchronize()
    assert M.mla_get_error() == 0
    ro, rl, bad = oracle.sparse_decode(q, cc, topk.numpy(), sm, tokens=tokens)
    assert bad == 0
    check_decode(out, lse, ro, rl, tokens=tokens)
    return q, gc, topk, sm, out, lse


def test_split_lists_with_empty_short_and_full_lists():
    counts = [0, 1, 31, 32, 33, 1024, 500, 0, 2, 777] * 4
    q, gc, topk, sm, out, lse = _run(counts, 16, 1024, seed=21)
    # Same inputs again: the merge order is fixed, so the result is bit-identical.
    out2, lse2 = M.mla_sparse_decode(q.to(dev()), gc, topk.to(dev()), sm)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))


def test_split_lists_with_a_short_last_head_group():
    # H = 20: head groups of 16 and 4.
    _run([2000, 0, 1500, 3, 999], 20, 2000, seed=22)


def test_split_lists_nope_rows():
    _run([900, 450, 1, 0, 64, 899, 300], 16, 900, seed=23, d_qk=512)


def test_planned_split_one_long_list_among_short_ones():
    # One full 2,304-entry list among 32 one-entry lists: the long list is cut into
    # many pieces (more than one merge batch of partials), the short ones into one.
    out = _run([2304] + [1] * 32, 16, 2304, seed=26)
    # The same call again is bit-identical (the plan and the merge order are fixed).
    q, gc, topk, sm, o1, l1 = out
    o2, l2 = M.mla_sparse_decode(q.to(dev()), gc, topk.to(dev()), sm)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_planned_split_near_the_sm_count_sampled():
    # 150 tokens (just under one unit per SM) with lists up to 2,304 entries: the
    # pieces just fit in one wave; compared on a sample of tokens.
    rng = np.random.default_rng(27)
    counts = rng.integers(0, 2305, size=150).tolist()
    counts[:4] = [2304, 0, 2304, 1]
    tokens = sorted(set(rng.choice(150, 12, replace=False).tolist()) | {0, 1, 2, 3, 149})
    _run(counts, 16, 2304, seed=27, tokens=tokens)


def test_planned_split_paged_with_holes_and_range():
    # The planned split through the block table: 6 tokens of 1,024 positions over
    # 3 sequences, unassigned pages and positions past the table (absent and flagged).
    gc, cc = _cache(28)
    rng = np.random.default_rng(28)
    T, H, W, page, n_seq, max_pages = 6, 16, 1024, 16, 3, 200
    bt = rng.permutation(np.arange(1, NUM_SLOTS // page))[: n_seq * max_pages].astype(np.int32).reshape(n_seq, max_pages)
    bt[rng.random(bt.shape) < 0.1] = -1
    pos = np.stack([rng.permutation(max_pages * page + 64)[:W] for _ in range(T)]).astype(np.int32)
    pos[rng.random(pos.shape) < 0.2] = -1
    pos[4, :] = -1                                          # an empty list
    seq = rng.integers(0, n_seq, size=T).astype(np.int32)
    q = torch.from_numpy(rng.standard_normal((T, H, 576)).astype(np.float32)).to(torch.bfloat16)
    assert M.mla_sparse_decode_workspace_bytes(T, H, W) > 0, "this case is meant to split"
    M.mla_get_error()
    out, lse = M.mla_sparse_decode_paged(q.to(dev()), gc, torch.from_numpy(pos).to(dev()),
                                         torch.from_numpy(bt).to(dev()), page, 0.05,
                                         token_seq=torch.from_numpy(seq).to(dev()))
    torch.cuda.synchronize()
    phys, bad = oracle.paged_to_physical(pos, bt, page, seq)
    assert bad > 0 and M.mla_get_error() == M.MLA_ERR_DECODE_INDEX_RANGE
    ro, rl, _ = oracle.sparse_decode(q, cc, phys, 0.05)
    check_decode(out, lse, ro, rl)


def test_many_units_random_counts_sampled():
    # 300 tokens with random counts: more units than SMs, one CTA per unit;
    # compared on a sample of tokens.
    rng = np.random.default_rng(24)
    counts = rng.integers(0, 601, size=300).tolist()
    counts[:3] = [0, 0, 0]
    tokens = sorted(set(rng.choice(300, 50, replace=False).tolist()) | {0, 1, 2, 299})
    _run(counts, 16, 600, seed=24, tokens=tokens)


def test_whole_units_many_tokens_sampled():
    # 1,300 tokens of 700 positions, one CTA per unit.
    rng = np.random.default_rng(25)
    counts = rng.integers(0, 700, size=1300).tolist()
    tokens = sorted(set(rng.choice(1300, 40, replace=False).tolist()) | {0, 1299})
    _run(counts, 16, 700, seed=25, tokens=tokens)
