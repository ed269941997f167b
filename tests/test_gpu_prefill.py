"""mla_sparse_prefill (one CTA per token pair, the pair's lists merged into
shared / first-only / second-only segments) against the float64 oracle.

Every token's result is the decode statement over its own list, so the oracle is
the same `sparse_decode`. The lists here reach the merge's corners: identical,
disjoint, empty and nested lists, partial overlaps around the 32-row block size,
slots listed twice (in the first list, in the second, shared or not), an odd
token count, and NaN rows listed by one token of a pair only (which must not
reach the other token, as for an absent entry in the decode)."""
import numpy as np
import pytest
import torch

import oracle
from fp8_mla_kv_gb300 import mlasparse as M
from fp8_mla_kv_gb300 import workloads

from _parity import build_both, check_decode, dev

pytestmark = pytest.mark.gpu

NUM_SLOTS = 16384


def _prefill(cache, db, q=None, topk=None):
    d = dev()
    q = db.q.to(d) if q is None else q
    topk = db.topk.to(d) if topk is None else topk
    out, lse = M.mla_sparse_prefill(q, cache, topk, db.sm_scale)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("name", ["tiny", "nope", "rope", "prefill", "sweep"])
def test_small_configs_match_oracle(name):
    wl = workloads.small(name)
    g, c = build_both(wl)
    db = wl.decode
    out, lse = _prefill(g, db)
    ro, rl, _ = oracle.sparse_decode(db.q, c, db.topk.numpy(), db.sm_scale)
    check_decode(out, lse, ro, rl)
    assert M.mla_get_error() == 0


def test_prefill_full_size_every_token():
    # The prefill-shaped workload at full size (T = 1,024 causal rows of a
    # 1,024-token sequence), in the launch configuration the bench times.
    wl = workloads.prefill()
    g, c = build_both(wl)
    db = wl.decode
    out, lse = _prefill(g, db)
    ro, rl, _ = oracle.sparse_decode(db.q, c, db.topk.numpy(), db.sm_scale)
    check_decode(out, lse, ro, rl)
    assert M.mla_get_error() == 0


def test_paged_prefill_is_the_physical_prefill():
    # Positions through the block table give exactly the physical slots, so the
    # merged lists and the results are the same bits.
    wl = workloads.small("prefill")
    g, _ = build_both(wl)
    db = wl.decode
    d = dev()
    a = M.mla_sparse_prefill(db.q.to(d), g, db.topk.to(d), db.sm_scale)
    bt = wl.block_table.to(torch.int32).to(d)
    b = M.mla_sparse_prefill_paged(db.q.to(d), g, wl.topk_logical.to(d), bt, wl.page_size, db.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))
    assert M.mla_get_error() == 0


def _random_cache(seed):
    gen = torch.Generator().manual_seed(seed)
    n = NUM_SLOTS - 1
    slots = torch.arange(1, NUM_SLOTS, dtype=torch.int64)
    lat = torch.randn((n, 512), generator=gen).to(torch.bfloat16)
    rope = torch.randn((n, 64), generator=gen).to(torch.bfloat16)
    gc = torch.zeros((NUM_SLOTS, 656), dtype=torch.uint8, device=dev())
    M.mla_kv_write(gc, slots.to(dev()), lat.to(dev()), rope.to(dev()))
    cc = np.zeros((NUM_SLOTS, 656), np.uint8)
    oracle.kv_write(cc, slots.numpy(), lat, rope)
    torch.cuda.synchronize()
    return gc, cc


def _corner_lists(W, seed):
    """Lists of 23 tokens (11 pairs and one token alone) built to reach the
    merge's corners; odd pairs scatter their entries among -1."""
    gen = torch.Generator().manual_seed(seed)
    pool = (torch.randperm(NUM_SLOTS - 1, generator=gen) + 1).to(torch.int32)
    cursor = [0]

    def fresh(n):
        v = pool[cursor[0]:cursor[0] + n].clone()
        cursor[0] += n
        return v

    def shuffled(v):
        return v[torch.randperm(v.numel(), generator=gen)]

    pairs = []
    s = fresh(700); pairs.append((s, shuffled(s)))                                  # identical
    pairs.append((fresh(300), fresh(400)))                                          # disjoint
    pairs.append((fresh(0), fresh(100)))                                            # first empty
    pairs.append((fresh(100), fresh(0)))                                            # second empty
    pairs.append((fresh(0), fresh(0)))                                              # both empty
    s = fresh(34); pairs.append((s[:33], shuffled(s)))                              # first inside second
    s = fresh(64); pairs.append((s, s[:31]))                                        # second inside first
    sh, oa, ob = fresh(40), fresh(1), fresh(32)
    pairs.append((shuffled(torch.cat([sh, oa])), shuffled(torch.cat([ob, sh]))))   # 40 shared, 1 + 32 own
    s = fresh(200); pairs.append((torch.cat([s, s[5:6]]), shuffled(s[:150])))      # first lists a slot twice
    s = fresh(200); pairs.append((s, torch.cat([s[:100], s[7:8]])))                # second lists a shared slot twice
    s, o = fresh(200), fresh(1); pairs.append((s, torch.cat([s[:90], o, o])))      # second lists its own slot twice
    lists = [x for p in pairs for x in p] + [fresh(500)]
    rows = []
    for t, v in enumerate(lists):
        row = torch.full((W,), -1, dtype=torch.int32)
        if (t // 2) % 2:
            row[torch.randperm(W, generator=gen)[:v.numel()]] = v
        else:
            row[:v.numel()] = v
        rows.append(row)
    return torch.stack(rows)


def test_merge_corners_match_oracle_and_repeat_bit_identically():
    gc, cc = _random_cache(31)
    W = 1024
    topk = _corner_lists(W, 32)
    T, H = topk.shape[0], 16
    gen = torch.Generator().manual_seed(33)
    q = torch.randn((T, H, 576), generator=gen).to(torch.bfloat16)
    sm = 1.0 / 24.0
    d = dev()
    out, lse = M.mla_sparse_prefill(q.to(d), gc, topk.to(d), sm)
    torch.cuda.synchronize()
    assert M.mla_get_error() == 0
    ro, rl, bad = oracle.sparse_decode(q, cc, topk.numpy(), sm)
    assert bad == 0
    check_decode(out, lse, ro, rl)
    out2, lse2 = M.mla_sparse_prefill(q.to(d), gc, topk.to(d), sm)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))


@pytest.mark.parametrize("H", [1, 20, 48])
def test_head_counts(H):
    wl = workloads.tiny(H=H, T=5)
    g, c = build_both(wl)
    db = wl.decode
    out, lse = _prefill(g, db)
    ro, rl, _ = oracle.sparse_decode(db.q, c, db.topk.numpy(), db.sm_scale)
    check_decode(out, lse, ro, rl)


def _nan_cache():
    """Rows 1..599 random, row 600 written from an all-NaN latent (E4M3 NaN codes)."""
    gen = torch.Generator().manual_seed(41)
    n = 600
    lat = torch.randn((n, 512), generator=gen)
    lat[n - 1] = float("nan")
    lat = lat.to(torch.bfloat16)
    rope = torch.randn((n, 64), generator=gen).to(torch.bfloat16)
    slots = torch.arange(1, n + 1, dtype=torch.int64)
    gc = torch.zeros((4096, 656), dtype=torch.uint8, device=dev())
    M.mla_kv_write(gc, slots.to(dev()), lat.to(dev()), rope.to(dev()))
    cc = np.zeros((4096, 656), np.uint8)
    oracle.kv_write(cc, slots.numpy(), lat, rope)
    torch.cuda.synchronize()
    return gc, cc, n


def test_nan_row_of_one_token_stays_out_of_the_other():
    # Pair 0: the NaN row in the second token's list only; pair 1: in the first
    # token's only; pair 2: in both. A token that does not list the row gets the
    # oracle's finite result; a token that lists it gets NaN out and lse, as the
    # decode (and the oracle) give.
    gc, cc, nan_slot = _nan_cache()
    gen = torch.Generator().manual_seed(42)
    W = 256
    base = (torch.randperm(nan_slot - 1, generator=gen)[:200] + 1).to(torch.int32)
    nan = torch.tensor([nan_slot], dtype=torch.int32)
    lists = [base, torch.cat([base, nan]), torch.cat([nan, base]), base[:150],
             torch.cat([base[:60], nan]), torch.cat([nan, base[10:90]])]
    topk = torch.full((len(lists), W), -1, dtype=torch.int32)
    for t, v in enumerate(lists):
        topk[t, :v.numel()] = v
    T, H = topk.shape[0], 16
    q = torch.randn((T, H, 576), generator=gen).to(torch.bfloat16)
    sm = 1.0 / 24.0
    d = dev()
    out, lse = M.mla_sparse_prefill(q.to(d), gc, topk.to(d), sm)
    dec_out, dec_lse = M.mla_sparse_decode(q.to(d), gc, topk.to(d), sm)
    torch.cuda.synchronize()
    clean = [0, 3]
    ro, rl, _ = oracle.sparse_decode(q, cc, topk.numpy(), sm, tokens=clean)
    check_decode(out, lse, ro, rl, tokens=clean)
    o, do = out.float().cpu(), dec_out.float().cpu()
    assert torch.equal(torch.isnan(o), torch.isnan(do))
    assert torch.isnan(o[[1, 2, 4, 5]]).all()
    assert torch.isnan(lse.cpu()[[1, 2, 4, 5]]).all()
    assert torch.equal(lse.cpu().isneginf(), dec_lse.cpu().isneginf())
    assert torch.equal(lse.cpu().isnan(), dec_lse.cpu().isnan())


def test_slot0_contents_bit_identical():
    wl = workloads.small("prefill")
    res = []
    for b in (0x00, 0xFF, 0x7F):
        g, _ = build_both(wl, slot0_byte=b)
        g[0].fill_(b)
        res.append(tuple(x.cpu() for x in _prefill(g, wl.decode)))
    for o, l in res[1:]:
        assert torch.equal(o.view(torch.int16), res[0][0].view(torch.int16))
        assert torch.equal(l.view(torch.int32), res[0][1].view(torch.int32))


def test_out_of_range_index_is_absent_and_flagged():
    wl = workloads.tiny()
    g, c = build_both(wl)
    M.mla_get_error()
    db = wl.decode
    tk = db.topk.clone()
    tk[1, 90] = wl.num_slots
    tk[2, 3] = 2**31 - 1
    out, lse = _prefill(g, db, topk=tk.to(dev()))
    assert M.mla_get_error() == M.MLA_ERR_DECODE_INDEX_RANGE
    ro, rl, _ = oracle.sparse_decode(db.q, c, tk.numpy(), db.sm_scale)
    check_decode(out, lse, ro, rl)


def test_empty_width_and_no_tokens():
    wl = workloads.tiny(T=3)
    g, _ = build_both(wl)
    d = dev()
    q = wl.decode.q.to(d)
    out, lse = M.mla_sparse_prefill(q, g, torch.empty((3, 0), dtype=torch.int32, device=d), 0.1)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
    out, lse = M.mla_sparse_prefill(q[:0], g, torch.empty((0, 8), dtype=torch.int32, device=d), 0.1)
    assert out.shape == (0, 16, 512)


def test_nope_rows_of_528_bytes():
    wl = workloads.small("nope")
    g, c = build_both(wl)
    db = wl.decode
    g528 = g[:, :528].contiguous()
    a = _prefill(g, db)
    b = _prefill(g528, db)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))
    ro, rl, _ = oracle.sparse_decode(db.q, c, db.topk.numpy(), db.sm_scale)
    check_decode(*b, ro, rl)


def test_paged_multi_sequence_holes_and_range():
    # Tokens of three sequences (a pair may mix two block tables), unassigned
    # pages, positions past the table (absent and flagged) and repeated positions
    # (a slot listed twice): the pairs' merged lists against the oracle.
    wl = workloads.small("sweep")
    g, c = build_both(wl)
    rng = np.random.default_rng(4)
    T, H, W, page, n_seq, max_pages = 7, 16, 96, 16, 3, 40
    n_pages = wl.num_slots // page
    bt = rng.integers(1, n_pages, size=(n_seq, max_pages)).astype(np.int32)
    bt[rng.random(bt.shape) < 0.1] = -1
    pos = rng.integers(-1, max_pages * page + 40, size=(T, W)).astype(np.int32)
    seq = rng.integers(0, n_seq, size=T).astype(np.int32)
    q = torch.from_numpy(rng.standard_normal((T, H, 576)).astype(np.float32)).to(torch.bfloat16)
    d = dev()
    M.mla_get_error()
    out, lse = M.mla_sparse_prefill_paged(q.to(d), g, torch.from_numpy(pos).to(d), torch.from_numpy(bt).to(d),
                                          page, 0.05, token_seq=torch.from_numpy(seq).to(d))
    torch.cuda.synchronize()
    err = M.mla_get_error()
    phys, bad = oracle.paged_to_physical(pos, bt, page, seq)
    assert bad > 0 and err == M.MLA_ERR_DECODE_INDEX_RANGE
    ro, rl, _ = oracle.sparse_decode(q, c, phys, 0.05)
    check_decode(out, lse, ro, rl)
