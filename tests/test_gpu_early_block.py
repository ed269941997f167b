"""GPU parity for the decode's early first block: when the first 32 positions of a
CTA's list are all present, its first copy-issuing warp copies them before the
list is compacted. Lists built around that rule (exactly 32 present, 31, a reserved
or out-of-range entry among the first 32, duplicates, entries of every kind after
them, a list split by positions, the paged entry point with an unassigned page)
must give what the float64 oracle gives, and out-of-range entries must still be
flagged."""
import numpy as np
import pytest
import torch

import oracle
from fp8_mla_kv_gb300 import mlasparse as M
from fp8_mla_kv_gb300 import workloads

from _parity import build_both, check_decode, dev

pytestmark = pytest.mark.gpu


def _lists(num_slots: int, W: int, rng: np.random.Generator) -> np.ndarray:
    def fresh(n):
        return rng.choice(np.arange(1, num_slots), size=n, replace=False).astype(np.int32)

    tk = np.full((8, W), -1, np.int32)
    tk[0, :32] = fresh(32)                                    # exactly one full block, then nothing
    tk[1, :32] = fresh(32)                                    # a full block, then every kind of entry
    tail = fresh(W - 32)
    kinds = rng.integers(0, 6, size=W - 32)
    tail[kinds == 1] = -1
    tail[kinds == 2] = 0                                      # the reserved slot
    tail[kinds == 3] = num_slots                              # one past the end: absent, flagged
    tail[kinds == 4] = tk[1, rng.integers(0, 32, size=int((kinds == 4).sum()))]   # duplicates
    tk[1, 32:] = tail
    tk[2, :] = fresh(W)
    tk[2, 31] = -1                                            # 31 present first: the usual path
    tk[3, :] = fresh(W)
    tk[3, 0] = 0                                              # the reserved slot first
    tk[4, :] = fresh(W)
    tk[4, 17] = 2**31 - 1                                     # out of range among the first 32
    tk[5, :] = fresh(W)                                       # all present
    # tk[6]: empty
    tk[7, :32] = fresh(32)
    tk[7, 5] = tk[7, 20]                                      # a duplicate inside the first block
    tk[7, 40:60] = fresh(20)
    return tk


def test_early_block_lists_match_oracle():
    wl = workloads.tiny(T=8, W=160)
    g, c = build_both(wl)
    db = wl.decode
    tk = _lists(wl.num_slots, 160, np.random.default_rng(5))
    M.mla_get_error()
    out, lse = M.mla_sparse_decode(db.q.to(dev()), g, torch.from_numpy(tk).to(dev()), db.sm_scale)
    torch.cuda.synchronize()
    assert M.mla_get_error() == M.MLA_ERR_DECODE_INDEX_RANGE
    ref_out, ref_lse, _ = oracle.sparse_decode(db.q, c, tk, db.sm_scale)
    check_decode(out, lse, ref_out, ref_lse)


def test_early_block_in_every_piece_of_a_list_split_by_positions():
    # 5,000 positions are more than one CTA compacts: the list is split by positions
    # and every piece whose first 32 positions are present takes the early path.
    wl = workloads.tiny(T=1, W=128)
    g, c = build_both(wl)
    rng = np.random.default_rng(9)
    W = 5000
    tk = rng.integers(1, wl.num_slots, size=(1, W)).astype(np.int32)
    tk[0, rng.integers(0, W, size=300)] = -1
    tk[0, :32] = rng.integers(1, wl.num_slots, size=32)      # the first piece's block 0 is whole
    q = torch.randn((1, 16, 576), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    ws = M.alloc_workspace(1, 16, W, dev())
    out, lse = M.mla_sparse_decode(q.to(dev()), g, torch.from_numpy(tk).to(dev()), 0.07, workspace=ws)
    torch.cuda.synchronize()
    ref_out, ref_lse, _ = oracle.sparse_decode(q, c, tk, 0.07)
    check_decode(out, lse, ref_out, ref_lse)
    assert M.mla_get_error() == 0


def test_early_block_through_the_block_table():
    # Positions of one sequence in 16-slot pages, logical page 3 unassigned and a
    # position past the table: the early path maps the first 32 positions with the
    # same rules as the compaction, or leaves the block to it.
    wl = workloads.tiny(T=8, W=160)
    g, c = build_both(wl)
    db = wl.decode
    rng = np.random.default_rng(21)
    page = 16
    n_pages = wl.num_slots // page
    table_pages = 40
    bt = rng.permutation(np.arange(1, n_pages))[:table_pages].astype(np.int32)[None, :]
    bt[0, 3] = -1
    pos = np.full((8, 160), -1, np.int32)
    for t in range(8):
        p = rng.permutation(np.arange(table_pages * page))[:160].astype(np.int32)
        if t % 2 == 0:
            p[:32] = rng.permutation(np.arange(0, 48))[:32]   # first 32 in assigned pages 0-2
        if t == 3:
            p[7] = 3 * page + 5                               # an unassigned page among the first 32
        if t == 5:
            p[9] = table_pages * page + 1                     # past the table: absent, flagged
        if t == 6:
            p[:] = -1
        pos[t] = p
    M.mla_get_error()
    out, lse = M.mla_sparse_decode_paged(db.q.to(dev()), g, torch.from_numpy(pos).to(dev()),
                                         torch.from_numpy(bt).to(dev()), page, db.sm_scale)
    torch.cuda.synchronize()
    assert M.mla_get_error() == M.MLA_ERR_DECODE_INDEX_RANGE
    phys, n_past = oracle.paged_to_physical(pos, bt, page)
    assert n_past == 1
    ref_out, ref_lse, _ = oracle.sparse_decode(db.q, c, phys, db.sm_scale)
    check_decode(out, lse, ref_out, ref_lse)
