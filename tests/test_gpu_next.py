"""GPU parity of the widened path against the oracle, through the C ABI:
528-byte NoPE rows (writer and decode), the paged decode (top-k as sequence
positions through a block table), and gather-and-upconvert to BF16."""
import numpy as np
import pytest
import torch

import oracle
from fp8_mla_kv_gb300 import mlasparse as M
from fp8_mla_kv_gb300 import workloads

from _parity import build_both, check_decode, dev, gpu_decode

pytestmark = pytest.mark.gpu


def _nope528(wl):
    """A workload's NoPE fill and writes into 528-byte caches on both sides."""
    g = torch.full((wl.num_slots, 528), wl.slot0_byte, dtype=torch.uint8, device=dev())
    c = np.full((wl.num_slots, 528), wl.slot0_byte, np.uint8)
    d = dev()
    for wb in ([wl.fill] if wl.fill is not None else []) + list(wl.writes):
        assert wb.rope is None
        M.mla_kv_write(g, wb.slot_idx.to(d), wb.latent.to(d), None)
        oracle.kv_write(c, wb.slot_idx.numpy(), wb.latent, None)
    torch.cuda.synchronize()
    return g, c


# ------------------------------------------------------------ 528-byte rows
@pytest.mark.parametrize("full", [False, True])
def test_528_rows_writer_and_decode(full):
    wl = workloads.nope() if full else workloads.small("nope")
    g528, c528 = _nope528(wl)
    assert M.mla_get_error() == 0
    assert np.array_equal(g528.cpu().numpy(), c528), "528-byte cache differs from the oracle's"
    db = wl.decode
    out, lse = gpu_decode(g528, db)
    ro, rl, _ = oracle.sparse_decode(db.q, c528, db.topk.numpy(), db.sm_scale)
    check_decode(out, lse, ro, rl)
    # the same rows in 656-byte form give the same bits
    g656, _ = build_both(wl)
    out6, lse6 = gpu_decode(g656, db)
    assert torch.equal(out.view(torch.int16), out6.view(torch.int16))
    assert torch.equal(lse, lse6)
    assert M.mla_get_error() == 0


def test_528_rows_refuse_rope_calls():
    g = torch.zeros((64, 528), dtype=torch.uint8, device=dev())
    d = dev()
    with pytest.raises(M.MlaError):
        M.mla_kv_write(g, torch.tensor([1], dtype=torch.int64, device=d),
                       torch.zeros((1, 512), dtype=torch.bfloat16, device=d),
                       torch.zeros((1, 64), dtype=torch.bfloat16, device=d))
    with pytest.raises(M.MlaError):
        M.mla_sparse_decode(torch.zeros((1, 16, 576), dtype=torch.bfloat16, device=d), g,
                            torch.ones((1, 8), dtype=torch.int32, device=d), 0.1)


# ------------------------------------------------------------ paged decode
@pytest.mark.parametrize("full", [False, True])
def test_paged_prefill_equals_physical(full):
    wl = workloads.prefill() if full else workloads.small("prefill")
    g, c = build_both(wl)
    db = wl.decode
    d = dev()
    ref_out, ref_lse = gpu_decode(g, db)
    out, lse = M.mla_sparse_decode_paged(db.q.to(d), g, wl.topk_logical.to(d),
                                         wl.block_table.to(torch.int32).to(d), wl.page_size, db.sm_scale)
    torch.cuda.synchronize()
    assert M.mla_get_error() == 0
    # the same slots in the same order: the same bits as the physical-slot decode
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lse, ref_lse)
    phys, bad = oracle.paged_to_physical(wl.topk_logical.numpy(), wl.block_table.numpy(), wl.page_size)
    assert bad == 0
    ro, rl, _ = oracle.sparse_decode(db.q, c, phys, db.sm_scale)
    check_decode(out, lse, ro, rl)


def test_paged_multi_sequence_holes_and_range():
    wl = workloads.small("sweep")
    g, c = build_both(wl)
    rng = np.random.default_rng(3)
    T, H, W, page, n_seq, max_pages = 5, 16, 96, 16, 3, 40
    n_pages = wl.num_slots // page
    bt = rng.integers(1, n_pages, size=(n_seq, max_pages)).astype(np.int32)
    bt[rng.random(bt.shape) < 0.1] = -1                    # unassigned pages
    pos = rng.integers(-1, max_pages * page + 40, size=(T, W)).astype(np.int32)   # some past the table
    seq = rng.integers(0, n_seq, size=T).astype(np.int32)
    q = torch.from_numpy(rng.standard_normal((T, H, 576)).astype(np.float32)).to(torch.bfloat16)
    d = dev()
    out, lse = M.mla_sparse_decode_paged(q.to(d), g, torch.from_numpy(pos).to(d), torch.from_numpy(bt).to(d),
                                         page, 0.05, token_seq=torch.from_numpy(seq).to(d))
    torch.cuda.synchronize()
    err = M.mla_get_error()
    phys, bad = oracle.paged_to_physical(pos, bt, page, seq)
    assert bad > 0 and err == M.MLA_ERR_DECODE_INDEX_RANGE
    ro, rl, _ = oracle.sparse_decode(q, c, phys, 0.05)
    check_decode(out, lse, ro, rl)


# ------------------------------------------------------------ gather-and-upconvert
def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("pe_dim", [64, 0])
def test_upconvert_matches_oracle(pe_dim):
    wl = workloads.small("sweep")
    g, c = build_both(wl)
    rng = np.random.default_rng(4)
    slots = rng.integers(-2, wl.num_slots + 3, size=3001).astype(np.int32)   # absent and out-of-range too
    out = M.mla_gather_upconvert(g, torch.from_numpy(slots).to(dev()), pe_dim)
    torch.cuda.synchronize()
    err = M.mla_get_error()
    ref, bad = oracle.gather_upconvert(c, slots, pe_dim)
    assert (err == M.MLA_ERR_GATHER_INDEX_RANGE) == (bad > 0)
    np.testing.assert_array_equal(_bits(out), ref)


def test_upconvert_rounding_cases():
    """Rows whose products sit on or near BF16 midpoints, tiny and huge scales,
    subnormal results, NaN and signed-zero codes."""
    rng = np.random.default_rng(5)
    rows = []
    for m in range(9, 16):
        found = 0
        for S in range(1 << 23, (1 << 23) + (1 << 21)):
            P = S * m
            L = P.bit_length()
            f32 = P >> (L - 24)
            if (P & ((1 << (L - 24)) - 1)) and ((f32 & 0xFFFF) in (0x8000, 0x7FFF)):
                codes = np.full(512, 0x38 | (m - 8), np.uint8)
                codes[1::2] = rng.integers(0, 256, size=256)
                rows.append((codes, [S * 2.0 ** -23, 1.0, S * 2.0 ** -30, S * 2.0 ** -10]))
                found += 1
                if found >= 4:
                    break
    for sc in ([2.0 ** -120, 2.0 ** -133, 1e-38, 3e-39], [2.0 ** 100, 1e30, 7.5e5, 0.3],
               [2.0 ** -126 * 1.7, 2.0 ** -110, 2.0 ** -101, 2.0 ** -99]):
        codes = np.arange(512, dtype=np.int64).astype(np.uint8)
        rows.append((codes, sc))
    cache = np.zeros((len(rows) + 1, 656), np.uint8)
    for i, (codes, sc) in enumerate(rows):
        cache[i + 1, :512] = codes
        cache[i + 1, 512:528] = np.asarray(sc, dtype="<f4").view(np.uint8)
        cache[i + 1, 528:] = rng.integers(0, 256, size=128)
    slots = np.arange(1, len(rows) + 1, dtype=np.int32)
    g = torch.from_numpy(cache).to(dev())
    out = M.mla_gather_upconvert(g, torch.from_numpy(slots).to(dev()), 64)
    torch.cuda.synchronize()
    ref, _ = oracle.gather_upconvert(cache, slots, 64)
    np.testing.assert_array_equal(_bits(out), ref)
    assert M.mla_get_error() == 0


def test_upconvert_528_rows():
    wl = workloads.small("nope")
    g528, c528 = _nope528(wl)
    slots = np.random.default_rng(6).integers(0, wl.num_slots, size=777).astype(np.int32)
    out = M.mla_gather_upconvert(g528, torch.from_numpy(slots).to(dev()), 0)
    torch.cuda.synchronize()
    ref, _ = oracle.gather_upconvert(c528, slots, 0)
    np.testing.assert_array_equal(_bits(out), ref)
    assert M.mla_get_error() == 0


def test_upconvert_full_size():
    """The bench's gather: 262,144 random slots of the 1M-slot RoPE cache."""
    wl = workloads.sweep()
    g, c = build_both(wl)
    slots = np.random.default_rng(7).integers(1, wl.num_slots, size=262144).astype(np.int32)
    out = M.mla_gather_upconvert(g, torch.from_numpy(slots).to(dev()), 64)
    torch.cuda.synchronize()
    ref, bad = oracle.gather_upconvert(c, slots, 64)
    assert bad == 0
    np.testing.assert_array_equal(_bits(out), ref)
    assert M.mla_get_error() == 0


@pytest.mark.parametrize("page", [16, 4])
def test_paged_with_head_groups_and_splits_equals_physical(page):
    """H = 64 (four head groups) and T = 3 (the list is split): an identity block
    table gives exactly the physical-slot decode, with 16-slot pages (a 1,024-page
    table) and 4-slot pages (4,096)."""
    wl = workloads.small("rope")
    g, _ = build_both(wl)
    db = wl.decode
    d = dev()
    bt = torch.arange(wl.num_slots // page, dtype=torch.int32, device=d)
    ref_out, ref_lse = gpu_decode(g, db)
    out, lse = M.mla_sparse_decode_paged(db.q.to(d), g, db.topk.to(d), bt, page, db.sm_scale)
    torch.cuda.synchronize()
    assert M.mla_sparse_decode_workspace_bytes(db.T, db.H, db.W) > 0
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)) and torch.equal(lse, ref_lse)
    assert M.mla_get_error() == 0


@pytest.mark.parametrize("n", [0, 1, 31, 33, 95])
def test_upconvert_partial_blocks(n):
    wl = workloads.small("sweep")
    g, c = build_both(wl)
    slots = np.random.default_rng(n).integers(-1, wl.num_slots, size=n).astype(np.int32)
    out = M.mla_gather_upconvert(g, torch.from_numpy(slots).to(dev()), 64)
    torch.cuda.synchronize()
    ref, _ = oracle.gather_upconvert(c, slots, 64)
    np.testing.assert_array_equal(_bits(out).reshape(n, 576), ref)
    assert M.mla_get_error() == 0
