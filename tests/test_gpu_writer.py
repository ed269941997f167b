"""GPU writer parity: bit-exact against the oracle on every byte of the cache
(FP8 codes, fp32 scales, RoPE / zero tail, untouched slots, reserved slot 0)."""
import numpy as np
import pytest
import torch

import oracle
from fp8_mla_kv_gb300 import mlasparse as M
from fp8_mla_kv_gb300 import workloads

from _parity import build_both, cpu_cache, cpu_write, dev, gpu_cache, gpu_write

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "nope", "rope", "prefill", "sweep"])
def test_small_configs_bit_exact(name):
    wl = workloads.small(name)
    g, c = build_both(wl)
    assert M.mla_get_error() == 0
    assert np.array_equal(g.cpu().numpy(), c)


@pytest.mark.parametrize("slot0", [0x00, 0xFF, 0xA5])
def test_reserved_slot_and_sentinel(slot0):
    wl = workloads.tiny()
    g, c = build_both(wl, slot0_byte=slot0)
    gc = g.cpu().numpy()
    assert np.all(gc[0] == slot0)
    assert np.array_equal(gc, c)


def test_every_bf16_value_with_unit_scale():
    # Tiles whose amax is exactly 448 have scale 1.0, so each byte is the E4M3
    # code of the bf16 value itself: this covers every bf16 pattern with |x| <= 448
    # (and the NaNs, which amax ignores).
    pats = np.arange(1 << 16, dtype=np.uint32)
    vals = (pats << 16).view(np.float32)
    keep = np.isnan(vals) | (np.abs(vals) <= 448.0)
    pats = pats[keep].astype(np.uint16)
    per_tile = 127
    n_tiles = (pats.size + per_tile - 1) // per_tile
    pats = np.concatenate([pats, np.zeros(n_tiles * per_tile - pats.size, np.uint16)])
    tiles = pats.reshape(n_tiles, per_tile)
    anchor = np.full((n_tiles, 1), 0x43E0, np.uint16)          # bf16 448.0
    tiles = np.concatenate([anchor, tiles], axis=1)             # [n_tiles, 128]
    n_rows = (n_tiles + 3) // 4
    tiles = np.concatenate([tiles, np.tile(tiles[:1], (n_rows * 4 - n_tiles, 1))])
    lat = torch.from_numpy(tiles.reshape(n_rows, 512).view(np.int16)).view(torch.bfloat16)
    slots = torch.arange(1, n_rows + 1, dtype=torch.int64)
    wb = workloads.WriteBatch(slots, lat, None)
    wl = workloads.Workload("bf16", n_rows + 1, 0, None, [wb], None)
    g, c = build_both(wl)
    gc = g.cpu().numpy()
    assert np.array_equal(gc, c)
    assert np.all(gc[1:, 512:528].view("<f4") == 1.0)


def test_out_of_range_slot_sets_error_and_is_dropped():
    wl = workloads.tiny()
    wb = wl.writes[0]
    slots = wb.slot_idx.clone()
    slots[3] = wl.num_slots + 11
    bad = workloads.WriteBatch(slots, wb.latent, wb.rope)
    M.mla_get_error()
    g, c = gpu_cache(wl), cpu_cache(wl)
    gpu_write(g, bad)
    cpu_write(c, bad)
    torch.cuda.synchronize()
    assert M.mla_get_error() == M.MLA_ERR_WRITE_SLOT_RANGE
    assert M.mla_get_error() == 0
    assert np.array_equal(g.cpu().numpy(), c)


def test_empty_and_invalid_calls():
    wl = workloads.tiny()
    g = gpu_cache(wl)
    d = dev()
    e = torch.empty(0, dtype=torch.int64, device=d)
    M.mla_kv_write(g, e, torch.empty((0, 512), dtype=torch.bfloat16, device=d), None)
    with pytest.raises(M.MlaError):
        # misaligned latent pointer
        lat = torch.empty(512 * 2 + 8, dtype=torch.bfloat16, device=d)[4:4 + 512 * 2].view(2, 512)
        M.mla_kv_write(g, torch.ones(2, dtype=torch.int64, device=d), lat, None)
    torch.cuda.synchronize()
    assert torch.all(g == 0)


@pytest.mark.parametrize("n_rows", [2432, 2433, 2440, 5001, 40000])
def test_batches_around_two_rows_per_warp(n_rows):
    # Large batches run two rows per warp (both rows' loads in flight together) and,
    # past four CTAs per SM, stride over the batch. Batch sizes on both sides of the
    # switch and with a ragged last group, a quarter of the rows aimed at the
    # reserved slot, a few out of range (dropped and flagged), RoPE and NoPE rows:
    # every byte of the cache as the oracle writes it.
    gen = torch.Generator().manual_seed(n_rows)
    num_slots = 2 * n_rows + 16
    slots = (torch.randperm(num_slots - 1, generator=gen)[:n_rows] + 1).to(torch.int64)
    slots[torch.randperm(n_rows, generator=gen)[: n_rows // 4]] = 0
    slots[torch.randperm(n_rows, generator=gen)[:3]] = num_slots + 5
    lat = (torch.randn((n_rows, 512), generator=gen) * 3.0).to(torch.bfloat16)
    rope = torch.randn((n_rows, 64), generator=gen).to(torch.bfloat16)
    for rp in (rope, None):
        wb = workloads.WriteBatch(slots, lat, rp)
        wl = workloads.Workload("writer-batch", num_slots, 0, None, [wb], None)
        M.mla_get_error()
        g, c = gpu_cache(wl), cpu_cache(wl)
        gpu_write(g, wb)
        cpu_write(c, wb)
        torch.cuda.synchronize()
        assert M.mla_get_error() == M.MLA_ERR_WRITE_SLOT_RANGE
        assert np.array_equal(g.cpu().numpy(), c)
