"""Pins for the oracle writer: the packed 656-byte row (vLLM PR #55277, Purpose
item 1), the reserved-slot drop (sglang PR #47013, Summary / Motivation) and the
per-tile FP8 quantisation, checked through invariants and through torch's fp8 cast."""
import os

import numpy as np
import pytest
import torch

import oracle
from fp8_mla_kv_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SENTINEL = 0xA5


def _layout():
    out = {}
    with open(os.path.join(GOLDEN, "row_layout.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                name, off, n = line.split()
                out[name] = (None if off == "-" else int(off), int(n))
    return out


def _bf16_bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _f32(t):
    return t.float().numpy()


def _scales(row):
    return row[512:528].copy().view("<f4")


def test_layout_constants_match_pages():
    L = _layout()
    assert L["latent_fp8"] == (0, 512)
    assert L["tile_scales_f32"] == (512, 16)
    assert L["rope_or_zero"] == (528, 128)
    assert L["row_total"] == (0, 656) == (0, oracle.ROW_BYTES)
    assert L["tile_values"][1] * L["num_tiles"][1] == 512
    assert L["rope_values_bf16"][1] * 2 == L["rope_or_zero"][1]


def _write_case(rope=True, seed=3):
    n, S = 40, 64
    g = torch.Generator().manual_seed(seed)
    lat = torch.randn((n, 512), generator=g).to(torch.bfloat16)
    rp = torch.randn((n, 64), generator=g).to(torch.bfloat16) if rope else None
    slots = torch.randperm(S - 1, generator=g)[:n] + 1
    slots[5] = 0           # reserved slot, NaN latent
    lat[5] = float("nan")
    slots[9] = -3          # negative slot: dropped too
    slots[11] = S + 7      # out of range: dropped and counted
    lat[12, 128:256] = 0.0         # an all-zero tile
    lat[13, 0:128] = -0.0          # an all-negative-zero tile
    cache = np.full((S, 656), SENTINEL, np.uint8)
    bad = oracle.kv_write(cache, slots.numpy(), lat, rp, reserved_slot=0)
    return cache, slots, lat, rp, bad


@pytest.mark.parametrize("rope", [True, False])
def test_untouched_bytes_and_reserved_slot(rope):
    cache, slots, lat, rp, bad = _write_case(rope)
    assert bad == 1
    written = {int(s) for s in slots if 0 < int(s) < cache.shape[0]}
    for s in range(cache.shape[0]):
        if s not in written:
            assert np.all(cache[s] == SENTINEL), s   # includes slot 0
    assert 0 not in written


@pytest.mark.parametrize("rope", [True, False])
def test_tail(rope):
    cache, slots, lat, rp, _ = _write_case(rope)
    for r, s in enumerate(slots.tolist()):
        if not 0 < s < cache.shape[0]:
            continue
        tail = cache[s, 528:656]
        if rope:
            assert np.array_equal(tail.view("<u2"), _bf16_bits(rp[r]))
        else:
            assert np.all(tail == 0)


def test_scale_amax_byte_and_dequant_bound():
    cache, slots, lat, rp, _ = _write_case(True)
    table = oracle.e4m3_decode_table()
    for r, s in enumerate(slots.tolist()):
        if not 0 < s < cache.shape[0]:
            continue
        row = cache[s]
        x = _f32(lat[r])
        sc = _scales(row)
        for t in range(4):
            xt = x[128 * t:128 * (t + 1)]
            bt = row[128 * t:128 * (t + 1)]
            amax = np.float32(np.max(np.abs(xt)))
            if amax == 0:
                assert sc[t] == 1.0
                assert np.all((bt & 0x7F) == 0)
                assert np.array_equal(bt >> 7, np.signbit(xt).astype(np.uint8))
                continue
            # scale = amax / 448 to within one fp32 rounding
            assert abs(float(sc[t]) * 448.0 - float(amax)) <= float(np.spacing(amax))
            i = int(np.argmax(np.abs(xt)))
            assert bt[i] == (0xFE if xt[i] < 0 else 0x7E)
            deq = table[bt] * float(sc[t])
            bound = 2.0 ** -4 * np.abs(xt) + 2.0 ** -10 * float(sc[t]) + 1e-6 * np.abs(xt)
            assert np.all(np.abs(deq - xt) <= bound)


def test_bytes_reduce_to_torch_cast():
    # One tile's bytes are torch's fp8 cast of x / scale (fp32 IEEE division),
    # saturated to +-448: an independent encoder for the whole row.
    cache, slots, lat, rp, _ = _write_case(True)
    for r, s in enumerate(slots.tolist()):
        if not 0 < s < cache.shape[0]:
            continue
        row = cache[s]
        sc = torch.from_numpy(_scales(row).copy())
        x = lat[r].float().view(4, 128)
        v = (x / sc[:, None]).clamp(-448, 448)
        ref = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy().ravel()
        assert np.array_equal(ref, row[:512])


def test_slot0_kept_whatever_it_holds():
    wl = workloads.tiny()
    wb = wl.writes[0]
    for fill in (0x00, 0xFF):
        cache = np.full((wl.num_slots, 656), fill, np.uint8)
        oracle.kv_write(cache, wb.slot_idx.numpy(), wb.latent, wb.rope)
        assert np.all(cache[0] == fill)
        assert int((wb.slot_idx == 0).sum()) == 32


def test_amax_ignores_quiet_and_signaling_nans():
    # "per-token FP8 quantization keeps BF16 NaNs" (sglang PR #47013, Motivation):
    # NaN elements encode as NaN and do not enter the tile amax, whether the bf16
    # NaN widens to a quiet (0x7FC1) or a signaling (0x7F97) fp32 NaN.
    bits = np.zeros((1, 512), np.uint16)
    bits[0, 0] = 0x43E0                       # 448.0
    bits[0, 1:40] = 0x7F97                    # signaling after widening
    bits[0, 40:60] = 0xFFC1                   # quiet, negative
    bits[0, 60:70] = 0x0015                   # bf16 subnormal
    bits[0, 128] = 0x7F81
    bits[0, 129] = 0x3F80                     # 1.0
    lat = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    cache = np.zeros((2, 656), np.uint8)
    oracle.kv_write(cache, np.array([1]), lat, None)
    sc = _scales(cache[1])
    assert sc[0] == 1.0 and sc[1] == np.float32(1.0) / np.float32(448.0)
    assert np.all(cache[1, 1:60] == 0x7F) and cache[1, 128] == 0x7F
    assert cache[1, 0] == 0x7E and cache[1, 129] == 0x7E
