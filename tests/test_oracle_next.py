"""Pins of the oracle's widened functions: 528-byte NoPE rows, top-k positions
through a block table, and gather-and-upconvert to BF16.

Each check compares the oracle with something other than itself: the 656-byte
row it already pins, the prefill generator's own position -> slot mapping,
torch's float8 -> bfloat16 conversion, and an integer nearest-even rounding.
"""
import os
import sys

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402
from fp8_mla_kv_gb300 import workloads  # noqa: E402


def _bf16(x):
    return x.to(torch.bfloat16)


# ---------------------------------------------------------------- 528-byte rows
def _nope_rows(n, seed):
    g = torch.Generator().manual_seed(seed)
    return _bf16(torch.randn(n, 512, generator=g))


def test_528_rows_are_the_656_rows_without_tail():
    n, S = 40, 97
    lat = _nope_rows(n, 1)
    slots = np.random.default_rng(2).choice(np.arange(1, S), size=n, replace=False)
    c656 = np.full((S, 656), 0xA5, np.uint8)
    c528 = np.full((S, 528), 0xA5, np.uint8)
    assert oracle.kv_write(c656, slots, lat, None) == 0
    assert oracle.kv_write(c528, slots, lat, None) == 0
    np.testing.assert_array_equal(c528, c656[:, :528])
    untouched = np.setdiff1d(np.arange(S), slots)
    assert (c528[untouched] == 0xA5).all()


def test_528_rows_refuse_rope():
    c528 = np.zeros((8, 528), np.uint8)
    with pytest.raises(AssertionError):
        oracle.kv_write(c528, [1], _nope_rows(1, 0), _nope_rows(1, 1)[:, :64])


def test_decode_over_528_rows_equals_656_nope():
    n, S, T, H, W = 60, 128, 3, 16, 48
    lat = _nope_rows(n, 3)
    slots = np.arange(1, n + 1)
    c656 = np.zeros((S, 656), np.uint8)
    c528 = np.zeros((S, 528), np.uint8)
    oracle.kv_write(c656, slots, lat, None)
    oracle.kv_write(c528, slots, lat, None)
    g = torch.Generator().manual_seed(4)
    q = _bf16(torch.randn(T, H, 512, generator=g))
    topk = torch.randint(-1, n + 1, (T, W), generator=g, dtype=torch.int32).numpy()
    a = oracle.sparse_decode(q, c656, topk, 0.05)
    b = oracle.sparse_decode(q, c528, topk, 0.05)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ---------------------------------------------------------------- paged top-k
def test_paged_matches_the_prefill_generator():
    wl = workloads.small("prefill")
    phys, bad = oracle.paged_to_physical(wl.topk_logical.numpy(), wl.block_table.numpy(), wl.page_size)
    assert bad == 0
    np.testing.assert_array_equal(phys, wl.decode.topk.numpy())


def test_paged_identity_table():
    g = np.random.default_rng(5)
    lg = g.integers(-1, 256, size=(4, 33)).astype(np.int32)
    phys, bad = oracle.paged_to_physical(lg, np.arange(16, dtype=np.int32), 16)
    assert bad == 0
    np.testing.assert_array_equal(phys, np.where(lg < 0, -1, lg))


def test_paged_hand_cases():
    # two sequences, page size 4: seq 0 pages -> [7, 2, -1], seq 1 pages -> [5]
    bt = np.array([[7, 2, -1], [5, -1, -1]], dtype=np.int32)
    lg = np.array([[0, 3, 4, 6, 9, -1, 12],
                   [1, 4, -5, 3, 0, 11, 2]], dtype=np.int32)
    seq = np.array([0, 1], dtype=np.int32)
    phys, bad = oracle.paged_to_physical(lg, bt, 4, seq)
    expect = np.array([[28, 31, 8, 10, -1, -1, -1],    # 9 -> page 2 unassigned; 12 -> past the table
                       [21, -1, -1, 23, 20, -1, 22]], dtype=np.int32)   # 4, 11 -> unassigned pages
    np.testing.assert_array_equal(phys, expect)
    assert bad == 1


# ---------------------------------------------------------------- upconvert
def _row_with(codes, scales, rope_bits=None):
    """One 656-byte row holding 512 given codes, four fp32 scales and a tail."""
    row = np.zeros(656, np.uint8)
    row[:512] = codes
    row[512:528] = np.asarray(scales, dtype="<f4").view(np.uint8)
    if rope_bits is not None:
        row[528:] = np.asarray(rope_bits, dtype="<u2").view(np.uint8)
    return row


def test_upconvert_power_of_two_scales_match_torch():
    codes = np.concatenate([np.arange(256), np.arange(256)]).astype(np.uint8)
    for scales in ([1.0, 2.0 ** -20, 2.0 ** 5, 0.5], [2.0 ** -100, 2.0 ** 60, 1.0, 2.0 ** -3]):
        cache = np.zeros((3, 656), np.uint8)
        cache[1] = _row_with(codes, scales)
        out, bad = oracle.gather_upconvert(cache, np.array([1], np.int32), 0)
        assert bad == 0
        vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32)
        sc = torch.tensor(np.repeat(np.asarray(scales, np.float32), 128))
        ref = (vals * sc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        nan = np.isnan(vals.numpy())
        np.testing.assert_array_equal(out[0, :512][~nan], ref[~nan])
        assert (out[0, :512][nan] == 0x7FC0).all()
        assert (out[0, 512:] == 0).all()


def _nearest_bf16_int(P: int, exp2: int) -> float:
    """Value nearest to P * 2^exp2 (P > 0) with an 8-bit significand, ties to even,
    by integer arithmetic (normal range only)."""
    L = P.bit_length()
    if L <= 8:
        return float(P) * 2.0 ** exp2
    sh = L - 8
    q, rem, half = P >> sh, P & ((1 << sh) - 1), 1 << (sh - 1)
    if rem > half or (rem == half and (q & 1)):
        q += 1
    return float(q) * 2.0 ** (exp2 + sh)


def test_upconvert_single_rounding_against_integer_reference():
    rng = np.random.default_rng(6)
    cases = []
    # Random 24-bit scale significands, and ones built so that rounding the product
    # first to fp32 lands exactly on a BF16 midpoint (double rounding would differ).
    for m in range(9, 16):                      # codes 0x39..0x3F: values m/8
        for S in rng.integers(1 << 23, 1 << 24, size=200):
            cases.append((m, int(S)))
        found = 0
        for S in range(1 << 23, (1 << 23) + (1 << 21)):
            P = S * m                           # exact product significand (27-28 bits)
            L = P.bit_length()
            f32 = P >> (L - 24)
            r = P & ((1 << (L - 24)) - 1)
            if r == 0:
                continue
            # the fp32 result (before its own rounding) equals a BF16 midpoint pattern
            if (f32 & 0xFFFF) == 0x8000 or (f32 & 0xFFFF) == 0x7FFF:
                cases.append((m, S))
                found += 1
                if found >= 6:
                    break
        assert found > 0
    codes = np.zeros(512, np.uint8)
    scales = []
    exp_vals = []
    for k, (m, S) in enumerate(cases):
        code = 0x38 | (m - 8)                   # exponent field 7 -> value m/8
        scale = float(np.float32(S * 2.0 ** -23))
        assert scale == S * 2.0 ** -23
        scales.append((code, scale, _nearest_bf16_int(S * m, -23 - 3)))
    # one row per (code, scale): value 0 of tile 0 carries the case
    cache = np.zeros((len(scales) + 1, 656), np.uint8)
    for i, (code, scale, _) in enumerate(scales):
        row_codes = np.zeros(512, np.uint8)
        row_codes[0] = code
        cache[i + 1] = _row_with(row_codes, [scale, 1.0, 1.0, 1.0])
    out, bad = oracle.gather_upconvert(cache, np.arange(1, len(scales) + 1, dtype=np.int32), 0)
    assert bad == 0
    got = out[:, 0].astype(np.uint32) << 16
    got_f = got.view(np.float32).astype(np.float64)
    want = np.array([e for _, _, e in scales])
    np.testing.assert_array_equal(got_f, want)


def test_upconvert_tail_absent_rows_and_528_rows():
    rng = np.random.default_rng(7)
    cache = np.zeros((6, 656), np.uint8)
    rope = rng.integers(0, 1 << 16, size=64).astype(np.uint16)
    codes = rng.integers(0, 256, size=512).astype(np.uint8)
    codes[codes & 0x7F == 0x7F] = 0x10           # no NaN codes here
    cache[3] = _row_with(codes, [0.25, 3.0, 1e-3, 7.5], rope)
    out, bad = oracle.gather_upconvert(cache, np.array([3, 0, -1, 9, 3], np.int32), 64)
    assert bad == 1                              # slot 9 >= num_slots
    np.testing.assert_array_equal(out[0, 512:], rope)
    assert (out[1:4] == 0).all()
    np.testing.assert_array_equal(out[4], out[0])
    out0, _ = oracle.gather_upconvert(cache, np.array([3], np.int32), 0)
    np.testing.assert_array_equal(out0[0, :512], out[0, :512])
    assert (out0[0, 512:] == 0).all()
    c528 = np.ascontiguousarray(cache[:, :528])
    out528, _ = oracle.gather_upconvert(c528, np.array([3], np.int32), 0)
    np.testing.assert_array_equal(out528, out0)
