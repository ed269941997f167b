"""Pins for the oracle's E4M3 codec (OCP OFP8 E4M3, round-to-nearest-even,
saturating). Pinned against torch's float8_e4m3fn (an independent library
implementation) and against closed-form points of the specification."""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_table():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_all_codes_match_torch():
    ours = oracle.e4m3_decode_table()
    ref = _torch_table()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2                       # 0x7F and 0xFF only
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def _golden_points():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_points.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            x, b = line.split()
            rows.append((float(eval(x)), int(b, 16)))
    return rows


@pytest.mark.parametrize("x,b", _golden_points())
def test_encode_golden_points(x, b):
    assert int(oracle.e4m3_encode(np.array([x], np.float32))[0]) == b


def test_encode_nan_reading():
    # Reading: NaN encodes as 0x7F whatever its sign (pinned on the GPU as well).
    x = np.array([0x7FC00000, 0xFFC00001], np.uint32).view(np.float32)  # +NaN, -NaN
    assert list(oracle.e4m3_encode(x)) == [0x7F, 0x7F]


def _structured_patterns():
    """fp32 bit patterns covering every exponent, every combination of the top 6
    mantissa bits and several low-bit (sticky) patterns, both signs, plus a
    uniform random sample."""
    exps = np.arange(0, 255, dtype=np.uint32)
    top = np.arange(64, dtype=np.uint32) << 17
    low = np.array([0, 1, 0x8000, 0xFFFF, 0x10000, 0x1FFFF, 0x0F0F0], dtype=np.uint32)
    m = (top[:, None] | low[None, :]).ravel()
    bits = (exps[:, None] << 23 | m[None, :]).ravel()
    bits = np.concatenate([bits, bits | np.uint32(0x80000000)])
    rng = np.random.default_rng(1234)
    rnd = rng.integers(0, 2**32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    bits = np.concatenate([bits, rnd])
    x = bits.view(np.float32)
    return x[~np.isnan(x)]


def test_encode_matches_torch_cast_with_saturation():
    x = _structured_patterns()
    ours = oracle.e4m3_encode(x)
    clamped = torch.from_numpy(x).clamp(-448.0, 448.0)
    ref = clamped.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(x[i]), hex(ours[i]), hex(ref[i])) for i in bad[:10]]


def test_encode_is_nearest_and_monotone():
    # Invariants that need no library: decode(encode(x)) is a nearest grid point
    # (within half a spacing) and the map is monotone.
    x = np.sort(_structured_patterns())
    x = x[np.abs(x) <= 448.0]
    table = oracle.e4m3_decode_table()
    v = table[oracle.e4m3_encode(x)]
    assert np.all(np.diff(v) >= 0)
    ax = np.abs(x.astype(np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -149)))
    spacing = np.where(ax < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))
    assert np.all(np.abs(v - x) <= spacing / 2)
