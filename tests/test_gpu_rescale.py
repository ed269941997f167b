"""GPU decode against the float64 oracle on lists built to drive the decode's
rescaling paths, which random N(0,1) inputs reach almost only on the first rows:

* rising scores: each row's score runs well above every earlier one, so the
  running softmax offset (and the O / l rescale that goes with it) moves on
  nearly every block of the list;
* rising tile scales: the rows' magnitudes, hence their fp32 tile scales, grow
  along the list, so the running maximum of the scales that normalises the PV
  operand moves repeatedly as well;
* mixed magnitudes: tile scales spread over many octaves inside one list and
  inside one row.

Each case runs through the decode and through the token-pair prefill kernel,
and is checked with the decode tolerance of the other parity tests
(max|out-ref| <= 1e-2 max|ref| + 1e-3, |lse-ref| <= 1e-3). The same check per
(token, head) row against that row's own max|ref| is printed as a diagnostic, and
asserted (within 2e-2) where the row scales span at most 2^12: the PV operand is
p * scale / sigma in f16 (sigma = the running maximum of the tile's scales), whose
normal range holds such ratios with full precision. In the 2^-30 case the rows
whose ratio falls below f16's range add nothing to O, which the per-row figure
shows.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_mla_kv_gb300 import mlasparse as M

from _parity import check_decode, dev

pytestmark = pytest.mark.gpu

NUM_SLOTS = 8192


def _write_rows(latent_f32, rope_f32):
    """A cache whose slots 1..n hold the given rows (GPU and oracle writers)."""
    n = latent_f32.shape[0]
    lat = latent_f32.to(torch.bfloat16)
    rope = None if rope_f32 is None else rope_f32.to(torch.bfloat16)
    slots = torch.arange(1, n + 1, dtype=torch.int64)
    g = torch.zeros((NUM_SLOTS, 656), dtype=torch.uint8, device=dev())
    M.mla_kv_write(g, slots.to(dev()), lat.to(dev()), None if rope is None else rope.to(dev()))
    c = np.zeros((NUM_SLOTS, 656), np.uint8)
    oracle.kv_write(c, slots.numpy(), lat, rope)
    torch.cuda.synchronize()
    assert np.array_equal(g.cpu().numpy(), c), "writer parity is a precondition here"
    return g, c


ENTRIES = {"decode": M.mla_sparse_decode, "prefill": M.mla_sparse_prefill}


def _run(g, c, q, topk, sm_scale, per_row_rtol=None, label="", entry="decode"):
    out, lse = ENTRIES[entry](q.to(dev()), g, topk.to(dev()), sm_scale)
    torch.cuda.synchronize()
    ro, rl, bad = oracle.sparse_decode(q, c, topk.numpy(), sm_scale)
    assert bad == 0
    check_decode(out, lse, ro, rl)
    o = out.float().cpu().numpy().astype(np.float64)
    row_max = np.abs(ro).max(axis=2)
    row_err = np.abs(o - ro).max(axis=2)
    rel = row_err / np.maximum(row_max, 1e-300)
    print(f"[{label}] worst per-(token, head) error / own max|ref|: {rel.max():.3e}; "
          f"max|lse-ref| {np.abs(lse.cpu().numpy() - rl).max():.3e}")
    if per_row_rtol is not None:
        assert (row_err <= per_row_rtol * row_max + 1e-6 * row_max.max()).all(), \
            f"per-row error {rel.max():.3e} above {per_row_rtol}"
    assert M.mla_get_error() == 0


def _topk(T, W, n, perm_seed=None):
    idx = torch.arange(1, n + 1, dtype=torch.int32)
    rows = []
    for t in range(T):
        r = idx.clone()
        if perm_seed is not None:
            r = r[torch.randperm(n, generator=torch.Generator().manual_seed(perm_seed + t))]
        full = torch.full((W,), -1, dtype=torch.int32)
        full[:n] = r
        rows.append(full)
    return torch.stack(rows)


@pytest.mark.parametrize("entry", ["decode", "prefill"])
@pytest.mark.parametrize("d_qk", [576, 512])
def test_rising_scores_and_scales_move_every_block(d_qk, entry):
    # Row j = a_j * v + small noise with a_j rising: its score against q = beta_h v
    # rises by about 20 log2 units per 32 rows (heads with beta_h > 0), its tile
    # scales rise with it. Heads with beta_h < 0 see falling scores instead.
    gen = torch.Generator().manual_seed(11)
    n, T, H = 1000, 3, 16
    v = torch.randn(512, generator=gen)
    a = 0.02 * torch.arange(1, n + 1, dtype=torch.float32)
    lat = a[:, None] * v[None, :] + 0.1 * torch.randn((n, 512), generator=gen)
    rope = torch.randn((n, 64), generator=gen) if d_qk == 576 else None
    g, c = _write_rows(lat, rope)
    beta = torch.tensor([1.0, -1.0, 0.5, -0.25, 2.0, 0.0, 0.75, -2.0] * 2)
    q = torch.empty((T, H, d_qk))
    q[:, :, :512] = beta[None, :, None] * v[None, None, :]
    if d_qk == 576:
        q[:, :, 512:] = torch.randn((T, H, 64), generator=gen)
    q = q.to(torch.bfloat16)
    topk = _topk(T, 1024, n)
    topk[1, :n] = torch.flip(topk[1, :n], [0])                              # falling order
    topk[2, :n] = topk[2, :n][torch.randperm(n, generator=gen)]              # random order
    _run(g, c, q, topk, 1.0 / d_qk ** 0.5, per_row_rtol=2e-2, label=f"rising d_qk={d_qk} {entry}", entry=entry)


@pytest.mark.parametrize("entry", ["decode", "prefill"])
def test_scales_growing_along_the_list(entry):
    # Row magnitudes grow geometrically (2^-11 .. 1) along the list with random
    # directions: sigma, the running maximum of the tile scales, is raised over
    # and over while the scores stay moderate.
    gen = torch.Generator().manual_seed(12)
    n, T, H = 768, 2, 16
    mag = torch.exp2(torch.linspace(-11.0, 0.0, n))
    lat = mag[:, None] * torch.randn((n, 512), generator=gen)
    rope = torch.randn((n, 64), generator=gen)
    g, c = _write_rows(lat, rope)
    q = (4.0 * torch.randn((T, H, 576), generator=gen)).to(torch.bfloat16)
    topk = _topk(T, 768, n)
    _run(g, c, q, topk, 1.0 / 24.0, per_row_rtol=2e-2, label=f"growing scales {entry}", entry=entry)


@pytest.mark.parametrize("entry", ["decode", "prefill"])
def test_tile_scales_spanning_many_octaves(entry):
    # Each tile of each row gets its own magnitude 2^-e, e uniform in 0..30, so a
    # list mixes tile scales from about 2^-39 to 2^-8 (scale = amax / 448).
    gen = torch.Generator().manual_seed(13)
    n, T, H = 1024, 4, 16
    e = torch.randint(0, 31, (n, 4), generator=gen).float()
    lat = torch.randn((n, 512), generator=gen) * torch.exp2(-e).repeat_interleave(128, dim=1)
    rope = 1e-3 * torch.randn((n, 64), generator=gen)
    g, c = _write_rows(lat, rope)
    q = (8.0 * torch.randn((T, H, 576), generator=gen)).to(torch.bfloat16)
    topk = _topk(T, 1024, n, perm_seed=5)
    _run(g, c, q, topk, 1.0 / 24.0, label=f"2^-30..1 tile magnitudes {entry}", entry=entry)


@pytest.mark.parametrize("entry", ["decode", "prefill"])
def test_tile_scales_spanning_twelve_octaves_per_row_check(entry):
    gen = torch.Generator().manual_seed(14)
    n, T, H = 900, 3, 16
    e = torch.randint(0, 13, (n, 4), generator=gen).float()
    lat = torch.randn((n, 512), generator=gen) * torch.exp2(-e).repeat_interleave(128, dim=1)
    rope = torch.randn((n, 64), generator=gen)
    g, c = _write_rows(lat, rope)
    q = (2.0 * torch.randn((T, H, 576), generator=gen)).to(torch.bfloat16)
    topk = _topk(T, 1024, n, perm_seed=9)
    _run(g, c, q, topk, 1.0 / 24.0, per_row_rtol=2e-2, label=f"2^-12..1 tile magnitudes {entry}", entry=entry)
