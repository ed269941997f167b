"""GPU sparse-decode parity against the float64 oracle on reduced versions of
the five workloads (several 32-row blocks, ragged tails, splits), plus the
masking properties the pages fix: -1 / slot-0 entries contribute nothing and
load nothing, so the output is bit-identical whatever slot 0 holds."""
import math

import numpy as np
import pytest
import torch

import oracle
from fp8_mla_kv_gb300 import mlasparse as M
from fp8_mla_kv_gb300 import workloads

from _parity import build_both, check_decode, dev, gpu_decode

pytestmark = pytest.mark.gpu


def _ref(c, db, topk=None, q=None):
    q = db.q if q is None else q
    topk = db.topk.numpy() if topk is None else topk
    out, lse, _ = oracle.sparse_decode(q, c, topk, db.sm_scale)
    return out, lse


@pytest.mark.parametrize("name", ["tiny", "nope", "rope", "prefill", "sweep"])
def test_small_configs_match_oracle(name):
    wl = workloads.small(name)
    g, c = build_both(wl)
    out, lse = gpu_decode(g, wl.decode)
    check_decode(out, lse, *_ref(c, wl.decode))
    assert M.mla_get_error() == 0


def test_tiny_config_full_size():
    wl = workloads.tiny()
    g, c = build_both(wl)
    out, lse = gpu_decode(g, wl.decode)
    check_decode(out, lse, *_ref(c, wl.decode))


def test_minus_one_anywhere():
    wl = workloads.tiny(scatter_minus_one=True, T=7)
    g, c = build_both(wl)
    out, lse = gpu_decode(g, wl.decode)
    check_decode(out, lse, *_ref(c, wl.decode))


@pytest.mark.parametrize("name", ["nope", "prefill", "tiny"])
def test_slot0_contents_bit_identical(name):
    wl = workloads.small(name)
    res = []
    for b in (0x00, 0xFF, 0x7F):
        g, _ = build_both(wl, slot0_byte=b)
        g[0].fill_(b)
        out, lse = gpu_decode(g, wl.decode)
        res.append((out.cpu(), lse.cpu()))
    for o, l in res[1:]:
        assert torch.equal(o.view(torch.int16), res[0][0].view(torch.int16))
        assert torch.equal(l.view(torch.int32), res[0][1].view(torch.int32))
        assert torch.isfinite(o.float()).all()


def test_reserved_index_zero_and_empty_rows():
    wl = workloads.tiny(T=5)
    g, c = build_both(wl)
    tk = wl.decode.topk.clone()
    tk[1, :] = -1                      # empty row
    tk[2, :] = 0                       # only the reserved slot: empty too
    tk[3, 5] = 0
    tk[4, :] = -1
    tk[4, 127] = tk[0, 0]              # single entry at the very end
    out, lse = gpu_decode(g, wl.decode, topk=tk.to(dev()))
    ro, rl = _ref(c, wl.decode, topk=tk.numpy())
    check_decode(out, lse, ro, rl)
    assert torch.all(out[1:3] == 0) and torch.all(torch.isneginf(lse[1:3]))


def test_out_of_range_index_is_absent_and_flagged():
    wl = workloads.tiny()
    g, c = build_both(wl)
    M.mla_get_error()
    tk = wl.decode.topk.clone()
    tk[0, 90] = wl.num_slots           # one past the end
    tk[2, 3] = 2**31 - 1
    out, lse = gpu_decode(g, wl.decode, topk=tk.to(dev()))
    assert M.mla_get_error() == M.MLA_ERR_DECODE_INDEX_RANGE
    check_decode(out, lse, *_ref(c, wl.decode, topk=tk.numpy()))


@pytest.mark.parametrize("H", [1, 8, 20, 48])
def test_head_counts(H):
    wl = workloads.tiny(H=H, T=3)
    g, c = build_both(wl)
    out, lse = gpu_decode(g, wl.decode)
    check_decode(out, lse, *_ref(c, wl.decode))


def test_zero_width_and_zero_tokens():
    wl = workloads.tiny(T=2)
    g, _ = build_both(wl)
    d = dev()
    q = wl.decode.q.to(d)
    out, lse = M.mla_sparse_decode(q, g, torch.empty((2, 0), dtype=torch.int32, device=d), 0.1)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
    out, lse = M.mla_sparse_decode(q[:0], g, torch.empty((0, 8), dtype=torch.int32, device=d), 0.1)
    assert out.shape == (0, 16, 512)


def test_rope_query_over_nope_rows_equals_nope_decode():
    # A zero RoPE tail makes q_rope . k_rope exactly 0 (vLLM PR #55277, Purpose item 1):
    # d_qk = 576 over NoPE-written rows is bit-identical to the d_qk = 512 decode.
    wl = workloads.small("nope")
    g, _ = build_both(wl)
    d = dev()
    q512 = wl.decode.q.to(d)
    q576 = torch.cat([q512, torch.randn(q512.shape[0], q512.shape[1], 64, device=d).to(torch.bfloat16)], -1)
    a = M.mla_sparse_decode(q512, g, wl.decode.topk.to(d), wl.decode.sm_scale)
    b = M.mla_sparse_decode(q576.contiguous(), g, wl.decode.topk.to(d), wl.decode.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1], b[1])


def test_large_query_magnitude_and_duplicates():
    # q far outside f16 range (the kernel rescales q by a power of two) and a
    # duplicated slot (counted twice, as in the oracle).
    wl = workloads.tiny(T=2)
    g, c = build_both(wl)
    q = wl.decode.q.clone()
    q[0] = q[0] * 1e6
    tk = wl.decode.topk.clone()
    tk[1, 100] = tk[1, 0]
    db = workloads.DecodeBatch(q, tk, 1e-7)
    out, lse = gpu_decode(g, db)
    check_decode(out, lse, *_ref(c, db))


def test_workspace_errors():
    wl = workloads.small("nope")
    g, _ = build_both(wl)
    d = dev()
    db = wl.decode
    need = M.mla_sparse_decode_workspace_bytes(db.T, db.H, db.W)
    if need == 0:
        pytest.skip("no workspace needed for this shape on this device")
    small = torch.empty(need - 16, dtype=torch.uint8, device=d)
    with pytest.raises(M.MlaError) as ei:
        M.mla_sparse_decode(db.q.to(d), g, db.topk.to(d), db.sm_scale, workspace=small)
    assert ei.value.code == M.MLA_ENOWORKSPACE


def test_maximum_head_count():
    # H = 128: eight head groups of 16 in one launch (the largest H the ABI takes).
    wl = workloads.tiny(H=128, T=2)
    g, c = build_both(wl)
    out, lse = gpu_decode(g, wl.decode)
    check_decode(out, lse, *_ref(c, wl.decode))
    assert M.mla_get_error() == 0


def test_wide_list_split_past_one_cta():
    # W = 5,000 positions (4,000 present) per token: more than one CTA's list, so
    # the list is split and the partials merged.
    wl = workloads.tiny(T=2, W=5000, n_valid=4000, n_rows=4200, num_slots=8192)
    g, c = build_both(wl)
    assert M.mla_sparse_decode_workspace_bytes(2, 16, 5000) > 0
    out, lse = gpu_decode(g, wl.decode)
    check_decode(out, lse, *_ref(c, wl.decode))
    assert M.mla_get_error() == 0


def test_many_tokens():
    # T = 2,048 query tokens in one launch, compared on a sample of them.
    wl = workloads.tiny(T=2048)
    g, c = build_both(wl)
    db = wl.decode
    out, lse = gpu_decode(g, db)
    tokens = sorted(set(np.random.default_rng(8).choice(db.T, 48, replace=False).tolist()) | {0, db.T - 1})
    ro, rl, _ = oracle.sparse_decode(db.q, c, db.topk.numpy(), db.sm_scale, tokens=tokens)
    check_decode(out, lse, ro, rl, tokens=tokens)
    assert M.mla_get_error() == 0


@pytest.mark.parametrize("T,W,n_valid", [(2, 1024, 900), (160, 128, 100)])
def test_nan_row_makes_the_tokens_that_list_it_nan(T, W, n_valid):
    # A row written from NaN latent values holds E4M3 NaN codes. A token that
    # lists it gets NaN out and NaN lse, as the decode statement (and the oracle)
    # gives, whether its list is split across CTAs (first case: 2 tokens, split by
    # present entries, partials merged) or not (second case); the other tokens
    # are untouched.
    gen = torch.Generator().manual_seed(51)
    n = 2000
    lat = torch.randn((n, 512), generator=gen)
    lat[7] = float("nan")                                  # slot 8
    lat = lat.to(torch.bfloat16)
    rope = torch.randn((n, 64), generator=gen).to(torch.bfloat16)
    slots = torch.arange(1, n + 1, dtype=torch.int64)
    g = torch.zeros((4096, 656), dtype=torch.uint8, device=dev())
    M.mla_kv_write(g, slots.to(dev()), lat.to(dev()), rope.to(dev()))
    c = np.zeros((4096, 656), np.uint8)
    oracle.kv_write(c, slots.numpy(), lat, rope)
    topk = torch.full((T, W), -1, dtype=torch.int32)
    for t in range(T):
        pick = torch.randperm(n, generator=gen)[:n_valid] + 1
        pick = pick[pick != 8]
        if t % 2 == 0:
            pick[int(torch.randint(0, pick.numel(), (1,), generator=gen))] = 8
        topk[t, :pick.numel()] = pick.to(torch.int32)
    q = torch.randn((T, 16, 576), generator=gen).to(torch.bfloat16)
    if T == 2:
        assert M.mla_sparse_decode_workspace_bytes(T, 16, W) > 0, "this case is meant to split"
    out, lse = M.mla_sparse_decode(q.to(dev()), g, topk.to(dev()), 1.0 / 24.0)
    torch.cuda.synchronize()
    assert M.mla_get_error() == 0
    even, odd = list(range(0, T, 2)), list(range(1, T, 2))
    o, l = out.float().cpu(), lse.cpu()
    assert torch.isnan(o[even]).all() and torch.isnan(l[even]).all()
    ro, rl, _ = oracle.sparse_decode(q, c, topk.numpy(), 1.0 / 24.0, tokens=odd)
    assert np.isnan(oracle.sparse_decode(q, c, topk.numpy(), 1.0 / 24.0, tokens=even[:1])[1][even[0]]).all()
    check_decode(out, lse, ro, rl, tokens=odd)
