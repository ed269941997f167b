"""Pins for the oracle's sparse top-k MLA decode.

The brute force below is an independent routine: it decodes the cache bytes with
torch's float8_e4m3fn table (not the oracle's codec), builds dense K/V for all
slots, and runs a textbook masked softmax in numpy float64. The other tests pin
closed forms and invariants the pages fix: masked (-1) and reserved-slot entries
contribute nothing (sglang PR #39288, Root cause), and a zero RoPE lane is
bit-exact NoPE (vLLM PR #55277, Purpose item 1)."""
import math

import numpy as np
import pytest
import torch

import oracle

S = 96


def _cache(seed=0, rope=True, slot0=0x00, same_rows=None):
    g = torch.Generator().manual_seed(seed)
    lat = torch.randn((S - 1, 512), generator=g).to(torch.bfloat16)
    rp = torch.randn((S - 1, 64), generator=g).to(torch.bfloat16) if rope else None
    if same_rows is not None:
        lat[same_rows] = lat[same_rows[0]].clone()
        if rp is not None:
            rp[same_rows] = rp[same_rows[0]].clone()
    cache = np.full((S, 656), slot0, np.uint8)
    oracle.kv_write(cache, np.arange(1, S), lat, rp)
    return cache


def _dense_kv(cache):
    """Independent decoder: torch's fp8 table and numpy's view of the fp32 scales."""
    table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    lat = table[cache[:, :512]]
    sc = cache[:, 512:528].copy().view("<f4").astype(np.float64)      # [S, 4]
    K = lat * np.repeat(sc, 128, axis=1)
    rope = cache[:, 528:656].copy().view("<u2").astype(np.uint32) << 16
    R = rope.view(np.float32).astype(np.float64)
    return K, R


def _brute(q, cache, topk, sm_scale):
    K, R = _dense_kv(cache)
    qf = q.float().numpy().astype(np.float64)
    T, H, D = qf.shape
    out = np.zeros((T, H, 512))
    lse = np.full((T, H), -np.inf)
    for t in range(T):
        mask = np.zeros(cache.shape[0], dtype=np.float64)    # multiplicity of each slot
        for idx in topk[t]:
            if 0 < idx < cache.shape[0]:
                mask[idx] += 1
        if mask.sum() == 0:
            continue
        sel = mask > 0
        Ks, Rs, w = K[sel], R[sel], mask[sel]
        s = qf[t, :, :512] @ Ks.T
        if D == 576:
            s = s + qf[t, :, 512:] @ Rs.T
        s = sm_scale * s                                      # [H, n]
        m = s.max(axis=1, keepdims=True)
        p = w[None, :] * np.exp(s - m)
        l = p.sum(axis=1, keepdims=True)
        out[t] = (p @ Ks) / l
        lse[t] = (m + np.log(l))[:, 0]
    return out, lse


def _q(T, H, D, seed=1):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((T, H, D), generator=g).to(torch.bfloat16)


def _topk(T, W, n_valid, seed=2, scatter=True, extra=()):
    g = torch.Generator().manual_seed(seed)
    tk = np.full((T, W), -1, np.int32)
    for t in range(T):
        k = n_valid[t] if hasattr(n_valid, "__len__") else n_valid
        slots = (torch.randperm(S - 1, generator=g)[:k] + 1).numpy()
        pos = torch.randperm(W, generator=g)[:k].numpy() if scatter else np.arange(k)
        tk[t, pos] = slots
    for (t, j, v) in extra:
        tk[t, j] = v
    return tk


@pytest.mark.parametrize("rope", [True, False])
def test_matches_brute_force(rope):
    cache = _cache(rope=rope)
    D = 576 if rope else 512
    q = _q(4, 5, D)
    tk = _topk(4, 48, [1, 17, 30, 48], extra=[(2, 3, 0), (2, 4, S + 5)])
    sm = 1.0 / math.sqrt(D)
    out, lse, bad = oracle.sparse_decode(q, cache, tk, sm, n_threads=2)
    ref_out, ref_lse = _brute(q, cache, tk, np.float64(np.float32(sm)))
    assert bad == (1 if tk[2, 4] == S + 5 else 0)
    np.testing.assert_allclose(out, ref_out, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_single_entry_closed_form():
    cache = _cache()
    K, R = _dense_kv(cache)
    q = _q(1, 3, 576)
    tk = np.full((1, 16), -1, np.int32)
    tk[0, 7] = 42
    sm = np.float32(0.05)
    out, lse, _ = oracle.sparse_decode(q, cache, tk, float(sm))
    qf = q.float().numpy().astype(np.float64)[0]
    s = float(sm) * (qf[:, :512] @ K[42] + qf[:, 512:] @ R[42])
    assert np.array_equal(out[0], np.broadcast_to(K[42], (3, 512)))
    np.testing.assert_allclose(lse[0], s, rtol=0, atol=1e-12)


def test_uniform_scores_give_mean_and_log_count():
    cache = _cache()
    K, _ = _dense_kv(cache)
    q = torch.zeros((1, 2, 576), dtype=torch.bfloat16)
    tk = _topk(1, 64, 37)
    out, lse, _ = oracle.sparse_decode(q, cache, tk, 0.1)
    sel = tk[0][tk[0] > 0]
    np.testing.assert_allclose(out[0, 0], K[sel].mean(axis=0), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse[0], math.log(37), rtol=0, atol=1e-13)


def test_all_equal_rows_give_that_row():
    rows = [3, 9, 27, 50]
    cache = _cache(same_rows=[r - 1 for r in rows])
    K, _ = _dense_kv(cache)
    q = _q(1, 4, 576)
    tk = np.array([[rows[0], -1, rows[1], rows[2], -1, rows[3]]], np.int32)
    out, _, _ = oracle.sparse_decode(q, cache, tk, 0.3)
    np.testing.assert_allclose(out[0], np.broadcast_to(K[rows[0]], (4, 512)), rtol=1e-13, atol=1e-14)


def test_empty_gives_zero_and_minus_inf():
    cache = _cache()
    q = _q(2, 3, 576)
    tk = np.array([[-1, 0, -1, -7], [0, 0, 0, 0]], np.int32)
    out, lse, _ = oracle.sparse_decode(q, cache, tk, 0.1)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_permutation_and_padding_position_invariance():
    cache = _cache()
    q = _q(3, 4, 576)
    tk = _topk(3, 40, [5, 20, 33], scatter=False)
    out0, lse0, _ = oracle.sparse_decode(q, cache, tk, 0.07)
    rng = np.random.default_rng(5)
    tk2 = np.stack([rng.permutation(r) for r in tk])
    out1, lse1, _ = oracle.sparse_decode(q, cache, tk2, 0.07)
    np.testing.assert_allclose(out1, out0, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse1, lse0, rtol=1e-13, atol=1e-13)


def test_slot0_contents_do_not_matter():
    q = _q(3, 4, 576)
    tk = _topk(3, 40, [5, 20, 33], extra=[(0, 39, 0), (1, 0, 0)])
    res = []
    for fill in (0x00, 0xFF, 0x7F):
        cache = _cache(slot0=fill)
        cache[0, :] = fill
        res.append(oracle.sparse_decode(q, cache, tk, 0.07))
    for r in res[1:]:
        assert np.array_equal(r[0], res[0][0]) and np.array_equal(r[1], res[0][1])
        assert not np.isnan(r[0]).any()


def test_zero_rope_equals_nope_exactly():
    cache = _cache(rope=False)
    q576 = _q(2, 4, 576)
    q512 = q576[:, :, :512].contiguous()
    tk = _topk(2, 32, [9, 31])
    a = oracle.sparse_decode(q576, cache, tk, 0.05)
    b = oracle.sparse_decode(q512, cache, tk, 0.05)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_token_subset_matches_full():
    cache = _cache()
    q = _q(5, 2, 576)
    tk = _topk(5, 32, [3, 4, 5, 6, 7])
    full = oracle.sparse_decode(q, cache, tk, 0.1)
    part = oracle.sparse_decode(q, cache, tk, 0.1, tokens=[1, 4])
    for t in (1, 4):
        assert np.array_equal(part[0][t], full[0][t]) and np.array_equal(part[1][t], full[1][t])
    assert np.isnan(part[0][0]).all()
