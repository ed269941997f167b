"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and the CPU oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from fp8_mla_kv_gb300 import mlasparse as M

OUT_RTOL = 1e-2     # max|out - ref| <= 1e-2 * max|ref| + 1e-3
OUT_ATOL = 1e-3
LSE_ATOL = 1e-3     # |lse - ref| <= 1e-3


def dev():
    return torch.device("cuda:0")


def gpu_cache(wl, slot0_byte=None):
    b = wl.slot0_byte if slot0_byte is None else slot0_byte
    return torch.full((wl.num_slots, 656), b, dtype=torch.uint8, device=dev())


def cpu_cache(wl, slot0_byte=None):
    b = wl.slot0_byte if slot0_byte is None else slot0_byte
    return np.full((wl.num_slots, 656), b, np.uint8)


def gpu_write(cache, wb):
    d = dev()
    M.mla_kv_write(cache, wb.slot_idx.to(d), wb.latent.to(d), None if wb.rope is None else wb.rope.to(d))


def cpu_write(cache, wb):
    oracle.kv_write(cache, wb.slot_idx.numpy(), wb.latent, wb.rope)


def build_both(wl, slot0_byte=None):
    """Fill + writes of a workload on both sides; returns (gpu cache, cpu cache)."""
    g = gpu_cache(wl, slot0_byte)
    c = cpu_cache(wl, slot0_byte)
    for wb in ([wl.fill] if wl.fill is not None else []) + list(wl.writes):
        gpu_write(g, wb)
        cpu_write(c, wb)
    torch.cuda.synchronize()
    return g, c


def gpu_decode(cache, db, q=None, topk=None):
    d = dev()
    q = db.q.to(d) if q is None else q
    topk = db.topk.to(d) if topk is None else topk
    out, lse = M.mla_sparse_decode(q, cache, topk, db.sm_scale)
    torch.cuda.synchronize()
    return out, lse


def check_decode(out, lse, ref_out, ref_lse, tokens=None):
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    if tokens is not None:
        o, l, ref_out, ref_lse = o[tokens], l[tokens], ref_out[tokens], ref_lse[tokens]
    empty = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(l), empty), "empty (token, head) pairs differ"
    assert np.all(o[empty] == 0)
    tol = OUT_RTOL * np.abs(ref_out).max() + OUT_ATOL
    err_o = np.abs(o - ref_out).max()
    err_l = np.abs(l[~empty] - ref_lse[~empty]).max() if (~empty).any() else 0.0
    assert np.isfinite(o).all()
    assert err_o <= tol, f"max|out-ref| = {err_o:.3e} > {tol:.3e}"
    assert err_l <= LSE_ATOL, f"max|lse-ref| = {err_l:.3e}"
    return err_o, tol, err_l
