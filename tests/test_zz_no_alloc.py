"""mla_sparse_decode_noalloc: the decode for callers that cannot allocate
device memory at the call site (for example code running inside another
framework's memory pool without an allocator handle, or a process that has
already committed its whole device-memory budget). It takes no workspace and
uses the library's fixed device array instead.

Called here through the C ABI (ctypes) and checked against mla_sparse_decode
with a caller-allocated workspace on the same inputs. Both run the same kernels
with the same split of the top-k lists, so the outputs must be bit-identical
(which is stricter than the decode tolerance the other tests use). Two calls in
a row use different inputs, so a call that read what the previous call left in
the shared array instead of what it wrote itself would be caught.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes when run alone.
"""
import ctypes

import numpy as np
import pytest
import torch

from fp8_mla_kv_gb300 import build as B
from fp8_mla_kv_gb300 import mlasparse as M
from fp8_mla_kv_gb300 import workloads

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 << 20


def _lib():
    B.build()
    lib = M.load()
    fn = lib.mla_sparse_decode_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, M.KVCache, ctypes.c_void_p,
                   ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return fn


def _noalloc(fn, q, cache, topk, T, H, d_qk, W, sm_scale):
    out = torch.full((T, H, 512), float("nan"), dtype=torch.bfloat16, device=q.device)
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device=q.device)
    rc = fn(q.data_ptr(), T, H, d_qk, M.kv_cache(cache), topk.data_ptr(), W, sm_scale, out.data_ptr(),
            lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == M.MLA_OK, M.strerror(rc)
    torch.cuda.synchronize()
    return out, lse


def _same(a_out, a_lse, b_out, b_lse):
    # Bit-identical, which also satisfies max|out-ref| <= 1e-2*max|ref| + 1e-3 and |lse-ref| <= 1e-3.
    assert torch.equal(a_out.view(torch.int16), b_out.view(torch.int16))
    assert torch.equal(a_lse.view(torch.int32), b_lse.view(torch.int32))


def _nope_inputs(dev):
    wl = workloads.small("nope")                 # ragged lengths, split across CTAs
    cache = torch.zeros((wl.num_slots, 656), dtype=torch.uint8, device=dev)
    f = wl.fill
    M.mla_kv_write(cache, f.slot_idx.to(dev), f.latent.to(dev), None)
    return wl, cache


def test_noalloc_matches_workspace_decode_on_two_calls():
    fn = _lib()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    wl, cache = _nope_inputs(dev)
    db = wl.decode
    need = M.mla_sparse_decode_workspace_bytes(db.T, db.H, db.W)
    assert 0 < need <= SCRATCH_BYTES, "the shape must exercise the scratch array"
    # Call 1: the workload's q and lists. Call 2: another q, and each token's
    # list reversed with a different number of present entries, so the partial
    # results the second call needs differ from the ones the first left behind.
    g = torch.Generator().manual_seed(1234)
    q2 = torch.randn(db.q.shape, generator=g).to(torch.bfloat16)
    topk2 = db.topk.clone()
    for t in range(db.T):
        row = topk2[t]
        present = row[row > 0]
        keep = max(1, int(present.numel() * (0.3 + 0.6 * ((t * 37) % 11) / 10)))
        new = torch.full_like(row, -1)
        new[: keep] = present.flip(0)[:keep]
        topk2[t] = new
    for q_h, topk_h in ((db.q, db.topk), (q2, topk2)):
        q, topk = q_h.to(dev), topk_h.to(dev)
        ref_out, ref_lse = M.mla_sparse_decode(q, cache, topk, db.sm_scale)
        torch.cuda.synchronize()
        out, lse = _noalloc(fn, q, cache, topk, db.T, db.H, db.d_qk, db.W, db.sm_scale)
        _same(out, lse, ref_out, ref_lse)
    assert M.mla_get_error() == 0


def test_noalloc_runs_small_shapes_and_rejects_large_ones():
    # The workspace grows with T * nsplit * H (nsplit: pieces per token list on
    # this device). Shapes whose workspace fits the array run; larger ones are
    # rejected before anything is launched and leave the error word untouched.
    fn = _lib()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    wl, cache = _nope_inputs(dev)
    g = torch.Generator().manual_seed(99)
    T, H, W = 1, 16, 512
    need = M.mla_sparse_decode_workspace_bytes(T, H, W)
    assert 0 < need <= SCRATCH_BYTES
    q = torch.randn((T, H, 512), generator=g).to(torch.bfloat16).to(dev)
    slots = torch.randperm(wl.num_slots - 1, generator=g)[:W].to(torch.int32) + 1
    slots[300:] = -1
    topk = slots.view(T, W).to(dev)
    ref_out, ref_lse = M.mla_sparse_decode(q, cache, topk, 0.05)
    torch.cuda.synchronize()
    out, lse = _noalloc(fn, q, cache, topk, T, H, 512, W, 0.05)
    _same(out, lse, ref_out, ref_lse)
    assert M.mla_get_error() == 0

    dummy = torch.empty(16, dtype=torch.uint8, device=dev)
    kv = M.KVCache(dummy.data_ptr(), 1, 656)
    rejected = 0
    for T, H, W in [(4096, 128, 2048), (64, 16, 2304 * 40), (65535, 128, 65536)]:
        need = M.mla_sparse_decode_workspace_bytes(T, H, W)
        if need <= SCRATCH_BYTES:
            continue
        rc = fn(dummy.data_ptr(), T, H, 576, kv, dummy.data_ptr(), W, 0.1, dummy.data_ptr(),
                dummy.data_ptr(), None)
        assert rc == M.MLA_ENOWORKSPACE
        rejected += 1
    assert rejected > 0
    assert M.mla_get_error() == 0
