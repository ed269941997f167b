"""mla_sparse_decode_noalloc: the decode for callers that cannot allocate
device memory at the call site (for example code running inside another
framework's memory pool without an allocator handle, or a process that has
already committed its whole device-memory budget). It takes no workspace and
uses the library's fixed device array instead.

Called here through the C ABI (ctypes) and checked against mla_sparse_decode
with a caller-allocated workspace, within the tolerance of the other decode
tests, on two calls in a row (the array keeps the previous call's contents).
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


def _close(a_out, a_lse, b_out, b_lse):
    a = a_out.float().cpu().numpy().astype(np.float64)
    b = b_out.float().cpu().numpy().astype(np.float64)
    assert np.abs(a - b).max() <= 1e-2 * np.abs(b).max() + 1e-3
    la, lb = a_lse.cpu().numpy(), b_lse.cpu().numpy()
    assert np.array_equal(np.isneginf(la), np.isneginf(lb))
    fin = ~np.isneginf(lb)
    assert np.abs(la[fin] - lb[fin]).max() <= 1e-3


def test_noalloc_matches_workspace_decode_on_two_calls():
    fn = _lib()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    wl = workloads.small("nope")                 # ragged lengths, split across CTAs
    db = wl.decode
    cache = torch.full((wl.num_slots, 656), 0, dtype=torch.uint8, device=dev)
    f = wl.fill
    M.mla_kv_write(cache, f.slot_idx.to(dev), f.latent.to(dev), None)
    q, topk = db.q.to(dev), db.topk.to(dev)
    need = M.mla_sparse_decode_workspace_bytes(db.T, db.H, db.W)
    assert 0 < need <= SCRATCH_BYTES, "the shape must exercise the scratch array"
    ref_out, ref_lse = M.mla_sparse_decode(q, cache, topk, db.sm_scale)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out = torch.full((db.T, db.H, 512), float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full((db.T, db.H), float("nan"), dtype=torch.float32, device=dev)
        rc = fn(q.data_ptr(), db.T, db.H, db.d_qk, M.kv_cache(cache), topk.data_ptr(), db.W,
                db.sm_scale, out.data_ptr(), lse.data_ptr(), stream)
        assert rc == M.MLA_OK, M.strerror(rc)
        torch.cuda.synchronize()
        _close(out, lse, ref_out, ref_lse)
    assert M.mla_get_error() == 0


def test_noalloc_covers_or_rejects_every_shape():
    # The decode's workspace is a few partial rows per resident CTA, so on this
    # device it is bounded whatever the token count or top-k width: either the
    # array holds it, or the call is rejected before anything runs.
    fn = _lib()
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda:0")
    kv = M.KVCache(dummy.data_ptr(), 1, 656)
    for T, H, W in [(1, 16, 128), (4096, 128, 2048), (64, 16, 2304 * 40), (65535, 128, 65536)]:
        need = M.mla_sparse_decode_workspace_bytes(T, H, W)
        if need > SCRATCH_BYTES:
            rc = fn(dummy.data_ptr(), T, H, 576, kv, dummy.data_ptr(), W, 0.1, dummy.data_ptr(),
                    dummy.data_ptr(), None)
            assert rc == M.MLA_ENOWORKSPACE
        else:
            assert need >= 0
