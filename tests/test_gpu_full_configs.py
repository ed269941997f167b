"""Full-size workloads, in the launch configuration the bench times: the whole
cache is compared byte for byte with the oracle's, and the decode output of
every token and head with the oracle's (a few seconds of oracle time each)."""
import numpy as np
import pytest
import torch

import oracle
from fp8_mla_kv_gb300 import mlasparse as M
from fp8_mla_kv_gb300 import workloads

from _parity import build_both, check_decode, gpu_decode

pytestmark = pytest.mark.gpu


def _run(wl, tokens, slot0_byte=None):
    g, c = build_both(wl, slot0_byte)
    assert M.mla_get_error() == 0
    assert np.array_equal(g.cpu().numpy(), c), "cache differs from the oracle's"
    db = wl.decode
    out, lse = gpu_decode(g, db)
    ro, rl, _ = oracle.sparse_decode(db.q, c, db.topk.numpy(), db.sm_scale, tokens=tokens)
    errs = check_decode(out, lse, ro, rl, tokens=tokens)
    assert M.mla_get_error() == 0
    return g, errs


def test_tiny_full():
    wl = workloads.tiny()
    _run(wl, None)


def test_nope_full_and_slot0_poison():
    wl = workloads.nope()
    g, _ = _run(wl, None)
    db = wl.decode
    a = gpu_decode(g, db)
    g[0].fill_(0xFF)
    b = gpu_decode(g, db)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))


def test_rope_full():
    wl = workloads.rope()
    _run(wl, None)


def test_prefill_full():
    wl = workloads.prefill()
    _run(wl, None)


def test_sweep_full():
    wl = workloads.sweep()
    _run(wl, None)
