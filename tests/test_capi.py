"""The C ABI library builds for sm_103a, loads, exports every entry point that
include/mlasparse.h declares, and rejects bad arguments on the host (no GPU)."""
import ctypes
import os
import re

import pytest

from fp8_mla_kv_gb300 import build as B
from fp8_mla_kv_gb300 import mlasparse as M

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "mlasparse.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(mla_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return M.load()


def test_header_declares_the_boundary():
    fns = declared_functions()
    for name in ("mla_kv_write", "mla_sparse_decode", "mla_sparse_decode_workspace_bytes",
                 "mla_get_error", "mla_strerror"):
        assert name in fns
    assert set(M.SYMBOLS) <= set(fns)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_host_validation_without_gpu(lib):
    kv = M.KVCache(None, 16, 656)
    # negative row count / wrong row size: rejected before any CUDA call
    assert lib.mla_kv_write(kv, None, None, None, -1, 0, None) == M.MLA_EINVAL
    assert lib.mla_kv_write(M.KVCache(None, 16, 600), None, None, None, 4, 0, None) == M.MLA_EINVAL
    assert lib.mla_kv_write(kv, None, None, None, 0, 0, None) == M.MLA_OK
    assert lib.mla_kv_write(kv, None, None, None, 3, 0, None) == M.MLA_EINVAL   # null pointers
    # unsupported head dim / head count
    assert lib.mla_sparse_decode(None, 1, 16, 300, kv, None, 8, 0.1, None, None, None, 0, None) == M.MLA_EUNSUPPORTED
    assert lib.mla_sparse_decode(None, 1, 0, 576, kv, None, 8, 0.1, None, None, None, 0, None) == M.MLA_EUNSUPPORTED
    assert lib.mla_sparse_decode(None, 1, 129, 576, kv, None, 8, 0.1, None, None, None, 0, None) == M.MLA_EUNSUPPORTED
    assert lib.mla_sparse_decode(None, 1, 16, 576, kv, None, 8, float("nan"), None, None, None, 0, None) == M.MLA_EINVAL
    assert lib.mla_sparse_decode(None, 0, 16, 576, kv, None, 8, 0.1, None, None, None, 0, None) == M.MLA_OK
    assert lib.mla_sparse_decode(None, 2, 16, 576, kv, None, 8, 0.1, None, None, None, 0, None) == M.MLA_EINVAL
    assert lib.mla_sparse_decode_workspace_bytes(0, 16, 8) == 0
    # 528-byte rows take NoPE calls only
    kv528 = M.KVCache(None, 16, 528)
    rope = ctypes.c_void_p(16)
    assert lib.mla_kv_write(kv528, None, None, rope, 3, 0, None) == M.MLA_EINVAL
    assert lib.mla_sparse_decode(None, 1, 16, 576, kv528, None, 8, 0.1, None, None, None, 0, None) == M.MLA_EUNSUPPORTED
    assert lib.mla_gather_upconvert(kv528, None, 4, 64, None, None) == M.MLA_EINVAL
    # gather-and-upconvert: bad pe_dim, empty call, null pointers
    assert lib.mla_gather_upconvert(kv, None, 4, 32, None, None) == M.MLA_EINVAL
    assert lib.mla_gather_upconvert(kv, None, 0, 64, None, None) == M.MLA_OK
    assert lib.mla_gather_upconvert(kv, None, 4, 64, None, None) == M.MLA_EINVAL
    # paged decode: page size, table and sequence count are checked first
    for ps, bt, nseq, mp in ((0, 16, 1, 4), (64, None, 1, 4), (64, 16, 0, 4), (64, 16, 1, 0)):
        assert lib.mla_sparse_decode_paged(None, 1, 16, 576, kv, None, 8, bt, nseq, mp, None, ps, 0.1,
                                           None, None, None, 0, None) == M.MLA_EINVAL
    # prefill: same checks as the decode, and W past one CTA's list is refused
    pf = lib.mla_sparse_prefill
    assert pf(None, 1, 16, 300, kv, None, 8, 0.1, None, None, None) == M.MLA_EUNSUPPORTED
    assert pf(None, 1, 129, 576, kv, None, 8, 0.1, None, None, None) == M.MLA_EUNSUPPORTED
    assert pf(None, 1, 16, 576, kv, None, 2305, 0.1, None, None, None) == M.MLA_EUNSUPPORTED
    assert pf(None, 1, 16, 576, kv, None, 8, float("inf"), None, None, None) == M.MLA_EINVAL
    assert pf(None, 0, 16, 576, kv, None, 8, 0.1, None, None, None) == M.MLA_OK
    assert pf(None, 2, 16, 576, kv, None, 8, 0.1, None, None, None) == M.MLA_EINVAL
    assert pf(None, 1, 16, 576, kv528, None, 8, 0.1, None, None, None) == M.MLA_EUNSUPPORTED
    for ps, bt, nseq, mp in ((0, 16, 1, 4), (64, None, 1, 4), (64, 16, 0, 4), (64, 16, 1, 0)):
        assert lib.mla_sparse_prefill_paged(None, 1, 16, 576, kv, None, 8, bt, nseq, mp, None, ps, 0.1,
                                            None, None, None) == M.MLA_EINVAL
    for code in (0, -1, -2, -3, -4):
        assert lib.mla_strerror(code)
