"""Thin ctypes binding to libmlasparse (include/mlasparse.h), same function names.

Argument marshalling only: torch tensors supply device memory and the current
CUDA stream; every step of the computation runs in the library's kernels. The
library is loaded on first use; if it is missing or no CUDA device is present,
the call raises. There is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import ROW_BYTES, ROW_BYTES_NOPE

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmlasparse.so")

MLA_OK = 0
MLA_EINVAL = -1
MLA_EUNSUPPORTED = -2
MLA_ENOWORKSPACE = -3
MLA_ECUDA = -4
MLA_ERR_WRITE_SLOT_RANGE = 0x1
MLA_ERR_DECODE_INDEX_RANGE = 0x2
MLA_ERR_PIPELINE_TIMEOUT = 0x4
MLA_ERR_GATHER_INDEX_RANGE = 0x8

SYMBOLS = ("mla_kv_write", "mla_sparse_decode", "mla_sparse_decode_workspace_bytes",
           "mla_sparse_decode_paged", "mla_sparse_prefill", "mla_sparse_prefill_paged",
           "mla_gather_upconvert", "mla_get_error", "mla_strerror")


class MlaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


class KVCache(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("num_slots", ctypes.c_int64), ("row_bytes", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the shared library (raises OSError if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise OSError(f"libmlasparse not built: {path} is missing "
                              "(run fp8_mla_kv_gb300.build.build() or __graft_entry__.build())")
            lib = ctypes.CDLL(path)
            c = ctypes
            lib.mla_kv_write.restype = c.c_int
            lib.mla_kv_write.argtypes = [KVCache, c.c_void_p, c.c_void_p, c.c_void_p, c.c_int64, c.c_int64,
                                         c.c_void_p]
            lib.mla_sparse_decode_workspace_bytes.restype = c.c_size_t
            lib.mla_sparse_decode_workspace_bytes.argtypes = [c.c_int, c.c_int, c.c_int]
            lib.mla_sparse_decode.restype = c.c_int
            lib.mla_sparse_decode.argtypes = [c.c_void_p, c.c_int, c.c_int, c.c_int, KVCache, c.c_void_p,
                                              c.c_int, c.c_float, c.c_void_p, c.c_void_p, c.c_void_p,
                                              c.c_size_t, c.c_void_p]
            lib.mla_sparse_decode_paged.restype = c.c_int
            lib.mla_sparse_decode_paged.argtypes = [c.c_void_p, c.c_int, c.c_int, c.c_int, KVCache, c.c_void_p,
                                                    c.c_int, c.c_void_p, c.c_int, c.c_int, c.c_void_p, c.c_int,
                                                    c.c_float, c.c_void_p, c.c_void_p, c.c_void_p, c.c_size_t,
                                                    c.c_void_p]
            lib.mla_sparse_prefill.restype = c.c_int
            lib.mla_sparse_prefill.argtypes = [c.c_void_p, c.c_int, c.c_int, c.c_int, KVCache, c.c_void_p,
                                               c.c_int, c.c_float, c.c_void_p, c.c_void_p, c.c_void_p]
            lib.mla_sparse_prefill_paged.restype = c.c_int
            lib.mla_sparse_prefill_paged.argtypes = [c.c_void_p, c.c_int, c.c_int, c.c_int, KVCache, c.c_void_p,
                                                     c.c_int, c.c_void_p, c.c_int, c.c_int, c.c_void_p, c.c_int,
                                                     c.c_float, c.c_void_p, c.c_void_p, c.c_void_p]
            lib.mla_gather_upconvert.restype = c.c_int
            lib.mla_gather_upconvert.argtypes = [KVCache, c.c_void_p, c.c_int64, c.c_int, c.c_void_p, c.c_void_p]
            lib.mla_get_error.restype = c.c_int
            lib.mla_get_error.argtypes = [c.POINTER(c.c_int32)]
            lib.mla_strerror.restype = c.c_char_p
            lib.mla_strerror.argtypes = [c.c_int]
            _lib = lib
    return _lib


def strerror(code: int) -> str:
    try:
        return load().mla_strerror(int(code)).decode()
    except OSError:
        return f"code {code}"


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libmlasparse takes device tensors only")


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def kv_cache(cache: torch.Tensor) -> KVCache:
    """View a uint8 [num_slots, 656] (or [num_slots, 528] NoPE-only) device tensor
    as the C cache descriptor."""
    if (cache.dtype != torch.uint8 or cache.dim() != 2 or cache.shape[1] not in (ROW_BYTES, ROW_BYTES_NOPE)
            or not cache.is_contiguous()):
        raise ValueError("cache must be a contiguous uint8 tensor [num_slots, 656] or [num_slots, 528]")
    return KVCache(cache.data_ptr(), cache.shape[0], int(cache.shape[1]))


def mla_kv_write(cache: torch.Tensor, slot_idx: torch.Tensor, latent: torch.Tensor,
                 rope: torch.Tensor | None, reserved_slot: int = 0, stream=None) -> None:
    _require_cuda(cache, slot_idx, latent, rope)
    n = int(slot_idx.shape[0])
    assert slot_idx.dtype == torch.int64 and slot_idx.is_contiguous()
    assert latent.dtype == torch.bfloat16 and latent.is_contiguous() and latent.numel() == n * 512
    if rope is not None:
        assert rope.dtype == torch.bfloat16 and rope.is_contiguous() and rope.numel() == n * 64
    rc = load().mla_kv_write(kv_cache(cache), slot_idx.data_ptr(), latent.data_ptr(),
                             rope.data_ptr() if rope is not None else None, n, int(reserved_slot),
                             _stream(stream))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_kv_write")


def mla_sparse_decode_workspace_bytes(T: int, H: int, W: int) -> int:
    return int(load().mla_sparse_decode_workspace_bytes(int(T), int(H), int(W)))


def alloc_workspace(T: int, H: int, W: int, device=None) -> torch.Tensor | None:
    n = mla_sparse_decode_workspace_bytes(T, H, W)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def mla_sparse_decode(q: torch.Tensor, cache: torch.Tensor, topk_idx: torch.Tensor, sm_scale: float,
                      out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, stream=None):
    """q bf16 [T, H, d_qk]; topk int32 [T, W]; returns (out bf16 [T, H, 512], lse fp32 [T, H])."""
    _require_cuda(q, cache, topk_idx)
    T, H, d_qk = (int(s) for s in q.shape)
    W = int(topk_idx.shape[1])
    assert q.dtype == torch.bfloat16 and q.is_contiguous()
    assert topk_idx.dtype == torch.int32 and topk_idx.is_contiguous() and topk_idx.shape[0] == T
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(T, H, W, q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_n = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load().mla_sparse_decode(q.data_ptr(), T, H, d_qk, kv_cache(cache), topk_idx.data_ptr(), W,
                                  float(sm_scale), out.data_ptr(), lse.data_ptr(), ws_ptr, ws_n,
                                  _stream(stream))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_sparse_decode")
    return out, lse


def mla_sparse_decode_paged(q: torch.Tensor, cache: torch.Tensor, topk_pos: torch.Tensor,
                            block_table: torch.Tensor, page_size: int, sm_scale: float,
                            token_seq: torch.Tensor | None = None, out: torch.Tensor | None = None,
                            lse: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None):
    """Decode with the top-k given as sequence positions: q bf16 [T, H, d_qk]; topk_pos
    int32 [T, W]; block_table int32 [n_seq, max_pages] (or [max_pages]); token_seq int32
    [T] or None. Returns (out bf16 [T, H, 512], lse fp32 [T, H])."""
    _require_cuda(q, cache, topk_pos, block_table, token_seq)
    T, H, d_qk = (int(s) for s in q.shape)
    W = int(topk_pos.shape[1])
    bt = block_table if block_table.dim() == 2 else block_table.view(1, -1)
    assert q.dtype == torch.bfloat16 and q.is_contiguous()
    assert topk_pos.dtype == torch.int32 and topk_pos.is_contiguous() and topk_pos.shape[0] == T
    assert bt.dtype == torch.int32 and bt.is_contiguous()
    if token_seq is not None:
        assert token_seq.dtype == torch.int32 and token_seq.is_contiguous() and token_seq.numel() == T
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(T, H, W, q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_n = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load().mla_sparse_decode_paged(q.data_ptr(), T, H, d_qk, kv_cache(cache), topk_pos.data_ptr(), W,
                                        bt.data_ptr(), int(bt.shape[0]), int(bt.shape[1]),
                                        token_seq.data_ptr() if token_seq is not None else None, int(page_size),
                                        float(sm_scale), out.data_ptr(), lse.data_ptr(), ws_ptr, ws_n,
                                        _stream(stream))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_sparse_decode_paged")
    return out, lse


def mla_sparse_prefill(q: torch.Tensor, cache: torch.Tensor, topk_idx: torch.Tensor, sm_scale: float,
                       out: torch.Tensor | None = None, lse: torch.Tensor | None = None, stream=None):
    """What mla_sparse_decode computes, by token pairs that share their rows (causal
    prefill): q bf16 [T, H, d_qk]; topk int32 [T, W] with W <= 2304; returns
    (out bf16 [T, H, 512], lse fp32 [T, H]). No workspace."""
    _require_cuda(q, cache, topk_idx)
    T, H, d_qk = (int(s) for s in q.shape)
    W = int(topk_idx.shape[1])
    assert q.dtype == torch.bfloat16 and q.is_contiguous()
    assert topk_idx.dtype == torch.int32 and topk_idx.is_contiguous() and topk_idx.shape[0] == T
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    rc = load().mla_sparse_prefill(q.data_ptr(), T, H, d_qk, kv_cache(cache), topk_idx.data_ptr(), W,
                                   float(sm_scale), out.data_ptr(), lse.data_ptr(), _stream(stream))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_sparse_prefill")
    return out, lse


def mla_sparse_prefill_paged(q: torch.Tensor, cache: torch.Tensor, topk_pos: torch.Tensor,
                             block_table: torch.Tensor, page_size: int, sm_scale: float,
                             token_seq: torch.Tensor | None = None, out: torch.Tensor | None = None,
                             lse: torch.Tensor | None = None, stream=None):
    """mla_sparse_prefill with the top-k given as sequence positions through a block
    table (arguments as mla_sparse_decode_paged, no workspace)."""
    _require_cuda(q, cache, topk_pos, block_table, token_seq)
    T, H, d_qk = (int(s) for s in q.shape)
    W = int(topk_pos.shape[1])
    bt = block_table if block_table.dim() == 2 else block_table.view(1, -1)
    assert q.dtype == torch.bfloat16 and q.is_contiguous()
    assert topk_pos.dtype == torch.int32 and topk_pos.is_contiguous() and topk_pos.shape[0] == T
    assert bt.dtype == torch.int32 and bt.is_contiguous()
    if token_seq is not None:
        assert token_seq.dtype == torch.int32 and token_seq.is_contiguous() and token_seq.numel() == T
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    rc = load().mla_sparse_prefill_paged(q.data_ptr(), T, H, d_qk, kv_cache(cache), topk_pos.data_ptr(), W,
                                         bt.data_ptr(), int(bt.shape[0]), int(bt.shape[1]),
                                         token_seq.data_ptr() if token_seq is not None else None,
                                         int(page_size), float(sm_scale), out.data_ptr(), lse.data_ptr(),
                                         _stream(stream))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_sparse_prefill_paged")
    return out, lse


def mla_gather_upconvert(cache: torch.Tensor, slots: torch.Tensor, pe_dim: int,
                         out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Rows at slots (int32 [n]) widened to bf16 [n, 576]."""
    _require_cuda(cache, slots, out)
    n = int(slots.numel())
    assert slots.dtype == torch.int32 and slots.is_contiguous()
    if out is None:
        out = torch.empty((n, 576), dtype=torch.bfloat16, device=cache.device)
    assert out.dtype == torch.bfloat16 and out.is_contiguous() and out.numel() == n * 576
    rc = load().mla_gather_upconvert(kv_cache(cache), slots.data_ptr(), n, int(pe_dim), out.data_ptr(),
                                     _stream(stream))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_gather_upconvert")
    return out


def mla_get_error() -> int:
    v = ctypes.c_int32(0)
    rc = load().mla_get_error(ctypes.byref(v))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_get_error")
    return int(v.value)
