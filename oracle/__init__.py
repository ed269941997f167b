"""Scalar CPU oracle for the FP8 MLA KV writer and the sparse top-k MLA decode.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package. The CUDA
library never loads it, and it shares no code with the CUDA library.

Parity status (what pins each function to something other than itself):
  * ``e4m3_encode`` / ``e4m3_decode`` - pinned: all 256 codes against torch's
    ``float8_e4m3fn`` table, closed-form values, and a structured sweep of fp32
    bit patterns against torch's cast (clamped to +-448 for the saturating form).
  * ``kv_write`` - pinned by invariants: layout, amax byte 0x7E/0xFE, the
    half-ulp dequantisation bound, sentinel bytes untouched, NoPE tail zero,
    rope tail bit-identical, reserved slot untouched; and by a reduction of one
    tile to torch's fp8 cast.
  * ``sparse_decode`` - pinned by a brute-force dense masked softmax in numpy
    (with torch's fp8 table as the decoder) on tiny inputs, closed forms
    (single entry, q = 0, all-equal rows), permutation invariance and the
    zero-RoPE == NoPE identity.
  * 528-byte rows (``kv_write`` / ``sparse_decode`` on a [N, 528] cache) -
    pinned: each row equals the first 528 bytes of the 656-byte NoPE row, and
    the decode over them equals the decode over the 656-byte NoPE cache.
  * ``paged_to_physical`` - pinned against the prefill workload's generator,
    which maps its positions to slots with its own code, and by the identity
    block table.
  * ``gather_upconvert`` - pinned: with power-of-two scales against torch's
    float8_e4m3fn -> bfloat16 conversion; with arbitrary scales against an
    exact rational nearest-BF16 search; RoPE tail bit-identical, NoPE tail and
    absent rows zero.

The arithmetic lives in ``mla_oracle.cpp`` (scalar C++17, float64 accumulation).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle_mla.so")
_lock = threading.Lock()
_lib = None

ROW_BYTES = 656       # restated from the row layout, not imported from the library
ROW_BYTES_NOPE = 528  # the canonical NoPE row: latent + scales, no tail


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (portable C++17, no SIMD intrinsics)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            c = ctypes
            lib.oracle_e4m3_decode.restype = c.c_double
            lib.oracle_e4m3_decode.argtypes = [c.c_uint8]
            lib.oracle_e4m3_encode.restype = c.c_uint8
            lib.oracle_e4m3_encode.argtypes = [c.c_float]
            lib.oracle_e4m3_encode_array.restype = None
            lib.oracle_e4m3_encode_array.argtypes = [c.c_void_p, c.c_void_p, c.c_int64]
            lib.oracle_e4m3_encode_bit_range.restype = None
            lib.oracle_e4m3_encode_bit_range.argtypes = [c.c_uint64, c.c_uint64, c.c_void_p, c.c_int]
            lib.oracle_kv_write.restype = c.c_int64
            lib.oracle_kv_write.argtypes = [c.c_void_p, c.c_int64, c.c_void_p, c.c_void_p,
                                            c.c_void_p, c.c_int64, c.c_int64]
            lib.oracle_sparse_decode.restype = c.c_int64
            lib.oracle_sparse_decode.argtypes = [c.c_void_p, c.c_int, c.c_int, c.c_int,
                                                 c.c_void_p, c.c_int64, c.c_void_p, c.c_int,
                                                 c.c_float, c.c_void_p, c.c_void_p,
                                                 c.c_void_p, c.c_int, c.c_int]
            lib.oracle_kv_write_rows.restype = c.c_int64
            lib.oracle_kv_write_rows.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_void_p, c.c_void_p,
                                                 c.c_void_p, c.c_int64, c.c_int64]
            lib.oracle_sparse_decode_rows.restype = c.c_int64
            lib.oracle_sparse_decode_rows.argtypes = [c.c_void_p, c.c_int, c.c_int, c.c_int,
                                                      c.c_void_p, c.c_int64, c.c_int64, c.c_void_p, c.c_int,
                                                      c.c_float, c.c_void_p, c.c_void_p,
                                                      c.c_void_p, c.c_int, c.c_int]
            lib.oracle_double_to_bf16.restype = c.c_uint16
            lib.oracle_double_to_bf16.argtypes = [c.c_double]
            lib.oracle_gather_upconvert.restype = c.c_int64
            lib.oracle_gather_upconvert.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_void_p, c.c_int64,
                                                    c.c_int, c.c_void_p]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _u16(x) -> np.ndarray:
    """bf16 data as raw uint16 bits (accepts a torch bf16 tensor or a uint16 array)."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def e4m3_decode(b: int) -> float:
    return _load().oracle_e4m3_decode(int(b) & 0xFF)


def e4m3_decode_table() -> np.ndarray:
    """Value of each of the 256 codes, float64."""
    return np.array([e4m3_decode(b) for b in range(256)], dtype=np.float64)


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def e4m3_encode_bit_range(lo: int, hi: int, n_threads: int | None = None) -> np.ndarray:
    """Codes of every fp32 bit pattern u in [lo, hi)."""
    out = np.empty(hi - lo, dtype=np.uint8)
    _load().oracle_e4m3_encode_bit_range(lo, hi, _ptr(out), n_threads or default_threads())
    return out


def kv_write(cache: np.ndarray, slot_idx, latent, rope, reserved_slot: int = 0) -> int:
    """Write rows into ``cache`` (uint8 [num_slots, 656] or [num_slots, 528] for
    NoPE-only rows; modified in place).

    latent: bf16 [n, 512]; rope: bf16 [n, 64] or None (NoPE; required for 528-byte
    rows). Returns the number of rows dropped for an out-of-range slot.
    """
    assert cache.dtype == np.uint8 and cache.ndim == 2 and cache.shape[1] in (ROW_BYTES, ROW_BYTES_NOPE)
    assert rope is None or cache.shape[1] == ROW_BYTES
    assert cache.flags.c_contiguous
    slots = np.ascontiguousarray(np.asarray(slot_idx, dtype=np.int64))
    lat = _u16(latent)
    n = slots.shape[0]
    assert lat.size == n * 512
    rp = None
    if rope is not None:
        rp = _u16(rope)
        assert rp.size == n * 64
    return int(_load().oracle_kv_write_rows(_ptr(cache), cache.shape[0], cache.shape[1], _ptr(slots), _ptr(lat),
                                            _ptr(rp) if rp is not None else None, n, reserved_slot))


def sparse_decode(q, cache: np.ndarray, topk, sm_scale: float, tokens=None,
                  n_threads: int | None = None):
    """Float64 sparse decode. q: bf16 [T, H, d_qk] (d_qk 576 or 512); topk int32 [T, W].

    Returns (out float64 [T, H, 512], lse float64 [T, H], n_out_of_range). When
    ``tokens`` is given only those token rows are computed (the others stay NaN).
    """
    qu = _u16(q)
    if hasattr(q, "shape"):
        T, H, d_qk = (int(s) for s in q.shape)
    assert d_qk in (512, 576)
    tk = np.ascontiguousarray(np.asarray(topk, dtype=np.int32))
    assert tk.shape[0] == T
    W = tk.shape[1]
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous and cache.shape[1] in (ROW_BYTES, ROW_BYTES_NOPE)
    assert cache.shape[1] == ROW_BYTES or d_qk == 512
    out = np.full((T, H, 512), np.nan, dtype=np.float64)
    lse = np.full((T, H), np.nan, dtype=np.float64)
    tok = None
    n_tok = 0
    if tokens is not None:
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        n_tok = tok.size
    bad = _load().oracle_sparse_decode_rows(_ptr(qu), T, H, d_qk, _ptr(cache), cache.shape[0], cache.shape[1],
                                            _ptr(tk), W, float(sm_scale), _ptr(out), _ptr(lse),
                                            _ptr(tok) if tok is not None else None, n_tok,
                                            n_threads or default_threads())
    return out, lse, int(bad)


def paged_to_physical(topk_logical, block_table, page_size: int, token_seq=None):
    """Physical slots of a top-k list given as sequence positions (vLLM PR #55277,
    Purpose item 2: the sparse top-k entries are read through block tables).

    topk_logical: int32 [T, W], -1 (any negative) = absent. block_table: int32
    [n_seq, max_pages], the physical page of each logical page; a negative entry
    is an unassigned page. token_seq: int32 [T], the block-table row of each token
    (None: row 0 for every token). Position p of token t maps to slot
    block_table[seq, p // page_size] * page_size + p % page_size. Returns (int32
    [T, W] physical slots with -1 where absent, number of positions past the end
    of the table, which are absent too).
    """
    lg = np.asarray(topk_logical, dtype=np.int64)
    bt = np.asarray(block_table, dtype=np.int64)
    if bt.ndim == 1:
        bt = bt[None, :]
    T, W = lg.shape
    seq = np.zeros(T, dtype=np.int64) if token_seq is None else np.asarray(token_seq, dtype=np.int64)
    out = np.full((T, W), -1, dtype=np.int64)
    bad = 0
    for t in range(T):
        row = bt[seq[t]]
        for j in range(W):
            p = lg[t, j]
            if p < 0:
                continue
            page = p // page_size
            if page >= row.shape[0]:
                bad += 1
                continue
            phys_page = row[page]
            if phys_page < 0:
                continue
            out[t, j] = phys_page * page_size + p % page_size
    return out.astype(np.int32), bad


def double_to_bf16(x: float) -> int:
    """BF16 bits of the value nearest to x (ties to even); NaN -> 0x7FC0."""
    return int(_load().oracle_double_to_bf16(float(x)))


def gather_upconvert(cache: np.ndarray, slots, pe_dim: int):
    """Rows of ``cache`` at ``slots`` (int32 [n]) widened to BF16 [n, 576] (uint16
    bits): the latent as the BF16 nearest to e4m3 * scale, then the RoPE tail
    (pe_dim 64) or zeros (pe_dim 0). Absent slots (<= 0 or >= num_slots) give
    zero rows. Returns (out, number of slots >= num_slots).
    """
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous and cache.shape[1] in (ROW_BYTES, ROW_BYTES_NOPE)
    assert pe_dim in (0, 64) and (cache.shape[1] == ROW_BYTES or pe_dim == 0)
    sl = np.ascontiguousarray(np.asarray(slots, dtype=np.int32))
    out = np.empty((sl.size, 576), dtype=np.uint16)
    bad = _load().oracle_gather_upconvert(_ptr(cache), cache.shape[0], cache.shape[1], _ptr(sl), sl.size,
                                          pe_dim, _ptr(out))
    return out, int(bad)
