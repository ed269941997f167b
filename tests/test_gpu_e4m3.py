"""The device E4M3 conversion the writer relies on agrees with the oracle codec
on every one of the 2^32 fp32 bit patterns (NaNs included: this fixes the NaN
code the oracle uses), and the pair intrinsic puts its first value in the low byte."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from fp8_mla_kv_gb300 import build as B

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gpu_helpers", "e4m3_cvt.cu")
OUT_DIR = os.path.join(HERE, "gpu_helpers", "_build")


def _helper():
    os.makedirs(OUT_DIR, exist_ok=True)
    so = os.path.join(OUT_DIR, "libe4m3_cvt.so")
    if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(SRC):
        subprocess.run([B.nvcc(), *B.ARCH, "-O3", "-shared", "-Xcompiler", "-fPIC", SRC, "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.e4m3_cvt_range.restype = ctypes.c_int
    lib.e4m3_cvt_range.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p]
    return lib


@pytest.mark.gpu
def test_exhaustive_fp32_to_e4m3_matches_oracle():
    lib = _helper()
    chunk = 1 << 28
    buf = torch.empty(chunk, dtype=torch.uint8, device="cuda:0")
    host = torch.empty(chunk, dtype=torch.uint8, pin_memory=True)
    for lo in range(0, 1 << 32, chunk):
        assert lib.e4m3_cvt_range(lo, chunk, buf.data_ptr()) == 0
        host.copy_(buf)
        got = host.numpy()
        ref = oracle.e4m3_encode_bit_range(lo, lo + chunk)
        bad = np.nonzero(got != ref)[0]
        assert bad.size == 0, [(hex(lo + int(i)), hex(got[i]), hex(ref[i])) for i in bad[:8]]


@pytest.mark.gpu
def test_writer_division_gives_ieee_codes_on_every_bf16_pair():
    src = os.path.join(HERE, "gpu_helpers", "div_check.cu")
    so = os.path.join(OUT_DIR, "libdiv_check.so")
    os.makedirs(OUT_DIR, exist_ok=True)
    subprocess.run([B.nvcc(), *B.ARCH, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC", src, "-o", so], check=True)
    lib = ctypes.CDLL(so)
    counts = (ctypes.c_ulonglong * 2)()
    ex = (ctypes.c_uint32 * 16)()
    assert lib.div_check(counts, ex) == 0
    checked, bad = counts[0], counts[1]
    assert checked > 500_000_000
    assert bad == 0, [(hex(ex[2 * i]), hex(ex[2 * i + 1])) for i in range(min(bad, 8))]
