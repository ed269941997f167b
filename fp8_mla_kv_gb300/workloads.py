"""Seeded synthetic inputs for the FP8 MLA KV writer and the sparse top-k decode.

This module only draws random inputs with the shapes, value distributions and
index structure of the workloads the pages describe (GLM-5.3-Flash-shaped NoPE
decode with a 2,176-wide top-k buffer, DeepSeek-style RoPE rows, prefill-shaped
causal top-k through a block table, padded writer batches aimed at slot 0). It
holds none of the method's arithmetic: no quantisation, no attention. Both the
CUDA path and the CPU oracle consume what it produces.

Every tensor is drawn from its own ``torch.Generator`` stream, seeded from the
workload seed and the tensor's name, on the CPU, so the same inputs come out on
any machine with the same PyTorch. bf16 values are N(0, 1) fp32 rounded to
nearest even.
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from typing import List, Optional

import torch

ROW_BYTES = 656
LATENT = 512
ROPE = 64


def _gen(seed: int, name: str) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed((seed * 0x9E3779B1 + zlib.crc32(name.encode())) % (2**63 - 1))
    return g


def _randn_bf16(shape, seed: int, name: str, chunk_rows: int = 1 << 16) -> torch.Tensor:
    """N(0,1) in fp32, rounded to bf16; drawn in row chunks to bound memory."""
    g = _gen(seed, name)
    out = torch.empty(shape, dtype=torch.bfloat16)
    flat = out.view(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        flat[r0:r1] = torch.randn((r1 - r0, flat.shape[1]), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return out


def _outliers_(x: torch.Tensor, seed: int, name: str, frac: float = 0.01, factor: float = 20.0,
               chunk_rows: int = 1 << 16) -> None:
    """Scale a Bernoulli(frac) subset of the values by ``factor`` in place."""
    g = _gen(seed, name + ".outliers")
    flat = x.view(x.shape[0], -1)
    for r0 in range(0, x.shape[0], chunk_rows):
        r1 = min(x.shape[0], r0 + chunk_rows)
        m = torch.rand((r1 - r0, flat.shape[1]), generator=g) < frac
        blk = flat[r0:r1].float()
        blk[m] *= factor
        flat[r0:r1] = blk.to(torch.bfloat16)


def _distinct_slots(k: int, lo: int, hi: int, g: torch.Generator) -> torch.Tensor:
    """k distinct slots drawn uniformly from [lo, hi)."""
    n = hi - lo
    assert k <= n
    if k * 8 < n:
        # rejection sampling keeps this O(k) for large caches
        picked = torch.unique(torch.randint(lo, hi, (2 * k + 16,), generator=g))
        while picked.numel() < k:
            picked = torch.unique(torch.cat([picked, torch.randint(lo, hi, (2 * k,), generator=g)]))
        perm = torch.randperm(picked.numel(), generator=g)[:k]
        return picked[perm]
    return torch.randperm(n, generator=g)[:k] + lo


@dataclasses.dataclass
class WriteBatch:
    slot_idx: torch.Tensor            # int64 [n]
    latent: torch.Tensor              # bf16 [n, 512]
    rope: Optional[torch.Tensor]      # bf16 [n, 64] or None (NoPE)
    label: str = ""


@dataclasses.dataclass
class DecodeBatch:
    q: torch.Tensor                   # bf16 [T, H, d_qk]
    topk: torch.Tensor                # int32 [T, W]
    sm_scale: float
    label: str = ""

    @property
    def T(self) -> int:
        return int(self.q.shape[0])

    @property
    def H(self) -> int:
        return int(self.q.shape[1])

    @property
    def d_qk(self) -> int:
        return int(self.q.shape[2])

    @property
    def W(self) -> int:
        return int(self.topk.shape[1])


@dataclasses.dataclass
class Workload:
    name: str
    num_slots: int
    slot0_byte: int                   # initial value of every byte of the cache (slot 0 included)
    fill: Optional[WriteBatch]        # rows written before anything else (cache contents)
    writes: List[WriteBatch]          # writer calls of the workload itself
    decode: Optional[DecodeBatch]
    description: str = ""
    block_table: Optional[torch.Tensor] = None   # C4 only: physical page of each logical page
    topk_logical: Optional[torch.Tensor] = None  # C4 only: the decode's top-k as sequence positions (-1 pad)
    page_size: int = 0                           # C4 only: slots per page

    def cache_bytes(self) -> int:
        return self.num_slots * ROW_BYTES


def _fill_all(num_slots: int, seed: int, nope: bool, outliers: bool) -> WriteBatch:
    n = num_slots - 1
    slots = torch.arange(1, num_slots, dtype=torch.int64)
    lat = _randn_bf16((n, LATENT), seed, "fill.latent")
    rope = None if nope else _randn_bf16((n, ROPE), seed, "fill.rope")
    if outliers:
        _outliers_(lat, seed, "fill.latent")
        if rope is not None:
            _outliers_(rope, seed, "fill.rope")
    return WriteBatch(slots, lat, rope, "fill")


# ---------------------------------------------------------------------------
# The five configurations (full size) and reduced variants with the same
# structure (``scale`` < 1 shrinks the cache, the token count and the top-k width
# while keeping several tiles and a ragged tail).
# ---------------------------------------------------------------------------

def tiny(seed: int = 0, T: int = 4, H: int = 16, W: int = 128, n_valid: int = 80,
         num_slots: int = 4096, n_rows: int = 256, n_pad: int = 32,
         scatter_minus_one: bool = False) -> Workload:
    """Tiny end-to-end: 256 rows to distinct random slots in 1..4095 plus 32
    NaN-latent padding rows aimed at slot 0 (shuffled in), then a 4-token decode
    with 80 present entries out of 128 (rest -1)."""
    g = _gen(seed, "tiny.slots")
    slots = _distinct_slots(n_rows, 1, num_slots, g)
    lat = _randn_bf16((n_rows + n_pad, LATENT), seed, "tiny.latent")
    lat[n_rows:] = float("nan")
    rope = _randn_bf16((n_rows + n_pad, ROPE), seed, "tiny.rope")
    all_slots = torch.cat([slots, torch.zeros(n_pad, dtype=torch.int64)])
    order = torch.randperm(n_rows + n_pad, generator=_gen(seed, "tiny.order"))
    wb = WriteBatch(all_slots[order].contiguous(), lat[order].contiguous(), rope[order].contiguous(), "tiny")
    q = _randn_bf16((T, H, LATENT + ROPE), seed, "tiny.q")
    gt = _gen(seed, "tiny.topk")
    topk = torch.full((T, W), -1, dtype=torch.int32)
    for t in range(T):
        pick = slots[torch.randperm(n_rows, generator=gt)[:n_valid]]
        if scatter_minus_one:
            pos = torch.randperm(W, generator=gt)[:n_valid]
            topk[t, pos] = pick.to(torch.int32)
        else:
            topk[t, :n_valid] = pick.to(torch.int32)
    return Workload("tiny", num_slots, 0x00, None, [wb],
                    DecodeBatch(q, topk, 1.0 / math.sqrt(576), "tiny"),
                    "4,096-slot cache; 256 rows + 32 NaN padding rows to slot 0; T=4 H=16 W=128 (80 present)")


def nope(seed: int = 0, num_slots: int = 131072, T: int = 64, H: int = 16, W: int = 2176,
         max_len: int = 2048, slot0_byte: int = 0x00) -> Workload:
    """NoPE decode (qk_rope_head_dim = 0): NoPE rows in every slot 1..N-1, T tokens
    with active length ~ U{1..max_len} of distinct random slots, the rest of the
    W-wide buffer -1."""
    fill = _fill_all(num_slots, seed, nope=True, outliers=False)
    q = _randn_bf16((T, H, LATENT), seed, "nope.q")
    g = _gen(seed, "nope.topk")
    lens = torch.randint(1, max_len + 1, (T,), generator=g)
    topk = torch.full((T, W), -1, dtype=torch.int32)
    for t in range(T):
        n = int(lens[t])
        topk[t, :n] = _distinct_slots(n, 1, num_slots, g).to(torch.int32)
    return Workload("nope", num_slots, slot0_byte, fill, [],
                    DecodeBatch(q, topk, 1.0 / math.sqrt(512), "nope"),
                    f"{num_slots}-slot NoPE cache; T={T} H={H} d_qk=512 W={W}, lengths U(1..{max_len})")


def rope(seed: int = 0, num_slots: int = 1048576, T: int = 128, H: int = 64, W: int = 2048) -> Workload:
    """RoPE decode with outliers: latent and rope N(0,1) with 1% of values x20;
    every top-k entry a distinct present slot; sm_scale = 1/sqrt(192)."""
    fill = _fill_all(num_slots, seed, nope=False, outliers=True)
    q = _randn_bf16((T, H, LATENT + ROPE), seed, "rope.q")
    g = _gen(seed, "rope.topk")
    topk = torch.stack([_distinct_slots(W, 1, num_slots, g) for _ in range(T)]).to(torch.int32)
    return Workload("rope", num_slots, 0x00, fill, [],
                    DecodeBatch(q, topk, 1.0 / math.sqrt(192), "rope"),
                    f"{num_slots}-slot RoPE cache with 1% x20 outliers; T={T} H={H} W={W} all present")


def prefill(seed: int = 0, num_pages: int = 1024, page: int = 64, T: int = 1024, H: int = 16,
            W: int = 2048) -> Workload:
    """Prefill-shaped sparse attention: one T-token sequence laid out through a
    random block table (physical pages drawn from 1..num_pages-1, page 0 holds the
    reserved slot); query row i selects min(i+1, W) distinct positions <= i and
    pads the rest with -1. Slot 0 is 0xFF."""
    num_slots = num_pages * page
    fill = _fill_all(num_slots, seed, nope=False, outliers=False)
    g = _gen(seed, "prefill.table")
    n_logical = (T + page - 1) // page
    table = (torch.randperm(num_pages - 1, generator=g)[:n_logical] + 1).to(torch.int64)
    pos = torch.arange(T, dtype=torch.int64)
    phys = table[pos // page] * page + pos % page
    q = _randn_bf16((T, H, LATENT + ROPE), seed, "prefill.q")
    topk = torch.full((T, W), -1, dtype=torch.int32)
    logical = torch.full((T, W), -1, dtype=torch.int32)
    for i in range(T):
        k = min(i + 1, W)
        chosen = torch.randperm(i + 1, generator=g)[:k]
        topk[i, :k] = phys[chosen].to(torch.int32)
        logical[i, :k] = chosen.to(torch.int32)
    return Workload("prefill", num_slots, 0xFF, fill, [],
                    DecodeBatch(q, topk, 1.0 / math.sqrt(576), "prefill"),
                    f"{num_slots}-slot cache in {num_pages} pages of {page}; T={T} causal rows; slot 0 = 0xFF",
                    block_table=table, topk_logical=logical, page_size=page)


def sweep(seed: int = 0, num_slots: int = 1048576, sizes=(1, 64, 1024, 8192), T: int = 256,
          H: int = 16, W: int = 2048, pad_frac: float = 0.25) -> Workload:
    """Writer sweep plus saturated decode: the cache is filled, then writer calls
    of each size with every row valid and again with a random quarter aimed at
    slot 0; then a T-token decode with every entry a distinct present slot."""
    fill = _fill_all(num_slots, seed, nope=False, outliers=False)
    writes = []
    for n in sizes:
        for padded in (False, True):
            tag = f"sweep.{n}.{'pad' if padded else 'valid'}"
            g = _gen(seed, tag)
            slots = _distinct_slots(n, 1, num_slots, g)
            if padded:
                m = torch.rand(n, generator=g) < pad_frac
                slots = torch.where(m, torch.zeros_like(slots), slots)
            lat = _randn_bf16((n, LATENT), seed, tag + ".latent")
            rp = _randn_bf16((n, ROPE), seed, tag + ".rope")
            writes.append(WriteBatch(slots, lat, rp, tag))
    q = _randn_bf16((T, H, LATENT + ROPE), seed, "sweep.q")
    g = _gen(seed, "sweep.topk")
    topk = torch.stack([_distinct_slots(W, 1, num_slots, g) for _ in range(T)]).to(torch.int32)
    return Workload("sweep", num_slots, 0x00, fill, writes,
                    DecodeBatch(q, topk, 1.0 / math.sqrt(576), "sweep"),
                    f"{num_slots}-slot cache; writer sizes {list(sizes)} valid and {int(pad_frac*100)}% padded; "
                    f"decode T={T} H={H} W={W} all present")


def by_name(name: str, **kw) -> Workload:
    return {"tiny": tiny, "nope": nope, "rope": rope, "prefill": prefill, "sweep": sweep}[name](**kw)


# Reduced variants: same structure, sizes the oracle finishes in seconds.
SMALL = {
    "tiny": dict(),
    "nope": dict(num_slots=8192, T=6, W=544, max_len=512),
    "rope": dict(num_slots=16384, T=3, H=64, W=512),
    "prefill": dict(num_pages=64, page=64, T=80, W=64),
    "sweep": dict(num_slots=16384, sizes=(1, 64, 1024), T=4, W=256),
}


def small(name: str, seed: int = 0) -> Workload:
    return by_name(name, seed=seed, **SMALL[name])
