"""Benchmark of the FP8 MLA KV hot path: one step = the KV writer on a padded
8,192-row batch (a random quarter aimed at slot 0) into a 1,048,576-slot cache,
then the sparse top-k decode of 256 query tokens (16 heads, d_qk 576, top-k
2,048, every entry present) over that cache.

Prints ONE JSON line (rank 0). ``value`` is decode query-tokens/s over whole
steps (writer + decode), all ranks together; the line also carries the decode's
gathered-KV GB/s, the writer's rows/s, the roofline of the dominant kernel
(decode) against the measured HBM peak, the clocks seen during the timed region,
an end-to-end figure through the public API with host buffers, and the CPU
oracle timed on a bounded sample on the host cores.

``--impl reference`` times the CPU oracle (the only reference this method has)
on the same workload, a bounded sample per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fp8_mla_kv_gb300 import workloads  # noqa: E402

METRIC = "sparse-MLA decode query-tokens/s & gathered-KV HBM GB/s; KV-writer rows/s"
UNIT = "query-tokens/s"
WRITE_LABEL = "sweep.8192.pad"
KERNEL_SRC = ["fp8_mla_kv_gb300/csrc/mla_sparse_decode.cu", "fp8_mla_kv_gb300/csrc/mla_device.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_sweep_traffic.txt")


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(values, world, device="cpu"):
    """Element-wise maximum of per-rank totals: the slowest rank sets the job's time."""
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def job_rate(world, units_per_rank, seconds):
    """Whole-job throughput under weak scaling: every rank processes the same units
    in parallel, so the job does world * units_per_rank in the slowest rank's time."""
    return world * units_per_rank / seconds


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_sha() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SRC:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """ncu DRAM bytes per decode launch, if recorded for the current kernel source."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    txt = open(TRAFFIC_FILE).read()
    m_b = re.search(r"traffic_bytes_per_launch\s*=\s*(\d+)", txt)
    m_s = re.search(r"kernel_source_sha\s*=\s*([0-9a-f]+)", txt)
    if m_b and m_s and m_s.group(1) == kernel_sha():
        return int(m_b.group(1))
    return None


class ClockSampler:
    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits", "-lms", "100"]
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            cmd += ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_cpu_baseline(wl, cache_np, wb, seconds: float = 12.0):
    """Oracle decode (float64, all host cores) on a bounded sample of the tokens."""
    import oracle
    db = wl.decode
    cores = oracle.default_threads()
    topk = db.topk.numpy()
    t0 = time.perf_counter()
    oracle.sparse_decode(db.q, cache_np, topk, db.sm_scale, tokens=[0], n_threads=1)
    one = max(time.perf_counter() - t0, 1e-3)          # single-thread seconds per token
    n_tok = int(max(cores, min(db.T, seconds * cores / one)))
    n_tok = min(n_tok, db.T)
    toks = list(range(n_tok))
    t0 = time.perf_counter()
    oracle.sparse_decode(db.q, cache_np, topk, db.sm_scale, tokens=toks, n_threads=cores)
    dt = time.perf_counter() - t0
    res = {"value": n_tok / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": f"float64 oracle decode of {n_tok} of the {db.T} query tokens "
                     f"(H={db.H}, W={db.W}, all present) in {dt:.2f} s on {cores} threads",
           "single_thread": {"value": 1.0 / one, "unit": UNIT, "cores": 1,
                             "sample": "one query token on one thread"}}
    if wb is not None:
        # The oracle writer (one thread) re-writing the step's batch: the same bytes land again.
        t0 = time.perf_counter()
        oracle.kv_write(cache_np, wb.slot_idx.numpy(), wb.latent, wb.rope)
        dtw = time.perf_counter() - t0
        res["writer_single_thread"] = {"value": int(wb.slot_idx.numel()) / dtw, "unit": "rows/s", "cores": 1,
                                       "sample": f"the {int(wb.slot_idx.numel())}-row step batch"}
    return res


WORKLOADS = {
    # default: writer sweep + saturated decode at full size
    "sweep": (lambda: workloads.sweep(),
              "writer sweep + saturated decode: 1,048,576-slot cache of 656-B rows; per step mla_kv_write of "
              "8,192 rows (random 25% aimed at slot 0) then mla_sparse_decode T=256, H=16, d_qk=576, top-k "
              "2,048 all present, sm_scale=1/sqrt(576)"),
    # reduced case of the same kernels for ncu captures (cache 172 MB > L2)
    "sweep-small": (lambda: workloads.sweep(num_slots=262144, T=256),
                    "reduced sweep for profiling: 262,144-slot cache (172 MB); 8,192-row padded write; decode "
                    "T=256, H=16, top-k 2,048 (the full sweep's launch shape)"),
    # reduced RoPE decode for section captures: the full launch shape (512 CTAs)
    # over a 262,144-slot cache (172 MB > L2)
    "rope-small": (lambda: workloads.rope(num_slots=262144),
                   "reduced RoPE decode for profiling: 262,144-slot cache (172 MB), T=128, H=64, d_qk=576, "
                   "top-k 2,048 (the full RoPE launch shape)"),
    "nope": (lambda: workloads.nope(),
             "NoPE decode: 131,072-slot cache, T=64, H=16, d_qk=512, W=2,176, active length U(1..2048)"),
    "rope": (lambda: workloads.rope(),
             "RoPE decode: 1,048,576-slot cache with 1% x20 outliers, T=128, H=64, d_qk=576, top-k 2,048"),
    "prefill": (lambda: workloads.prefill(),
                "prefill-shaped: 65,536-slot paged cache, T=1,024 causal rows, H=16, W=2,048"),
    "tiny": (lambda: workloads.tiny(), "tiny end-to-end: 4,096 slots, 288-row write, T=4, H=16, W=128"),
}


def time_graph(flush, fn, reps=20, calls=1):
    """Seconds per call of fn: `calls` calls captured in one CUDA graph, the graph
    replayed `reps` times (after 3 untimed replays) with L2 flushed before each
    replay, CUDA events around each replay; the median replay divided by calls."""
    fn()
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        for _ in range(calls):
            fn()
    ts = []
    for it in range(reps + 3):
        flush.zero_()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        gr.replay()
        a1.record()
        a1.synchronize()
        if it >= 3:
            ts.append(a0.elapsed_time(a1) * 1e-3 / calls)
    ts.sort()
    del gr
    return ts[len(ts) // 2]


def load_bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def decode_figures(db, num_slots, t_s, row_read=None):
    """Throughput, algorithmic bytes and flops of one decode call of db taking t_s."""
    n_valid = int(((db.topk > 0) & (db.topk < num_slots)).sum())
    rr = row_read or (656 if db.d_qk == 576 else 528)
    gathered = n_valid * rr
    alg = gathered + db.T * db.W * 4 + db.T * db.H * db.d_qk * 2 + db.T * db.H * 512 * 2 + db.T * db.H * 4
    flops = 2.0 * n_valid * db.H * (db.d_qk + 512)
    hbm, _ = load_peaks()
    tf, _ = load_bf16_peak()
    return {"us": t_s * 1e6, "query_tokens_per_s": db.T / t_s, "present_entries": n_valid,
            "gathered_bytes": gathered, "gathered_kv_gbs": gathered / t_s / 1e9,
            "algorithmic_bytes": alg, "algorithmic_gbs": alg / t_s / 1e9, "hbm_frac": alg / t_s / 1e9 / hbm,
            "tflops": flops / t_s / 1e12, "tensor_frac_of_bf16_peak": flops / t_s / 1e12 / tf}


def measure_configs(dev, flush):
    """The four other configurations: decode timed by graph replay with L2 flushed
    before each replay (median), plus the 528-byte rows (NoPE), the paged entry
    point and the token-pair prefill kernel (prefill)."""
    from fp8_mla_kv_gb300 import mlasparse as M
    res = {}
    for name in ("tiny", "nope", "rope", "prefill"):
        wl = workloads.by_name(name)
        cache = build_cache_gpu(wl, dev)
        for w in wl.writes:
            M.mla_kv_write(cache, w.slot_idx.to(dev), w.latent.to(dev), None if w.rope is None else w.rope.to(dev))
        db = wl.decode
        q, tk = db.q.to(dev), db.topk.to(dev)
        out = torch.empty((db.T, db.H, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((db.T, db.H), dtype=torch.float32, device=dev)
        ws = M.alloc_workspace(db.T, db.H, db.W, dev)
        t = time_graph(flush, lambda: M.mla_sparse_decode(q, cache, tk, db.sm_scale, out=out, lse=lse, workspace=ws))
        rec = decode_figures(db, wl.num_slots, t)
        rec["shape"] = {"T": db.T, "H": db.H, "d_qk": db.d_qk, "W": db.W, "num_slots": wl.num_slots}
        if name == "nope":
            c528 = torch.full((wl.num_slots, 528), wl.slot0_byte, dtype=torch.uint8, device=dev)
            f = wl.fill
            M.mla_kv_write(c528, f.slot_idx.to(dev), f.latent.to(dev), None)
            t528 = time_graph(flush, lambda: M.mla_sparse_decode(q, c528, tk, db.sm_scale, out=out, lse=lse,
                                                                  workspace=ws))
            rec["rows_528"] = decode_figures(db, wl.num_slots, t528, row_read=528)
            rec["rows_528"]["cache_bytes"] = int(c528.numel())
            del c528
        if name == "prefill":
            pos, bt = wl.topk_logical.to(dev), wl.block_table.to(torch.int32).to(dev)
            tp = time_graph(flush, lambda: M.mla_sparse_decode_paged(q, cache, pos, bt, wl.page_size, db.sm_scale,
                                                                     out=out, lse=lse, workspace=ws))
            rec["paged"] = decode_figures(db, wl.num_slots, tp)
            # The token-pair prefill kernel on the same batch (physical and paged).
            tk2 = time_graph(flush, lambda: M.mla_sparse_prefill(q, cache, tk, db.sm_scale, out=out, lse=lse))
            rec["prefill_kernel"] = decode_figures(db, wl.num_slots, tk2)
            tk2p = time_graph(flush, lambda: M.mla_sparse_prefill_paged(q, cache, pos, bt, wl.page_size, db.sm_scale,
                                                                         out=out, lse=lse))
            rec["prefill_kernel_paged"] = decode_figures(db, wl.num_slots, tk2p)
        res[name] = rec
        del cache, q, tk, out, lse, ws
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return res


def step_write_batch(wl):
    for w in wl.writes:
        if w.label == WRITE_LABEL:
            return w
    return wl.writes[0] if wl.writes else None


def build_cache_gpu(wl, dev):
    from fp8_mla_kv_gb300 import mlasparse as M
    cache = torch.full((wl.num_slots, 656), wl.slot0_byte, dtype=torch.uint8, device=dev)
    f = wl.fill
    if f is None:
        return cache
    chunk = 1 << 18
    for r0 in range(0, f.slot_idx.shape[0], chunk):
        r1 = min(f.slot_idx.shape[0], r0 + chunk)
        M.mla_kv_write(cache, f.slot_idx[r0:r1].to(dev), f.latent[r0:r1].to(dev),
                       None if f.rope is None else f.rope[r0:r1].to(dev))
    torch.cuda.synchronize()
    return cache


def run_ours(args, rank, world, local_rank):
    from fp8_mla_kv_gb300 import build as B
    from fp8_mla_kv_gb300 import mlasparse as M
    B.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    make_wl, wl_desc = WORKLOADS[args.workload]
    wl = make_wl()
    wb = step_write_batch(wl)
    db = wl.decode
    cache = build_cache_gpu(wl, dev)

    if wb is not None:
        slots_d, lat_d = wb.slot_idx.to(dev), wb.latent.to(dev)
        rope_d = None if wb.rope is None else wb.rope.to(dev)
    q_d, topk_d = db.q.to(dev), db.topk.to(dev)
    out_d = torch.empty((db.T, db.H, 512), dtype=torch.bfloat16, device=dev)
    lse_d = torch.empty((db.T, db.H), dtype=torch.float32, device=dev)
    use_prefill = args.kernel == "prefill"
    ws = None if use_prefill else M.alloc_workspace(db.T, db.H, db.W, dev)
    launches_per_step = (1 if wb is not None else 0) + 1 + (1 if ws is not None else 0)   # per timed step

    def attend(qd, tkd, o, l, w):
        # The attention call of the step: the per-token decode, or the token-pair
        # prefill kernel (--kernel prefill; same result, no workspace).
        if use_prefill:
            M.mla_sparse_prefill(qd, cache, tkd, db.sm_scale, out=o, lse=l)
        else:
            M.mla_sparse_decode(qd, cache, tkd, db.sm_scale, out=o, lse=l, workspace=w)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)

    def write():
        if wb is not None:
            M.mla_kv_write(cache, slots_d, lat_d, rope_d)

    def step():
        write()
        attend(q_d, topk_d, out_d, lse_d, ws)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert M.mla_get_error() == 0
    # The step is captured once as a CUDA graph (writer then decode, as a caller
    # would run it; the decode may start launching while the writer finishes) and
    # replayed; the pages time their kernels by graph replay too. A second timed
    # phase replays the two calls as separate graphs for the writer / decode
    # breakdown and the decode's roofline.
    g_step, g_write, g_decode = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step):
        step()
    if wb is not None:
        with torch.cuda.graph(g_write):
            write()
    with torch.cuda.graph(g_decode):
        attend(q_d, topk_d, out_d, lse_d, ws)
    for _ in range(3):
        flush.zero_()
        g_step.replay()
        flush.zero_()
        if wb is not None:
            g_write.replay()
        g_decode.replay()
    torch.cuda.synchronize()

    K = args.steps
    K2 = min(K, 1000)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K2)]
    sampler = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    wall0 = time.perf_counter()
    for k in range(K):
        flush.zero_()                      # L2 flushed between timed steps (not timed)
        ev[k][0].record()
        g_step.replay()
        ev[k][1].record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    for k in range(K2):
        flush.zero_()
        ev2[k][0].record()
        if wb is not None:
            g_write.replay()
        ev2[k][1].record()
        g_decode.replay()
        ev2[k][2].record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    s_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]
    w_ms = [ev2[k][0].elapsed_time(ev2[k][1]) for k in range(K2)]
    d_ms = [ev2[k][1].elapsed_time(ev2[k][2]) for k in range(K2)]
    assert M.mla_get_error() == 0

    # Writer sweep (every batch of the workload). Two figures per batch: the pages'
    # method (sglang PR #47013, Speed Tests: CUDA-graph replay) with 100 calls in
    # one graph, reported per call (L2 flushed once before each replay, the 100
    # calls then run back to back), and one call per graph replay with L2 flushed.
    sweep = {}
    for w in wl.writes:
        sd, ld = w.slot_idx.to(dev), w.latent.to(dev)
        rd = None if w.rope is None else w.rope.to(dev)
        t_one = time_graph(flush, lambda: M.mla_kv_write(cache, sd, ld, rd), reps=20)
        t_100 = time_graph(flush, lambda: M.mla_kv_write(cache, sd, ld, rd), reps=10, calls=100)
        n_rows, n_wr = int(w.slot_idx.numel()), int((w.slot_idx > 0).sum())
        alg = n_wr * (1024 + (128 if rd is not None else 0) + 656) + n_rows * 8
        sweep[w.label] = {"rows": n_rows, "written": n_wr, "us_per_call_graph100": t_100 * 1e6,
                          "us_single_call": t_one * 1e6, "rows_per_s": n_rows / t_100,
                          "hbm_frac_graph100": alg / t_100 / 1e9 / load_peaks()[0]}
    # Large-N writer points over every slot but the reserved one, in one call:
    # the workload's own fill (sequential slots, re-writing the same rows so the
    # cache contents stay as they are), and the same rows scattered to a random
    # permutation of the slots of a second cache of the same size.
    fill_pt = None
    f = wl.fill
    if f is not None and args.workload == "sweep":
        fs, fl = f.slot_idx.to(dev), f.latent.to(dev)
        fr = None if f.rope is None else f.rope.to(dev)
        n_fill = int(fs.numel())
        fill_alg = n_fill * (1024 + (128 if fr is not None else 0) + 656 + 8)
        t_seq = time_graph(flush, lambda: M.mla_kv_write(cache, fs, fl, fr), reps=5)
        perm = (torch.randperm(n_fill, generator=torch.Generator().manual_seed(11)) + 1).to(torch.int64).to(dev)
        cache2 = torch.zeros_like(cache)
        t_rnd = time_graph(flush, lambda: M.mla_kv_write(cache2, perm, fl, fr), reps=5)
        peak_hbm = load_peaks()[0]
        fill_pt = {
            "sequential": {"rows": n_fill, "us": t_seq * 1e6, "rows_per_s": n_fill / t_seq,
                           "algorithmic_gbs": fill_alg / t_seq / 1e9, "hbm_frac": fill_alg / t_seq / 1e9 / peak_hbm},
            "random": {"rows": n_fill, "us": t_rnd * 1e6, "rows_per_s": n_fill / t_rnd,
                       "algorithmic_gbs": fill_alg / t_rnd / 1e9, "hbm_frac": fill_alg / t_rnd / 1e9 / peak_hbm},
            "algorithmic_bytes": fill_alg,
            "note": "one call over every slot 1..N-1 (sequential slots / a random permutation into a second "
                    "1,048,576-slot cache), CUDA-graph replay, L2 flushed",
        }
        del fs, fl, fr, perm, cache2
    torch.cuda.synchronize()
    assert M.mla_get_error() == 0

    # The widened rows of the path, each timed the same way (graph replay, L2
    # flushed before each replay, median): gather-and-upconvert on the sweep cache.
    widened = {}
    peak_hbm = load_peaks()[0]
    if args.workload == "sweep":
        n_up = 262144
        up_slots = torch.randint(1, wl.num_slots, (n_up,), generator=torch.Generator().manual_seed(7),
                                 dtype=torch.int32).to(dev)
        up_out = torch.empty((n_up, 576), dtype=torch.bfloat16, device=dev)
        t_up = time_graph(flush, lambda: M.mla_gather_upconvert(cache, up_slots, 64, out=up_out))
        up_alg = n_up * (4 + 656 + 576 * 2)
        widened["gather_upconvert"] = {"rows": n_up, "us": t_up * 1e6, "rows_per_s": n_up / t_up,
                                       "algorithmic_bytes": up_alg, "algorithmic_gbs": up_alg / t_up / 1e9,
                                       "hbm_frac": up_alg / t_up / 1e9 / peak_hbm}
        del up_out
    torch.cuda.synchronize()
    assert M.mla_get_error() == 0

    # The other four configurations, measured in the same run with the same method
    # (their own caches, decode graph-replayed, L2 flushed before each replay).
    configs = None
    if args.workload == "sweep" and not args.no_configs:
        configs = measure_configs(dev, flush)
    torch.cuda.synchronize()
    assert M.mla_get_error() == 0

    # End to end through the public API with pinned host buffers: every step's
    # inputs go host -> device and its outputs come back device -> host inside the
    # timed region. Consecutive steps are pipelined, as a serving loop would run
    # them: step k+1's inputs are copied in (one stream) while step k computes
    # (the launching stream) and step k-1's outputs are copied out (a third
    # stream), with two sets of device buffers. No flush between these steps: the
    # 1M-slot cache (688 MB) is larger than L2. One event pair brackets all steps.
    # A step's inputs sit in one pinned host buffer and its outputs in one device
    # buffer (each tensor a 256-byte aligned view), so a step moves them with one
    # copy each way: fewer host-side calls per step in the serving loop.
    w_in = [] if wb is None else [t for t in (wb.slot_idx, wb.latent, wb.rope) if t is not None]
    src_in = w_in + [db.q, db.topk]

    def _layout(tensors):
        offs, off = [], 0
        for t in tensors:
            offs.append(off)
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, off

    def _views(buf, tensors, offs):
        return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for t, o in zip(tensors, offs)]

    in_offs, in_bytes = _layout(src_in)
    h_pack = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    h_in = _views(h_pack, src_in, in_offs)
    for h, t in zip(h_in, src_in):
        h.copy_(t)
    d_pack = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    d_ins = [_views(b, src_in, in_offs) for b in d_pack]
    out_like = [torch.empty((db.T, db.H, 512), dtype=torch.bfloat16), torch.empty((db.T, db.H), dtype=torch.float32)]
    out_offs, out_bytes = _layout(out_like)
    h_opack = [torch.empty(out_bytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
    h_outs = [tuple(_views(b, out_like, out_offs)) for b in h_opack]
    d_opack = [torch.empty(out_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    d_outs = [tuple(_views(b, out_like, out_offs)) for b in d_opack]
    ws2 = [ws, None if ws is None else torch.empty_like(ws)]
    h2d = in_bytes                                 # bytes each step copies in (the packed buffer)
    d2h = out_bytes
    e2e_steps = 0 if args.no_e2e else max(4, min(K, 200))
    xs = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def copy_in(k):
        i = k % 2
        if k >= 2:
            s_in.wait_event(ev_done[i])            # step k-2 no longer reads these buffers
        with torch.cuda.stream(s_in):
            d_pack[i].copy_(h_pack, non_blocking=True)
        ev_in[i].record(s_in)

    def e2e_run(n):
        copy_in(0)
        for k in range(n):
            i = k % 2
            if k + 1 < n:
                copy_in(k + 1)
            xs.wait_event(ev_in[i])
            if k >= 2:
                xs.wait_event(ev_out[i])           # step k-2's outputs have left
            d = d_ins[i]
            if wb is not None:
                M.mla_kv_write(cache, d[0], d[1], d[2] if len(w_in) == 3 else None)
            attend(d[-2], d[-1], d_outs[i][0], d_outs[i][1], ws2[i])
            ev_done[i].record(xs)
            s_out.wait_event(ev_done[i])
            with torch.cuda.stream(s_out):
                h_opack[i].copy_(d_opack[i], non_blocking=True)
            ev_out[i].record(s_out)
        xs.wait_stream(s_out)

    e2e_ms = [float("nan")]
    if e2e_steps:
        e2e_run(3)                                 # warm-up
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(xs)
        e2e_run(e2e_steps)
        e1.record(xs)
        e1.synchronize()
        e2e_ms = [e0.elapsed_time(e1) / e2e_steps] * e2e_steps
        # the pipelined steps computed what the timed graph replays computed
        last = (e2e_steps - 1) % 2
        assert torch.equal(h_outs[last][0].view(torch.int16), out_d.cpu().view(torch.int16))
        assert torch.equal(h_outs[last][1], lse_d.cpu())

    # reduce: max over ranks of the summed device time
    tot = max_over_ranks([sum(s_ms), sum(w_ms), sum(d_ms), sum(e2e_ms)], world, dev)
    step_ms, writer_ms, decode_ms, e2e_tot = (tot[0] / K, tot[1] / K2, tot[2] / K2, tot[3] / len(e2e_ms))

    n_valid = int(((db.topk > 0) & (db.topk < wl.num_slots)).sum())
    row_read = 656 if db.d_qk == 576 else 528
    gathered = n_valid * row_read
    decode_alg = (gathered + db.T * db.W * 4 + db.T * db.H * db.d_qk * 2 + db.T * db.H * 512 * 2
                  + db.T * db.H * 4)
    n_rows = 0 if wb is None else int(wb.slot_idx.numel())
    n_written = 0 if wb is None else int((wb.slot_idx > 0).sum())
    writer_alg = n_written * (1024 + (128 if wb is not None and wb.rope is not None else 0) + 656) + n_rows * 8
    peak, peak_kind = load_peaks()
    achieved = decode_alg / (decode_ms * 1e-3) / 1e9
    traffic = recorded_traffic()

    result = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline and args.workload == "sweep":
            cache_np = cache.cpu().numpy()
            cpu = oracle_cpu_baseline(wl, cache_np, wb, seconds=args.cpu_seconds)
        result = {
            "metric": METRIC,
            "value": job_rate(world, db.T, step_ms * 1e-3),
            "unit": UNIT,
            "n_gpus": world,
            "steps": K,
            "warmup": args.warmup,
            "ms_per_step": step_ms,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "e4m3 cache; bf16 q/out; f16/bf16 tensor-core MMA with fp32 accumulate",
            "data": "synthetic (seeded N(0,1) bf16; no model weights)",
            "config": {
                "workload": wl_desc,
                "T": db.T, "H": db.H, "d_qk": db.d_qk, "topk": db.W, "num_slots": wl.num_slots,
                "present_entries": n_valid,
                "attention_call": "mla_sparse_prefill" if use_prefill else "mla_sparse_decode",
                "writer_rows": n_rows, "writer_rows_written": n_written,
                "l2": "flushed between timed steps (256 MiB write, outside the timed events)",
                "timing": "CUDA-graph replay of the whole step (writer + decode in one graph); CUDA events on "
                          "the launching stream around each step; device time summed over steps; the writer / "
                          "decode split from a second timed phase of separate graphs",
            },
            "decode": {
                "us": decode_ms * 1e3,
                "query_tokens_per_s": job_rate(world, db.T, decode_ms * 1e-3),
                "gathered_kv_gbs": gathered / (decode_ms * 1e-3) / 1e9,
                "gathered_bytes": gathered,
                "nsplit_workspace_bytes": 0 if ws is None else int(ws.numel()),
            },
            "writer_sweep": sweep or None,
            "widened": widened or None,
            "writer_large": fill_pt,
            "configs": configs,
            "writer": None if wb is None else {
                "us": writer_ms * 1e3,
                "rows_per_s": job_rate(world, n_rows, writer_ms * 1e-3),
                "algorithmic_gbs": writer_alg / (writer_ms * 1e-3) / 1e9,
                "hbm_frac": writer_alg / (writer_ms * 1e-3) / 1e9 / peak,
            },
            "roofline": {
                "kernel": "mla_sparse_pair_kernel" if use_prefill else "mla_sparse_decode_kernel (+ split combine)",
                "bound": "hbm",
                "achieved": achieved,
                "peak": peak,
                "unit": "GB/s",
                "frac": achieved / peak,
                "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured" else "fallback 6.8 TB/s",
                "algorithmic_bytes_per_launch": decode_alg,
                "traffic": traffic if args.workload == "sweep" and not use_prefill else None,
            },
            "clocks": clocks,
            "e2e": {
                "value": job_rate(world, db.T, e2e_tot * 1e-3),
                "unit": UNIT,
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "pipelined": "steps overlap: inputs in, compute, outputs out on three streams",
                "ms_per_step": e2e_tot,
            },
            "gpu_launches": K * launches_per_step,
            "cpu_baseline": cpu,
            "wall_s_timed_region": wall,
        }
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return result


def run_reference(args, rank, world):
    """CPU oracle arm: each step writes the 8,192-row batch with the oracle
    writer and decodes a bounded sample of the query tokens with the oracle."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    wl = workloads.sweep()
    wb = next(w for w in wl.writes if w.label == WRITE_LABEL)
    db = wl.decode
    cache = np.full((wl.num_slots, 656), wl.slot0_byte, np.uint8)
    oracle.kv_write(cache, wl.fill.slot_idx.numpy(), wl.fill.latent, wl.fill.rope)
    cores = oracle.default_threads()
    topk = db.topk.numpy()
    per_step = max(1, min(db.T, cores))
    times = []
    for k in range(args.warmup + args.steps):
        toks = [(k * per_step + i) % db.T for i in range(per_step)]
        t0 = time.perf_counter()
        oracle.kv_write(cache, wb.slot_idx.numpy(), wb.latent, wb.rope)
        oracle.sparse_decode(db.q, cache, topk, db.sm_scale, tokens=toks, n_threads=cores)
        dt = time.perf_counter() - t0
        if k >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = per_step * len(times) / total
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": "same as the GPU arm; per step the oracle writes the 8,192-row batch and "
                               f"decodes {per_step} of the 256 query tokens",
                   "T": db.T, "H": db.H, "d_qk": db.d_qk, "topk": db.W, "num_slots": wl.num_slots},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} query tokens + the 8,192-row write per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="sweep")
    ap.add_argument("--kernel", choices=["decode", "prefill"], default="decode",
                    help="attention call of the step: mla_sparse_decode or the token-pair mla_sparse_prefill")
    args = ap.parse_args()
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local_rank)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
