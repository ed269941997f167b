"""The writer and the decode captured together in one CUDA graph, the way a
serving step replays them: the decode is launched with programmatic stream
serialization behind the writer, so it may start while the writer runs but must
not read the cache before the writer's rows are in it. The rows the writer
stores are poisoned (0xFF: NaN codes and NaN scales) before every replay; the
decode must still give, bit for bit, what it gives when the rows were written
before it by a separate call."""
import numpy as np
import pytest
import torch

from fp8_mla_kv_gb300 import mlasparse as M
from fp8_mla_kv_gb300 import workloads

from _parity import build_both, dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "sweep"])
def test_writer_then_decode_in_one_graph(name):
    # tiny: 4 tokens of 128 positions, one CTA per token; sweep: 200 tokens of
    # 512 positions, cut across CTAs (partials and the merge launch).
    wl = workloads.tiny() if name == "tiny" else workloads.sweep(num_slots=16384, sizes=(1, 64, 1024), T=200, W=512)
    g, c = build_both(wl)
    d = dev()
    db = wl.decode
    last = wl.writes[-1]
    slots = last.slot_idx.to(d)
    lat = last.latent.to(d)
    rope = None if last.rope is None else last.rope.to(d)
    q, topk = db.q.to(d), db.topk.to(d)
    ws = M.alloc_workspace(db.T, db.H, db.W, d)
    ref_out, ref_lse = M.mla_sparse_decode(q, g, topk, db.sm_scale, workspace=ws)
    torch.cuda.synchronize()
    assert M.mla_get_error() == 0
    targets = slots[slots > 0]
    # the decode reads some of the rows the writer stores
    assert np.isin(db.topk.numpy(), targets.cpu().numpy()).any()

    out = torch.empty_like(ref_out)
    lse = torch.empty_like(ref_lse)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        M.mla_kv_write(g, slots, lat, rope)
        M.mla_sparse_decode(q, g, topk, db.sm_scale, out=out, lse=lse, workspace=ws)
    for _ in range(3):
        g[targets] = 0xFF
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert M.mla_get_error() == 0
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
    assert np.array_equal(g.cpu().numpy(), c), "cache after the replays differs from the oracle's"
