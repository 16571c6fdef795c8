"""The calls never synchronise, so a serving loop can capture a decode step
(cache write + decode with its programmatic-dependent merge) and the context
gather in a CUDA graph: replaying the graph gives bit-identical results to
the eager calls, for the folded-tile kernel, the cluster kernel and fp8."""
import pytest
import torch

import mla_latent_kv_cache_gb300 as m
from mla_latent_kv_cache_gb300 import build as mbuild
from mla_latent_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mbuild.build()
    m.load()
    torch.cuda.set_device(DEV)
    yield


@pytest.mark.parametrize("shape", [
    dict(Hq=16, Qt=1, page_size=16, kind=0),   # folded tiles, 16 rows
    dict(Hq=16, Qt=2, page_size=64, kind=0),   # folded tiles, 32 rows
    dict(Hq=16, Qt=4, page_size=16, kind=0),   # folded tiles, 64 rows
    dict(Hq=16, Qt=8, page_size=16, kind=0),   # 128 rows: a CTA pair on multicast tiles
    dict(Hq=16, Qt=4, page_size=5, kind=0),    # cluster kernel (load/convert warps), 64 rows
    dict(Hq=64, Qt=1, page_size=64, kind=1),   # fp8 pool
])
def test_decode_step_replays_from_a_cuda_graph(shape):
    sl = [900, 0, 3000, 1, 257]
    kind = shape["kind"]
    wl = W.make("graph", B=len(sl), Hq=shape["Hq"], Qt=shape["Qt"], page_size=shape["page_size"], seq_lens=sl,
                kind=kind, write_all=(kind == 1), seed=123, device=DEV)
    if kind == 1:
        m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
    B, Qt, Hq = wl.B, wl.Qt, wl.Hq
    ws = torch.empty((m.mla_decode_workspace_bytes(B, Qt, Hq),), dtype=torch.uint8, device=DEV)
    out_e = torch.empty((B * Qt, Hq, 512), dtype=torch.bfloat16, device=DEV)
    lse_e = torch.empty((B * Qt, Hq), dtype=torch.float32, device=DEV)
    out_g, lse_g = torch.empty_like(out_e), torch.empty_like(lse_e)

    def step(out, lse, stream=None):
        m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind, stream=stream)
        m.mla_decode(wl.q_lat, wl.q_pe, wl.pool, wl.kind, wl.page_size, wl.block_table, wl.seq_lens, Qt, wl.scale,
                     out, lse, ws, stream=stream)

    step(out_e, lse_e)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(out_g, lse_g, stream=s)
    for _ in range(3):
        out_g.zero_()
        lse_g.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert m.device_status(ws) == 0
    assert torch.equal(out_g, out_e) and torch.equal(lse_g, lse_e)


def test_context_gather_replays_from_a_cuda_graph():
    sl = [40, 0, 300, 77]
    wl = W.make("graphg", B=len(sl), Hq=8, Qt=1, page_size=16, seq_lens=sl, kind=1, write_all=True, seed=124,
                device=DEV)
    m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
    cu = torch.tensor([0, 40, 40, 340, 417], dtype=torch.int32, device=DEV)
    eager = torch.empty((417, 576), dtype=torch.bfloat16, device=DEV)
    m.mla_gather_upconvert(wl.pool, wl.page_size, wl.block_table, cu, eager)
    graphed = torch.zeros_like(eager)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        m.mla_gather_upconvert(wl.pool, wl.page_size, wl.block_table, cu, graphed, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(graphed.view(torch.int16), eager.view(torch.int16))
