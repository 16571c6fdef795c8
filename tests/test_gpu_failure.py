"""Device-side failure path without a GPU fault: a test hook withholds one
hand-off inside the decode kernel, a bounded wait gives up after about a
second, the call's status words say so and where, and the same context then
decodes correctly."""
import numpy as np
import pytest
import torch

import mla_latent_kv_cache_gb300 as m
import oracle
from mla_latent_kv_cache_gb300 import build as mbuild
from mla_latent_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
WAIT_TIMEOUT = 1          # status bit: a bounded wait gave up


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mbuild.build()
    m.load()
    torch.cuda.set_device(DEV)
    yield


@pytest.mark.parametrize("Qt,kind", [(1, 0), (4, 0), (8, 0), (4, 1)])
def test_bounded_wait_reports_and_context_survives(Qt, kind):
    # 16 query rows, 64 (the folded kernel with one O accumulator), 128 (two
    # row groups as a CTA pair sharing multicast tiles), and an fp8 pool at 64
    # rows (expand warps)
    wl = W.make("hold", B=3, Hq=16, Qt=Qt, page_size=16, seq_lens=[700, 1500, 300], seed=91, device=DEV, kind=kind,
                write_all=(kind == 1))
    m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
    m.test_hold_next_decode()
    out, lse, ws = m.decode(wl.q_lat, wl.q_pe, wl.pool, wl.kind, wl.page_size, wl.block_table, wl.seq_lens,
                            wl.Qt, wl.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()  # returns: the kernel left through its abort path
    words = m.device_status_words(ws)
    assert words[0] & WAIT_TIMEOUT, words
    assert words[1] != 0, words  # the wait site (PV issuers' or the last output's, as a rule)
    assert any(w != 0 for w in words[4:12]), words  # a role recorded where it gave up

    # the hook is spent; the same context decodes the same inputs correctly
    c = W.compact(wl, range(wl.B))
    pool = c["pool"].copy()
    oracle.cache_write(c["w_latent"], c["w_k_pe"], c["w_slots"], pool, wl.kind)
    ref_o, ref_l = oracle.decode(c["q_lat"], c["q_pe"], pool, wl.kind, wl.page_size, c["block_table"],
                                 c["seq_lens"], wl.B, wl.Qt, wl.Hq, wl.scale)
    out, lse, ws = m.decode(wl.q_lat, wl.q_pe, wl.pool, wl.kind, wl.page_size, wl.block_table, wl.seq_lens,
                            wl.Qt, wl.scale, out_dtype=torch.float32, workspace=ws)
    torch.cuda.synchronize()
    assert m.device_status(ws) == 0
    o = out.cpu().numpy()[c["rows"]].astype(np.float64)
    tol = (1e-2 + 2e-2 * np.abs(ref_o)) if kind == 0 else 5e-2
    assert np.all(np.abs(o - ref_o) <= tol)
    assert np.abs(lse.cpu().numpy()[c["rows"]] - ref_l).max() <= (1e-3 if kind == 0 else 5e-2)
