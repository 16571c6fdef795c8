"""The softmax -> PV hand-off under issuer skew: a test hook holds one of the
two PV-issuing warps about 20 us after each of its first 32 tiles, so the
softmax warps run up to two tiles ahead of it. The delayed call must finish
with status 0 and give exactly the undelayed call's outputs (the arithmetic
and its order do not depend on timing), and both match the oracle.

Zero queries make every score 0, so no tile after the first rescales O and the
softmax never waits for the lagging issuer's latest product: the skew is as
large as the pipeline allows."""
import numpy as np
import pytest
import torch

import mla_latent_kv_cache_gb300 as m
import oracle
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
    torch.cuda.empty_cache()


CASES = [
    # name, kind, Hq, page size: the folded-tile kernel at 16, 32 and 64
    # query rows, the cluster kernel (fp8 pool) at 16, and its load/convert-warp
    # variants (pages that are not a multiple of 8 rows) at 16 and 32
    ("fold16", W.KIND_BF16, 16, 16),
    ("fold32", W.KIND_BF16, 32, 64),
    ("fold64", W.KIND_BF16, 64, 16),
    ("fold128_pair", W.KIND_BF16, 128, 16),
    ("fold64_fp8", W.KIND_FP8, 64, 64),
    ("cluster16_fp8", W.KIND_FP8, 16, 64),
    ("lsu16", W.KIND_BF16, 16, 3),
    ("lsu32", W.KIND_BF16, 32, 5),
]


@pytest.mark.parametrize("zero_q", [True, False])
@pytest.mark.parametrize("name,kind,Hq,ps", CASES)
def test_lagging_pv_issuer(name, kind, Hq, ps, zero_q):
    sl = [9000, 5000, 130]
    extra = dict(write_all=True) if kind == W.KIND_FP8 else {}
    wl = W.make(name, B=len(sl), Hq=Hq, Qt=1, page_size=ps, seq_lens=sl, kind=kind, seed=300 + Hq + kind,
                device=DEV, **extra)
    if zero_q:
        wl.q_lat.zero_()
        wl.q_pe.zero_()
    c = W.compact(wl, range(wl.B))
    pool = c["pool"].copy()
    oracle.cache_write(c["w_latent"], c["w_k_pe"], c["w_slots"], pool, kind)
    ref_o, ref_l = oracle.decode(c["q_lat"], c["q_pe"], pool, kind, ps, c["block_table"], c["seq_lens"], wl.B,
                                 wl.Qt, wl.Hq, wl.scale)

    m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, kind)
    args = (wl.q_lat, wl.q_pe, wl.pool, kind, ps, wl.block_table, wl.seq_lens, wl.Qt, wl.scale)
    # four workers: each runs dozens of tiles, more than the hook's 32
    out0, lse0, ws0 = m.decode(*args, out_dtype=torch.float32, num_ctas=4)
    torch.cuda.synchronize()
    assert m.device_status(ws0) == 0
    m.test_slow_pv_next_decode()
    out1, lse1, ws1 = m.decode(*args, out_dtype=torch.float32, num_ctas=4)
    torch.cuda.synchronize()
    assert m.device_status(ws1) == 0, m.device_status_words(ws1)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)

    o = out1.cpu().numpy()[c["rows"]].astype(np.float64)
    l = lse1.cpu().numpy()[c["rows"]].astype(np.float64)
    tol = (1e-2 + 2e-2 * np.abs(ref_o)) if kind == W.KIND_BF16 else 5e-2
    assert np.all(np.abs(o - ref_o) <= tol), np.abs(o - ref_o).max()
    assert np.abs(l - ref_l).max() <= (1e-3 if kind == W.KIND_BF16 else 5e-2)
