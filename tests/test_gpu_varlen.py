"""GPU parity of mla_decode_varlen (a verify step of its own length per
request) against the oracle's varlen decode: the folded-tile kernel at 16
and 32 rows, the cluster kernel at 64, two row groups, an fp8 pool, requests
shorter than their verify step, and several CTA counts. Bars as mla_decode's."""
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


def _check(out, lse, ref_o, ref_l, kind, what):
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    tol = (1e-2 + 2e-2 * np.abs(ref_o)) if kind == 0 else 5e-2
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    assert np.all(np.abs(o - ref_o) <= tol), f"{what}: max|d|={np.abs(o - ref_o).max():.3e}"
    ninf = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(l), ninf), f"{what}: -inf pattern of lse"
    if (~ninf).any():
        assert np.abs(l[~ninf] - ref_l[~ninf]).max() <= (1e-3 if kind == 0 else 5e-2), f"{what}: lse"
    assert np.all(o[ninf] == 0), f"{what}: rows with no visible token must be 0"


CASES = [
    # (Hq, verify lengths, page size, kind, num_ctas)
    (8, [1, 2, 2, 1, 2, 1, 1], 16, 0, 0),    # folded tiles, 16 rows
    (16, [2, 1, 1, 2, 2, 1, 2], 64, 0, 5),   # folded tiles, 32 rows
    (16, [4, 1, 3, 2, 4, 1, 2], 16, 0, 0),   # folded tiles, 64 rows
    (16, [4, 1, 3, 2, 4, 1, 2], 8, 0, 9),    # folded tiles, 64 rows, requests cut across workers
    (16, [6, 1, 5, 2, 3, 6, 1], 16, 0, 7),   # 96 rows: two row groups sharing each tile (a CTA pair)
    (16, [8, 1, 7, 3, 8, 5, 8], 16, 0, 0),   # 1 + 7 drafts: 128 rows, one cache read per request
    (16, [8, 2, 8, 1, 6, 8, 4], 64, 0, 11),  # the same with 64-token pages, requests cut across pairs
    (16, [3, 4, 1, 2, 4, 2, 1], 64, 1, 0),   # fp8 pool, 64 rows
]


@pytest.mark.parametrize("Hq,qlens,page_size,kind,num_ctas", CASES)
def test_decode_varlen_matches_the_oracle(Hq, qlens, page_size, kind, num_ctas):
    sl = [700, 2, 1500, 0, 257, 3, 64 * 5 + 1]   # requests shorter than their step, and an empty one
    assert len(qlens) == len(sl)  # one verify length per request (checked before any device indexing)
    qmax = max(qlens)
    wl = W.make("varlen", B=len(sl), Hq=Hq, Qt=qmax, page_size=page_size, seq_lens=sl, kind=kind,
                write_all=(kind == 1), seed=300 + Hq + page_size + kind, device=DEV)
    m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
    cu = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    R = int(cu[-1])
    # request b's queries: the first q_len_b of its uniform-length rows
    pick = torch.tensor([b * qmax + t for b, q in enumerate(qlens) for t in range(q)], dtype=torch.int64, device=DEV)
    q_lat = wl.q_lat[pick].contiguous()
    q_pe = wl.q_pe[pick].contiguous()
    out = torch.empty((R, Hq, 512), dtype=torch.float32, device=DEV)
    lse = torch.empty((R, Hq), dtype=torch.float32, device=DEV)
    ws = torch.empty((m.mla_decode_workspace_bytes(wl.B, qmax, Hq, num_ctas),), dtype=torch.uint8, device=DEV)
    m.mla_decode_varlen(q_lat, q_pe, wl.pool, wl.kind, wl.page_size, wl.block_table, wl.seq_lens,
                        torch.from_numpy(cu).to(DEV), qmax, wl.scale, out, lse, ws, num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert m.device_status(ws) == 0
    c = W.compact(wl, range(wl.B))
    ref_o, ref_l = oracle.decode_varlen(q_lat.cpu(), q_pe.cpu(), c["pool"], wl.kind, wl.page_size, c["block_table"],
                                        c["seq_lens"], cu, Hq, wl.scale)
    _check(out, lse, ref_o, ref_l, kind, f"Hq={Hq} qlens={qlens} ps={page_size} kind={kind}")


def test_uniform_lengths_match_mla_decode_bitwise():
    sl = [900, 0, 3000, 1, 257]
    wl = W.make("varlen_u", B=len(sl), Hq=16, Qt=2, page_size=16, seq_lens=sl, seed=311, device=DEV)
    m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
    out1, lse1, ws = m.decode(wl.q_lat, wl.q_pe, wl.pool, wl.kind, wl.page_size, wl.block_table, wl.seq_lens,
                              wl.Qt, wl.scale, out_dtype=torch.float32)
    cu = torch.arange(0, 2 * wl.B + 1, 2, dtype=torch.int32, device=DEV)
    out2, lse2 = torch.empty_like(out1), torch.empty_like(lse1)
    m.mla_decode_varlen(wl.q_lat, wl.q_pe, wl.pool, wl.kind, wl.page_size, wl.block_table, wl.seq_lens, cu, 2,
                        wl.scale, out2, lse2, ws)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_verify_workload_sampled():
    """The bench's verify workload at full size: the MTP pool above the int32
    wrap, 128 requests with verify lengths U{1..4}, one mla_decode_varlen call
    as the bench times it; sampled requests (empty and one-token ones, the
    longest, the one holding the pool's last page) against the oracle."""
    import bench

    wl = W.CONFIGS["mtp"](device=DEV)
    qlens = bench.verify_qlens(wl.B)
    sl = wl.seq_lens.cpu().numpy()
    zero_one = [int(i) for i in np.nonzero(sl <= 1)[0]][:3]
    last = int(np.nonzero((wl.block_table == wl.num_slots // wl.page_size - 1).any(dim=1).cpu().numpy())[0][0])
    reqs = sorted(set(zero_one + [int(np.argmax(sl)), last, 7, 60]))
    c = W.compact(wl, reqs)
    pool = c["pool"].copy()
    oracle.cache_write(c["w_latent"], c["w_k_pe"], c["w_slots"], pool, wl.kind)
    sel = [k * wl.Qt + t for k, b in enumerate(reqs) for t in range(int(qlens[b]))]
    cu_c = np.concatenate([[0], np.cumsum([int(qlens[b]) for b in reqs])]).astype(np.int32)
    ref_o, ref_l = oracle.decode_varlen(c["q_lat"][sel], c["q_pe"][sel], pool, wl.kind, wl.page_size,
                                        c["block_table"], c["seq_lens"], cu_c, wl.Hq, wl.scale)

    # the device step: each request's first q_len_b query rows, packed
    pick = torch.tensor([b * wl.Qt + t for b in range(wl.B) for t in range(int(qlens[b]))], dtype=torch.int64,
                        device=DEV)
    q_lat = wl.q_lat[pick].contiguous()
    q_pe = wl.q_pe[pick].contiguous()
    cu = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    total = int(cu[-1])
    m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
    out = torch.empty((total, wl.Hq, 512), dtype=torch.float32, device=DEV)
    lse = torch.empty((total, wl.Hq), dtype=torch.float32, device=DEV)
    ws = torch.empty(m.mla_decode_workspace_bytes(wl.B, wl.Qt, wl.Hq, 0), dtype=torch.uint8, device=DEV)
    m.mla_decode_varlen(q_lat, q_pe, wl.pool, wl.kind, wl.page_size, wl.block_table, wl.seq_lens,
                        torch.from_numpy(cu).to(DEV), wl.Qt, wl.scale, out, lse, ws)
    torch.cuda.synchronize()
    assert m.device_status(ws) == 0
    rows = [int(cu[b]) + t for b in reqs for t in range(int(qlens[b]))]
    _check(out[rows], lse[rows], ref_o, ref_l, wl.kind, "verify workload")
