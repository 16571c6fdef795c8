"""GPU parity for other latent widths ("qwen-mla-vllm" README, "How it works":
per-layer latents of rank 256, 768 or 1792 plus a small rotary tail):
mla_cache_write_latent is a bit copy, mla_decode_latent meets the decode bar
(|d| <= 1e-2 + 2e-2 |ref|, LSE within 1e-3) against oracle.decode_latent,
over ragged requests (empty, one token, page and tile boundaries) with
shuffled pages, split across several workers."""
import numpy as np
import pytest
import torch

import mla_latent_kv_cache_gb300 as m
import oracle
from mla_latent_kv_cache_gb300 import build as mbuild

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mbuild.build()
    m.load()
    torch.cuda.set_device(DEV)
    yield


def bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def case(D, seq, Qt, Hq, ps, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    rng = np.random.default_rng(seed)
    B = len(seq)
    pages = [-(-t // ps) for t in seq]
    nblocks = int(sum(pages) * 1.25) + 2
    perm = rng.permutation(nblocks)
    bt = np.full((B, max(1, max(pages))), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[k:k + n]
        k += n
    rows = torch.randn(nblocks * ps, D + 64, generator=g).to(torch.bfloat16)
    ql = torch.randn(B * Qt, Hq, D, generator=g).to(torch.bfloat16)
    qp = torch.randn(B * Qt, Hq, 64, generator=g).to(torch.bfloat16)
    return rows, ql, qp, bt, np.asarray(seq, np.int32)


@pytest.mark.parametrize("D,Hq,Qt,ps,num_ctas", [(256, 16, 1, 16, 0), (256, 32, 1, 64, 5), (256, 8, 4, 16, 3),
                                                 (768, 16, 1, 16, 0), (768, 8, 2, 64, 7), (512, 16, 1, 16, 0),
                                                 (1792, 16, 1, 16, 0), (1792, 8, 2, 64, 6), (1792, 4, 1, 8, 2)])
def test_decode_latent_matches_oracle(D, Hq, Qt, ps, num_ctas):
    seq = [0, 1, 63, 64, 65, 700, 3000, 129]
    rows, ql, qp, bt, sl = case(D, seq, Qt, Hq, ps, seed=D + Hq + ps)
    # the pool is written by the cache-write kernel, row by row
    pool = torch.full((rows.shape[0], 2 * (D + 64)), 0xFF, dtype=torch.uint8, device=DEV)
    slots = torch.arange(rows.shape[0], dtype=torch.int64, device=DEV)
    lat = rows[:, :D].contiguous().to(DEV)
    kpe = rows[:, D:].contiguous().to(DEV)
    m.mla_cache_write_latent(lat, kpe, slots, pool, D)
    torch.cuda.synchronize()
    assert np.array_equal(pool.cpu().numpy().view(np.uint16), bits(rows))
    out = torch.empty((len(seq) * Qt, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((len(seq) * Qt, Hq), dtype=torch.float32, device=DEV)
    ws = torch.empty(m.mla_decode_latent_workspace_bytes(len(seq), Qt, Hq, D, num_ctas), dtype=torch.uint8,
                     device=DEV)
    scale = 1.0 / np.sqrt(192)
    m.mla_decode_latent(ql.to(DEV), qp.to(DEV), pool, D, ps, torch.from_numpy(bt).to(DEV),
                        torch.from_numpy(sl).to(DEV), Qt, scale, out, lse, ws, num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert m.device_status(ws) == 0
    ro, rl = oracle.decode_latent(bits(ql), bits(qp), bits(rows), D, 64, ps, bt, sl, len(seq), Qt, Hq, scale)
    o = out.cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(o - ro) <= 1e-2 + 2e-2 * np.abs(ro)), np.abs(o - ro).max()
    ninf = np.isneginf(rl)
    assert np.array_equal(np.isneginf(l), ninf)
    assert np.abs(l[~ninf] - rl[~ninf]).max() <= 1e-3


def test_unsupported_shapes_are_refused():
    D = 768
    rows, ql, qp, bt, sl = case(D, [100], 1, 32, 16, seed=1)
    pool = torch.zeros((rows.shape[0], 2 * (D + 64)), dtype=torch.uint8, device=DEV)
    out = torch.empty((1, 32, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((1, 32), dtype=torch.float32, device=DEV)
    ws = torch.empty(m.mla_decode_latent_workspace_bytes(1, 1, 32, D, 0), dtype=torch.uint8, device=DEV)
    with pytest.raises(m.MlaError):
        m.mla_decode_latent(ql.to(DEV), qp.to(DEV), pool, D, 16, torch.from_numpy(bt).to(DEV),
                            torch.from_numpy(sl).to(DEV), 1, 0.1, out, lse, ws)


@pytest.mark.parametrize("D", [256, 768, 1792])
def test_cache_write_latent_skips_slots_past_the_pool(D):
    rb = 2 * (D + 64)
    n = 32
    big = torch.full((n + 4, rb), 0x5A, dtype=torch.uint8, device=DEV)
    pool = big[:n]
    g = torch.Generator(device=DEV).manual_seed(D)
    lat = torch.randn(3, D, generator=g, device=DEV).to(torch.bfloat16)
    kpe = torch.randn(3, 64, generator=g, device=DEV).to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.mla_cache_write_latent(lat, kpe, torch.tensor([5, n, n + 2], dtype=torch.int64, device=DEV), pool, D,
                             status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 2
    assert bool((big[n:] == 0x5A).all())
    want = torch.cat([lat[0], kpe[0]]).cpu().view(torch.int16).numpy().view(np.uint8)
    assert np.array_equal(pool[5].cpu().numpy(), want)
