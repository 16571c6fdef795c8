"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars: cache writes and indexing bit-exact; decode outputs within
|d| <= 1e-2 + 2e-2 |ref| per element and LSE within 1e-3 (bf16 cache);
|d| <= 5e-2 (outputs and LSE) for fp8_ds_mla caches against the oracle run on
the same (dequantised) cache. Inputs are seeded (mla_latent_kv_cache_gb300.workloads);
pools start as NaN sentinels so a read of a wrong slot shows up.
"""
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


def check_decode(out, lse, ref_o, ref_l, rows, kind=0, what=""):
    o = out.float().cpu().numpy()[rows].astype(np.float64)
    l = lse.cpu().numpy()[rows].astype(np.float64)
    assert o.size > 0
    if kind == 0:
        excess = np.abs(o - ref_o) - (1e-2 + 2e-2 * np.abs(ref_o))
    else:
        excess = np.abs(o - ref_o) - 5e-2
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    assert excess.max() <= 0, f"{what}: max|d|={np.abs(o - ref_o).max():.3e}"
    ninf = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(l), ninf), f"{what}: -inf pattern of lse"
    if (~ninf).any():
        # fp8 pools: the dequantised rows reach the MMA rounded to bf16 (f16 up
        # to 64 rows), which moves every score (and so the LSE) by up to ~1e-2
        # on short requests
        lse_tol = 1e-3 if kind == 0 else 5e-2
        assert np.abs(l[~ninf] - ref_l[~ninf]).max() <= lse_tol, \
            f"{what}: lse off by {np.abs(l[~ninf] - ref_l[~ninf]).max():.3e}"
    assert np.all(o[ninf] == 0), f"{what}: rows with no visible token must be 0"


def run_step(wl, out_dtype=torch.float32, num_ctas=0):
    """The step on the device: write the new rows, then decode."""
    m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
    out, lse, ws = m.decode(wl.q_lat, wl.q_pe, wl.pool, wl.kind, wl.page_size, wl.block_table, wl.seq_lens, wl.Qt,
                            wl.scale, out_dtype=out_dtype, num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert m.device_status(ws) == 0
    return out, lse


def oracle_step(wl, reqs):
    """The same step on the host, restricted to requests `reqs` (call before
    the device step: it reads the pool's state before the writes)."""
    c = W.compact(wl, reqs)
    pool = c["pool"].copy()
    oracle.cache_write(c["w_latent"], c["w_k_pe"], c["w_slots"], pool, wl.kind)
    o, l = oracle.decode(c["q_lat"], c["q_pe"], pool, wl.kind, wl.page_size, c["block_table"], c["seq_lens"],
                         len(reqs), wl.Qt, wl.Hq, wl.scale)
    return o, l, c["rows"]


# ---------------------------------------------------------------- cache write

def _write_inputs(T, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    lat = (torch.randn(T, 512, generator=g, device=DEV) *
           torch.exp(torch.randn(T, 1, generator=g, device=DEV))).to(torch.bfloat16)
    kpe = torch.randn(T, 64, generator=g, device=DEV).to(torch.bfloat16)
    return lat, kpe


@pytest.mark.parametrize("kind", [0, 1])
def test_cache_write_bit_exact_incl_high_slots(kind):
    rb = W.ROW_BYTES[kind]
    wrap = (2 ** 31) // (576 if kind == 0 else 656)   # element / byte offset wrap of a 32-bit index
    num_slots = wrap + 5000
    pool = torch.full((num_slots, rb), 0xA5, dtype=torch.uint8, device=DEV)
    T = 3000
    rng = np.random.default_rng(kind)
    slots = np.concatenate([rng.choice(wrap - 100, 1000, replace=False),
                            wrap - 50 + rng.choice(5049, 1998, replace=False),
                            [num_slots - 1, -1]]).astype(np.int64)
    lat, kpe = _write_inputs(T, 10 + kind)
    lat[5] = 0                                              # all-zero blocks: scale 1
    kpe[7] = 0
    sm = torch.from_numpy(slots).to(DEV)
    m.mla_cache_write(lat, kpe, sm, pool, kind)
    # strided views (rows of a wider tensor) must give the same bytes
    wide = torch.zeros(T, 640, dtype=torch.bfloat16, device=DEV)
    wide[:, :512] = lat
    wide[:, 576:] = kpe
    pool2 = torch.full_like(pool, 0xA5)
    m.mla_cache_write(wide[:, :512], wide[:, 576:], sm, pool2, kind)
    torch.cuda.synchronize()
    # oracle on a compact copy holding just the written rows
    ok = slots >= 0
    comp = np.full((T, rb), 0xA5, dtype=np.uint8)
    idx = np.full(T, -1, dtype=np.int64)
    idx[ok] = np.arange(T)[ok]
    oracle.cache_write(lat.cpu(), kpe.cpu(), idx, comp, kind)
    got = pool[torch.from_numpy(slots[ok]).to(DEV)].cpu().numpy()
    assert np.array_equal(got, comp[ok])
    assert torch.equal(pool, pool2)
    # untouched rows keep their bytes
    mask = torch.ones(num_slots, dtype=torch.bool, device=DEV)
    mask[torch.from_numpy(slots[ok]).to(DEV)] = False
    assert bool((pool[mask] == 0xA5).all())


@pytest.mark.parametrize("kind", [0, 1])
def test_cache_write_skips_slots_past_the_pool(kind):
    """Slots at or past num_slots are skipped on the device and reported in
    the status word. The pool is a view of the front of a larger allocation,
    so even an unguarded write would land in mapped memory: the test checks
    that the bytes past the pool are unchanged."""
    rb = W.ROW_BYTES[kind]
    n = 64
    big = torch.full((n + 8, rb), 0x5A, dtype=torch.uint8, device=DEV)
    pool = big[:n]
    lat, kpe = _write_inputs(5, 40 + kind)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sm = torch.tensor([3, n, n + 5, -1, n - 1], dtype=torch.int64, device=DEV)
    m.mla_cache_write(lat, kpe, sm, pool, kind, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 2
    assert bool((big[n:] == 0x5A).all())
    ref = np.full((n, rb), 0x5A, dtype=np.uint8)
    oracle.cache_write(lat[[0, 4]].cpu(), kpe[[0, 4]].cpu(), np.array([3, n - 1]), ref, kind)
    assert np.array_equal(pool.cpu().numpy(), ref)
    # in-range slots only: the status word stays clear
    status.zero_()
    m.mla_cache_write(lat[:1], kpe[:1], sm[:1], pool, kind, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_fp8_encoder_on_every_bf16_value():
    """Blocks whose absmax is 448 have scale 1, so codes are the e4m3
    encoding of the bf16 inputs themselves: compare every finite bf16 value
    with |x| <= 448 against the oracle's encoder."""
    allv = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float()
    vals = allv[torch.isfinite(allv) & (allv.abs() <= 448)]
    per = 127
    nb = -(-vals.numel() // per)
    pad = torch.zeros(nb * per)
    pad[:vals.numel()] = vals
    blocks = torch.cat([torch.full((nb, 1), 448.0), pad.view(nb, per)], dim=1)   # [nb, 128]
    nt = -(-nb // 4)
    lat = torch.zeros(nt * 4, 128)
    lat[:nb] = blocks
    lat = lat.view(nt, 512).to(torch.bfloat16)
    kpe = torch.zeros(nt, 64, dtype=torch.bfloat16)
    pool = torch.zeros((nt, 656), dtype=torch.uint8, device=DEV)
    m.mla_cache_write(lat.to(DEV), kpe.to(DEV), torch.arange(nt, device=DEV), pool, 1)
    ref = np.zeros((nt, 656), dtype=np.uint8)
    oracle.cache_write(lat, kpe, np.arange(nt), ref, 1)
    got = pool.cpu().numpy()
    assert np.all(got[:, 512:528].view(np.float32)[:nb // 4] == 1.0)
    assert np.array_equal(got, ref)


# -------------------------------------------------------------------- decode

def test_decode_tiny_all_rows():
    wl = W.tiny(device=DEV)
    o, l, rows = oracle_step(wl, range(wl.B))
    out, lse = run_step(wl)
    check_decode(out, lse, o, l, rows, what="tiny")


@pytest.mark.parametrize("num_ctas", [1, 3, 7, 300])
def test_decode_cta_counts(num_ctas):
    """Any number of CTAs cuts the token stream differently (segments,
    partials, merge) but must give the same result."""
    wl = W.make("cta", B=5, Hq=16, Qt=1, page_size=16, seq_lens=[1, 700, 129, 0, 2000], seed=21, device=DEV)
    o, l, rows = oracle_step(wl, range(wl.B))
    out, lse = run_step(wl, num_ctas=num_ctas)
    check_decode(out, lse, o, l, rows, what=f"ctas={num_ctas}")


@pytest.mark.parametrize("page_size", [1, 8, 16, 32, 64, 96, 784])
def test_decode_page_sizes_ragged(page_size):
    sl = [1, 17, 300, 1000, 129, 784, 785]
    wl = W.make("ps", B=len(sl), Hq=8, Qt=1, page_size=page_size, seq_lens=sl, seed=30 + page_size,
                rms_spread=1.5, device=DEV)
    o, l, rows = oracle_step(wl, range(wl.B))
    out, lse = run_step(wl, out_dtype=torch.bfloat16)
    check_decode(out, lse, o, l, rows, what=f"page_size={page_size}")


@pytest.mark.parametrize("Hq,Qt,num_ctas", [(32, 1, 0), (16, 4, 0), (48, 3, 9), (16, 8, 5), (64, 1, 3)])
def test_bf16_outputs_at_32_to_128_rows(Hq, Qt, num_ctas):
    """bf16 outputs through the drain's paired stores, for whole requests and
    for split ones (partials then the merge), at 32, 64, 48 and 128 rows."""
    sl = [Qt, 64 + Qt, 999, 4096, 130]
    wl = W.make("b16", B=len(sl), Hq=Hq, Qt=Qt, page_size=16, seq_lens=sl, seed=40 + Hq + Qt, device=DEV)
    o, l, rows = oracle_step(wl, range(wl.B))
    out, lse = run_step(wl, out_dtype=torch.bfloat16, num_ctas=num_ctas)
    check_decode(out, lse, o, l, rows, what=f"bf16 out Hq={Hq} Qt={Qt} ctas={num_ctas}")


@pytest.mark.parametrize("kind,Hq,Qt,page_size", [(1, 16, 1, 64), (1, 32, 4, 64), (0, 16, 1, 5), (0, 32, 1, 7)])
def test_bf16_outputs_on_the_cluster_kernel(kind, Hq, Qt, page_size):
    """The same for the cluster kernel's paths: fp8 pools at 16 and 128 rows,
    page sizes that are not a multiple of 8 (load/convert warps)."""
    sl = [Qt, 300, 2500, 70]
    wl = W.make("cb16", B=len(sl), Hq=Hq, Qt=Qt, page_size=page_size, seq_lens=sl, kind=kind, write_all=(kind == 1),
                seed=60 + Hq + page_size, device=DEV)
    o, l, rows = oracle_step(wl, range(wl.B))
    out, lse = run_step(wl, out_dtype=torch.bfloat16, num_ctas=6)
    check_decode(out, lse, o, l, rows, kind=kind, what=f"cluster bf16 out kind={kind} Hq={Hq} ps={page_size}")


@pytest.mark.parametrize("Hq,Qt", [(16, 4), (8, 3), (32, 1), (64, 1), (80, 1), (20, 4), (16, 8), (32, 3), (128, 1),
                                   (48, 3)])
def test_decode_row_shapes_and_causal(Hq, Qt):
    sl = [0, 1, 2, 3, 5, 130, 400]
    wl = W.make("rows", B=len(sl), Hq=Hq, Qt=Qt, page_size=16, seq_lens=sl, seed=40 + Hq + Qt, device=DEV)
    o, l, rows = oracle_step(wl, range(wl.B))
    out, lse = run_step(wl)
    check_decode(out, lse, o, l, rows, what=f"Hq={Hq} Qt={Qt}")


@pytest.mark.parametrize("rows", [16, 32, 64])
@pytest.mark.parametrize("num_ctas", [2, 6, 40, 400])
def test_many_request_boundaries(rows, num_ctas):
    """Short, empty and long requests against few and many clusters: request
    boundaries inside a cluster's range, drains overtaken by one-tile
    segments, clusters with empty ranges, and at 32 and 64 rows the split
    softmax columns (exchanged P blocks, rescale factors and row sums)."""
    rng = np.random.default_rng(100 + rows + num_ctas)
    sl = [int(x) for x in rng.choice([0, 1, 2, 127, 128, 129, 300, 1000, 2500], size=24)]
    Hq, Qt = {16: (16, 1), 32: (8, 4), 64: (16, 4)}[rows]
    wl = W.make("bounds", B=len(sl), Hq=Hq, Qt=Qt, page_size=16, seq_lens=sl, seed=50 + rows + num_ctas,
                device=DEV)
    o, l, rr = oracle_step(wl, range(wl.B))
    out, lse = run_step(wl, num_ctas=num_ctas)
    check_decode(out, lse, o, l, rr, what=f"rows={rows} ctas={num_ctas}")


@pytest.mark.parametrize("num_ctas,page_size,Hq,Qt", [(5, 64, 16, 1), (0, 16, 32, 1), (9, 8, 8, 3), (3, 32, 16, 2)])
def test_fp8_16_and_32_rows_folded(num_ctas, page_size, Hq, Qt):
    """fp8 pools at 1..32 query rows on the folded kernel (codes widened to f16,
    the queries converted to f16 in shared memory), ragged requests, tile and
    page boundaries, requests cut across workers."""
    sl = [0, 1, 64, 65, 127, 300, 900, 2049, 5]
    wl = W.make("fp8s", B=len(sl), Hq=Hq, Qt=Qt, page_size=page_size, seq_lens=sl, kind=W.KIND_FP8, write_all=True,
                seed=91 + num_ctas + page_size + Hq, device=DEV)
    o, l, rr = oracle_step(wl, range(wl.B))
    out, lse = run_step(wl, num_ctas=num_ctas)
    check_decode(out, lse, o, l, rr, kind=1, what=f"fp8 {Hq * Qt} rows ctas={num_ctas}")


@pytest.mark.parametrize("num_ctas,page_size,Hq,Qt", [(4, 64, 64, 1), (0, 64, 64, 1), (7, 16, 16, 4), (40, 8, 64, 1),
                                                     (3, 32, 16, 3)])
def test_fp8_64_rows_boundaries(num_ctas, page_size, Hq, Qt):
    """fp8 pools at 33..64 query rows (folded tiles: TMA-landed codes widened
    in place by the expand warps) with ragged requests, tile and page
    boundaries, requests cut across workers."""
    sl = [0, 1, 64, 65, 127, 300, 900, 2049, 5]
    wl = W.make("fp8b", B=len(sl), Hq=Hq, Qt=Qt, page_size=page_size, seq_lens=sl, kind=W.KIND_FP8, write_all=True,
                seed=77 + num_ctas + page_size, device=DEV)
    o, l, rr = oracle_step(wl, range(wl.B))
    out, lse = run_step(wl, num_ctas=num_ctas)
    check_decode(out, lse, o, l, rr, kind=1, what=f"fp8 ctas={num_ctas}")
    # these rows compute in f16 (the widened codes, the queries, P): well inside
    # the fp8 bar (measured ~2e-3 on outputs and LSE)
    d = out.cpu().numpy()[rr].astype(np.float64) - o
    fin = np.isfinite(l)
    dl = lse.cpu().numpy()[rr].astype(np.float64)[fin] - l[fin]
    assert np.abs(d).max() <= 1e-2 and (dl.size == 0 or np.abs(dl).max() <= 1e-2), (np.abs(d).max(), np.abs(dl).max())


def test_fp8_64_rows_f16_range_flag():
    """The 64-row fp8 path widens codes to f16: a block whose scale passes 146
    (a latent value above ~65,400 in magnitude) sets status bit 4, and the
    same pool without it leaves the word clear."""
    sl = [300, 700]
    for big, want in ((1.0e5, 4), (3.0e4, 0)):
        wl = W.make("fp8r", B=2, Hq=64, Qt=1, page_size=64, seq_lens=sl, kind=W.KIND_FP8, write_all=True, seed=81,
                    device=DEV)
        wl.w_latent[5, 130] = big
        m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
        out, lse, ws = m.decode(wl.q_lat, wl.q_pe, wl.pool, wl.kind, wl.page_size, wl.block_table, wl.seq_lens,
                                wl.Qt, wl.scale, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert m.device_status(ws) & 4 == want, (big, m.device_status(ws))
        assert m.device_status(ws) & 3 == 0


def test_single_token_is_bit_exact():
    """seq_len 1: softmax weight 1, so the bf16 output is exactly the row."""
    wl = W.make("one", B=6, Hq=16, Qt=1, page_size=16, seq_lens=[1] * 6, seed=50, device=DEV)
    out, lse = run_step(wl, out_dtype=torch.bfloat16)
    rows = wl.pool.view(torch.bfloat16)[W.token_slots(wl.block_table, wl.seq_lens, 16)]
    assert torch.equal(out, rows[:, None, :512].expand(-1, 16, -1))


def test_peaked_attention():
    """One token per request holds (a multiple of) the query, so the output
    is close to that token's row rather than an average near zero."""
    wl = W.make("peak", B=3, Hq=16, Qt=1, page_size=64, seq_lens=[300, 5000, 1200], seed=60, device=DEV)
    slots = W.token_slots(wl.block_table, wl.seq_lens, 64)
    pv = wl.pool.view(torch.bfloat16)
    start = 0
    for b, T in enumerate(wl.seq_lens.tolist()):
        tgt = slots[start + T // 3]
        pv[tgt, :512] = (wl.q_lat[b, 0].float() * 0.25).to(torch.bfloat16)
        start += T
    o, l, rows = oracle_step(wl, range(wl.B))
    out, lse = run_step(wl)
    check_decode(out, lse, o, l, rows, what="peaked")
    assert np.abs(o[:, 0]).max() > 0.3   # the test really is peaked


def test_merge_lse_api():
    g = torch.Generator(device=DEV).manual_seed(70)
    S, N = 7, 333
    po = torch.randn(S, N, 512, generator=g, device=DEV)
    pl = torch.randn(S, N, generator=g, device=DEV) * 5
    pl[:, 3] = -float("inf")
    pl[2:5, 10] = -float("inf")
    out = torch.empty(N, 512, device=DEV)
    lse = torch.empty(N, device=DEV)
    m.mla_merge_lse(po, pl, out, lse)
    out16 = torch.empty(N, 512, dtype=torch.bfloat16, device=DEV)
    m.mla_merge_lse(po, pl, out16)
    torch.cuda.synchronize()
    ro, rl = oracle.merge(po.cpu(), pl.cpu())
    o = out.cpu().double().numpy()
    assert np.abs(o - ro).max() <= 1e-5 * (1 + np.abs(ro).max())
    ln = lse.cpu().double().numpy()
    assert np.array_equal(np.isneginf(ln), np.isneginf(rl))
    fin = np.isfinite(rl)
    assert np.abs(ln[fin] - rl[fin]).max() <= 1e-5
    assert np.all(o[3] == 0)
    # bf16 output: the decode bar (half a bf16 ulp is 2^-9 relative)
    assert (np.abs(out16.cpu().double().numpy() - ro) - (1e-2 + 2e-2 * np.abs(ro))).max() <= 0


# ----------------------------------------------- the five named workloads

def _sample(wl, extra):
    sl = wl.seq_lens.cpu().numpy()
    pick = set(extra)
    pick.add(int(np.argmax(sl)))
    pick.add(int(np.argmin(sl)))
    return sorted(pick)


@pytest.mark.parametrize("name", ["batched", "long", "mtp", "fp8"])
def test_named_workload_sampled(name):
    wl = W.CONFIGS[name](device=DEV)
    sl = wl.seq_lens.cpu().numpy()
    if name == "batched":
        reqs = _sample(wl, [5, 40])
    elif name == "long":
        reqs = [0, 1, 2, 3]
    elif name == "mtp":
        # the empty and one-token requests, and the request holding the last pool slot
        zero_one = [int(i) for i in np.nonzero(sl <= 1)[0]][:6]
        last = int(np.nonzero((wl.block_table == wl.num_slots // wl.page_size - 1).any(dim=1).cpu().numpy())[0][0])
        reqs = sorted(set(zero_one + [last, 3]))
    else:
        reqs = [0, 9, 17, 26, 33, 41, 50, 63]
    o, l, rows = oracle_step(wl, reqs)
    out, lse = run_step(wl)
    check_decode(out, lse, o, l, rows, kind=wl.kind, what=name)
    if name == "mtp":
        assert (wl.block_table[wl.block_table >= 0] >= W.INT32_WRAP_SLOT // 16).all()


@pytest.mark.parametrize("page_size,Hq,Qt,kind,num_ctas", [
    (3, 16, 1, 0, 0), (5, 8, 4, 0, 6), (3, 16, 4, 0, 5), (7, 16, 1, 1, 0), (1, 8, 4, 1, 6), (3, 16, 4, 1, 0)])
def test_load_convert_warps_ragged(page_size, Hq, Qt, kind, num_ctas):
    """Page sizes that are not a multiple of 8 rows go through the load/convert
    warps (a four-slot pair ring): 16, 32 and 64 rows, bf16 and fp8 pools,
    request boundaries inside and across workers."""
    sl = [0, 1, 2, 130, 129, 700, 1500, 257, 5]
    extra = dict(write_all=True) if kind == 1 else {}
    wl = W.make("lsu", B=len(sl), Hq=Hq, Qt=Qt, page_size=page_size, seq_lens=sl, kind=kind,
                seed=70 + page_size + Hq + Qt + kind, device=DEV, **extra)
    o, l, rr = oracle_step(wl, range(wl.B))
    out, lse = run_step(wl, num_ctas=num_ctas)
    check_decode(out, lse, o, l, rr, kind=kind, what=f"page={page_size} rows={Hq * Qt} kind={kind}")
