"""GPU checks of the guards the decode and gather kernels keep against bad
indexing inputs, which the caller hands over in device memory where the host
cannot look at them without a synchronisation:
- a block-table entry outside the pool (past its end, or negative): the
  decode reads page 0 in its place and sets status bit 2 ("sabi-mla-vllm"
  README, "B300 fix (0.2.0)": the out-of-range access this guards against);
- a sequence longer than its block-table row: the page indices past the row
  count as entries outside the pool (decode: page 0 and bit 2; gather: rows of
  zeros, as for any entry outside the pool);
- per-request verify lengths whose prefix sums pass the query count of the
  call: the sums are clamped to it, so the rows past it are neither read nor
  written.
Every case is laid out so that even an unguarded access would stay inside
memory the test allocated (the tables and the outputs carry spare rows); the
checks are that the kernels flag or skip the bad part, leave the spare rows
as they were, and compute every other row as the oracle does."""
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


def _check(out, lse, ref_o, ref_l, kind, what):
    o = out.float().cpu().numpy().astype(np.float64).reshape(ref_o.shape)
    l = lse.cpu().numpy().astype(np.float64).reshape(ref_l.shape)
    tol = (1e-2 + 2e-2 * np.abs(ref_o)) if kind == 0 else 5e-2
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    assert np.all(np.abs(o - ref_o) <= tol), f"{what}: max|d|={np.abs(o - ref_o).max():.3e}"
    ninf = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(l), ninf), f"{what}: -inf pattern of lse"
    if (~ninf).any():
        assert np.abs(l[~ninf] - ref_l[~ninf]).max() <= (1e-3 if kind == 0 else 5e-2), f"{what}: lse"


def _oracle_with_table(wl, table):
    """The step on the host (its writes, then the decode) with `table` in
    place of the workload's block table; called before the device step."""
    keep = wl.block_table
    wl.block_table = table
    try:
        c = W.compact(wl, range(wl.B))
    finally:
        wl.block_table = keep
    pool = c["pool"].copy()
    oracle.cache_write(c["w_latent"], c["w_k_pe"], c["w_slots"], pool, wl.kind)
    return oracle.decode(c["q_lat"], c["q_pe"], pool, wl.kind, wl.page_size, c["block_table"], c["seq_lens"],
                         wl.B, wl.Qt, wl.Hq, wl.scale)


BAD_ENTRY_CASES = [
    # (kind, Hq, Qt, page size): the kernel each one takes
    (0, 8, 1, 16),    # folded tiles, 16 rows
    (0, 16, 4, 64),   # folded tiles, 64 rows (scores transposed)
    (0, 16, 6, 16),   # 96 rows: a CTA pair sharing multicast tiles
    (1, 16, 4, 64),   # fp8 pool, folded tiles, 64 rows
    (1, 64, 2, 64),   # fp8 pool, 128 rows: the cluster kernel
    (0, 8, 1, 7),     # a page size that is not a multiple of 8: load/convert warps
]


@pytest.mark.parametrize("kind,Hq,Qt,page_size", BAD_ENTRY_CASES)
def test_block_entries_outside_the_pool_read_page_0_and_flag(kind, Hq, Qt, page_size):
    sl = [300, 1000, 150, 513]
    wl = W.make("oob", B=4, Hq=Hq, Qt=Qt, page_size=page_size, seq_lens=sl, kind=kind, force_block=0,
                write_all=(kind == 1), seed=900 + 10 * kind + Hq + page_size, device=DEV)
    pages = wl.num_slots // page_size
    assert int(wl.block_table[1, 0]) == 0  # page 0 is the first page of the longest request: every row written
    bad = wl.block_table.clone()
    bad[2, 1] = pages + 5      # past the end of the pool
    bad[3, 0] = -7             # negative
    ref_table = wl.block_table.clone()
    ref_table[2, 1] = 0
    ref_table[3, 0] = 0
    ref_o, ref_l = _oracle_with_table(wl, ref_table)
    m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
    out, lse, ws = m.decode(wl.q_lat, wl.q_pe, wl.pool, wl.kind, page_size, bad, wl.seq_lens, Qt, wl.scale,
                            out_dtype=torch.float32)
    torch.cuda.synchronize()
    st = m.device_status(ws)
    assert st & 2 and not st & 1, st
    _check(out, lse, ref_o, ref_l, kind, f"kind={kind} Hq={Hq} Qt={Qt} ps={page_size}")


@pytest.mark.parametrize("kind,Hq,Qt", [(0, 8, 1), (0, 16, 4), (1, 16, 4)])
def test_sequence_longer_than_its_table_row(kind, Hq, Qt):
    """Request 0 needs 13 pages of 16 tokens, its table row holds 9: its last
    four pages are read as page 0 and bit 2 is set. The table is the front of
    a larger allocation, so the row after the last one exists (and names a
    real page that the guarded kernel must not use)."""
    sl = [200, 50, 130]
    ps = 16
    wl = W.make("short_table", B=3, Hq=Hq, Qt=Qt, page_size=ps, seq_lens=sl, kind=kind, force_block=0,
                write_all=(kind == 1), seed=950 + Hq + kind, device=DEV)
    assert int(wl.block_table[0, 0]) == 0 and wl.block_table.shape[1] == 13
    width = 9
    alloc = torch.zeros((wl.B + 1, width), dtype=torch.int32, device=DEV)
    alloc[: wl.B] = wl.block_table[:, :width]
    alloc[wl.B] = wl.block_table[1, 0]
    short = alloc[: wl.B]
    ref_table = wl.block_table.clone()
    ref_table[0, width:] = 0
    ref_o, ref_l = _oracle_with_table(wl, ref_table)
    m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
    out, lse, ws = m.decode(wl.q_lat, wl.q_pe, wl.pool, wl.kind, ps, short, wl.seq_lens, Qt, wl.scale,
                            out_dtype=torch.float32)
    torch.cuda.synchronize()
    st = m.device_status(ws)
    assert st & 2 and not st & 1, st
    _check(out, lse, ref_o, ref_l, kind, f"short table kind={kind} Hq={Hq} Qt={Qt}")
    # a table wide enough for every request: no flag
    out, lse, ws = m.decode(wl.q_lat, wl.q_pe, wl.pool, wl.kind, ps, wl.block_table, wl.seq_lens, Qt, wl.scale)
    torch.cuda.synchronize()
    assert m.device_status(ws) == 0


@pytest.mark.parametrize("Hq,qlens,kind", [
    (8, [1, 2, 1, 2], 0),        # 16 rows
    (16, [2, 3, 1, 4], 0),       # 64 rows
    (16, [5, 8, 2, 7], 0),       # 128 rows: a CTA pair
    (16, [2, 3, 1, 4], 1),       # fp8 pool, 64 rows
])
def test_varlen_rows_past_the_query_count_are_left_alone(Hq, qlens, kind):
    """cu_q_lens ends two tokens past the query count the call is given: the
    sums are clamped to it (the last request verifies only its tokens below
    it, with the shorter length that gives), the spare rows of the output and
    LSE buffers keep their sentinel, and every other row is the oracle's on
    the clamped sums."""
    sl = [400, 90, 1300, 257]
    qmax = max(qlens)
    wl = W.make("varlen_short", B=len(sl), Hq=Hq, Qt=qmax, page_size=16, seq_lens=sl, kind=kind,
                write_all=(kind == 1), seed=970 + Hq + kind + qmax, device=DEV)
    m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
    cu = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    R = int(cu[-1])
    given = R - 2
    pick = torch.tensor([b * qmax + t for b, q in enumerate(qlens) for t in range(q)], dtype=torch.int64, device=DEV)
    q_lat = wl.q_lat[pick].contiguous()
    q_pe = wl.q_pe[pick].contiguous()
    out_all = torch.full((R, Hq, 512), 7.0, dtype=torch.float32, device=DEV)
    lse_all = torch.full((R, Hq), 7.0, dtype=torch.float32, device=DEV)
    ws = torch.empty((m.mla_decode_workspace_bytes(wl.B, qmax, Hq, 0),), dtype=torch.uint8, device=DEV)
    m.mla_decode_varlen(q_lat[:given], q_pe[:given], wl.pool, wl.kind, wl.page_size, wl.block_table, wl.seq_lens,
                        torch.from_numpy(cu).to(DEV), qmax, wl.scale, out_all[:given], lse_all[:given], ws)
    torch.cuda.synchronize()
    assert m.device_status(ws) & 1 == 0
    assert torch.all(out_all[given:] == 7.0) and torch.all(lse_all[given:] == 7.0)
    c = W.compact(wl, range(wl.B))
    cu_c = np.minimum(cu, given).astype(np.int32)
    ref_o, ref_l = oracle.decode_varlen(q_lat[:given].cpu(), q_pe[:given].cpu(), c["pool"], wl.kind, wl.page_size,
                                        c["block_table"], c["seq_lens"], cu_c, Hq, wl.scale)
    _check(out_all[:given], lse_all[:given], ref_o, ref_l, kind, f"varlen Hq={Hq} qlens={qlens} kind={kind}")


def test_gather_past_the_table_row_gives_zero_rows():
    """Request 1 has 40 tokens of 16-token pages but a two-entry table row:
    its tokens 32..39 come out as zero rows; the row after the table exists
    and names a real page."""
    sl = [20, 40]
    wl = W.make("gshort", B=2, Hq=8, Qt=1, page_size=16, seq_lens=sl, kind=W.KIND_FP8, write_all=True, seed=990,
                device=DEV)
    m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
    alloc = torch.zeros((3, 2), dtype=torch.int32, device=DEV)
    alloc[:2] = wl.block_table[:, :2]
    alloc[2] = wl.block_table[1, 2]
    cu = np.array([0, 20, 60], dtype=np.int32)
    dst = torch.full((60, 576), 0x7FFF, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    m.mla_gather_upconvert(wl.pool, 16, alloc[:2], torch.from_numpy(cu).to(DEV), dst)
    torch.cuda.synchronize()
    got = dst.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.all(got[52:60] == 0)
    c = W.compact(wl, [0, 1])
    want = oracle.gather_upconvert(c["pool"], 16, c["block_table"], cu, 60)
    assert np.array_equal(got[:52], want[:52])
