"""Seeded synthetic workloads for paged MLA decode.

This module only draws random inputs and lays out page tables. It holds none
of the method's arithmetic, so both the GPU path and the CPU oracle can be fed
from it.

Shapes follow the five decode workloads the method is measured on:

  tiny      B=2,   Hq=8,  Qt=1, seq {37, 200},      page 16, bf16 rows
  batched   B=64,  Hq=16, Qt=1, seq U{1024..8192},  page 16, bf16 rows
  long      B=4,   Hq=32, Qt=1, seq 262,144 each,   page 64, bf16 rows
  mtp       B=128, Hq=16, Qt=4 (1 + 3 drafts, causal), 9.8M-slot pool of 16-token
            pages, every block above slot 3,728,270, seq 0 / 1 / U{2048..100000}
  fp8       B=64,  Hq=64, Qt=1, seq 32,768,         page 64, 656-byte fp8_ds_mla
            rows written by the cache-write kernel from N(0,1) bf16 sources

Values are N(0,1) drawn in fp32 and rounded to bf16. The pool starts filled
with NaN sentinels (bf16 0x7FC0 / fp8 0xFF bytes) so that any read of a slot
that holds no token of the request poisons the result. Block tables are
seeded permutations of pool blocks (non-contiguous); unused table entries are
-1. The decode softmax scale is 1/sqrt(192) (128 no-rope + 64 rope dims).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

D, P, W = 512, 64, 576
ROW_BYTES = {0: 1152, 1: 656}
KIND_BF16, KIND_FP8 = 0, 1
SCALE = 1.0 / math.sqrt(192.0)
INT32_WRAP_SLOT = (2 ** 31) // 576  # first slot whose element offset overflows int32


@dataclass
class Workload:
    name: str
    kind: int
    B: int
    Hq: int
    Qt: int
    page_size: int
    num_slots: int
    scale: float
    seq_lens: torch.Tensor        # [B] int32
    block_table: torch.Tensor     # [B, max_blocks] int32, -1 past the last page
    q_lat: torch.Tensor           # [B*Qt, Hq, 512] bf16
    q_pe: torch.Tensor            # [B*Qt, Hq, 64] bf16
    pool: torch.Tensor            # [num_slots, row_bytes] uint8, state before `writes`
    w_latent: torch.Tensor        # [Tw, 512] bf16 rows the step writes first
    w_k_pe: torch.Tensor          # [Tw, 64] bf16
    w_slots: torch.Tensor         # [Tw] int64 (-1 = skip)
    meta: dict = field(default_factory=dict)
    lat_dim: int = D              # latent width of a bf16 row [latent | rope 64]

    @property
    def row_bytes(self) -> int:
        return 2 * (self.lat_dim + P) if self.kind == KIND_BF16 else ROW_BYTES[self.kind]

    def context_tokens(self) -> int:
        return int(self.seq_lens.to(torch.int64).sum().item())

    def cache_bytes(self) -> int:
        """Latent-cache bytes one decode step must read (each row once)."""
        return self.context_tokens() * self.row_bytes


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, g, device) -> torch.Tensor:
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def _nan_pool(num_slots: int, kind: int, device, lat_dim: int = D) -> torch.Tensor:
    row_bytes = 2 * (lat_dim + P) if kind == KIND_BF16 else ROW_BYTES[kind]
    pool = torch.empty((num_slots, row_bytes), dtype=torch.uint8, device=device)
    if kind == KIND_BF16:
        pool.view(torch.int16).fill_(0x7FC0)
    else:
        pool.fill_(0xFF)
    return pool


def _block_table(seq_lens: np.ndarray, page_size: int, block_ids: np.ndarray) -> np.ndarray:
    """Hand out `block_ids` (already shuffled) to requests in order."""
    nblk = [(int(t) + page_size - 1) // page_size for t in seq_lens]
    mb = max(1, max(nblk))
    bt = np.full((len(seq_lens), mb), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = block_ids[pos:pos + n]
        pos += n
    assert pos <= len(block_ids)
    return bt


def token_slots(block_table: torch.Tensor, seq_lens: torch.Tensor, page_size: int) -> torch.Tensor:
    """All (request, position) slots, concatenated request by request (int64)."""
    dev = block_table.device
    out = []
    for b in range(block_table.shape[0]):
        T = int(seq_lens[b])
        if T == 0:
            continue
        j = torch.arange(T, device=dev, dtype=torch.int64)
        blk = block_table[b].to(torch.int64)[j // page_size]
        out.append(blk * page_size + j % page_size)
    if not out:
        return torch.empty((0,), dtype=torch.int64, device=dev)
    return torch.cat(out)


def _fill_rows(pool: torch.Tensor, slots: torch.Tensor, g, device, rms_spread: float = 0.0,
               chunk: int = 1 << 20) -> None:
    """Write N(0,1) bf16 rows into `slots` of a bf16 pool, in chunks."""
    pv = pool.view(torch.bfloat16)
    width = pv.shape[1]
    for s in range(0, slots.numel(), chunk):
        idx = slots[s:s + chunk]
        rows = torch.randn((idx.numel(), width), generator=g, device=device, dtype=torch.float32)
        if rms_spread:
            f = torch.exp(rms_spread * (2 * torch.rand((idx.numel(), 1), generator=g, device=device) - 1))
            rows = rows * f
        pv[idx] = rows.to(torch.bfloat16)


def make(name: str, *, B: int, Hq: int, Qt: int, page_size: int, seq_lens, kind: int = KIND_BF16,
         num_blocks: int | None = None, min_block: int = 0, force_block: int | None = None,
         seed: int = 0, device="cpu", write_last: int | None = None, rms_spread: float = 0.0,
         write_all: bool = False, lat_dim: int = D) -> Workload:
    """General builder.

    seq_lens     per-request context lengths, counting the Qt query tokens.
    num_blocks   pool size in pages (default: 1.25x what the requests need).
    min_block    lowest block id handed out (blocks below stay NaN).
    force_block  a block id that must appear, as the first (full) page of the
                 longest request, so every one of its slots holds a token.
    write_last   how many trailing tokens per request the step writes with the
                 cache-write kernel (default Qt; bf16 pools only).
    write_all    (fp8) every token's row is written by the cache-write kernel.
    lat_dim      (bf16) latent width of a row [latent lat_dim | rope 64].
    """
    assert lat_dim == D or kind == KIND_BF16
    g_np = np.random.default_rng(seed)
    sl = np.asarray(seq_lens, dtype=np.int64)
    need = int(sum((int(t) + page_size - 1) // page_size for t in sl))
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(need * 1.25)))
    avail = np.arange(min_block, num_blocks, dtype=np.int64)
    if need > len(avail):
        raise ValueError(f"{name}: requests need {need} pages, pool offers {len(avail)}")
    ids = g_np.permutation(avail)[:need]
    bt_np = _block_table(sl, page_size, ids)
    if force_block is not None and need > 0:
        b = int(np.argmax(sl))
        hit = np.argwhere(bt_np == force_block)
        if len(hit):
            bt_np[hit[0][0], hit[0][1]] = bt_np[b, 0]
        bt_np[b, 0] = force_block
    num_slots = num_blocks * page_size

    g = _gen(seed, device)
    block_table = torch.from_numpy(bt_np).to(device)
    seq = torch.from_numpy(sl.astype(np.int32)).to(device)
    q_lat = _randn_bf16((B * Qt, Hq, lat_dim), g, device)
    q_pe = _randn_bf16((B * Qt, Hq, P), g, device)
    pool = _nan_pool(num_slots, kind, device, lat_dim)
    slots = token_slots(block_table, seq, page_size)

    if kind == KIND_BF16:
        _fill_rows(pool, slots, g, device, rms_spread)
        wl = Qt if write_last is None else write_last
        ws = []
        for b in range(B):
            T = int(sl[b])
            for j in range(max(0, T - wl), T):
                ws.append(int(bt_np[b, j // page_size]) * page_size + j % page_size)
        w_slots = torch.tensor(ws, dtype=torch.int64, device=device)
    else:
        assert write_all, "fp8 pools are written by the cache-write kernel"
        w_slots = slots
    Tw = w_slots.numel()
    w_latent = _randn_bf16((Tw, lat_dim), g, device)
    w_k_pe = _randn_bf16((Tw, P), g, device)
    if rms_spread and Tw:
        f = torch.exp(rms_spread * (2 * torch.rand((Tw, 1), generator=g, device=device) - 1))
        w_latent = (w_latent.float() * f).to(torch.bfloat16)
    return Workload(name=name, kind=kind, B=B, Hq=Hq, Qt=Qt, page_size=page_size,
                    num_slots=num_slots, scale=SCALE, seq_lens=seq, block_table=block_table,
                    q_lat=q_lat, q_pe=q_pe, pool=pool, w_latent=w_latent, w_k_pe=w_k_pe,
                    w_slots=w_slots, meta={"seed": seed, "num_blocks": num_blocks}, lat_dim=lat_dim)


# ------------------------------------------------------------ named configs

def tiny(device="cpu", seed: int = 1) -> Workload:
    """B=2, Hq=8, seq {37, 200}, page 16, a 64-block pool; request 0 gets the
    first 3 blocks of a seeded permutation of the pool, request 1 the next 13."""
    return make("tiny", B=2, Hq=8, Qt=1, page_size=16, seq_lens=[37, 200], num_blocks=64,
                seed=seed, device=device)


def batched_seq_lens(seed: int = 2) -> np.ndarray:
    return np.random.default_rng(seed).integers(1024, 8192, size=64, endpoint=True)


def batched(device="cpu", seed: int = 2) -> Workload:
    return make("batched", B=64, Hq=16, Qt=1, page_size=16, seq_lens=batched_seq_lens(seed),
                seed=seed, device=device)


def long(device="cpu", seed: int = 3, B: int = 4) -> Workload:
    """B requests of 262,144 tokens (4 in the named workload; fewer give a
    cut-down copy of the same shape for profiling)."""
    return make("long", B=B, Hq=32, Qt=1, page_size=64, seq_lens=[262144] * B, num_blocks=4096 * B,
                seed=seed, device=device)


MTP_POOL_SLOTS = 9_800_000
MTP_PAGE = 16


def mtp_seq_lens(seed: int = 4) -> np.ndarray:
    """8 empty requests, 8 one-token requests, 112 of U{2048..100000} tokens,
    redrawn (deterministically) until they fit in the pool above the int32
    wrap slot."""
    rng = np.random.default_rng(seed)
    nb = MTP_POOL_SLOTS // MTP_PAGE
    first = -(-INT32_WRAP_SLOT // MTP_PAGE)
    while True:
        long_ = rng.integers(2048, 100000, size=112, endpoint=True)
        sl = np.concatenate([np.zeros(8, np.int64), np.ones(8, np.int64), long_])
        sl = sl[rng.permutation(sl.size)]
        if sum(-(-int(t) // MTP_PAGE) for t in sl) <= nb - first:
            return sl


def mtp(device="cpu", seed: int = 4, Qt: int = 4, B: int = 128) -> Workload:
    """The large-pool verify workload; Qt = 4 (1 + 3 drafts) as named, or a
    longer step (1 + 7 drafts: Qt = 8) on the same pool and requests. B < 128
    keeps the first B requests in a pool of their own size (a cut-down copy of
    the same row shape for profiling; no slot past the int32 wrap)."""
    if B < 128:
        return make(f"mtp_b{B}", B=B, Hq=16, Qt=Qt, page_size=MTP_PAGE, seq_lens=mtp_seq_lens(seed)[:B], seed=seed,
                    device=device)
    nb = MTP_POOL_SLOTS // MTP_PAGE            # 612,500 pages
    first = -(-INT32_WRAP_SLOT // MTP_PAGE)    # 233,017: first page wholly above the wrap slot
    return make("mtp" if Qt == 4 else f"mtp_q{Qt}", B=128, Hq=16, Qt=Qt, page_size=MTP_PAGE,
                seq_lens=mtp_seq_lens(seed), num_blocks=nb, min_block=first, force_block=nb - 1, seed=seed,
                device=device)


def fp8(device="cpu", seed: int = 5, B: int = 64) -> Workload:
    """B requests of 32,768 tokens (64 in the named workload; fewer give a
    cut-down copy of the same shape for profiling)."""
    return make("fp8", B=B, Hq=64, Qt=1, page_size=64, seq_lens=[32768] * B, num_blocks=512 * B,
                kind=KIND_FP8, write_all=True, seed=seed, device=device)


def latent(D: int, device="cpu", seed: int = 2) -> Workload:
    """The batched shape (B=64, Hq=16, seq U{1024..8192}, page 16) over bf16
    rows of another latent width: [latent D | rope 64]."""
    return make(f"latent{D}", B=64, Hq=16, Qt=1, page_size=16, seq_lens=batched_seq_lens(seed), seed=seed,
                device=device, lat_dim=D)


CONFIGS = {"tiny": tiny, "batched": batched, "long": long, "mtp": mtp, "fp8": fp8}


# ----------------------------------------------------- host copies for checks

def compact(wl: Workload, reqs) -> dict:
    """Host copy of just what requests `reqs` read, with renumbered pages.

    Returns numpy arrays for a pool holding only those requests' pages (in
    their state before the step's writes, so call this before running the
    step on the device), the matching block table, the step's writes that
    land in those pages, and the requests' queries. Plumbing only: no
    arithmetic of the method happens here."""
    reqs = [int(r) for r in reqs]
    ps = wl.page_size
    bt = wl.block_table.cpu().numpy()
    sl = wl.seq_lens.cpu().numpy()
    pages = []
    for b in reqs:
        n = -(-int(sl[b]) // ps)
        pages.extend(int(x) for x in bt[b, :n])
    uniq = sorted(set(pages))
    remap = {p: i for i, p in enumerate(uniq)}
    nb = max(1, len(uniq))
    pool_rows = torch.empty((nb * ps, wl.row_bytes), dtype=torch.uint8)
    if uniq:
        pg = torch.tensor(uniq, dtype=torch.int64, device=wl.pool.device)
        idx = (pg[:, None] * ps + torch.arange(ps, device=pg.device)[None, :]).reshape(-1)
        pool_rows[: idx.numel()] = wl.pool[idx].cpu()
    mb = max(1, max(-(-int(sl[b]) // ps) for b in reqs) if reqs else 1)
    bt_c = np.full((len(reqs), mb), -1, dtype=np.int32)
    for i, b in enumerate(reqs):
        n = -(-int(sl[b]) // ps)
        bt_c[i, :n] = [remap[int(x)] for x in bt[b, :n]]
    ws = wl.w_slots.cpu().numpy()
    keep, new_slots = [], []
    for t, s in enumerate(ws):
        if s < 0:
            continue
        p = int(s) // ps
        if p in remap:
            keep.append(t)
            new_slots.append(remap[p] * ps + int(s) % ps)
    keep_t = torch.tensor(keep, dtype=torch.int64)
    rows = torch.tensor([q for b in reqs for q in range(b * wl.Qt, (b + 1) * wl.Qt)], dtype=torch.int64)
    return {
        "pool": pool_rows.numpy(),
        "block_table": bt_c,
        "seq_lens": sl[reqs].astype(np.int32),
        "q_lat": wl.q_lat.cpu()[rows],
        "q_pe": wl.q_pe.cpu()[rows],
        "w_latent": wl.w_latent.cpu()[keep_t] if keep else wl.w_latent.cpu()[:0],
        "w_k_pe": wl.w_k_pe.cpu()[keep_t] if keep else wl.w_k_pe.cpu()[:0],
        "w_slots": np.asarray(new_slots, dtype=np.int64),
        "rows": rows.numpy(),
    }
