"""GPU parity of mla_gather_upconvert (the fp8_ds_mla prefill-context gather)
against the oracle: bit-exact bf16 rows, at small and full workload sizes,
slots above the int32 byte-offset wrap, strides, row limits and bad pages."""
import numpy as np
import pytest
import torch

import mla_latent_kv_cache_gb300 as m
import oracle
from mla_latent_kv_cache_gb300 import build as mbuild
from mla_latent_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SENTINEL = 0x7FFF  # a NaN bit pattern no gathered row can produce


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mbuild.build()
    m.load()
    torch.cuda.set_device(DEV)
    yield


def _written(wl):
    """The workload's fp8 pool after the cache-write kernel wrote every token."""
    m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
    torch.cuda.synchronize()
    return wl


def _cu(seq_lens):
    sl = np.asarray(seq_lens, dtype=np.int64)
    return np.concatenate([[0], np.cumsum(sl)]).astype(np.int32)


def _gpu_gather(wl, cu, rows, stride=576, num_rows=None):
    dst = torch.full((rows, stride), 0, dtype=torch.int16, device=DEV)
    dst.fill_(SENTINEL)
    dst = dst.view(torch.bfloat16)
    m.mla_gather_upconvert(wl.pool, wl.page_size, wl.block_table, torch.from_numpy(cu).to(DEV), dst,
                           num_rows=num_rows)
    torch.cuda.synchronize()
    return dst.view(torch.int16).cpu().numpy().view(np.uint16)


def _oracle_gather(wl, reqs, rows, stride=576, num_rows=None):
    c = W.compact(wl, reqs)
    dst = np.full((rows, stride), SENTINEL, dtype=np.uint16)
    oracle.gather_upconvert(c["pool"], wl.page_size, c["block_table"], _cu(c["seq_lens"]),
                            rows if num_rows is None else num_rows, dst=dst, dst_stride=stride)
    return dst


@pytest.mark.parametrize("page_size", [1, 3, 16, 64, 784])
def test_gather_is_bit_exact(page_size):
    sl = [1, 17, 300, 0, 129, 784, 785]
    wl = _written(W.make("g", B=len(sl), Hq=8, Qt=1, page_size=page_size, seq_lens=sl, kind=W.KIND_FP8,
                         write_all=True, seed=70 + page_size, device=DEV))
    cu = _cu(sl)
    rows = int(cu[-1]) + 5  # the last five rows are named by no request
    got = _gpu_gather(wl, cu, rows)
    want = _oracle_gather(wl, range(wl.B), rows)
    assert np.array_equal(got, want)
    assert np.all(got[-5:] == SENTINEL)


def test_gather_row_limit_and_wide_rows():
    sl = [40, 0, 90, 7]
    wl = _written(W.make("gs", B=len(sl), Hq=8, Qt=1, page_size=16, seq_lens=sl, kind=W.KIND_FP8,
                         write_all=True, seed=81, device=DEV))
    cu = _cu(sl)
    rows, limit = int(cu[-1]), 100  # rows >= 100 are skipped
    got = _gpu_gather(wl, cu, rows, stride=640, num_rows=limit)
    want = _oracle_gather(wl, range(wl.B), rows, stride=640, num_rows=limit)
    assert np.array_equal(got, want)
    assert np.all(got[limit:] == SENTINEL) and np.all(got[:, 576:] == SENTINEL)


def test_gather_slots_above_the_int32_byte_wrap():
    # 2^31 / 656 = 3,273,603: every page handed out starts above that slot
    first = 3_273_603 // 16 + 1
    sl = [700, 1500, 33, 16]
    wl = _written(W.make("gw", B=len(sl), Hq=8, Qt=1, page_size=16, seq_lens=sl, kind=W.KIND_FP8,
                         write_all=True, num_blocks=first + 400, min_block=first, force_block=first + 399,
                         seed=82, device=DEV))
    assert int(wl.block_table[wl.block_table >= 0].min()) * 16 > 3_273_603
    cu = _cu(sl)
    rows = int(cu[-1])
    assert np.array_equal(_gpu_gather(wl, cu, rows), _oracle_gather(wl, range(wl.B), rows))


def test_gather_full_fp8_workload_on_whole_requests():
    wl = _written(W.fp8(device=DEV))
    sl = wl.seq_lens.cpu().numpy()
    cu = _cu(sl)
    rows = int(cu[-1])  # 2,097,152 rows of 576 bf16 (2.4 GB)
    got = _gpu_gather(wl, cu, rows)
    for b in (0, 37, 63):  # three whole requests, against the oracle
        c = W.compact(wl, [b])
        want = oracle.gather_upconvert(c["pool"], wl.page_size, c["block_table"], _cu(c["seq_lens"]), int(sl[b]))
        assert np.array_equal(got[cu[b]:cu[b + 1]], want)


def test_gather_page_outside_the_pool_gives_zero_rows():
    sl = [20, 20]
    wl = _written(W.make("gb", B=2, Hq=8, Qt=1, page_size=16, seq_lens=sl, kind=W.KIND_FP8,
                         write_all=True, seed=83, device=DEV))
    wl.block_table[1, 1] = wl.num_slots // 16 + 5  # request 1, tokens 16..19: a page past the pool
    cu = _cu(sl)
    got = _gpu_gather(wl, cu, 40)
    assert np.all(got[36:40] == 0)
    c = W.compact(wl, [0])
    want = oracle.gather_upconvert(c["pool"], 16, c["block_table"], _cu(c["seq_lens"]), 20)
    assert np.array_equal(got[:20], want)


def test_gather_empty_calls_do_nothing():
    wl = _written(W.make("ge", B=2, Hq=8, Qt=1, page_size=16, seq_lens=[0, 0], kind=W.KIND_FP8,
                         write_all=True, seed=84, device=DEV))
    got = _gpu_gather(wl, _cu([0, 0]), 8)
    assert np.all(got == SENTINEL)
