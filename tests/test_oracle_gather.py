"""Pins of the oracle's fp8_ds_mla context gather (``oracle.gather_upconvert``)
against what the pages and IEEE arithmetic fix, independently of the oracle's
own code: torch's bf16 and float8_e4m3fn conversions (library routines),
numpy's float32 multiply, closed forms at power-of-two scales, the cache
write's round-trip bound, and brute-force row bookkeeping."""
import numpy as np
import pytest
import torch

import oracle

D, P, W = 512, 64, 576


def _bf16_bits_of_f32(x32: np.ndarray) -> np.ndarray:
    """torch's fp32 -> bf16 conversion (round to nearest even), as bits."""
    return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def _e4m3_values(codes: np.ndarray) -> np.ndarray:
    """torch's float8_e4m3fn decode of raw codes, as float32."""
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float32).numpy()


def _pool(rng, num_slots, scales=None):
    """A random fp8_ds_mla pool: finite e4m3 codes, positive fp32 scales, bf16 rope bits."""
    pool = np.zeros((num_slots, 656), dtype=np.uint8)
    codes = rng.integers(0, 256, size=(num_slots, 512), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    pool[:, :512] = codes
    if scales is None:
        scales = (np.abs(rng.standard_normal((num_slots, 4))) / 448.0 + 1e-6).astype(np.float32)
    pool[:, 512:528] = np.ascontiguousarray(scales, dtype=np.float32).view(np.uint8).reshape(num_slots, 16)
    rope = rng.integers(0, 1 << 16, size=(num_slots, 64), dtype=np.uint16)
    rope[(rope & 0x7F80) == 0x7F80] = 0x3F80  # finite bf16
    pool[:, 528:] = rope.view(np.uint8).reshape(num_slots, 128)
    return pool


def _one_request(num_slots):
    """Request 0 holds every slot in order: page size 1, block table = identity."""
    bt = np.arange(num_slots, dtype=np.int32)[None, :]
    cu = np.array([0, num_slots], dtype=np.int32)
    return bt, cu


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(20000).astype(np.float32) * np.float32(3.7)
    # exact ties: one ulp of bf16 is 2^-7 at 1.0, so 1 + k 2^-8 (k odd) is a tie
    ties = np.array([1 + k * 2.0 ** -8 for k in range(1, 64, 2)], dtype=np.float32)
    x = np.concatenate([x, ties, -ties, np.array([0.0, -0.0, 3.0e38, 1e-40], dtype=np.float32)])
    got = np.array([oracle.f32_to_bf16(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, _bf16_bits_of_f32(x))


def test_power_of_two_scales_are_exact():
    rng = np.random.default_rng(2)
    n = 97
    k = rng.integers(-4, 5, size=(n, 4))
    scales = np.ldexp(np.ones((n, 4)), k).astype(np.float32)
    pool = _pool(rng, n, scales)
    bt, cu = _one_request(n)
    dst = oracle.gather_upconvert(pool, 1, bt, cu, n)
    want = _e4m3_values(pool[:, :512]) * np.repeat(scales, 128, axis=1)  # exact: 4 significant bits
    assert np.array_equal(_bits_to_f32(dst[:, :512]), want.astype(np.float32))
    assert np.array_equal(dst[:, 512:], pool[:, 528:].view(np.uint16))


def test_products_round_as_float32_then_bf16():
    rng = np.random.default_rng(3)
    n = 211
    pool = _pool(rng, n)
    bt, cu = _one_request(n)
    dst = oracle.gather_upconvert(pool, 1, bt, cu, n)
    scales = pool[:, 512:528].copy().view(np.float32)
    prod32 = _e4m3_values(pool[:, :512]) * np.repeat(scales, 128, axis=1).astype(np.float32)  # float32 multiply
    assert prod32.dtype == np.float32
    assert np.array_equal(dst[:, :512], _bf16_bits_of_f32(prod32))


def test_round_trip_through_the_cache_write():
    rng = np.random.default_rng(4)
    T = 300
    lat = torch.randn(T, D).to(torch.bfloat16)
    kpe = torch.randn(T, P).to(torch.bfloat16)
    pool = np.zeros((T, 656), dtype=np.uint8)
    oracle.cache_write(lat, kpe, np.arange(T, dtype=np.int64), pool, 1)
    bt, cu = _one_request(T)
    dst = oracle.gather_upconvert(pool, 1, bt, cu, T)
    x = lat.float().numpy().astype(np.float64)
    g = _bits_to_f32(dst[:, :512]).astype(np.float64)
    scale = np.repeat(np.abs(x).reshape(T, 4, 128).max(axis=2) / 448.0, 128, axis=1)
    # e4m3: relative 2^-4 in the normal range, 2^-10 * scale below it; then a bf16 rounding (2^-8)
    bound = (2.0 ** -4 * np.abs(x) + 2.0 ** -10 * scale) * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(x) + 1e-30
    assert np.all(np.abs(g - x) <= bound)
    assert np.array_equal(dst[:, 512:], kpe.view(torch.int16).numpy().view(np.uint16))


@pytest.mark.parametrize("page_size", [1, 3, 16, 64])
def test_rows_follow_the_block_table_and_the_rest_stay_untouched(page_size):
    rng = np.random.default_rng(10 + page_size)
    lens = [5, 0, 130, 1, 0, 77]
    pages = [(t + page_size - 1) // page_size for t in lens]
    num_blocks = sum(pages) + 7
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.full((len(lens), max(pages) + 2), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[k:k + n]
        k += n
    num_slots = num_blocks * page_size
    pool = _pool(rng, num_slots)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    rows = int(cu[-1]) + 9  # rows past the last request keep their sentinel
    dst = oracle.gather_upconvert(pool, page_size, bt, cu, rows)
    rope = pool[:, 528:].copy().view(np.uint16)
    for b, T in enumerate(lens):
        for j in range(T):
            slot = int(bt[b, j // page_size]) * page_size + j % page_size
            assert np.array_equal(dst[cu[b] + j, 512:], rope[slot])
    assert np.all(dst[int(cu[-1]):] == 0xFFFF)


def test_rows_past_num_rows_are_skipped_and_bad_pages_zeroed():
    rng = np.random.default_rng(5)
    pool = _pool(rng, 32)
    bt = np.array([[0, 1], [40, 2]], dtype=np.int32)  # page 40 is outside a 32-slot pool (page size 16)
    cu = np.array([0, 20, 40], dtype=np.int32)
    dst = np.full((30, W), 0xFFFF, dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.gather_upconvert(pool, 16, bt, cu, 30, dst=dst)
    assert np.all(dst[20:30] == 0)        # request 1, page 40: zeros
    assert not np.any(dst[:20] == 0xFFFF)  # request 0 written
    dst2 = oracle.gather_upconvert(pool, 16, bt[:1], cu[:2], 12)
    assert dst2.shape == (12, W)           # rows 12..19 of request 0 not written anywhere


def test_slot_above_the_int32_byte_offset_wrap():
    # 2^31 / 656 = 3,273,603: a 32-bit byte offset slot * 656 wraps past it
    n = 3_273_700
    pool = np.zeros((n, 656), dtype=np.uint8)  # untouched pages stay unallocated
    slot = n - 3
    pool[slot, :512] = 0x38                    # e4m3 1.0
    pool[slot, 512:528] = np.array([0.5, 1.0, 2.0, 4.0], dtype=np.float32).view(np.uint8)
    pool[slot, 528:530] = [0x80, 0x3F]         # bf16 1.0
    bt = np.array([[slot]], dtype=np.int32)
    dst = oracle.gather_upconvert(pool, 1, bt, np.array([0, 1], dtype=np.int32), 1)
    assert np.array_equal(_bits_to_f32(dst[0, :512]), np.repeat(np.float32([0.5, 1.0, 2.0, 4.0]), 128))
    assert dst[0, 512] == 0x3F80
