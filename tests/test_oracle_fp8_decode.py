"""Pins of the oracle's decode over fp8_ds_mla rows (cache kind 1).

The oracle's fp8 decode dequantises each 656-byte row (vLLM PR #55543, PR
description "Approach" and "Memory tradeoff"; commits 5.1-5.4: per-128-block
fp8 quantisation of the NoPE bytes, the bf16 rope kept as stored) and runs the
plain decode definition on it. Here a numpy fp64 brute force recomputes that
definition from the bytes with torch's float8_e4m3fn decode, the scale of
dims [128 j, 128 j + 128) read at byte 512 + 4 j, and the rope read from bytes
528..655 as bf16. A wrong scale index (d % 4 instead of d // 128) or a rope
read at byte 512 fails the comparison; the tests below show that either slip
moves the brute force away from the oracle by far more than the tolerance.
"""
import numpy as np
import torch
from scipy.special import logsumexp

import oracle
from mla_latent_kv_cache_gb300 import workloads as W

ROW = 656


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _fp8_pool(num_slots, slots, seed, block_gain=(1.0, 1e-2, 30.0, 0.25)):
    """A pool of fp8 rows written by the oracle's cache write from N(0,1)
    bf16 sources whose four 128-blocks are scaled by very different gains,
    so that the four block scales of a row differ by orders of magnitude."""
    g = torch.Generator().manual_seed(seed)
    T = len(slots)
    lat = torch.randn((T, 512), generator=g)
    gain = torch.tensor(block_gain, dtype=torch.float32).repeat_interleave(128)
    lat = (lat * gain).to(torch.bfloat16)
    kpe = torch.randn((T, 64), generator=g).to(torch.bfloat16)
    pool = np.full((num_slots, ROW), 0xFF, dtype=np.uint8)
    oracle.cache_write(lat, kpe, np.asarray(slots, dtype=np.int64), pool, 1)
    return pool


def _dequant(pool, scale_index=lambda d: d // 128, rope_byte=528):
    """Brute-force dequantisation of every row: [num_slots, 576] fp64."""
    codes = torch.from_numpy(pool[:, :512].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    scales = pool[:, 512:528].copy().view(np.float32).astype(np.float64)  # [n, 4], little endian
    d = np.arange(512)
    lat = codes * scales[:, scale_index(d)]
    rope = torch.from_numpy(pool[:, rope_byte:rope_byte + 128].copy().view(np.int16)).view(torch.bfloat16)
    return np.concatenate([lat, rope.to(torch.float64).numpy()], axis=1)


def _brute_decode(rows, q_lat, q_pe, block_table, seq_lens, page_size, Qt, Hq, scale):
    """fp64 softmax over each query row's visible tokens (numpy, scipy)."""
    B = len(seq_lens)
    ql = torch.from_numpy(_bits(q_lat).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    qp = torch.from_numpy(_bits(q_pe).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    ql = ql.reshape(B * Qt, Hq, 512)
    qp = qp.reshape(B * Qt, Hq, 64)
    out = np.zeros((B * Qt, Hq, 512))
    lse = np.full((B * Qt, Hq), -np.inf)
    for b in range(B):
        T = int(seq_lens[b])
        j = np.arange(T)
        slots = block_table[b, j // page_size].astype(np.int64) * page_size + j % page_size
        c = rows[slots]
        for t in range(Qt):
            nvis = T - Qt + t + 1
            if nvis <= 0:
                continue
            r = b * Qt + t
            q = np.concatenate([ql[r], qp[r]], axis=1)  # [Hq, 576]
            s = scale * (q @ c[:nvis].T)                # [Hq, nvis]
            L = logsumexp(s, axis=1)
            out[r] = np.exp(s - L[:, None]) @ c[:nvis, :512]
            lse[r] = L
    return out, lse


def _case(seed=0, page_size=16, seq_lens=(1, 37, 200, 0), Qt=1, Hq=8):
    rng = np.random.default_rng(seed)
    need = [-(-t // page_size) for t in seq_lens]
    nb = sum(need) + 3
    perm = rng.permutation(nb)
    bt = np.full((len(seq_lens), max(1, max(need))), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[pos:pos + n]
        pos += n
    num_slots = nb * page_size
    slots = [int(bt[b, j // page_size]) * page_size + j % page_size
             for b, T in enumerate(seq_lens) for j in range(T)]
    pool = _fp8_pool(num_slots, slots, seed)
    g = torch.Generator().manual_seed(seed + 100)
    B = len(seq_lens)
    q_lat = torch.randn((B * Qt, Hq, 512), generator=g).to(torch.bfloat16)
    q_pe = torch.randn((B * Qt, Hq, 64), generator=g).to(torch.bfloat16)
    return pool, bt, np.asarray(seq_lens, dtype=np.int32), q_lat, q_pe


def _oracle(pool, bt, sl, q_lat, q_pe, page_size=16, Qt=1, Hq=8):
    return oracle.decode(q_lat, q_pe, pool, 1, page_size, bt, sl, len(sl), Qt, Hq, W.SCALE)


def test_fp8_decode_matches_brute_force():
    for seed, ps, Qt in ((0, 16, 1), (1, 3, 1), (2, 64, 4)):
        seq = (1, 37, 200, 0) if Qt == 1 else (2, 5, 130, 64)
        pool, bt, sl, ql, qp = _case(seed=seed, page_size=ps, seq_lens=seq, Qt=Qt)
        o, l = _oracle(pool, bt, sl, ql, qp, page_size=ps, Qt=Qt)
        ro, rl = _brute_decode(_dequant(pool), ql, qp, bt, sl, ps, Qt, 8, W.SCALE)
        np.testing.assert_allclose(o, ro, rtol=1e-12, atol=1e-12)
        fin = np.isfinite(rl)
        assert np.array_equal(fin, np.isfinite(l))
        np.testing.assert_allclose(l[fin], rl[fin], rtol=0, atol=1e-12)
        assert np.all(l[~fin] == -np.inf) and np.all(o[~fin] == 0.0)


def test_fp8_one_token_request_returns_its_dequantised_row():
    pool, bt, sl, ql, qp = _case(seed=3, seq_lens=(1, 1, 1))
    o, l = _oracle(pool, bt, sl, ql, qp)
    rows = _dequant(pool)
    for b in range(3):
        slot = int(bt[b, 0]) * 16
        # p = 1: the output is the row's 512 dequantised latent values (each
        # exactly e4m3(code) x fp32 scale in fp64), identically for all heads
        assert np.array_equal(o[b], np.broadcast_to(rows[slot, :512], (8, 512)))
        q = np.concatenate([ql[b].to(torch.float64).numpy(), qp[b].to(torch.float64).numpy()], axis=1)
        np.testing.assert_allclose(l[b], W.SCALE * (q @ rows[slot]), rtol=1e-13, atol=1e-13)


def test_fp8_block_scales_have_teeth():
    pool, bt, sl, ql, qp = _case(seed=4)
    o, l = _oracle(pool, bt, sl, ql, qp)
    swapped = pool.copy()
    s = swapped[:, 512:528].copy().view(np.float32)
    s[:, [1, 2]] = s[:, [2, 1]]
    swapped[:, 512:528] = s.view(np.uint8)
    o2, l2 = _oracle(swapped, bt, sl, ql, qp)
    live = np.isfinite(l)
    assert np.abs(o2[live] - o[live]).max() > 1e-2
    assert np.abs(l2[live] - l[live]).max() > 1e-2


def test_plausible_slips_fail_the_pin():
    # the brute force with a wrong scale index, or with the rope read from the
    # scale bytes, is far from the oracle: the comparison above would catch
    # either slip in the oracle's row reader
    pool, bt, sl, ql, qp = _case(seed=5)
    o, l = _oracle(pool, bt, sl, ql, qp)
    live = np.isfinite(l)
    for rows in (_dequant(pool, scale_index=lambda d: d % 4), _dequant(pool, rope_byte=512)):
        ro, rl = _brute_decode(rows, ql, qp, bt, sl, 16, 1, 8, W.SCALE)
        assert np.abs(rl[live] - l[live]).max() > 1e-3 or np.abs(ro[live] - o[live]).max() > 1e-3


def test_fp8_decode_equals_bf16_decode_of_the_dequantised_rows_when_exact():
    # rows whose dequantised values are bf16-exact (scale a power of two and
    # values on the e4m3 grid): the fp8 decode must equal the bf16 decode of a
    # pool holding those values, which pins the fp8 branch to the pinned bf16 one
    rng = np.random.default_rng(6)
    n = 48
    # finite codes of both signs (0x7F and 0xFF are NaN)
    codes = (rng.integers(0, 0x7F, size=(n, 512)) | (rng.integers(0, 2, size=(n, 512)) << 7)).astype(np.uint8)
    sc = (2.0 ** rng.integers(-4, 5, size=(n, 4))).astype(np.float32)
    kpe = torch.randn((n, 64), generator=torch.Generator().manual_seed(6)).to(torch.bfloat16)
    pool8 = np.zeros((n, ROW), dtype=np.uint8)
    pool8[:, :512] = codes
    pool8[:, 512:528] = sc.view(np.uint8).reshape(n, 16)
    pool8[:, 528:] = _bits(kpe).view(np.uint8).reshape(n, 128)
    deq = _dequant(pool8)
    as_bf16 = torch.from_numpy(deq).to(torch.bfloat16)
    assert np.array_equal(as_bf16.to(torch.float64).numpy(), deq)  # exact in bf16
    pool16 = _bits(as_bf16).view(np.uint8).reshape(n, 1152).copy()
    bt = np.arange(3, dtype=np.int32).reshape(1, 3)
    sl = np.array([n], dtype=np.int32)
    g = torch.Generator().manual_seed(7)
    ql = torch.randn((1, 8, 512), generator=g).to(torch.bfloat16)
    qp = torch.randn((1, 8, 64), generator=g).to(torch.bfloat16)
    o8, l8 = oracle.decode(ql, qp, pool8, 1, 16, bt, sl, 1, 1, 8, W.SCALE)
    o16, l16 = oracle.decode(ql, qp, pool16, 0, 16, bt, sl, 1, 1, 8, W.SCALE)
    assert np.array_equal(o8, o16) and np.array_equal(l8, l16)
