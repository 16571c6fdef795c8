"""Pins of the oracle's decode over other latent widths (oracle.decode_latent).

The pages name per-layer latents of rank 256, 768 and 1792, each with a small
rotary and normalisation tail. The reading here is that the normalisation is
applied before a row is cached, so a cached row is [latent D | rope P] in bf16.

The oracle is checked against:
- a numpy brute force of the definition (gather through the block table,
  scipy's softmax and logsumexp) at each width;
- its own 512-wide decode, which is pinned separately;
- closed forms: a single token, identical rows, no visible token, and the
  causal limit of a verify step.
"""
import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import oracle


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def make_case(D, P, seq_lens, Qt, Hq, page_size, seed):
    g = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    B = len(seq_lens)
    pages = [-(-t // page_size) for t in seq_lens]
    nblocks = sum(pages) + 3
    perm = rng.permutation(nblocks)
    bt = np.full((B, max(1, max(pages))), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[k:k + n]
        k += n
    cache = bf16_bits(torch.randn(nblocks * page_size, D + P, generator=g))
    ql = bf16_bits(torch.randn(B * Qt, Hq, D, generator=g))
    qp = bf16_bits(torch.randn(B * Qt, Hq, P, generator=g))
    return cache, ql, qp, bt, np.asarray(seq_lens, dtype=np.int32)


def brute(cache, ql, qp, bt, sl, D, P, Qt, Hq, page_size, scale):
    B = len(sl)
    c = bits_to_f64(cache)
    out = np.zeros((B * Qt, Hq, D))
    lse = np.full((B * Qt, Hq), -np.inf)
    for b in range(B):
        for qt in range(Qt):
            nvis = max(0, int(sl[b]) - Qt + qt + 1)
            if nvis == 0:
                continue
            rows = np.array([c[int(bt[b, j // page_size]) * page_size + j % page_size] for j in range(nvis)])
            for h in range(Hq):
                r = b * Qt + qt
                q = np.concatenate([bits_to_f64(ql[r, h]), bits_to_f64(qp[r, h])])
                s = scale * (rows @ q)
                out[r, h] = softmax(s) @ rows[:, :D]
                lse[r, h] = logsumexp(s)
    return out, lse


@pytest.mark.parametrize("D,P", [(256, 64), (768, 64), (1792, 64), (256, 32)])
def test_matches_brute_force(D, P):
    seq, Qt, Hq, ps = [5, 0, 23, 1], 2, 3, 4
    cache, ql, qp, bt, sl = make_case(D, P, seq, Qt, Hq, ps, seed=D + P)
    scale = 1.0 / np.sqrt(D + P)
    o, l = oracle.decode_latent(ql, qp, cache, D, P, ps, bt, sl, len(seq), Qt, Hq, scale)
    ro, rl = brute(cache, ql, qp, bt, sl, D, P, Qt, Hq, ps, scale)
    assert np.array_equal(np.isneginf(l), np.isneginf(rl))
    fin = ~np.isneginf(rl)
    assert np.abs(l[fin] - rl[fin]).max() < 1e-12
    assert np.abs(o - ro).max() < 1e-12


def test_512_equals_the_pinned_decode():
    D, P, ps, Qt, Hq = 512, 64, 16, 2, 4
    seq = [40, 1, 0, 77]
    cache, ql, qp, bt, sl = make_case(D, P, seq, Qt, Hq, ps, seed=5)
    scale = 0.05
    o, l = oracle.decode_latent(ql, qp, cache, D, P, ps, bt, sl, len(seq), Qt, Hq, scale)
    pool = np.ascontiguousarray(cache).view(np.uint8).reshape(cache.shape[0], 1152)
    ro, rl = oracle.decode(ql, qp, pool, 0, ps, bt, sl, len(seq), Qt, Hq, scale)
    assert np.array_equal(o, ro) and np.array_equal(l, rl)


@pytest.mark.parametrize("D", [256, 768, 1792])
def test_closed_forms(D):
    P, ps, Hq = 64, 8, 2
    g = torch.Generator().manual_seed(D)
    row = bf16_bits(torch.randn(1, D + P, generator=g))
    T = 37
    cache = np.repeat(row, 40, axis=0)                       # every slot holds the same row
    bt = np.arange(5, dtype=np.int32)[None, :]
    ql = bf16_bits(torch.randn(1, Hq, D, generator=g))
    qp = bf16_bits(torch.randn(1, Hq, P, generator=g))
    scale = 0.03
    s = scale * (np.concatenate([bits_to_f64(ql[0]), bits_to_f64(qp[0])], axis=1) @ bits_to_f64(row[0]))
    # identical rows: out is the row's latent, lse = s + ln T
    o, l = oracle.decode_latent(ql, qp, cache, D, P, ps, bt, np.array([T], np.int32), 1, 1, Hq, scale)
    assert np.allclose(o[0], bits_to_f64(row[0, :D])[None, :], rtol=0, atol=1e-12)
    assert np.abs(l[0] - (s + np.log(T))).max() < 1e-12
    # a single token: out is its latent exactly, lse = s
    o, l = oracle.decode_latent(ql, qp, cache, D, P, ps, bt, np.array([1], np.int32), 1, 1, Hq, scale)
    assert np.array_equal(o[0], np.repeat(bits_to_f64(row[0, :D])[None, :], Hq, axis=0))
    assert np.abs(l[0] - s).max() < 1e-12


def test_causal_verify_equals_truncated_requests():
    """Query token qt of a verify step of Qt tokens over T tokens sees what a
    single-token step over T - Qt + qt + 1 tokens sees."""
    D, P, ps, Qt, Hq = 768, 64, 4, 3, 2
    cache, ql, qp, bt, sl = make_case(D, P, [19], Qt, Hq, ps, seed=11)
    scale = 0.04
    o, l = oracle.decode_latent(ql, qp, cache, D, P, ps, bt, sl, 1, Qt, Hq, scale)
    for qt in range(Qt):
        T1 = np.array([19 - Qt + qt + 1], np.int32)
        o1, l1 = oracle.decode_latent(ql[qt:qt + 1], qp[qt:qt + 1], cache, D, P, ps, bt, T1, 1, 1, Hq, scale)
        assert np.array_equal(o[qt], o1[0]) and np.array_equal(l[qt], l1[0])


def test_no_visible_token_and_bad_block():
    D, P, ps = 256, 64, 4
    cache, ql, qp, bt, sl = make_case(D, P, [0, 2], 3, 1, ps, seed=3)
    o, l = oracle.decode_latent(ql, qp, cache, D, P, ps, bt, sl, 2, 3, 1, 0.1)
    # request 0 has no token; request 1's first query sees none (2 tokens, 3 queries)
    assert np.all(o[0:3] == 0) and np.all(np.isneginf(l[0:3]))
    assert np.all(o[3] == 0) and np.isneginf(l[3, 0]) and np.isfinite(l[4:]).all()
    bt_bad = bt.copy()
    bt_bad[1, 0] = cache.shape[0] // ps + 5
    with pytest.raises(ValueError):
        oracle.decode_latent(ql, qp, cache, D, P, ps, bt_bad, sl, 2, 3, 1, 0.1)
