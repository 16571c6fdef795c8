"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks the oracle against something fixed independently of it: a
number the pages print (tests/golden/geometry.json), a mathematical identity
(absorbed == naive MLA attention), a closed form (identical rows, one-hot
rows, a single token), a library routine (torch's float8_e4m3fn cast,
scipy's softmax / logsumexp), brute force (nearest-value table search), or an
invariant (page-size and partition invariance, causal truncation, rope-free
invariance). A slip in the oracle (a dropped term, a wrong index, the softmax
over heads instead of tokens, a missing scale) fails at least one of them.
"""
import json
import math
import os
import tempfile

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import oracle
from mla_latent_kv_cache_gb300 import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden", "geometry.json")


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def bf16_pool(rows: torch.Tensor) -> np.ndarray:
    """[n, 576] bf16 -> uint8 pool of 1152-byte rows."""
    return bits(rows).view(np.uint8).reshape(rows.shape[0], 1152).copy()


# ----------------------------------------------------------------- geometry

def test_geometry_matches_pages():
    g = json.load(open(GOLD))
    assert oracle.row_values() == g["values_per_token"]["value"]
    assert oracle.D + oracle.P == g["values_per_token"]["value"]
    assert oracle.D == g["latent_dims"]["value"] and oracle.P == g["rope_dims"]["value"]
    assert oracle.row_bytes(0) == g["bf16_row_bytes"]["value"] == 2 * oracle.row_values()
    assert oracle.row_bytes(1) == g["fp8_ds_mla_row_bytes"]["value"]
    # 656 = 512 e4m3 codes + 4 fp32 scales (one per 128-block) + 64 bf16 rope
    blk = g["fp8_quant_block"]["value"]
    assert oracle.D + 4 * (oracle.D // blk) + 2 * oracle.P == oracle.row_bytes(1)
    assert 2 ** 31 // oracle.row_values() == g["int32_wrap_slot"]["value"]
    assert round(100 * (656 / g["nope_fp8_row_bytes"]["value"] - 1)) == g["fp8_vs_nope_overhead_pct"]["value"]
    assert round(100 * (1 - 656 / 1152)) == g["fp8_vs_bf16_reduction_pct"]["value"]
    # the B300 pool reaches past the wrap slot, the H100 pool does not
    assert g["h100_pool_slots_approx"]["value"] < g["int32_wrap_slot"]["value"] < g["b300_pool_slots_approx"]["value"]
    assert W.INT32_WRAP_SLOT == g["int32_wrap_slot"]["value"]


# -------------------------------------------------------------------- codecs

def test_bf16_decode_matches_torch():
    allb = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(allb.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_f64(int(b)) for b in allb[::97]])
    r = ref[::97]
    assert np.array_equal(np.isnan(got), np.isnan(r))
    assert np.array_equal(got[~np.isnan(r)], r[~np.isnan(r)])


def _e4m3_table():
    codes = np.arange(256, dtype=np.uint8)
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_matches_torch_all_codes():
    ref = _e4m3_table()
    got = np.array([oracle.e4m3_to_f64(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF])
    assert got[0x7E] == 448.0 and got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9


def _codec_sample(rng) -> np.ndarray:
    tab = _e4m3_table()[:0x7F]                  # non-negative finite values, increasing
    mids = (tab[1:] + tab[:-1]) / 2             # exact ties (all are fp32 values)
    m32 = mids.astype(np.float32)
    near = np.concatenate([m32, np.nextafter(m32, np.float32(np.inf)), np.nextafter(m32, np.float32(0))])
    allbf = torch.from_numpy(np.arange(65536, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).float().numpy()
    rnd = (rng.standard_normal(400_000) * np.exp2(rng.uniform(-14, 9, 400_000))).astype(np.float32)
    x = np.concatenate([near, -near, tab.astype(np.float32), allbf, rnd])
    x = x[np.isfinite(x) & (np.abs(x) <= 448.0)]
    return x


def test_e4m3_encode_matches_torch_cast():
    """torch's float8_e4m3fn cast rounds to nearest-even inside the finite
    range; there the oracle must agree bit for bit."""
    x = _codec_sample(np.random.default_rng(0))
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.f32_to_e4m3_array(x)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], ref[bad[:5]])


def test_e4m3_encode_matches_bruteforce_nearest():
    """Nearest table value, ties to the even code (the code LSB is the
    mantissa LSB), saturating at 448."""
    tab = _e4m3_table()[:0x7F]
    x = _codec_sample(np.random.default_rng(1))[::7]
    a = np.abs(x.astype(np.float64))
    d = np.abs(a[:, None] - tab[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    codes = np.arange(0x7F)
    even = cand & (codes[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1)).astype(np.uint8)
    pick = pick | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    assert np.array_equal(oracle.f32_to_e4m3_array(x), pick)


def test_e4m3_encode_saturates_and_specials():
    x = np.array([448.0, 449.0, 463.9, 464.0, 1e30, np.inf, -np.inf, -1e9, np.nan, -0.0, 0.0,
                  2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -9, 1.0, 240.0, 2.0 ** -6], dtype=np.float32)
    got = oracle.f32_to_e4m3_array(x).tolist()
    assert got[:8] == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert got[8] & 0x7F == 0x7F                 # NaN stays NaN
    assert got[9] == 0x80 and got[10] == 0x00    # signed zero kept
    assert got[11] == 0x00                       # 2^-10 ties between 0 and 2^-9: even code 0
    assert got[12] == 0x02                       # 1.5*2^-9 ties between codes 1 and 2: even 2
    assert got[13] == 0x01 and got[14] == 0x38 and got[15] == 0x77 and got[16] == 0x08


# ---------------------------------------------------------------- cache write

def _write_case(kind, T=40, num_slots=97, seed=0, zero_kpe=False):
    g = torch.Generator().manual_seed(seed)
    lat = (torch.randn(T, 512, generator=g) * torch.exp(torch.randn(T, 1, generator=g))).to(torch.bfloat16)
    kpe = torch.zeros(T, 64, dtype=torch.bfloat16) if zero_kpe else torch.randn(T, 64, generator=g).to(torch.bfloat16)
    rng = np.random.default_rng(seed)
    slots = rng.permutation(num_slots)[:T].astype(np.int64)
    slots[::7] = -1
    pool = np.full((num_slots, oracle.ROW_BYTES[kind]), 0xA5, dtype=np.uint8)
    before = pool.copy()
    oracle.cache_write(lat, kpe, slots, pool, kind)
    return lat, kpe, slots, pool, before


def test_cache_write_bf16_is_a_bit_copy():
    lat, kpe, slots, pool, before = _write_case(0)
    lb, kb = bits(lat), bits(kpe)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        assert np.array_equal(pool[s, :1024].view(np.uint16), lb[t])
        assert np.array_equal(pool[s, 1024:].view(np.uint16), kb[t])
    written = set(int(s) for s in slots if s >= 0)
    untouched = [i for i in range(pool.shape[0]) if i not in written]
    assert np.array_equal(pool[untouched], before[untouched])


def test_cache_write_rejects_out_of_range_slot():
    lat = torch.zeros(1, 512, dtype=torch.bfloat16)
    kpe = torch.zeros(1, 64, dtype=torch.bfloat16)
    pool = np.zeros((4, 1152), dtype=np.uint8)
    with pytest.raises(ValueError):
        oracle.cache_write(lat, kpe, np.array([4]), pool, 0)


def test_cache_write_fp8_round_trip():
    lat, kpe, slots, pool, before = _write_case(1)
    x = f64(lat)
    kb = bits(kpe)
    tab = _e4m3_table()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        row = pool[s]
        sc = row[512:528].view(np.float32).astype(np.float64)
        assert np.array_equal(row[528:].view(np.uint16), kb[t])       # rope stored unchanged
        for j in range(4):
            blk = x[t, 128 * j:128 * (j + 1)]
            amax = np.float32(np.abs(blk).max())
            assert sc[j] == np.float32(amax / np.float32(448.0))       # absmax / 448 in fp32
            deq = tab[row[128 * j:128 * (j + 1)]] * sc[j]
            q = np.abs(blk) / sc[j]
            normal = q >= 2.0 ** -6
            # e4m3 has 3 mantissa bits: half an ulp is 2^-4 of the value
            assert np.all(np.abs(deq - blk)[normal] <= 2.0 ** -4 * np.abs(blk)[normal] * (1 + 1e-6))
            assert np.all(np.abs(deq - blk)[~normal] <= 2.0 ** -10 * sc[j] * (1 + 1e-6))
            i = int(np.argmax(np.abs(blk)))
            assert row[128 * j + i] & 0x7F == 0x7E                     # absmax -> +-448
            assert abs(abs(deq[i]) - amax) <= 2 * np.spacing(np.float32(amax))


def test_cache_write_fp8_zero_block_and_zero_rope():
    lat = torch.zeros(2, 512, dtype=torch.bfloat16)
    lat[1, 300] = 3.0
    kpe = torch.zeros(2, 64, dtype=torch.bfloat16)
    pool = np.full((2, 656), 0xFF, dtype=np.uint8)
    oracle.cache_write(lat, kpe, np.array([0, 1]), pool, 1)
    assert np.all(pool[0, :512] == 0) and np.all(pool[0, 512:528].view(np.float32) == 1.0)
    assert np.all(pool[:, 528:] == 0)                                  # bf16 zero rope bytes
    assert pool[1, 300] == 0x7E and pool[1, 512:528].view(np.float32)[2] == np.float32(3.0) / np.float32(448.0)


# --------------------------------------------------------------------- decode

def _decode_single(rows: torch.Tensor, q_lat, q_pe, scale=W.SCALE, Qt=1, page_size=16, seed=0):
    """One request whose tokens are `rows` [T, 576] bf16, stored on shuffled pages."""
    T = rows.shape[0]
    nb = max(1, -(-T // page_size))
    rng = np.random.default_rng(seed)
    perm = rng.permutation(nb + 3)[:nb]
    pool_t = torch.full(((nb + 3) * page_size, 576), float("nan"), dtype=torch.bfloat16)
    for j in range(T):
        pool_t[perm[j // page_size] * page_size + j % page_size] = rows[j]
    bt = perm.astype(np.int32)[None, :]
    out, lse = oracle.decode(q_lat, q_pe, bf16_pool(pool_t), 0, page_size, bt, np.array([T], np.int32),
                             1, Qt, q_lat.shape[-2], scale)
    return out, lse


def test_absorbed_equals_naive_attention():
    """MLA identity: with K_h = W_UK[h] c (+) k_pe and V_h = W_UV[h] c, naive
    per-head attention equals W_UV[h] applied to the absorbed latent output
    with q_lat = W_UK[h]^T q_nope. W_UK and q_nope are drawn on a coarse grid
    so that q_lat is exact in bf16 and the identity holds to fp64 rounding."""
    wl = W.tiny()
    Hq, B = wl.Hq, wl.B
    rng = np.random.default_rng(11)
    W_UK = rng.integers(-1, 2, size=(Hq, 128, 512)).astype(np.float64) / 16
    W_UV = rng.standard_normal((Hq, 128, 512)) / math.sqrt(512)
    q_nope = rng.integers(-2, 3, size=(B, Hq, 128)).astype(np.float64)
    q_lat64 = np.einsum("hkd,bhk->bhd", W_UK, q_nope)
    q_lat = torch.from_numpy(q_lat64).to(torch.bfloat16)
    assert np.array_equal(f64(q_lat), q_lat64)            # exact in bf16
    pool = wl.pool.numpy()
    out, lse = oracle.decode(q_lat, wl.q_pe, pool, 0, wl.page_size, wl.block_table, wl.seq_lens,
                             B, 1, Hq, wl.scale)
    rows = W.token_slots(wl.block_table, wl.seq_lens, wl.page_size).numpy()
    allrows = torch.from_numpy(pool.view(np.int16).reshape(-1, 576)).view(torch.bfloat16).to(torch.float64).numpy()
    qpe = f64(wl.q_pe)
    start = 0
    for b in range(B):
        T = int(wl.seq_lens[b])
        R = allrows[rows[start:start + T]]
        start += T
        c, kpe = R[:, :512], R[:, 512:]
        for h in range(Hq):
            K = np.concatenate([c @ W_UK[h].T, kpe], axis=1)        # [T, 192]
            V = c @ W_UV[h].T                                        # [T, 128]
            q = np.concatenate([q_nope[b, h], qpe[b, h]])
            s = wl.scale * (K @ q)
            p = softmax(s)
            ref_o = p @ V
            got_o = W_UV[h] @ out[b, h]
            assert np.allclose(got_o, ref_o, rtol=1e-10, atol=1e-12)
            assert abs(lse[b, h] - logsumexp(s)) < 1e-10


def test_single_token_returns_its_row():
    g = torch.Generator().manual_seed(3)
    row = torch.randn(1, 576, generator=g).to(torch.bfloat16)
    q_lat = torch.zeros(1, 2, 512, dtype=torch.bfloat16)
    q_lat[0, 0, 5] = 1.0
    q_pe = torch.zeros(1, 2, 64, dtype=torch.bfloat16)
    out, lse = _decode_single(row, q_lat, q_pe)
    assert np.array_equal(out[0, 0], f64(row[0, :512]))
    assert np.array_equal(out[0, 1], f64(row[0, :512]))
    assert lse[0, 0] == W.SCALE * float(row[0, 5]) and lse[0, 1] == 0.0


def test_identical_rows_closed_form():
    g = torch.Generator().manual_seed(4)
    T = 300
    row = torch.randn(1, 576, generator=g).to(torch.bfloat16)
    rows = row.repeat(T, 1)
    q_lat = torch.zeros(1, 1, 512, dtype=torch.bfloat16)
    q_pe = torch.zeros(1, 1, 64, dtype=torch.bfloat16)
    q_lat[0, 0, 0] = 2.0
    q_pe[0, 0, 1] = -1.0
    out, lse = _decode_single(rows, q_lat, q_pe)
    s = W.SCALE * (2.0 * float(row[0, 0]) - float(row[0, 513]))
    assert np.allclose(out[0, 0], f64(row[0, :512]), rtol=1e-13, atol=1e-13)
    assert abs(lse[0, 0] - (s + math.log(T))) < 1e-12


def test_softmax_over_tokens_one_hot_rows():
    """Token j holds the unit vector e_j, so out[j] is exactly the softmax
    weight of token j and q_lat[j] its logit: pins the scale, the softmax
    axis (tokens, not heads) and the token -> slot order."""
    T, Hq = 200, 3
    rows = torch.zeros(T, 576, dtype=torch.bfloat16)
    rows[torch.arange(T), torch.arange(T)] = 1.0
    g = torch.Generator().manual_seed(5)
    q_lat = (3 * torch.randn(1, Hq, 512, generator=g)).to(torch.bfloat16)
    q_pe = torch.randn(1, Hq, 64, generator=g).to(torch.bfloat16)   # k_pe = 0: rope adds nothing
    out, lse = _decode_single(rows, q_lat, q_pe, page_size=7)
    for h in range(Hq):
        s = W.SCALE * f64(q_lat[0, h, :T])
        assert np.allclose(out[0, h, :T], softmax(s), rtol=1e-12, atol=1e-15)
        assert np.all(out[0, h, T:] == 0)
        assert abs(out[0, h].sum() - 1.0) < 1e-12
        assert abs(lse[0, h] - logsumexp(s)) < 1e-12


def test_page_size_and_layout_invariance():
    g = torch.Generator().manual_seed(6)
    T = 513
    rows = torch.randn(T, 576, generator=g).to(torch.bfloat16)
    q_lat = torch.randn(1, 4, 512, generator=g).to(torch.bfloat16)
    q_pe = torch.randn(1, 4, 64, generator=g).to(torch.bfloat16)
    ref = _decode_single(rows, q_lat, q_pe, page_size=16, seed=1)
    for ps, seed in [(1, 2), (64, 3), (784, 4), (16, 5)]:
        o, l = _decode_single(rows, q_lat, q_pe, page_size=ps, seed=seed)
        assert np.array_equal(o, ref[0]) and np.array_equal(l, ref[1])


def test_causal_query_equals_truncated_request():
    """Query qt of a Qt-token verify step sees tokens 0..T-Qt+qt: the same as
    a one-query decode over the first T-Qt+qt+1 tokens."""
    g = torch.Generator().manual_seed(7)
    T, Qt, Hq = 90, 4, 2
    rows = torch.randn(T, 576, generator=g).to(torch.bfloat16)
    q_lat = torch.randn(Qt, Hq, 512, generator=g).to(torch.bfloat16)
    q_pe = torch.randn(Qt, Hq, 64, generator=g).to(torch.bfloat16)
    out, lse = _decode_single(rows, q_lat, q_pe, Qt=Qt)
    for qt in range(Qt):
        n = T - Qt + qt + 1
        o1, l1 = _decode_single(rows[:n], q_lat[qt:qt + 1], q_pe[qt:qt + 1])
        assert np.allclose(out[qt], o1[0], rtol=1e-13, atol=1e-14)
        assert np.allclose(lse[qt], l1[0], rtol=0, atol=1e-13)


def test_short_and_empty_requests():
    """T=0: every query is (0, -inf). T=2 < Qt=4: queries 0 and 1 see nothing."""
    g = torch.Generator().manual_seed(8)
    rows = torch.randn(8, 576, generator=g).to(torch.bfloat16)
    pool = bf16_pool(rows)
    bt = np.array([[0], [-1]], dtype=np.int32)
    q_lat = torch.randn(8, 2, 512, generator=g).to(torch.bfloat16)
    q_pe = torch.randn(8, 2, 64, generator=g).to(torch.bfloat16)
    out, lse = oracle.decode(q_lat, q_pe, pool, 0, 8, bt, np.array([2, 0], np.int32), 2, 4, 2, W.SCALE)
    assert np.all(out[0:2] == 0) and np.all(np.isneginf(lse[0:2]))
    assert np.all(np.isfinite(lse[2:4]))
    assert np.all(out[4:8] == 0) and np.all(np.isneginf(lse[4:8]))
    assert np.array_equal(out[2, 0], f64(rows[0, :512]))          # sees only token 0


def test_rope_free_invariance_and_teeth():
    """q_pe = 0 makes k_pe irrelevant (exactly); with q_pe != 0 a garbage k_pe
    must change the result (the test has teeth)."""
    g = torch.Generator().manual_seed(9)
    T = 150
    rows = torch.randn(T, 576, generator=g).to(torch.bfloat16)
    junk = rows.clone()
    junk[:, 512:] = (100 * torch.randn(T, 64, generator=g)).to(torch.bfloat16)
    q_lat = torch.randn(1, 2, 512, generator=g).to(torch.bfloat16)
    zero = torch.zeros(1, 2, 64, dtype=torch.bfloat16)
    a = _decode_single(rows, q_lat, zero)
    b = _decode_single(junk, q_lat, zero)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    q_pe = torch.randn(1, 2, 64, generator=g).to(torch.bfloat16)
    c = _decode_single(rows, q_lat, q_pe)
    d = _decode_single(junk, q_lat, q_pe)
    assert np.abs(c[0] - d[0]).max() > 1e-2


def test_slots_above_int32_wrap():
    """Rows stored above slot 2^31/576 are read at their own address (64-bit
    offsets). A sparse memory map keeps the 4.3 GB pool cheap."""
    first = W.INT32_WRAP_SLOT - 5
    nslots = first + 40
    with tempfile.TemporaryDirectory() as d:
        pool = np.memmap(os.path.join(d, "pool"), dtype=np.uint8, mode="w+", shape=(nslots, 1152))
        g = torch.Generator().manual_seed(10)
        rows = torch.randn(40, 576, generator=g).to(torch.bfloat16)
        pool[first:first + 40] = bf16_pool(rows)
        q_lat = torch.zeros(1, 1, 512, dtype=torch.bfloat16)
        q_pe = torch.zeros(1, 1, 64, dtype=torch.bfloat16)
        # page size 1: block id = slot; check single-token requests one by one
        for j in [0, 4, 5, 6, 39]:
            slot = first + j
            bt = np.array([[slot]], dtype=np.int32)
            out, _ = oracle.decode(q_lat, q_pe, np.asarray(pool), 0, 1, bt, np.array([1], np.int32),
                                   1, 1, 1, W.SCALE)
            assert np.array_equal(out[0, 0], f64(rows[j, :512]))
        del pool


# ---------------------------------------------------------------------- merge

def test_merge_equals_single_pass():
    """Decoding disjoint token ranges separately and merging the partial
    (out, lse) equals one pass over all tokens; empty parts carry no weight."""
    g = torch.Generator().manual_seed(12)
    T, Hq = 700, 3
    rows = torch.randn(T, 576, generator=g).to(torch.bfloat16)
    q_lat = torch.randn(1, Hq, 512, generator=g).to(torch.bfloat16)
    q_pe = torch.randn(1, Hq, 64, generator=g).to(torch.bfloat16)
    ref_o, ref_l = _decode_single(rows, q_lat, q_pe)
    cuts = [0, 1, 129, 129, 500, T]           # includes an empty part
    po, pl = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        if b > a:
            o, l = _decode_single(rows[a:b], q_lat, q_pe)
        else:
            o, l = np.zeros((1, Hq, 512)), np.full((1, Hq), -np.inf)
        po.append(o[0])
        pl.append(l[0])
    po = np.stack(po).astype(np.float32)
    pl = np.stack(pl).astype(np.float32)
    mo, ml = oracle.merge(po, pl)
    # partials were stored in fp32: compare at fp32 resolution
    assert np.allclose(mo, ref_o[0], rtol=1e-5, atol=1e-6)
    assert np.allclose(ml, ref_l[0], rtol=0, atol=1e-5)


def test_merge_closed_forms():
    o = np.random.default_rng(0).standard_normal((2, 3, 512)).astype(np.float32)
    lse = np.array([[1.5, -np.inf, 0.25], [1.5, -np.inf, -np.inf]], dtype=np.float32)
    mo, ml = oracle.merge(o, lse)
    assert np.allclose(mo[0], (o[0, 0].astype(np.float64) + o[1, 0]) / 2, rtol=1e-12, atol=1e-12)
    assert abs(ml[0] - (1.5 + math.log(2))) < 1e-12
    assert np.all(mo[1] == 0) and np.isneginf(ml[1])                   # all -inf -> (0, -inf)
    assert np.array_equal(mo[2], o[0, 2].astype(np.float64)) and ml[2] == np.float32(0.25)
