"""Pins of the oracle's verify step with a length of its own per request
(``oracle.decode_varlen``): an independent fp64 brute force of the definition
on tiny inputs, agreement with the uniform-length decode, the causal rule per
request, and queries with nothing visible."""
import math

import numpy as np
import torch

import oracle

D, P, W = 512, 64, 576


def _tiny(seed, seq_lens, q_lens, Hq, page_size):
    """bf16 pool [slots, 576], shuffled block table, queries for sum(q_lens) tokens."""
    rng = np.random.default_rng(seed)
    pages = [-(-t // page_size) for t in seq_lens]
    nb = sum(pages) + 3
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.full((len(seq_lens), max(pages) + 1), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[k:k + n]
        k += n
    vals = torch.from_numpy(rng.standard_normal((nb * page_size, W)).astype(np.float32)).to(torch.bfloat16)
    pool = vals.view(torch.int16).numpy().view(np.uint8).reshape(nb * page_size, 2 * W).copy()
    R = sum(q_lens)
    q = torch.from_numpy(rng.standard_normal((R, Hq, W)).astype(np.float32)).to(torch.bfloat16)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    return pool, vals.double().numpy(), bt, q, cu


def _brute(vals, bt, seq_lens, q, cu, Hq, page_size, scale):
    R = int(cu[-1])
    out = np.zeros((R, Hq, D))
    lse = np.full((R, Hq), -np.inf)
    qd = q.double().numpy()
    for b, T in enumerate(seq_lens):
        Qt = int(cu[b + 1] - cu[b])
        for qt in range(Qt):
            r = int(cu[b]) + qt
            nvis = T - Qt + qt + 1
            if nvis <= 0:
                continue
            rows = np.array([bt[b, j // page_size] * page_size + j % page_size for j in range(nvis)])
            c = vals[rows]                      # [nvis, 576]
            for h in range(Hq):
                s = scale * (c @ qd[r, h])      # q_lat . c + q_pe . k_pe in one dot
                m = s.max()
                p = np.exp(s - m)
                out[r, h] = (p[:, None] * c[:, :D]).sum(0) / p.sum()
                lse[r, h] = m + math.log(p.sum())
    return out, lse


def test_brute_force_definition():
    seq_lens, q_lens, Hq, ps = [5, 9, 4, 1], [1, 3, 2, 1], 2, 2
    pool, vals, bt, q, cu = _tiny(1, seq_lens, q_lens, Hq, ps)
    scale = 1 / math.sqrt(192)
    o, l = oracle.decode_varlen(q[:, :, :D].contiguous(), q[:, :, D:].contiguous(), pool, 0, ps, bt,
                                np.array(seq_lens, dtype=np.int32), cu, Hq, scale)
    bo, bl = _brute(vals, bt, seq_lens, q, cu, Hq, ps, scale)
    assert np.abs(o - bo).max() < 1e-12 and np.abs(l - bl).max() < 1e-12


def test_uniform_lengths_equal_the_uniform_decode():
    seq_lens, Qt, Hq, ps = [40, 7, 130], 3, 4, 16
    pool, _, bt, q, cu = _tiny(2, seq_lens, [Qt] * 3, Hq, ps)
    scale = 0.07
    ql, qp = q[:, :, :D].contiguous(), q[:, :, D:].contiguous()
    sl = np.array(seq_lens, dtype=np.int32)
    o1, l1 = oracle.decode_varlen(ql, qp, pool, 0, ps, bt, sl, cu, Hq, scale)
    o2, l2 = oracle.decode(ql, qp, pool, 0, ps, bt, sl, 3, Qt, Hq, scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_each_request_is_its_own_verify_step():
    seq_lens, q_lens, Hq, ps = [33, 70, 5, 64], [2, 1, 4, 3], 3, 8
    pool, _, bt, q, cu = _tiny(3, seq_lens, q_lens, Hq, ps)
    ql, qp = q[:, :, :D].contiguous(), q[:, :, D:].contiguous()
    sl = np.array(seq_lens, dtype=np.int32)
    o, l = oracle.decode_varlen(ql, qp, pool, 0, ps, bt, sl, cu, Hq, 0.05)
    for b, Qt in enumerate(q_lens):
        r0, r1 = int(cu[b]), int(cu[b + 1])
        ob, lb = oracle.decode(ql[r0:r1], qp[r0:r1], pool, 0, ps, bt[b:b + 1], sl[b:b + 1], 1, Qt, Hq, 0.05)
        assert np.array_equal(o[r0:r1], ob) and np.array_equal(l[r0:r1], lb)


def test_queries_with_nothing_visible_are_zero_and_minus_inf():
    # T = 2 < q_len = 4: queries 0 and 1 of the request see no token
    seq_lens, q_lens, Hq, ps = [2, 6], [4, 1], 2, 4
    pool, _, bt, q, cu = _tiny(4, seq_lens, q_lens, Hq, ps)
    o, l = oracle.decode_varlen(q[:, :, :D].contiguous(), q[:, :, D:].contiguous(), pool, 0, ps, bt,
                                np.array(seq_lens, dtype=np.int32), cu, Hq, 0.1)
    assert np.all(o[0:2] == 0) and np.all(l[0:2] == -np.inf)
    assert np.all(np.isfinite(l[2:]))


def test_a_request_that_verifies_no_token_adds_no_rows():
    # the verify step of request 1 is empty (cu_q_lens repeats a value): the
    # other requests' rows are those of a batch without it
    seq_lens, q_lens, Hq, ps = [30, 50, 17], [2, 0, 3], 2, 8
    pool, _, bt, q, cu = _tiny(5, seq_lens, q_lens, Hq, ps)
    ql, qp = q[:, :, :D].contiguous(), q[:, :, D:].contiguous()
    sl = np.array(seq_lens, dtype=np.int32)
    o, l = oracle.decode_varlen(ql, qp, pool, 0, ps, bt, sl, cu, Hq, 0.08)
    assert o.shape[0] == 5 and l.shape[0] == 5
    keep = [0, 2]
    cu2 = np.array([0, 2, 5], dtype=np.int32)
    o2, l2 = oracle.decode_varlen(ql, qp, pool, 0, ps, bt[keep], sl[keep], cu2, Hq, 0.08)
    assert np.array_equal(o, o2) and np.array_equal(l, l2)
