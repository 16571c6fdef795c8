"""GLA-g2 (qwen-mla-vllm README: the latent split into two head groups; at
tensor-parallel size 1 it runs like plain MLA). With absorbed queries a head
of group g has q_lat zero outside its group's 256 latent dims, so plain MLA
decode computes GLA-g2 exactly: each head's output is its group's half of the
512-wide result. Pinned on the oracle by an independent per-group numpy
computation; the GPU path is checked on GLA-shaped queries."""
import math

import numpy as np
import pytest
import torch

import oracle

D, P, W = 512, 64, 576


def _gla_reference(vals, bt, seq_lens, q_grp, groups, page_size, scale):
    """Per group g: scores from q_g . c[g*256:(g+1)*256] + q_pe . k_pe, softmax over
    the tokens, output sum p * c[g half] (256 values); fp64, from the definition."""
    B, H = q_grp.shape[0], q_grp.shape[1]
    out = np.zeros((B, H, 256))
    lse = np.zeros((B, H))
    for b, T in enumerate(seq_lens):
        rows = np.array([bt[b, j // page_size] * page_size + j % page_size for j in range(T)])
        c = vals[rows]
        for h in range(H):
            g = groups[h]
            lat = c[:, 256 * g:256 * (g + 1)]
            s = scale * (lat @ q_grp[b, h, :256] + c[:, D:] @ q_grp[b, h, 256:])
            m = s.max()
            p = np.exp(s - m)
            out[b, h] = (p[:, None] * lat).sum(0) / p.sum()
            lse[b, h] = m + math.log(p.sum())
    return out, lse


def _gla_case(seed, seq_lens, H, page_size):
    rng = np.random.default_rng(seed)
    pages = [-(-t // page_size) for t in seq_lens]
    nb = sum(pages) + 2
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.full((len(seq_lens), max(pages)), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[k:k + n]
        k += n
    vals = torch.from_numpy(rng.standard_normal((nb * page_size, W)).astype(np.float32)).to(torch.bfloat16)
    pool = vals.view(torch.int16).numpy().view(np.uint8).reshape(nb * page_size, 2 * W).copy()
    groups = np.array([h * 2 // H for h in range(H)])  # first half of the heads: group 0
    q_grp = torch.from_numpy(rng.standard_normal((len(seq_lens), H, 256 + P)).astype(np.float32)).to(torch.bfloat16)
    # the absorbed 512-wide query: the group's 256 values in its half, zeros elsewhere
    q_lat = torch.zeros((len(seq_lens), H, D), dtype=torch.bfloat16)
    for h in range(H):
        g = groups[h]
        q_lat[:, h, 256 * g:256 * (g + 1)] = q_grp[:, h, :256]
    q_pe = q_grp[:, :, 256:].contiguous()
    return pool, vals.double().numpy(), bt, groups, q_grp, q_lat, q_pe


def test_gla_g2_is_plain_mla_with_group_padded_queries():
    seq_lens, H, ps = [37, 200, 5], 8, 16
    pool, vals, bt, groups, q_grp, q_lat, q_pe = _gla_case(1, seq_lens, H, ps)
    scale = 1 / math.sqrt(192)
    o, l = oracle.decode(q_lat, q_pe, pool, 0, ps, bt, np.array(seq_lens, dtype=np.int32), len(seq_lens), 1, H, scale)
    ro, rl = _gla_reference(vals, bt, seq_lens, q_grp.double().numpy(), groups, ps, scale)
    for h in range(H):
        g = groups[h]
        assert np.abs(o[:, h, 256 * g:256 * (g + 1)] - ro[:, h]).max() < 1e-12
    assert np.abs(l - rl).max() < 1e-12


@pytest.mark.gpu
def test_gla_g2_shaped_queries_on_the_gpu():
    import mla_latent_kv_cache_gb300 as m
    from mla_latent_kv_cache_gb300 import build as mbuild
    mbuild.build()
    m.load()
    dev = torch.device("cuda:0")
    seq_lens, H, ps = [700, 1, 3000, 129], 16, 16
    pool, vals, bt, groups, q_grp, q_lat, q_pe = _gla_case(2, seq_lens, H, ps)
    scale = 1 / math.sqrt(192)
    out, lse, _ = m.decode(q_lat.to(dev), q_pe.to(dev), torch.from_numpy(pool).to(dev), 0, ps,
                           torch.from_numpy(bt).to(dev), torch.tensor(seq_lens, dtype=torch.int32, device=dev), 1,
                           scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ro, rl = _gla_reference(vals, bt, seq_lens, q_grp.double().numpy(), groups, ps, scale)
    o = out.cpu().numpy().astype(np.float64)
    for h in range(H):
        g = groups[h]
        ref = ro[:, h]
        assert np.all(np.abs(o[:, h, 256 * g:256 * (g + 1)] - ref) <= 1e-2 + 2e-2 * np.abs(ref))
    assert np.abs(lse.cpu().numpy() - rl).max() <= 1e-3
