"""mla_decode_static_scratch (the library's static device scratch as the
decode workspace) against mla_decode with a caller-allocated workspace.

Collected last (file name) so it also runs after every other GPU test has
used the device; it passes on its own as well."""
import pytest
import torch

import mla_latent_kv_cache_gb300 as m
from mla_latent_kv_cache_gb300 import build as mbuild
from mla_latent_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
MLA_ERR_SCRATCH_LIMIT = -5
MLA_STATIC_SCRATCH_BYTES = 64 << 20


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mbuild.build()
    m.load()
    torch.cuda.set_device(DEV)
    yield


def _outputs(wl, out_dtype):
    R = wl.seq_lens.numel() * wl.Qt
    Hq = wl.q_lat.shape[-2]
    return (torch.full((R, Hq, 512), float("nan"), dtype=out_dtype, device=DEV),
            torch.full((R, Hq), float("nan"), dtype=torch.float32, device=DEV))


def _reference(wl, out_dtype):
    out, lse = _outputs(wl, out_dtype)
    ws = torch.empty(m.mla_decode_workspace_bytes(wl.seq_lens.numel(), wl.Qt, wl.q_lat.shape[-2]),
                     dtype=torch.uint8, device=DEV)
    m.mla_decode(wl.q_lat, wl.q_pe, wl.pool, wl.kind, wl.page_size, wl.block_table, wl.seq_lens, wl.Qt, wl.scale,
                 out, lse, ws)
    return out, lse


def _reference_ctas(wl, out_dtype, num_ctas):
    out, lse = _outputs(wl, out_dtype)
    ws = torch.empty(m.mla_decode_workspace_bytes(wl.seq_lens.numel(), wl.Qt, wl.q_lat.shape[-2], num_ctas),
                     dtype=torch.uint8, device=DEV)
    m.mla_decode(wl.q_lat, wl.q_pe, wl.pool, wl.kind, wl.page_size, wl.block_table, wl.seq_lens, wl.Qt, wl.scale,
                 out, lse, ws, num_ctas)
    return out, lse


def _static(wl, out_dtype, num_ctas=0):
    out, lse = _outputs(wl, out_dtype)
    m.mla_decode_static_scratch(wl.q_lat, wl.q_pe, wl.pool, wl.kind, wl.page_size, wl.block_table, wl.seq_lens,
                                wl.Qt, wl.scale, out, lse, num_ctas)
    return out, lse


def test_two_calls_in_a_row_match_the_workspace_entry():
    # two different workloads back to back on one stream: the second call
    # reuses the scratch the first one left behind
    wa = W.tiny(device=DEV)
    wb = W.batched(device=DEV)
    for wl in (wa, wb):
        m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
    ref_a = _reference(wa, torch.float32)
    ref_b = _reference(wb, torch.bfloat16)
    got_a = _static(wa, torch.float32)
    got_b = _static(wb, torch.bfloat16)
    torch.cuda.synchronize()
    for got, ref in ((got_a, ref_a), (got_b, ref_b)):
        assert torch.equal(got[0], ref[0])
        assert torch.equal(got[1], ref[1])


def test_repeated_call_is_identical():
    wl = W.tiny(device=DEV, seed=7)
    m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
    first = _static(wl, torch.float32)
    second = _static(wl, torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(first[0], second[0]) and torch.equal(first[1], second[1])
    assert torch.isfinite(first[0]).all()


def test_every_bench_workload_fits_the_scratch():
    # batched, long, MTP verify and fp8 shapes at one CTA per SM
    for B, q, Hq in [(64, 1, 16), (4, 1, 32), (128, 4, 16), (64, 1, 64)]:
        assert 0 < m.mla_decode_workspace_bytes(B, q, Hq) <= MLA_STATIC_SCRATCH_BYTES


def test_oversized_call_is_rejected_before_any_launch():
    B, Hq = 4096, 16
    assert m.mla_decode_workspace_bytes(B, 1, Hq) > MLA_STATIC_SCRATCH_BYTES
    q_lat = torch.zeros((B, Hq, 512), dtype=torch.bfloat16, device=DEV)
    q_pe = torch.zeros((B, Hq, 64), dtype=torch.bfloat16, device=DEV)
    pool = torch.zeros((16, 1152), dtype=torch.uint8, device=DEV)
    bt = torch.zeros((B, 1), dtype=torch.int32, device=DEV)
    sl = torch.zeros((B,), dtype=torch.int32, device=DEV)
    out = torch.zeros((B, Hq, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.zeros((B, Hq), dtype=torch.float32, device=DEV)
    with pytest.raises(m.MlaError) as e:
        m.mla_decode_static_scratch(q_lat, q_pe, pool, 0, 16, bt, sl, 1, 0.1, out, lse)
    assert e.value.status == MLA_ERR_SCRATCH_LIMIT
    assert "static decode scratch" in m.mla_status_string(MLA_ERR_SCRATCH_LIMIT)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0  # nothing ran


def test_other_kernels_reuse_the_scratch():
    # an fp8 pool at 64 query rows (the cluster kernel with its expand warps),
    # split over a CTA count of its own, after a bf16 call that left a larger
    # partial-slot layout behind; then odd page sizes (load/convert warps)
    wb = W.batched(device=DEV)
    w8 = W.make("fp8_small", B=3, Hq=64, Qt=1, page_size=64, seq_lens=[3000, 1, 4500], kind=W.KIND_FP8,
                write_all=True, seed=31, device=DEV)
    wo = W.make("odd_pages", B=4, Hq=16, Qt=4, page_size=3, seq_lens=[0, 2, 900, 2100], seed=32, device=DEV)
    for wl in (wb, w8, wo):
        m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
    ref = [_reference(wb, torch.bfloat16), _reference_ctas(w8, torch.float32, 12),
           _reference_ctas(wo, torch.float32, 10)]
    got = [_static(wb, torch.bfloat16), _static(w8, torch.float32, 12), _static(wo, torch.float32, 10)]
    torch.cuda.synchronize()
    for (go, gl), (ro, rl) in zip(got, ref):
        assert torch.equal(go, ro) and torch.equal(gl, rl)
    assert m.static_scratch_status_words()[0] == 0


def test_status_words_of_a_static_call():
    # a bounded wait that gives up inside a static-scratch call is reported
    # through mla_static_scratch_status; the next call clears it
    wl = W.make("hold_static", B=3, Hq=16, Qt=1, page_size=16, seq_lens=[700, 1500, 300], seed=93, device=DEV)
    m.mla_cache_write(wl.w_latent, wl.w_k_pe, wl.w_slots, wl.pool, wl.kind)
    ref = _reference(wl, torch.float32)
    m.test_hold_next_decode()
    _static(wl, torch.float32)
    torch.cuda.synchronize()
    words = m.static_scratch_status_words()
    assert words[0] & 1 and words[1] != 0, words
    got = _static(wl, torch.float32)
    torch.cuda.synchronize()
    assert m.static_scratch_status_words()[0] == 0
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
