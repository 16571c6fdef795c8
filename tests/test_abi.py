"""The C-ABI library loads and exports what include/mla.h declares; host-side
argument checks reject bad calls before any GPU work (no device needed)."""
import ctypes
import os
import re

import pytest

import mla_latent_kv_cache_gb300 as m
from mla_latent_kv_cache_gb300 import build as mbuild

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mla.h")


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return m.load()


def declared_functions():
    txt = open(HDR).read()
    return sorted(set(re.findall(r"MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", txt)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["mla_cache_write", "mla_decode", "mla_merge_lse", "mla_decode_workspace_bytes"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_status_strings(lib):
    assert m.mla_status_string(0) == "ok"
    assert "invalid" in m.mla_status_string(-1)
    assert m.mla_row_bytes(0) == 1152 and m.mla_row_bytes(1) == 656 and m.mla_row_bytes(7) == 0


def test_host_validation_rejects_bad_arguments(lib):
    # every one of these is rejected on the host before any CUDA call
    assert lib.mla_cache_write(None, 512, None, 64, None, -1, None, 10, 0, None, None) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_cache_write(None, 512, None, 64, None, 0, None, 10, 0, None, None) == m.MLA_OK  # nothing to do
    assert lib.mla_cache_write(16, 512, 16, 64, 16, 4, 16, 10, 5, None, None) == m.MLA_ERR_INVALID_ARG  # kind
    assert lib.mla_cache_write(16, 500, 16, 64, 16, 4, 16, 10, 0, None, None) == m.MLA_ERR_INVALID_ARG  # stride
    assert lib.mla_cache_write(8, 512, 16, 64, 16, 4, 16, 10, 0, None, None) == m.MLA_ERR_INVALID_ARG   # alignment
    assert lib.mla_cache_write(16, 512, 16, 64, 16, 4, 16, 10, 0, 18, None) == m.MLA_ERR_INVALID_ARG    # status word
    args = [16, 16, 16, 0, 100, 16, 16, 4, 16, 2, 1, 8, 0.1, 16, 0, 16, 256, 1 << 20, 0, None]
    bad = list(args)
    bad[9] = 0                                                     # B = 0
    assert lib.mla_decode(*bad) == m.MLA_ERR_INVALID_ARG
    bad = list(args)
    bad[5] = 0                                                     # page_size = 0
    assert lib.mla_decode(*bad) == m.MLA_ERR_INVALID_ARG
    bad = list(args)
    bad[16] = 264                                                  # workspace not 256-aligned
    assert lib.mla_decode(*bad) == m.MLA_ERR_INVALID_ARG
    bad = list(args)
    bad[3] = 9                                                     # cache kind
    assert lib.mla_decode(*bad) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_merge_lse(16, 16, -1, 4, 16, 0, 16, None) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_merge_lse(16, 16, 2, 0, 16, 0, 16, None) == m.MLA_OK
    # other latent widths: only 256 / 512 / 768 / 1792
    assert lib.mla_cache_write_latent(16, 384, 16, 64, 16, 4, 16, 10, 384, None, None) == m.MLA_ERR_UNSUPPORTED
    assert lib.mla_cache_write_latent(16, 200, 16, 64, 16, 4, 16, 10, 256, None, None) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_decode_latent_workspace_bytes(4, 1, 16, 300, 8) == 0
    assert lib.mla_decode_latent_workspace_bytes(4, 1, 16, 768, 8) > lib.mla_decode_workspace_bytes(4, 1, 16, 8)
    lat = [16, 16, 16, 384, 100, 16, 16, 4, 16, 2, 1, 8, 0.1, 16, 0, 16, 256, 1 << 20, 0, None]
    assert lib.mla_decode_latent(*lat) == m.MLA_ERR_UNSUPPORTED
    assert lib.mla_static_scratch_status(None, 12, None) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_static_scratch_status(16, 0, None) == m.MLA_ERR_INVALID_ARG
    assert lib.mla_static_scratch_status(16, 13, None) == m.MLA_ERR_INVALID_ARG
    # mla_decode_varlen(q_lat, q_pe, total_q, cache, kind, num_slots, page_size, bt, bt_stride, seq_lens, cu_q, B,
    #                   max_q_len, Hq, scale, out, out_dtype, lse, ws, ws_bytes, num_ctas, stream)
    v = [16, 16, 6, 16, 0, 100, 16, 16, 4, 16, 16, 2, 3, 8, 0.1, 16, 0, 16, 256, 1 << 20, 0, None]
    assert lib.mla_decode_varlen(*(v[:10] + [None] + v[11:])) == m.MLA_ERR_INVALID_ARG  # no prefix sums
    assert lib.mla_decode_varlen(*(v[:2] + [0] + v[3:])) == m.MLA_ERR_INVALID_ARG       # no query tokens
    assert lib.mla_decode_varlen(*(v[:12] + [0] + v[13:])) == m.MLA_ERR_INVALID_ARG     # max_q_len = 0
    # mla_gather_upconvert(cache, num_slots, page_size, block_table, bt_stride, cu, B, num_rows, dst, dst_stride, stream)
    g = [16, 100, 16, 16, 4, 16, 2, 10, 16, 576, None]
    assert lib.mla_gather_upconvert(*(g[:6] + [0] + g[7:])) == m.MLA_OK             # B = 0: nothing to do
    assert lib.mla_gather_upconvert(*(g[:7] + [0] + g[8:])) == m.MLA_OK             # no rows: nothing to do
    assert lib.mla_gather_upconvert(*(g[:2] + [0] + g[3:])) == m.MLA_ERR_INVALID_ARG  # page_size
    assert lib.mla_gather_upconvert(*(g[:9] + [512] + g[10:])) == m.MLA_ERR_INVALID_ARG  # rows narrower than 576
    assert lib.mla_gather_upconvert(*(g[:9] + [580] + g[10:])) == m.MLA_ERR_INVALID_ARG  # stride not a multiple of 8
    assert lib.mla_gather_upconvert(*(g[:8] + [24] + g[9:])) == m.MLA_ERR_INVALID_ARG   # dst not 16-byte aligned
    assert lib.mla_gather_upconvert(*([None] + g[1:])) == m.MLA_ERR_INVALID_ARG       # no cache
    assert lib.mla_gather_upconvert(*(g[:6] + [-1] + g[7:])) == m.MLA_ERR_INVALID_ARG  # B < 0


def test_workspace_size_formula(lib):
    # header + [CTAs][16] int32 status records + [groups][CTAs + B][64] lse
    # + [groups][CTAs + B][64][512] partial outputs, CTAs = max(2, num_ctas),
    # each part rounded up to 256 bytes
    def up(x):
        return -(-x // 256) * 256
    for B, q, H, G in [(2, 1, 8, 152), (64, 1, 16, 152), (128, 4, 16, 152), (3, 1, 80, 7), (5, 1, 16, 1)]:
        gy = -(-(H * q) // 64)
        ctas = max(2, G)
        slots = gy * (ctas + B) * 64
        rec_b = up(ctas * gy * 16 * 4)
        assert m.mla_decode_workspace_bytes(B, q, H, G) == 256 + rec_b + up(slots * 4) + slots * 512 * 4
    assert lib.mla_decode_workspace_bytes(0, 1, 8, 4) == 0
