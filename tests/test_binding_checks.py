"""The Python binding's own argument checks (no GPU needed).

The library validates sizes, pointers and alignment on the host but cannot
tell a host tensor from a device one, nor how large a caller's output is; the
binding checks both before it calls the library and raises
MlaError(MLA_ERR_INVALID_ARG). Here host tensors must be refused outright;
the shape, dtype and size checks are then exercised with the device test
replaced (any tensor counts as on the device) and a stand-in library that
records what reached it."""
import pytest
import torch

import mla_latent_kv_cache_gb300 as m


class _Recorder:
    """Stands in for the compiled library: every entry point returns MLA_OK
    and records its arguments."""

    def __init__(self, real):
        self.calls = []
        self.real = real

    def __getattr__(self, name):
        if name in ("mla_row_bytes", "mla_status_string"):
            return getattr(self.real, name)

        def call(*args):
            self.calls.append((name, args))
            return m.MLA_OK
        return call


@pytest.fixture
def fake(monkeypatch):
    rec = _Recorder(m.load())  # the real library answers mla_row_bytes and the status strings
    monkeypatch.setattr(m, "_is_cuda", lambda t: isinstance(t, torch.Tensor))
    monkeypatch.setattr(m, "load", lambda: rec)
    monkeypatch.setattr(m, "_stream", lambda s: 0)
    return rec


def _decode_inputs(B=2, q_len=2, Hq=8, D=512, out_dtype=torch.bfloat16):
    R = B * q_len
    return dict(
        q_lat=torch.zeros((R, Hq, D), dtype=torch.bfloat16),
        q_pe=torch.zeros((R, Hq, 64), dtype=torch.bfloat16),
        cache=torch.zeros((64, 2 * (D + 64)), dtype=torch.uint8),
        block_table=torch.zeros((B, 4), dtype=torch.int32),
        seq_lens=torch.full((B,), 10, dtype=torch.int32),
        out=torch.empty((R, Hq, D), dtype=out_dtype),
        lse=torch.empty((R, Hq), dtype=torch.float32),
        workspace=torch.empty((1 << 16,), dtype=torch.uint8),
    )


def _decode(a, q_len=2, **over):
    a = {**a, **over}
    m.mla_decode(a["q_lat"], a["q_pe"], a["cache"], 0, 16, a["block_table"], a["seq_lens"], q_len, 0.1, a["out"],
                 a["lse"], a["workspace"])


def _refused(fn, words):
    with pytest.raises(m.MlaError) as e:
        fn()
    assert e.value.status == m.MLA_ERR_INVALID_ARG
    assert words in str(e.value), str(e.value)


def test_host_tensors_are_refused_before_the_library_is_called():
    a = _decode_inputs()
    _refused(lambda: _decode(a), "must be a CUDA tensor")
    _refused(lambda: m.mla_cache_write(torch.zeros((1, 512), dtype=torch.bfloat16),
                                       torch.zeros((1, 64), dtype=torch.bfloat16), torch.zeros(1, dtype=torch.int64),
                                       torch.zeros((4, 1152), dtype=torch.uint8)), "must be a CUDA tensor")
    _refused(lambda: m.mla_merge_lse(torch.zeros((2, 3, 512)), torch.zeros((2, 3)), torch.empty((3, 512))),
             "must be a CUDA tensor")
    _refused(lambda: m.mla_gather_upconvert(torch.zeros((16, 656), dtype=torch.uint8), 16,
                                            torch.zeros((1, 1), dtype=torch.int32),
                                            torch.tensor([0, 4], dtype=torch.int32),
                                            torch.empty((4, 576), dtype=torch.bfloat16)), "must be a CUDA tensor")


def test_decode_reaches_the_library_with_consistent_arguments(fake):
    a = _decode_inputs()
    _decode(a)
    name, args = fake.calls[-1]
    assert name == "mla_decode"
    assert args[4] == 64 * 1152 // 1152          # num_slots from the pool's bytes
    assert args[9:12] == (2, 2, 8)                # B, q_len, Hq
    assert args[14] == m.MLA_OUT_BF16
    _decode(a, out=torch.empty((4, 8, 512), dtype=torch.float32))
    assert fake.calls[-1][1][14] == m.MLA_OUT_F32


def test_decode_argument_checks(fake):
    a = _decode_inputs()
    _refused(lambda: _decode(a, out=torch.empty((3, 8, 512), dtype=torch.bfloat16)), "the call writes")
    _refused(lambda: _decode(a, out=torch.empty((4, 8, 512), dtype=torch.float16)), "bf16 or fp32")
    _refused(lambda: _decode(a, out=torch.empty((8, 4, 512), dtype=torch.bfloat16).transpose(0, 1)), "contiguous")
    _refused(lambda: _decode(a, lse=torch.empty((3, 8), dtype=torch.float32)), "lse")
    _refused(lambda: _decode(a, lse=torch.empty((4, 8), dtype=torch.float64)), "lse")
    _refused(lambda: _decode(a, block_table=torch.zeros((1, 4), dtype=torch.int32)), "rows for 2 requests")
    _refused(lambda: _decode(a, block_table=torch.zeros((2, 4), dtype=torch.int64)), "block_table")
    _refused(lambda: _decode(a, block_table=torch.zeros((4, 2), dtype=torch.int32).t()), "block_table")
    _refused(lambda: _decode(a, seq_lens=torch.full((2,), 10, dtype=torch.int64)), "seq_lens")
    _refused(lambda: _decode(a, q_len=3), "rows of 512")
    _refused(lambda: _decode(a, q_lat=a["q_lat"].float()), "bf16")
    _refused(lambda: _decode(a, cache=torch.zeros((1152, 64), dtype=torch.uint8).t()), "cache")
    assert not fake.calls  # nothing reached the library


def test_latent_and_static_scratch_checks(fake):
    a = _decode_inputs(D=768)
    m.mla_decode_latent(a["q_lat"], a["q_pe"], a["cache"], 768, 16, a["block_table"], a["seq_lens"], 2, 0.1,
                        a["out"], a["lse"], a["workspace"])
    assert fake.calls[-1][0] == "mla_decode_latent"
    _refused(lambda: m.mla_decode_latent(a["q_lat"], a["q_pe"], a["cache"], 768, 16, a["block_table"],
                                         a["seq_lens"], 2, 0.1, a["out"][:3], a["lse"], a["workspace"]),
             "the call writes")
    b = _decode_inputs()
    m.mla_decode_static_scratch(b["q_lat"], b["q_pe"], b["cache"], 0, 16, b["block_table"], b["seq_lens"], 2, 0.1,
                                b["out"], b["lse"])
    assert fake.calls[-1][0] == "mla_decode_static_scratch"
    _refused(lambda: m.mla_decode_static_scratch(b["q_lat"], b["q_pe"], b["cache"], 0, 16, b["block_table"],
                                                 b["seq_lens"], 2, 0.1, b["out"], b["lse"][:1]), "lse")


def test_varlen_checks(fake):
    a = _decode_inputs()  # 4 query tokens
    cu = torch.tensor([0, 1, 4], dtype=torch.int32)

    def call(**over):
        x = {**a, "cu": cu, **over}
        m.mla_decode_varlen(x["q_lat"], x["q_pe"], x["cache"], 0, 16, x["block_table"], x["seq_lens"], x["cu"], 3,
                            0.1, x["out"], x["lse"], x["workspace"])

    call()
    name, args = fake.calls[-1]
    assert name == "mla_decode_varlen" and args[2] == 4 and args[5] == 64  # total_q, num_slots
    _refused(lambda: call(cu=torch.tensor([0, 4], dtype=torch.int32)), "3 entries")
    _refused(lambda: call(cu=cu.long()), "cu_q_lens")
    _refused(lambda: call(out=a["out"][:3]), "the call writes")
    _refused(lambda: call(q_pe=a["q_pe"][:3]), "q_pe")


def test_cache_write_checks(fake):
    lat = torch.zeros((3, 512), dtype=torch.bfloat16)
    kpe = torch.zeros((3, 64), dtype=torch.bfloat16)
    slots = torch.tensor([0, 5, -1], dtype=torch.int64)
    pool = torch.zeros((8, 1152), dtype=torch.uint8)
    m.mla_cache_write(lat, kpe, slots, pool, 0)
    assert fake.calls[-1][0] == "mla_cache_write" and fake.calls[-1][1][7] == 8  # num_slots
    wide = torch.zeros((3, 640), dtype=torch.bfloat16)
    m.mla_cache_write(wide[:, :512], wide[:, 576:], slots, pool, 0)  # row-strided views
    assert fake.calls[-1][1][1] == 640 and fake.calls[-1][1][3] == 640
    _refused(lambda: m.mla_cache_write(lat[:2], kpe, slots, pool, 0), "rows")
    _refused(lambda: m.mla_cache_write(lat, kpe, slots.int(), pool, 0), "slot_mapping")
    _refused(lambda: m.mla_cache_write(lat, kpe, slots, pool, 0, status=torch.zeros(1)), "status")
    _refused(lambda: m.mla_cache_write(lat, kpe, slots, pool, 9), "cache kind")
    _refused(lambda: m.mla_cache_write_latent(lat, kpe, slots, pool, 256), "latent must be")
    m.mla_cache_write_latent(torch.zeros((3, 256), dtype=torch.bfloat16), kpe, slots, pool, 256)
    assert fake.calls[-1][0] == "mla_cache_write_latent"


def test_gather_and_merge_checks(fake):
    pool = torch.zeros((32, 656), dtype=torch.uint8)
    bt = torch.zeros((2, 2), dtype=torch.int32)
    cu = torch.tensor([0, 4, 9], dtype=torch.int32)
    m.mla_gather_upconvert(pool, 16, bt, cu, torch.empty((9, 576), dtype=torch.bfloat16))
    assert fake.calls[-1][0] == "mla_gather_upconvert"
    _refused(lambda: m.mla_gather_upconvert(pool, 16, bt, cu, torch.empty((9, 512), dtype=torch.bfloat16)), "dst")
    _refused(lambda: m.mla_gather_upconvert(pool, 16, bt[:1], cu, torch.empty((9, 576), dtype=torch.bfloat16)),
             "fewer rows")
    _refused(lambda: m.mla_gather_upconvert(pool, 16, bt, cu, torch.empty((9, 576), dtype=torch.bfloat16),
                                            num_rows=10), "num_rows")
    po, pl = torch.zeros((2, 3, 512)), torch.zeros((2, 3))
    m.mla_merge_lse(po, pl, torch.empty((3, 512)), torch.empty(3))
    assert fake.calls[-1][0] == "mla_merge_lse"
    _refused(lambda: m.mla_merge_lse(po[:, :2], pl, torch.empty((3, 512))), "part_out")
    _refused(lambda: m.mla_merge_lse(po, pl, torch.empty((2, 512))), "out must be")
    _refused(lambda: m.mla_merge_lse(po, pl, torch.empty((3, 512)), torch.empty(2)), "lse")
