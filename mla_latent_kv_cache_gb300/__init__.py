"""Paged MLA decode for GB300 (sm_103a): Python binding of the C ABI.

The compute path lives in ``_lib/libmla_gb300.so`` (built from ``csrc/`` by
``mla_latent_kv_cache_gb300.build``). This module only marshals arguments:
torch tensors -> device pointers, the current CUDA stream, and status codes ->
exceptions. Before a call it checks what the library cannot see (that every
tensor is a CUDA tensor on one device, and the dtypes, layouts and sizes of
the buffers the call reads and writes) and raises MlaError with
MLA_ERR_INVALID_ARG otherwise. There is no fallback: if the library is
missing, every call raises.

Entry points mirror ``include/mla.h``:
  mla_cache_write, mla_decode_workspace_bytes, mla_decode, mla_decode_varlen,
  mla_merge_lse, mla_gather_upconvert, mla_cache_write_latent,
  mla_decode_latent_workspace_bytes, mla_decode_latent,
  mla_decode_static_scratch (+ mla_static_scratch_status), mla_num_sms,
  mla_row_bytes, mla_status_string.
``decode(...)`` is a convenience wrapper that allocates the outputs and the
workspace with torch and calls ``mla_decode``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmla_gb300.so")

MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_WORKSPACE, MLA_ERR_CUDA = 0, -1, -2, -3, -4
MLA_CACHE_BF16_576, MLA_CACHE_FP8_DS_MLA_656 = 0, 1
MLA_OUT_BF16, MLA_OUT_F32 = 0, 1
STATUS_WAIT_TIMEOUT, STATUS_BAD_BLOCK = 1, 2

_lock = threading.Lock()
_lib = None


class MlaError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {mla_status_string(status)} ({status})" + (f": {detail}" if detail else ""))


def load() -> ctypes.CDLL:
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build it with `python -m mla_latent_kv_cache_gb300.build` "
                    "(there is no CPU fallback)")
            lib = ctypes.CDLL(LIB_PATH)
            vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
            lib.mla_row_bytes.argtypes = [i32]
            lib.mla_row_bytes.restype = i32
            lib.mla_status_string.argtypes = [i32]
            lib.mla_status_string.restype = ctypes.c_char_p
            lib.mla_num_sms.argtypes = []
            lib.mla_num_sms.restype = i32
            lib.mla_cache_write.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, i32, vp, vp]
            lib.mla_cache_write.restype = i32
            lib.mla_decode_workspace_bytes.argtypes = [i32, i32, i32, i32]
            lib.mla_decode_workspace_bytes.restype = sz
            lib.mla_decode.argtypes = [vp, vp, vp, i32, i64, i32, vp, i64, vp, i32, i32, i32, f32, vp, i32, vp,
                                       vp, sz, i32, vp]
            lib.mla_decode.restype = i32
            lib.mla_decode_static_scratch.argtypes = [vp, vp, vp, i32, i64, i32, vp, i64, vp, i32, i32, i32, f32, vp,
                                                      i32, vp, i32, vp]
            lib.mla_decode_static_scratch.restype = i32
            lib.mla_static_scratch_status.argtypes = [vp, i32, vp]
            lib.mla_static_scratch_status.restype = i32
            lib.mla_test_hold_next_decode.argtypes = []
            lib.mla_test_hold_next_decode.restype = None
            lib.mla_test_slow_pv_next_decode.argtypes = []
            lib.mla_test_slow_pv_next_decode.restype = None
            lib.mla_merge_lse.argtypes = [vp, vp, i32, i64, vp, i32, vp, vp]
            lib.mla_decode_varlen.argtypes = [vp, vp, i64, vp, i32, i64, i32, vp, i64, vp, vp, i32, i32, i32, f32,
                                              vp, i32, vp, vp, ctypes.c_size_t, i32, vp]
            lib.mla_decode_varlen.restype = i32
            lib.mla_gather_upconvert.argtypes = [vp, i64, i32, vp, i64, vp, i32, i64, vp, i64, vp]
            lib.mla_gather_upconvert.restype = i32
            lib.mla_cache_write_latent.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, i32, vp, vp]
            lib.mla_cache_write_latent.restype = i32
            lib.mla_decode_latent_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
            lib.mla_decode_latent_workspace_bytes.restype = sz
            lib.mla_decode_latent.argtypes = [vp, vp, vp, i32, i64, i32, vp, i64, vp, i32, i32, i32, f32, vp, i32,
                                              vp, vp, sz, i32, vp]
            lib.mla_decode_latent.restype = i32
            lib.mla_merge_lse.restype = i32
            _lib = lib
    return _lib


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status: int, where: str) -> None:
    if status != MLA_OK:
        raise MlaError(status, where)


# Argument checks of the binding. The library validates sizes, pointers and
# alignment on the host, but it cannot tell a host pointer from a device one
# or how large a caller's buffer is: a host tensor handed to a kernel is an
# illegal address (or, where the GPU reaches host memory, a silent slow
# path), and an output smaller than the call writes is overrun. These checks
# run before the library is called and raise MlaError(MLA_ERR_INVALID_ARG).

def _is_cuda(t) -> bool:
    return isinstance(t, torch.Tensor) and t.is_cuda


def _need(ok: bool, where: str, detail: str) -> None:
    if not ok:
        raise MlaError(MLA_ERR_INVALID_ARG, where, detail)


def _on_device(where: str, **tensors) -> None:
    """Every tensor passed as a device pointer is a CUDA tensor, all on one device."""
    dev = None
    for name, t in tensors.items():
        if t is None:
            continue
        _need(_is_cuda(t), where, f"{name} must be a CUDA tensor")
        if dev is None:
            dev = t.device
        _need(t.device == dev, where, f"{name} is on {t.device}, the other arguments on {dev}")


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


def _decode_args(where, q_lat, q_pe, cache, block_table, seq_lens, out, lse, workspace, rows, width):
    """Checks shared by the decode entry points: `rows` query rows of `width`
    latent values (query tokens x heads)."""
    _on_device(where, q_lat=q_lat, q_pe=q_pe, cache=cache, block_table=block_table, seq_lens=seq_lens, out=out,
               lse=lse, workspace=workspace)
    _need(q_lat.dtype == torch.bfloat16 and q_pe.dtype == torch.bfloat16, where, "q_lat and q_pe must be bf16")
    _need(q_lat.is_contiguous() and q_pe.is_contiguous(), where, "q_lat and q_pe must be contiguous")
    _need(q_lat.numel() == rows * width and q_pe.numel() == rows * 64, where,
          f"q_lat / q_pe hold {q_lat.numel()} / {q_pe.numel()} values, {rows} rows of {width} / 64 expected")
    _need(out.dtype in (torch.bfloat16, torch.float32) and out.is_contiguous(), where,
          "out must be a contiguous bf16 or fp32 tensor")
    _need(out.numel() >= rows * width, where, f"out holds {out.numel()} values, the call writes {rows * width}")
    _need(lse.dtype == torch.float32 and lse.is_contiguous() and lse.numel() >= rows, where,
          f"lse must be a contiguous fp32 tensor of at least {rows} values")
    _need(cache.is_contiguous(), where, "cache must be contiguous")
    _need(block_table.dtype == torch.int32 and block_table.dim() == 2 and block_table.stride(1) == 1, where,
          "block_table must be a 2-D int32 tensor with contiguous rows")
    B = seq_lens.numel()
    _need(block_table.shape[0] >= B, where, f"block_table has {block_table.shape[0]} rows for {B} requests")
    _need(seq_lens.dtype == torch.int32 and seq_lens.is_contiguous(), where, "seq_lens must be contiguous int32")
    if workspace is not None:
        _need(workspace.is_contiguous(), where, "workspace must be contiguous")


def _write_args(where, latent, k_pe, slot_mapping, cache, status, width):
    """Checks shared by the cache writes: rows of `width` latent values."""
    _on_device(where, latent=latent, k_pe=k_pe, slot_mapping=slot_mapping, cache=cache, status=status)
    _need(latent.dtype == torch.bfloat16 and k_pe.dtype == torch.bfloat16, where, "latent and k_pe must be bf16")
    _need(latent.dim() in (1, 2) and k_pe.dim() in (1, 2) and latent.shape[-1] == width and k_pe.shape[-1] == 64,
          where, f"latent must be [T, {width}] and k_pe [T, 64]")
    _need(latent.stride(-1) == 1 and k_pe.stride(-1) == 1, where, "latent and k_pe rows must be contiguous")
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.is_contiguous(), where,
          "slot_mapping must be contiguous int64")
    T = slot_mapping.numel()
    rows = lambda t: t.shape[0] if t.dim() == 2 else 1
    _need(rows(latent) >= T and rows(k_pe) >= T, where, f"latent / k_pe have fewer than the {T} rows slot_mapping names")
    _need(cache.is_contiguous(), where, "cache must be contiguous")
    _need(status is None or (status.dtype == torch.int32 and status.numel() >= 1), where,
          "status must be an int32 tensor")


def mla_status_string(status: int) -> str:
    try:
        return load().mla_status_string(status).decode()
    except ImportError:
        return f"status {status}"


def mla_row_bytes(cache_kind: int) -> int:
    return load().mla_row_bytes(cache_kind)


def mla_num_sms() -> int:
    return load().mla_num_sms()


def mla_cache_write(latent: torch.Tensor, k_pe: torch.Tensor, slot_mapping: torch.Tensor, cache: torch.Tensor,
                    cache_kind: int = MLA_CACHE_BF16_576, stream=None, status: torch.Tensor = None) -> None:
    """latent [T,512] bf16, k_pe [T,64] bf16 (row-strided views allowed),
    slot_mapping [T] int64 (-1 = skip), cache [num_slots, row_bytes] (any dtype
    viewable as bytes). Scatters rows in place; slots >= num_slots are skipped
    and, when `status` (a device int32 tensor) is given, OR bit 2 into its
    first element."""
    _write_args("mla_cache_write", latent, k_pe, slot_mapping, cache, status, 512)
    T = slot_mapping.numel()
    nbytes = cache.numel() * cache.element_size()
    rb = mla_row_bytes(cache_kind)
    _need(rb > 0, "mla_cache_write", f"unknown cache kind {cache_kind}")
    _check(load().mla_cache_write(latent.data_ptr(), latent.stride(0) if latent.dim() == 2 else 512,
                                  k_pe.data_ptr(), k_pe.stride(0) if k_pe.dim() == 2 else 64,
                                  slot_mapping.data_ptr(), T, cache.data_ptr(), nbytes // rb, cache_kind,
                                  status.data_ptr() if status is not None else None,
                                  _stream(stream)), "mla_cache_write")


def mla_decode_varlen(q_lat, q_pe, cache, cache_kind, page_size, block_table, seq_lens, cu_q_lens, max_q_len,
                      scale, out, lse, workspace, num_ctas: int = 0, stream=None) -> None:
    """Decode with per-request verify lengths (include/mla.h): q_lat [total_q, Hq, 512],
    cu_q_lens int32 [B+1] on the device."""
    where = "mla_decode_varlen"
    _need(isinstance(q_lat, torch.Tensor) and q_lat.dim() == 3, where, "q_lat must be [total_q, Hq, 512]")
    total_q, Hq = q_lat.shape[0], q_lat.shape[1]
    _need(q_lat.shape == (total_q, Hq, 512) and tuple(q_pe.shape) == (total_q, Hq, 64), where,
          "q_lat must be [total_q, Hq, 512] and q_pe [total_q, Hq, 64]")
    _decode_args(where, q_lat, q_pe, cache, block_table, seq_lens, out, lse, workspace, total_q * Hq, 512)
    _on_device(where, q_lat=q_lat, cu_q_lens=cu_q_lens)
    B = seq_lens.numel()
    _need(cu_q_lens.dtype == torch.int32 and cu_q_lens.is_contiguous() and cu_q_lens.numel() == B + 1, where,
          f"cu_q_lens must be contiguous int32 with {B + 1} entries")
    rb = mla_row_bytes(cache_kind)
    _need(rb > 0, where, f"unknown cache kind {cache_kind}")
    odt = MLA_OUT_F32 if out.dtype == torch.float32 else MLA_OUT_BF16
    st = load().mla_decode_varlen(q_lat.data_ptr(), q_pe.data_ptr(), total_q, cache.data_ptr(), int(cache_kind),
                                  _nbytes(cache) // rb, int(page_size), block_table.data_ptr(),
                                  block_table.stride(0), seq_lens.data_ptr(), cu_q_lens.data_ptr(), B,
                                  int(max_q_len), Hq, float(scale), out.data_ptr(), odt, lse.data_ptr(),
                                  workspace.data_ptr(), _nbytes(workspace), int(num_ctas), _stream(stream))
    _check(st, "mla_decode_varlen")


def mla_gather_upconvert(cache: torch.Tensor, page_size: int, block_table: torch.Tensor, cu_seq_lens: torch.Tensor,
                         dst: torch.Tensor, num_rows: int = None, stream=None) -> None:
    """Context gather of an fp8_ds_mla pool into bf16 rows (include/mla.h)."""
    where = "mla_gather_upconvert"
    _on_device(where, cache=cache, block_table=block_table, cu_seq_lens=cu_seq_lens, dst=dst)
    _need(cache.dtype == torch.uint8 and cache.dim() == 2 and cache.shape[1] == 656 and cache.is_contiguous(), where,
          "cache must be a contiguous uint8 [num_slots, 656] tensor")
    _need(block_table.dtype == torch.int32 and block_table.dim() == 2 and block_table.stride(1) == 1, where,
          "block_table must be a 2-D int32 tensor with contiguous rows")
    _need(cu_seq_lens.dtype == torch.int32 and cu_seq_lens.is_contiguous() and cu_seq_lens.numel() >= 1, where,
          "cu_seq_lens must be contiguous int32 with B + 1 entries")
    _need(block_table.shape[0] >= cu_seq_lens.numel() - 1, where, "block_table has fewer rows than requests")
    _need(dst.dtype == torch.bfloat16 and dst.dim() == 2 and dst.stride(1) == 1 and dst.shape[1] >= 576, where,
          "dst must be a bf16 [rows, >= 576] tensor with contiguous rows")
    rows = dst.shape[0] if num_rows is None else int(num_rows)
    _need(0 <= rows <= dst.shape[0], where, f"num_rows {rows} outside [0, {dst.shape[0]}]")
    st = load().mla_gather_upconvert(cache.data_ptr(), cache.shape[0], int(page_size), block_table.data_ptr(),
                                     block_table.stride(0), cu_seq_lens.data_ptr(), cu_seq_lens.shape[0] - 1, rows,
                                     dst.data_ptr(), dst.stride(0), _stream(stream))
    _check(st, "mla_gather_upconvert")


def mla_cache_write_latent(latent, k_pe, slot_mapping, cache, lat_dim, stream=None, status=None) -> None:
    """bf16 rows [latent lat_dim | rope 64] (include/mla.h): latent
    [T, lat_dim] bf16, k_pe [T, 64] bf16, slot_mapping [T] int64, cache
    [num_slots, 2 (lat_dim + 64)] bytes."""
    _write_args("mla_cache_write_latent", latent, k_pe, slot_mapping, cache, status, int(lat_dim))
    T = slot_mapping.numel()
    row_bytes = 2 * (lat_dim + 64)
    nbytes = cache.numel() * cache.element_size()
    _check(load().mla_cache_write_latent(latent.data_ptr(), latent.stride(0), k_pe.data_ptr(), k_pe.stride(0),
                                         slot_mapping.data_ptr(), T, cache.data_ptr(), nbytes // row_bytes,
                                         int(lat_dim), status.data_ptr() if status is not None else None,
                                         _stream(stream)), "mla_cache_write_latent")


def mla_decode_latent_workspace_bytes(B: int, q_len: int, Hq: int, lat_dim: int, num_ctas: int = 0) -> int:
    n = load().mla_decode_latent_workspace_bytes(B, q_len, Hq, lat_dim, num_ctas)
    if n == 0:
        raise MlaError(MLA_ERR_INVALID_ARG, "mla_decode_latent_workspace_bytes")
    return n


def mla_decode_latent(q_lat, q_pe, cache, lat_dim, page_size, block_table, seq_lens, q_len, scale, out, lse,
                      workspace, num_ctas: int = 0, stream=None) -> None:
    """Decode over bf16 rows of latent width lat_dim (include/mla.h):
    q_lat [B*q_len, Hq, lat_dim], out [B*q_len, Hq, lat_dim]."""
    B = seq_lens.numel()
    Hq = q_lat.shape[-2]
    where = "mla_decode_latent"
    _need(q_lat.shape[-1] == lat_dim and q_pe.shape[-1] == 64 and out.shape[-1] == lat_dim, where,
          f"q_lat and out must end in {lat_dim} values, q_pe in 64")
    _decode_args(where, q_lat, q_pe, cache, block_table, seq_lens, out, lse, workspace, B * int(q_len) * Hq,
                 int(lat_dim))
    out_dtype = MLA_OUT_F32 if out.dtype == torch.float32 else MLA_OUT_BF16
    row_bytes = 2 * (lat_dim + 64)
    nbytes = cache.numel() * cache.element_size()
    _check(load().mla_decode_latent(q_lat.data_ptr(), q_pe.data_ptr(), cache.data_ptr(), int(lat_dim),
                                    nbytes // row_bytes, int(page_size), block_table.data_ptr(),
                                    block_table.stride(0), seq_lens.data_ptr(), B, int(q_len), Hq, float(scale),
                                    out.data_ptr(), out_dtype, lse.data_ptr(), workspace.data_ptr(),
                                    workspace.numel() * workspace.element_size(), int(num_ctas), _stream(stream)),
           "mla_decode_latent")


def mla_decode_workspace_bytes(B: int, q_len: int, Hq: int, num_ctas: int = 0) -> int:
    n = load().mla_decode_workspace_bytes(B, q_len, Hq, num_ctas)
    if n == 0:
        raise MlaError(MLA_ERR_INVALID_ARG, "mla_decode_workspace_bytes")
    return n


def mla_decode(q_lat, q_pe, cache, cache_kind, page_size, block_table, seq_lens, q_len, scale, out, lse,
               workspace, num_ctas: int = 0, stream=None) -> None:
    """Raw entry point: every buffer is caller-allocated (see include/mla.h)."""
    B = seq_lens.numel()
    Hq = q_lat.shape[-2]
    _decode_args("mla_decode", q_lat, q_pe, cache, block_table, seq_lens, out, lse, workspace, B * int(q_len) * Hq,
                 512)
    out_dtype = MLA_OUT_F32 if out.dtype == torch.float32 else MLA_OUT_BF16
    nbytes = cache.numel() * cache.element_size()
    rb = mla_row_bytes(cache_kind)
    _need(rb > 0, "mla_decode", f"unknown cache kind {cache_kind}")
    _check(load().mla_decode(q_lat.data_ptr(), q_pe.data_ptr(), cache.data_ptr(), cache_kind, nbytes // rb,
                             page_size, block_table.data_ptr(), block_table.stride(0), seq_lens.data_ptr(), B, q_len,
                             Hq, float(scale), out.data_ptr(), out_dtype, lse.data_ptr(), workspace.data_ptr(),
                             workspace.numel() * workspace.element_size(), num_ctas, _stream(stream)),
           "mla_decode")


def mla_decode_static_scratch(q_lat, q_pe, cache, cache_kind, page_size, block_table, seq_lens, q_len, scale, out,
                              lse, num_ctas: int = 0, stream=None) -> None:
    """mla_decode with the library's static device scratch as its workspace
    (see include/mla.h: at most MLA_STATIC_SCRATCH_BYTES; calls sharing a
    device must be ordered on one stream)."""
    B = seq_lens.numel()
    Hq = q_lat.shape[-2]
    _decode_args("mla_decode_static_scratch", q_lat, q_pe, cache, block_table, seq_lens, out, lse, None,
                 B * int(q_len) * Hq, 512)
    out_dtype = MLA_OUT_F32 if out.dtype == torch.float32 else MLA_OUT_BF16
    nbytes = cache.numel() * cache.element_size()
    rb = mla_row_bytes(cache_kind)
    _need(rb > 0, "mla_decode_static_scratch", f"unknown cache kind {cache_kind}")
    _check(load().mla_decode_static_scratch(q_lat.data_ptr(), q_pe.data_ptr(), cache.data_ptr(), cache_kind,
                                            nbytes // rb, page_size, block_table.data_ptr(), block_table.stride(0),
                                            seq_lens.data_ptr(), B, q_len, Hq, float(scale), out.data_ptr(),
                                            out_dtype, lse.data_ptr(), num_ctas, _stream(stream)),
           "mla_decode_static_scratch")


def static_scratch_status_words(n: int = 12, stream=None) -> list:
    """The status words the last mla_decode_static_scratch call on the
    current device left in the static scratch (mla_static_scratch_status):
    word 0 status bits, words 1..11 where a wait gave up (as
    device_status_words for a caller workspace)."""
    dst = torch.zeros(n, dtype=torch.int32, device=torch.cuda.current_device())
    _check(load().mla_static_scratch_status(dst.data_ptr(), n, _stream(stream)), "mla_static_scratch_status")
    return [int(v) for v in dst.tolist()]


def mla_merge_lse(part_out: torch.Tensor, part_lse: torch.Tensor, out: torch.Tensor, lse=None, stream=None) -> None:
    """part_out [S,N,512] fp32, part_lse [S,N] fp32 -> out [N,512] (bf16/fp32), lse [N]."""
    where = "mla_merge_lse"
    _on_device(where, part_out=part_out, part_lse=part_lse, out=out, lse=lse)
    _need(part_lse.dim() == 2, where, "part_lse must be [S, N]")
    S, N = part_lse.shape
    _need(part_out.dtype == torch.float32 and part_lse.dtype == torch.float32, where, "partials must be fp32")
    _need(part_out.is_contiguous() and part_lse.is_contiguous() and part_out.numel() == S * N * 512, where,
          f"part_out must be a contiguous [{S}, {N}, 512] tensor")
    _need(out.dtype in (torch.bfloat16, torch.float32) and out.is_contiguous() and out.numel() >= N * 512, where,
          f"out must be a contiguous bf16 or fp32 tensor of at least {N} x 512 values")
    _need(lse is None or (lse.dtype == torch.float32 and lse.is_contiguous() and lse.numel() >= N), where,
          f"lse must be a contiguous fp32 tensor of at least {N} values")
    out_dtype = MLA_OUT_F32 if out.dtype == torch.float32 else MLA_OUT_BF16
    _check(load().mla_merge_lse(part_out.data_ptr(), part_lse.data_ptr(), S, N, out.data_ptr(), out_dtype,
                                lse.data_ptr() if lse is not None else None, _stream(stream)), "mla_merge_lse")


def decode(q_lat, q_pe, cache, cache_kind, page_size, block_table, seq_lens, q_len, scale,
           out_dtype=torch.bfloat16, num_ctas: int = 0, workspace=None, stream=None):
    """Allocate out/lse (and the workspace unless given) and run mla_decode.
    Returns (out [B*q_len, Hq, 512], lse [B*q_len, Hq], workspace)."""
    B = seq_lens.numel()
    Hq = q_lat.shape[-2]
    dev = q_lat.device
    out = torch.empty((B * q_len, Hq, 512), dtype=out_dtype, device=dev)
    lse = torch.empty((B * q_len, Hq), dtype=torch.float32, device=dev)
    need = mla_decode_workspace_bytes(B, q_len, Hq, num_ctas)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    mla_decode(q_lat, q_pe, cache, cache_kind, page_size, block_table, seq_lens, q_len, scale, out, lse, workspace,
               num_ctas, stream)
    return out, lse, workspace


def device_status_words(workspace: torch.Tensor, n: int = 12) -> list:
    """The workspace status header of the last mla_decode that used it:
    word 0 status bits, words 1..3 the first failing CTA's wait site, tile and
    index, words 4..11 where each of its roles gave up ((site << 24) | tile)."""
    return [int(v) for v in workspace[:4 * n].view(torch.int32).tolist()]


def test_hold_next_decode() -> None:
    """Test support: make the next mla_decode's PV issuers time out (see
    include/mla.h)."""
    load().mla_test_hold_next_decode()


def test_slow_pv_next_decode() -> None:
    """Test support: make one PV issuer of the next mla_decode lag the
    softmax warps by up to two tiles; its results are unchanged (see
    include/mla.h)."""
    load().mla_test_slow_pv_next_decode()


def device_status(workspace: torch.Tensor) -> int:
    """Device-side status word of the last mla_decode that used `workspace`
    (0 = ok; bit 1 = a bounded wait gave up; bit 2 = a block id outside the
    pool or a page index past the table row; bit 4 = an fp8 value past the
    f16 range of the fp8 path up to 64 rows)."""
    return int(workspace[:4].view(torch.int32).item())
