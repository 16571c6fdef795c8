"""CPU oracle for paged MLA decode (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The GPU library does not depend on it
and it does not depend on the GPU library: the two share no code.

The arithmetic lives in ``mla_oracle.c`` (plain C, fp64, optional OpenMP over
independent (request, query, head) rows); this module compiles it with gcc and
exposes it to numpy through ctypes.

Functions whose result is pinned by tests (see ``tests/test_oracle_pins.py``):
``cache_write`` (byte geometry, bf16 bit copy, e4m3 round trip), ``decode``
(absorbed == naive identity, closed forms, causal truncation, rope-free
invariance), ``merge`` (partition invariance) and the e4m3 codec (agreement
with torch's float8_e4m3fn cast and with a brute-force table search); and
``decode_varlen`` in ``tests/test_oracle_varlen.py`` (fp64 brute force of the
definition, per-request verify lengths, empty leading queries); and
``gather_upconvert`` / ``f32_to_bf16`` in ``tests/test_oracle_gather.py``
(torch's bf16 and e4m3 conversions, numpy float32 products, exact power-of-two
scales, the cache write's round-trip bound, brute-force row bookkeeping); and
``decode_latent`` (other latent widths) in ``tests/test_oracle_latent.py``
(numpy brute force at widths 256 / 768 / 1792, equality with ``decode`` at
512, closed forms).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libmla_oracle.so")
_lock = threading.Lock()
_lib = None

D, P, W = 512, 64, 576
ROW_BYTES = {0: 1152, 1: 656}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no GPU code, no fast-math)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            p = ctypes.c_void_p
            i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = dbl
            lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_f64.restype = dbl
            lib.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_e4m3.restype = ctypes.c_uint8
            lib.oracle_f32_to_e4m3_n.argtypes = [p, p, i64]
            lib.oracle_f32_to_e4m3_n.restype = None
            lib.oracle_cache_write.argtypes = [p, i64, p, i64, p, i64, p, i64, i32]
            lib.oracle_cache_write.restype = i32
            lib.oracle_decode.argtypes = [p, p, p, i32, i64, i32, p, i64, p, i32, i32,
                                          i32, dbl, p, i32, p, p]
            lib.oracle_decode.restype = i32
            lib.oracle_decode_varlen.argtypes = [p, p, p, i32, i64, i32, p, i64, p, p, i32, i32, dbl, p, p]
            lib.oracle_decode_varlen.restype = i32
            lib.oracle_decode_latent.argtypes = [p, p, p, i32, i32, i64, i32, p, i64, p, i32, i32, i32, dbl, p, p]
            lib.oracle_decode_latent.restype = i32
            lib.oracle_merge.argtypes = [p, p, i32, i64, p, p]
            lib.oracle_merge.restype = None
            lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
            lib.oracle_gather_upconvert.argtypes = [p, i64, i32, p, i64, p, i32, i64, p, i64]
            lib.oracle_gather_upconvert.restype = i32
            lib.oracle_row_values.restype = i32
            lib.oracle_num_threads.restype = i32
            lib.oracle_set_num_threads.argtypes = [i32]
            lib.oracle_set_num_threads.restype = None
            lib.oracle_row_bytes.argtypes = [i32]
            lib.oracle_row_bytes.restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _as_bits16(a) -> np.ndarray:
    """Accept a torch bf16 tensor or a uint16 array of bf16 bit patterns."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def _as_np(a, dtype) -> np.ndarray:
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    """OpenMP threads the decode loop runs on (OMP_NUM_THREADS)."""
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    """Threads the decode loops use from now on (the CPU-baseline leg times
    one thread as well as all of them)."""
    _load().oracle_set_num_threads(int(n))


def row_values() -> int:
    return _load().oracle_row_values()


def row_bytes(kind: int) -> int:
    return _load().oracle_row_bytes(kind)


def bf16_to_f64(bits: int) -> float:
    return _load().oracle_bf16_to_f64(bits)


def e4m3_to_f64(code: int) -> float:
    return _load().oracle_e4m3_to_f64(code)


def f32_to_e4m3(x: float) -> int:
    return _load().oracle_f32_to_e4m3(x)


def f32_to_e4m3_array(x) -> np.ndarray:
    xs = _as_np(x, np.float32).reshape(-1)
    out = np.empty(xs.shape, dtype=np.uint8)
    _load().oracle_f32_to_e4m3_n(_ptr(xs), _ptr(out), xs.size)
    return out


def cache_write(latent, k_pe, slot_mapping, cache: np.ndarray, kind: int) -> None:
    """In-place scatter into `cache` (uint8 [num_slots, row_bytes])."""
    lib = _load()
    lat = _as_bits16(latent)
    kpe = _as_bits16(k_pe)
    sm = _as_np(slot_mapping, np.int64)
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous
    assert cache.shape[1] == ROW_BYTES[kind]
    T = sm.shape[0]
    rc = lib.oracle_cache_write(_ptr(lat), lat.shape[1] if lat.ndim == 2 else D,
                                _ptr(kpe), kpe.shape[1] if kpe.ndim == 2 else P,
                                _ptr(sm), T, _ptr(cache), cache.shape[0], kind)
    if rc != 0:
        raise ValueError("oracle_cache_write: slot out of range")


def decode(q_lat, q_pe, cache: np.ndarray, kind: int, page_size: int, block_table,
           seq_lens, B: int, Qt: int, Hq: int, scale: float, reqs=None):
    """Returns (out [B*Qt, Hq, 512] fp64, lse [B*Qt, Hq] fp64).

    Rows of requests outside `reqs` (when given) are NaN."""
    lib = _load()
    ql = _as_bits16(q_lat).reshape(B * Qt, Hq, D)
    qp = _as_bits16(q_pe).reshape(B * Qt, Hq, P)
    bt = _as_np(block_table, np.int32)
    sl = _as_np(seq_lens, np.int32)
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous
    out = np.full((B * Qt, Hq, D), np.nan, dtype=np.float64)
    lse = np.full((B * Qt, Hq), np.nan, dtype=np.float64)
    if reqs is None:
        rq, nr = None, B
    else:
        rq = np.ascontiguousarray(np.asarray(reqs, dtype=np.int32))
        nr = rq.shape[0]
    rc = lib.oracle_decode(_ptr(ql), _ptr(qp), _ptr(cache), kind, cache.shape[0], page_size,
                           _ptr(bt), bt.shape[1], _ptr(sl), B, Qt, Hq, float(scale),
                           _ptr(rq) if rq is not None else None, nr, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_decode: block id or slot out of range")
    return out, lse


def decode_varlen(q_lat, q_pe, cache: np.ndarray, kind: int, page_size: int, block_table, seq_lens, cu_q_lens,
                  Hq: int, scale: float):
    """Decode with a verify length of its own per request: cu_q_lens [B+1]
    prefix sums of query tokens; returns (out [cu_q[B], Hq, 512] fp64,
    lse [cu_q[B], Hq] fp64)."""
    lib = _load()
    cu = _as_np(cu_q_lens, np.int32)
    B = cu.shape[0] - 1
    R = int(cu[-1])
    ql = _as_bits16(q_lat).reshape(R, Hq, D)
    qp = _as_bits16(q_pe).reshape(R, Hq, P)
    bt = _as_np(block_table, np.int32)
    sl = _as_np(seq_lens, np.int32)
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous
    out = np.empty((R, Hq, D), dtype=np.float64)
    lse = np.empty((R, Hq), dtype=np.float64)
    rc = lib.oracle_decode_varlen(_ptr(ql), _ptr(qp), _ptr(cache), kind, cache.shape[0], page_size, _ptr(bt),
                                  bt.shape[1], _ptr(sl), _ptr(cu), B, Hq, float(scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_decode_varlen: block id or slot out of range")
    return out, lse


def decode_latent(q_lat, q_pe, cache, D: int, P: int, page_size: int, block_table, seq_lens, B: int, Qt: int,
                  Hq: int, scale: float):
    """Decode over a bf16 cache of rows [latent D | rope P] (uint16 bits
    [num_slots, D + P]); q_lat [B*Qt, Hq, D], q_pe [B*Qt, Hq, P]. Returns
    (out [B*Qt, Hq, D] fp64, lse [B*Qt, Hq] fp64)."""
    lib = _load()
    ql = _as_bits16(q_lat).reshape(B * Qt, Hq, D)
    qp = _as_bits16(q_pe).reshape(B * Qt, Hq, P) if P else np.zeros((B * Qt, Hq, 1), dtype=np.uint16)
    c = _as_bits16(cache)
    assert c.ndim == 2 and c.shape[1] == D + P, c.shape
    bt = _as_np(block_table, np.int32)
    sl = _as_np(seq_lens, np.int32)
    out = np.empty((B * Qt, Hq, D), dtype=np.float64)
    lse = np.empty((B * Qt, Hq), dtype=np.float64)
    rc = lib.oracle_decode_latent(_ptr(ql), _ptr(qp), _ptr(c), D, P, c.shape[0], page_size, _ptr(bt),
                                  bt.shape[1], _ptr(sl), B, Qt, Hq, float(scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_decode_latent: block id or slot out of range")
    return out, lse


def merge(part_o, part_lse):
    """part_o [S, N, 512] fp32, part_lse [S, N] fp32 -> (out [N,512], lse [N]) fp64."""
    lib = _load()
    po = _as_np(part_o, np.float32)
    pl = _as_np(part_lse, np.float32)
    S, N = pl.shape
    assert po.shape == (S, N, D)
    out = np.empty((N, D), dtype=np.float64)
    lse = np.empty((N,), dtype=np.float64)
    lib.oracle_merge(_ptr(po), _ptr(pl), S, N, _ptr(out), _ptr(lse))
    return out, lse


def f32_to_bf16(x: float) -> int:
    """bf16 bits of an fp32 value, round to nearest even."""
    return int(_load().oracle_f32_to_bf16(float(x)))


def gather_upconvert(cache: np.ndarray, page_size: int, block_table, cu_seq_lens, num_rows: int,
                     dst: np.ndarray = None, dst_stride: int = W) -> np.ndarray:
    """Context gather of an fp8_ds_mla pool (uint8 [num_slots, 656]) into bf16
    rows: returns `dst` (uint16 bits [num_rows, dst_stride], a fresh array of
    0xFFFF sentinels when not given) with rows cu[b] + j filled."""
    lib = _load()
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous and cache.shape[1] == ROW_BYTES[1]
    bt = _as_np(block_table, np.int32)
    cu = _as_np(cu_seq_lens, np.int32)
    B = cu.shape[0] - 1
    if dst is None:
        dst = np.full((num_rows, dst_stride), 0xFFFF, dtype=np.uint16)
    assert dst.dtype == np.uint16 and dst.flags.c_contiguous and dst.shape[1] == dst_stride
    rc = lib.oracle_gather_upconvert(_ptr(cache), cache.shape[0], page_size, _ptr(bt),
                                     bt.shape[1] if bt.ndim == 2 else 1, _ptr(cu), B, num_rows, _ptr(dst), dst_stride)
    if rc != 0:
        raise ValueError("oracle_gather_upconvert: block id or slot out of range")
    return dst
