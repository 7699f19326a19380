"""fp64 CPU oracle for split-KV flash attention (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never loads it, and it
imports nothing from the library.  The arithmetic lives in ``splitkv_oracle.c``
(plain C, OpenMP over independent output rows); this module compiles it with
gcc on first use and marshals numpy arrays through ctypes.

Functions (all results float64 numpy arrays):

* ``half_to_double(bits)``            IEEE binary16 decoding.
* ``dequant(type, raw, n_values)``    q8_0 / q4_0 / f16 decoding.
* ``attention(...)``                  two-pass softmax attention over a logical
                                      key list (window+tail regions, kv_rows
                                      indirection with -1 padding, causal
                                      positions, additive fp16 mask).
* ``combine(o_parts, lse_parts)``     log-sum-exp merge of partial results.

Also in the package, in plain Python: ``planner`` (the residency planner's
rules in the Rolling KV page's order) and ``bcache_model`` (the block cache's
CLOCK residency decisions as a sequential loop).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F16, Q8_0, Q4_0 = 0, 1, 2
CELL_MAJOR, PAGED = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "splitkv_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libsplitkv_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (OpenMP when available)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # SPLITKV_ORACLE_LIB points the tests at another build of this oracle
        # (the mutation tests load deliberately broken copies this way).
        override = os.environ.get("SPLITKV_ORACLE_LIB")
        lib = ctypes.CDLL(override if override else build())
        P, I, L, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.orc_half_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_half_to_double.restype = D
        lib.orc_dequant.argtypes = [I, P, L, P]
        lib.orc_dequant.restype = I
        lib.orc_attention.argtypes = [I, I, I, I, I, D, P, I, I,
                                      P, P, L, L, L,
                                      P, P, L, L, L,
                                      I, I, L, P, I, P, P, L, P, P]
        lib.orc_attention.restype = I
        lib.orc_combine.argtypes = [I, L, I, P, P, P, P]
        lib.orc_combine.restype = I
        lib.orc_max_threads.restype = I
        lib.orc_set_threads.argtypes = [I]
        lib.orc_segment_bytes.argtypes = [I, I]
        lib.orc_segment_bytes.restype = L
        lib.orc_float_to_half.argtypes = [ctypes.c_float]
        lib.orc_float_to_half.restype = ctypes.c_uint16
        lib.orc_quantize.argtypes = [I, P, L, P]
        lib.orc_quantize.restype = I
        lib.orc_kv_append.argtypes = [I, I, I, L, P, P, L, P, L, P, L]
        lib.orc_kv_append.restype = L
        lib.orc_paged_append.argtypes = [I, I, I, L, P, P, L, P]
        lib.orc_paged_append.restype = L
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def max_threads() -> int:
    return int(_load().orc_max_threads())


def set_threads(n: int) -> None:
    _load().orc_set_threads(int(n))


def segment_bytes(type_: int, D: int) -> int:
    return int(_load().orc_segment_bytes(type_, D))


def half_to_double(bits) -> np.ndarray:
    lib = _load()
    bits = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.orc_half_to_double(int(b)) for b in bits], dtype=np.float64)


def dequant(type_: int, raw, n_values: int) -> np.ndarray:
    raw = np.ascontiguousarray(np.asarray(raw, dtype=np.uint8))
    out = np.empty(n_values, dtype=np.float64)
    rc = _load().orc_dequant(type_, _ptr(raw), n_values, _ptr(out))
    if rc:
        raise ValueError("orc_dequant rejected its arguments")
    return out


def _bytes_view(a):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    return a.view(np.uint8).reshape(-1) if a.size else np.zeros(1, np.uint8)


def attention(q, *, D, H, Hk, scale, k_type=F16, v_type=F16,
              k0, v0, n_rows0, k_row_bytes0=0, v_row_bytes0=0,
              k1=None, v1=None, n_rows1=0, k_row_bytes1=0, v_row_bytes1=0,
              layout=CELL_MAJOR, page_rows=0,
              n_keys, kv_rows=None, rows_per_head=False,
              mask=None, q_pos=None, key_pos0=0):
    """Two-pass fp64 attention.  ``q`` holds fp16 values (any float16 array
    shaped [S, nq, H, D]); caches are raw byte buffers (numpy arrays of any
    dtype, reinterpreted as bytes).  Returns (O [S,nq,H,D], lse [S,nq,H])."""
    q = np.ascontiguousarray(np.asarray(q, dtype=np.float16))
    S, nq = q.shape[0], q.shape[1]
    assert q.shape[2] == H and q.shape[3] == D
    qb = q.view(np.uint16)
    kr = None if kv_rows is None else np.ascontiguousarray(kv_rows, dtype=np.int32)
    mk = None if mask is None else np.ascontiguousarray(np.asarray(mask, np.float16)).view(np.uint16)
    qp = None if q_pos is None else np.ascontiguousarray(q_pos, dtype=np.int32)
    kb0, vb0, kb1, vb1 = (_bytes_view(x) for x in (k0, v0, k1, v1))
    if kb1 is None:
        kb1 = vb1 = np.zeros(1, np.uint8)
    o = np.empty((S, nq, H, D), dtype=np.float64)
    lse = np.empty((S, nq, H), dtype=np.float64)
    rc = _load().orc_attention(S, nq, H, Hk, D, float(scale), _ptr(qb), k_type, v_type,
                               _ptr(kb0), _ptr(vb0), int(n_rows0), int(k_row_bytes0), int(v_row_bytes0),
                               _ptr(kb1), _ptr(vb1), int(n_rows1), int(k_row_bytes1), int(v_row_bytes1),
                               layout, int(page_rows), int(n_keys), _ptr(kr), int(bool(rows_per_head)),
                               _ptr(mk), _ptr(qp), int(key_pos0), _ptr(o), _ptr(lse))
    if rc:
        raise ValueError(f"orc_attention failed ({rc})")
    return o, lse


def combine(o_parts, lse_parts):
    """Merge partials: o_parts [P, rows, D], lse_parts [P, rows] (float64)."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    P, rows, D = o_parts.shape
    o = np.empty((rows, D), dtype=np.float64)
    lse = np.empty(rows, dtype=np.float64)
    rc = _load().orc_combine(P, rows, D, _ptr(o_parts), _ptr(lse_parts), _ptr(o), _ptr(lse))
    if rc:
        raise ValueError("orc_combine rejected its arguments")
    return o, lse


def float_to_half(x) -> np.ndarray:
    """Binary16 bit patterns (uint16) of fp32 values, nearest-even rounding."""
    lib = _load()
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.orc_float_to_half(float(v)) for v in x], dtype=np.uint16)


def quantize(type_: int, x) -> np.ndarray:
    """Encode fp32 values as fp16 / q8_0 / q4_0 bytes."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32).ravel())
    n = x.size
    nbytes = 2 * n if type_ == F16 else segment_bytes(type_, 32) * (n // 32)
    out = np.zeros(max(nbytes, 1), dtype=np.uint8)
    if _load().orc_quantize(type_, _ptr(x), n, _ptr(out)):
        raise ValueError("orc_quantize rejected its arguments")
    return out[:nbytes]


def kv_append(type_: int, x, positions, dst0, n_rows0: int, dst1, n_rows1: int, row_bytes: int) -> int:
    """Write x ([n][Hk][D] fp32) into two cell-major uint8 regions in place;
    returns how many positions fell outside both regions."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    n, Hk, D = x.shape
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int32))
    for a in (dst0, dst1):
        assert a is None or (a.dtype == np.uint8 and a.flags["C_CONTIGUOUS"])
    bad = _load().orc_kv_append(type_, Hk, D, int(row_bytes), _ptr(x), _ptr(pos), n, _ptr(dst0), int(n_rows0),
                                _ptr(dst1), int(n_rows1))
    if bad < 0:
        raise ValueError("orc_kv_append rejected its arguments")
    return int(bad)


def paged_append(x, positions, host, *, block_rows: int, n_blocks: int) -> int:
    """Write x ([n][Hk][D] fp32) into a paged fp16 host copy (uint16
    [n_blocks][Hk][block_rows][D]) in place; returns the out-of-range count."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    n, Hk, D = x.shape
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int32))
    assert host.dtype == np.uint16 and host.flags["C_CONTIGUOUS"]
    bad = _load().orc_paged_append(Hk, D, int(block_rows), int(n_blocks), _ptr(x), _ptr(pos), n, _ptr(host))
    if bad < 0:
        raise ValueError("orc_paged_append rejected its arguments")
    return int(bad)
