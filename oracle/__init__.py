"""CPU oracle for the Conditional Program (CP) lookup-decode -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never loads it, and this package never loads the CUDA library.

The arithmetic lives in ``cp_oracle.cpp`` (plain C++17, fp64 unless a step says
fp32, compiled without contraction of multiply-adds).  This module only
marshals numpy arrays through ctypes.

Pages are cited by title:
  [P4] "2비트 코드와 공유 트렐리스로 n-gram 룩업 테이블을 4~8배 압축한다"
       (onedev.kr/papers/1189), sections 어떻게 동작하나 (how it works) and
       무엇과 다른가 (how it differs).

Parity pins for every function are in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "cp_oracle.cpp"
_LIB_PATH = _HERE / "_build" / "libcp_oracle.so"

BRUTE, EXACT, TWO_PASS = 0, 1, 2

_lib = None


def compile_oracle(force: bool = False) -> Path:
    """Compile cp_oracle.cpp into oracle/_build/libcp_oracle.so (g++, -ffp-contract=off)."""
    if force or not _LIB_PATH.exists() or _LIB_PATH.stat().st_mtime < _SRC.stat().st_mtime:
        _LIB_PATH.parent.mkdir(parents=True, exist_ok=True)
        tmp = _LIB_PATH.with_suffix(f".{os.getpid()}.tmp.so")
        subprocess.run(
            ["g++", "-std=c++17", "-O2", "-fPIC", "-shared", "-pthread",
             "-ffp-contract=off", "-fno-fast-math", "-o", str(tmp), str(_SRC)],
            check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(str(compile_oracle()))
        u8p, u16p, u32p, i64p, f64p = (C.POINTER(C.c_uint8), C.POINTER(C.c_uint16),
                                       C.POINTER(C.c_uint32), C.POINTER(C.c_int64),
                                       C.POINTER(C.c_double))
        L = _lib
        L.orc_half_to_double.restype = C.c_double
        L.orc_half_to_double.argtypes = [C.c_uint16]
        L.orc_double_to_half.restype = C.c_uint16
        L.orc_double_to_half.argtypes = [C.c_double]
        L.orc_float_to_bf16.restype = C.c_uint16
        L.orc_float_to_bf16.argtypes = [C.c_float]
        L.orc_double_to_bf16.restype = C.c_uint16
        L.orc_double_to_bf16.argtypes = [C.c_double]
        L.orc_bf16_to_float.restype = C.c_float
        L.orc_bf16_to_float.argtypes = [C.c_uint16]
        L.orc_splitmix64.restype = C.c_uint64
        L.orc_splitmix64.argtypes = [C.c_uint64]
        L.orc_normal_pairs.restype = None
        L.orc_normal_pairs.argtypes = [C.c_uint64, C.c_uint64, C.c_uint64, f64p]
        L.orc_lloyd_lut.restype = C.c_double
        L.orc_lloyd_lut.argtypes = [C.c_uint64, C.c_uint64, C.c_uint32, C.c_uint32, C.c_int,
                                    f64p, u16p]
        L.orc_window_states.restype = None
        L.orc_window_states.argtypes = [u8p, C.c_uint32, C.c_uint32, u32p]
        L.orc_state_hash.restype = None
        L.orc_state_hash.argtypes = [u32p, C.c_uint64, u32p, u32p]
        L.orc_decode_f.restype = None
        L.orc_decode_f.argtypes = [u8p, C.c_uint32, C.c_uint32, u16p, f64p]
        L.orc_lookup_decode.restype = C.c_uint64
        L.orc_lookup_decode.argtypes = [u8p, C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint64,
                                        u16p, i64p, C.c_uint64, u16p, C.c_int]
        L.orc_lookup_decode_reduce.restype = C.c_uint64
        L.orc_lookup_decode_reduce.argtypes = [u8p, C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint64,
                                               u16p, i64p, C.c_uint64, C.c_uint32,
                                               C.POINTER(C.c_float), u16p, C.c_int]
        L.orc_lookup_decode_mixed.restype = C.c_uint64
        L.orc_lookup_decode_mixed.argtypes = [u8p, C.POINTER(C.c_uint64), C.c_uint64, C.c_uint32,
                                              u16p, i64p, C.c_uint64, u16p]
        L.orc_distortion.restype = C.c_double
        L.orc_distortion.argtypes = [f64p, u8p, C.c_uint32, C.c_uint32, u16p]
        L.orc_encode_z.restype = C.c_double
        L.orc_encode_z.argtypes = [f64p, C.c_uint32, C.c_uint32, u16p, C.c_int, u8p]
        L.orc_encode_rows.restype = C.c_int
        L.orc_encode_rows.argtypes = [f64p, C.c_uint64, C.c_uint32, C.c_uint32, u16p, C.c_int,
                                      C.c_int, u8p, f64p, f64p]
        f32p = C.POINTER(C.c_float)
        L.orc_distortion_f32.restype = C.c_float
        L.orc_distortion_f32.argtypes = [f32p, u8p, C.c_uint32, C.c_uint32, u16p]
        L.orc_encode_z_f32.restype = C.c_float
        L.orc_encode_z_f32.argtypes = [f32p, C.c_uint32, C.c_uint32, u16p, C.c_int, u8p]
        L.orc_encode_rows_f32.restype = C.c_int
        L.orc_encode_rows_f32.argtypes = [f32p, C.c_uint64, C.c_uint32, C.c_uint32, u16p, C.c_int,
                                          u8p, f32p]
        L.orc_free_start_f.restype = C.c_float
        L.orc_free_start_f.argtypes = [f32p, C.c_uint32, C.c_uint32, u16p, C.c_uint32, u32p]
        L.orc_free_start_brute_f.restype = C.c_float
        L.orc_free_start_brute_f.argtypes = [f32p, C.c_uint32, C.c_uint32, u16p, C.c_uint32, u32p]
        L.orc_rtn2.restype = None
        L.orc_rtn2.argtypes = [f64p, C.c_uint32, C.c_int, f64p]
    return _lib


def _p(a: np.ndarray, ct):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.POINTER(ct))


def n_threads_default() -> int:
    return max(1, os.cpu_count() or 1)


# ---- formats ---------------------------------------------------------------

def half_to_double(h: int) -> float:
    return lib().orc_half_to_double(int(h))


def double_to_half(x: float) -> int:
    return lib().orc_double_to_half(float(x))


def float_to_bf16(x: float) -> int:
    return lib().orc_float_to_bf16(float(x))


def double_to_bf16(x: float) -> int:
    return lib().orc_double_to_bf16(float(x))


def bf16_to_float(b: int) -> float:
    return lib().orc_bf16_to_float(int(b))


def lut_values(lut: np.ndarray) -> np.ndarray:
    """fp16 LUT bits (512, 2) -> float64 values."""
    return np.asarray(lut, dtype=np.uint16).view(np.float16).astype(np.float64)


# ---- LUT construction --------------------------------------------------------

def normal_pairs(seed: int, first: int, count: int) -> np.ndarray:
    out = np.empty((count, 2), dtype=np.float64)
    lib().orc_normal_pairs(seed, first, count, _p(out, C.c_double))
    return out


def lloyd_lut(seed: int, n_pairs: int, n_cent: int, iters: int, n_threads: int | None = None):
    """Lloyd k-means centroids (n_cent, 2) float64, their fp16 bits, and the MSE per coordinate."""
    cent = np.empty((n_cent, 2), dtype=np.float64)
    lut = np.empty((n_cent, 2), dtype=np.uint16)
    mse = lib().orc_lloyd_lut(seed, n_pairs, n_cent, iters, n_threads or n_threads_default(),
                              _p(cent, C.c_double), _p(lut, C.c_uint16))
    return cent, lut, mse


# ---- decoder -------------------------------------------------------------------

def window_states(code: np.ndarray, d: int, k: int) -> np.ndarray:
    code = np.ascontiguousarray(code, dtype=np.uint8)
    out = np.empty(d // 2, dtype=np.uint32)
    lib().orc_window_states(_p(code, C.c_uint8), d, k, _p(out, C.c_uint32))
    return out


def state_hash(states: np.ndarray):
    states = np.ascontiguousarray(states, dtype=np.uint32)
    idx = np.empty_like(states)
    neg = np.empty_like(states)
    lib().orc_state_hash(_p(states, C.c_uint32), states.size, _p(idx, C.c_uint32),
                         _p(neg, C.c_uint32))
    return idx, neg


def decode_f(code: np.ndarray, d: int, k: int, lut: np.ndarray) -> np.ndarray:
    code = np.ascontiguousarray(code, dtype=np.uint8)
    lut = np.ascontiguousarray(lut, dtype=np.uint16)
    f = np.empty(d, dtype=np.float64)
    lib().orc_decode_f(_p(code, C.c_uint8), d, k, _p(lut, C.c_uint16), _p(f, C.c_double))
    return f


def lookup_decode(records: np.ndarray, n_rows: int, d: int, k: int, rec_bytes: int,
                  lut: np.ndarray, idx: np.ndarray, n_threads: int = 1):
    """bf16 bits (n, d) of the reconstructed rows, and the count of out-of-range ids."""
    records = np.ascontiguousarray(records, dtype=np.uint8)
    lut = np.ascontiguousarray(lut, dtype=np.uint16)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty((idx.size, d), dtype=np.uint16)
    bad = lib().orc_lookup_decode(_p(records, C.c_uint8), n_rows, d, k, rec_bytes,
                                  _p(lut, C.c_uint16), _p(idx, C.c_int64), idx.size,
                                  _p(out, C.c_uint16), n_threads)
    return out, int(bad)


def lookup_decode_mixed(records: np.ndarray, offsets: np.ndarray, d: int, lut: np.ndarray,
                        idx: np.ndarray):
    """bf16 bits (n, d) for a table with one bit rate per row (record r at
    [offsets[r], offsets[r+1])), and the count of unusable ids."""
    records = np.ascontiguousarray(records, dtype=np.uint8)
    offsets = np.ascontiguousarray(offsets, dtype=np.uint64)
    lut = np.ascontiguousarray(lut, dtype=np.uint16)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty((idx.size, d), dtype=np.uint16)
    bad = lib().orc_lookup_decode_mixed(_p(records, C.c_uint8), _p(offsets, C.c_uint64),
                                        offsets.size - 1, d, _p(lut, C.c_uint16),
                                        _p(idx, C.c_int64), idx.size, _p(out, C.c_uint16))
    return out, int(bad)


def lookup_decode_reduce(records: np.ndarray, n_rows: int, d: int, k: int, rec_bytes: int,
                         lut: np.ndarray, idx: np.ndarray, group: int,
                         weights: np.ndarray | None = None, n_threads: int = 1):
    """bf16 bits (n_groups, d): per group of `group` lookups, the fp32 fmaf-accumulated
    weighted sum of the decoded bf16 rows, rounded once to bf16; and the out-of-range count."""
    records = np.ascontiguousarray(records, dtype=np.uint8)
    lut = np.ascontiguousarray(lut, dtype=np.uint16)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    assert idx.size % group == 0
    n_groups = idx.size // group
    wp = None
    if weights is not None:
        weights = np.ascontiguousarray(weights, dtype=np.float32)
        assert weights.size == idx.size
        wp = _p(weights, C.c_float)
    out = np.empty((n_groups, d), dtype=np.uint16)
    bad = lib().orc_lookup_decode_reduce(_p(records, C.c_uint8), n_rows, d, k, rec_bytes,
                                         _p(lut, C.c_uint16), _p(idx, C.c_int64), n_groups, group,
                                         wp, _p(out, C.c_uint16), n_threads)
    return out, int(bad)


# ---- encoder -------------------------------------------------------------------

def distortion(z: np.ndarray, code: np.ndarray, d: int, k: int, lut: np.ndarray) -> float:
    z = np.ascontiguousarray(z, dtype=np.float64)
    code = np.ascontiguousarray(code, dtype=np.uint8)
    lut = np.ascontiguousarray(lut, dtype=np.uint16)
    return lib().orc_distortion(_p(z, C.c_double), _p(code, C.c_uint8), d, k, _p(lut, C.c_uint16))


def encode_z(z: np.ndarray, d: int, k: int, lut: np.ndarray, mode: int):
    z = np.ascontiguousarray(z, dtype=np.float64)
    lut = np.ascontiguousarray(lut, dtype=np.uint16)
    code = np.zeros((d * k // 2 + 7) // 8, dtype=np.uint8)
    cost = lib().orc_encode_z(_p(z, C.c_double), d, k, _p(lut, C.c_uint16), mode,
                              _p(code, C.c_uint8))
    if cost < 0:
        raise ValueError("search mode does not apply to this geometry")
    return code, cost


def encode_rows(e: np.ndarray, d: int, k: int, lut: np.ndarray, mode: int = TWO_PASS,
                n_threads: int | None = None):
    """AoS records (rows, d*k/16 + 2) uint8, pre-rounding alphas, and search costs."""
    e = np.ascontiguousarray(e, dtype=np.float64).reshape(-1, d)
    lut = np.ascontiguousarray(lut, dtype=np.uint16)
    rows = e.shape[0]
    rec_bytes = d * k // 16 + 2
    rec = np.zeros((rows, rec_bytes), dtype=np.uint8)
    alpha = np.empty(rows, dtype=np.float64)
    cost = np.empty(rows, dtype=np.float64)
    rc = lib().orc_encode_rows(_p(e, C.c_double), rows, d, k, _p(lut, C.c_uint16), mode,
                               n_threads or n_threads_default(), _p(rec, C.c_uint8),
                               _p(alpha, C.c_double), _p(cost, C.c_double))
    if rc != 0:
        raise ValueError("encode_rows failed (geometry or mode)")
    return rec, alpha, cost


def distortion_f32(z: np.ndarray, code: np.ndarray, d: int, k: int, lut: np.ndarray) -> float:
    z = np.ascontiguousarray(z, dtype=np.float32)
    code = np.ascontiguousarray(code, dtype=np.uint8)
    lut = np.ascontiguousarray(lut, dtype=np.uint16)
    return lib().orc_distortion_f32(_p(z, C.c_float), _p(code, C.c_uint8), d, k,
                                    _p(lut, C.c_uint16))


def encode_z_f32(z: np.ndarray, d: int, k: int, lut: np.ndarray, mode: int):
    """fp32 search (the GPU encoder's precision): code and fp32 cost."""
    z = np.ascontiguousarray(z, dtype=np.float32)
    lut = np.ascontiguousarray(lut, dtype=np.uint16)
    code = np.zeros((d * k // 2 + 7) // 8, dtype=np.uint8)
    cost = lib().orc_encode_z_f32(_p(z, C.c_float), d, k, _p(lut, C.c_uint16), mode,
                                  _p(code, C.c_uint8))
    if cost < 0:
        raise ValueError("search mode does not apply to this geometry")
    return code, cost


def free_start_f32(z: np.ndarray, d: int, k: int, lut: np.ndarray, rho: int | None = None,
                   brute: bool = False):
    """First pass of the two-pass search (test hook): free-start fp32 Viterbi over the
    steps in the order rho, rho + 1, ... (mod T; default rho = T/2).  Returns (cost,
    states of the best path at each original step).  brute=True: the same minimum by
    enumerating every path (small T only)."""
    T = d // 2
    rho = T // 2 if rho is None else rho
    z = np.ascontiguousarray(z, dtype=np.float32)
    lut = np.ascontiguousarray(lut, dtype=np.uint16)
    states = np.zeros(T, dtype=np.uint32)
    fn = lib().orc_free_start_brute_f if brute else lib().orc_free_start_f
    cost = fn(_p(z, C.c_float), d, k, _p(lut, C.c_uint16), rho, _p(states, C.c_uint32))
    return cost, states


def encode_rows_f32(e: np.ndarray, d: int, k: int, lut: np.ndarray,
                    n_threads: int | None = None):
    """AoS records (rows, d*k/16 + 2) from fp32 rows with the fp32 two-pass search, and costs."""
    e = np.ascontiguousarray(e, dtype=np.float32).reshape(-1, d)
    lut = np.ascontiguousarray(lut, dtype=np.uint16)
    rows = e.shape[0]
    rec = np.zeros((rows, d * k // 16 + 2), dtype=np.uint8)
    cost = np.empty(rows, dtype=np.float32)
    rc = lib().orc_encode_rows_f32(_p(e, C.c_float), rows, d, k, _p(lut, C.c_uint16),
                                   n_threads or n_threads_default(), _p(rec, C.c_uint8),
                                   _p(cost, C.c_float))
    if rc != 0:
        raise ValueError("encode_rows_f32: geometry not supported")
    return rec, cost


def rtn2(e: np.ndarray, variant: int = 0) -> np.ndarray:
    e = np.ascontiguousarray(e, dtype=np.float64)
    out = np.empty_like(e)
    lib().orc_rtn2(_p(e, C.c_double), e.size, variant, _p(out, C.c_double))
    return out
