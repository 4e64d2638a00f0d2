"""ctypes shim over ``w12_oracle.c`` (test infrastructure, never the product path).

The C file is compiled with plain ``gcc`` into ``oracle/_build/libw12oracle.so``
on first use (or by ``build()``).  Every wrapper takes and returns numpy arrays
of BF16 *bit patterns* (uint16) so that no floating-point conversion happens on
the Python side.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w12_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_NAME = "libw12oracle.so"

TILE_ROWS = 128
TILE_COLS = 256

_lock = threading.Lock()
_lib = None


def lib_path(src: str = _SRC, build_dir: str = _BUILD, name: str = _LIB_NAME) -> str:
    return os.path.join(build_dir, name)


def build(src: str = _SRC, build_dir: str = _BUILD, name: str = _LIB_NAME,
          extra_flags: tuple = ()) -> str:
    """Compile the oracle (no optimisation flags that change fp semantics)."""
    os.makedirs(build_dir, exist_ok=True)
    out = os.path.join(build_dir, name)
    if (not os.path.exists(out)) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c99", "-O2", "-fno-fast-math", "-ffp-contract=off",
               "-shared", "-fPIC", *extra_flags, src, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


_I64 = ctypes.c_int64
_P = ctypes.c_void_p


def _declare(lib):
    lib.orc_encoded_size.argtypes = [_P, _I64, _I64]
    lib.orc_encoded_size.restype = _I64
    lib.orc_encode.argtypes = [_P, _I64, _I64, _P, _I64]
    lib.orc_encode.restype = _I64
    lib.orc_encoded_size_count_max.argtypes = [_P, _I64, _I64]
    lib.orc_encoded_size_count_max.restype = _I64
    lib.orc_encode_count_max.argtypes = [_P, _I64, _I64, _P, _I64]
    lib.orc_encode_count_max.restype = _I64
    lib.orc_row_ebase_count_max.argtypes = [_P, _I64]
    lib.orc_row_ebase_count_max.restype = ctypes.c_int
    lib.orc_blob_header.argtypes = [_P, _I64, _P]
    lib.orc_blob_header.restype = ctypes.c_int
    lib.orc_decode.argtypes = [_P, _I64, _P]
    lib.orc_decode.restype = ctypes.c_int
    lib.orc_decode_rows.argtypes = [_P, _I64, _I64, _I64, _P]
    lib.orc_decode_rows.restype = ctypes.c_int
    lib.orc_decode_q8.argtypes = [_P, _I64, _P]
    lib.orc_decode_q8.restype = ctypes.c_int
    lib.orc_gemm.argtypes = [_P, _P, _I64, _I64, _I64, _P]
    lib.orc_gemm.restype = None
    lib.orc_gemm_rows.argtypes = [_P, _P, _I64, _I64, _I64, _I64, _I64, _P]
    lib.orc_gemm_rows.restype = None
    lib.orc_abs_gemm.argtypes = [_P, _P, _I64, _I64, _I64, _P]
    lib.orc_abs_gemm.restype = None
    lib.orc_row_ebase.argtypes = [_P, _I64]
    lib.orc_row_ebase.restype = ctypes.c_int
    lib.orc_num_tiles.argtypes = [_I64, _I64]
    lib.orc_num_tiles.restype = _I64
    lib.orc_b_row_bytes.argtypes = [_I64]
    lib.orc_b_row_bytes.restype = _I64
    lib.orc_i8_quantize.argtypes = [_P, _I64, _I64, _P, _P]
    lib.orc_i8_quantize.restype = None
    lib.orc_gemm_i8.argtypes = [_P, _P, _P, _I64, _I64, _I64, _P]
    lib.orc_gemm_i8.restype = None
    lib.orc_abs_gemm_i8.argtypes = [_P, _P, _P, _I64, _I64, _I64, _P]
    lib.orc_abs_gemm_i8.restype = None
    lib.orc_round_bf16.argtypes = [_P, _I64, _P]
    lib.orc_round_bf16.restype = None
    lib.orc_silu_mul.argtypes = [_P, _I64, _I64, _P]
    lib.orc_silu_mul.restype = None
    return lib


def load(path: str):
    """Load an oracle shared library from an explicit path (used for mutants)."""
    return _declare(ctypes.CDLL(path))


def _get():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load(build())
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("expected BF16 bit patterns as uint16")
    return a


def encode(w_bits: np.ndarray, lib=None, count_max: bool = False) -> bytes:
    """W[N][K] (uint16 BF16 bits) -> W12 blob bytes; count_max selects the
    count-maximising window (R13) instead of the max-anchored one (R1)."""
    lib = lib or _get()
    w = _u16(w_bits)
    N, K = w.shape
    size_fn = lib.orc_encoded_size_count_max if count_max else lib.orc_encoded_size
    enc_fn = lib.orc_encode_count_max if count_max else lib.orc_encode
    size = size_fn(_ptr(w), N, K)
    out = np.zeros(max(size, 1), dtype=np.uint8)
    n = enc_fn(_ptr(w), N, K, _ptr(out), size)
    if n != size:
        raise RuntimeError("oracle encode failed")
    return out[:size].tobytes()


def blob_header(blob: bytes, lib=None):
    """(N, K, n_esc, T) of a blob, or ValueError if it is malformed."""
    lib = lib or _get()
    b = np.frombuffer(blob, dtype=np.uint8)
    out = np.zeros(4, dtype=np.int64)
    if lib.orc_blob_header(_ptr(b), b.size, _ptr(out)) != 0:
        raise ValueError("malformed W12 blob")
    return tuple(int(v) for v in out)


def decode(blob: bytes, lib=None) -> np.ndarray:
    lib = lib or _get()
    N, K, _, _ = blob_header(blob, lib)
    b = np.frombuffer(blob, dtype=np.uint8)
    out = np.zeros((N, K), dtype=np.uint16)
    if lib.orc_decode(_ptr(b), b.size, _ptr(out)) != 0:
        raise ValueError("oracle decode failed")
    return out


def decode_rows(blob: bytes, n0: int, n1: int, lib=None) -> np.ndarray:
    lib = lib or _get()
    N, K, _, _ = blob_header(blob, lib)
    b = np.frombuffer(blob, dtype=np.uint8)
    out = np.zeros((n1 - n0, K), dtype=np.uint16)
    if lib.orc_decode_rows(_ptr(b), b.size, n0, n1, _ptr(out)) != 0:
        raise ValueError("oracle decode failed")
    return out


def decode_q8(blob: bytes, lib=None) -> np.ndarray:
    lib = lib or _get()
    N, K, _, _ = blob_header(blob, lib)
    b = np.frombuffer(blob, dtype=np.uint8)
    out = np.zeros((N, K), dtype=np.uint16)
    if lib.orc_decode_q8(_ptr(b), b.size, _ptr(out)) != 0:
        raise ValueError("oracle decode failed")
    return out


def gemm(x_bits: np.ndarray, w_bits: np.ndarray, lib=None) -> np.ndarray:
    """y[M][N] = x[M][K] . W[N][K]^T in float64, k in increasing order."""
    lib = lib or _get()
    x, w = _u16(x_bits), _u16(w_bits)
    M, K = x.shape
    N, K2 = w.shape
    assert K == K2
    y = np.zeros((M, N), dtype=np.float64)
    lib.orc_gemm(_ptr(x), _ptr(w), M, N, K, _ptr(y))
    return y


def gemm_rows(x_bits: np.ndarray, w_rows: np.ndarray, lib=None) -> np.ndarray:
    """The same GEMM for a block of already-decoded rows: returns [M][rows]."""
    lib = lib or _get()
    x, w = _u16(x_bits), _u16(w_rows)
    M, K = x.shape
    R, K2 = w.shape
    assert K == K2
    y = np.zeros((M, R), dtype=np.float64)
    lib.orc_gemm_rows(_ptr(x), _ptr(w), M, R, K, 0, R, _ptr(y))
    return y


def abs_gemm(x_bits: np.ndarray, w_bits: np.ndarray, lib=None) -> np.ndarray:
    """s[M][N] = sum_k |x[m][k] * W[n][k]| in float64."""
    lib = lib or _get()
    x, w = _u16(x_bits), _u16(w_bits)
    M, K = x.shape
    N, _ = w.shape
    s = np.zeros((M, N), dtype=np.float64)
    lib.orc_abs_gemm(_ptr(x), _ptr(w), M, N, K, _ptr(s))
    return s


def row_ebase(row_bits: np.ndarray, lib=None, count_max: bool = False) -> int:
    lib = lib or _get()
    r = _u16(row_bits).reshape(-1)
    fn = lib.orc_row_ebase_count_max if count_max else lib.orc_row_ebase
    return int(fn(_ptr(r), r.size))


def num_tiles(N: int, K: int, lib=None) -> int:
    return int((lib or _get()).orc_num_tiles(N, K))


def b_row_bytes(K: int, lib=None) -> int:
    return int((lib or _get()).orc_b_row_bytes(K))


def round_bf16(v, lib=None) -> np.ndarray:
    """FP32 values -> BF16 bit patterns, round to nearest, ties to even."""
    lib = lib or _get()
    a = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    out = np.zeros(a.shape, dtype=np.uint16)
    lib.orc_round_bf16(_ptr(a), a.size, _ptr(out))
    return out


def silu_mul(y, lib=None) -> np.ndarray:
    """h[M][N/2] = silu(y[:, 0::2]) * y[:, 1::2] in float64 (gate/up rows interleaved)."""
    lib = lib or _get()
    a = np.ascontiguousarray(np.asarray(y, dtype=np.float64))
    M, N = a.shape
    if N % 2:
        raise ValueError("silu_mul needs an even number of columns")
    h = np.zeros((M, N // 2), dtype=np.float64)
    lib.orc_silu_mul(_ptr(a), M, N, _ptr(h))
    return h


def i8_quantize(w_bits, lib=None):
    """INT8 copy (R14): (q[N][K] int8, scale[N] float32) of BF16 weights."""
    lib = lib or _get()
    w = _u16(w_bits)
    N, K = w.shape
    q = np.zeros((N, K), dtype=np.int8)
    sc = np.zeros(N, dtype=np.float32)
    lib.orc_i8_quantize(_ptr(w), N, K, _ptr(q), _ptr(sc))
    return q, sc


def gemm_i8(x_bits, q, scale, lib=None) -> np.ndarray:
    """y[M][N] = x . (q * scale)^T in float64, k ascending."""
    lib = lib or _get()
    x = _u16(x_bits)
    q = np.ascontiguousarray(q, dtype=np.int8)
    sc = np.ascontiguousarray(scale, dtype=np.float32)
    M, K = x.shape
    N = q.shape[0]
    y = np.zeros((M, N), dtype=np.float64)
    lib.orc_gemm_i8(_ptr(x), _ptr(q), _ptr(sc), M, N, K, _ptr(y))
    return y


def abs_gemm_i8(x_bits, q, scale, lib=None) -> np.ndarray:
    """s[M][N] = sum_k |x q scale| in float64."""
    lib = lib or _get()
    x = _u16(x_bits)
    q = np.ascontiguousarray(q, dtype=np.int8)
    sc = np.ascontiguousarray(scale, dtype=np.float32)
    M, K = x.shape
    N = q.shape[0]
    s = np.zeros((M, N), dtype=np.float64)
    lib.orc_abs_gemm_i8(_ptr(x), _ptr(q), _ptr(sc), M, N, K, _ptr(s))
    return s
