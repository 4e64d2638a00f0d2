"""Python binding of the W12 library (lossless 12-bit BF16 weights + skinny GEMM).

Argument marshalling only: every step of the encode, upload, decode and GEMM
runs in ``_lib/libw12.so`` (host C++ and sm_103a CUDA kernels).  PyTorch is
used for device memory and streams.  There is no fallback: if the library is
missing or fails to load, importing this package raises ImportError.

Function names mirror the C ABI in ``include/w12.h``:

    h = w12_encode(w_bits)                 # host handle (CPU)
    d = w12_upload(h)                      # device handle, current device/stream
    y = w12_gemm(x, d)                     # x: cuda bf16 [M][K] -> y: cuda f32 [M][N]
    y = w12_gemm_q8view(x, d)              # Q pass over the nested 8-bit view
    w = w12_decode(d)                      # cuda int16 [N][K], bit-exact BF16 patterns
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libw12.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"W12 library not built: {LIB_PATH} is missing "
        "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
try:
    _lib = ctypes.CDLL(LIB_PATH)
except OSError as e:  # pragma: no cover - load failure is fatal
    raise ImportError(f"W12 library failed to load: {e}") from e

W12_OK = 0
STATUS_NAMES = {
    0: "OK", 1: "INVALID_ARG", 2: "SHAPE", 3: "ALIGNMENT", 4: "UNSUPPORTED", 5: "OOM",
    6: "CUDA", 7: "CORRUPT", 8: "TIMEOUT", 9: "IO",
}

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_ST = ctypes.c_int


class GemmPlan(ctypes.Structure):
    _fields_ = [
        ("kernel", ctypes.c_int), ("tile_rows", ctypes.c_int), ("block_rows", ctypes.c_int),
        ("grid", ctypes.c_int), ("row_blocks", ctypes.c_int64), ("k_steps", ctypes.c_int64),
        ("split_row_blocks", ctypes.c_int64), ("separate_fixup", ctypes.c_int), ("partial_bytes", ctypes.c_size_t),
    ]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class Stats(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("n_escapes", ctypes.c_int64),
        ("n_tiles", ctypes.c_int64), ("max_escapes_per_tile", ctypes.c_int64),
        ("bits_per_weight", ctypes.c_double), ("escape_fraction", ctypes.c_double),
        ("bytes_total", ctypes.c_size_t), ("bytes_ae", ctypes.c_size_t),
        ("bytes_b", ctypes.c_size_t),
    ]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


def _sig(name, args, res=_ST):
    f = getattr(_lib, name)
    f.argtypes = args
    f.restype = res
    return f


_sig("w12_status_string", [_ST], ctypes.c_char_p)
_sig("w12_encode", [_P, _I64, _I64, _I, ctypes.POINTER(_P)])
_sig("w12_encode_ex", [_P, _I64, _I64, _I, ctypes.c_uint, ctypes.POINTER(_P)])
_sig("w12_host_free", [_P], None)
_sig("w12_host_stats", [_P, ctypes.POINTER(Stats)])
_sig("w12_host_view", [_P] + [ctypes.POINTER(_P)] * 5)
_sig("w12_validate", [_P])
_sig("w12_serialize", [_P, _P, ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t)])
_sig("w12_deserialize", [_P, ctypes.c_size_t, ctypes.POINTER(_P)])
_sig("w12_save", [_P, ctypes.c_char_p])
_sig("w12_load", [ctypes.c_char_p, ctypes.POINTER(_P)])
_sig("w12_upload", [_P, _P, ctypes.POINTER(_P)])
_sig("w12_dev_free", [_P], None)
_sig("w12_encode_device", [_P, _I64, _I64, _P, ctypes.POINTER(_P)])
_sig("w12_encode_device_ex", [_P, _I64, _I64, ctypes.c_uint, _P, ctypes.POINTER(_P)])
_sig("w12_i8_encode_device", [_P, _I64, _I64, _P, ctypes.POINTER(_P)])
_sig("w12_i8_from_dev", [_P, _P, ctypes.POINTER(_P)])
_sig("w12_i8_free", [_P], None)
_sig("w12_i8_download", [_P, _P, _P, _P])
_sig("w12_i8_status", [_P, _P])
_sig("w12_gemm_i8", [_P, _P, _P, _I, _I, _I, ctypes.c_uint, _P])
_sig("w12_gemm_plan", [_I, _I64, _I64, _I, ctypes.POINTER(GemmPlan)])
_sig("w12_gemm_plan_grouped", [_I, ctypes.POINTER(_I64), _I, _I64, _I, ctypes.POINTER(GemmPlan)])
_sig("w12_download", [_P, _P, ctypes.POINTER(_P)])
_sig("w12_dev_info", [_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64), ctypes.POINTER(ctypes.c_size_t)])
_sig("w12_gemm", [_P, _P, _P, _I, _I, _I, _P])
_sig("w12_gemm_q8view", [_P, _P, _P, _I, _I, _I, _P])
_sig("w12_gemm_ex", [_P, _P, _P, _I, _I, _I, ctypes.c_uint, _P])
_sig("w12_gemm_grouped", [_P, _P, _P, _I, _I, _I, ctypes.c_uint, _P])
_sig("w12_gemm_grouped_host", [_P, _P, _P, _P, _P, _I, _I, _I, ctypes.c_uint, _P])
_sig("w12_gemm_host", [_P, _P, _P, _P, _P, _I, _I, _I, _P])
_sig("w12_gemm_noalloc", [_P, _P, _P, _I, _I, _I, _P])
_sig("w12_last_cuda_error", [], ctypes.c_char_p)
_sig("w12_decode", [_P, _P, _P])
_sig("w12_dev_status", [_P, _P])
_sig("w12_release_workspaces", [])
_sig("w12_set_spin_limit", [ctypes.c_uint32], None)
_sig("w12_debug_inject_stall", [_I], None)

EXPORTED = (
    "w12_status_string", "w12_encode", "w12_host_free", "w12_host_stats", "w12_host_view",
    "w12_validate", "w12_serialize", "w12_deserialize", "w12_save", "w12_load", "w12_upload",
    "w12_dev_free", "w12_dev_info", "w12_gemm", "w12_gemm_q8view", "w12_gemm_host",
    "w12_decode", "w12_dev_status", "w12_release_workspaces", "w12_set_spin_limit",
    "w12_debug_inject_stall", "w12_gemm_noalloc", "w12_last_cuda_error", "w12_gemm_ex",
    "w12_encode_device", "w12_download", "w12_encode_ex", "w12_encode_device_ex",
    "w12_i8_encode_device", "w12_i8_from_dev", "w12_i8_free", "w12_i8_download", "w12_i8_status", "w12_gemm_i8",
    "w12_gemm_plan", "w12_gemm_grouped", "w12_gemm_grouped_host", "w12_gemm_plan_grouped",
)

W12_GEMM_Q8VIEW = 1
W12_GEMM_INPUT_READY = 2
W12_GEMM_OUT_BF16 = 4
W12_GEMM_SILU_MUL = 8
W12_ENCODE_COUNT_MAX = 1


class W12Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.w12_status_string(status).decode()
        if status == 6:
            msg += ": " + _lib.w12_last_cuda_error().decode()
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({msg})")


def _check(st: int, where: str):
    if st != W12_OK:
        raise W12Error(st, where)


def _u16_host(w) -> np.ndarray:
    """Host BF16 bit patterns as a contiguous uint16 numpy array."""
    try:
        import torch
        if isinstance(w, torch.Tensor):
            if w.is_cuda:
                raise ValueError("w12_encode takes a host tensor")
            if w.dtype == torch.bfloat16:
                w = w.view(torch.int16)
            w = w.contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(w)
    if a.dtype in (np.int16,):
        a = a.view(np.uint16)
    if a.dtype != np.uint16 or a.ndim != 2:
        raise TypeError("expected a 2-D array of BF16 bit patterns (uint16/int16/bfloat16)")
    return a


class Host:
    """An encoded matrix in host memory (owns a ``w12_host*``)."""

    def __init__(self, ptr: int, N: int, K: int):
        self._ptr = ptr
        self.N, self.K = N, K

    @property
    def ptr(self):
        return self._ptr

    def __del__(self):
        if getattr(self, "_ptr", None):
            _lib.w12_host_free(self._ptr)
            self._ptr = None

    def stats(self) -> dict:
        s = Stats()
        _check(_lib.w12_host_stats(self._ptr, ctypes.byref(s)), "w12_host_stats")
        return s.as_dict()

    def validate(self) -> int:
        return _lib.w12_validate(self._ptr)

    def view(self):
        """(ebase, ae, b, tile_ptr, esc) as numpy arrays (copies)."""
        ptrs = [_P() for _ in range(5)]
        _check(_lib.w12_host_view(self._ptr, *[ctypes.byref(p) for p in ptrs]), "w12_host_view")
        st = self.stats()
        N, K = self.N, self.K
        brow = 4 * ((K + 7) // 8)
        sizes = [(N, np.uint8), (N * K, np.uint8), (N * brow, np.uint8),
                 (st["n_tiles"] + 1, np.uint32), (st["n_escapes"], np.uint32)]
        out = []
        for p, (n, dt) in zip(ptrs, sizes):
            if n == 0 or not p.value:
                out.append(np.zeros(n, dtype=dt))
            else:
                buf = (ctypes.c_char * (n * np.dtype(dt).itemsize)).from_address(p.value)
                out.append(np.frombuffer(buf, dtype=dt).copy())
        ebase, ae, b, tptr, esc = out
        return ebase, ae.reshape(N, K), b.reshape(N, brow), tptr, esc

    def serialize(self) -> bytes:
        n = ctypes.c_size_t()
        _check(_lib.w12_serialize(self._ptr, None, 0, ctypes.byref(n)), "w12_serialize")
        buf = ctypes.create_string_buffer(max(n.value, 1))
        _check(_lib.w12_serialize(self._ptr, buf, n.value, ctypes.byref(n)), "w12_serialize")
        return buf.raw[:n.value]

    def save(self, path: str):
        _check(_lib.w12_save(self._ptr, path.encode()), "w12_save")

    def upload(self, stream=None) -> "Dev":
        return w12_upload(self, stream)


class Dev:
    """An encoded matrix in device memory (owns a ``w12_dev*``)."""

    def __init__(self, ptr: int, N: int, K: int, host: Host | None = None):
        self._ptr = ptr
        self.N, self.K = N, K
        self._host = host  # keeps the source alive until the uploads have run

    @property
    def ptr(self):
        return self._ptr

    def free(self):
        if getattr(self, "_ptr", None):
            _lib.w12_dev_free(self._ptr)
            self._ptr = None

    def __del__(self):
        self.free()

    def device_bytes(self) -> int:
        n, k, b = _I64(), _I64(), ctypes.c_size_t()
        _check(_lib.w12_dev_info(self._ptr, ctypes.byref(n), ctypes.byref(k), ctypes.byref(b)), "w12_dev_info")
        return b.value


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ---- the C ABI, one Python function per entry point -------------------------

def w12_encode(w_bits, n_threads: int = 0, count_max: bool = False) -> Host:
    """Encode host BF16 bit patterns [N][K]; count_max selects count-maximising
    windows (W12_ENCODE_COUNT_MAX) instead of max-anchored ones."""
    a = _u16_host(w_bits)
    N, K = a.shape
    out = _P()
    flags = W12_ENCODE_COUNT_MAX if count_max else 0
    _check(_lib.w12_encode_ex(a.ctypes.data_as(_P), N, K, n_threads, flags, ctypes.byref(out)), "w12_encode")
    return Host(out.value, N, K)


def w12_deserialize(blob: bytes) -> Host:
    out = _P()
    buf = ctypes.create_string_buffer(blob, len(blob))
    _check(_lib.w12_deserialize(buf, len(blob), ctypes.byref(out)), "w12_deserialize")
    h = Host(out.value, 0, 0)
    st = h.stats()
    h.N, h.K = st["N"], st["K"]
    return h


def w12_load(path: str) -> Host:
    out = _P()
    _check(_lib.w12_load(path.encode(), ctypes.byref(out)), "w12_load")
    h = Host(out.value, 0, 0)
    st = h.stats()
    h.N, h.K = st["N"], st["K"]
    return h


def w12_upload(h: Host, stream=None) -> Dev:
    out = _P()
    _check(_lib.w12_upload(h.ptr, _stream_ptr(stream), ctypes.byref(out)), "w12_upload")
    return Dev(out.value, h.N, h.K, host=h)


def w12_encode_device(w, stream=None, count_max: bool = False) -> Dev:
    """Encode a CUDA tensor of BF16 weights [N][K] (bfloat16 or its int16 /
    uint16 bit view) on the device; the arrays equal
    w12_upload(w12_encode(w, count_max=count_max))."""
    import torch
    if not (isinstance(w, torch.Tensor) and w.is_cuda and w.dim() == 2 and w.is_contiguous() and w.element_size() == 2
            and w.dtype in (torch.bfloat16, torch.int16, torch.uint16)):
        raise TypeError("w must be a contiguous CUDA [N][K] tensor of BF16 (or its 16-bit pattern)")
    N, K = w.shape
    out = _P()
    flags = W12_ENCODE_COUNT_MAX if count_max else 0
    _check(_lib.w12_encode_device_ex(ctypes.c_void_p(w.data_ptr()), N, K, flags, _stream_ptr(stream),
                                     ctypes.byref(out)), "w12_encode_device")
    return Dev(out.value, N, K)


class I8:
    """An INT8 copy of a weight matrix for the Q pass (owns a ``w12_i8*``)."""

    def __init__(self, ptr: int, N: int, K: int):
        self._ptr = ptr
        self.N, self.K = N, K

    @property
    def ptr(self):
        return self._ptr

    def free(self):
        if getattr(self, "_ptr", None):
            _lib.w12_i8_free(self._ptr)
            self._ptr = None

    def __del__(self):
        self.free()


def w12_i8_encode_device(w, stream=None) -> I8:
    """INT8 copy (per-row FP32 scale, round half to even) of a CUDA [N][K]
    tensor of BF16 weights (bfloat16 or its 16-bit pattern)."""
    import torch
    if not (isinstance(w, torch.Tensor) and w.is_cuda and w.dim() == 2 and w.is_contiguous() and w.element_size() == 2
            and w.dtype in (torch.bfloat16, torch.int16, torch.uint16)):
        raise TypeError("w must be a contiguous CUDA [N][K] tensor of BF16 (or its 16-bit pattern)")
    N, K = w.shape
    out = _P()
    _check(_lib.w12_i8_encode_device(ctypes.c_void_p(w.data_ptr()), N, K, _stream_ptr(stream), ctypes.byref(out)),
           "w12_i8_encode_device")
    return I8(out.value, N, K)


def w12_i8_from_dev(d: Dev, stream=None) -> I8:
    """INT8 copy of the weights a W12 device handle holds."""
    out = _P()
    _check(_lib.w12_i8_from_dev(d.ptr, _stream_ptr(stream), ctypes.byref(out)), "w12_i8_from_dev")
    return I8(out.value, d.N, d.K)


def w12_i8_download(q: I8, stream=None):
    """(q [N][K] int8, scale [N] float32) as numpy arrays."""
    qh = np.zeros((q.N, q.K), dtype=np.int8)
    sh = np.zeros(q.N, dtype=np.float32)
    _check(_lib.w12_i8_download(q.ptr, qh.ctypes.data_as(_P), sh.ctypes.data_as(_P), _stream_ptr(stream)),
           "w12_i8_download")
    return qh, sh


def w12_i8_status(q: I8, stream=None) -> int:
    return int(_lib.w12_i8_status(q.ptr, _stream_ptr(stream)))


def w12_gemm_i8(x, q: I8, y=None, stream=None, input_ready=False, out_bf16=False, silu_mul=False):
    """The Q pass over an INT8 copy: y = scale * (x . q^T), flags as w12_gemm_ex."""
    import torch
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()):
        raise TypeError("x must be a contiguous CUDA bfloat16 [M][K] tensor")
    M, K = x.shape
    cols = q.N // 2 if silu_mul else q.N
    dt = torch.bfloat16 if out_bf16 else torch.float32
    y = _out(x, y, M, cols, dt)
    flags = ((W12_GEMM_INPUT_READY if input_ready else 0) | (W12_GEMM_OUT_BF16 if out_bf16 else 0)
             | (W12_GEMM_SILU_MUL if silu_mul else 0))
    _check(_lib.w12_gemm_i8(ctypes.c_void_p(x.data_ptr()), q.ptr, ctypes.c_void_p(y.data_ptr()), M, q.N, K, flags,
                            _stream_ptr(stream)), "w12_gemm_i8")
    return y


def w12_download(d: Dev, stream=None) -> Host:
    """The device handle's arrays copied into a new host handle."""
    out = _P()
    _check(_lib.w12_download(d.ptr, _stream_ptr(stream), ctypes.byref(out)), "w12_download")
    return Host(out.value, d.N, d.K)


def _out(x, y, M, cols, dt):
    """The output buffer: a new [M][cols] tensor of dtype dt, or the caller's,
    which must be a contiguous CUDA tensor of that dtype on x's device with at
    least M * cols elements."""
    import torch
    if y is None:
        return torch.empty((M, cols), dtype=dt, device=x.device)
    if not (isinstance(y, torch.Tensor) and y.is_cuda and y.dtype == dt and y.is_contiguous()
            and y.device == x.device and y.numel() >= M * cols):
        raise TypeError(f"y must be a contiguous CUDA {dt} tensor on {x.device} of at least {M} x {cols} elements")
    return y


def _gemm(fn, name, x, d: Dev, y=None, stream=None):
    import torch
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()):
        raise TypeError("x must be a contiguous CUDA bfloat16 [M][K] tensor")
    M, K = x.shape
    y = _out(x, y, M, d.N, torch.float32)
    _check(fn(ctypes.c_void_p(x.data_ptr()), d.ptr, ctypes.c_void_p(y.data_ptr()), M, d.N, K,
              _stream_ptr(stream)), name)
    return y


def w12_gemm(x, d: Dev, y=None, stream=None):
    """y[M][N] = x[M][K] . W^T on the device (W decoded exactly on the fly)."""
    return _gemm(_lib.w12_gemm, "w12_gemm", x, d, y, stream)


def w12_gemm_q8view(x, d: Dev, y=None, stream=None):
    """The Q pass: the same product over the 8-bit A+E view only."""
    return _gemm(_lib.w12_gemm_q8view, "w12_gemm_q8view", x, d, y, stream)


def w12_gemm_ex(x, d: Dev, y=None, stream=None, q8view=False, input_ready=False, out_bf16=False,
                silu_mul=False):
    """w12_gemm (or the Q pass) with flags.  input_ready states that x was
    complete before the previous operation on the stream started, so the
    launch may read it at once and overlap that operation's tail.  out_bf16
    writes y as BF16 (round to nearest even); silu_mul treats rows 2i / 2i+1
    as a gate / up pair and writes y[M][N/2] = silu(gate) * up."""
    import torch
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()):
        raise TypeError("x must be a contiguous CUDA bfloat16 [M][K] tensor")
    M, K = x.shape
    cols = d.N // 2 if silu_mul else d.N
    dt = torch.bfloat16 if out_bf16 else torch.float32
    y = _out(x, y, M, cols, dt)
    flags = ((W12_GEMM_Q8VIEW if q8view else 0) | (W12_GEMM_INPUT_READY if input_ready else 0)
             | (W12_GEMM_OUT_BF16 if out_bf16 else 0) | (W12_GEMM_SILU_MUL if silu_mul else 0))
    _check(_lib.w12_gemm_ex(ctypes.c_void_p(x.data_ptr()), d.ptr, ctypes.c_void_p(y.data_ptr()), M, d.N, K,
                            flags, _stream_ptr(stream)), "w12_gemm_ex")
    return y


W12_MAX_GROUP = 4


def w12_gemm_grouped(x, devs, ys=None, stream=None, q8view=False, input_ready=False, out_bf16=False):
    """y_i = x . W_i^T for every handle in devs (all with x's K), in ONE
    launch: the q/k/v or gate/up projections that read the same activations.
    Returns the list of outputs (new tensors, or the caller's ys)."""
    import torch
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()):
        raise TypeError("x must be a contiguous CUDA bfloat16 [M][K] tensor")
    devs = list(devs)
    n = len(devs)
    if not 1 <= n <= W12_MAX_GROUP:
        raise ValueError(f"between 1 and {W12_MAX_GROUP} matrices per launch, not {n}")
    M, K = x.shape
    dt = torch.bfloat16 if out_bf16 else torch.float32
    ys = [None] * n if ys is None else list(ys)
    if len(ys) != n:
        raise ValueError("one output per matrix")
    ys = [_out(x, y, M, d.N, dt) for y, d in zip(ys, devs)]
    hs = (_P * n)(*[d.ptr for d in devs])
    ps = (_P * n)(*[y.data_ptr() for y in ys])
    flags = ((W12_GEMM_Q8VIEW if q8view else 0) | (W12_GEMM_INPUT_READY if input_ready else 0)
             | (W12_GEMM_OUT_BF16 if out_bf16 else 0))
    _check(_lib.w12_gemm_grouped(ctypes.c_void_p(x.data_ptr()), hs, ps, n, M, K, flags, _stream_ptr(stream)),
           "w12_gemm_grouped")
    return ys


def w12_gemm_grouped_host(x_host, x_dev, devs, ys_dev, ys_host, stream=None, out_bf16=False):
    """H2D copy of x, one grouped GEMM over devs, a D2H copy of every output,
    all on one stream (pinned host buffers; synchronise before reading)."""
    devs = list(devs)
    n = len(devs)
    M, K = x_host.shape
    hs = (_P * n)(*[d.ptr for d in devs])
    pd = (_P * n)(*[y.data_ptr() for y in ys_dev])
    ph = (_P * n)(*[y.data_ptr() for y in ys_host])
    flags = W12_GEMM_OUT_BF16 if out_bf16 else 0
    _check(_lib.w12_gemm_grouped_host(ctypes.c_void_p(x_host.data_ptr()), ctypes.c_void_p(x_dev.data_ptr()), hs, pd,
                                      ph, n, M, K, flags, _stream_ptr(stream)), "w12_gemm_grouped_host")
    return ys_host


def w12_gemm_noalloc(x, d: Dev, y, stream=None):
    """w12_gemm with its scratch in the library's fixed device array: no
    device allocation at all (y must be given).  Overlapping calls race."""
    return _gemm(_lib.w12_gemm_noalloc, "w12_gemm_noalloc", x, d, y, stream)


def w12_gemm_host(x_host, x_dev, d: Dev, y_dev, y_host, stream=None):
    """H2D copy of x, GEMM, D2H copy of y, all on one stream (pinned buffers)."""
    M, K = x_host.shape
    _check(_lib.w12_gemm_host(ctypes.c_void_p(x_host.data_ptr()), ctypes.c_void_p(x_dev.data_ptr()),
                              d.ptr, ctypes.c_void_p(y_dev.data_ptr()), ctypes.c_void_p(y_host.data_ptr()),
                              M, d.N, K, _stream_ptr(stream)), "w12_gemm_host")
    return y_host


def w12_decode(d: Dev, out=None, stream=None):
    """Bit-exact BF16 patterns [N][K] (int16 CUDA tensor)."""
    import torch
    if out is None:
        out = torch.empty((d.N, d.K), dtype=torch.int16, device="cuda")
    _check(_lib.w12_decode(d.ptr, ctypes.c_void_p(out.data_ptr()), _stream_ptr(stream)), "w12_decode")
    return out


def w12_dev_status(d: Dev, stream=None) -> int:
    """Synchronise and return (then clear) the handle's device status code."""
    return _lib.w12_dev_status(d.ptr, _stream_ptr(stream))


def w12_release_workspaces():
    _check(_lib.w12_release_workspaces(), "w12_release_workspaces")


def w12_set_spin_limit(limit_ns: int):
    _lib.w12_set_spin_limit(int(limit_ns))


def w12_debug_inject_stall(on: bool):
    _lib.w12_debug_inject_stall(1 if on else 0)


def lib():
    """The loaded ctypes library (for tests that call the C ABI directly)."""
    return _lib


def w12_gemm_plan_grouped(M: int, Ns, K: int, sm_count: int = 0) -> dict:
    """The launch w12_gemm_grouped makes for matrices of Ns rows (same K)."""
    Ns = list(Ns)
    arr = (_I64 * max(1, len(Ns)))(*Ns)
    p = GemmPlan()
    _check(_lib.w12_gemm_plan_grouped(M, arr, len(Ns), K, sm_count, ctypes.byref(p)), "w12_gemm_plan_grouped")
    return p.as_dict()


def w12_gemm_plan(M: int, N: int, K: int, sm_count: int = 0) -> dict:
    """The launch w12_gemm makes for M x N x K on a GPU with sm_count SMs
    (0: the current device's): kernel, tile rows, grid, split-K shape."""
    p = GemmPlan()
    _check(_lib.w12_gemm_plan(M, N, K, sm_count, ctypes.byref(p)), "w12_gemm_plan")
    return p.as_dict()
