"""The INT8 copy for the Q pass against the oracle (needs a GB300; every test is
marked gpu).

The device quantiser must give the oracle's q and FP32 scales bit for bit
(integer results decided in FP32 on both sides: amax / 127, w / scale, round
half to even).  The product must meet |y - y_ref| <= 2^-8 sum_k |x q scale|
against the oracle's float64 sum, and with one-hot activations it must be
exactly the FP32 value of q * scale.
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL

pytestmark = pytest.mark.gpu

BOUND = 2.0 ** -8


@pytest.fixture(scope="module")
def w12():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__._load_builder().build()
    import lossless_bit_weight_skinny_gb300 as m

    return m


def _dev(W):
    import torch

    return torch.from_numpy(np.ascontiguousarray(W).view(np.int16)).cuda()


def _xdev(x_bits):
    import torch

    return _dev(x_bits).view(torch.bfloat16)


def _specials():
    rng = np.random.Generator(np.random.PCG64(61))
    W = rng.integers(0, 65536, size=(70, 320), dtype=np.uint16)  # every kind of pattern, Inf/NaN included
    W[3] = 0
    W[4] = 0x0001  # a subnormal row
    W[5, :] = 0x7F80  # all +Inf
    return W


CASES = {
    "projection_300x800": lambda: WL.projection_weights(300, 800, seed=62, outlier_frac=2e-3),
    "heavy_640x1024": lambda: WL.heavy_weights(640, 1024, seed=63),
    "specials_70x320": _specials,
    "ragged_k_129x777": lambda: WL.projection_weights(129, 777, seed=64),
    "kv_1024x5120": lambda: WL.projection_weights(1024, 5120, seed=65),
}
_cache = {}


def _prepared(w12, name):
    if name not in _cache:
        W = CASES[name]()
        q, sc = O.i8_quantize(W)
        _cache[name] = (W, q, sc, w12.w12_i8_encode_device(_dev(W)))
    return _cache[name]


@pytest.mark.parametrize("name", list(CASES.keys()))
def test_quantise_bit_exact(w12, name):
    W, q, sc, qd = _prepared(w12, name)
    gq, gsc = w12.w12_i8_download(qd)
    assert np.array_equal(gq, q)
    assert np.array_equal(gsc.view(np.uint32), sc.view(np.uint32))


def test_from_dev_equals_direct(w12):
    W, q, sc, _ = _prepared(w12, "projection_300x800")
    d = w12.w12_upload(w12.w12_encode(W))
    gq, gsc = w12.w12_i8_download(w12.w12_i8_from_dev(d))
    assert np.array_equal(gq, q) and np.array_equal(gsc, sc)


@pytest.mark.parametrize("M", (1, 2, 3, 16, 33, 64, 128, 200))
@pytest.mark.parametrize("name", ["projection_300x800", "heavy_640x1024", "kv_1024x5120"])
def test_gemm_i8_parity(w12, name, M):
    W, q, sc, qd = _prepared(w12, name)
    x = WL.activations(M, W.shape[1], seed=900 + M)
    y = w12.w12_gemm_i8(_xdev(x), qd).cpu().numpy().astype(np.float64)
    assert w12.w12_i8_status(qd) == 0
    ref = O.gemm_i8(x, q, sc)
    scale = O.abs_gemm_i8(x, q, sc)
    bad = ~(np.abs(y - ref) <= BOUND * scale)
    assert not bad.any(), f"{name} M={M}: {bad.sum()} outside the bound"


@pytest.mark.parametrize("M", (1, 16, 64))
def test_gemm_i8_one_hot_exact(w12, M):
    W, q, sc, qd = _prepared(w12, "heavy_640x1024")
    K = W.shape[1]
    want = (q.astype(np.float64) * sc.astype(np.float64)[:, None]).astype(np.float32)
    for k0 in (0, 1, 255, 256, 700, K - M):
        x = np.zeros((M, K), dtype=np.uint16)
        for m in range(M):
            x[m, k0 + m] = 0x3F80
        y = w12.w12_gemm_i8(_xdev(x), qd).cpu().numpy()
        for m in range(M):
            np.testing.assert_array_equal(y[m], want[:, k0 + m], err_msg=f"M={M} k={k0 + m}")


def test_gemm_i8_epilogues_and_errors(w12):
    import ctypes

    import torch

    W, q, sc, qd = _prepared(w12, "projection_300x800")
    x = WL.activations(5, W.shape[1], seed=950)
    xd = _xdev(x)
    yf = w12.w12_gemm_i8(xd, qd)
    yb = w12.w12_gemm_i8(xd, qd, out_bf16=True, input_ready=True)
    assert torch.equal(yb.cpu(), yf.cpu().to(torch.bfloat16))
    h = w12.w12_gemm_i8(xd, qd, silu_mul=True).cpu().numpy().astype(np.float64)
    ref = O.gemm_i8(x, q, sc)
    hr = O.silu_mul(ref)
    tol = BOUND * O.abs_gemm_i8(x, q, sc)
    g = ref[:, 0::2]
    sg = np.abs(O.silu_mul(np.stack([g, np.ones_like(g)], axis=2).reshape(g.shape[0], -1)))
    lim = (sg + 1.1 * tol[:, 0::2]) * tol[:, 1::2] + 1.1 * tol[:, 0::2] * np.abs(ref[:, 1::2])
    lim = (lim + 2.0 ** -20 * (np.abs(hr) + lim)) * (1 + 1e-6)
    assert np.all(np.abs(h - hr) <= lim)
    lib = w12.lib()
    P = ctypes.c_void_p
    s = P(torch.cuda.current_stream().cuda_stream)
    y = torch.empty((5, 300), device="cuda")
    assert lib.w12_gemm_i8(P(xd.data_ptr()), qd.ptr, P(y.data_ptr()), 5, 300, 800, 1, s) == 1  # Q8VIEW: not a flag here
    assert lib.w12_gemm_i8(P(xd.data_ptr()), qd.ptr, P(y.data_ptr()), 5, 301, 800, 0, s) == 2
    assert lib.w12_gemm_i8(P(xd.data_ptr()), qd.ptr, P(y.data_ptr()), 257, 300, 800, 0, s) == 4
    out = P()
    assert lib.w12_i8_encode_device(None, 4, 4, s, ctypes.byref(out)) == 1


@pytest.mark.parametrize("M", (1, 64))
def test_gemm_i8_full_size_sampled(w12, M):
    import torch

    W = WL.projection_weights(17408, 5120, seed=66)
    qd = w12.w12_i8_encode_device(torch.from_numpy(W.view(np.int16)).cuda())
    gq, gsc = w12.w12_i8_download(qd)
    rows = np.unique(np.concatenate([np.random.Generator(np.random.PCG64(M)).choice(17408, 64, replace=False),
                                     [0, 127, 128, 17407]]))
    q, sc = O.i8_quantize(W[rows])
    assert np.array_equal(gq[rows], q) and np.array_equal(gsc[rows], sc)
    x = WL.activations(M, 5120, seed=960 + M)
    y = w12.w12_gemm_i8(_xdev(x), qd).cpu().numpy().astype(np.float64)[:, rows]
    ref = O.gemm_i8(x, q, sc)
    assert np.all(np.abs(y - ref) <= BOUND * O.abs_gemm_i8(x, q, sc))
