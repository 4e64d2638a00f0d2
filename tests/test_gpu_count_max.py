"""Count-maximising windows on the GPU (needs a GB300; every test is marked gpu).

With W12_ENCODE_COUNT_MAX the weights above a row's window escape too, and
their slot holds the saturated placeholder.  The device encoder must write
the oracle's blob byte for byte; the exact GEMM (both kernels) must meet the
GEMM bound against the oracle's float64 product of the decoded weights, and
be exact for one-hot activations (which pins the CUDA-core kernel's escape
correction, whose placeholder now depends on the escape); the Q pass must
meet the bound against the oracle's 8-bit view of the same blob, where the
top outliers read as the saturated value.
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


def _xdev(x_bits):
    import torch

    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda().view(torch.bfloat16)


def _outliers():
    W = WL.projection_weights(384, 2048, seed=71, outlier_frac=2e-3)
    W[130, 7] = 0x7180   # +2^100
    W[300, 2000] = 0xEC80  # -2^90
    W[17, 900] = 0x4300  # +128
    W[255, 5] = 0xC280   # -64
    return W


CASES = {
    "heavy_640x1024": lambda: WL.heavy_weights(640, 1024, seed=9),
    "outliers_384x2048": _outliers,
    "ragged_300x800": lambda: WL.projection_weights(300, 800, seed=7, outlier_frac=2e-3),
}
_cache = {}


def _prepared(w12, name):
    if name not in _cache:
        import torch

        W = CASES[name]()
        blob = O.encode(W, count_max=True)
        d = w12.w12_encode_device(torch.from_numpy(W.view(np.int16)).cuda(), count_max=True)
        _cache[name] = (W, blob, O.decode(blob), O.decode_q8(blob), d)
    return _cache[name]


def _check(y, x, Wref, what):
    ref = O.gemm_rows(x, Wref)
    scale = O.abs_gemm(x, Wref)
    fin = np.isfinite(ref)
    bad = fin & ~(np.abs(y - ref) <= BOUND * scale)
    assert not bad.any(), f"{what}: {bad.sum()} elements outside the bound"


@pytest.mark.parametrize("name", list(CASES.keys()))
def test_device_count_max_blob_equals_oracle(w12, name):
    W, blob, Wdec, _, d = _prepared(w12, name)
    assert w12.w12_download(d).serialize() == blob
    assert np.array_equal(Wdec, W)
    assert O.blob_header(blob)[2] <= O.blob_header(O.encode(W))[2]


@pytest.mark.parametrize("M", (1, 2, 3, 16, 64, 128))
@pytest.mark.parametrize("name", list(CASES.keys()))
def test_count_max_gemm_parity(w12, name, M):
    W, _, Wdec, _, d = _prepared(w12, name)
    x = WL.activations(M, W.shape[1], seed=700 + M)
    y = w12.w12_gemm(_xdev(x), d).cpu().numpy().astype(np.float64)
    assert w12.w12_dev_status(d) == 0
    _check(y, x, Wdec, f"{name} M={M}")


@pytest.mark.parametrize("M", (1, 2, 16, 64))
@pytest.mark.parametrize("name", list(CASES.keys()))
def test_count_max_q8_parity(w12, name, M):
    W, _, _, Wq, d = _prepared(w12, name)
    x = WL.activations(M, W.shape[1], seed=800 + M)
    y = w12.w12_gemm_q8view(_xdev(x), d).cpu().numpy().astype(np.float64)
    _check(y, x, Wq, f"q8 {name} M={M}")


@pytest.mark.parametrize("M", (1, 2, 16))
def test_count_max_one_hot_exact(w12, M):
    """x = unit rows: every output is exactly a weight, so the escape
    correction must cancel the saturated placeholder exactly."""
    W, _, _, _, d = _prepared(w12, "outliers_384x2048")
    K = W.shape[1]
    want = WL.bf16_bits_to_f32(W).astype(np.float64)
    cols = sorted({7, 2000, 900, 5, 0, 1, 1023, 2047} | set(range(3 * M, 3 * M + M)))
    for k0 in cols:
        x = np.zeros((M, K), dtype=np.uint16)
        x[0, k0] = 0x3F80
        if M > 1:
            x[M - 1, (k0 + 1) % K] = 0xBF80  # -1
        y = w12.w12_gemm(_xdev(x), d).cpu().numpy().astype(np.float64)
        np.testing.assert_array_equal(y[0], want[:, k0], err_msg=f"M={M} k={k0}")
        if M > 1:
            np.testing.assert_array_equal(y[M - 1], -want[:, (k0 + 1) % K], err_msg=f"M={M} k={k0 + 1}")


def test_count_max_decode_kernel(w12):
    W, _, _, _, d = _prepared(w12, "heavy_640x1024")
    assert np.array_equal(w12.w12_decode(d).cpu().numpy().view(np.uint16), W)
