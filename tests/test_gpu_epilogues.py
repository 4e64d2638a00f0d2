"""BF16 output and the gated-MLP epilogue against the oracle (needs a GB300).

w12_gemm_ex(..., out_bf16=True) must write each FP32 result rounded to the
nearest BF16; w12_gemm_ex(..., silu_mul=True) treats rows 2i / 2i+1 as a gate /
up pair and writes silu(gate) * up.  Both are compared with the oracle's
float64 GEMM under the GEMM's bound |y - ref| <= 2^-8 sum_k |x W|, carried
through the epilogue:
  * BF16 rounding adds at most half an ulp, 2^-9 of the magnitude;
  * silu(g) * u - silu(gr) * ur = silu(g)(u - ur) + ur (silu(g) - silu(gr)),
    with |silu'| <= 1.1, plus a few FP32 roundings (2^-20 relative).
Two properties need no oracle: the BF16 output is bit-for-bit PyTorch's
round-to-nearest-even of the FP32 output of the same launch configuration,
and both output paths (direct store and split-K fix-up) are exercised.
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL

pytestmark = pytest.mark.gpu

BOUND = 2.0 ** -8
SILU_SLOPE = 1.1  # max |d silu / dg| = 1.0998...


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


def _interleave(gate, up):
    W = np.empty((2 * gate.shape[0], gate.shape[1]), dtype=np.uint16)
    W[0::2], W[1::2] = gate, up
    return W


def _bf16_to_f64(t):
    import torch

    return t.float().cpu().numpy().astype(np.float64)


CASES = {
    # gate/up pairs of one dense layer, merged by rows
    "pairs_150x800": lambda: _interleave(WL.projection_weights(150, 800, seed=31, outlier_frac=2e-3),
                                         WL.projection_weights(150, 800, seed=32, outlier_frac=2e-3)),
    "pairs_512x5120": lambda: _interleave(WL.projection_weights(512, 5120, seed=33),
                                          WL.projection_weights(512, 5120, seed=34)),
    "heavy_640x1024": lambda: WL.heavy_weights(640, 1024, seed=9),
    "tiny_512x256": lambda: WL.tiny_weights(1)[0],
}
_cache = {}


def _prepared(w12, name):
    if name not in _cache:
        W = CASES[name]()
        blob = O.encode(W)
        _cache[name] = (W, O.decode(blob), O.decode_q8(blob), w12.w12_upload(w12.w12_encode(W)))
    return _cache[name]


def _ref(x, Wref):
    return O.gemm_rows(x, Wref), BOUND * O.abs_gemm(x, Wref)


def _check_bf16(got, ref, tol, what):
    fin = np.isfinite(ref)
    err = np.abs(got - ref)
    lim = (tol + 2.0 ** -9 * (np.abs(ref) + tol)) * (1 + 1e-6)
    bad = fin & ~(err <= lim)
    assert not bad.any(), f"{what}: {bad.sum()} outside the bound"


def _check_silu(got, ref, tol, what, bf16=False):
    gr, ur = ref[:, 0::2], ref[:, 1::2]
    tg, tu = tol[:, 0::2], tol[:, 1::2]
    hr = O.silu_mul(ref)
    s = np.abs(O.silu_mul(np.stack([gr, np.ones_like(gr)], axis=2).reshape(gr.shape[0], -1)))
    lim = (s + SILU_SLOPE * tg) * tu + np.abs(ur) * SILU_SLOPE * tg
    lim = lim + 2.0 ** -20 * (np.abs(hr) + lim)
    if bf16:
        lim = lim + 2.0 ** -9 * (np.abs(hr) + lim)
    lim = lim * (1 + 1e-6) + 1e-30
    fin = np.isfinite(hr)
    err = np.abs(got - hr)
    bad = fin & ~(err <= lim)
    assert not bad.any(), f"{what}: {bad.sum()} outside the bound; worst {(err / lim)[fin].max()}"


@pytest.mark.parametrize("M", (1, 2, 3, 16, 33, 64, 128, 200))
@pytest.mark.parametrize("name", list(CASES.keys()))
def test_bf16_output(w12, name, M):
    import torch

    W, Wdec, _, d = _prepared(w12, name)
    x = WL.activations(M, W.shape[1], seed=300 + M)
    xd = _xdev(x)
    yb = w12.w12_gemm_ex(xd, d, out_bf16=True)
    assert yb.dtype == torch.bfloat16 and tuple(yb.shape) == (M, W.shape[0])
    yf = w12.w12_gemm_ex(xd, d)
    assert w12.w12_dev_status(d) == 0
    # the BF16 epilogue is round-to-nearest-even of the FP32 result
    assert torch.equal(yb.cpu(), yf.cpu().to(torch.bfloat16)), f"{name} M={M}"
    ref, tol = _ref(x, Wdec)
    _check_bf16(_bf16_to_f64(yb), ref, tol, f"{name} M={M}")


@pytest.mark.parametrize("bf16", (False, True))
@pytest.mark.parametrize("M", (1, 2, 3, 16, 33, 64, 96, 256))
@pytest.mark.parametrize("name", list(CASES.keys()))
def test_silu_mul(w12, name, M, bf16):
    import torch

    W, Wdec, _, d = _prepared(w12, name)
    x = WL.activations(M, W.shape[1], seed=400 + M)
    xd = _xdev(x)
    h = w12.w12_gemm_ex(xd, d, silu_mul=True, out_bf16=bf16)
    assert tuple(h.shape) == (M, W.shape[0] // 2)
    assert w12.w12_dev_status(d) == 0
    if bf16:
        hf = w12.w12_gemm_ex(xd, d, silu_mul=True)
        assert torch.equal(h.cpu(), hf.cpu().to(torch.bfloat16))
    ref, tol = _ref(x, Wdec)
    _check_silu(_bf16_to_f64(h), ref, tol, f"{name} M={M}", bf16=bf16)


@pytest.mark.parametrize("M", (1, 16, 64))
def test_q8view_with_epilogues(w12, M):
    W, _, Wq, d = _prepared(w12, "pairs_512x5120")
    x = WL.activations(M, W.shape[1], seed=500 + M)
    h = w12.w12_gemm_ex(_xdev(x), d, q8view=True, silu_mul=True, out_bf16=True)
    assert w12.w12_dev_status(d) == 0
    ref, tol = _ref(x, Wq)
    _check_silu(_bf16_to_f64(h), ref, tol, f"q8 M={M}", bf16=True)


@pytest.fixture(scope="module")
def gate_up_full(w12):
    """The gate and up projections of one layer (17408 x 5120 each) merged by
    rows into one 34816 x 5120 matrix, encoded on the device."""
    import torch

    gate = WL.projection_weights(17408, 5120, seed=41)
    up = WL.projection_weights(17408, 5120, seed=42)
    W = _interleave(gate, up)
    d = w12.w12_encode_device(torch.from_numpy(W.view(np.int16)).cuda())
    assert w12.w12_dev_status(d) == 0
    return W, d


@pytest.mark.parametrize("M", (1, 2, 32, 64, 128))
def test_gate_up_full_size_sampled(w12, gate_up_full, M):
    W, d = gate_up_full
    rng = np.random.Generator(np.random.PCG64(M))
    pairs = np.unique(np.concatenate([rng.choice(17408, 48, replace=False), [0, 1, 63, 64, 17407]]))
    rows = np.stack([2 * pairs, 2 * pairs + 1], axis=1).reshape(-1)
    x = WL.activations(M, 5120, seed=600 + M)
    h = w12.w12_gemm_ex(_xdev(x), d, silu_mul=True, out_bf16=True, input_ready=True)
    assert w12.w12_dev_status(d) == 0
    ref, tol = _ref(x, W[rows])
    _check_silu(_bf16_to_f64(h)[:, pairs], ref, tol, f"gate_up M={M}", bf16=True)


def test_epilogue_errors_and_edges(w12):
    import ctypes

    import torch

    W = WL.projection_weights(7, 64, seed=3)  # odd N: no gate/up pairs
    d = w12.w12_upload(w12.w12_encode(W))
    x = _xdev(WL.activations(2, 64, seed=1))
    with pytest.raises(w12.W12Error):
        w12.w12_gemm_ex(x, d, y=torch.empty((2, 4), device="cuda"), silu_mul=True)
    with pytest.raises(TypeError):
        w12.w12_gemm_ex(x, d, y=torch.empty((2, 7), device="cuda"), out_bf16=True)
    lib = w12.lib()
    P = ctypes.c_void_p
    s = P(torch.cuda.current_stream().cuda_stream)
    y = torch.empty((2, 7), device="cuda")
    assert lib.w12_gemm_ex(P(x.data_ptr()), d.ptr, P(y.data_ptr()), 2, 7, 64, 16, s) == 1  # unknown flag
    assert lib.w12_gemm_ex(P(x.data_ptr()), d.ptr, P(y.data_ptr()), 2, 7, 64, 8, s) == 2  # odd N
    # K = 0: the product is zero, and silu(0) * 0 = 0; only [M][N/2] BF16 is written
    d0 = w12.w12_upload(w12.w12_encode(np.zeros((6, 0), dtype=np.uint16)))
    x0 = torch.zeros((3, 8), dtype=torch.bfloat16, device="cuda")
    h = torch.full((4, 3), 7.0, dtype=torch.bfloat16, device="cuda")
    assert lib.w12_gemm_ex(P(x0.data_ptr()), d0.ptr, P(h.data_ptr()), 3, 6, 0, 4 | 8, s) == 0
    torch.cuda.synchronize()
    assert torch.count_nonzero(h[:3]).item() == 0 and torch.all(h[3] == 7.0)
