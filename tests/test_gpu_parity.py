"""CUDA path against the oracle (needs a GB300; every test is marked gpu).

Decode must be bit-exact.  GEMM outputs must satisfy
|y - y_ref| <= 2^-8 * sum_k |x[m][k] W[n][k]| per element (FP32 accumulation
against the oracle's float64 sum of the decoded weights); the Q pass the same
bound against the oracle's A+E-only decode.  One-hot activations make the
product exact whatever the summation order, which catches a dropped B plane
or a misplaced escape that the 2^-8 bound would miss.
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


def _gemm(w12, d, x_bits, q8=False):
    fn = w12.w12_gemm_q8view if q8 else w12.w12_gemm
    y = fn(_xdev(x_bits), d)
    assert w12.w12_dev_status(d) == 0
    return y.cpu().numpy().astype(np.float64)


def _check(y, x, Wref, rows=None, what=""):
    """y: [M][len(rows)] GPU result for rows `rows` of Wref (decoded, oracle)."""
    Wr = Wref if rows is None else Wref[rows]
    ref = O.gemm_rows(x, Wr)
    scale = O.abs_gemm(x, Wr)
    fin = np.isfinite(ref)
    err = np.abs(y - ref)
    bad = fin & ~(err <= BOUND * scale)
    assert not bad.any(), f"{what}: {bad.sum()} elements outside the bound; worst {err[fin].max()}"
    # non-finite references (Inf/NaN escapes) must propagate the same way
    nf = ~fin
    if nf.any():
        assert np.array_equal(np.isnan(y[nf]), np.isnan(ref[nf])), what
        inf = nf & ~np.isnan(ref)
        assert np.array_equal(y[inf], ref[inf]), what
    return float((err[fin] / np.maximum(scale[fin], 1e-300)).max()) if fin.any() else 0.0


# ---- decode ------------------------------------------------------------------

def _decode_cases():
    rng = np.random.Generator(np.random.PCG64(5))
    return {
        "tiny": WL.tiny_weights(1)[0],
        "ragged_k_not_mult8": WL.projection_weights(300, 777, seed=3, outlier_frac=3e-3),
        "heavy": WL.heavy_weights(257, 1024, seed=4),
        "random_bits": rng.integers(0, 65536, size=(131, 264), dtype=np.uint16),
        "all_patterns": rng.permutation(np.arange(65536, dtype=np.uint32)).astype(np.uint16).reshape(2, 32768),
        "q_proj": WL.projection_weights(5120, 5120, seed=2),
    }


@pytest.mark.parametrize("name", list(_decode_cases().keys()))
def test_decode_bit_exact(w12, name):
    W = _decode_cases()[name]
    blob = O.encode(W)
    h = w12.w12_encode(W)
    assert h.serialize() == blob
    d = w12.w12_upload(h)
    got = w12.w12_decode(d).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, O.decode(blob))
    assert np.array_equal(got, W)


# ---- GEMM parity on small shapes (several tiles and ragged tails) ---------------

def _flooded_rows():
    """Rows whose window a single huge outlier drags up: row 130 (and 300, of
    negative sign) escape almost entirely, row 131 and 40 partly, so single
    tiles hold far more entries than the staged list and one row owns most of
    them."""
    W = WL.projection_weights(384, 2048, seed=27)
    W[130, 7] = 0x7180  # +2^100: every other weight of the row is below the window
    W[300, 2000] = 0xEC80  # -2^90
    W[131, 900] = 0x4300  # +128: weights under 2^-8 escape
    W[40, 5] = 0x4280  # +64
    return W


SHAPES = {
    "tiny_512x256": lambda: WL.tiny_weights(1)[0],
    "flooded_384x2048": _flooded_rows,
    "ragged_300x800": lambda: WL.projection_weights(300, 800, seed=7, outlier_frac=2e-3),
    "heavy_640x1024": lambda: WL.heavy_weights(640, 1024, seed=9),
    "rows_200x4096": lambda: WL.projection_weights(200, 4096, seed=10),
}
MS = (1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 31, 32, 33, 48, 63, 64, 65, 96, 127, 128, 129, 200, 256)
_cache = {}


def _prepared(w12, name):
    if name not in _cache:
        W = SHAPES[name]()
        blob = O.encode(W)
        d = w12.w12_upload(w12.w12_encode(W))
        _cache[name] = (W, O.decode(blob), O.decode_q8(blob), d)
    return _cache[name]


@pytest.mark.parametrize("M", MS)
@pytest.mark.parametrize("name", list(SHAPES.keys()))
def test_gemm_parity(w12, name, M):
    W, Wdec, Wq, d = _prepared(w12, name)
    x = WL.activations(M, W.shape[1], seed=1000 + M)
    _check(_gemm(w12, d, x), x, Wdec, what=f"{name} M={M}")


def test_error_statistics_logged(w12, capsys):
    """The gating bound is 2^-8 sum|x w|; this logs how far inside it the
    results are (largest ratio, and the share of elements above 2^-16)."""
    W, Wdec, Wq, d = _prepared(w12, "rows_200x4096")
    lines = []
    for M in (1, 2, 16, 64, 128, 256):
        x = WL.activations(M, W.shape[1], seed=5000 + M)
        y = _gemm(w12, d, x)
        ref = O.gemm_rows(x, Wdec)
        scale = O.abs_gemm(x, Wdec)
        r = np.abs(y - ref) / np.maximum(scale, 1e-300)
        assert r.max() <= BOUND
        lines.append(f"M={M}: max err/sum|xw| = 2^{np.log2(max(r.max(), 2.0 ** -60)):.1f}, "
                     f"share above 2^-16 = {np.mean(r > 2.0 ** -16):.4f}")
    with capsys.disabled():
        print("\n" + "\n".join(lines))


@pytest.mark.parametrize("M", (1, 2, 4, 8, 16, 32, 64, 128, 256))
@pytest.mark.parametrize("name", list(SHAPES.keys()))
def test_q8view_parity(w12, name, M):
    W, Wdec, Wq, d = _prepared(w12, name)
    x = WL.activations(M, W.shape[1], seed=2000 + M)
    _check(_gemm(w12, d, x, q8=True), x, Wq, what=f"q8 {name} M={M}")


@pytest.mark.parametrize("M", (1, 4, 8, 16, 64, 128, 200))
def test_deterministic(w12, M):
    W, Wdec, Wq, d = _prepared(w12, "heavy_640x1024")
    x = WL.activations(M, W.shape[1], seed=3000 + M)
    y1, y2 = _gemm(w12, d, x), _gemm(w12, d, x)
    assert np.array_equal(y1, y2)


def _one_hot_matrix():
    W = WL.heavy_weights(384, 512, seed=17)
    rng = np.random.Generator(np.random.PCG64(18))
    # zeros, subnormals and below-window values as escapes next to large ones
    W[5, 10:20] = 0
    W[6, 30:40] = 0x8000
    W[7, 40:60] = rng.integers(1, 0x7F, size=20).astype(np.uint16)  # subnormals
    W[8, 0] = 0x7F7F  # huge: everything else in row 8 escapes
    return W


@pytest.mark.parametrize("M", (1, 2, 4, 8, 16, 32, 64, 128, 256))
def test_one_hot_exact(w12, M):
    W = _one_hot_matrix()
    K = W.shape[1]
    d = w12.w12_upload(w12.w12_encode(W))
    want = WL.bf16_bits_to_f32(W).astype(np.float64)
    for k0 in range(0, K, M):
        rows = min(M, K - k0)
        x = np.zeros((M, K), dtype=np.uint16)
        for m in range(rows):
            x[m, k0 + m] = 0x3F80
        y = _gemm(w12, d, x)
        for m in range(rows):
            np.testing.assert_array_equal(y[m], want[:, k0 + m], err_msg=f"M={M} k={k0 + m}")


def test_nonfinite_escapes_propagate(w12):
    W = WL.projection_weights(256, 512, seed=23)
    W[3, 100] = 0x7F80   # +Inf
    W[4, 200] = 0xFF80   # -Inf
    W[5, 300] = 0x7FC1   # NaN
    blob = O.encode(W)
    d = w12.w12_upload(w12.w12_encode(W))
    for M in (1, 16):
        x = WL.activations(M, 512, seed=40 + M)
        _check(_gemm(w12, d, x), x, O.decode(blob), what=f"nonfinite M={M}")


# ---- full-size workloads, sampled rows -----------------------------------------

def _sample_rows(N, n=96, seed=0):
    rng = np.random.Generator(np.random.PCG64(seed))
    pick = rng.choice(N, size=min(n, N), replace=False)
    return np.unique(np.concatenate([pick, [0, N - 1], np.arange(min(N, 130))]))


@pytest.fixture(scope="module")
def full_shapes(w12):
    out = {}
    for i, (N, K) in enumerate(WL.PROJECTION_SHAPES):
        W = WL.projection_weights(N, K, seed=2 + i)
        blob = O.encode(W)
        h = w12.w12_encode(W)
        assert h.serialize() == blob
        out[(N, K)] = (W, blob, w12.w12_upload(h))
    return out


@pytest.mark.parametrize("shape", WL.PROJECTION_SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
def test_projection_shapes_m1(w12, full_shapes, shape):
    W, blob, d = full_shapes[shape]
    N, K = shape
    rows = _sample_rows(N, seed=N + K)
    Wdec = O.decode_rows(blob, 0, N)[rows]
    assert np.array_equal(Wdec, W[rows])
    x = WL.activations(1, K, seed=5)
    y = _gemm(w12, d, x)
    _check(y[:, rows], x, Wdec, what=f"{shape} M=1")
    got = w12.w12_decode(d).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, W)


@pytest.mark.parametrize("M", (1, 2, 4, 8, 16, 32, 64, 128, 256))
@pytest.mark.parametrize("shape", [(17408, 5120), (5120, 17408)], ids=lambda s: f"{s[0]}x{s[1]}")
def test_m_sweep(w12, full_shapes, shape, M):
    W, blob, d = full_shapes[shape]
    N, K = shape
    rows = _sample_rows(N, n=64, seed=M)
    x = WL.activations(M, K, seed=77 + M)
    y = _gemm(w12, d, x)
    _check(y[:, rows], x, W[rows], what=f"{shape} M={M}")


@pytest.mark.parametrize("dist", ["projection", "heavy"])
def test_two_level_verification_pair(w12, dist):
    N, K = 17408, 5120
    W = WL.projection_weights(N, K, seed=55) if dist == "projection" else WL.heavy_weights(N, K, seed=56)
    blob = O.encode(W)
    h = w12.w12_encode(W)
    assert h.serialize() == blob
    d = w12.w12_upload(h)
    rows = _sample_rows(N, n=64, seed=3)
    xq = WL.activations(64, K, seed=90)
    yq = _gemm(w12, d, xq, q8=True)
    Wq = O.decode_q8(blob)
    _check(yq[:, rows], xq, Wq[rows], what=f"{dist} Q pass M=64")
    xe = WL.activations(16, K, seed=91)
    ye = _gemm(w12, d, xe)
    _check(ye[:, rows], xe, W[rows], what=f"{dist} exact pass M=16")


# ---- edges, errors and the failure path -----------------------------------------

def test_edges_and_errors(w12):
    import torch

    W = WL.projection_weights(256, 512, seed=61)
    d = w12.w12_upload(w12.w12_encode(W))
    x = _xdev(WL.activations(4, 512, seed=62))
    lib = w12.lib()
    import ctypes

    y = torch.empty((257, 256), dtype=torch.float32, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = ctypes.c_void_p
    assert lib.w12_gemm(P(x.data_ptr()), d.ptr, P(y.data_ptr()), 0, 256, 512, s) == 0
    assert lib.w12_gemm(P(x.data_ptr()), d.ptr, P(y.data_ptr()), 4, 255, 512, s) == 2
    assert lib.w12_gemm(P(x.data_ptr()), d.ptr, P(y.data_ptr()), 257, 256, 512, s) == 4
    assert lib.w12_gemm(P(x.data_ptr() + 2), d.ptr, P(y.data_ptr()), 4, 256, 512, s) == 3
    assert lib.w12_gemm(None, d.ptr, P(y.data_ptr()), 4, 256, 512, s) == 1
    # K not a multiple of 32: the GEMM refuses, decode still works
    W2 = WL.projection_weights(64, 200, seed=63)
    d2 = w12.w12_upload(w12.w12_encode(W2))
    x2 = _xdev(WL.activations(1, 200, seed=64))
    assert lib.w12_gemm(P(x2.data_ptr()), d2.ptr, P(y.data_ptr()), 1, 64, 200, s) == 4
    assert np.array_equal(w12.w12_decode(d2).cpu().numpy().view(np.uint16), W2)
    # K = 0: y = 0
    d3 = w12.w12_upload(w12.w12_encode(np.zeros((16, 0), dtype=np.uint16)))
    y3 = torch.full((2, 16), 7.0, device="cuda")
    x3 = torch.zeros((2, 8), dtype=torch.bfloat16, device="cuda")
    assert lib.w12_gemm(P(x3.data_ptr()), d3.ptr, P(y3.data_ptr()), 2, 16, 0, s) == 0
    assert torch.all(y3 == 0)
    # N = 0: nothing to do
    d4 = w12.w12_upload(w12.w12_encode(np.zeros((0, 64), dtype=np.uint16)))
    assert lib.w12_gemm(P(x.data_ptr()), d4.ptr, P(y.data_ptr()), 4, 0, 64, s) == 0


def test_gemm_host_entry(w12):
    import torch

    W, Wdec, Wq, d = _prepared(w12, "ragged_300x800")
    for M in (1, 16):
        x = WL.activations(M, 800, seed=70 + M)
        xh = torch.from_numpy(x.view(np.int16)).pin_memory()
        xd = torch.empty((M, 800), dtype=torch.int16, device="cuda")
        yd = torch.empty((M, 300), dtype=torch.float32, device="cuda")
        yh = torch.empty((M, 300), dtype=torch.float32).pin_memory()
        w12.w12_gemm_host(xh, xd, d, yd, yh)
        torch.cuda.synchronize()
        _check(yh.numpy().astype(np.float64), x, Wdec, what=f"host entry M={M}")


@pytest.mark.parametrize("M", (1, 16, 128))
def test_timeout_reports_and_recovers(w12, M):
    """A wait that nothing satisfies ends in W12_ERR_TIMEOUT, not a hang, and
    the next call on the same handle and workspace is correct again."""
    W, Wdec, Wq, d = _prepared(w12, "heavy_640x1024")
    x = WL.activations(M, 1024, seed=80 + M)
    w12.w12_set_spin_limit(2_000_000)  # 2 ms
    w12.w12_debug_inject_stall(True)
    try:
        w12.w12_gemm(_xdev(x), d)
        assert w12.w12_dev_status(d) == 8
    finally:
        w12.w12_debug_inject_stall(False)
        w12.w12_set_spin_limit(0)
    _check(_gemm(w12, d, x), x, Wdec, what="after timeout")


def test_input_ready_chain(w12):
    """Launches flagged input-ready read x at once and overlap the previous
    kernel's tail, but write only after it has completed: a chain of them
    (both kernels, split-K shapes, one y reused by consecutive launches) gives
    bitwise the results of plain w12_gemm."""
    import torch

    cases = []
    for name in ("rows_200x4096", "ragged_300x800", "heavy_640x1024", "flooded_384x2048"):
        W, Wdec, Wq, d = _prepared(w12, name)
        for M in (1, 2, 16, 64):
            x = _xdev(WL.activations(M, W.shape[1], seed=4000 + M))
            cases.append((d, x, w12.w12_gemm(x, d)))
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ys = [torch.full_like(ref, float("nan")) for _, _, ref in cases]
    shared = {}
    for i, (d, x, ref) in enumerate(cases):
        w12.w12_gemm_ex(x, d, ys[i], stream, input_ready=(i > 0))
        # the same output buffer written by two consecutive launches
        key = tuple(ref.shape)
        if key in shared:
            w12.w12_gemm_ex(x, d, shared[key], stream, input_ready=True)
        else:
            shared[key] = torch.full_like(ref, float("nan"))
            w12.w12_gemm_ex(x, d, shared[key], stream, input_ready=True)
        shared[key + ("last",)] = ref
    torch.cuda.synchronize()
    for i, (d, x, ref) in enumerate(cases):
        assert w12.w12_dev_status(d) == 0
        assert torch.equal(ys[i], ref), f"case {i}"
    for key, buf in shared.items():
        if key[-1] != "last":
            assert torch.equal(buf, shared[key + ("last",)]), f"shared {key}"
    # unknown flag bits are refused
    d, x, ref = cases[0]
    P = __import__("ctypes").c_void_p
    assert w12.lib().w12_gemm_ex(P(x.data_ptr()), d.ptr, P(ys[0].data_ptr()), x.shape[0], d.N, x.shape[1],
                                 16, P(stream.cuda_stream)) == 1
