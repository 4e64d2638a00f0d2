"""w12_gemm_grouped: several matrices that read the same x, in one launch.

The q, k and v projections of a layer (or its gate and up projections) read
the same activations; one launch runs all of them with their row blocks laid
end to end.  Each output is compared with the oracle (decoded matrix, float64
GEMM) under the bound every GEMM test uses, |y - ref| <= 2^-8 sum_k |x W|;
for the Q pass against the oracle's 8-bit view, and for BF16 output with the
extra half ulp of the final rounding.  The groups mix ragged row counts (a
matrix ending inside a row block, so the next one's first block starts a new
tile), heavy escape tails, and a matrix with no rows, across the CUDA-core
sizes (M <= 2) and every tensor-core tile height.
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL

pytestmark = pytest.mark.gpu

BOUND = 2.0 ** -8
INVALID_ARG, SHAPE = 1, 2


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


GROUPS = {
    # q / k / v of a small attention block, rows not multiples of 128
    "qkv_ragged_800": lambda: [WL.projection_weights(300, 800, seed=41, outlier_frac=2e-3),
                               WL.projection_weights(70, 800, seed=42),
                               WL.projection_weights(129, 800, seed=43)],
    # a heavy-tailed matrix next to a plain one, and an empty one in between
    "heavy_mix_1024": lambda: [WL.heavy_weights(640, 1024, seed=9),
                               np.zeros((0, 1024), dtype=np.uint16),
                               WL.projection_weights(256, 1024, seed=44),
                               WL.projection_weights(64, 1024, seed=45)],
    # q / k / v shapes of a 5120-wide layer with 8 KV heads of 128
    "qkv_5120": lambda: [WL.projection_weights(5120, 5120, seed=46),
                         WL.projection_weights(1024, 5120, seed=47),
                         WL.projection_weights(1024, 5120, seed=48)],
}
MS = {"qkv_ragged_800": (1, 2, 3, 16, 17, 33, 64, 100, 200, 256),
      "heavy_mix_1024": (1, 2, 16, 64, 128),
      "qkv_5120": (1, 2, 16, 32, 64)}
_cache = {}


def _prepared(w12, name):
    if name not in _cache:
        Ws = GROUPS[name]()
        blobs = [O.encode(W) for W in Ws]
        _cache[name] = (Ws, [O.decode(b) for b in blobs], [O.decode_q8(b) for b in blobs],
                        [w12.w12_upload(w12.w12_encode(W)) for W in Ws])
    return _cache[name]


@pytest.mark.parametrize("name", sorted(GROUPS))
def test_grouped_matches_oracle(w12, name):
    Ws, Wdec, _, devs = _prepared(w12, name)
    K = Ws[0].shape[1]
    for M in MS[name]:
        x = WL.activations(M, K, seed=700 + M)
        ys = w12.w12_gemm_grouped(_xdev(x), devs)
        for i, (W, Wd, y) in enumerate(zip(Ws, Wdec, ys)):
            assert y.shape == (M, W.shape[0])
            if W.shape[0] == 0:
                continue
            got = y.cpu().numpy().astype(np.float64)
            bad = np.abs(got - O.gemm(x, Wd)) > BOUND * O.abs_gemm(x, W)
            assert not bad.any(), f"{name} M={M} matrix {i}: {int(bad.sum())} outside the bound"
        for d in devs:
            assert w12.w12_dev_status(d) == 0


@pytest.mark.parametrize("M", (1, 16, 64))
def test_grouped_q8view_and_bf16(w12, M):
    """The Q pass over every matrix of the group, and BF16 output (the FP32
    result rounded to nearest: half an ulp, 2^-9 of |y|, on top of the bound)."""
    import torch

    Ws, Wdec, Wq8, devs = _prepared(w12, "qkv_ragged_800")
    K = Ws[0].shape[1]
    x = WL.activations(M, K, seed=800 + M)
    xd = _xdev(x)
    for W, Wq, y in zip(Ws, Wq8, w12.w12_gemm_grouped(xd, devs, q8view=True)):
        got = y.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - O.gemm(x, Wq)) <= BOUND * O.abs_gemm(x, Wq)), f"Q pass M={M}"
    for W, Wd, y in zip(Ws, Wdec, w12.w12_gemm_grouped(xd, devs, out_bf16=True)):
        assert y.dtype == torch.bfloat16
        ref = O.gemm(x, Wd)
        got = y.float().cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref) <= BOUND * O.abs_gemm(x, W) * (1 + 2.0 ** -8) + 2.0 ** -9 * np.abs(ref)), \
            f"BF16 M={M}"


def test_grouped_input_ready_and_caller_outputs(w12):
    """input_ready and caller-owned outputs; a second call overwrites them."""
    import torch

    Ws, Wdec, _, devs = _prepared(w12, "heavy_mix_1024")
    K = Ws[0].shape[1]
    for M in (2, 33):
        x = WL.activations(M, K, seed=900 + M)
        ys = [torch.full((M, W.shape[0]), float("nan"), device="cuda") for W in Ws]
        for _ in range(2):
            w12.w12_gemm_grouped(_xdev(x), devs, ys=ys, input_ready=True)
            for W, Wd, y in zip(Ws, Wdec, ys):
                if W.shape[0]:
                    got = y.cpu().numpy().astype(np.float64)
                    assert np.all(np.abs(got - O.gemm(x, Wd)) <= BOUND * O.abs_gemm(x, W)), f"M={M}"


def test_grouped_refusals(w12):
    """Arguments the entry point refuses before any launch."""
    import ctypes

    import torch

    _, _, _, devs = _prepared(w12, "qkv_ragged_800")
    _, _, _, other = _prepared(w12, "heavy_mix_1024")
    lib = w12.lib()
    P = ctypes.c_void_p
    x = torch.zeros((4, 800), dtype=torch.bfloat16, device="cuda")
    ys = [torch.empty((4, d.N), device="cuda") for d in devs]

    def call(ds, n, flags=0, K=800):
        k = max(len(ds), 1)
        hs = (P * k)(*[d.ptr for d in ds])
        ps = (P * k)(*[ys[i % len(ys)].data_ptr() for i in range(len(ds))])
        return lib.w12_gemm_grouped(P(x.data_ptr()), hs, ps, n, 4, K, flags, P(0))

    assert call(devs, 0) == INVALID_ARG
    assert call(devs + devs[:2], 5) == INVALID_ARG  # more than four matrices
    assert call([devs[0], other[0]], 2) == SHAPE  # K differs
    assert call(devs, 3, flags=w12.W12_GEMM_SILU_MUL) == INVALID_ARG
    assert call(devs, 3, flags=1 << 20) == INVALID_ARG
    assert call(devs, 3) == 0


@pytest.mark.parametrize("M", (1, 16))
def test_grouped_timeout_then_correct(w12, M):
    """A wait that nothing satisfies (test hook) ends the grouped launch with
    W12_ERR_TIMEOUT in every handle of the group, not a hang; after the abort
    the kernels run on whatever their rings hold, and every read of an escape
    list stays inside its own matrix's list.  The next call is correct."""
    TIMEOUT = 8
    Ws, Wdec, _, devs = _prepared(w12, "heavy_mix_1024")
    K = Ws[0].shape[1]
    x = WL.activations(M, K, seed=950 + M)
    xd = _xdev(x)
    w12.w12_set_spin_limit(2_000_000)  # 2 ms
    w12.w12_debug_inject_stall(True)
    try:
        w12.w12_gemm_grouped(xd, devs)
        for W, d in zip(Ws, devs):
            assert w12.w12_dev_status(d) == (TIMEOUT if W.shape[0] else 0)
    finally:
        w12.w12_debug_inject_stall(False)
        w12.w12_set_spin_limit(0)
    ys = w12.w12_gemm_grouped(xd, devs)
    for W, Wd, y, d in zip(Ws, Wdec, ys, devs):
        assert w12.w12_dev_status(d) == 0
        if W.shape[0]:
            got = y.cpu().numpy().astype(np.float64)
            assert np.all(np.abs(got - O.gemm(x, Wd)) <= BOUND * O.abs_gemm(x, W)), f"M={M}"


@pytest.mark.parametrize("M", (1, 16))
def test_grouped_host_buffers(w12, M):
    """w12_gemm_grouped_host: x from pinned host memory, every output back in
    pinned host memory, one stream; results against the oracle."""
    import torch

    Ws, Wdec, _, devs = _prepared(w12, "qkv_ragged_800")
    K = Ws[0].shape[1]
    x = WL.activations(M, K, seed=990 + M)
    xh = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).pin_memory()
    xd = torch.empty((M, K), dtype=torch.int16, device="cuda")
    yd = [torch.empty((M, W.shape[0]), dtype=torch.float32, device="cuda") for W in Ws]
    yh = [torch.full((M, W.shape[0]), float("nan"), dtype=torch.float32).pin_memory() for W in Ws]
    st = torch.cuda.current_stream()
    w12.w12_gemm_grouped_host(xh, xd, devs, yd, yh, stream=st)
    st.synchronize()
    for W, Wd, y in zip(Ws, Wdec, yh):
        got = y.numpy().astype(np.float64)
        assert np.all(np.abs(got - O.gemm(x, Wd)) <= BOUND * O.abs_gemm(x, W)), f"M={M}"


@pytest.mark.parametrize("M", (1, 2, 16, 32, 64))
def test_grouped_gate_up_full_size(w12, M):
    """The gate/up group of the benchmark layer at full size (two 17408x5120
    matrices, one x, the launch the benchmark times), on sampled rows of each
    matrix against the oracle (rows decode independently, so a sample's own
    encoding decodes to the same rows)."""
    K = 5120
    Ws = [WL.projection_weights(17408, K, seed=s) for s in (61, 62)]
    devs = [w12.w12_upload(w12.w12_encode(W)) for W in Ws]
    x = WL.activations(M, K, seed=960 + M)
    ys = w12.w12_gemm_grouped(_xdev(x), devs)
    rng = np.random.Generator(np.random.PCG64(M))
    for i, (W, y) in enumerate(zip(Ws, ys)):
        rows = np.unique(np.concatenate([rng.choice(17408, size=96, replace=False), [0, 127, 128, 17407]]))
        Wr = O.decode(O.encode(W[rows]))
        assert np.array_equal(Wr, W[rows])
        got = y.cpu().numpy().astype(np.float64)[:, rows]
        assert np.all(np.abs(got - O.gemm(x, Wr)) <= BOUND * O.abs_gemm(x, Wr)), f"gate/up matrix {i} M={M}"
    for d in devs:
        assert w12.w12_dev_status(d) == 0


def test_grouped_host_packed_outputs(w12):
    """Outputs laid end to end on the device and on the host go back in one
    transfer; the results are the same as with separate buffers.  (Every
    output must start on a 16-byte boundary: M = 4 keeps the ragged row
    counts' offsets aligned.)"""
    import torch

    Ws, Wdec, _, devs = _prepared(w12, "qkv_ragged_800")
    M, K = 4, Ws[0].shape[1]
    x = WL.activations(M, K, seed=997)
    xh = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).pin_memory()
    xd = torch.empty((M, K), dtype=torch.int16, device="cuda")
    n = sum(M * W.shape[0] for W in Ws)
    yd_all = torch.empty(n, dtype=torch.float32, device="cuda")
    yh_all = torch.full((n,), float("nan"), dtype=torch.float32).pin_memory()
    yd, yh, off = [], [], 0
    for W in Ws:
        yd.append(yd_all[off:off + M * W.shape[0]].view(M, -1))
        yh.append(yh_all[off:off + M * W.shape[0]].view(M, -1))
        off += M * W.shape[0]
    st = torch.cuda.current_stream()
    w12.w12_gemm_grouped_host(xh, xd, devs, yd, yh, stream=st)
    st.synchronize()
    for W, Wd, y in zip(Ws, Wdec, yh):
        got = y.numpy().astype(np.float64)
        assert np.all(np.abs(got - O.gemm(x, Wd)) <= BOUND * O.abs_gemm(x, W))
