"""w12_gemm_noalloc: the GEMM for callers that may not allocate device memory.

Some callers cannot let a library call cudaMalloc (a host process that has
handed all device memory to its own pool, a plug-in whose framework must own
every allocation, a loop that may not take allocator locks).  For them the
library offers an entry point whose split-K scratch lives in a fixed array in
device memory.  These tests call it through the C ABI, twice in a row on the
same buffers, and check each result against the oracle (decoded matrix,
float64 GEMM) within the 2^-8 bound used by every GEMM test; they also check
that a call whose scratch would not fit is refused, and that a forced timeout
is reported and leaves the array's counters ready for the next call.  The file
is named to run last.
"""
import ctypes

import numpy as np
import pytest

import oracle as O
import workloads as WL

pytestmark = pytest.mark.gpu

BOUND = 2.0 ** -8
SCRATCH_BYTES = 16 << 20      # the fixed array
COUNTER_BYTES = 64 << 10      # its arrival counters
UNSUPPORTED, TIMEOUT = 4, 8


@pytest.fixture(scope="module")
def w12():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__._load_builder().build()
    import lossless_bit_weight_skinny_gb300 as m

    return m


def _noalloc(w12, x, d, y):
    import torch

    P = ctypes.c_void_p
    M, K = x.shape
    return w12.lib().w12_gemm_noalloc(P(x.data_ptr()), d.ptr, P(y.data_ptr()), M, y.shape[1], K,
                                      P(torch.cuda.current_stream().cuda_stream))


CASES = [
    ("kv_1024x5120", lambda: WL.projection_weights(1024, 5120, seed=2), (1, 2, 5, 16, 64, 100)),
    ("heavy_640x1024", lambda: WL.heavy_weights(640, 1024, seed=9), (1, 8, 16, 33, 64, 128, 200)),
    ("ragged_300x800", lambda: WL.projection_weights(300, 800, seed=7, outlier_frac=2e-3), (3, 17)),
]


@pytest.mark.parametrize("name,make,ms", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_oracle(w12, name, make, ms):
    import torch

    W = make()
    N, K = W.shape
    blob = O.encode(W)
    Wdec = O.decode(blob)
    d = w12.w12_upload(w12.w12_encode(W))
    for M in ms:
        x_bits = WL.activations(M, K, seed=500 + M)
        x = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)
        want = O.gemm(x_bits, Wdec)
        bound = BOUND * O.abs_gemm(x_bits, W)
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        for call in range(2):  # the array keeps the previous call's contents
            y.fill_(float("nan"))
            st = _noalloc(w12, x, d, y)
            assert st == 0, w12.STATUS_NAMES.get(st, st)
            assert w12.w12_dev_status(d) == 0
            got = y.cpu().numpy().astype(np.float64)
            assert np.all(np.abs(got - want) <= bound), f"{name} M={M} call {call}"
    # sizes past the supported range are refused, not run
    x = torch.zeros((257, K), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((257, N), dtype=torch.float32, device="cuda")
    assert _noalloc(w12, x, d, y) == UNSUPPORTED


def test_noalloc_refuses_scratch_overflow(w12):
    """A tensor-core call whose grid fills every SM at 128 rows needs more
    partial sums than the array holds, and is refused before any launch."""
    import torch

    N = K = 5120
    plan = w12.w12_gemm_plan(128, N, K)
    assert COUNTER_BYTES + 2 * plan["grid"] * 128 * 128 * 4 > SCRATCH_BYTES, plan
    wt = torch.randn((N, K), device="cuda").to(torch.bfloat16)
    d = w12.w12_encode_device(wt)
    x = torch.zeros((128, K), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((128, N), dtype=torch.float32, device="cuda")
    assert _noalloc(w12, x, d, y) == UNSUPPORTED
    assert w12.w12_dev_status(d) == 0


@pytest.mark.parametrize("M", (1, 16))
def test_noalloc_timeout_then_correct(w12, M):
    """A wait that nothing satisfies (test hook) ends in W12_ERR_TIMEOUT, not a
    hang; the array's counters come back to zero, so the next call is correct."""
    import torch

    W = WL.heavy_weights(640, 1024, seed=9)
    N, K = W.shape
    Wdec = O.decode(O.encode(W))
    d = w12.w12_upload(w12.w12_encode(W))
    x_bits = WL.activations(M, K, seed=90 + M)
    x = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    w12.w12_set_spin_limit(2_000_000)  # 2 ms
    w12.w12_debug_inject_stall(True)
    try:
        assert _noalloc(w12, x, d, y) == 0
        assert w12.w12_dev_status(d) == TIMEOUT
    finally:
        w12.w12_debug_inject_stall(False)
        w12.w12_set_spin_limit(0)
    y.fill_(float("nan"))
    assert _noalloc(w12, x, d, y) == 0
    assert w12.w12_dev_status(d) == 0
    got = y.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - O.gemm(x_bits, Wdec)) <= BOUND * O.abs_gemm(x_bits, W))
