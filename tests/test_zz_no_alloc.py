"""w12_gemm_noalloc: the GEMM for callers that may not allocate device memory.

Some callers cannot let a library call cudaMalloc (a host process that has
handed all device memory to its own pool, a plug-in whose framework must own
every allocation, a loop that may not take allocator locks).  For them the
library offers an entry point whose split-K scratch lives in a fixed array in
device memory.  This test calls it through the C ABI, twice in a row on the
same buffers, and checks each result against w12_gemm's within the 2^-8
bound used by every GEMM test.  The file is named to run last.
"""
import ctypes

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


CASES = [
    ("kv_1024x5120", lambda: WL.projection_weights(1024, 5120, seed=2), (1, 2, 5, 16, 64, 100)),
    ("heavy_640x1024", lambda: WL.heavy_weights(640, 1024, seed=9), (1, 8, 16, 33, 64, 128, 200)),
    ("ragged_300x800", lambda: WL.projection_weights(300, 800, seed=7, outlier_frac=2e-3), (3, 17)),
]


@pytest.mark.parametrize("name,make,ms", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_gemm(w12, name, make, ms):
    import torch

    W = make()
    N, K = W.shape
    d = w12.w12_upload(w12.w12_encode(W))
    lib = w12.lib()
    P = ctypes.c_void_p
    stream = torch.cuda.current_stream()
    for M in ms:
        x_bits = WL.activations(M, K, seed=500 + M)
        x = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)
        y_ref = w12.w12_gemm(x, d)
        bound = BOUND * O.abs_gemm(x_bits, W)
        want = y_ref.cpu().numpy().astype(np.float64)
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        for call in range(2):
            y.fill_(float("nan"))
            st = lib.w12_gemm_noalloc(P(x.data_ptr()), d.ptr, P(y.data_ptr()), M, N, K,
                                      P(stream.cuda_stream))
            assert st == 0, w12.STATUS_NAMES.get(st, st)
            assert w12.w12_dev_status(d) == 0
            got = y.cpu().numpy().astype(np.float64)
            assert np.all(np.abs(got - want) <= bound), f"{name} M={M} call {call}"
    # sizes past the supported range are refused, not run
    x = torch.zeros((257, K), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((257, N), dtype=torch.float32, device="cuda")
    assert lib.w12_gemm_noalloc(P(x.data_ptr()), d.ptr, P(y.data_ptr()), 257, N, K,
                                P(stream.cuda_stream)) == 4
