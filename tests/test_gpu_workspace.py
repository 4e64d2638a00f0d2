"""The GEMM workspace and CUDA graphs.

w12_gemm keeps its split-K scratch in a workspace cached per (device, stream)
and grows it, outside stream capture, when a call needs more room.  A graph
captured before the growth still holds the old workspace's addresses, so the
old workspace must stay allocated: this test captures a split-K GEMM at 64
rows, grows the workspace with an uncaptured 256-row call on the same stream,
and replays the graph, whose result must still match the oracle.
"""
import numpy as np
import pytest

import oracle as O
import workloads as WL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w12():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__._load_builder().build()
    import lossless_bit_weight_skinny_gb300 as m

    return m


def test_graph_survives_workspace_growth(w12):
    import torch

    N, K = 1024, 5120
    W = WL.projection_weights(N, K, seed=2)
    Wdec = O.decode(O.encode(W))
    plan = w12.w12_gemm_plan(64, N, K)
    assert plan["split_row_blocks"] > 0, plan  # the launch uses the workspace
    st = torch.cuda.Stream()  # a stream of its own: a fresh workspace
    with torch.cuda.stream(st):
        d = w12.w12_upload(w12.w12_encode(W), st)
        x_bits = WL.activations(64, K, seed=11)
        x = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)
        y = torch.empty((64, N), dtype=torch.float32, device="cuda")
        w12.w12_gemm_ex(x, d, y, st)  # first call: allocates the workspace
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            w12.w12_gemm_ex(x, d, y, st)
        # a 256-row call needs more partial sums: the workspace grows
        x2_bits = WL.activations(256, K, seed=12)
        x2 = torch.from_numpy(x2_bits.view(np.int16)).cuda().view(torch.bfloat16)
        y2 = w12.w12_gemm(x2, d, stream=st)
        st.synchronize()
        y.fill_(float("nan"))
        g.replay()
        st.synchronize()
    assert w12.w12_dev_status(d, st) == 0
    bound = 2.0 ** -8 * O.abs_gemm(x_bits, W)
    assert np.all(np.abs(y.cpu().numpy().astype(np.float64) - O.gemm(x_bits, Wdec)) <= bound)
    bound2 = 2.0 ** -8 * O.abs_gemm(x2_bits, W)
    assert np.all(np.abs(y2.cpu().numpy().astype(np.float64) - O.gemm(x2_bits, Wdec)) <= bound2)
