"""Encoding on the device (needs a GB300; every test is marked gpu).

w12_encode_device must produce, from BF16 weights already in device memory,
exactly the arrays the oracle's encoder produces: the test downloads the
handle, serialises it and compares the blob byte for byte with the oracle's.
A GEMM through the device-encoded handle must equal, bit for bit, the GEMM
through the uploaded host encoding (same arrays, same row-group index).
"""
import ctypes

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


def _flooded():
    W = WL.projection_weights(384, 2048, seed=27)
    W[130, 7] = 0x7180
    W[300, 2000] = 0xEC80
    W[131, 900] = 0x4300
    return W


def _cases():
    rng = np.random.Generator(np.random.PCG64(6))
    return {
        "tiny": lambda: WL.tiny_weights(1)[0],
        "ragged_k_not_mult8": lambda: WL.projection_weights(300, 777, seed=3, outlier_frac=3e-3),
        "heavy": lambda: WL.heavy_weights(257, 1024, seed=4),
        "random_bits": lambda: rng.integers(0, 65536, size=(131, 264), dtype=np.uint16),
        "all_patterns": lambda: np.random.Generator(np.random.PCG64(7)).permutation(
            np.arange(65536, dtype=np.uint32)).astype(np.uint16).reshape(2, 32768),
        "kv_proj": lambda: WL.projection_weights(1024, 5120, seed=2),
        "flooded_rows": _flooded,
        "one_row": lambda: WL.projection_weights(1, 300, seed=8),
    }


def _dev_tensor(W):
    import torch

    return torch.from_numpy(np.ascontiguousarray(W).view(np.int16)).cuda()


@pytest.mark.parametrize("name", list(_cases().keys()))
def test_device_encode_blob_equals_oracle(w12, name):
    W = _cases()[name]()
    d = w12.w12_encode_device(_dev_tensor(W))
    blob = w12.w12_download(d).serialize()
    assert blob == O.encode(W), name
    assert w12.w12_dev_status(d) == 0


@pytest.mark.parametrize("shape", [(0, 16), (16, 0), (0, 0)])
def test_device_encode_empty(w12, shape):
    import torch

    W = np.zeros(shape, dtype=np.uint16)
    d = w12.w12_encode_device(torch.zeros(shape, dtype=torch.int16, device="cuda"))
    assert w12.w12_download(d).serialize() == O.encode(W)


@pytest.mark.parametrize("M", (1, 2, 16, 64))
@pytest.mark.parametrize("name", ["kv_proj", "flooded_rows", "heavy"])
def test_device_encoded_gemm_equals_uploaded(w12, name, M):
    import torch

    W = _cases()[name]()
    if W.shape[1] % 32:
        pytest.skip("GEMMs need K % 32 == 0")
    d_dev = w12.w12_encode_device(_dev_tensor(W))
    d_up = w12.w12_upload(w12.w12_encode(W))
    x = torch.from_numpy(WL.activations(M, W.shape[1], seed=60 + M).view(np.int16)).cuda().view(torch.bfloat16)
    assert torch.equal(w12.w12_gemm(x, d_dev), w12.w12_gemm(x, d_up))
    assert w12.w12_dev_status(d_dev) == 0


def test_device_encode_errors(w12):
    lib = w12.lib()
    out = ctypes.c_void_p()
    P = ctypes.c_void_p
    assert lib.w12_encode_device(P(0), -1, 4, P(0), ctypes.byref(out)) == 1
    assert lib.w12_encode_device(P(0), 4, 4, P(0), ctypes.byref(out)) == 1  # no weights
    assert lib.w12_download(P(0), P(0), ctypes.byref(out)) == 1
    with pytest.raises(TypeError):
        w12.w12_encode_device(np.zeros((4, 4), dtype=np.uint16))
