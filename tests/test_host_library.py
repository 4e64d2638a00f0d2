"""The library's host side against the oracle (CPU only, no GPU needed).

The library encoder is separate code from the oracle's; its blob must be byte
for byte the oracle's on every input.  Also: the C ABI exports every symbol
include/w12.h declares, the validator rejects corrupted handles, and the file
format round-trips.
"""
import os
import re
import subprocess
import sys

import numpy as np
import pytest

import oracle as O
import workloads as WL

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def w12():
    import __graft_entry__

    __graft_entry__._load_builder().build()
    import lossless_bit_weight_skinny_gb300 as m

    return m


def _cases():
    rng = np.random.Generator(np.random.PCG64(5))
    allpat = rng.permutation(np.arange(65536, dtype=np.uint32)).astype(np.uint16).reshape(2, 32768)
    return {
        "tiny": WL.tiny_weights(1)[0],
        "ragged": WL.projection_weights(300, 777, seed=3, outlier_frac=3e-3),
        "heavy": WL.heavy_weights(257, 1000, seed=4),
        "random_bits": rng.integers(0, 65536, size=(131, 263), dtype=np.uint16),
        "all_patterns": allpat,
        "empty_rows": np.zeros((0, 64), dtype=np.uint16),
        "empty_cols": np.zeros((7, 0), dtype=np.uint16),
        "single": np.array([[0x3F80]], dtype=np.uint16),
        "zeros": np.zeros((130, 300), dtype=np.uint16),
        "k5120": WL.projection_weights(1024, 5120, seed=2),
    }


@pytest.mark.parametrize("name", list(_cases().keys()))
def test_encoder_matches_oracle_bytes(w12, name):
    W = _cases()[name]
    blob = O.encode(W)
    for threads in (1, 0):
        h = w12.w12_encode(W, n_threads=threads)
        assert h.validate() == 0
        assert h.serialize() == blob
    st = h.stats()
    N, K, n_esc, T = O.blob_header(blob)
    assert (st["N"], st["K"], st["n_escapes"], st["n_tiles"]) == (N, K, n_esc, T)
    assert st["bytes_total"] == len(blob)


@pytest.mark.parametrize("name", ["tiny", "ragged", "heavy", "random_bits", "all_patterns", "empty_rows",
                                  "empty_cols", "single", "zeros"])
def test_count_max_encoder_matches_oracle_bytes(w12, name):
    """Count-maximising windows: the library's blob is the oracle's, it
    validates and decodes losslessly, and never has more escapes than the
    max-anchored encoding of the same matrix."""
    W = _cases()[name]
    blob = O.encode(W, count_max=True)
    for threads in (1, 0):
        h = w12.w12_encode(W, n_threads=threads, count_max=True)
        assert h.validate() == 0
        assert h.serialize() == blob
    assert np.array_equal(O.decode(blob), W)
    assert O.blob_header(blob)[2] <= O.blob_header(O.encode(W))[2]
    h2 = w12.w12_deserialize(blob)
    assert h2.validate() == 0


def test_encoder_full_projection_shape(w12):
    W = WL.projection_weights(5120, 5120, seed=2)
    h = w12.w12_encode(W)
    assert h.serialize() == O.encode(W)
    st = h.stats()
    assert 12.0 < st["bits_per_weight"] < 12.05


def test_deserialize_roundtrip_and_view(w12):
    W = WL.projection_weights(200, 512, seed=8, outlier_frac=2e-3)
    blob = O.encode(W)
    h = w12.w12_deserialize(blob)
    assert h.serialize() == blob
    ebase, ae, b, tptr, esc = h.view()
    assert ae.shape == (200, 512) and b.shape == (200, 256)
    assert tptr[-1] == esc.size


def test_save_load(w12, tmp_path):
    W = WL.heavy_weights(64, 96, seed=12)
    h = w12.w12_encode(W)
    p = str(tmp_path / "m.w12")
    h.save(p)
    h2 = w12.w12_load(p)
    assert h2.serialize() == h.serialize()
    raw = bytearray(open(p, "rb").read())
    raw[100] ^= 0x40
    open(p, "wb").write(bytes(raw))
    with pytest.raises(w12.W12Error) as e:
        w12.w12_load(p)
    assert e.value.status == 7  # CORRUPT (checksum)


def _corrupt(blob: bytes, N: int, K: int, what: str) -> bytes:
    b = bytearray(blob)
    n_esc = int.from_bytes(b[24:32], "little")
    T = int.from_bytes(b[32:40], "little")
    brow = 4 * ((K + 7) // 8)
    off_eb = 40
    off_ae = off_eb + N
    off_b = off_ae + N * K
    off_ptr = off_b + N * brow
    off_esc = off_ptr + 4 * (T + 1)
    if what == "ebase_zero":
        b[off_eb] = 0
    elif what == "ebase_high":
        b[off_eb + 1] = 240
    elif what == "unsorted":
        e0 = b[off_esc:off_esc + 4]
        b[off_esc:off_esc + 4] = b[off_esc + 4:off_esc + 8]
        b[off_esc + 4:off_esc + 8] = e0
    elif what == "ptr":
        v = int.from_bytes(b[off_ptr + 4:off_ptr + 8], "little") + 1
        b[off_ptr + 4:off_ptr + 8] = v.to_bytes(4, "little")
    elif what == "placeholder":
        e = int.from_bytes(b[off_esc:off_esc + 4], "little")
        n, k = e >> 24, (e >> 16) & 0xFF
        b[off_ae + n * K + k] ^= 0x01
    elif what == "in_window_escape":
        # rewrite the first escape's bits to a value inside its row's window
        e = int.from_bytes(b[off_esc:off_esc + 4], "little")
        n = e >> 24
        eb = b[off_eb + n]
        e = (e & 0xFFFF0000) | ((eb + 3) << 7)
        b[off_esc:off_esc + 4] = e.to_bytes(4, "little")
    elif what == "saturated_placeholder":
        # an escape above its row's window must carry A = s<<3|7, E = 15
        for i in range(n_esc):
            e = int.from_bytes(b[off_esc + 4 * i:off_esc + 4 * i + 4], "little")
            n_in_tile = e >> 24
            ex = (e >> 7) & 0xFF
            if 1 <= ex <= 254 and ex > b[off_eb + n_in_tile] + 15:
                b[off_ae + n_in_tile * K + ((e >> 16) & 0xFF)] &= 0xF0
                break
        else:
            raise AssertionError("no escape above a window")
    elif what == "truncated":
        return bytes(b[:-4])
    return bytes(b)


@pytest.mark.parametrize("what", ["ebase_zero", "ebase_high", "unsorted", "ptr", "placeholder",
                                  "in_window_escape", "truncated", "saturated_placeholder"])
def test_validator_rejects_corruption(w12, what):
    W = WL.projection_weights(64, 256, seed=21, outlier_frac=5e-3)
    W[0, :3] = 0  # a few escapes in row 0
    W[1, 5] = 0x7F00  # a huge weight that a count-maximising window leaves above it
    blob = O.encode(W, count_max=(what == "saturated_placeholder"))
    bad = _corrupt(blob, 64, 256, what)
    with pytest.raises(w12.W12Error) as e:
        w12.w12_deserialize(bad)
    assert e.value.status == 7


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "w12.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(w12_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(w12):
    declared = _declared_functions()
    assert len(declared) >= 18
    out = subprocess.run(["nm", "-D", "--defined-only", w12.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(w12_\w+)", out))
    missing = [n for n in declared if n not in exported]
    assert not missing, missing
    for n in declared:
        assert hasattr(w12.lib(), n)
    assert set(w12.EXPORTED) == set(declared)


def test_invalid_arguments(w12):
    import ctypes

    lib = w12.lib()
    out = ctypes.c_void_p()
    assert lib.w12_encode(None, 4, 4, 0, ctypes.byref(out)) == 1
    assert lib.w12_encode(None, -1, 4, 0, ctypes.byref(out)) == 1
    assert lib.w12_validate(None) == 1
    assert lib.w12_encode_ex(None, 0, 0, 0, 2, ctypes.byref(out)) == 1  # unknown flag
    assert lib.w12_status_string(8) == b"device wait timed out"


def test_no_oracle_on_product_path():
    """The package and its C++/CUDA sources never reference the oracle."""
    pkg = os.path.join(ROOT, "lossless_bit_weight_skinny_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f


def test_c_client_compiles_and_runs(w12, tmp_path):
    """include/w12.h is plain C99, and a C program linked against the library
    drives the host-side calls without Python or a GPU."""
    src = os.path.join(ROOT, "tests", "c_abi", "host_roundtrip.c")
    exe = str(tmp_path / "host_roundtrip")
    libdir = os.path.dirname(w12.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), src, "-o", exe,
                    "-L", libdir, "-lw12", "-Wl,-rpath," + libdir], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok")
    esc = [int(line.split()[3]) for line in r.stdout.splitlines() if line.startswith("window rule")]
    assert len(esc) == 2 and esc[1] <= esc[0]


def test_package_fails_loudly_without_the_library(tmp_path):
    """A copy of the package without its built library refuses to import:
    there is no fallback path."""
    import shutil

    pkg = tmp_path / "lossless_bit_weight_skinny_gb300"
    pkg.mkdir()
    shutil.copy(os.path.join(ROOT, "lossless_bit_weight_skinny_gb300", "__init__.py"), pkg / "__init__.py")
    r = subprocess.run([sys.executable, "-c", "import lossless_bit_weight_skinny_gb300"], cwd=str(tmp_path),
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "not built" in r.stderr


@pytest.mark.parametrize("M,N,K,kernel,tile,grid,split", [
    (1, 17408, 5120, 1, 1, 136, 0),    # aligned: one whole row block per CTA
    (1, 1024, 5120, 1, 1, 80, 8),      # aligned: 10 CTAs share each of 8 row blocks
    (1, 5120, 5120, 1, 1, 136, 40),    # stream-K over 152 - 16 SMs (both kernels)
    (1, 5120, 17408, 1, 1, 136, 40),
    (2, 5120, 5120, 1, 2, 136, 40),
    (3, 5120, 5120, 2, 16, 136, 40),   # tensor cores from 3 rows
    (16, 17408, 5120, 2, 16, 136, 0),
    (64, 17408, 5120, 2, 64, 136, 0),
    (65, 1024, 5120, 2, 128, 80, 8),
    (256, 17408, 5120, 2, 256, 136, 0),
])
def test_gemm_plan_projection_shapes(w12, M, N, K, kernel, tile, grid, split):
    """The launch planning w12_gemm uses, for the projection shapes on a
    152-SM GB300 (kernel by M, tile rows, grid, split row blocks)."""
    p = w12.w12_gemm_plan(M, N, K, 152)
    assert (p["kernel"], p["tile_rows"], p["grid"], p["split_row_blocks"]) == (kernel, tile, grid, split)
    assert p["separate_fixup"] == (1 if (M > 64 and split) else 0)


def test_gemm_plan_invariants(w12):
    rng = np.random.Generator(np.random.PCG64(77))
    for _ in range(300):
        M = int(rng.integers(1, 257))
        N = int(rng.integers(1, 40000))
        K = 32 * int(rng.integers(1, 700))
        sms = int(rng.choice([8, 76, 132, 152]))
        p = w12.w12_gemm_plan(M, N, K, sms)
        units = p["row_blocks"] * p["k_steps"]
        assert p["kernel"] == (1 if M <= 2 else 2)
        assert p["tile_rows"] >= M and (p["tile_rows"] == M or p["tile_rows"] // 2 < M or p["tile_rows"] == 16)
        assert p["row_blocks"] == -(-N // p["block_rows"]) and p["k_steps"] == -(-K // 256)
        assert 1 <= p["grid"] <= min(units, sms - min(16, sms // 8))
        assert 0 <= p["split_row_blocks"] <= p["row_blocks"]
        if p["split_row_blocks"]:
            assert p["partial_bytes"] == 4 * 2 * p["grid"] * M * p["block_rows"]
        else:
            assert p["partial_bytes"] == 0
    assert w12.w12_gemm_plan(0, 5, 5, 152)["kernel"] == 0
    with pytest.raises(w12.W12Error):
        w12.w12_gemm_plan(1, 64, 200, 152)   # K % 32 != 0
    with pytest.raises(w12.W12Error):
        w12.w12_gemm_plan(257, 64, 256, 152)


def test_gemm_plan_grouped(w12):
    """The grouped launch's planning: the row blocks of all matrices end to
    end.  When every matrix's rows fill whole row blocks, the group plans
    exactly like one matrix of all their rows; ragged matrices each start a
    row block of their own; a group of one is w12_gemm_plan."""
    rng = np.random.Generator(np.random.PCG64(78))
    for M in (1, 2, 3, 16, 32, 64, 65, 128, 256):
        # q/k/v and gate/up of a 5120-wide layer
        for Ns in ([5120, 1024, 1024], [17408, 17408]):
            g = w12.w12_gemm_plan_grouped(M, Ns, 5120, 152)
            assert g == w12.w12_gemm_plan(M, sum(Ns), 5120, 152), (M, Ns)
        for _ in range(20):
            Ns = [int(v) for v in rng.integers(0, 9000, size=int(rng.integers(1, 5)))]
            K = 32 * int(rng.integers(1, 400))
            sms = int(rng.choice([8, 132, 152]))
            g = w12.w12_gemm_plan_grouped(M, Ns, K, sms)
            if sum(Ns) == 0:
                assert g["kernel"] == 0
                continue
            assert g["row_blocks"] == sum(-(-n // g["block_rows"]) for n in Ns)
            assert g["k_steps"] == -(-K // 256)
            assert 1 <= g["grid"] <= min(g["row_blocks"] * g["k_steps"], sms - min(16, sms // 8))
            assert g["kernel"] == (1 if M <= 2 else 2)
            if len(Ns) == 1:
                assert g == w12.w12_gemm_plan(M, Ns[0], K, sms)
    with pytest.raises(w12.W12Error):
        w12.w12_gemm_plan_grouped(1, [64] * 5, 256, 152)   # more than four matrices
    with pytest.raises(w12.W12Error):
        w12.w12_gemm_plan_grouped(1, [], 256, 152)
    with pytest.raises(w12.W12Error):
        w12.w12_gemm_plan_grouped(1, [64, -1], 256, 152)
