"""Pins that tie the scalar oracle to facts fixed outside the oracle itself.

Each ``pin_*`` function takes an oracle library handle (``None`` = the real
oracle) and raises AssertionError when the oracle disagrees with:
  * a hand-derived worked example (tests/golden/w12_worked_example.txt);
  * a closed form (brute force over all 65536 BF16 patterns, constructed rows);
  * the definition of losslessness (bit-exact round trip);
  * a library routine (numpy float64 matmul) or exact integer arithmetic;
  * the figures the pages print (escape fraction, bits per weight).
The same functions run against deliberately broken copies of the oracle in
test_oracle_mutants.py, which is how we know the pins can fail.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

import oracle as O
import workloads as WL

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden_example():
    rows = {}
    with open(os.path.join(GOLDEN, "w12_worked_example.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            rows.setdefault(key, []).append(vals)
    return rows


def _blob_arrays(blob: bytes, N: int, K: int):
    b = np.frombuffer(blob, dtype=np.uint8)
    n_esc = int(b[24:32].view(np.uint64)[0])
    T = int(b[32:40].view(np.uint64)[0])
    brow = 4 * ((K + 7) // 8)
    off = 40
    ebase = b[off:off + N]
    off += N
    ae = b[off:off + N * K].reshape(N, K)
    off += N * K
    bpl = b[off:off + N * brow].reshape(N, brow)
    off += N * brow
    tptr = b[off:off + 4 * (T + 1)].view("<u4")
    off += 4 * (T + 1)
    esc = b[off:off + 4 * n_esc].view("<u4")
    return ebase, ae, bpl, tptr, esc


# ---- hand-derived worked example -------------------------------------------

def pin_worked_example(lib=None):
    g = _golden_example()
    N, K = int(g["N"][0][0]), int(g["K"][0][0])
    W = np.array([[int(v, 16) for v in r] for r in g["W"]], dtype=np.uint16)
    blob = O.encode(W, lib=lib)
    assert len(blob) == int(g["BLOBLEN"][0][0]), "blob length"
    assert blob[:4] == b"W12\x00"
    ebase, ae, bpl, tptr, esc = _blob_arrays(blob, N, K)
    assert list(ebase) == [int(v) for v in g["EBASE"][0]], "ebase"
    want_ae = np.array([[int(v, 16) for v in r] for r in g["AE"]], dtype=np.uint8)
    assert np.array_equal(ae, want_ae), "AE plane"
    words = bpl.view("<u4").reshape(N, -1)
    want_w = [int(r[0], 16) for r in g["BWORD"]]
    assert [int(words[n, 0]) for n in range(N)] == want_w, "B plane"
    assert [int(v) for v in tptr] == [int(v) for v in g["TILEPTR"][0]], "tile_ptr"
    assert [int(v) for v in esc] == [int(v, 16) for v in g["ESC"][0]], "escapes"
    dec = O.decode(blob, lib=lib)
    assert np.array_equal(dec, W), "lossless decode"
    q8 = O.decode_q8(blob, lib=lib)
    want_q8 = np.array([[int(v, 16) for v in r] for r in g["Q8"]], dtype=np.uint16)
    assert np.array_equal(q8, want_q8), "Q8 view"


# ---- closed forms ------------------------------------------------------------

def pin_all_patterns(lib=None, seed=7):
    """One channel holding every BF16 pattern once: ebase 239, 4096 in window."""
    rng = np.random.Generator(np.random.PCG64(seed))
    row = rng.permutation(np.arange(65536, dtype=np.uint32)).astype(np.uint16)[None, :]
    blob = O.encode(row, lib=lib)
    N, K, n_esc, T = O.blob_header(blob, lib=lib)
    assert (N, K) == (1, 65536)
    assert T == 256
    ebase, ae, bpl, tptr, esc = _blob_arrays(blob, 1, 65536)
    assert int(ebase[0]) == 239, int(ebase[0])
    # 16 binades x 2 signs x 128 mantissas in the window
    assert n_esc == 65536 - 4096, n_esc
    assert np.array_equal(O.decode(blob, lib=lib), row)
    # every escape entry carries the exact original pattern at its position
    k_of = np.empty(65536, dtype=np.int64)
    k_of[row[0].astype(np.int64)] = np.arange(65536)
    for t in range(T):
        for i in range(int(tptr[t]), int(tptr[t + 1])):
            e = int(esc[i])
            k = t * 256 + ((e >> 16) & 0xFF)
            assert (e >> 24) == 0
            assert int(row[0, k]) == (e & 0xFFFF)


def pin_constructed_rows(lib=None):
    # (a) every pattern with exponent 0..16: emax 16 -> ebase 1; only the 256
    #     e = 0 patterns (+-0 and subnormals) escape
    pats = np.array([(s << 15) | (e << 7) | m for s in (0, 1) for e in range(17)
                     for m in range(128)], dtype=np.uint16)[None, :]
    blob = O.encode(pats, lib=lib)
    _, _, n_esc, _ = O.blob_header(blob, lib=lib)
    ebase = _blob_arrays(blob, 1, pats.shape[1])[0]
    assert int(ebase[0]) == 1 and n_esc == 256, (int(ebase[0]), n_esc)
    assert np.array_equal(O.decode(blob, lib=lib), pats)
    # (b) a row of zeros: no finite normal -> ebase 1, all escape
    z = np.zeros((3, 40), dtype=np.uint16)
    z[1] = 0x8000
    blob = O.encode(z, lib=lib)
    _, _, n_esc, _ = O.blob_header(blob, lib=lib)
    assert n_esc == 120 and list(_blob_arrays(blob, 3, 40)[0]) == [1, 1, 1]
    assert np.array_equal(O.decode(blob, lib=lib), z)
    # (c) +-Inf and NaN never set the window; they escape with payload kept
    r = np.full((1, 16), 0x3F80, dtype=np.uint16)  # 1.0, e = 127
    r[0, 3] = 0x7F80
    r[0, 5] = 0xFF80
    r[0, 9] = 0x7FC3
    blob = O.encode(r, lib=lib)
    _, _, n_esc, _ = O.blob_header(blob, lib=lib)
    assert int(_blob_arrays(blob, 1, 16)[0][0]) == 112 and n_esc == 3
    assert np.array_equal(O.decode(blob, lib=lib), r)
    # (d) window edges: emax 20 -> ebase 5; e = 5 is in, e = 4 escapes
    r = np.array([[(20 << 7), (5 << 7) | 0x7F, (4 << 7) | 0x7F, 0x8000 | (19 << 7)]],
                 dtype=np.uint16)
    blob = O.encode(r, lib=lib)
    ebase, ae, _, _, esc = _blob_arrays(blob, 1, 4)
    assert int(ebase[0]) == 5
    assert [int(v) for v in esc] == [(2 << 16) | int(r[0, 2])]
    assert int(ae[0, 1]) == ((0x7F >> 4) << 4) | 0  # A = top mantissa bits, E = 0
    assert int(ae[0, 3]) == ((8 | 0) << 4) | 14     # negative, E = 19 - 5
    # (e) the largest finite exponent 254 sets ebase 239 exactly
    r = np.array([[0x7F7F, 0x3F80, (239 << 7), (238 << 7)]], dtype=np.uint16)
    blob = O.encode(r, lib=lib)
    ebase, _, _, _, esc = _blob_arrays(blob, 1, 4)
    assert int(ebase[0]) == 239 and len(esc) == 2


def pin_roundtrip(lib=None):
    """Lossless: decode(encode(W)) == W bit for bit, shapes with ragged tiles."""
    rng = np.random.Generator(np.random.PCG64(11))
    cases = [
        WL.tiny_weights(1)[0],
        WL.projection_weights(300, 777, seed=3, outlier_frac=3e-3),
        WL.heavy_weights(129, 520, seed=4),
        rng.integers(0, 65536, size=(130, 259), dtype=np.uint16),  # any pattern
        np.zeros((0, 16), dtype=np.uint16),
        np.zeros((5, 0), dtype=np.uint16),
        WL.normal_rows(1, 1, seed=5),
    ]
    for W in cases:
        blob = O.encode(W, lib=lib)
        N, K, _, T = O.blob_header(blob, lib=lib)
        assert (N, K) == W.shape
        assert T == (-(-N // 128)) * (-(-K // 256))
        assert np.array_equal(O.decode(blob, lib=lib), W), W.shape
        if N >= 2:
            part = O.decode_rows(blob, 1, N - 1, lib=lib)
            assert np.array_equal(part, W[1:N - 1])


def pin_escape_list_structure(lib=None):
    """Escape entries: sorted and unique per tile, positions hold placeholders."""
    W = WL.heavy_weights(300, 700, seed=9)
    blob = O.encode(W, lib=lib)
    N, K, n_esc, T = O.blob_header(blob, lib=lib)
    ebase, ae, bpl, tptr, esc = _blob_arrays(blob, N, K)
    assert tptr[0] == 0 and tptr[-1] == n_esc
    tiles_c = -(-K // 256)
    seen = np.zeros((N, K), dtype=bool)
    for t in range(T):
        seg = esc[int(tptr[t]):int(tptr[t + 1])]
        assert np.all(np.diff(seg.astype(np.int64)) > 0)
        for e in seg:
            e = int(e)
            n = (t // tiles_c) * 128 + (e >> 24)
            k = (t % tiles_c) * 256 + ((e >> 16) & 0xFF)
            assert n < N and k < K
            seen[n, k] = True
            s = (int(W[n, k]) >> 15) & 1
            assert int(ae[n, k]) == (s << 7), "placeholder A = s<<3, E = 0"
    # every weight that is not an escape is in its row's window
    e = (W.astype(np.int32) >> 7) & 0xFF
    inwin = (e >= 1) & (e <= 254) & (e >= ebase[:, None]) & (e <= ebase[:, None].astype(np.int32) + 15)
    assert np.array_equal(~inwin, seen)


# ---- the 8-bit view ------------------------------------------------------------

def pin_tiny_composition(lib=None):
    """The 512 x 256 configuration: its 13 forced zeros escape at their
    positions; each row holding a +-50 outlier has window base 117 (50 =
    1.5625 * 2^5, biased exponent 132, minus 15) and escapes exactly its
    weights below 2^-10 (plus its zeros); every other escape is a zero or lies
    below its own row's window."""
    W, _, zpos, opos = WL.tiny_weights(1)
    N, K = W.shape
    blob = O.encode(W, lib=lib)
    ebase, ae, bpl, tptr, esc = _blob_arrays(blob, N, K)
    tiles_c = (K + 255) // 256
    escaped = set()
    for t in range(len(tptr) - 1):
        n0, k0 = (t // tiles_c) * 128, (t % tiles_c) * 256
        for e in esc[tptr[t]:tptr[t + 1]]:
            escaped.add((n0 + (int(e) >> 24), k0 + ((int(e) >> 16) & 0xFF)))
    assert len(escaped) == len(esc)
    for p in zpos:
        assert (p // K, p % K) in escaped
    orows = sorted({int(p) // K for p in opos})
    for n in orows:
        assert int(ebase[n]) == 117, (n, int(ebase[n]))
        row = W[n].astype(np.int32)
        small = ((row & 0x7FFF) < (117 << 7))  # |w| < 2^-10, zeros included
        assert {(n, k) for k in range(K) if small[k]} == {(n, k) for (m, k) in escaped if m == n}
    for (n, k) in escaped:
        e = (int(W[n, k]) >> 7) & 0xFF
        assert (int(W[n, k]) & 0x7FFF) == 0 or e < int(ebase[n])


def pin_q8_nesting(lib=None):
    """Q8 = the weight with its low four mantissa bits cleared (in window);
    escaped slots read +-2^(ebase-127); the AE byte is the record's top byte."""
    W = WL.projection_weights(256, 512, seed=21, outlier_frac=2e-3)
    blob = O.encode(W, lib=lib)
    N, K, _, _ = O.blob_header(blob, lib=lib)
    ebase, ae, bpl, _, _ = _blob_arrays(blob, N, K)
    q8 = O.decode_q8(blob, lib=lib)
    e = (W.astype(np.int32) >> 7) & 0xFF
    inwin = (e >= 1) & (e <= 254) & (e >= ebase[:, None]) & (e <= ebase[:, None].astype(np.int32) + 15)
    assert np.array_equal(q8[inwin], W[inwin] & 0xFFF0)
    s = W.astype(np.int32) >> 15
    ph = (s << 15) | (ebase[:, None].astype(np.int32) << 7)
    assert np.array_equal(q8[~inwin].astype(np.int32), ph[~inwin])
    # the value the Q pass sees is A+E only: the full decode differs from it
    # exactly in the low four mantissa bits of in-window weights
    full = O.decode(blob, lib=lib)
    assert np.array_equal(full[inwin] & 0xFFF0, q8[inwin])
    assert np.array_equal((full[inwin] & 0xF), (W[inwin] & 0xF))


# ---- GEMM ----------------------------------------------------------------------

def pin_gemm_numpy(lib=None):
    """fp64 reference against numpy's float64 matmul of the decoded matrix."""
    W = WL.projection_weights(200, 300, seed=5, outlier_frac=1e-3)
    x = WL.activations(5, 300, seed=6)
    y = O.gemm(x, W, lib=lib)
    xf = WL.bf16_bits_to_f32(x).astype(np.float64)
    wf = WL.bf16_bits_to_f32(W).astype(np.float64)
    ref = xf @ wf.T
    scale = np.abs(xf) @ np.abs(wf).T
    assert np.all(np.abs(y - ref) <= 1e-12 * scale + 1e-300)
    s = O.abs_gemm(x, W, lib=lib)
    assert np.allclose(s, scale, rtol=1e-12, atol=0)
    # rows computed block-wise agree with the full call
    blk = O.gemm_rows(x, W[17:40], lib=lib)
    assert np.array_equal(blk, y[:, 17:40])


def pin_gemm_one_hot(lib=None):
    """x = unit rows e_k: y[m][n] is exactly W[n][k] (any finite W)."""
    W = WL.heavy_weights(64, 96, seed=13)
    W[0, :] = np.arange(96, dtype=np.uint16) | 0x0001  # subnormals
    K = W.shape[1]
    for k0 in (0, 37, 95):
        x = np.zeros((1, K), dtype=np.uint16)
        x[0, k0] = 0x3F80  # 1.0
        y = O.gemm(x, W, lib=lib)
        assert np.array_equal(y[0], WL.bf16_bits_to_f32(W[:, k0]).astype(np.float64))


def pin_gemm_exact_integers(lib=None):
    """All-ones x and W of powers of two: sums are exact integers."""
    rng = np.random.Generator(np.random.PCG64(17))
    N, K = 40, 200
    ex = rng.integers(-4, 6, size=(N, K))
    sg = rng.integers(0, 2, size=(N, K))
    W = ((sg << 15) | ((127 + ex) << 7)).astype(np.uint16)
    x = np.full((2, K), 0x3F80, dtype=np.uint16)
    x[1, ::2] = 0xBF80  # -1 on even k
    y = O.gemm(x, W, lib=lib)
    for n in range(N):
        v = [Fraction(-1 if sg[n, k] else 1) * Fraction(2) ** int(ex[n, k]) for k in range(K)]
        assert y[0, n] == float(sum(v))
        assert y[1, n] == float(sum(-v[k] if k % 2 == 0 else v[k] for k in range(K)))


# ---- count-maximising window (encoder option) ------------------------------------

def _brute_count_max_base(row):
    """The rule written out directly: every base b from 1 up to the
    max-anchored one, counting the row's finite normal weights whose exponent
    lies in [b, b + 15]; the largest b with the most."""
    e = [(int(v) >> 7) & 0xFF for v in row]
    normal = [x for x in e if 1 <= x <= 254]
    b1 = max(max(normal, default=0), 16) - 15
    best, best_b = -1, 1
    for b in range(1, b1 + 1):
        c = sum(1 for x in normal if b <= x <= b + 15)
        if c >= best:
            best, best_b = c, b
    return best_b


def pin_count_max_window(lib=None):
    """Window bases against the brute-force rule on constructed and random
    rows, and the escape count never above the max-anchored one."""
    rng = np.random.Generator(np.random.PCG64(93))
    rows = [
        np.zeros(64, dtype=np.uint16),                      # no normal weight: b = 1
        np.array([0x7F80, 0x3F80, 0x0001] * 8, dtype=np.uint16),
        np.array([0x7F7F] + [0x3F80] * 40, dtype=np.uint16),  # one huge outlier: the window drops
        np.array([0x7F7F] * 40 + [0x3F80] * 40, dtype=np.uint16),  # a tie: the higher window
        np.array([(e << 7) for e in range(1, 255)], dtype=np.uint16),  # one of every exponent
        np.array([(e << 7) | 0x8000 for e in range(100, 140)] * 3 + [200 << 7], dtype=np.uint16),
    ]
    for i in range(40):
        centre = int(rng.integers(20, 230))
        e = np.clip(rng.normal(centre, rng.uniform(2, 20), size=97).round(), 0, 255).astype(np.uint16)
        rows.append(((rng.integers(0, 2, 97).astype(np.uint16) << 15) | (e << 7)
                     | rng.integers(0, 128, 97).astype(np.uint16)).astype(np.uint16))
    for r in rows:
        got = O.row_ebase(r, lib=lib, count_max=True)
        assert got == _brute_count_max_base(r), (got, _brute_count_max_base(r), r[:8])
    # the outlier row keeps 1.0 (exponent 127) in its window and lets 2^127 escape
    b = O.row_ebase(rows[2], lib=lib, count_max=True)
    assert b <= 127 <= b + 15 and b + 15 < 254
    W = WL.heavy_weights(64, 1024, seed=94)
    for n in range(64):
        bm = O.row_ebase(W[n], lib=lib)
        bc = O.row_ebase(W[n], lib=lib, count_max=True)
        e = (W[n].astype(np.int32) >> 7) & 0xFF
        normal = (e >= 1) & (e <= 254)
        assert np.sum(normal & (e >= bc) & (e <= bc + 15)) >= np.sum(normal & (e >= bm) & (e <= bm + 15))


def pin_count_max_encoding(lib=None):
    """Blobs with the count-maximising window: lossless; weights above the
    window escape with the saturated placeholder (A = s<<3|7, E = 15, B = 15),
    which the 8-bit view reads as +-1.875 * 2^(ebase+15-127); weights below it
    keep the ordinary placeholder; fewer escapes on heavy tails."""
    W = WL.projection_weights(96, 520, seed=95, outlier_frac=5e-3)
    W[3, 7] = 0x7F7F   # huge, positive
    W[4, 9] = 0xFF00   # huge, negative
    W[5, :] = 0x3F80   # a flat row: every weight in one binade
    blob = O.encode(W, lib=lib, count_max=True)
    N, K, n_esc, T = O.blob_header(blob, lib=lib)
    assert np.array_equal(O.decode(blob, lib=lib), W)
    ebase, ae, bpl, tptr, esc = _blob_arrays(blob, N, K)
    e = (W.astype(np.int32) >> 7) & 0xFF
    eb = ebase.astype(np.int32)[:, None]
    normal = (e >= 1) & (e <= 254)
    inwin = normal & (e >= eb) & (e <= eb + 15)
    above = normal & (e > eb + 15)
    assert above[3, 7] and above[4, 9] and above.sum() >= 2
    s = (W.astype(np.int32) >> 15)
    assert np.array_equal(ae[above].astype(np.int32), (s[above] << 7) | 0x7F)
    below = ~inwin & ~above
    assert np.array_equal(ae[below].astype(np.int32), s[below] << 7)
    kk = np.arange(K)
    slot = np.where(kk % 2 == 1, 4 + kk % 8 // 2, kk % 8 // 2)
    words = bpl.reshape(N, -1).view("<u4")
    nib = (words[:, kk // 8] >> (4 * slot)) & 0xF
    assert np.all(nib[above] == 15) and np.all(nib[below] == 0)
    assert n_esc == int((~inwin).sum())
    q8 = O.decode_q8(blob, lib=lib).astype(np.int32)
    assert np.array_equal(q8[above], (s[above] << 15) | ((eb + 15) * np.ones_like(e))[above] << 7 | 0x70)
    # max-anchored blobs of the same matrix have no weight above the window
    blob1 = O.encode(W, lib=lib)
    e1 = O.blob_header(blob1, lib=lib)[2]
    assert n_esc <= e1
    H = WL.heavy_weights(128, 2048, seed=96)
    f_max = O.blob_header(O.encode(H, lib=lib), lib=lib)[2] / H.size
    f_cnt = O.blob_header(O.encode(H, lib=lib, count_max=True), lib=lib)[2] / H.size
    assert f_cnt < 0.4 * f_max, (f_cnt, f_max)
    pats = np.random.Generator(np.random.PCG64(97)).permutation(
        np.arange(65536, dtype=np.uint32)).astype(np.uint16).reshape(8, 8192)
    assert np.array_equal(O.decode(O.encode(pats, lib=lib, count_max=True), lib=lib), pats)


# ---- INT8 copy for the Q pass -------------------------------------------------------

def _bf16(vals):
    """BF16 bit patterns of values that BF16 holds exactly."""
    a = np.asarray(vals, dtype=np.float32).view(np.uint32)
    assert np.all((a & 0xFFFF) == 0)
    return (a >> 16).astype(np.uint16)


def pin_i8_quantize(lib=None):
    """Worked rows whose scale is exact (amax 127 -> scale 1, amax 254 ->
    scale 2), so every tie is a true tie and goes to the even integer; Inf,
    NaN and zero rows; and on random rows the properties any such
    quantisation has: |q| <= 127, the largest finite weight maps to +-127,
    |w - q scale| <= scale / 2, order and sign kept."""
    inf, nan = float("inf"), float("nan")
    rows = [
        ([127.0, 2.5, 3.5, -2.5, 126.5, 0.5, 1.5, -1.5, inf, -inf, nan, 0.0, -0.0, 64.0],
         [127, 2, 4, -2, 126, 0, 2, -2, 127, -127, 0, 0, 0, 64], 1.0),
        ([254.0, 3.0, 5.0, -7.0, 1.0, -254.0, 9.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0],
         [127, 2, 2, -4, 0, -127, 4, 0, 0, 0, 0, 0, 0, 0], 2.0),
        ([0.0] * 14, [0] * 14, 0.0),
    ]
    W = np.stack([_bf16(np.array(r[0], dtype=np.float32)) for r in rows])
    q, sc = O.i8_quantize(W, lib=lib)
    for i, (_, want, s) in enumerate(rows):
        assert sc[i] == np.float32(s), (i, sc[i])
        assert q[i].tolist() == want, (i, q[i].tolist())
    W = WL.projection_weights(64, 700, seed=98, outlier_frac=3e-3)
    W[5, :] = 0
    q, sc = O.i8_quantize(W, lib=lib)
    wf = WL.bf16_bits_to_f32(W).astype(np.float64)
    assert np.all(np.abs(q.astype(np.int32)) <= 127)
    for n in range(64):
        amax = np.abs(wf[n]).max()
        if amax == 0:
            assert sc[n] == 0 and not q[n].any()
            continue
        assert abs(float(sc[n]) - amax / 127) <= 2.0 ** -23 * amax / 127
        assert np.abs(q[n]).max() == 127 and abs(int(q[n][np.argmax(np.abs(wf[n]))])) == 127
        err = np.abs(wf[n] - q[n].astype(np.float64) * float(sc[n]))
        assert np.all(err <= 0.5 * float(sc[n]) * (1 + 2.0 ** -18))
        assert np.all((np.sign(q[n]) == np.sign(wf[n])) | (q[n] == 0))
        o = np.argsort(wf[n], kind="stable")
        assert np.all(np.diff(q[n][o].astype(np.int32)) >= 0)


def pin_gemm_i8(lib=None):
    """The INT8 product against numpy's float64 matmul of the dequantised
    weights, and one-hot activations picking single q * scale values."""
    W = WL.projection_weights(90, 333, seed=99, outlier_frac=2e-3)
    q, sc = O.i8_quantize(W, lib=lib)
    x = WL.activations(4, 333, seed=100)
    y = O.gemm_i8(x, q, sc, lib=lib)
    xf = WL.bf16_bits_to_f32(x).astype(np.float64)
    deq = q.astype(np.float64) * sc.astype(np.float64)[:, None]
    ref = xf @ deq.T
    scale = np.abs(xf) @ np.abs(deq).T
    assert np.all(np.abs(y - ref) <= 1e-12 * scale + 1e-300)
    assert np.allclose(O.abs_gemm_i8(x, q, sc, lib=lib), scale, rtol=1e-12, atol=0)
    for k0 in (0, 100, 332):
        e = np.zeros((1, 333), dtype=np.uint16)
        e[0, k0] = 0x3F80
        assert np.array_equal(O.gemm_i8(e, q, sc, lib=lib)[0], deq[:, k0])


# ---- epilogues: BF16 output and the gated-MLP product ----------------------------

def _f32(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


def pin_round_bf16(lib=None):
    """Round to nearest, ties to even: worked bit patterns (ties both ways,
    sign, overflow, subnormals, infinities) and agreement with PyTorch's CPU
    float32 -> bfloat16 conversion on random bit patterns."""
    table = [
        (0x3F800000, 0x3F80),  # exact
        (0x3F808000, 0x3F80),  # 1 + 2^-8: tie, even stays
        (0x3F818000, 0x3F82),  # 1 + 3*2^-8: tie, odd rounds up
        (0x3F808001, 0x3F81),  # just above the tie
        (0x3F807FFF, 0x3F80),  # just below the tie
        (0xBF808001, 0xBF81),  # sign kept, magnitude rounded
        (0xBF818000, 0xBF82),
        (0x7F7F7FFF, 0x7F7F),  # largest finite BF16 stays
        (0x7F7F8000, 0x7F80),  # its tie with 2^128 goes to infinity (even)
        (0xFF7FFFFF, 0xFF80),  # largest finite FP32 overflows
        (0x00008000, 0x0000),  # subnormal tie, even
        (0x00018000, 0x0002),  # subnormal tie, odd rounds up
        (0x80000001, 0x8000),
        (0x7F800000, 0x7F80),
        (0xFF800000, 0xFF80),
    ]
    got = O.round_bf16(_f32([t[0] for t in table]), lib=lib)
    for (i, o), g in zip(table, got):
        assert int(g) == o, (hex(i), hex(int(g)), hex(o))
    nan = O.round_bf16(_f32([0x7FC00001, 0xFF800001]), lib=lib)
    assert all((int(v) & 0x7F80) == 0x7F80 and (int(v) & 0x7F) for v in nan)
    import torch

    rng = np.random.Generator(np.random.PCG64(91))
    bits = rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    bits = bits[(bits & 0x7F800000) != 0x7F800000]
    want = torch.from_numpy(_f32(bits).copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.round_bf16(_f32(bits), lib=lib), want)


def pin_silu_mul(lib=None):
    """h = silu(gate) * up with gate/up interleaved by row: worked values, the
    identity silu(g) - silu(-g) = g, and the large-|g| limits."""
    e = np.exp(1.0)
    y = np.array([[0.0, 5.0, 1.0, 2.0, -1.0, 3.0, 2.0, -0.5]])
    want = [0.0, 2.0 * (1.0 / (1.0 + 1.0 / e)), 3.0 * (-1.0 / (1.0 + e)), -0.5 * (2.0 / (1.0 + np.exp(-2.0)))]
    h = O.silu_mul(y, lib=lib)
    assert h.shape == (1, 4)
    assert np.allclose(h[0], want, rtol=1e-15, atol=0)
    g = np.random.Generator(np.random.PCG64(92)).normal(0, 3, size=1000)
    pos = O.silu_mul(np.stack([g, np.ones_like(g)], 1).reshape(1, -1), lib=lib)[0]
    neg = O.silu_mul(np.stack([-g, np.ones_like(g)], 1).reshape(1, -1), lib=lib)[0]
    assert np.allclose(pos - neg, g, rtol=1e-13, atol=1e-13)
    big = O.silu_mul(np.array([[60.0, 1.0, -60.0, 1.0, -800.0, 1.0]]), lib=lib)[0]
    assert big[0] == 60.0 and -1e-24 < big[1] < 0 and big[2] == 0.0


# ---- the printed figures -------------------------------------------------------

def printed_figures():
    out = {}
    with open(os.path.join(GOLDEN, "printed_figures.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()
                out[k] = float(v)
    return out


def expected_escape_fraction(K: int, sigma0: float = 0.02, n_scale: int = 400) -> float:
    """Analytic escape probability of one weight for rows W ~ N(0, (sigma0 c)^2),
    c ~ U(0.5, 2), with the window anchored at the row maximum's binade.

    A weight escapes iff |w| < 2^(j-15) where 2^j <= max|row| < 2^(j+1); since
    such a weight cannot be the maximum, P = sum_j F(2^(j-15)) *
    [F(2^(j+1))^(K-1) - F(2^j)^(K-1)] with F(t) = erf(t / (sigma sqrt 2)).
    """
    from scipy.special import erf

    j = np.arange(-40, 8, dtype=np.float64)
    acc = 0.0
    cs = 0.5 + 1.5 * (np.arange(n_scale) + 0.5) / n_scale
    for c in cs:
        sig = sigma0 * c

        def F(t):
            return erf(t / (sig * np.sqrt(2.0)))

        p = F(2.0 ** (j - 15)) * (F(2.0 ** (j + 1)) ** (K - 1) - F(2.0 ** j) ** (K - 1))
        acc += p.sum()
    return acc / len(cs)


def pin_escape_fraction(lib=None, N=2048, K=5120, seed=31):
    """Normal weights: the oracle's escape fraction matches the analytic value
    for the max-anchored window and lands near the pages' 7.3e-5."""
    W = WL.normal_rows(N, K, seed=seed)
    blob = O.encode(W, lib=lib)
    _, _, n_esc, _ = O.blob_header(blob, lib=lib)
    frac = n_esc / (N * K)
    # per-row escape counts -> a standard error that includes the row-level
    # correlation through the shared maximum
    ebase = _blob_arrays(blob, N, K)[0].astype(np.int32)
    e = (W.astype(np.int32) >> 7) & 0xFF
    per_row = ((e < ebase[:, None]) | (e == 0)).sum(axis=1) / K
    se = per_row.std(ddof=1) / np.sqrt(N)
    ana = expected_escape_fraction(K)
    assert abs(frac - ana) <= 5 * se + 0.03 * ana, (frac, ana, se)
    fig = printed_figures()["escape_fraction"]
    assert abs(frac - fig) <= 0.15 * fig, (frac, fig)
    return frac, ana


def pin_bits_per_weight(lib=None):
    """Storage: 12 bits + escapes + metadata, within the pages' 12.01-12.02."""
    N, K = 1024, 5120
    W = WL.normal_rows(N, K, seed=41)
    blob = O.encode(W, lib=lib)
    _, _, n_esc, T = O.blob_header(blob, lib=lib)
    bpw = 8 * len(blob) / (N * K)
    fig = printed_figures()
    assert 12.0 < bpw <= fig["bits_per_weight_max"], bpw
    # the size is fixed by the layout: 12 bits + 8/K (ebase) + tile pointers + escapes
    want = 40 + N + N * K + N * 4 * ((K + 7) // 8) + 4 * (T + 1) + 4 * n_esc
    assert len(blob) == want
    return bpw


def pin_converted_size(lib=None):
    """The pages' converted size: 44.67 GB of BF16 layers become 33.58 GB,
    i.e. 16 * 33.58 / 44.67 = 12.03 bits per weight.  The format's own
    accounting on normal weights (every byte of the blob) must land within
    0.5 % of that."""
    fig = printed_figures()
    bpw = pin_bits_per_weight(lib)
    predicted = fig["converted_gb_before"] * bpw / 16.0
    assert abs(predicted - fig["converted_gb_after"]) <= 0.005 * fig["converted_gb_after"], (predicted, bpw)
    return predicted


FAST_PINS = (
    pin_worked_example,
    pin_all_patterns,
    pin_constructed_rows,
    pin_roundtrip,
    pin_escape_list_structure,
    pin_q8_nesting,
    pin_tiny_composition,
    pin_gemm_numpy,
    pin_gemm_one_hot,
    pin_gemm_exact_integers,
    pin_round_bf16,
    pin_silu_mul,
    pin_count_max_window,
    pin_count_max_encoding,
    pin_i8_quantize,
    pin_gemm_i8,
)
