"""Pins of the CPU oracle against things other than itself.

Each test fixes one part of the oracle against a library routine, a closed form,
a brute-force computation in exact (Python integer / Fraction) arithmetic, a value
printed on the pages, or a hand-derived fixture under tests/golden/.  A plausible
mistake anywhere in the oracle (a dropped term, a wrong sign or index, a swapped
operand, a wrong tie rule) fails at least one of them.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.linalg

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
D = 256


# ----------------------------------------------------------------------------- fp16

def test_fp16_matches_numpy_on_every_exponent(orc):
    """The oracle's binary16 rounding equals numpy's float32 -> float16 cast (a
    library routine) for every fp32 exponent, random mantissas and every exact tie."""
    rng = np.random.default_rng(1)
    ef = np.arange(256, dtype=np.uint32)
    pats = []
    for sign in (0, 1):
        mant = rng.integers(0, 1 << 23, size=(256, 2048), dtype=np.uint32)
        pats.append((sign << 31) | (ef[:, None] << 23) | mant)
        # ties and near-ties for every possible number of dropped bits
        for drop in range(1, 24):
            half = np.uint32(1 << (drop - 1))
            base = rng.integers(0, 1 << 23, size=(256, 8), dtype=np.uint32) & ~np.uint32((1 << drop) - 1)
            for delta in (0, 1):
                m = (base | half) + np.uint32(delta) if delta else (base | half)
                pats.append((sign << 31) | (ef[:, None] << 23) | (m & np.uint32(0x7FFFFF)))
            pats.append((sign << 31) | (ef[:, None] << 23) | ((base | half) - np.uint32(1)) & np.uint32(0x7FFFFF))
    bits = np.concatenate([p.reshape(-1) for p in pats]).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = orc.f32_to_f16_array(x)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first {x[bad[0]]!r}: {got[bad[0]]:#x} vs {ref[bad[0]]:#x}"


def test_fp16_back_conversion_exact(orc):
    allh = np.arange(1 << 16, dtype=np.uint16)
    ref = allh.view(np.float16).astype(np.float32)
    got = np.array([orc.f16_bits_to_f32(int(h)) for h in allh[::7]], np.float32)
    fin = np.isfinite(ref[::7])
    assert np.array_equal(got[fin], ref[::7][fin])


# ----------------------------------------------------------------------------- Hadamard

def H_oracle():
    return np.array([[synth_entry(i, j) for j in range(D)] for i in range(D)])


_H = None


def synth_entry(i, j):
    import oracle
    return oracle.hadamard_entry(i, j)


def test_hadamard_is_sylvester_and_orthogonal(orc):
    """H equals scipy's Sylvester Hadamard matrix and H.H = 256 I exactly."""
    H = np.array([[orc.hadamard_entry(i, j) for j in range(D)] for i in range(D)], dtype=np.int64)
    assert np.array_equal(H, scipy.linalg.hadamard(D).astype(np.int64))
    assert np.array_equal(H @ H, 256 * np.eye(D, dtype=np.int64))


def test_rotate_unit_vectors(orc):
    """rotate(e_k) = H[:, k] / 16 (column k), e.g. e_0 -> all 1/16."""
    Hs = scipy.linalg.hadamard(D)
    for k in (0, 1, 37, 128, 255):
        e = np.zeros(D, np.float32)
        e[k] = 1.0
        assert np.array_equal(orc.rotate(e), (Hs[:, k] / 16.0).astype(np.float32))


def _round_to_f32(v: Fraction) -> np.float32:
    """Correct rounding of an exact rational to fp32 (nearest, ties to even), by
    brute force over the three fp32 neighbours of float32(float(v))."""
    if v == 0:
        return np.float32(0.0)
    c = np.float32(float(v))
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    best = None
    for cand in cands:
        if not np.isfinite(cand):
            continue
        err = abs(Fraction(float(cand)) - v)
        key = (err, int(np.float32(cand).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, cand)
    return np.float32(best[1])


def _exact_rotation(x: np.ndarray) -> np.ndarray:
    Hs = scipy.linalg.hadamard(D).astype(np.int64)
    xs = [Fraction(float(t)) for t in x]
    return np.array([_round_to_f32(sum((xs[j] if Hs[i, j] > 0 else -xs[j]) for j in range(D)) / 16)
                     for i in range(D)], np.float32)


@pytest.mark.parametrize("case", ["normal", "wide", "subnormal", "cancel"])
def test_rotate_equals_exact_rational_rounding(orc, case):
    """The oracle's multi-limb rotation equals exact rational arithmetic followed by
    one correct fp32 rounding, including extreme exponent spreads."""
    rng = np.random.default_rng({"normal": 2, "wide": 3, "subnormal": 4, "cancel": 5}[case])
    if case == "normal":
        x = rng.standard_normal(D).astype(np.float32)
    elif case == "wide":
        x = (rng.standard_normal(D) * 10.0 ** rng.integers(-30, 30, D)).astype(np.float32)
    elif case == "subnormal":
        x = (rng.standard_normal(D) * 1e-39).astype(np.float32)   # mostly subnormal fp32
        x[:4] = [1e-45, -1e-45, 3e-45, 1e-38]
    else:
        # near-total cancellation: the sums are tiny, so low-order bits decide
        x = np.zeros(D, np.float32)
        x[0], x[1] = 1.0, 1.0 + 2.0 ** -23
        x[2] = 2.0 ** -60
        x[3] = -(2.0 ** -100)
    got = orc.rotate(x)
    ref = _exact_rotation(x)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_rotate_round_trip_and_norm(orc):
    """For dyadic sparse y, x = (H/16) y is exact in fp32 and rotate(x) = y exactly;
    the rotation is orthonormal: ||rotate(x)|| = ||x|| up to fp32 rounding."""
    Hs = scipy.linalg.hadamard(D).astype(np.float64)
    rng = np.random.default_rng(6)
    y = np.zeros(D)
    idx = rng.choice(D, 12, replace=False)
    y[idx] = rng.integers(-64, 64, 12) / 8.0
    x = (Hs @ y) / 16.0
    assert np.array_equal(x.astype(np.float32).astype(np.float64), x)
    assert np.array_equal(orc.rotate(x.astype(np.float32)).astype(np.float64), y)
    z = rng.standard_normal(D).astype(np.float32)
    rz = orc.rotate(z).astype(np.float64)
    assert abs(np.linalg.norm(rz) - np.linalg.norm(z.astype(np.float64))) < 1e-6 * np.linalg.norm(z)
    # the rotation is its own inverse up to the two roundings
    assert np.max(np.abs(orc.rotate(orc.rotate(z)) - z)) < 1e-6


# ----------------------------------------------------------------------------- int8

def _read_int8_golden():
    rows = []
    for line in open(os.path.join(GOLDEN, "int8_ties.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        parts = line.split()
        s = float(parts[0])
        pairs = [(float(a), int(b)) for a, b in (p.split(":") for p in parts[1:])]
        rows.append((s, pairs))
    return rows


def test_int8_hand_ties(orc):
    for s, pairs in _read_int8_golden():
        x = np.zeros(128, np.float32)
        for i, (n, _) in enumerate(pairs):
            x[i] = n * s
        c, got_s = orc.quant_int8(x)
        assert got_s == s
        assert [int(t) for t in c[:len(pairs)]] == [code for _, code in pairs]


def test_int8_bound_and_extremes(orc):
    rng = np.random.default_rng(7)
    for trial in range(200):
        x = (rng.standard_normal(128) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
        c, s = orc.quant_int8(x)
        a = np.max(np.abs(x))
        assert s == np.float32(a) / np.float32(127.0)
        err = np.abs(x.astype(np.float64) - c.astype(np.float64) * s)
        assert np.all(err <= s / 2 * (1 + 2.0 ** -20))
        assert abs(int(c[np.argmax(np.abs(x))])) == 127
        assert np.all(np.abs(c.astype(np.int32)) <= 127)
    c, s = orc.quant_int8(np.zeros(128, np.float32))
    assert s == 0.0 and not c.any()


def _read_quotient_golden(name):
    """Rows of int8_quotient.txt / q4_quotient.txt: the fp32 inputs (exact hex)
    and, per reading of the quotient, the code it gives."""
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if not line:
            continue
        fields = [f.split() for f in line.split("|")]
        vals = [float.fromhex(t) for t in fields[0]]
        codes = [int(f[0]) for f in fields[1:]]
        rows.append((vals, codes))
    return rows


def test_int8_quotient_is_one_ieee_division(orc):
    """Codes that tell x / s apart from x * (1 / s) and from (x * 127) / a (the
    PR's Tests section fixes the rounding of the code, half to even; the
    quotient is read as one correctly rounded fp32 division).  Each fixture line
    was derived with exact rational arithmetic; a non-power-of-two absmax makes
    the three readings differ."""
    rows = _read_quotient_golden("int8_quotient.txt")
    assert len(rows) >= 8
    recip_differs = absmax_differs = 0
    for (a, x, s), (code, code_recip, code_absmax) in rows:
        # the fixture's own consistency, checked exactly
        assert Fraction(s) == _round_to_f32(Fraction(a) / 127)
        recip_differs += code_recip != code
        absmax_differs += code_absmax != code
        half = np.zeros(128, np.float32)
        half[0], half[1] = a, x
        c, got_s = orc.quant_int8(half)
        assert got_s == s
        assert int(c[0]) == 127 and int(c[1]) == code, (a, x, int(c[1]), code)
    assert recip_differs >= 4 and absmax_differs >= 4


# ----------------------------------------------------------------------------- Q4_0

def _read_q4_golden():
    rows = []
    for line in open(os.path.join(GOLDEN, "q4_ties.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        parts = line.split()
        blk, d = int(parts[0]), float(parts[1])
        trip = [(int(a), float(b), int(c)) for a, b, c in (p.split(":") for p in parts[2:])]
        rows.append((blk, d, trip))
    return rows


def test_q4_hand_ties_through_rotation(orc):
    """Blocks built in the rotated domain, fed through x = (H/16) y and the oracle's
    rotation, give the hand-derived codes and scales."""
    for blk, d, trip in _read_q4_golden():
        y = np.zeros(32, np.float32)
        for lane, val, _ in trip:
            y[lane] = val
        Hs = scipy.linalg.hadamard(D).astype(np.float64)
        full = np.zeros(D)
        full[32 * blk:32 * blk + 32] = y
        x = ((Hs @ full) / 16.0).astype(np.float32)
        yr = orc.rotate(x)
        assert np.array_equal(yr[32 * blk:32 * blk + 32], y)
        nib, db = orc.quant_q4_block(yr[32 * blk:32 * blk + 32])
        assert np.float16(d).view(np.uint16) == db
        codes = np.concatenate([nib & 15, nib >> 4])
        want = np.full(32, 8)
        for lane, _, code in trip:
            want[lane] = code
        assert np.array_equal(codes, want), (blk, codes, want)
        # the other blocks are all zero: d = -0 (0 / -8) and every code 8
        other = (blk + 1) % 8
        nib0, d0 = orc.quant_q4_block(yr[32 * other:32 * other + 32])
        assert d0 == 0x8000 and np.all(nib0 == 0x88)


def test_q4_quotient_is_one_ieee_division(orc):
    """Q4_0 codes that tell y / d apart from y * (1 / d): blocks whose fp16
    scale d has a non-power-of-two significand, with y next to a half-integer
    multiple of d (fixture derived with exact rational arithmetic)."""
    rows = _read_quotient_golden("q4_quotient.txt")
    assert len(rows) >= 6
    for (m, y, d), (code, code_recip) in rows:
        assert code_recip != code
        blk = np.zeros(32, np.float32)
        blk[0], blk[1] = m, y
        nib, db = orc.quant_q4_block(blk)
        assert db == int(np.float16(d).view(np.uint16)) and float(np.float16(d)) == d
        codes = np.concatenate([nib & 15, nib >> 4])
        assert codes[0] == 0 and codes[1] == code, (m, y, int(codes[1]), code)
        assert np.all(codes[2:] == 8)


def test_q4_error_bounds(orc):
    """|y - (q-8) d| <= |d|/2 for unclamped codes; a clamped code (y/d >= 7.5, only
    for elements opposite in sign to m) errs by at most |d| (1 + 2^-10); m -> 0."""
    rng = np.random.default_rng(8)
    n_clamped = 0
    for trial in range(400):
        y = (rng.standard_normal(32) * 10.0 ** rng.uniform(-2, 2)).astype(np.float32)
        if trial % 3 == 0:
            y[rng.integers(32)] = -np.max(np.abs(y)) * rng.uniform(0.94, 1.0)
        nib, db = orc.quant_q4_block(y)
        d = float(np.uint16(db).view(np.float16))
        q = np.concatenate([nib & 15, nib >> 4]).astype(np.int64)
        err = np.abs(y.astype(np.float64) - (q - 8) * d)
        clamped = (q == 15) & (y.astype(np.float64) / d >= 7.5)
        n_clamped += int(clamped.sum())
        assert np.all(err[~clamped] <= abs(d) / 2 * (1 + 2.0 ** -20))
        assert np.all(err[clamped] <= abs(d) * (1 + 2.0 ** -10))
        im = int(np.argmax(np.abs(y)))
        assert q[im] == 0
        assert db == np.float16(np.float32(y[im]) / np.float32(-8.0)).view(np.uint16)
    assert n_clamped > 0


# ----------------------------------------------------------------------------- layout

def test_bytes_per_cell(orc):
    assert 2 * orc.bytes_per_cell_head(orc.FMT_K8V4) == 816
    assert 2 * orc.bytes_per_cell_head(orc.FMT_INT8) == 1056
    # the k8v4 PR (#120, section "What") gives 816 B per cell against 1,056 for
    # all-int8 and 576 for all-q4_0
    assert 2 * orc.bytes_per_cell_head(orc.FMT_Q4) == 576
    # 816 = 512 K codes + 16 K scales + 256 V nibbles + 32 V scales
    assert 2 * (256 + 8 + 128 + 16) == 816


def test_memory_figures_printed_on_pages(orc):
    sizes = {"k8v4": 2 * orc.bytes_per_cell_head(orc.FMT_K8V4), "int8": 2 * orc.bytes_per_cell_head(orc.FMT_INT8)}
    n = 0
    for line in open(os.path.join(GOLDEN, "memory_figures.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        cells, layers, fmt, printed, unit, _src = line.split()
        gib = int(cells) * int(layers) * sizes[fmt] / 2 ** 30
        decimals = len(printed.split(".")[1])
        assert round(gib, decimals) == float(printed), (line, gib)
        n += 1
    assert n == 6
    # the 131K-context KV bytes 1.80 GB -> 1.39 GB (same PR, "Measured" table)
    assert round(1.80 * 816 / 1056, 2) == 1.39


def test_page_layout_hand_offsets(orc):
    """Cell c of a sequence lives in page pt[c // P], slot c % P; within a page of P
    cells and H heads the four runs are K codes [P][H][256], K scales [P][H][2] f32,
    V nibbles [P][H][8][16], V scales [P][H][8] f16 (offsets derived by hand)."""
    P, H = 2, 2
    cache = orc.Cache(n_pages=3, P=P, H=H)
    pt = np.array([[2, 0]], np.int32)                     # cells 0,1 -> page 2; 2,3 -> page 0
    k = np.zeros((1, 1, H, D), np.float32)
    v = np.zeros((1, 1, H, D), np.float32)
    k[0, 0, 1, 5] = 127.0                                # head 1, half 0: s = 1, code[5] = 127
    k[0, 0, 1, 200] = -2.0 * 127                         # head 1, half 1: s = 2, code[200] = -127
    v[0, 0, 1, :] = 1.0                                  # rotates to 16 e_0 -> block 0: m = 16, d = -2
    cache.append(pt, np.array([3]), k, v)                # logical cell 3 -> page 0, slot 1
    page = 0 * P * 816
    kc = page + (1 * H + 1) * 256
    ks = page + 512 * P + (1 * H + 1) * 8
    vq = page + 528 * P + (1 * H + 1) * 128
    vs = page + 784 * P + (1 * H + 1) * 16
    b = cache.buf
    assert b[kc + 5] == 127 and b[kc + 200].view(np.int8) == -127
    assert np.frombuffer(b[ks:ks + 8].tobytes(), np.float32).tolist() == [1.0, 2.0]
    assert b[vq] == (0 | (8 << 4)) and np.all(b[vq + 1:vq + 128] == 0x88)
    dv = np.frombuffer(b[vs:vs + 16].tobytes(), np.uint16)
    assert dv[0] == np.float16(-2.0).view(np.uint16) and np.all(dv[1:] == 0x8000)
    # head 0 of the same cell: all-zero input -> codes 0, scales 0, V codes 8, d = -0
    kc0 = page + (1 * H + 0) * 256
    assert not b[kc0:kc0 + 256].any()
    # nothing else was written
    touched = np.zeros(b.size, bool)
    for base, n in ((page + (1 * H) * 256, 512), (page + 512 * P + 2 * H * 8 - 16, 16),
                    (page + 528 * P + (1 * H) * 128, 256), (page + 784 * P + (1 * H) * 16, 32)):
        touched[base:base + n] = True
    assert not b[~touched].any()


# ----------------------------------------------------------------------------- attention

def _small_cache(orc, fmt, seed=11, n=77, P=8, H=2):
    rng = np.random.default_rng(seed)
    n_pages = (n + P - 1) // P
    pt = rng.permutation(n_pages + 3)[:n_pages].astype(np.int32)[None]
    k = rng.standard_normal((1, n, H, D)).astype(np.float32)
    v = rng.standard_normal((1, n, H, D)).astype(np.float32)
    k[..., 3] *= 20
    v[..., 7] *= 20
    cache = orc.Cache(n_pages + 3, P, H, fmt)
    cache.append(pt, np.array([0]), k, v)
    return cache, pt, n


@pytest.mark.parametrize("fmt", ["k8v4", "int8"])
def test_attention_matches_torch_sdpa(orc, fmt):
    """fp64 attention equals torch's scaled_dot_product_attention (float64, CPU)
    over the dequantised K and the un-rotated dequantised V, for several visible
    counts and all 16 query heads (GQA 8)."""
    import torch
    f = orc.FMT_K8V4 if fmt == "k8v4" else orc.FMT_INT8
    cache, pt, n = _small_cache(orc, f)
    kh, vr, vo = cache.dequant(pt, 0, n)
    Hs = scipy.linalg.hadamard(D).astype(np.float64)
    vhat = vr.astype(np.float64) @ Hs.T / 16.0 if fmt == "k8v4" else vr.astype(np.float64)
    rng = np.random.default_rng(12)
    q = rng.standard_normal((16, D)).astype(np.float32)
    for vis in (1, 2, 40, n):
        rs, rh, rv = orc.decode_rows(1, 16, [vis])
        got = cache.attention(pt, rs, rh, rv, q)
        for h in range(16):
            g = h // 8
            Q = torch.tensor(q[h], dtype=torch.float64)[None, None, None]
            K = torch.tensor(kh[:vis, g].astype(np.float64))[None, None]
            V = torch.tensor(vhat[:vis, g])[None, None]
            ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=1.0 / 16.0)[0, 0, 0].numpy()
            assert np.max(np.abs(got[h] - ref)) < 1e-12 * max(1.0, np.max(np.abs(ref)))


def _merge_partials(parts):
    """sum_r e^(m_r - M) o_r / sum_r e^(m_r - M) l_r over (o, m, l) triples, fp64."""
    M = np.max(np.stack([m for _, m, _ in parts]), axis=0)
    num = np.zeros_like(parts[0][0])
    den = np.zeros_like(parts[0][1])
    for o, m, l in parts:
        w = np.where(np.isneginf(m), 0.0, np.exp(np.where(np.isneginf(m), 0.0, m - M)))
        num += w[:, None] * o
        den += w * l
    return num / np.where(den > 0, den, 1.0)[:, None]


@pytest.mark.parametrize("fmt", ["k8v4", "int8"])
def test_attention_partial_merge_equals_full(orc, fmt):
    """The partial attention of a cell range (the cell-range split of one decode
    across GPUs) merges back to the full attention: for random partitions of the
    visible cells into ranges (empty ones included), the merge of the ranges'
    (o, m, l) equals the full fp64 attention, itself pinned to torch SDPA; a
    single range [0, n) gives o / l = attention and l >= 1; an empty range gives
    m = -inf, l = 0, o = 0."""
    f = orc.FMT_K8V4 if fmt == "k8v4" else orc.FMT_INT8
    cache, pt, n = _small_cache(orc, f, seed=21, n=93)
    rng = np.random.default_rng(22)
    q = rng.standard_normal((16, D)).astype(np.float32)
    rs, rh, rv = orc.decode_rows(1, 16, [n])
    full = cache.attention(pt, rs, rh, rv, q)
    for trial in range(6):
        cuts = np.sort(rng.integers(0, n + 1, size=rng.integers(1, 5)))
        bounds = [0, *cuts.tolist(), n]
        parts = []
        for lo, hi in zip(bounds[:-1], bounds[1:]):
            parts.append(cache.attention_partial(pt, rs, rh, np.full(16, lo), np.full(16, hi), q))
        got = _merge_partials(parts)
        assert np.max(np.abs(got - full)) < 1e-12 * max(1.0, np.max(np.abs(full)))
    o, m, l = cache.attention_partial(pt, rs, rh, np.zeros(16), np.full(16, n), q)
    assert np.max(np.abs(o / l[:, None] - full)) < 1e-12 * max(1.0, np.max(np.abs(full)))
    assert np.all(l >= 1.0)
    o, m, l = cache.attention_partial(pt, rs, rh, np.full(16, 50), np.full(16, 50), q)
    assert np.all(np.isneginf(m)) and np.all(l == 0.0) and np.all(o == 0.0)


def test_attention_closed_forms(orc):
    """One visible cell returns that cell's V; q = 0 returns the plain mean of the
    visible cells' V (equal scores)."""
    cache, pt, n = _small_cache(orc, orc.FMT_K8V4)
    kh, vr, vo = cache.dequant(pt, 0, n)
    Hs = scipy.linalg.hadamard(D).astype(np.float64)
    vhat = vr.astype(np.float64) @ Hs.T / 16.0
    rng = np.random.default_rng(13)
    q = rng.standard_normal((16, D)).astype(np.float32)
    rs, rh, rv = orc.decode_rows(1, 16, [1])
    one = cache.attention(pt, rs, rh, rv, q)
    for h in range(16):
        assert np.max(np.abs(one[h] - vhat[0, h // 8])) < 1e-12
    rs, rh, rv = orc.decode_rows(1, 16, [n])
    zero = cache.attention(pt, rs, rh, rv, np.zeros((16, D), np.float32))
    for h in range(16):
        assert np.max(np.abs(zero[h] - vhat[:n, h // 8].mean(0))) < 1e-12
    # V after the exact inverse rotation is close to the un-quantised V's scale
    assert np.all(np.isfinite(vo))


def test_attention_page_permutation_invariance(orc):
    """The same cells written through two different page tables give identical
    dequantised values and identical attention."""
    rng = np.random.default_rng(14)
    n, P, H = 50, 4, 2
    k = rng.standard_normal((1, n, H, D)).astype(np.float32)
    v = rng.standard_normal((1, n, H, D)).astype(np.float32)
    n_pages = (n + P - 1) // P
    outs = []
    for seed in (0, 1):
        pt = np.random.default_rng(seed).permutation(n_pages)[None].astype(np.int32)
        c = orc.Cache(n_pages, P, H)
        c.append(pt, np.array([0]), k, v)
        q = np.random.default_rng(99).standard_normal((16, D)).astype(np.float32)
        rs, rh, rv = orc.decode_rows(1, 16, [n])
        outs.append((c.dequant(pt, 0, n), c.attention(pt, rs, rh, rv, q), c.buf.copy()))
    for a, b in zip(outs[0][0], outs[1][0]):
        assert np.array_equal(a, b)
    assert np.array_equal(outs[0][1], outs[1][1])
    assert not np.array_equal(outs[0][2], outs[1][2])        # the bytes did move


def test_attention_modes_cross_check(orc):
    """Verify query i (sees len - 4 + i cells) equals decode at length len - 4 + i;
    a prefill row t (sees offset + t + 1) equals decode at that length; the
    rotated-space result brought back with (H/16) equals the default output."""
    cache, pt, n = _small_cache(orc, orc.FMT_K8V4, n=60)
    rng = np.random.default_rng(15)
    q = rng.standard_normal((5, 16, D)).astype(np.float32)
    steps = np.array([[n - 4 + i for i in range(5)]])
    rs, rh, rv = orc.multi_query_rows(steps, 16)
    ver = cache.attention(pt, rs, rh, rv, q.reshape(-1, D)).reshape(5, 16, D)
    for i in range(5):
        a, b, c = orc.decode_rows(1, 16, [n - 4 + i])
        dec = cache.attention(pt, a, b, c, q[i])
        assert np.array_equal(dec, ver[i])
    rot = cache.attention(pt, rs, rh, rv, q.reshape(-1, D), rotate_back=False)
    Hs = scipy.linalg.hadamard(D).astype(np.float64)
    assert np.max(np.abs(rot @ Hs.T / 16.0 - ver.reshape(-1, D))) < 1e-12


def test_negative_control_detects_corruption(orc):
    """Planted mistake (in the oracle's cache, on the CPU): one flipped V-scale byte
    changes the attention output well beyond the comparison tolerance."""
    cache, pt, n = _small_cache(orc, orc.FMT_K8V4, n=33)
    rng = np.random.default_rng(16)
    q = rng.standard_normal((16, D)).astype(np.float32)
    rs, rh, rv = orc.decode_rows(1, 16, [n])
    good = cache.attention(pt, rs, rh, rv, q)
    P, H = cache.P, cache.H
    page = int(pt[0, 1])
    vs = page * cache.page_bytes + 784 * P + (0 * H + 0) * 16 + 1
    cache.buf[vs] ^= 0x40
    bad = cache.attention(pt, rs, rh, rv, q)
    assert np.max(np.abs(bad - good)) > 1e-3


def test_tie_cells_round_trip(orc):
    """The generator's tie cells quantise to the hand-derived codes."""
    tk, tv = synth.tie_cells()
    c, s = orc.quant_int8(tk[0, 0, :128])
    assert s == 0.0625
    assert [int(t) for t in c[:11]] == [127, 2, -2, 126, 4, -4, 0, 2, 0, 126, -126]
    y = orc.rotate(tv[0, 0])
    nib, db = orc.quant_q4_block(y[:32])
    codes = np.concatenate([nib & 15, nib >> 4])
    assert codes[:9].tolist() == [0, 10, 12, 8, 15, 6, 8, 10, 0]


# ----------------------------------------------------------------------------- q4_0 K+V format

def _q4_runs(buf, page, P, H, slot, g):
    """Byte runs of (page, slot, head) in the q4_0 format, from the layout
    K nibbles [P][H][8][16], K scales f16 [P][H][8], V nibbles, V scales."""
    base = page * P * H * 288
    r = slot * H + g
    kq = buf[base + r * 128: base + r * 128 + 128]
    ks = buf[base + 128 * H * P + r * 16: base + 128 * H * P + r * 16 + 16]
    vq = buf[base + 144 * H * P + r * 128: base + 144 * H * P + r * 128 + 128]
    vs = buf[base + 272 * H * P + r * 16: base + 272 * H * P + r * 16 + 16]
    return kq, ks, vq, vs


def _q4_values(nib, scales):
    """(code - 8) * d of eight blocks: byte j holds codes j (low) and j + 16 (high)."""
    d = np.frombuffer(scales.tobytes(), np.float16).astype(np.float64)
    out = np.zeros(D)
    for b in range(8):
        for j in range(16):
            byte = int(nib[16 * b + j])
            out[32 * b + j] = ((byte & 15) - 8) * d[b]
            out[32 * b + j + 16] = ((byte >> 4) - 8) * d[b]
    return out


def test_q4_format_quantises_k_like_v(orc):
    """In the q4_0 format K goes through the same rotation + Q4_0 as V: equal K
    and V inputs give equal K and V runs, and those equal the V runs the k8v4
    format writes for the same vector."""
    rng = np.random.default_rng(31)
    P, H = 4, 2
    x = rng.standard_normal((1, 3, H, D)).astype(np.float32)
    x[..., 9] *= 20
    pt = np.array([[0]], np.int32)
    q4 = orc.Cache(1, P, H, orc.FMT_Q4)
    q4.append(pt, np.array([0]), x, x)
    k8 = orc.Cache(1, P, H, orc.FMT_K8V4)
    k8.append(pt, np.array([0]), x, x)
    for slot in range(3):
        for g in range(H):
            kq, ks, vq, vs = _q4_runs(q4.buf, 0, P, H, slot, g)
            assert np.array_equal(kq, vq) and np.array_equal(ks, vs)
            r = slot * H + g
            assert np.array_equal(vq, k8.buf[264 * H * P + r * 128: 264 * H * P + r * 128 + 128])
            assert np.array_equal(vs, k8.buf[392 * H * P + r * 16: 392 * H * P + r * 16 + 16])


def test_q4_format_dequant_and_attention(orc):
    """Dequantised K of the q4_0 format is the exact inverse rotation of its
    rotated-space values (decoded here from the raw bytes), and fp64 attention
    equals torch SDPA over K = (H/16) Khat_rot and V = (H/16) Vhat_rot formed
    in float64 from those bytes."""
    import torch
    cache, pt, n = _small_cache(orc, orc.FMT_Q4)
    kh, vr, vo = cache.dequant(pt, 0, n)
    Hs = scipy.linalg.hadamard(D).astype(np.float64)
    P, H = 8, 2
    krot = np.zeros((n, H, D))
    vrot = np.zeros((n, H, D))
    for c in range(n):
        for g in range(H):
            kq, ks, vq, vs = _q4_runs(cache.buf, int(pt[0, c // P]), P, H, c % P, g)
            krot[c, g] = _q4_values(kq, ks)
            vrot[c, g] = _q4_values(vq, vs)
    assert np.array_equal(vr.astype(np.float64), vrot)
    for c in (0, 5, n - 1):
        for g in range(H):
            assert np.array_equal(kh[c, g], orc.rotate(krot[c, g].astype(np.float32)))
    kd = krot @ Hs.T / 16.0
    vd = vrot @ Hs.T / 16.0
    rng = np.random.default_rng(14)
    q = rng.standard_normal((16, D)).astype(np.float32)
    for vis in (1, 33, n):
        rs, rh, rv = orc.decode_rows(1, 16, [vis])
        got = cache.attention(pt, rs, rh, rv, q)
        for h in range(16):
            g = h // 8
            Q = torch.tensor(q[h], dtype=torch.float64)[None, None, None]
            K = torch.tensor(kd[:vis, g])[None, None]
            V = torch.tensor(vd[:vis, g])[None, None]
            ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=1.0 / 16.0)[0, 0, 0].numpy()
            assert np.max(np.abs(got[h] - ref)) < 1e-11 * max(1.0, np.max(np.abs(ref)))


# ---------------------------------------------------------------- streaming block lookups
def test_stream_resolve_worked_example(orc):
    """A lookup worked by hand: P = 4, lengths 9 and 4 (three and one pages), host
    pages 5, 2, 7 | 2; pages 2 and 7 resident in slots 0 and 1, two staging slots.
    The one miss (page 5) goes to the first staging slot; page 2 is a hit for both
    sequences; entries no cell reaches stay -1."""
    pt = np.array([[5, 2, 7], [2, 0, 0]], np.int32)
    slot_of_page = np.full(8, -1, np.int32)
    slot_of_page[2], slot_of_page[7] = 0, 1
    dev, moves, over = orc.stream_resolve(pt, [9, 4], slot_of_page, 2, 4, 4, 12)
    assert dev.tolist() == [[2, 0, 1], [0, -1, -1]]
    assert moves == [(5, 2)]
    assert not over


def test_stream_resolve_extremes_and_overflow(orc):
    """Everything resident: the table is slot_of_page of the host table and
    nothing moves.  Nothing resident: every needed page moves, in lookup order,
    to consecutive staging slots.  One staging slot short: the last miss is not
    read and overflow is reported.  Lengths are clipped to max_seq_len."""
    rng = np.random.default_rng(3)
    P, n_host = 16, 40
    pt = rng.permutation(n_host)[:30].reshape(3, 10).astype(np.int32)
    lens = [160, 17, 0]
    need = [10, 2, 0]
    every = rng.permutation(n_host).astype(np.int32)
    dev, moves, over = orc.stream_resolve(pt, lens, every, n_host, n_host, P, 160)
    for b in range(3):
        assert dev[b, :need[b]].tolist() == [int(every[p]) for p in pt[b, :need[b]]]
        assert np.all(dev[b, need[b]:] == -1)
    assert moves == [] and not over
    none = np.full(n_host, -1, np.int32)
    dev, moves, over = orc.stream_resolve(pt, lens, none, 5, 5 + 12, P, 160)
    order = [int(p) for b in range(3) for p in pt[b, :need[b]]]
    assert moves == [(p, 5 + r) for r, p in enumerate(order)] and not over
    assert dev[0, :10].tolist() == list(range(5, 15)) and dev[1, :2].tolist() == [15, 16]
    dev, moves, over = orc.stream_resolve(pt, lens, none, 5, 5 + 11, P, 160)
    assert over and len(moves) == 11 and dev[1, 1] == -1
    dev, moves, over = orc.stream_resolve(pt, [1000, 17, 0], none, 0, 64, P, 48)
    assert dev[0, :3].tolist() == [0, 1, 2] and np.all(dev[0, 3:] == -1)


def test_stream_resolve_reads_the_right_bytes(orc):
    """Invariant on random tables: emulate VRAM (resident slots filled from the
    host copy, then the returned copies applied) and check that every cell a
    sequence reads through the returned table holds the bytes of the host page
    its own page table names, and that no copy overwrites a resident slot."""
    rng = np.random.default_rng(11)
    for trial in range(20):
        P = int(rng.choice([16, 64]))
        n_host, n_res = 50, int(rng.integers(0, 20))
        n_seqs, max_pages = int(rng.integers(1, 5)), 8
        pt = rng.integers(0, n_host, (n_seqs, max_pages)).astype(np.int32)
        lens = rng.integers(0, max_pages * P + 1, n_seqs)
        host = rng.integers(0, 256, (n_host, 4), dtype=np.uint8)
        slot_of_page = np.full(n_host, -1, np.int32)
        res_pages = rng.permutation(n_host)[:n_res]
        slot_of_page[res_pages] = rng.permutation(n_res)
        n_dev = n_res + n_seqs * max_pages
        dev_mem = np.zeros((n_dev, 4), np.uint8)
        for p in res_pages:
            dev_mem[slot_of_page[p]] = host[p]
        dev, moves, over = orc.stream_resolve(pt, lens, slot_of_page, n_res, n_dev, P, max_pages * P)
        assert not over
        for hp, slot in moves:
            assert slot >= n_res
            dev_mem[slot] = host[hp]
        for b in range(n_seqs):
            for i in range(max_pages):
                if i * P < lens[b]:
                    assert np.array_equal(dev_mem[dev[b, i]], host[pt[b, i]])
                else:
                    assert dev[b, i] == -1


@pytest.mark.parametrize("fmt", ["k8v4", "int8", "q4"])
def test_head_count_separability(orc, fmt):
    """A cache of 3 KV heads agrees head by head with three 1-head caches of the
    same rows (same page table, same bytes per head, same dequantised values),
    and its attention rows for query head h equal those of the 1-head cache of
    KV head h // 8: the (slot, head) interleaving and the GQA map hold for any
    head count."""
    f = {"k8v4": orc.FMT_K8V4, "int8": orc.FMT_INT8, "q4": orc.FMT_Q4}[fmt]
    rng = np.random.default_rng(21)
    n, P, H = 45, 8, 3
    n_pages = (n + P - 1) // P
    pt = rng.permutation(n_pages + 2)[:n_pages].astype(np.int32)[None]
    k = rng.standard_normal((1, n, H, D)).astype(np.float32)
    v = rng.standard_normal((1, n, H, D)).astype(np.float32)
    v[..., 5] *= 20
    big = orc.Cache(n_pages + 2, P, H, f)
    big.append(pt, np.array([0]), k, v)
    kb, vb, ob = big.dequant(pt, 0, n)
    q = rng.standard_normal((8 * H, D)).astype(np.float32)
    rs, rh, rv = orc.decode_rows(1, 8 * H, [n])
    att = big.attention(pt, rs, rh, rv, q)
    chb = orc.bytes_per_cell_head(f)
    for g in range(H):
        one = orc.Cache(n_pages + 2, P, 1, f)
        one.append(pt, np.array([0]), k[:, :, g:g + 1], v[:, :, g:g + 1])
        k1, v1, o1 = one.dequant(pt, 0, n)
        assert np.array_equal(k1[:, 0], kb[:, g]) and np.array_equal(v1[:, 0], vb[:, g])
        assert np.array_equal(o1[:, 0], ob[:, g])
        r1s, r1h, r1v = orc.decode_rows(1, 8, [n])
        att1 = one.attention(pt, r1s, r1h, r1v, q[8 * g:8 * g + 8])
        assert np.array_equal(att1, att[8 * g:8 * g + 8])
        # byte runs: every run of (cell, head g) in the big page equals the
        # 1-head page's run, at offsets scaled by H
        for c in (0, 9, n - 1):
            page = int(pt[0, c // P])
            pb_big, pb_one = P * H * chb, P * chb
            slot = c % P
            big_page = big.buf[page * pb_big:(page + 1) * pb_big]
            one_page = one.buf[page * pb_one:(page + 1) * pb_one]
            run_off, off1 = 0, 0
            for run in orc_runs(f):
                a = big_page[run_off * H * P + (slot * H + g) * run: run_off * H * P + (slot * H + g + 1) * run]
                b = one_page[off1 * P + slot * run: off1 * P + (slot + 1) * run]
                assert np.array_equal(a, b), (fmt, g, c, run)
                run_off += run
                off1 += run


def orc_runs(fmt_code):
    """Bytes per (cell, head) of each run of a format, in page order (K, K
    scales, V, V scales), from the layout the pages describe."""
    import oracle
    if fmt_code == oracle.FMT_K8V4:
        return (256, 8, 128, 16)
    if fmt_code == oracle.FMT_INT8:
        return (256, 8, 256, 8)
    return (128, 16, 128, 16)
