"""GPU parity of the append and dequant kernels: cache bytes must equal the
oracle's bit for bit (codes, scales, nibble order, page placement, untouched
canary pages), through non-identity page tables."""
import numpy as np
import pytest
import torch

import quantized_paged_kv_q8_gb300 as k8
import synth
from gpu_util import CANARY, append_both, dev_tensor, make_caches

pytestmark = pytest.mark.gpu


def _assert_bytes_equal(gpu, ref):
    got = gpu.pages.cpu().numpy()
    bad = np.nonzero(got != ref.buf)[0]
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[0]} (page {bad[0] // gpu.page_bytes})"


def test_append_tiny_fp32_roundtrip_bytes():
    """1,024 fp32 cells (hand-placed ties in cells 0-3), P = 16, 64 of 80 pages used:
    every byte equals the oracle's and the 16 canary pages keep 0xA5."""
    w = synth.config1()
    gpu, ref = make_caches(w.n_pages, w.page_size, w.n_kv)
    k = synth.Tensor(w.k.f32[None], "f32")
    v = synth.Tensor(w.v.f32[None], "f32")
    append_both(gpu, ref, w.page_table, w.pos, k, v)
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    _assert_bytes_equal(gpu, ref)
    used = set(int(p) for p in w.page_table.reshape(-1))
    pages = gpu.pages.cpu().numpy().reshape(w.n_pages, -1)
    for p in range(w.n_pages):
        if p not in used:
            assert np.all(pages[p] == CANARY)


@pytest.mark.parametrize("fmt", [k8.FORMAT_K8V4, k8.FORMAT_Q4])
def test_append_bf16_32k_bytes(fmt):
    w = synth.config2()
    gpu, ref = make_caches(w.n_pages, w.page_size, w.n_kv, fmt)
    k = synth.Tensor(w.k.f32[None], "bf16")
    v = synth.Tensor(w.v.f32[None], "bf16")
    append_both(gpu, ref, w.page_table, w.pos, k, v)
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    _assert_bytes_equal(gpu, ref)


@pytest.mark.parametrize("fmt", [k8.FORMAT_K8V4, k8.FORMAT_INT8, k8.FORMAT_Q4])
def test_append_shared_pool_chunks(fmt):
    """Three sequences in one interleaved pool, written in two appends (a history
    then a chunk at its offset), ragged lengths, every format."""
    seed = synth.config_seed(4) + 17
    lens = np.array([700, 1333, 64], np.int32)
    P = 64
    pt, n_pages = synth.interleaved_pool(seed, lens + 40, P)
    gpu, ref = make_caches(n_pages + 3, P, 2, fmt)
    hist = 37
    for b in range(3):
        k = synth.kv_values(seed, synth.T_K, b, int(lens[b]), 2, 3, "bf16")
        v = synth.kv_values(seed, synth.T_V, b, int(lens[b]), 2, 3, "bf16")
        row = pt[b:b + 1]
        for lo, hi in ((0, hist), (hist, int(lens[b]))):
            kk = synth.Tensor(k.f32[None, lo:hi], "bf16")
            vv = synth.Tensor(v.f32[None, lo:hi], "bf16")
            append_both(gpu, ref, row, np.array([lo]), kk, vv)
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    _assert_bytes_equal(gpu, ref)


@pytest.mark.parametrize("fmt", [k8.FORMAT_K8V4, k8.FORMAT_Q4])
def test_append_exact_rotation_wide_exponents(fmt):
    """fp32 V rows whose values span far more than 2^55 (the rotation's slow path),
    subnormals, all-zero rows, and rows with one huge value: bytes still equal
    (in the Q4 format the K rows take the rotation too)."""
    rng = np.random.default_rng(123)
    n, P = 64, 16
    k = rng.standard_normal((1, n, 2, 256)).astype(np.float32)
    v = rng.standard_normal((1, n, 2, 256)).astype(np.float32)
    v[0, 0, 0] *= 1e30
    v[0, 1, 1, :] = (rng.standard_normal(256) * 10.0 ** rng.integers(-35, 35, 256)).astype(np.float32)
    v[0, 2, 0, :] = 0.0
    v[0, 3, 1, :] = (rng.standard_normal(256) * 1e-40).astype(np.float32)
    v[0, 4, 0, :] = 0.0
    v[0, 4, 0, 17] = 3e-45
    k[0, 5, 0, :128] = 0.0
    k[0, 6, 1, :] = (rng.standard_normal(256) * 1e-38).astype(np.float32)
    v[0, 7, 0, ::3] *= 2.0 ** 60
    k[0, 8, 0, :] = (rng.standard_normal(256) * 10.0 ** rng.integers(-35, 35, 256)).astype(np.float32)
    k[0, 9, 1, ::5] *= 2.0 ** 70
    pt = np.random.default_rng(5).permutation(n // P)[None].astype(np.int32)
    gpu, ref = make_caches(n // P, P, 2, fmt)
    append_both(gpu, ref, pt, np.array([0]), synth.Tensor(k, "f32"), synth.Tensor(v, "f32"))
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    _assert_bytes_equal(gpu, ref)


@pytest.mark.parametrize("fmt", [k8.FORMAT_K8V4, k8.FORMAT_INT8, k8.FORMAT_Q4])
def test_dequant_matches_oracle(fmt):
    """kv_dequant_k8v4: Khat = c*s (Q4: the exact inverse rotation of the stored
    K), Vhat_rot = (q-8)*d and the exact inverse rotation equal the oracle's
    dequantisation bit for bit."""
    w = synth.config1()
    gpu, ref = make_caches(w.n_pages, w.page_size, w.n_kv, fmt)
    pt_d = append_both(gpu, ref, w.page_table, w.pos, synth.Tensor(w.k.f32[None], "f32"),
                       synth.Tensor(w.v.f32[None], "f32"))
    start, n = 5, 1000
    ko = torch.empty(n, 2, 256, device="cuda")
    vr = torch.empty_like(ko)
    vo = torch.empty_like(ko)
    k8.kv_dequant_k8v4(gpu, pt_d, start, n, ko, vr, vo)
    torch.cuda.synchronize()
    rk, rvr, rvo = ref.dequant(w.page_table, start, n)
    assert np.array_equal(ko.cpu().numpy().view(np.uint32), rk.view(np.uint32))
    assert np.array_equal(vr.cpu().numpy().view(np.uint32), rvr.view(np.uint32))
    assert np.array_equal(vo.cpu().numpy().view(np.uint32), rvo.view(np.uint32))


def test_append_out_of_range_page_is_skipped_and_reported():
    """A page-table entry outside [0, n_pages) is never written through: the cells
    that map to it are skipped, K8V4_ERANGE is recorded, everything else is
    written exactly, and the device stays usable."""
    n, P = 96, 16
    rng = np.random.default_rng(9)
    k = synth.Tensor(rng.standard_normal((1, n, 2, 256)).astype(np.float32), "f32")
    v = synth.Tensor(rng.standard_normal((1, n, 2, 256)).astype(np.float32), "f32")
    gpu, ref = make_caches(8, P)
    pt = np.array([[3, 1, 99, 0, 5, 7]], np.int32)        # page index 2 -> id 99 (bad)
    pt_d = torch.from_numpy(pt).cuda()
    k8.kv_append_k8v4(gpu, pt_d, torch.zeros(1, dtype=torch.int64, device="cuda"), dev_tensor(k), dev_tensor(v))
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == k8.ERANGE
    assert k8.k8v4_last_device_status() == 0              # read-and-clear
    pt_ok = np.array([[3, 1, 2, 0, 5, 7]], np.int32)     # index 2 is never used below
    ref.append(pt_ok, np.array([0]), k.f32[:, :32], v.f32[:, :32])
    ref.append(pt_ok, np.array([48]), k.f32[:, 48:], v.f32[:, 48:])
    _assert_bytes_equal(gpu, ref)


@pytest.mark.parametrize("fmt", [k8.FORMAT_K8V4, k8.FORMAT_Q4])
def test_append_rotation_fixed_point_edges(fmt):
    """Rows whose values span exactly 23 and 24 bits in fixed point (sums
    reaching 255 x (2^24 - 1) + 1), same-sign, negated and alternating-sign,
    plus rows of 8-bit mantissas over 16 binades with one huge value: the exact
    rotation's integer butterflies and its final rounding give the oracle's
    bytes."""
    n, P = 32, 16
    rng = np.random.default_rng(77)
    k = rng.standard_normal((1, n, 2, 256)).astype(np.float32)
    v = rng.standard_normal((1, n, 2, 256)).astype(np.float32)
    big23, big24 = float(2 ** 23 - 1), float(2 ** 24 - 1)
    rows = []
    for big in (big23, big24):
        r = np.full(256, big, np.float32); r[5] = 1.0; rows.append(r)                 # all positive
        rows.append(-rows[-1])                                                          # all negative
        r = np.full(256, big, np.float32); r[1::2] *= -1; r[7] = 1.0; rows.append(r)  # alternating
        r = (rng.integers(1, 2 ** 8, 256) * 2.0 ** rng.integers(0, 16, 256)).astype(np.float32)
        r[3] = 1.0; r[4] = big; rows.append(r)                                          # mixed exponents
    for i, r in enumerate(rows):
        v[0, i, i % 2] = r
        k[0, 16 + i, i % 2] = r
    pt = np.random.default_rng(6).permutation(n // P)[None].astype(np.int32)
    gpu, ref = make_caches(n // P, P, 2, fmt)
    append_both(gpu, ref, pt, np.array([0]), synth.Tensor(k, "f32"), synth.Tensor(v, "f32"))
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    _assert_bytes_equal(gpu, ref)


def _sylvester():
    i = np.arange(256)
    return np.where(np.vectorize(lambda a: bin(a).count("1") & 1)(i[:, None] & i[None, :]), -1.0, 1.0)


def _from_rotated(y: np.ndarray) -> np.ndarray:
    """The row x whose exact rotation H x / 16 is y (H H = 256 I); x must be
    exactly representable in bf16."""
    x = _sylvester() @ np.asarray(y, np.float64) / 16.0
    xb = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(x.astype(np.float32))).astype(np.float64)
    assert np.array_equal(xb, x), "crafted row is not exact in bf16"
    return x.astype(np.float32)


def _rotation_edge_rows(rng) -> list[np.ndarray]:
    """bf16 rows at the edges of the append's int32 rotation path and of its
    q4_0 quantiser: L1 norms just inside and just outside 2^30 units of the
    smallest element's last bit, wide exponent spans, the smallest admitted
    exponent and its neighbour, huge values, exact zeros, subnormals, +/- ties
    for a block's largest magnitude in either order, fp16 scales that are
    subnormal (codes clamped at 0 and 15), zero or infinite, and quotients
    exactly halfway between codes."""
    rows = []
    mant = lambda n: (rng.integers(128, 256, n) / 128.0) * rng.choice([-1.0, 1.0], n)
    for big in (32.0, 32.25):                            # L1 * 2^17 = 1.0696e9 / 1.0779e9 vs 2^30
        r = np.full(256, big); r[1::2] *= -1; r[200] = 2.0 ** -10
        rows.append(r)
    for e in (-115, -116):                                # smallest element's exponent field 12 / 11
        r = mant(256) * 2.0 ** (e + rng.integers(0, 8, 256))
        r[17] = 2.0 ** e
        rows.append(r)
    mant = lambda n: (rng.integers(128, 256, n) / 128.0) * rng.choice([-1.0, 1.0], n)
    for span in (14, 15):
        r = mant(256) * 2.0 ** rng.integers(-4, 3, 256)
        r[0] = 255 / 128 * 8.0
        r[1] = -255 / 128 * 2.0 ** (3 - span)
        rows.append(r)
    for e in (-101, -102, 73, 74, 75, 80):               # huge and tiny rows; 80: smallest field 202
        r = mant(256) * 2.0 ** (e - rng.integers(0, 6, 256))
        r[9] = 1.5 * 2.0 ** e
        rows.append(r)
    r = mant(256); r[77] = 0.0; rows.append(r)           # one exact zero
    r = mant(256); r[3] = 2.0 ** -130; rows.append(r)    # one subnormal
    rows.append(np.zeros(256))
    rows.append(mant(256) * 2.0 ** -126)                 # all at the smallest normal binade
    # rotated-domain rows: y sparse, x = H y / 16 exact and without zeros
    for j1, j2 in ((3, 20), (20, 3), (17, 2), (0, 31)):
        y = np.zeros(256); y[j1] = 1.0; y[j2] = -1.0; y[200] = 4.0
        rows.append(_from_rotated(y))
    # block 1's largest is 11 u: its fp16 scale -11 u / 8 is subnormal and rounds to
    # -u (codes -11 + 8 and 10 + 8 clamp to 0 and 15), flushes to zero, or overflows;
    # every signed sum of 11, 10, 3, 1 is odd, so x has no zeros
    for u in (2.0 ** -24, 2.0 ** -30, 2.0 ** 17):
        y = np.zeros(256); y[40] = 11 * u; y[41] = -10 * u; y[42] = 3 * u; y[230] = u
        rows.append(_from_rotated(y))
    y = np.zeros(256); y[64:68] = (-8.0, 2.5, 3.5, -1.5); y[100] = 0.25; y[101] = 0.5
    rows.append(_from_rotated(y))                        # q = y / 1 exactly k + 1/2
    return [np.asarray(r, np.float32) for r in rows]


def _int8_edge_rows(rng) -> list[np.ndarray]:
    """bf16 rows at the edges of the int8 quantiser's fast path: quotients that
    are exact half-integers (scale 1), a zero half, a tiny scale below 2^-125
    (the general quantiser), and halves whose largest magnitude sits in either
    lane group."""
    rows = []
    r = np.zeros(256); r[0] = 127.0; r[1:6] = (2.5, -3.5, 0.5, -0.5, 126.5); r[128] = -127.0; r[129:131] = (1.5, -2.5)
    rows.append(r)
    r = rng.standard_normal(256); r[:128] = 0.0; rows.append(r)
    r = rng.standard_normal(256) * 2.0 ** -120; rows.append(r)
    r = rng.standard_normal(256); r[127] = 40.0; r[255] = -40.0; rows.append(r)
    return [synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(np.asarray(r, np.float32))) for r in rows]


@pytest.mark.parametrize("fmt", [k8.FORMAT_K8V4, k8.FORMAT_INT8, k8.FORMAT_Q4])
def test_append_bf16_fast_path_edges(fmt):
    """A long bf16 append (the persistent bulk kernel) whose rows include every
    edge of its int32 rotation and rounding shortcuts: bytes equal the oracle's
    (rows that leave a shortcut take the general exact path)."""
    rng = np.random.default_rng(2024)
    n, P = 1024, 16
    k = rng.standard_normal((1, n, 2, 256)).astype(np.float32)
    v = rng.standard_normal((1, n, 2, 256)).astype(np.float32)
    rot, i8 = _rotation_edge_rows(rng), _int8_edge_rows(rng)
    rot_dst, i8_dst = (k if fmt == k8.FORMAT_Q4 else v), (v if fmt == k8.FORMAT_INT8 else k)
    for i, r in enumerate(rot):
        rot_dst[0, 100 + 7 * i, i % 2] = r
        if fmt == k8.FORMAT_K8V4:
            v[0, 600 + 5 * i, (i + 1) % 2] = -r
    for i, r in enumerate(i8):
        i8_dst[0, 300 + 11 * i, i % 2] = r
    pt = np.random.default_rng(8).permutation(n // P)[None].astype(np.int32)
    gpu, ref = make_caches(n // P, P, 2, fmt)
    append_both(gpu, ref, pt, np.array([0]), synth.Tensor(k, "bf16"), synth.Tensor(v, "bf16"))
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    _assert_bytes_equal(gpu, ref)


def test_append_bf16_bulk_bad_page_is_skipped_and_reported():
    """The persistent bf16 kernel (a long append) over a page table with one bad
    id: the cells of that page are skipped and K8V4_ERANGE is recorded; every
    other cell's bytes equal the oracle's, including cells after the bad page."""
    n, P = 1024, 64
    rng = np.random.default_rng(31)
    k = synth.Tensor(rng.standard_normal((1, n, 2, 256)).astype(np.float32), "bf16")
    v = synth.Tensor(rng.standard_normal((1, n, 2, 256)).astype(np.float32), "bf16")
    n_pages = n // P
    perm = np.random.default_rng(32).permutation(n_pages).astype(np.int32)
    pt = perm.copy()[None]
    pt[0, 5] = n_pages + 7                                  # page index 5 -> a bad id
    gpu, ref = make_caches(n_pages, P)
    pt_d = torch.from_numpy(pt).cuda()
    k8.kv_append_k8v4(gpu, pt_d, torch.zeros(1, dtype=torch.int64, device="cuda"), dev_tensor(k), dev_tensor(v))
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == k8.ERANGE
    assert k8.k8v4_last_device_status() == 0
    ok = perm[None].copy()
    ref.append(ok, np.array([0]), k.f32[:, :5 * P], v.f32[:, :5 * P])
    ref.append(ok, np.array([6 * P]), k.f32[:, 6 * P:], v.f32[:, 6 * P:])
    got = gpu.pages.cpu().numpy()
    # the page the bad entry would have used stays a canary
    assert np.all(got.reshape(n_pages, -1)[perm[5]] == CANARY)
    mask = np.ones(n_pages, bool)
    mask[perm[5]] = False
    assert np.array_equal(got.reshape(n_pages, -1)[mask], ref.buf.reshape(n_pages, -1)[mask])
