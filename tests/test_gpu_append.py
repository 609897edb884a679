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
