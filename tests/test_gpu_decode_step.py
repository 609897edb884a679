"""The fused decode step (attn_k8v4_decode_step): appending each sequence's
newest token inside the decode grid must write the same cache bytes and give the
same output as kv_append_k8v4 followed by attn_k8v4_decode, and match the fp64
oracle on the full cache."""
import numpy as np
import pytest
import torch

import oracle
import quantized_paged_kv_q8_gb300 as k8
import synth
from gpu_util import TOL, dev_tensor, make_caches, rel_err

pytestmark = pytest.mark.gpu


def _setup(fmt, kvdt, lens, P=64, seed_off=0):
    seed = synth.config_seed(3) + 500 + seed_off
    H = 2
    lens = np.asarray(lens, np.int32)
    pt, n_pages = synth.interleaved_pool(seed, np.maximum(lens, 1), P)
    ks = [synth.kv_values(seed, synth.T_K, b, max(int(n), 1), H, 3, kvdt) for b, n in enumerate(lens)]
    vs = [synth.kv_values(seed, synth.T_V, b, max(int(n), 1), H, 3, kvdt) for b, n in enumerate(lens)]
    q = synth.q_values(seed, 0, len(lens), H, "bf16")
    # two GPU caches holding cells 0 .. len-2, the oracle holding all len cells
    gpu_a, ref = make_caches(n_pages, P, H, fmt)
    gpu_b, _ = make_caches(n_pages, P, H, fmt)
    for b, n in enumerate(lens):
        if n > 1:
            for g in (gpu_a, gpu_b):
                k8.kv_append_k8v4(g, torch.from_numpy(pt[b:b + 1]).cuda(), torch.zeros(1, dtype=torch.int64).cuda(),
                                  dev_tensor(synth.Tensor(ks[b].f32[None, :n - 1], kvdt)),
                                  dev_tensor(synth.Tensor(vs[b].f32[None, :n - 1], kvdt)))
        if n > 0:
            ref.append(pt[b:b + 1], np.array([0]), ks[b].f32[None, :n], vs[b].f32[None, :n])
    # the new token of each sequence (a zero row where the sequence stays empty)
    k_new = np.stack([ks[b].f32[max(int(n), 1) - 1] for b, n in enumerate(lens)])
    v_new = np.stack([vs[b].f32[max(int(n), 1) - 1] for b, n in enumerate(lens)])
    return pt, lens, q, gpu_a, gpu_b, ref, synth.Tensor(k_new, kvdt), synth.Tensor(v_new, kvdt)


@pytest.mark.parametrize("fmt,kvdt,P", [(k8.FORMAT_K8V4, "bf16", 64), (k8.FORMAT_K8V4, "f32", 64),
                                          (k8.FORMAT_INT8, "bf16", 64), (k8.FORMAT_INT8, "f32", 64),
                                          (k8.FORMAT_K8V4, "bf16", 16), (k8.FORMAT_K8V4, "bf16", 256),
                                          (k8.FORMAT_Q4, "bf16", 64), (k8.FORMAT_Q4, "f32", 16)])
def test_decode_step_equals_append_then_decode(fmt, kvdt, P):
    lens = [1, 17, 64, 1000, 5000, 0, 4097]
    pt, lens, q, gpu_a, gpu_b, ref, k_new, v_new = _setup(fmt, kvdt, lens, P=P)
    n = len(lens)
    max_len = int(lens.max())
    pt_d = torch.from_numpy(pt).cuda()
    lens_d = torch.from_numpy(lens).cuda()
    qd = dev_tensor(q, (n, 16, 256))
    kd, vd = dev_tensor(k_new, (n, 2, 256)), dev_tensor(v_new, (n, 2, 256))
    # A: the two calls (sequences with a token only)
    has = lens > 0
    pos = torch.from_numpy(np.maximum(lens - 1, 0).astype(np.int64)).cuda()
    for b in np.nonzero(has)[0]:
        k8.kv_append_k8v4(gpu_a, pt_d[b:b + 1], pos[b:b + 1], kd[b:b + 1, None].contiguous(),
                          vd[b:b + 1, None].contiguous())
    out_a = torch.empty(n, 16, 256, dtype=torch.float32, device="cuda")
    ws = k8.workspace(gpu_a, n, 1, max_len)
    k8.attn_k8v4_decode(gpu_a, qd, pt_d, lens_d, max_len, out_a, ws)
    # B: the fused step
    out_b = torch.empty(n, 16, 256, dtype=torch.float32, device="cuda")
    k8.attn_k8v4_decode_step(gpu_b, qd, kd, vd, pt_d, lens_d, max_len, out_b, ws)
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    assert torch.equal(gpu_a.pages, gpu_b.pages)                 # same bytes written
    assert np.array_equal(gpu_b.pages.cpu().numpy(), ref.buf)    # and they are the oracle's
    assert torch.equal(out_a, out_b)                             # same arithmetic
    got = out_b.cpu().numpy()
    assert np.all(got[~has] == 0.0)
    rs, rh, rv = oracle.decode_rows(n, 16, lens)
    want = ref.attention(pt, rs, rh, rv, q.f32.reshape(-1, 256))
    assert rel_err(got.reshape(-1, 256), want) <= TOL


def test_decode_step_bad_page_is_reported():
    """The newest cell's page id out of range: recorded, the token not written,
    the other sequences unaffected."""
    pt, lens, q, gpu_a, gpu_b, ref, k_new, v_new = _setup(k8.FORMAT_K8V4, "bf16", [300, 700], seed_off=1)
    bad = pt.copy()
    bad[0, (300 - 1) // 64] = 10 ** 6                  # page of sequence 0's newest cell
    before = gpu_b.pages.clone()
    out = torch.empty(2, 16, 256, dtype=torch.float32, device="cuda")
    ws = k8.workspace(gpu_b, 2, 1, 700)
    k8.attn_k8v4_decode_step(gpu_b, dev_tensor(q, (2, 16, 256)), dev_tensor(k_new, (2, 2, 256)),
                             dev_tensor(v_new, (2, 2, 256)), torch.from_numpy(bad).cuda(),
                             torch.from_numpy(lens).cuda(), 700, out, ws)
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == k8.ERANGE
    # sequence 1's token was written, sequence 0's page stayed as it was
    changed = np.nonzero(gpu_b.pages.cpu().numpy() != before.cpu().numpy())[0]
    page_bytes = 64 * 816
    assert len(changed) > 0 and set((changed // page_bytes).tolist()) == {int(pt[1, (700 - 1) // 64])}


def test_decode_step_config3_full():
    """The bench's step at full size: 237,567 cells in the cache, the step appends
    cell 237,567 and attends over all 237,568; every row against the oracle and
    the cache bytes equal to the oracle's."""
    n = 237568
    w = synth.config3(n, seed=synth.config_seed(3))
    gpu, ref = make_caches(w.n_pages, w.page_size, w.n_kv)
    pt_d = torch.from_numpy(w.page_table).cuda()
    k8.kv_append_k8v4(gpu, pt_d, torch.zeros(1, dtype=torch.int64).cuda(),
                      dev_tensor(synth.Tensor(w.k.f32[None, :n - 1], "bf16")),
                      dev_tensor(synth.Tensor(w.v.f32[None, :n - 1], "bf16")))
    ref.append(w.page_table, w.pos, w.k.f32[None], w.v.f32[None])
    out = torch.empty(1, 16, 256, dtype=torch.float32, device="cuda")
    ws = k8.workspace(gpu, 1, 1, n)
    k_new = dev_tensor(synth.Tensor(w.k.f32[n - 1:], "bf16"), (1, 2, 256))
    v_new = dev_tensor(synth.Tensor(w.v.f32[n - 1:], "bf16"), (1, 2, 256))
    k8.attn_k8v4_decode_step(gpu, dev_tensor(w.q, (1, 16, 256)), k_new, v_new, pt_d,
                             torch.from_numpy(w.seq_lens).cuda(), n, out, ws)
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    assert np.array_equal(gpu.pages.cpu().numpy(), ref.buf)
    rs, rh, rv = oracle.decode_rows(1, 16, w.seq_lens)
    want = ref.attention(w.page_table, rs, rh, rv, w.q.f32.reshape(-1, 256))
    assert rel_err(out.cpu().numpy().reshape(-1, 256), want) <= TOL


def test_decode_step_many_sequences():
    """The engine's batched shape at scale: 40 sequences of seeded ragged lengths
    (80 (sequence, KV head) pairs, more than half the SMs, so the split plan
    trades ranges per pair against waves), pages interleaved in one pool.  The
    fused step appends every newest token and attends; cache bytes and every
    row against the oracle."""
    rng = np.random.default_rng(synth.config_seed(3) + 777)
    lens = rng.integers(700, 6000, size=40).astype(np.int32)
    lens[3] = 1
    lens[11] = 64
    pt, lens, q, _, gpu_b, ref, k_new, v_new = _setup(k8.FORMAT_K8V4, "bf16", lens, seed_off=7)
    n = len(lens)
    max_len = int(lens.max())
    pt_d = torch.from_numpy(pt).cuda()
    out = torch.empty(n, 16, 256, dtype=torch.float32, device="cuda")
    ws = k8.workspace(gpu_b, n, 1, max_len)
    k8.attn_k8v4_decode_step(gpu_b, dev_tensor(q, (n, 16, 256)), dev_tensor(k_new, (n, 2, 256)),
                             dev_tensor(v_new, (n, 2, 256)), pt_d, torch.from_numpy(lens).cuda(), max_len, out, ws)
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    assert np.array_equal(gpu_b.pages.cpu().numpy(), ref.buf)
    rs, rh, rv = oracle.decode_rows(n, 16, lens)
    want = ref.attention(pt, rs, rh, rv, q.f32.reshape(-1, 256))
    assert rel_err(out.cpu().numpy().reshape(-1, 256), want) <= TOL


@pytest.mark.parametrize("fmt,kvdt", [(k8.FORMAT_K8V4, "bf16"), (k8.FORMAT_INT8, "bf16"), (k8.FORMAT_Q4, "f32")])
def test_decode_step_host_buffers_equal_device_buffers(fmt, kvdt):
    """q, the new rows and the output may live in page-locked host memory: the
    kernels read and write them over the host link.  Same cache bytes and the
    same output, bit for bit, as with device buffers, for the fused step and the
    plain decode."""
    lens = [1, 17, 1000, 5000, 0, 4097]
    pt, lens, q, gpu_a, gpu_b, ref, k_new, v_new = _setup(fmt, kvdt, lens, seed_off=7)
    n = len(lens)
    max_len = int(lens.max())
    pt_d = torch.from_numpy(pt).cuda()
    lens_d = torch.from_numpy(lens).cuda()
    qd = dev_tensor(q, (n, 16, 256))
    kd, vd = dev_tensor(k_new, (n, 2, 256)), dev_tensor(v_new, (n, 2, 256))
    qh, kh, vh = qd.cpu().pin_memory(), kd.cpu().pin_memory(), vd.cpu().pin_memory()
    ws = k8.workspace(gpu_a, n, 1, max_len)
    out_d = torch.empty(n, 16, 256, dtype=torch.float32, device="cuda")
    out_h = torch.full((n, 16, 256), float("nan"), dtype=torch.float32).pin_memory()
    k8.attn_k8v4_decode_step(gpu_a, qd, kd, vd, pt_d, lens_d, max_len, out_d, ws)
    k8.attn_k8v4_decode_step(gpu_b, qh, kh, vh, pt_d, lens_d, max_len, out_h, ws)
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    assert torch.equal(gpu_a.pages, gpu_b.pages)
    assert np.array_equal(gpu_b.pages.cpu().numpy(), ref.buf)
    assert torch.equal(out_d.cpu(), out_h)
    rs, rh, rv = oracle.decode_rows(n, 16, lens)
    want = ref.attention(pt, rs, rh, rv, q.f32.reshape(-1, 256))
    assert rel_err(out_h.numpy().reshape(-1, 256), want) <= TOL
    out_h.fill_(float("nan"))
    k8.attn_k8v4_decode(gpu_b, qh, pt_d, lens_d, max_len, out_h, ws)
    k8.attn_k8v4_decode(gpu_b, qd, pt_d, lens_d, max_len, out_d, ws)
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    assert torch.equal(out_d.cpu(), out_h)
