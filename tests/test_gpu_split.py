"""The cell-range split of one decode across GPUs, device side, on one GPU:
attn_k8v4_decode_partial over each rank's range of cell_ranges(), then
attn_k8v4_combine_partials over the stacked partials, equals the oracle's full
attention (and the single-call decode) within the suite's bar; each range's
partial matches the oracle's partial over the same cells."""
import math

import numpy as np
import pytest
import torch

import oracle
import quantized_paged_kv_q8_gb300 as k8
import synth
from gpu_util import TOL, append_both, decode_gpu, dev_tensor, make_caches, rel_err

pytestmark = pytest.mark.gpu


def _split_decode(gpu, q_d, pt_d, lens_d, max_len, world):
    n, rows = q_d.shape[0], q_d.shape[1]
    parts = torch.empty(world, n, rows, k8.PARTIAL_ROW, device="cuda")
    for r, (lo, hi) in enumerate(k8.cell_ranges(max_len, world)):
        ws = k8.partial_workspace(gpu, n, lo, hi)
        k8.attn_k8v4_decode_partial(gpu, q_d, pt_d, lens_d, max_len, lo, hi, parts[r], ws)
    out = torch.empty(n, rows, 256, device="cuda")
    k8.attn_k8v4_combine_partials(parts, out)
    torch.cuda.synchronize()
    return parts, out


@pytest.mark.parametrize("fmt", [k8.FORMAT_K8V4, k8.FORMAT_INT8])
def test_split_decode_ragged(fmt):
    """Sequences of 1, 17, 1,000, 4,097 and 5,000 cells over one 5,000-cell
    cache, split 2 and 3 ways (short sequences leave later ranges empty)."""
    w = synth.decode_workload(synth.config_seed(2) + 41, 5000, P=64)
    gpu, ref = make_caches(w.n_pages, w.page_size, w.n_kv, fmt)
    append_both(gpu, ref, w.page_table, w.pos, synth.Tensor(w.k.f32[None], "bf16"),
                synth.Tensor(w.v.f32[None], "bf16"))
    lens = np.array([1, 17, 1000, 4097, 5000], np.int32)
    n = len(lens)
    pt = np.repeat(w.page_table, n, axis=0)
    pt_d, lens_d = torch.from_numpy(pt).cuda(), torch.from_numpy(lens).cuda()
    q = synth.q_values(w.seed, 5, n, 2, "bf16")
    q_d = dev_tensor(q, (n, 16, 256))
    rs, rh, rv = oracle.decode_rows(n, 16, lens)
    want = ref.attention(pt, rs, rh, rv, q.f32.reshape(-1, 256))
    one = decode_gpu(gpu, q_d, pt_d, lens, 5000)
    for world in (2, 3):
        parts, out = _split_decode(gpu, q_d, pt_d, lens_d, 5000, world)
        got = out.cpu().numpy()
        assert rel_err(got.reshape(-1, 256), want) <= TOL, world
        assert rel_err(got, one) <= TOL, world
        # each range's partial against the oracle's partial over the same cells
        for r, (lo, hi) in enumerate(k8.cell_ranges(5000, world)):
            p = parts[r].cpu().numpy().reshape(-1, 260).astype(np.float64)
            o, m, l = ref.attention_partial(pt, rs, rh, np.full(rs.shape, lo), np.minimum(rv, hi), q.f32.reshape(-1, 256))
            empty = np.isneginf(m)
            assert np.all(np.isneginf(p[empty, 256])) and np.all(p[empty, 257] == 0.0)
            ok = ~empty
            assert rel_err(p[ok, :256] / p[ok, 257:258], o[ok] / l[ok, None]) <= TOL
            # the same total weight: l 2^m (base 2) against l e^m
            lhs = np.log(p[ok, 257]) + p[ok, 256] * math.log(2.0)
            rhs = np.log(l[ok]) + m[ok]
            assert np.max(np.abs(lhs - rhs)) < 1e-5
    assert k8.k8v4_last_device_status() == 0


def test_split_decode_238k_two_ranks():
    """The 237,568-cell workload split over two ranks (118,784 cells each)."""
    w = synth.config3(237568, seed=synth.config_seed(3))
    gpu, ref = make_caches(w.n_pages, w.page_size, w.n_kv)
    pt_d = append_both(gpu, ref, w.page_table, w.pos, synth.Tensor(w.k.f32[None], w.dtype),
                       synth.Tensor(w.v.f32[None], w.dtype))
    q_d = dev_tensor(w.q, (1, 16, 256))
    lens_d = torch.from_numpy(np.asarray(w.seq_lens, np.int32)).cuda()
    _, out = _split_decode(gpu, q_d, pt_d, lens_d, 237568, 2)
    rs, rh, rv = oracle.decode_rows(1, 16, w.seq_lens)
    want = ref.attention(w.page_table, rs, rh, rv, w.q.f32.reshape(-1, 256))
    assert rel_err(out.cpu().numpy().reshape(-1, 256), want) <= TOL
    assert k8.k8v4_last_device_status() == 0


def test_split_decode_rejects_bad_ranges():
    w = synth.decode_workload(synth.config_seed(2) + 42, 256, P=64)
    gpu, _ = make_caches(w.n_pages, w.page_size, w.n_kv)
    q = torch.zeros(1, 16, 256, dtype=torch.bfloat16, device="cuda")
    pt_d = torch.from_numpy(w.page_table).cuda()
    lens = torch.full((1,), 256, dtype=torch.int32, device="cuda")
    part = torch.empty(1, 16, 260, device="cuda")
    ws = k8.partial_workspace(gpu, 1, 0, 256)
    for lo, hi in ((8, 256), (0, 100), (64, 32)):
        with pytest.raises(k8.K8V4Error) as e:
            k8.attn_k8v4_decode_partial(gpu, q, pt_d, lens, 256, lo, hi, part, ws)
        assert e.value.code == k8.EINVAL
    q4, _ = make_caches(w.n_pages, w.page_size, w.n_kv, k8.FORMAT_Q4)
    with pytest.raises(k8.K8V4Error):
        k8.attn_k8v4_decode_partial(q4, q, pt_d, lens, 256, 0, 256, part, ws)
