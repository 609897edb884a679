"""GPU parity of decode and verify attention against the fp64 oracle, which
builds its own cache from the same seeded inputs.  Bar: elementwise
|gpu - ref| <= 2e-5 * max(1, |ref|) in fp32."""
import numpy as np
import pytest
import torch

import oracle
import quantized_paged_kv_q8_gb300 as k8
import synth
from gpu_util import TOL, append_both, decode_gpu, dev_tensor, make_caches, rel_err, verify_gpu

pytestmark = pytest.mark.gpu


def _single_seq(w, fmt=k8.FORMAT_K8V4, dtype=None):
    dtype = dtype or w.dtype
    gpu, ref = make_caches(w.n_pages, w.page_size, w.n_kv, fmt)
    pt_d = append_both(gpu, ref, w.page_table, w.pos, synth.Tensor(w.k.f32[None], dtype),
                       synth.Tensor(w.v.f32[None], dtype))
    return gpu, ref, pt_d


@pytest.mark.parametrize("fmt", [k8.FORMAT_K8V4, k8.FORMAT_Q4])
def test_decode_tiny_fp32(fmt):
    """Config 1: 1,024 fp32 cells with ties, one fp32 decode query."""
    w = synth.config1()
    gpu, ref, pt_d = _single_seq(w, fmt)
    got = decode_gpu(gpu, dev_tensor(w.q, (1, 16, 256)), pt_d, w.seq_lens, int(w.seq_lens[0]))
    rs, rh, rv = oracle.decode_rows(1, 16, w.seq_lens)
    want = ref.attention(w.page_table, rs, rh, rv, w.q.f32.reshape(-1, 256))
    assert rel_err(got.reshape(-1, 256), want) <= TOL
    assert k8.k8v4_last_device_status() == 0


@pytest.mark.parametrize("fmt", [k8.FORMAT_K8V4, k8.FORMAT_INT8, k8.FORMAT_Q4])
def test_decode_ragged_lengths(fmt):
    """One 5,000-cell cache read by 9 sequences that share its page table and see
    1, 15, 16, 17, 37, 1,000, 4,095, 4,999 and 5,000 cells (ragged tails, tiles
    split across CTAs)."""
    w = synth.decode_workload(synth.config_seed(2) + 7, 5000, P=64)
    gpu, ref, _ = _single_seq(w, fmt)
    lens = np.array([1, 15, 16, 17, 37, 1000, 4095, 4999, 5000], np.int32)
    n = len(lens)
    pt = np.repeat(w.page_table, n, axis=0)
    pt_d = torch.from_numpy(pt).cuda()
    q = synth.q_values(w.seed, 3, n, 2, "bf16")
    got = decode_gpu(gpu, dev_tensor(q, (n, 16, 256)), pt_d, lens, 5000)
    rs, rh, rv = oracle.decode_rows(n, 16, lens)
    want = ref.attention(pt, rs, rh, rv, q.f32.reshape(-1, 256))
    assert rel_err(got.reshape(-1, 256), want) <= TOL


def test_decode_32k():
    """Config 2: 32,768 bf16 cells, P = 64, shuffled pages, bf16 q."""
    w = synth.config2()
    gpu, ref, pt_d = _single_seq(w)
    got = decode_gpu(gpu, dev_tensor(w.q, (1, 16, 256)), pt_d, w.seq_lens, 32768)
    rs, rh, rv = oracle.decode_rows(1, 16, w.seq_lens)
    want = ref.attention(w.page_table, rs, rh, rv, w.q.f32.reshape(-1, 256))
    assert rel_err(got.reshape(-1, 256), want) <= TOL
    # attention never writes the cache
    assert np.array_equal(gpu.pages.cpu().numpy(), ref.buf)


def test_decode_wide_v_scales():
    """V rows whose q4_0 scales reach |d| >= 256 (values in the thousands) mixed
    with ordinary rows: tiles holding one are read through the wide-scale path of
    the decode PV, the others through the narrow one.  An output element here is
    a sum of terms up to ~1e4 that cancel down to ~1, which no fp32 sum resolves
    to 2e-5 of the small result, so the bar is norm-wise: 2e-5 of the largest
    |ref| of the row (the fp32 rounding scale of its terms)."""
    w = synth.decode_workload(synth.config_seed(2) + 9, 3000, P=64)
    v = w.v.f32.copy()
    v[100:400] *= 5000.0           # whole tiles of wide scales
    v[1000::37] *= 3000.0          # one wide cell in many otherwise narrow tiles
    v[2000:2100] *= 1e-6           # tiny scales (subnormal fp16 d) next to them
    gpu, ref = make_caches(w.n_pages, w.page_size, w.n_kv)
    pt_d = append_both(gpu, ref, w.page_table, w.pos, synth.Tensor(w.k.f32[None], w.dtype),
                       synth.Tensor(v[None], w.dtype))
    got = decode_gpu(gpu, dev_tensor(w.q, (1, 16, 256)), pt_d, w.seq_lens, 3000)
    rs, rh, rv = oracle.decode_rows(1, 16, w.seq_lens)
    want = ref.attention(w.page_table, rs, rh, rv, w.q.f32.reshape(-1, 256))
    assert np.abs(want).max() > 100.0          # the wide rows carry weight
    assert _normwise(got.reshape(-1, 256), want) <= TOL
    # and a length that ends inside the wide run
    got = decode_gpu(gpu, dev_tensor(w.q, (1, 16, 256)), pt_d, np.array([250], np.int32), 3000)
    rs, rh, rv = oracle.decode_rows(1, 16, [250])
    want = ref.attention(w.page_table, rs, rh, rv, w.q.f32.reshape(-1, 256))
    assert _normwise(got.reshape(-1, 256), want) <= TOL


def _normwise(got: np.ndarray, ref: np.ndarray) -> float:
    """max over rows of max |got - ref| / max(1, max |ref|)."""
    e = np.abs(got.astype(np.float64) - ref).max(axis=1)
    return float((e / np.maximum(1.0, np.abs(ref).max(axis=1))).max())


def test_decode_zero_length_rows_are_zero():
    w = synth.decode_workload(synth.config_seed(2) + 8, 200, P=16)
    gpu, ref, _ = _single_seq(w)
    pt = np.repeat(w.page_table, 2, axis=0)
    lens = np.array([0, 200], np.int32)
    q = synth.q_values(w.seed, 4, 2, 2, "bf16")
    got = decode_gpu(gpu, dev_tensor(q, (2, 16, 256)), torch.from_numpy(pt).cuda(), lens, 200)
    assert np.all(got[0] == 0.0)
    rs, rh, rv = oracle.decode_rows(1, 16, [200])
    want = ref.attention(w.page_table, rs, rh, rv, q.f32[1].reshape(-1, 256))
    assert rel_err(got[1].reshape(-1, 256), want) <= TOL


@pytest.mark.parametrize("n_q", [1, 2, 3, 5, 8])
def test_verify_small(n_q):
    """Verify with per-query steps len - (n_q-1) + i over three sequences in one
    interleaved pool; every row of every query checked."""
    seed = synth.config_seed(4) + 100 + n_q
    lens = np.array([130, 2049, 777], np.int32)
    w = synth.config4(seed=seed, lens=lens, n_q=n_q)
    gpu, ref = make_caches(w.n_pages, w.page_size, w.n_kv)
    pt_d = torch.from_numpy(w.page_table).cuda()
    for b in range(len(lens)):
        append_both(gpu, ref, w.page_table[b:b + 1], np.array([0]), synth.Tensor(w.k[b].f32[None], "bf16"),
                    synth.Tensor(w.v[b].f32[None], "bf16"))
    q = torch.stack([dev_tensor(w.q[b]) for b in range(len(lens))])
    got = verify_gpu(gpu, q, pt_d, w.steps, int(lens.max()))
    rs, rh, rv = oracle.multi_query_rows(w.steps, 16)
    qrows = np.concatenate([w.q[b].f32.reshape(-1, 256) for b in range(len(lens))])
    want = ref.attention(w.page_table, rs, rh, rv, qrows)
    assert rel_err(got.reshape(-1, 256), want) <= TOL


@pytest.mark.parametrize("fmt", [k8.FORMAT_K8V4, k8.FORMAT_INT8, k8.FORMAT_Q4])
@pytest.mark.parametrize("P,qdt", [(16, "f32"), (64, "bf16")])
def test_verify_irregular_steps(fmt, P, qdt):
    """Verify with irregular per-query steps (0, 1, page and tile edges,
    mid-tile, the whole sequence): three sequences, 7 queries each, every row
    checked; 16-cell pages with fp32 queries (warp-MMA kernel) and 64-cell pages
    with bf16 queries (the team-of-warps TMA kernel for k8v4)."""
    seed = synth.config_seed(4) + 77
    H, n_q = 2, 7
    lens = np.array([1500, 33, 700], np.int32)
    pt, n_pages = synth.interleaved_pool(seed, lens, P)
    ks = [synth.kv_values(seed, synth.T_K, b, int(n), H, 3, "bf16") for b, n in enumerate(lens)]
    vs = [synth.kv_values(seed, synth.T_V, b, int(n), H, 3, "bf16") for b, n in enumerate(lens)]
    qs = [synth.q_values(seed, b, n_q, H, qdt) for b in range(len(lens))]
    steps = np.array([[0, 1, 16, 17, 499, 1499, 1500],
                      [33, 0, 1, 31, 32, 16, 15],
                      [700, 699, 64, 65, 0, 2, 350]], np.int32)
    gpu, ref = make_caches(n_pages, P, H, fmt)
    pt_d = torch.from_numpy(pt).cuda()
    for b in range(len(lens)):
        append_both(gpu, ref, pt[b:b + 1], np.array([0]), synth.Tensor(ks[b].f32[None], "bf16"),
                    synth.Tensor(vs[b].f32[None], "bf16"))
    q = torch.stack([dev_tensor(qs[b]) for b in range(len(lens))])
    got = verify_gpu(gpu, q, pt_d, steps, int(lens.max()))
    assert k8.k8v4_last_device_status() == 0
    rs, rh, rv = oracle.multi_query_rows(steps, 16)
    qrows = np.concatenate([qs[b].f32.reshape(-1, 256) for b in range(len(lens))])
    want = ref.attention(pt, rs, rh, rv, qrows)
    got = got.reshape(-1, 256)
    assert np.all(got[rv == 0] == 0.0)
    assert rel_err(got, want) <= TOL


def test_verify_rows_equal_decode_at_step():
    """Mode cross-check on the GPU: verify query i equals decode with seq_len =
    len - 4 + i (same q, same cache) within the tolerance."""
    seed = synth.config_seed(4) + 55
    lens = np.array([3000, 1500], np.int32)
    w = synth.config4(seed=seed, lens=lens)
    gpu, ref = make_caches(w.n_pages, w.page_size, w.n_kv)
    pt_d = torch.from_numpy(w.page_table).cuda()
    for b in range(2):
        append_both(gpu, ref, w.page_table[b:b + 1], np.array([0]), synth.Tensor(w.k[b].f32[None], "bf16"),
                    synth.Tensor(w.v[b].f32[None], "bf16"))
    q = torch.stack([dev_tensor(w.q[b]) for b in range(2)])
    ver = verify_gpu(gpu, q, pt_d, w.steps, 3000)
    for i in range(5):
        dec = decode_gpu(gpu, q[:, i].contiguous(), pt_d, w.steps[:, i], 3000)
        assert rel_err(ver[:, i].reshape(-1, 256), dec.reshape(-1, 256)) <= 2 * TOL


def test_verify_config4_full_sampled():
    """Config 4 at full size: 8 sequences, lengths U[16,384, 65,536], 5 queries
    each; every one of the 640 rows (8 sequences x 5 queries x 16 heads)."""
    w = synth.config4()
    gpu, ref = make_caches(w.n_pages, w.page_size, w.n_kv)
    pt_d = torch.from_numpy(w.page_table).cuda()
    for b in range(w.n_seqs):
        append_both(gpu, ref, w.page_table[b:b + 1], np.array([0]), synth.Tensor(w.k[b].f32[None], "bf16"),
                    synth.Tensor(w.v[b].f32[None], "bf16"))
    q = torch.stack([dev_tensor(w.q[b]) for b in range(w.n_seqs)])
    got = verify_gpu(gpu, q, pt_d, w.steps, int(w.seq_lens.max()))
    assert k8.k8v4_last_device_status() == 0
    sel = [(b, i, h) for b in range(w.n_seqs) for i in range(w.n_q) for h in range(16)]
    rs = np.array([s[0] for s in sel], np.int32)
    rh = np.array([s[2] for s in sel], np.int32)
    rv = np.array([w.steps[b, i] for b, i, _ in sel], np.int32)
    qrows = np.stack([w.q[b].f32[i, h] for b, i, h in sel])
    want = ref.attention(w.page_table, rs, rh, rv, qrows)
    gsel = np.stack([got[b, i, h] for b, i, h in sel])
    assert rel_err(gsel, want) <= TOL


@pytest.mark.parametrize("n_cells", [14848, 118784, 237568, 262144, 118784 + 37])
def test_decode_long_context(n_cells):
    """Config 3 lengths (and one non-aligned length): all 16 rows against the oracle;
    the INT8 and Q4 comparison arms at the 238K point too."""
    seed = synth.config_seed(3)
    w = synth.config3(n_cells, seed=seed)
    fmts = [k8.FORMAT_K8V4] + ([k8.FORMAT_INT8, k8.FORMAT_Q4] if n_cells == 237568 else [])
    for fmt in fmts:
        gpu, ref, pt_d = _single_seq(w, fmt)
        got = decode_gpu(gpu, dev_tensor(w.q, (1, 16, 256)), pt_d, w.seq_lens, n_cells)
        rs, rh, rv = oracle.decode_rows(1, 16, w.seq_lens)
        want = ref.attention(w.page_table, rs, rh, rv, w.q.f32.reshape(-1, 256))
        assert rel_err(got.reshape(-1, 256), want) <= TOL, fmt
        assert k8.k8v4_last_device_status() == 0
        del gpu, ref
        torch.cuda.empty_cache()


def test_decode_bad_length_and_page_are_reported():
    """A device length beyond max_seq_len is clipped and reported; a bad page id is
    skipped and reported; the call still completes and the GPU stays usable."""
    w = synth.decode_workload(synth.config_seed(2) + 9, 256, P=16)
    gpu, ref, pt_d = _single_seq(w)
    q = dev_tensor(w.q, (1, 16, 256))
    got = decode_gpu(gpu, q, pt_d, np.array([300], np.int32), 256)
    assert k8.k8v4_last_device_status() == k8.ERANGE
    rs, rh, rv = oracle.decode_rows(1, 16, [256])
    assert rel_err(got.reshape(-1, 256), ref.attention(w.page_table, rs, rh, rv, w.q.f32.reshape(-1, 256))) <= TOL
    bad = w.page_table.copy()
    bad[0, 3] = 1 << 20
    decode_gpu(gpu, q, torch.from_numpy(bad).cuda(), w.seq_lens, 256)
    assert k8.k8v4_last_device_status() == k8.ERANGE
    assert np.all(gpu.pages.cpu().numpy() == ref.buf)


@pytest.mark.parametrize("fmt,H", [(k8.FORMAT_K8V4, 1), (k8.FORMAT_K8V4, 3), (k8.FORMAT_Q4, 3), (k8.FORMAT_INT8, 3)])
def test_other_kv_head_counts(fmt, H):
    """1 and 3 KV heads (8 and 24 query heads), 32-cell pages, two sequences in
    one interleaved pool: cache bytes equal the oracle's and decode and verify
    are within the tolerance (the index arithmetic divides by H, P and the
    token count; 3 is the first divisor that is not a power of two)."""
    seed = synth.config_seed(2) + 40 + H
    P = 32
    lens = np.array([1111, 300], np.int32)
    pt, n_pages = synth.interleaved_pool(seed, lens, P)
    ks = [synth.kv_values(seed, synth.T_K, b, int(n), H, 3, "bf16") for b, n in enumerate(lens)]
    vs = [synth.kv_values(seed, synth.T_V, b, int(n), H, 3, "bf16") for b, n in enumerate(lens)]
    gpu, ref = make_caches(n_pages, P, H, fmt)
    for b in range(len(lens)):
        append_both(gpu, ref, pt[b:b + 1], np.array([0]), synth.Tensor(ks[b].f32[None], "bf16"),
                    synth.Tensor(vs[b].f32[None], "bf16"))
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    assert np.array_equal(gpu.pages.cpu().numpy(), ref.buf)
    pt_d = torch.from_numpy(pt).cuda()
    HQ = 8 * H
    q = synth.q_values(seed, 0, len(lens), H, "bf16")
    got = decode_gpu(gpu, dev_tensor(q, (len(lens), HQ, 256)), pt_d, lens, int(lens.max()))
    rs, rh, rv = oracle.decode_rows(len(lens), HQ, lens)
    assert rel_err(got.reshape(-1, 256), ref.attention(pt, rs, rh, rv, q.f32.reshape(-1, 256))) <= TOL
    steps = np.stack([np.maximum(int(L) - 4 + np.arange(5), 0) for L in lens]).astype(np.int32)
    qs = [synth.q_values(seed, 1 + b, 5, H, "bf16") for b in range(len(lens))]
    got = verify_gpu(gpu, torch.stack([dev_tensor(x) for x in qs]), pt_d, steps, int(lens.max()))
    assert k8.k8v4_last_device_status() == 0
    rs, rh, rv = oracle.multi_query_rows(steps, HQ)
    qrows = np.concatenate([x.f32.reshape(-1, 256) for x in qs])
    assert rel_err(got.reshape(-1, 256), ref.attention(pt, rs, rh, rv, qrows)) <= TOL


def test_one_kv_head_long_sequence_many_splits():
    """One KV head (8 query heads) and one 65,536-cell sequence: decode cuts it
    into more than 96 cell ranges and verify into more still, so the combine's
    many-split instantiation folds each warp's splits over several rounds (12
    splits a round), rescaling its running sum at each new round maximum.  All
    decode rows and a 5-query verify window against the oracle."""
    n, H, P = 65536, 1, 64
    seed = synth.config_seed(3) + 211
    n_pages = n // P
    k = synth.kv_values(seed, synth.T_K, 0, n, H, 3, "bf16")
    v = synth.kv_values(seed, synth.T_V, 0, n, H, 3, "bf16")
    pt = synth.page_table_shuffled(seed, synth.stream_id(synth.T_PT, 0), n_pages, n_pages).reshape(1, -1)
    gpu, ref = make_caches(n_pages, P, H)
    pt_d = append_both(gpu, ref, pt, np.array([0]), synth.Tensor(k.f32[None], "bf16"), synth.Tensor(v.f32[None], "bf16"))
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    row_bytes = 8 * H * 1040                    # one partial row (260 floats) per query head
    assert k8.attn_k8v4_workspace_bytes(gpu, 1, 1, n) // row_bytes > 96
    assert k8.attn_k8v4_workspace_bytes(gpu, 1, 5, n) // (5 * row_bytes) > 96
    lens = np.array([n], np.int32)
    q = synth.q_values(seed, 0, 1, H, "bf16")
    got = decode_gpu(gpu, dev_tensor(q, (1, 8, 256)), pt_d, lens, n)
    assert k8.k8v4_last_device_status() == 0
    rs, rh, rv = oracle.decode_rows(1, 8, lens)
    assert rel_err(got.reshape(-1, 256), ref.attention(pt, rs, rh, rv, q.f32.reshape(-1, 256))) <= TOL
    steps = (n - 4 + np.arange(5)).astype(np.int32)[None]
    qv = synth.q_values(seed, 1, 5, H, "bf16")
    got = verify_gpu(gpu, dev_tensor(qv)[None], pt_d, steps, n)
    assert k8.k8v4_last_device_status() == 0
    rs, rh, rv = oracle.multi_query_rows(steps, 8)
    assert rel_err(got.reshape(-1, 256), ref.attention(pt, rs, rh, rv, qv.f32.reshape(-1, 256))) <= TOL
