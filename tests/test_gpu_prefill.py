"""GPU parity of the tcgen05 chunked-prefill attention against the fp64 oracle:
ragged chunks, explicit step arrays (including 0 and 1 visible cells), and the
full 8,192-token chunk at offset 229,376 on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
import quantized_paged_kv_q8_gb300 as k8
import synth
from gpu_util import TOL, append_both, dev_tensor, make_caches, rel_err

pytestmark = pytest.mark.gpu


def _build(seed, n_cells, P=64):
    w = synth.decode_workload(seed, n_cells, P=P, name="prefill_small")
    gpu, ref = make_caches(w.n_pages, P, 2)
    pt_d = append_both(gpu, ref, w.page_table, w.pos, synth.Tensor(w.k.f32[None], "bf16"),
                       synth.Tensor(w.v.f32[None], "bf16"))
    return w, gpu, ref, pt_d


def _prefill(gpu, q_dev, pt_row, seq_len, steps=None):
    out = torch.full(q_dev.shape, float("nan"), dtype=torch.float32, device="cuda")
    st = None if steps is None else torch.from_numpy(np.asarray(steps, np.int32)).cuda()
    k8.attn_k8v4_prefill(gpu, q_dev, pt_row, seq_len, out, step_arrays=st)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("n_cells,n_tok", [(700, 100), (1000, 37), (300, 300), (2048, 16)])
def test_prefill_causal_small(n_cells, n_tok):
    """A chunk of n_tok tokens ending at n_cells (token t sees n_cells - n_tok + t + 1
    cells); every row compared."""
    w, gpu, ref, pt_d = _build(synth.config_seed(5) + n_cells + n_tok, n_cells)
    q = synth.q_values(w.seed, 7, n_tok, 2, "bf16")
    got = _prefill(gpu, dev_tensor(q, (n_tok, 16, 256)), pt_d[0], n_cells)
    assert k8.k8v4_last_device_status() == 0
    steps = (n_cells - n_tok + 1 + np.arange(n_tok))[None].astype(np.int32)
    rs, rh, rv = oracle.multi_query_rows(steps, 16)
    want = ref.attention(w.page_table, rs, rh, rv, q.f32.reshape(-1, 256))
    assert rel_err(got.reshape(-1, 256), want) <= TOL


@pytest.mark.parametrize("P", [128, 256])
def test_prefill_page_sizes(P):
    """Pages of 128 and 256 cells (several 64-cell tiles per page), a ragged last
    page and a ragged last block of 16 tokens."""
    n_cells, n_tok = 1500, 77
    w, gpu, ref, pt_d = _build(synth.config_seed(5) + P, n_cells, P=P)
    q = synth.q_values(w.seed, 9, n_tok, 2, "bf16")
    got = _prefill(gpu, dev_tensor(q, (n_tok, 16, 256)), pt_d[0], n_cells)
    assert k8.k8v4_last_device_status() == 0
    steps = (n_cells - n_tok + 1 + np.arange(n_tok))[None].astype(np.int32)
    rs, rh, rv = oracle.multi_query_rows(steps, 16)
    want = ref.attention(w.page_table, rs, rh, rv, q.f32.reshape(-1, 256))
    assert rel_err(got.reshape(-1, 256), want) <= TOL


def test_prefill_rejects_pages_below_a_tile():
    """16-cell pages cannot hold a 64-cell tile: the call is refused before any
    launch and the output is untouched."""
    w, gpu, ref, pt_d = _build(synth.config_seed(5) + 16, 200, P=16)
    q = synth.q_values(w.seed, 10, 8, 2, "bf16")
    out = torch.full((8, 16, 256), 7.0, dtype=torch.float32, device="cuda")
    with pytest.raises(k8.K8V4Error) as e:
        k8.attn_k8v4_prefill(gpu, dev_tensor(q, (8, 16, 256)), pt_d[0], 200, out)
    assert e.value.code == k8.EINVAL
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)


def test_prefill_step_arrays():
    """Explicit per-token visible counts in any order, including 0 (zero output)
    and 1 (exactly the first cell's V)."""
    n_cells, n_tok = 900, 40
    w, gpu, ref, pt_d = _build(synth.config_seed(5) + 11, n_cells)
    rng = np.random.default_rng(3)
    steps = rng.integers(1, n_cells + 1, n_tok).astype(np.int32)
    steps[0], steps[5], steps[17] = 0, 1, n_cells
    q = synth.q_values(w.seed, 8, n_tok, 2, "bf16")
    got = _prefill(gpu, dev_tensor(q, (n_tok, 16, 256)), pt_d[0], n_cells, steps=steps)
    assert k8.k8v4_last_device_status() == 0
    assert np.all(got[0] == 0.0)
    rs, rh, rv = oracle.multi_query_rows(steps[None], 16)
    want = ref.attention(w.page_table, rs, rh, rv, q.f32.reshape(-1, 256))
    assert rel_err(got.reshape(-1, 256)[16:], want[16:]) <= TOL


def test_prefill_rows_equal_decode():
    """Mode cross-check: prefill token t equals decode at seq_len - n + t + 1."""
    n_cells, n_tok = 1500, 24
    w, gpu, ref, pt_d = _build(synth.config_seed(5) + 12, n_cells)
    q = synth.q_values(w.seed, 9, n_tok, 2, "bf16")
    qd = dev_tensor(q, (n_tok, 16, 256))
    got = _prefill(gpu, qd, pt_d[0], n_cells)
    lens = (n_cells - n_tok + 1 + np.arange(n_tok)).astype(np.int32)
    out = torch.empty(n_tok, 16, 256, device="cuda")
    ws = k8.workspace(gpu, n_tok, 1, n_cells)
    k8.attn_k8v4_decode(gpu, qd, torch.from_numpy(np.repeat(w.page_table, n_tok, 0)).cuda(),
                        torch.from_numpy(lens).cuda(), n_cells, out, ws)
    torch.cuda.synchronize()
    assert rel_err(got.reshape(-1, 256), out.cpu().numpy().reshape(-1, 256)) <= 2 * TOL


def test_prefill_config5_full_sampled():
    """Config 5: append an 8,192-token chunk at offset 229,376 (after the 229,376-cell
    history), then causal prefill of the chunk over 237,568 cells; the appended
    chunk's bytes are checked in full, attention on 540 rows: the edge tokens and
    one seeded row in each of the 512 token blocks."""
    w = synth.config5()
    gpu, ref = make_caches(w.n_pages, w.page_size, w.n_kv)
    hk, hv = synth.prefill_kv(w, 0, w.history)
    append_both(gpu, ref, w.page_table, np.array([0]), synth.Tensor(hk.f32[None], "bf16"),
                synth.Tensor(hv.f32[None], "bf16"))
    ck, cv = synth.prefill_kv(w, w.history, w.chunk)
    pt_d = append_both(gpu, ref, w.page_table, np.array([w.history]), synth.Tensor(ck.f32[None], "bf16"),
                       synth.Tensor(cv.f32[None], "bf16"))
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    assert np.array_equal(gpu.pages.cpu().numpy(), ref.buf)
    q = synth.prefill_q(w)
    got = _prefill(gpu, dev_tensor(q, (w.chunk, 16, 256)), pt_d[0], w.total)
    assert k8.k8v4_last_device_status() == 0
    # hand-picked edges, plus one seeded (token, head) row in every 16-token block
    # (every CTA row group and both KV heads' CTAs), 540 rows in all
    sel = [(t, h) for t in (0, 1, 15, 16, 1000, 4095, 8191) for h in (0, 7, 8, 15)]
    rng = np.random.default_rng(20251)
    sel += [(16 * blk + int(rng.integers(16)), int(rng.integers(16))) for blk in range(w.chunk // 16)]
    rs = np.zeros(len(sel), np.int32)
    rh = np.array([h for _, h in sel], np.int32)
    rv = np.array([w.history + t + 1 for t, _ in sel], np.int32)
    qrows = np.stack([q.f32[t, h] for t, h in sel])
    want = ref.attention(w.page_table, rs, rh, rv, qrows)
    gsel = np.stack([got[t, h] for t, h in sel])
    assert rel_err(gsel, want) <= TOL
