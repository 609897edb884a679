"""The bounded-wait failure path of the mbarrier-driven kernels, made to run on
the GPU without a fault: with the wait bound set below 1 us every wait that is
not already complete gives up after one poll (the barrier would still complete on its
own), so the kernel records K8V4_ECUDA, waits (with its default bound) for its
own copies and MMAs, releases what it holds (tensor memory for prefill) and
returns.  The decode kernel's first waits usually find their copies landed
(it issues them before it sets up q), so there a diagnostic switch withholds
one tile's copies instead, and the wait on that stage runs out.  A normal call
in the same process afterwards must match the oracle, which shows the context
and the tensor memory are intact."""
import numpy as np
import pytest
import torch

import oracle
import quantized_paged_kv_q8_gb300 as k8
import synth
from gpu_util import TOL, append_both, decode_gpu, dev_tensor, make_caches, rel_err, verify_gpu

pytestmark = pytest.mark.gpu


def _cache(seed, n_cells):
    w = synth.decode_workload(seed, n_cells, P=64, name="timeout")
    gpu, ref = make_caches(w.n_pages, 64, 2)
    pt_d = append_both(gpu, ref, w.page_table, w.pos, synth.Tensor(w.k.f32[None], "bf16"),
                       synth.Tensor(w.v.f32[None], "bf16"))
    return w, gpu, ref, pt_d


def test_prefill_wait_timeout_then_recovery():
    w, gpu, ref, pt_d = _cache(synth.config_seed(5) + 901, 256)
    n_tok = 16
    q = synth.q_values(w.seed, 9, n_tok, 2, "bf16")
    q_d = dev_tensor(q, (n_tok, 16, 256))
    out = torch.empty(n_tok, 16, 256, device="cuda")
    assert k8.k8v4_last_device_status() == 0
    try:
        k8.k8v4_set_wait_limit_ns(1)
        k8.attn_k8v4_prefill(gpu, q_d, pt_d[0], 256, out)
        assert k8.k8v4_last_device_status() == k8.ECUDA
    finally:
        k8.k8v4_set_wait_limit_ns(0)   # back to each kernel's default
    k8.attn_k8v4_prefill(gpu, q_d, pt_d[0], 256, out)
    assert k8.k8v4_last_device_status() == 0
    steps = (256 - n_tok + 1 + np.arange(n_tok)).astype(np.int32)
    rs, rh, rv = oracle.multi_query_rows(steps[None], 16)
    want = ref.attention(w.page_table, rs, rh, rv, q.f32.reshape(-1, 256))
    assert rel_err(out.cpu().numpy().reshape(-1, 256), want) <= TOL


@pytest.mark.parametrize("qdt", ["f32", "bf16"])
def test_decode_wait_timeout_then_recovery(qdt):
    """Both query types of the TMA decode kernel (fp32 queries carry a second q
    term and run fewer worker warps).  With the withheld-copy diagnostic on,
    worker 0 of the first CTA never issues its first tile, so its wait on that
    stage runs out after the 200 us bound -- a phase that nothing completes,
    while every other wait of the call completes well within the bound: the
    kernel records K8V4_ECUDA, closes that stage itself, waits for its copies in
    flight and returns.  A normal call in the same process afterwards matches
    the oracle."""
    n = 32768
    w, gpu, ref, pt_d = _cache(synth.config_seed(2) + 902, n)
    q = synth.q_values(w.seed, 9, 1, 2, qdt)
    q_d = dev_tensor(q, (1, 16, 256))
    assert k8.k8v4_last_device_status() == 0
    try:
        k8.k8v4_set_wait_limit_ns(200_000)
        k8.k8v4_set_withheld_copy(True)
        decode_gpu(gpu, q_d, pt_d, w.seq_lens, n)
    finally:
        k8.k8v4_set_withheld_copy(False)
        k8.k8v4_set_wait_limit_ns(0)
    assert k8.k8v4_last_device_status() == k8.ECUDA
    got = decode_gpu(gpu, q_d, pt_d, w.seq_lens, n)
    assert k8.k8v4_last_device_status() == 0
    rs, rh, rv = oracle.decode_rows(1, 16, w.seq_lens)
    want = ref.attention(w.page_table, rs, rh, rv, q.f32.reshape(-1, 256))
    assert rel_err(got.reshape(-1, 256), want) <= TOL


def test_verify_team_kernel_wait_timeout_then_recovery():
    """The team-of-warps verify kernel (bf16 queries, pages that are not a
    multiple of 64 cells): the same bounded-wait failure path, then a normal
    call in the same process against the oracle."""
    n, P, n_q = 32768, 16, 3
    w = synth.decode_workload(synth.config_seed(4) + 903, n, P=P, name="timeout-verify")
    gpu, ref = make_caches(w.n_pages, P, 2)
    pt_d = append_both(gpu, ref, w.page_table, w.pos, synth.Tensor(w.k.f32[None], "bf16"),
                       synth.Tensor(w.v.f32[None], "bf16"))
    q = synth.q_values(w.seed, 9, n_q, 2, "bf16")
    q_d = dev_tensor(q, (1, n_q, 16, 256))
    steps = np.array([[n - 2, n - 1, n]], np.int32)
    assert k8.k8v4_last_device_status() == 0
    flush = torch.ones(128 << 20, dtype=torch.float32, device="cuda")
    statuses = []
    try:
        for _ in range(5):
            float(flush.sum())
            torch.cuda.synchronize()
            k8.k8v4_set_wait_limit_ns(1)
            verify_gpu(gpu, q_d, pt_d, steps, n)
            k8.k8v4_set_wait_limit_ns(0)
            statuses.append(k8.k8v4_last_device_status())
            if statuses[-1] == k8.ECUDA:
                break
    finally:
        k8.k8v4_set_wait_limit_ns(0)
    assert statuses[-1] == k8.ECUDA and set(statuses) <= {0, k8.ECUDA}, statuses
    del flush
    got = verify_gpu(gpu, q_d, pt_d, steps, n)
    assert k8.k8v4_last_device_status() == 0
    rs, rh, rv = oracle.multi_query_rows(steps, 16)
    want = ref.attention(w.page_table, rs, rh, rv, q.f32.reshape(-1, 256))
    assert rel_err(got.reshape(-1, 256), want) <= TOL
