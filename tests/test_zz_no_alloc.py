"""attn_k8v4_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (no allocator of their own, or a loop where cudaFree's
device-wide synchronisation is not acceptable).  Its split-K partials live in
the library's fixed device array, so its output must match the regular decode
(which uses a caller workspace) bit for bit, call after call.

This file is named to be collected last, so a stopping run has already run
every other test if it fails; it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import quantized_paged_kv_q8_gb300 as k8
import synth
from gpu_util import append_both, dev_tensor, make_caches

pytestmark = pytest.mark.gpu


def _noalloc(cache, q, pt_d, lens_d, max_len, out):
    L = k8.lib()
    rc = L.attn_k8v4_decode_noalloc(cache.ref(), ctypes.c_void_p(q.data_ptr()), k8.BF16,
                                    ctypes.c_void_p(pt_d.data_ptr()), pt_d.shape[-1],
                                    ctypes.c_void_p(lens_d.data_ptr()), q.shape[0], max_len, 1.0 / 16.0,
                                    ctypes.c_void_p(out.data_ptr()), k8._stream(None))
    return rc


def test_noalloc_decode_matches_workspace_decode_twice():
    w = synth.decode_workload(synth.config_seed(2) + 77, 6000, P=64)
    gpu, ref = make_caches(w.n_pages, w.page_size, w.n_kv)
    append_both(gpu, ref, w.page_table, w.pos, synth.Tensor(w.k.f32[None], "bf16"),
                synth.Tensor(w.v.f32[None], "bf16"))
    # two calls in a row with different batches, lengths and queries; the
    # first writes more partials than the second reads, so a second call that
    # picked up a stale partial of the first would differ
    for call, lens in enumerate((np.array([1, 4097, 5999], np.int32), np.array([6000], np.int32))):
        n = len(lens)
        pt_d = torch.from_numpy(np.repeat(w.page_table, n, axis=0)).cuda()
        lens_d = torch.from_numpy(lens).cuda()
        q = dev_tensor(synth.q_values(w.seed, 10 + call, n, 2, "bf16"), (n, 16, 256))
        want = torch.empty(n, 16, 256, device="cuda")
        ws = k8.workspace(gpu, n, 1, 6000)
        k8.attn_k8v4_decode(gpu, q, pt_d, lens_d, 6000, want, ws)
        got = torch.full((n, 16, 256), float("nan"), device="cuda")
        assert _noalloc(gpu, q, pt_d, lens_d, 6000, got) == k8.OK
        torch.cuda.synchronize()
        assert k8.k8v4_last_device_status() == 0
        # both paths launch the same kernels with the same split plan, so the
        # results agree bit for bit; a tolerance could hide a wrong scratch
        # offset or a partial left over from the previous call
        assert torch.equal(got, want)


def test_noalloc_rejects_batches_beyond_its_array():
    """A batch whose partials exceed the fixed 4 MiB array is refused up front."""
    w = synth.decode_workload(synth.config_seed(2) + 78, 64, P=64)
    gpu, _ = make_caches(w.n_pages, w.page_size, w.n_kv)
    n = 1000
    assert k8.attn_k8v4_workspace_bytes(gpu, n, 1, 64) > (4 << 20)
    pt_d = torch.from_numpy(np.repeat(w.page_table, n, axis=0)).cuda()
    lens_d = torch.full((n,), 64, dtype=torch.int32, device="cuda")
    q = torch.zeros(n, 16, 256, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(n, 16, 256, device="cuda")
    assert _noalloc(gpu, q, pt_d, lens_d, 64, out) == k8.ENOSPACE
