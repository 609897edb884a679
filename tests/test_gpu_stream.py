"""KV streaming on the GPU (the "kv: --kv k8v4 streams with --kv-resident" pull
request): a host mirror in page-locked memory holds every page, a device cache
holds the resident slots plus staging slots.  Checked here: the mirrored append
writes the oracle's bytes to both copies; the lookup table and the copies equal
the oracle's block lookups; streamed attention is bitwise equal to resident
attention (and within the tolerance of the fp64 oracle); a writer that skips the
mirror is caught (the pull request's negative control)."""
import numpy as np
import pytest
import torch

import oracle
import quantized_paged_kv_q8_gb300 as k8
import synth
from gpu_util import CANARY, TOL, dev_tensor, rel_err

pytestmark = pytest.mark.gpu

H = 2


class Streamed:
    """One streamed cache built by mirrored appends, and the same cells appended
    to a fully resident device cache (the reference) and to the oracle."""

    def __init__(self, fmt, lens, P, n_res, seed, kvdt="bf16", extra_stage=0):
        self.fmt, self.P = fmt, P
        self.lens = np.asarray(lens, np.int32)
        self.pt, self.n_host = synth.interleaved_pool(seed, np.maximum(self.lens, 1), P)
        self.ks = [synth.kv_values(seed, synth.T_K, b, max(int(n), 1), H, 3, kvdt) for b, n in enumerate(self.lens)]
        self.vs = [synth.kv_values(seed, synth.T_V, b, max(int(n), 1), H, 3, kvdt) for b, n in enumerate(self.lens)]
        rng = np.random.default_rng(seed)
        self.n_res = n_res
        self.slot_of_page = np.full(self.n_host, -1, np.int32)
        self.slot_of_page[rng.permutation(self.n_host)[:n_res]] = rng.permutation(n_res)
        need = int(((self.lens + P - 1) // P).sum())
        self.host = k8.PagedCache(self.n_host, P, H, fmt, device="pinned")
        self.host.pages.fill_(CANARY)
        self.dev = k8.PagedCache(n_res + need + extra_stage, P, H, fmt)
        self.dev.pages.fill_(CANARY)
        self.full = k8.PagedCache(self.n_host, P, H, fmt)
        self.full.pages.fill_(CANARY)
        self.ref = oracle.Cache(self.n_host, P, H, fmt, fill=CANARY)
        self.pt_d = torch.from_numpy(self.pt).cuda()
        self.sop_d = torch.from_numpy(self.slot_of_page).cuda()
        for b, n in enumerate(self.lens):
            cut = int(n) // 3                      # two appends: a history, then the rest at its offset
            for lo, hi in ((0, cut), (cut, int(n))):
                if hi <= lo:
                    continue
                kk = dev_tensor(synth.Tensor(self.ks[b].f32[None, lo:hi], kvdt))
                vv = dev_tensor(synth.Tensor(self.vs[b].f32[None, lo:hi], kvdt))
                pos = torch.tensor([lo], dtype=torch.int64, device="cuda")
                k8.kv_append_k8v4_mirrored(self.host, self.dev, self.sop_d, self.pt_d[b:b + 1], pos, kk, vv)
                k8.kv_append_k8v4(self.full, self.pt_d[b:b + 1], pos, kk, vv)
            if n > 0:
                self.ref.append(self.pt[b:b + 1], np.array([0]), self.ks[b].f32[None, :n], self.vs[b].f32[None, :n])
        torch.cuda.synchronize()
        assert k8.k8v4_last_device_status() == 0

    def resolve(self, lens, max_len):
        dev_pt = torch.full(self.pt.shape, -7, dtype=torch.int32, device="cuda")
        ws = torch.empty(k8.kv_stream_workspace_bytes(*self.pt.shape), dtype=torch.uint8, device="cuda")
        k8.kv_stream_resolve(self.host, self.dev, self.sop_d, self.n_res, self.pt_d,
                             torch.from_numpy(np.asarray(lens, np.int32)).cuda(), max_len, dev_pt, ws)
        return dev_pt

    def slot_bytes(self, s):
        pb = self.dev.page_bytes
        return self.dev.pages[s * pb:(s + 1) * pb].cpu().numpy()

    def ref_page(self, p):
        pb = self.dev.page_bytes
        return self.ref.buf[p * pb:(p + 1) * pb]


def _decode(cache, q, pt_d, lens, max_len):
    n = q.shape[0]
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    ws = k8.workspace(cache, n, 1, max_len)
    k8.attn_k8v4_decode(cache, q, pt_d, torch.from_numpy(np.asarray(lens, np.int32)).cuda(), max_len, out, ws)
    return out


def _verify(cache, q, pt_d, steps, max_len):
    n, nq = q.shape[0], q.shape[1]
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    ws = k8.workspace(cache, n, nq, max_len)
    k8.attn_k8v4_verify(cache, q, pt_d, torch.from_numpy(np.asarray(steps, np.int32)).cuda(), max_len, out, ws)
    return out


@pytest.mark.parametrize("fmt", [k8.FORMAT_K8V4, k8.FORMAT_Q4, k8.FORMAT_INT8])
def test_mirrored_append_writes_both_copies(fmt):
    """The mirror holds the oracle's bytes for every page; each resident slot
    holds the oracle's bytes of its page; staging slots are untouched."""
    s = Streamed(fmt, [700, 1333, 64, 0], 64, 9, synth.config_seed(4) + 301)
    assert np.array_equal(s.host.pages.numpy(), s.ref.buf)
    for p in range(s.n_host):
        slot = int(s.slot_of_page[p])
        if slot >= 0:
            assert np.array_equal(s.slot_bytes(slot), s.ref_page(p)), (p, slot)
    tail = s.dev.pages[s.n_res * s.dev.page_bytes:].cpu().numpy()
    assert np.all(tail == CANARY)


def test_resolve_matches_oracle_lookups():
    """The device page table equals the oracle's block lookups; every staging
    slot the lookups name holds its host page's bytes; resident slots keep
    theirs; nothing past the copies is touched."""
    s = Streamed(k8.FORMAT_K8V4, [1500, 33, 700, 64], 64, 11, synth.config_seed(4) + 302)
    before = s.dev.pages.cpu().numpy().copy()
    lens = np.array([1500, 20, 650, 0], np.int32)
    dev_pt = s.resolve(lens, 1500)
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    want, moves, over = oracle.stream_resolve(s.pt, lens, s.slot_of_page, s.n_res, s.dev.n_pages, s.P, 1500)
    assert not over
    assert np.array_equal(dev_pt.cpu().numpy(), want)
    after = s.dev.pages.cpu().numpy()
    pb = s.dev.page_bytes
    moved = set()
    for hp, slot in moves:
        assert np.array_equal(after[slot * pb:(slot + 1) * pb], s.ref_page(hp))
        moved.add(slot)
    for slot in range(s.dev.n_pages):
        if slot not in moved:
            assert np.array_equal(after[slot * pb:(slot + 1) * pb], before[slot * pb:(slot + 1) * pb]), slot


@pytest.mark.parametrize("fmt,P", [(k8.FORMAT_K8V4, 64), (k8.FORMAT_K8V4, 16), (k8.FORMAT_Q4, 64),
                                   (k8.FORMAT_INT8, 64)])
def test_streamed_attention_bitwise_equals_resident(fmt, P):
    """Decode and verify over the device table of a streamed call are bitwise
    equal to the same calls over a fully resident cache, and decode is within
    the tolerance of the fp64 oracle."""
    seed = synth.config_seed(4) + 303
    lens = np.array([2500, 17, 1024, 700], np.int32)
    s = Streamed(fmt, lens, P, 13 if P == 64 else 40, seed)
    n = len(lens)
    q = dev_tensor(synth.q_values(seed, 0, n, H, "bf16"), (n, 16, 256))
    dev_pt = s.resolve(lens, 2500)
    streamed = _decode(s.dev, q, dev_pt, lens, 2500)
    resident = _decode(s.full, q, s.pt_d, lens, 2500)
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    assert torch.equal(streamed, resident)
    rs, rh, rv = oracle.decode_rows(n, 16, lens)
    qf = synth.q_values(seed, 0, n, H, "bf16").f32.reshape(-1, 256)
    assert rel_err(streamed.cpu().numpy().reshape(-1, 256), s.ref.attention(s.pt, rs, rh, rv, qf)) <= TOL
    # verify: five queries per sequence, steps up to the length
    steps = np.stack([np.maximum(int(L) - 4 + np.arange(5), 0) for L in lens]).astype(np.int32)
    steps[1, 0] = 0
    qv = torch.stack([dev_tensor(synth.q_values(seed, 1 + b, 5, H, "bf16")) for b in range(n)])
    dev_pt = s.resolve(steps.max(axis=1), 2500)
    a = _verify(s.dev, qv, dev_pt, steps, 2500)
    b = _verify(s.full, qv, s.pt_d, steps, 2500)
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    assert torch.equal(a, b)


def test_negative_control_writer_that_skips_the_mirror():
    """A token written to its resident slot only (a writer that does not write
    both copies): while the page stays resident the streamed result is still
    right, but once the page is streamed from the mirror the result differs
    from the resident reference -- the check catches the skipped host write."""
    seed = synth.config_seed(4) + 304
    lens = np.array([900], np.int32)
    s = Streamed(k8.FORMAT_K8V4, lens - 1, 64, 15, seed)   # cells 0 .. 898 mirrored, all 15 pages resident
    cell = 899
    hp = int(s.pt[0, cell // 64])
    slot = int(s.slot_of_page[hp])
    assert slot >= 0
    k = synth.kv_values(seed, synth.T_K, 7, 1, H, 3, "bf16")
    v = synth.kv_values(seed, synth.T_V, 7, 1, H, 3, "bf16")
    kk, vv = dev_tensor(synth.Tensor(k.f32[None], "bf16")), dev_tensor(synth.Tensor(v.f32[None], "bf16"))
    pos = torch.tensor([cell], dtype=torch.int64, device="cuda")
    slot_pt = torch.full_like(s.pt_d[:1], -1)
    slot_pt[0, cell // 64] = slot
    k8.kv_append_k8v4(s.dev, slot_pt, pos, kk, vv)        # device slot only: the mirror misses it
    k8.kv_append_k8v4(s.full, s.pt_d, pos, kk, vv)
    q = dev_tensor(synth.q_values(seed, 0, 1, H, "bf16"), (1, 16, 256))
    resident = _decode(s.full, q, s.pt_d, lens, 900)
    hit = _decode(s.dev, q, s.resolve(lens, 900), lens, 900)
    s.slot_of_page[hp] = -1                                 # the page leaves the resident window
    s.sop_d = torch.from_numpy(s.slot_of_page).cuda()
    missed = _decode(s.dev, q, s.resolve(lens, 900), lens, 900)
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    assert torch.equal(hit, resident)
    assert not torch.equal(missed, resident)


def test_resolve_without_enough_staging_is_reported():
    """Two staging slots for more misses: the first two misses are copied, the
    rest are -1 and K8V4_ENOSPACE is recorded; the table still equals the
    oracle's lookups."""
    s = Streamed(k8.FORMAT_K8V4, [640, 320], 64, 3, synth.config_seed(4) + 305)
    s.dev = k8.PagedCache(s.n_res + 2, s.P, H, k8.FORMAT_K8V4)
    lens = np.array([640, 320], np.int32)
    dev_pt = s.resolve(lens, 640)
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == k8.ENOSPACE
    want, moves, over = oracle.stream_resolve(s.pt, lens, s.slot_of_page, s.n_res, s.n_res + 2, s.P, 640)
    assert over and len(moves) == 2
    assert np.array_equal(dev_pt.cpu().numpy(), want)


def test_streamed_decode_238k_with_32k_resident():
    """The 238K workload with a 32,768-cell resident window (512 of 3,712 pages,
    the streaming PR's --kv-resident 32768): streamed decode is bitwise equal to
    resident decode, and the mirror equals the resident cache byte for byte."""
    n_cells, P = 237568, 64
    w = synth.config3(n_cells)
    n_host = w.n_pages
    need = n_cells // P
    host = k8.PagedCache(n_host, P, H, device="pinned")
    full = k8.PagedCache(n_host, P, H)
    n_res = 32768 // P
    slot_of_page = np.full(n_host, -1, np.int32)
    last = w.page_table[0, need - n_res:need]              # the window holds the newest cells
    slot_of_page[last] = np.arange(n_res, dtype=np.int32)
    dev = k8.PagedCache(n_res + need, P, H)
    pt = torch.from_numpy(w.page_table).cuda()
    sop = torch.from_numpy(slot_of_page).cuda()
    kd, vd = dev_tensor(w.k, (1, n_cells, H, 256)), dev_tensor(w.v, (1, n_cells, H, 256))
    z = torch.zeros(1, dtype=torch.int64, device="cuda")
    k8.kv_append_k8v4_mirrored(host, dev, sop, pt, z, kd, vd)
    k8.kv_append_k8v4(full, pt, z, kd, vd)
    q = dev_tensor(w.q, (1, 16, 256))
    lens = np.array([n_cells], np.int32)
    dev_pt = torch.empty_like(pt)
    ws = torch.empty(k8.kv_stream_workspace_bytes(1, pt.shape[1]), dtype=torch.uint8, device="cuda")
    k8.kv_stream_resolve(host, dev, sop, n_res, pt, torch.from_numpy(lens).cuda(), n_cells, dev_pt, ws)
    a = _decode(dev, q, dev_pt, lens, n_cells)
    b = _decode(full, q, pt, lens, n_cells)
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    assert torch.equal(a, b)
    assert torch.equal(host.pages, full.pages.cpu())
