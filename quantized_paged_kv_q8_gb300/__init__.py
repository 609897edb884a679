"""Python binding of libk8v4.so -- the k8v4 quantized paged KV cache and its
fused attention on one GB300 (sm_103a).

Argument marshalling only: every step runs in the library's CUDA kernels.  The
functions carry the C ABI's names (include/k8v4.h); tensors are torch CUDA
tensors (PyTorch provides device memory and streams, nothing else).  If the
compiled library is missing this module raises on first use -- there is no CPU
or PyTorch fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libk8v4.so")

OK, EINVAL, ERANGE, EALIGN, ECUDA, EDEVICE, ENOSPACE = 0, -1, -2, -3, -4, -5, -6
F32, BF16 = 0, 1
FORMAT_INT8, FORMAT_Q4, FORMAT_K8V4 = 1, 2, 3
HEAD_DIM = 256
GQA = 8


class K8V4Error(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


class k8v4_cache(ctypes.Structure):
    _fields_ = [("pages", ctypes.c_void_p), ("n_pages", ctypes.c_int64), ("page_size", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("format", ctypes.c_int32)]


_lib = None


def build(force: bool = False) -> str:
    from . import buildlib
    return buildlib.build(force=force)


def lib():
    """The loaded libk8v4.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libk8v4.so is not built ({LIB_PATH}); call quantized_paged_kv_q8_gb300.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, I64, F, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        C = ctypes.POINTER(k8v4_cache)
        sigs = {
            "k8v4_bytes_per_cell": ([I32, I32], SZ),
            "k8v4_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "k8v4_device_check": ([], ctypes.c_int),
            "kv_append_k8v4": ([C, P, I64, I32, P, I32, P, P, I32, P], ctypes.c_int),
            "attn_k8v4_workspace_bytes": ([C, I32, I32, I32], SZ),
            "attn_k8v4_decode": ([C, P, I32, P, I64, P, I32, I32, F, P, P, SZ, P], ctypes.c_int),
            "attn_k8v4_decode_noalloc": ([C, P, I32, P, I64, P, I32, I32, F, P, P], ctypes.c_int),
            "attn_k8v4_decode_step": ([C, P, I32, P, P, I32, P, I64, P, I32, I32, F, P, P, SZ, P], ctypes.c_int),
            "attn_k8v4_verify": ([C, P, I32, P, I64, P, I32, I32, I32, F, P, P, SZ, P], ctypes.c_int),
            "attn_k8v4_prefill": ([C, P, I32, P, I64, I32, I32, P, F, P, P], ctypes.c_int),
            "kv_dequant_k8v4": ([C, P, I64, I64, I64, P, P, P, P], ctypes.c_int),
            "k8v4_last_device_status": ([P], ctypes.c_int),
            "kv_append_k8v4_mirrored": ([C, C, P, P, I64, I32, P, I32, P, P, I32, P], ctypes.c_int),
            "kv_stream_workspace_bytes": ([I32, I64], SZ),
            "kv_stream_resolve": ([C, C, P, I32, P, I64, P, I32, I32, P, P, SZ, P], ctypes.c_int),
            "kv_stream_copy": ([C, C, P, I32, P], ctypes.c_int),
            "attn_k8v4_partial_workspace_bytes": ([C, I32, I32, I32], SZ),
            "attn_k8v4_decode_partial": ([C, P, I32, P, I64, P, I32, I32, I32, I32, F, P, P, SZ, P], ctypes.c_int),
            "attn_k8v4_combine_partials": ([P, I32, I32, I32, P, P], ctypes.c_int),
            "k8v4_set_wait_limit_ns": ([ctypes.c_uint32], None),
            "k8v4_set_withheld_copy": ([ctypes.c_int32], None),
        }
        for name, (args, res) in sigs.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


EXPORTED = ("k8v4_bytes_per_cell", "k8v4_status_string", "k8v4_device_check", "kv_append_k8v4",
            "attn_k8v4_workspace_bytes", "attn_k8v4_decode", "attn_k8v4_decode_noalloc", "attn_k8v4_decode_step",
            "attn_k8v4_verify",
            "attn_k8v4_prefill",
            "kv_dequant_k8v4", "k8v4_last_device_status",
            "kv_append_k8v4_mirrored", "kv_stream_workspace_bytes", "kv_stream_resolve", "kv_stream_copy",
            "attn_k8v4_partial_workspace_bytes", "attn_k8v4_decode_partial", "attn_k8v4_combine_partials",
            "k8v4_set_wait_limit_ns", "k8v4_set_withheld_copy")


def status_string(code: int) -> str:
    try:
        return lib().k8v4_status_string(int(code)).decode()
    except Exception:  # noqa: BLE001 - message formatting only
        return "status"


def _check(rc: int, what: str) -> None:
    if rc != OK:
        raise K8V4Error(rc, what)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def k8v4_bytes_per_cell(fmt: int = FORMAT_K8V4, n_kv_heads: int = 2) -> int:
    return int(lib().k8v4_bytes_per_cell(fmt, n_kv_heads))


def k8v4_device_check() -> int:
    return int(lib().k8v4_device_check())


class PagedCache:
    """A caller-owned paged cache: `pages` is one uint8 CUDA tensor of
    n_pages * page_size * bytes_per_cell bytes; `desc` is the C descriptor."""

    def __init__(self, n_pages: int, page_size: int, n_kv_heads: int = 2, fmt: int = FORMAT_K8V4,
                 device: str | torch.device = "cuda", pages: torch.Tensor | None = None):
        """device="pinned" allocates the pages in page-locked host memory: the
        host mirror of a streamed cache."""
        self.n_pages, self.page_size, self.n_kv_heads, self.fmt = n_pages, page_size, n_kv_heads, fmt
        self.bytes_per_cell = k8v4_bytes_per_cell(fmt, n_kv_heads)
        self.page_bytes = page_size * self.bytes_per_cell
        nbytes = n_pages * self.page_bytes
        if pages is None and device == "pinned":
            pages = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
            pages.zero_()
        elif pages is None:
            pages = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        assert pages.dtype == torch.uint8 and pages.numel() == nbytes and pages.is_contiguous()
        self.pages = pages
        self.desc = k8v4_cache(ctypes.c_void_p(pages.data_ptr()), n_pages, page_size, n_kv_heads, HEAD_DIM, fmt)

    def ref(self):
        return ctypes.byref(self.desc)


def kv_append_k8v4(cache: PagedCache, page_table: torch.Tensor, pos: torch.Tensor, k: torch.Tensor,
                   v: torch.Tensor, stream=None) -> None:
    """k, v: [n_seqs, n_tok, H, 256] (bf16 or f32); page_table int32 [n_seqs, max_pages];
    pos int64 [n_seqs]."""
    n_seqs, n_tok = k.shape[0], k.shape[1]
    assert k.shape == v.shape and k.dtype == v.dtype and k.is_contiguous() and v.is_contiguous()
    assert page_table.dtype == torch.int32 and pos.dtype == torch.int64
    rc = lib().kv_append_k8v4(cache.ref(), _ptr(page_table), page_table.shape[-1], n_seqs, _ptr(pos), n_tok,
                              _ptr(k), _ptr(v), _dtype(k), _stream(stream))
    _check(rc, "kv_append_k8v4")


def attn_k8v4_workspace_bytes(cache: PagedCache, n_seqs: int, n_q: int, max_seq_len: int) -> int:
    return int(lib().attn_k8v4_workspace_bytes(cache.ref(), n_seqs, n_q, max_seq_len))


def workspace(cache: PagedCache, n_seqs: int, n_q: int, max_seq_len: int, device="cuda") -> torch.Tensor:
    n = attn_k8v4_workspace_bytes(cache, n_seqs, n_q, max_seq_len)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def attn_k8v4_decode(cache: PagedCache, q: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                     max_seq_len: int, out: torch.Tensor, ws: torch.Tensor, sm_scale: float = 1.0 / 16.0,
                     stream=None) -> torch.Tensor:
    """q: [n_seqs, 8H, 256]; seq_lens int32 [n_seqs]; out float32 [n_seqs, 8H, 256]."""
    assert q.is_contiguous() and out.is_contiguous() and out.dtype == torch.float32
    rc = lib().attn_k8v4_decode(cache.ref(), _ptr(q), _dtype(q), _ptr(page_table), page_table.shape[-1],
                                _ptr(seq_lens), q.shape[0], max_seq_len, sm_scale, _ptr(out), _ptr(ws),
                                ws.numel(), _stream(stream))
    _check(rc, "attn_k8v4_decode")
    return out


def attn_k8v4_decode_step(cache: PagedCache, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                          page_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int, out: torch.Tensor,
                          ws: torch.Tensor, sm_scale: float = 1.0 / 16.0, stream=None) -> torch.Tensor:
    """Append each sequence's newest token (k_new, v_new: [n_seqs, H, 256], at cell
    seq_lens[b] - 1) and decode over seq_lens[b] cells, in one call."""
    assert q.is_contiguous() and out.is_contiguous() and out.dtype == torch.float32
    assert k_new.is_contiguous() and v_new.is_contiguous() and k_new.dtype == v_new.dtype
    rc = lib().attn_k8v4_decode_step(cache.ref(), _ptr(q), _dtype(q), _ptr(k_new), _ptr(v_new), _dtype(k_new),
                                     _ptr(page_table), page_table.shape[-1], _ptr(seq_lens), q.shape[0],
                                     max_seq_len, sm_scale, _ptr(out), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "attn_k8v4_decode_step")
    return out


def attn_k8v4_verify(cache: PagedCache, q: torch.Tensor, page_table: torch.Tensor, step_arrays: torch.Tensor,
                     max_seq_len: int, out: torch.Tensor, ws: torch.Tensor, sm_scale: float = 1.0 / 16.0,
                     stream=None) -> torch.Tensor:
    """q: [n_seqs, n_q, 8H, 256]; step_arrays int32 [n_seqs, n_q]; out float32 like q."""
    assert q.is_contiguous() and out.is_contiguous() and out.dtype == torch.float32
    rc = lib().attn_k8v4_verify(cache.ref(), _ptr(q), _dtype(q), _ptr(page_table), page_table.shape[-1],
                                _ptr(step_arrays), q.shape[0], q.shape[1], max_seq_len, sm_scale, _ptr(out),
                                _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "attn_k8v4_verify")
    return out


def attn_k8v4_prefill(cache: PagedCache, q: torch.Tensor, page_table: torch.Tensor, seq_len: int,
                      out: torch.Tensor, step_arrays: torch.Tensor | None = None, sm_scale: float = 1.0 / 16.0,
                      stream=None) -> torch.Tensor:
    """q: bf16 [n_q_tok, 8H, 256]; page_table int32 [max_pages]; out float32 like q."""
    assert q.is_contiguous() and out.is_contiguous() and out.dtype == torch.float32
    rc = lib().attn_k8v4_prefill(cache.ref(), _ptr(q), _dtype(q), _ptr(page_table), page_table.shape[-1],
                                 seq_len, q.shape[0], _ptr(step_arrays), sm_scale, _ptr(out), _stream(stream))
    _check(rc, "attn_k8v4_prefill")
    return out


def kv_dequant_k8v4(cache: PagedCache, page_table: torch.Tensor, start: int, n_cells: int, k_out: torch.Tensor,
                    v_rot_out: torch.Tensor, v_out: torch.Tensor | None = None, stream=None) -> None:
    rc = lib().kv_dequant_k8v4(cache.ref(), _ptr(page_table), page_table.shape[-1], start, n_cells, _ptr(k_out),
                               _ptr(v_rot_out), _ptr(v_out), _stream(stream))
    _check(rc, "kv_dequant_k8v4")


def kv_append_k8v4_mirrored(host: PagedCache, dev: PagedCache, slot_of_page: torch.Tensor, page_table: torch.Tensor,
                            pos: torch.Tensor, k: torch.Tensor, v: torch.Tensor, stream=None) -> None:
    """Append to a streamed cache: page_table holds host page ids; every row goes to
    the pinned mirror `host` and, where slot_of_page[page] >= 0, to that slot of `dev`."""
    n_seqs, n_tok = k.shape[0], k.shape[1]
    assert k.shape == v.shape and k.dtype == v.dtype and k.is_contiguous() and v.is_contiguous()
    assert page_table.dtype == torch.int32 and pos.dtype == torch.int64 and slot_of_page.dtype == torch.int32
    rc = lib().kv_append_k8v4_mirrored(host.ref(), dev.ref(), _ptr(slot_of_page), _ptr(page_table),
                                       page_table.shape[-1], n_seqs, _ptr(pos), n_tok, _ptr(k), _ptr(v), _dtype(k),
                                       _stream(stream))
    _check(rc, "kv_append_k8v4_mirrored")


def kv_stream_workspace_bytes(n_seqs: int, max_pages: int) -> int:
    return int(lib().kv_stream_workspace_bytes(n_seqs, max_pages))


def kv_stream_resolve(host: PagedCache, dev: PagedCache, slot_of_page: torch.Tensor, n_resident: int,
                      page_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                      dev_page_table: torch.Tensor, ws: torch.Tensor, stream=None) -> torch.Tensor:
    """Look up the pages each sequence reads (resident slot, or a copy from the
    mirror into a staging slot) and write the device page table."""
    assert page_table.dtype == torch.int32 and dev_page_table.shape == page_table.shape
    rc = lib().kv_stream_resolve(host.ref(), dev.ref(), _ptr(slot_of_page), n_resident, _ptr(page_table),
                                 page_table.shape[-1], _ptr(seq_lens), page_table.shape[0], max_seq_len,
                                 _ptr(dev_page_table), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "kv_stream_resolve")
    return dev_page_table


def kv_stream_copy(host: PagedCache, dev: PagedCache, pages: torch.Tensor, stream=None) -> None:
    """Copy host pages pages[i, 0] into device slots pages[i, 1]."""
    assert pages.dtype == torch.int32 and pages.is_contiguous() and pages.shape[-1] == 2
    rc = lib().kv_stream_copy(host.ref(), dev.ref(), _ptr(pages), pages.shape[0], _stream(stream))
    _check(rc, "kv_stream_copy")


def k8v4_last_device_status(stream=None) -> int:
    return int(lib().k8v4_last_device_status(_stream(stream)))


# ---------------------------------------------------------------- split across GPUs
PARTIAL_ROW = 260      # floats per partial row: o[256], m (base-2 exponent), l, 2 unused


def cell_ranges(max_seq_len: int, world: int, align: int = 16) -> list[tuple[int, int]]:
    """Split cells [0, max_seq_len) into `world` contiguous ranges of whole
    16-cell tiles, as even as the tiles allow; the last range ends at
    max_seq_len (possibly past a shorter sequence's length, which is fine)."""
    assert world >= 1 and max_seq_len >= 0
    tiles = (max_seq_len + align - 1) // align
    bounds = [align * ((tiles * r) // world) for r in range(world)] + [max_seq_len]
    return [(min(bounds[r], max_seq_len), bounds[r + 1] if r + 1 < world else max_seq_len) for r in range(world)]


def attn_k8v4_partial_workspace_bytes(cache: PagedCache, n_seqs: int, cell_begin: int, cell_end: int) -> int:
    return int(lib().attn_k8v4_partial_workspace_bytes(cache.ref(), n_seqs, cell_begin, cell_end))


def partial_workspace(cache: PagedCache, n_seqs: int, cell_begin: int, cell_end: int, device="cuda") -> torch.Tensor:
    n = attn_k8v4_partial_workspace_bytes(cache, n_seqs, cell_begin, cell_end)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def attn_k8v4_decode_partial(cache: PagedCache, q: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                             max_seq_len: int, cell_begin: int, cell_end: int, partial: torch.Tensor,
                             ws: torch.Tensor, sm_scale: float = 1.0 / 16.0, stream=None) -> torch.Tensor:
    """Decode over cells [cell_begin, cell_end) only; partial: float32
    [n_seqs, 8H, 260] (o[256] unnormalised, m, l)."""
    assert q.is_contiguous() and partial.is_contiguous() and partial.dtype == torch.float32
    assert partial.shape[-1] == PARTIAL_ROW
    rc = lib().attn_k8v4_decode_partial(cache.ref(), _ptr(q), _dtype(q), _ptr(page_table), page_table.shape[-1],
                                        _ptr(seq_lens), q.shape[0], max_seq_len, cell_begin, cell_end, sm_scale,
                                        _ptr(partial), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "attn_k8v4_decode_partial")
    return partial


def attn_k8v4_combine_partials(parts: torch.Tensor, out: torch.Tensor, stream=None) -> torch.Tensor:
    """parts: float32 [n_parts, n_seqs, rows, 260] -> out float32 [n_seqs, rows, 256]."""
    assert parts.is_contiguous() and out.is_contiguous() and parts.dtype == torch.float32
    n_parts, n_seqs, rows = parts.shape[0], parts.shape[1], parts.shape[2]
    assert parts.shape[3] == PARTIAL_ROW and tuple(out.shape) == (n_seqs, rows, HEAD_DIM)
    rc = lib().attn_k8v4_combine_partials(_ptr(parts), n_parts, n_seqs, rows, _ptr(out), _stream(stream))
    _check(rc, "attn_k8v4_combine_partials")
    return out


def decode_across_ranks(cache: PagedCache, q: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                        max_seq_len: int, out: torch.Tensor, group=None, sm_scale: float = 1.0 / 16.0,
                        stream=None) -> torch.Tensor:
    """Decode split by cell range across the ranks of `group` (one GPU each,
    every rank holding the same cache layout and page table): rank r attends
    over its range of cell_ranges(max_seq_len, world), the partial rows are
    all-gathered (n_seqs * 8H * 260 floats per rank), and every rank merges
    them into `out`."""
    import torch.distributed as dist
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    lo, hi = cell_ranges(max_seq_len, world)[rank]
    n_seqs, rows = q.shape[0], q.shape[1]
    part = torch.empty(n_seqs, rows, PARTIAL_ROW, dtype=torch.float32, device=q.device)
    ws = partial_workspace(cache, n_seqs, lo, hi, device=q.device)
    attn_k8v4_decode_partial(cache, q, page_table, seq_lens, max_seq_len, lo, hi, part, ws, sm_scale, stream)
    return attn_k8v4_combine_partials(gather_partials(part, group), out, stream)


def gather_partials(part: torch.Tensor, group=None) -> torch.Tensor:
    """The exchange step of the cell-range split: every rank's partial rows
    [n_seqs, rows, 260] stacked in rank order, [world, n_seqs, rows, 260]
    (an all-gather; any torch.distributed backend, NCCL on GPUs)."""
    import torch.distributed as dist
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    parts = torch.empty((world,) + tuple(part.shape), dtype=part.dtype, device=part.device)
    if world > 1:
        dist.all_gather(list(parts.unbind(0)), part.contiguous(), group=group)
    else:
        parts[0].copy_(part)
    return parts


def k8v4_set_wait_limit_ns(ns: int) -> None:
    """Failure-handling diagnostics: bound of every mbarrier wait (0: default)."""
    lib().k8v4_set_wait_limit_ns(int(ns))


def k8v4_set_withheld_copy(on: bool) -> None:
    """Failure-handling diagnostics: the TMA decode kernel withholds one tile's copies."""
    lib().k8v4_set_withheld_copy(1 if on else 0)
