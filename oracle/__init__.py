"""ctypes front end of the k8v4 CPU oracle (k8v4_oracle.c).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The CUDA library never imports it.

Every function restates the cache's arithmetic as described by the hybrid
k8v4 pull request (What section: K as INT8 and V rotated by a Hadamard
transform and stored as Q4_0, 816 B per cell; Tests section: int8 codes round
half to even, the rotated q4_0 rules, attention on the host over the
dequantised K and V) with the readings listed at the top of k8v4_oracle.c.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "k8v4_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "liboracle.so")
CFLAGS = ["-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread",
          "-Wall", "-Wno-unused-function"]

FMT_INT8 = 1
FMT_Q4 = 2
FMT_K8V4 = 3
D = 256
GQA = 8

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host compiler (no fast-math, no FP contraction)."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"], check=True)
        os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(LIB)
            P, I, I64, F, Dd = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
            L.orc_f32_to_f16.argtypes = [F]
            L.orc_f32_to_f16.restype = ctypes.c_uint16
            L.orc_f32_to_f16_array.argtypes = [P, P, I64]
            L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_f16_to_f32.restype = F
            L.orc_hadamard_entry.argtypes = [I, I]
            L.orc_hadamard_entry.restype = I
            L.orc_hadamard_rotate.argtypes = [P, P]
            L.orc_quant_int8.argtypes = [P, I, P, P]
            L.orc_quant_q4_block.argtypes = [P, P, P]
            L.orc_bytes_per_cell_head.argtypes = [I]
            L.orc_bytes_per_cell_head.restype = I64
            L.orc_append.argtypes = [P, I, I, I, P, I64, I, P, I, P, P, I]
            L.orc_append.restype = I
            L.orc_dequant.argtypes = [P, I, I, I, P, I64, I, I64, I64, P, P, P]
            L.orc_dequant.restype = I
            L.orc_attention.argtypes = [P, I, I, I, P, I64, I64, P, P, P, P, Dd, P, I, I]
            L.orc_attention.restype = I
            L.orc_attention_partial.argtypes = [P, I, I, I, P, I64, I64, P, P, P, P, P, Dd, P, P, P, I]
            L.orc_attention_partial.restype = I
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def n_threads_default() -> int:
    return max(1, os.cpu_count() or 1)


# --------------------------------------------------------------------------- scalars

def f32_to_f16_bits(x: float) -> int:
    return int(lib().orc_f32_to_f16(ctypes.c_float(x)))


def f32_to_f16_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().orc_f32_to_f16_array(_ptr(x), _ptr(out), x.size)
    return out


def f16_bits_to_f32(b: int) -> float:
    return float(lib().orc_f16_to_f32(int(b)))


def hadamard_entry(i: int, j: int) -> int:
    return int(lib().orc_hadamard_entry(i, j))


def rotate(x: np.ndarray) -> np.ndarray:
    """y = RN_fp32((H x) / 16) with the sum taken exactly; x: [..., 256] float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    flat = x.reshape(-1, D)
    y = np.empty_like(flat)
    L = lib()
    for r in range(flat.shape[0]):
        L.orc_hadamard_rotate(_ptr(flat[r]), _ptr(y[r]))
    return y.reshape(x.shape)


def quant_int8(x: np.ndarray) -> tuple[np.ndarray, float]:
    x = np.ascontiguousarray(x, dtype=np.float32)
    c = np.empty(x.size, np.int8)
    s = np.zeros(1, np.float32)
    lib().orc_quant_int8(_ptr(x), x.size, _ptr(c), _ptr(s))
    return c, float(s[0])


def quant_q4_block(y: np.ndarray) -> tuple[np.ndarray, int]:
    y = np.ascontiguousarray(y, dtype=np.float32)
    assert y.size == 32
    nib = np.empty(16, np.uint8)
    d = np.zeros(1, np.uint16)
    lib().orc_quant_q4_block(_ptr(y), _ptr(nib), _ptr(d))
    return nib, int(d[0])


def bytes_per_cell_head(fmt: int = FMT_K8V4) -> int:
    return int(lib().orc_bytes_per_cell_head(fmt))


# --------------------------------------------------------------------------- cache

class Cache:
    """A paged cache held in host memory: n_pages pages of P cells, H KV heads."""

    def __init__(self, n_pages: int, P: int, H: int = 2, fmt: int = FMT_K8V4, fill: int = 0):
        self.n_pages, self.P, self.H, self.fmt = n_pages, P, H, fmt
        self.page_bytes = P * H * bytes_per_cell_head(fmt)
        self.buf = np.full(n_pages * self.page_bytes, fill, dtype=np.uint8)

    def append(self, page_table: np.ndarray, pos: np.ndarray, k: np.ndarray, v: np.ndarray,
               n_threads: int | None = None) -> None:
        """k, v: [n_seqs, n_tok, H, 256] float32; cell pos[b] + t of sequence b."""
        pt = np.ascontiguousarray(page_table, dtype=np.int32)
        if pt.ndim == 1:
            pt = pt[None]
        k = np.ascontiguousarray(k, dtype=np.float32)
        v = np.ascontiguousarray(v, dtype=np.float32)
        n_seqs, n_tok = k.shape[0], k.shape[1]
        pos = np.ascontiguousarray(pos, dtype=np.int64)
        assert pt.shape[0] == n_seqs and pos.shape[0] == n_seqs
        need = int((pos + n_tok).max())
        assert need <= pt.shape[1] * self.P
        assert int(pt[:, :((need + self.P - 1) // self.P)].max()) < self.n_pages
        rc = lib().orc_append(_ptr(self.buf), self.fmt, self.P, self.H, _ptr(pt), pt.shape[1], n_seqs,
                              _ptr(pos), n_tok, _ptr(k), _ptr(v), n_threads or n_threads_default())
        assert rc == 0

    def dequant(self, page_table: np.ndarray, start: int, n: int, seq: int = 0, with_v: bool = True):
        pt = np.ascontiguousarray(page_table, dtype=np.int32)
        if pt.ndim == 1:
            pt = pt[None]
        ko = np.empty((n, self.H, D), np.float32)
        vr = np.empty((n, self.H, D), np.float32)
        vo = np.empty((n, self.H, D), np.float32) if with_v else None
        lib().orc_dequant(_ptr(self.buf), self.fmt, self.P, self.H, _ptr(pt), pt.shape[1], seq, start, n,
                          _ptr(ko), _ptr(vr), _ptr(vo))
        return ko, vr, vo

    def attention(self, page_table: np.ndarray, row_seq, row_head, row_vis, q_rows: np.ndarray,
                  sm_scale: float = 1.0 / 16.0, rotate_back: bool = True,
                  n_threads: int | None = None) -> np.ndarray:
        """fp64 attention, one output row per (sequence, query head, visible count)."""
        pt = np.ascontiguousarray(page_table, dtype=np.int32)
        if pt.ndim == 1:
            pt = pt[None]
        rs = np.ascontiguousarray(row_seq, dtype=np.int32)
        rh = np.ascontiguousarray(row_head, dtype=np.int32)
        rv = np.ascontiguousarray(row_vis, dtype=np.int32)
        q = np.ascontiguousarray(q_rows, dtype=np.float32).reshape(-1, D)
        n = rs.shape[0]
        assert rh.shape[0] == n and rv.shape[0] == n and q.shape[0] == n
        out = np.empty((n, D), np.float64)
        lib().orc_attention(_ptr(self.buf), self.fmt, self.P, self.H, _ptr(pt), pt.shape[1], n, _ptr(rs),
                            _ptr(rh), _ptr(rv), _ptr(q), float(sm_scale), _ptr(out), int(rotate_back),
                            n_threads or n_threads_default())
        return out


    def attention_partial(self, page_table: np.ndarray, row_seq, row_head, row_lo, row_hi, q_rows: np.ndarray,
                          sm_scale: float = 1.0 / 16.0, n_threads: int | None = None):
        """fp64 partial attention over cells [row_lo, row_hi) per row: (o, m, l)
        with o un-rotated and unnormalised, m the natural-log maximum score."""
        pt = np.ascontiguousarray(page_table, dtype=np.int32)
        if pt.ndim == 1:
            pt = pt[None]
        rs, rh = np.ascontiguousarray(row_seq, np.int32), np.ascontiguousarray(row_head, np.int32)
        lo, hi = np.ascontiguousarray(row_lo, np.int32), np.ascontiguousarray(row_hi, np.int32)
        q = np.ascontiguousarray(q_rows, dtype=np.float32).reshape(-1, D)
        n = rs.shape[0]
        assert rh.shape[0] == n and lo.shape[0] == n and hi.shape[0] == n and q.shape[0] == n
        o = np.empty((n, D), np.float64)
        m = np.empty(n, np.float64)
        lsum = np.empty(n, np.float64)
        lib().orc_attention_partial(_ptr(self.buf), self.fmt, self.P, self.H, _ptr(pt), pt.shape[1], n, _ptr(rs),
                                    _ptr(rh), _ptr(lo), _ptr(hi), _ptr(q), float(sm_scale), _ptr(o), _ptr(m),
                                    _ptr(lsum), n_threads or n_threads_default())
        return o, m, lsum


def stream_resolve(page_table: np.ndarray, seq_lens, slot_of_page, n_resident: int, n_dev_pages: int, P: int,
                   max_seq_len: int):
    """Block lookups of one streamed attention call, from the streaming pull
    request ("kv: --kv k8v4 streams with --kv-resident", "How" and "Tests"): every
    page a sequence reads is looked up; a page resident in VRAM is read from its
    slot, a miss is copied from the host copy into a VRAM staging slot.

    Readings (the pages give the mechanism, not an order): lookups run in
    (sequence, page index) order over the pages that hold a sequence's first
    min(seq_lens[b], max_seq_len) cells; the r-th miss takes staging slot
    n_resident + r; a miss with no staging slot left (n_resident + r >=
    n_dev_pages) is not read (-1) and reported; table entries no cell reaches are
    -1.  Returns (device page table, [(host page, slot)] copies, overflow)."""
    page_table = np.asarray(page_table)
    n_seqs, max_pages = page_table.shape
    dev = np.full((n_seqs, max_pages), -1, np.int32)
    moves = []
    rank = 0
    overflow = False
    for b in range(n_seqs):
        n = min(max(int(seq_lens[b]), 0), max_seq_len)
        for i in range((n + P - 1) // P):
            hp = int(page_table[b, i])
            s = int(slot_of_page[hp])
            if s >= 0:
                dev[b, i] = s
                continue
            slot = n_resident + rank
            rank += 1
            if slot < n_dev_pages:
                dev[b, i] = slot
                moves.append((hp, slot))
            else:
                overflow = True
    return dev, moves, overflow


def decode_rows(n_seqs: int, n_q_heads: int, seq_lens) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Row descriptors for decode: row (b, h) sees seq_lens[b] cells."""
    b = np.repeat(np.arange(n_seqs), n_q_heads)
    h = np.tile(np.arange(n_q_heads), n_seqs)
    v = np.repeat(np.asarray(seq_lens), n_q_heads)
    return b.astype(np.int32), h.astype(np.int32), v.astype(np.int32)


def multi_query_rows(steps: np.ndarray, n_q_heads: int) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Row descriptors for verify / prefill: steps[b, i] cells visible to query i of
    sequence b; rows ordered (b, i, h)."""
    steps = np.asarray(steps)
    n_seqs, n_q = steps.shape
    b = np.repeat(np.arange(n_seqs), n_q * n_q_heads)
    h = np.tile(np.arange(n_q_heads), n_seqs * n_q)
    v = np.repeat(steps.reshape(-1), n_q_heads)
    return b.astype(np.int32), h.astype(np.int32), v.astype(np.int32)
