"""Seeded synthetic inputs for the k8v4 cache: the one module both the CPU oracle
and the CUDA path are fed from.

It produces inputs only (K/V/q values, page tables, lengths, step arrays) and
holds none of the cache's arithmetic: no quantiser, no rotation, no attention.

Generator (stated once, used everywhere):
  * SplitMix64 as a counter-based generator: value i of stream (seed, sid) is
    mix(seed + sid * 0xD1B54A32D192ED03 + (i + 1) * 0x9E3779B97F4A7C15), where mix
    is the published SplitMix64 finaliser.
  * uniform u = ((z >> 11) + 1) * 2^-53, in (0, 1].
  * Box-Muller on consecutive pairs (u1, u2): sqrt(-2 ln u1) * (cos, sin)(2 pi u2)
    in float64.
  * outlier channels: chosen without replacement per (tensor, KV head) by a
    Fisher-Yates draw, fixed across cells, multiplied by 20 before rounding.
  * rounding: float64 -> float32 (round to nearest even); bf16 inputs then round
    the float32 value to bf16 (round to nearest even on the bit pattern).

The workloads mirror the five k8v4 configurations: the tiny fp32 round trip,
single-sequence decode at 32,768 cells, the long-context sweep, the 8-sequence
speculative verify, and the 8,192-token chunked prefill at offset 229,376.
"""
from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
SID_MUL = np.uint64(0xD1B54A32D192ED03)
D = 256          # head_dim
GQA = 8          # query heads per KV head
MASTER_SEED = 0x6B38763400

# stream tags
T_K, T_V, T_Q, T_OUTK, T_OUTV, T_PT, T_LEN, T_POOL = 1, 2, 3, 4, 5, 6, 7, 8


def config_seed(k: int) -> int:
    return MASTER_SEED + int(k)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def stream_id(tag: int, a: int = 0, b: int = 0) -> int:
    return ((int(tag) & 0xFF) << 48) | ((int(a) & 0xFFFFFF) << 24) | (int(b) & 0xFFFFFF)


def raw_u64(seed: int, sid: int, start: int, n: int) -> np.ndarray:
    with np.errstate(over="ignore"):
        base = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + np.uint64(sid) * SID_MUL
        idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        return _mix(base + idx * GOLDEN)


def uniform(seed: int, sid: int, start: int, n: int) -> np.ndarray:
    z = raw_u64(seed, sid, start, n)
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normal(seed: int, sid: int, n: int, start_pair: int = 0) -> np.ndarray:
    """n standard normals (float64) from stream sid; pair p uses counters 2p, 2p+1."""
    npairs = (n + 1) // 2
    u = uniform(seed, sid, 2 * start_pair, 2 * npairs)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * np.pi * u2
    out = np.empty(2 * npairs, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out[:n]


def randint_below(seed: int, sid: int, start: int, bounds: np.ndarray) -> np.ndarray:
    """Uniform integers in [0, bound) (multiply-shift on the top 32 bits)."""
    bounds = np.asarray(bounds, dtype=np.uint64)
    z = raw_u64(seed, sid, start, bounds.size) >> np.uint64(32)
    return ((z * bounds) >> np.uint64(32)).astype(np.int64)


def permutation(seed: int, sid: int, n: int) -> np.ndarray:
    """Fisher-Yates shuffle of range(n)."""
    perm = np.arange(n, dtype=np.int64)
    if n <= 1:
        return perm
    bounds = np.arange(n, 1, -1, dtype=np.uint64)          # i+1 for i = n-1 .. 1
    r = randint_below(seed, sid, 0, bounds)
    for k, i in enumerate(range(n - 1, 0, -1)):
        j = int(r[k])
        perm[i], perm[j] = perm[j], perm[i]
    return perm


def choose_channels(seed: int, sid: int, count: int, n: int = D) -> np.ndarray:
    return np.sort(permutation(seed, sid, n)[:count])


def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


class Tensor:
    """A synthetic input in both forms: `f32` (exact float32 values, what the oracle
    reads) and `dev` (the bytes handed to the device: float32 or bf16 bits)."""

    def __init__(self, f32: np.ndarray, dtype: str):
        self.dtype = dtype
        if dtype == "bf16":
            self.dev = f32_to_bf16_bits(f32)
            self.f32 = bf16_bits_to_f32(self.dev).reshape(f32.shape)
            self.dev = self.dev.reshape(f32.shape)
        else:
            self.f32 = np.ascontiguousarray(f32, dtype=np.float32)
            self.dev = self.f32

    @property
    def shape(self):
        return self.f32.shape


def kv_values(seed: int, tag: int, seq: int, n_cells: int, n_kv: int, n_out: int,
              dtype: str, cell0: int = 0, outlier_scale: float = 20.0) -> Tensor:
    """[n_cells, n_kv, 256] N(0,1) values, n_out outlier channels per KV head x20.

    Cell c of sequence `seq` always draws the same numbers, whatever cell0/n_cells
    slice is asked for (pairs are indexed by absolute cell), so a history and a
    later chunk of one sequence come from one stream."""
    x = normal(seed, stream_id(tag, seq), n_cells * n_kv * D, start_pair=cell0 * n_kv * D // 2)
    x = x.reshape(n_cells, n_kv, D)
    if n_out:
        for g in range(n_kv):
            ch = choose_channels(seed, stream_id(T_OUTK if tag == T_K else T_OUTV, seq, g), n_out)
            x[:, g, ch] *= outlier_scale
    return Tensor(x.astype(np.float32), dtype)


def q_values(seed: int, seq: int, n_q: int, n_kv: int, dtype: str) -> Tensor:
    x = normal(seed, stream_id(T_Q, seq), n_q * n_kv * GQA * D).reshape(n_q, n_kv * GQA, D)
    return Tensor(x.astype(np.float32), dtype)


# ----------------------------------------------------------------------------
# hand-placed exact cases for the fp32 round trip (cells 0-3)
# ----------------------------------------------------------------------------

def _sylvester(n: int = D) -> np.ndarray:
    i = np.arange(n)
    bits = np.bitwise_and.outer(i, i)
    pc = np.zeros_like(bits)
    b = bits.copy()
    while b.any():
        pc += b & 1
        b >>= 1
    return np.where(pc % 2 == 0, 1, -1).astype(np.int64)


def tie_cells() -> tuple[np.ndarray, np.ndarray]:
    """K and V values [4, 2, 256] (float32) holding exact ties.

    K: a half whose absmax is 127 * 2^k has scale exactly 2^k, so x = (n + 1/2) 2^k
    sits on a rounding tie.  V: rotated-domain blocks are chosen first (dyadic,
    sparse) and the input is x = (H/16) y, which is exact in float32, so the
    rotation returns y exactly and the Q4_0 ties land where placed."""
    k = np.zeros((4, 2, D), dtype=np.float64)
    v_rot = np.zeros((4, 2, D), dtype=np.float64)
    # cell 0, head 0, half 0: s = 2^-4
    s = 2.0 ** -4
    k[0, 0, 0] = 127 * s
    for i, n in enumerate([2.5, -2.5, 126.5, 3.5, -3.5, 0.5, 1.5, -0.5, 125.5, -126.5]):
        k[0, 0, 1 + i] = n * s
    # cell 0, head 0, half 1: s = 1
    k[0, 0, 128] = -127.0
    for i, n in enumerate([0.5, 1.5, -1.5, 125.5, 2.5, 64.5, -64.5]):
        k[0, 0, 129 + i] = n
    # cell 0, head 1: half 0 all zero (s = 0), half 1 s = 2^3
    k[0, 1, 128] = 127 * 8.0
    k[0, 1, 129:133] = [0.5 * 8, 1.5 * 8, 2.5 * 8, -2.5 * 8]
    # cells 1-3: smooth random-ish ties at other scales
    for c in range(1, 4):
        for g in range(2):
            for h in range(2):
                sc = 2.0 ** (c - 3 + g - h)
                base = 128 * h
                k[c, g, base] = 127 * sc * (1 if (c + g) % 2 == 0 else -1)
                for i in range(1, 40):
                    k[c, g, base + i] = (((i * 7 + c * 3) % 120) - 60 + 0.5) * sc
    # V, rotated domain. cell 0 head 0 block 0: m = -8 -> d = 1
    y = v_rot
    y[0, 0, 0] = -8.0
    y[0, 0, 1:5] = [2.5, 3.5, -0.5, 7.5]
    y[0, 0, 5:9] = [-2.5, 0.5, 1.5, -7.5]
    # block 1: m = +8 -> d = -1
    y[0, 0, 32] = 8.0
    y[0, 0, 33:37] = [2.5, -7.5, 4.5, -4.5]
    # block 2: |y| tie between +4 (first) and -4 -> m = +4, d = -0.5
    y[0, 0, 64 + 3] = 4.0
    y[0, 0, 64 + 10] = -4.0
    y[0, 0, 64 + 11] = 1.25
    # block 3: m = -2 -> d = 0.25; 0.375/0.25 = 1.5 -> 2
    y[0, 0, 96] = -2.0
    y[0, 0, 97:101] = [0.375, 0.625, -0.125, 1.875]
    # head 1 block 7 only (others zero -> d == 0)
    y[0, 1, 224] = 16.0
    y[0, 1, 225:229] = [5.0, -3.0, 6.0, 10.0]
    # cells 1-3: a couple of ties per head at varying scales
    for c in range(1, 4):
        for g in range(2):
            sc = 2.0 ** (c - 2 - g)
            b0 = 32 * ((c + g) % 8)
            y[c, g, b0] = -8 * sc
            y[c, g, b0 + 1:b0 + 5] = [0.5 * sc, 1.5 * sc, -2.5 * sc, 6.5 * sc]
    H = _sylvester()
    v = np.einsum("ij,cgj->cgi", H.astype(np.float64), y) / 16.0
    assert np.all(v.astype(np.float32).astype(np.float64) == v)   # exact in float32
    return k.astype(np.float32), v.astype(np.float32)


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------

class Workload:
    """Everything one configuration feeds to both sides."""

    def __init__(self, **kw):
        self.__dict__.update(kw)


def page_table_shuffled(seed: int, sid: int, n_pages_needed: int, pool: int) -> np.ndarray:
    perm = permutation(seed, sid, pool)
    return perm[:n_pages_needed].astype(np.int32)


def config1(seed: int | None = None) -> Workload:
    """Tiny fp32 round trip: 1 seq, 1,024 cells, P=16, 64 pages used out of an
    80-page pool (16 canary pages), 4 outlier channels/head x20, ties in cells 0-3,
    one fp32 decode query."""
    seed = config_seed(1) if seed is None else seed
    n, P, H = 1024, 16, 2
    k = kv_values(seed, T_K, 0, n, H, 4, "f32")
    v = kv_values(seed, T_V, 0, n, H, 4, "f32")
    tk, tv = tie_cells()
    k.f32[:4] = tk
    v.f32[:4] = tv
    k = Tensor(k.f32, "f32")
    v = Tensor(v.f32, "f32")
    pool = 80
    pt = page_table_shuffled(seed, stream_id(T_PT, 0), n // P, pool)
    q = q_values(seed, 0, 1, H, "f32")
    return Workload(name="tiny_roundtrip_1024", seed=seed, n_seqs=1, page_size=P, n_kv=H,
                    n_pages=pool, max_pages=n // P, page_table=pt.reshape(1, -1),
                    seq_lens=np.array([n], np.int32), pos=np.array([0], np.int64),
                    k=k, v=v, q=q, dtype="f32")


def decode_workload(seed: int, n_cells: int, P: int = 64, dtype: str = "bf16", n_out: int = 3,
                    name: str = "") -> Workload:
    """Single sequence, shuffled page table over exactly the pages needed."""
    H = 2
    n_pages = (n_cells + P - 1) // P
    k = kv_values(seed, T_K, 0, n_cells, H, n_out, dtype)
    v = kv_values(seed, T_V, 0, n_cells, H, n_out, dtype)
    pt = page_table_shuffled(seed, stream_id(T_PT, 0), n_pages, n_pages)
    q = q_values(seed, 0, 1, H, dtype)
    return Workload(name=name or f"decode_{n_cells}", seed=seed, n_seqs=1, page_size=P, n_kv=H,
                    n_pages=n_pages, max_pages=n_pages, page_table=pt.reshape(1, -1),
                    seq_lens=np.array([n_cells], np.int32), pos=np.array([0], np.int64),
                    k=k, v=v, q=q, dtype=dtype)


def config2(seed: int | None = None) -> Workload:
    seed = config_seed(2) if seed is None else seed
    return decode_workload(seed, 32768, name="decode_32768")


CONFIG3_LENGTHS = (14848, 118784, 237568, 262144)


def config3(n_cells: int, seed: int | None = None) -> Workload:
    seed = config_seed(3) if seed is None else seed
    return decode_workload(seed, n_cells, name=f"decode_{n_cells}")


def verify_lengths(seed: int, n_seqs: int = 8, lo: int = 16384, hi: int = 65536) -> np.ndarray:
    return (lo + randint_below(seed, stream_id(T_LEN), 0, np.full(n_seqs, hi - lo + 1))).astype(np.int32)


def interleaved_pool(seed: int, lens: np.ndarray, P: int) -> tuple[np.ndarray, int]:
    """Pages handed out round-robin across sequences from one pool, then the
    physical ids permuted: page_table[b, j] for each sequence's j-th page."""
    need = (lens + P - 1) // P
    max_pages = int(need.max())
    order = []
    for j in range(max_pages):
        for b in range(len(lens)):
            if j < need[b]:
                order.append((b, j))
    n_pages = len(order)
    perm = permutation(seed, stream_id(T_POOL), n_pages)
    pt = np.zeros((len(lens), max_pages), np.int32)
    for slot, (b, j) in enumerate(order):
        pt[b, j] = perm[slot]
    return pt, n_pages


def config4(seed: int | None = None, lens: np.ndarray | None = None, n_q: int = 5) -> Workload:
    """Speculative verify: 8 sequences, lengths U[16384, 65536], 5 queries each,
    query i sees len - (n_q - 1) + i cells; pages interleaved in a shared pool."""
    seed = config_seed(4) if seed is None else seed
    P, H = 64, 2
    lens = verify_lengths(seed) if lens is None else np.asarray(lens, np.int32)
    pt, n_pages = interleaved_pool(seed, lens, P)
    ks, vs, qs = [], [], []
    for b, n in enumerate(lens):
        ks.append(kv_values(seed, T_K, b, int(n), H, 3, "bf16"))
        vs.append(kv_values(seed, T_V, b, int(n), H, 3, "bf16"))
        qs.append(q_values(seed, b, n_q, H, "bf16"))
    steps = (lens[:, None] - (n_q - 1) + np.arange(n_q)[None, :]).astype(np.int32)
    return Workload(name="verify_8x5", seed=seed, n_seqs=len(lens), page_size=P, n_kv=H,
                    n_pages=n_pages, max_pages=pt.shape[1], page_table=pt, seq_lens=lens,
                    pos=np.zeros(len(lens), np.int64), k=ks, v=vs, q=qs, steps=steps,
                    n_q=n_q, dtype="bf16")


def config5(seed: int | None = None, history: int = 229376, chunk: int = 8192) -> Workload:
    """Chunked prefill: history cells appended first, then a chunk of `chunk`
    tokens at offset `history`; causal attention of the chunk's queries."""
    seed = config_seed(5) if seed is None else seed
    P, H = 64, 2
    total = history + chunk
    n_pages = (total + P - 1) // P
    pt = page_table_shuffled(seed, stream_id(T_PT, 0), n_pages, n_pages)
    return Workload(name=f"prefill_{chunk}_at_{history}", seed=seed, n_seqs=1, page_size=P,
                    n_kv=H, n_pages=n_pages, max_pages=n_pages, page_table=pt.reshape(1, -1),
                    history=history, chunk=chunk, total=total, dtype="bf16")


def prefill_kv(w: Workload, cell0: int, n: int) -> tuple[Tensor, Tensor]:
    return (kv_values(w.seed, T_K, 0, n, w.n_kv, 3, "bf16", cell0=cell0),
            kv_values(w.seed, T_V, 0, n, w.n_kv, 3, "bf16", cell0=cell0))


def prefill_q(w: Workload) -> Tensor:
    return q_values(w.seed, 0, w.chunk, w.n_kv, "bf16")
