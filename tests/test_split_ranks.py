"""The cell-range split of one decode across GPUs, host side, on CPU: two gloo
ranks (127.0.0.1) each take their range of cell_ranges(), compute its partial
rows (here with the oracle, standing for attn_k8v4_decode_partial on a GPU),
exchange them with gather_partials (the all-gather the GPUs run over NCCL), and
merge them; the result equals the full attention on every rank."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str, n_cells: int):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    import quantized_paged_kv_q8_gb300 as k8
    from test_oracle_pins import _merge_partials
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(31)                     # every rank builds the same cache
        P, H = 16, 2
        n_pages = (n_cells + P - 1) // P
        pt = rng.permutation(n_pages).astype(np.int32)[None]
        k = rng.standard_normal((1, n_cells, H, 256)).astype(np.float32)
        v = rng.standard_normal((1, n_cells, H, 256)).astype(np.float32)
        cache = oracle.Cache(n_pages, P, H)
        cache.append(pt, np.array([0]), k, v)
        q = rng.standard_normal((16, 256)).astype(np.float32)
        rs, rh, _ = oracle.decode_rows(1, 16, [n_cells])
        lo, hi = k8.cell_ranges(n_cells, world)[rank]
        o, m, l = cache.attention_partial(pt, rs, rh, np.full(16, lo), np.full(16, hi), q, n_threads=1)
        row = np.concatenate([o, m[:, None], l[:, None], np.zeros((16, 2))], axis=1)   # the 260-float rows
        parts = k8.gather_partials(torch.from_numpy(row)[None], group=None)             # [world, 1, 16, 260]
        assert parts.shape == (world, 1, 16, 260)
        pieces = [(p[0, :, :256].numpy(), p[0, :, 256].numpy(), p[0, :, 257].numpy()) for p in parts]
        got = _merge_partials(pieces)
        full = cache.attention(pt, rs, rh, np.full(16, n_cells), q, n_threads=1)
        err = float(np.max(np.abs(got - full)) / max(1.0, np.max(np.abs(full))))
        ranges = k8.cell_ranges(n_cells, world)
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{err} {ranges[rank][0]} {ranges[rank][1]}\n")
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("n_cells", [300, 37])
def test_two_rank_split_decode_merges_to_full(tmp_path, n_cells):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path), n_cells), nprocs=world,
                       start_method="spawn")
    spans = []
    for r in range(world):
        err, lo, hi = open(tmp_path / f"r{r}.txt").read().split()
        assert float(err) < 1e-12
        spans.append((int(lo), int(hi)))
    # the ranges tile [0, n) in rank order, each starting on a 16-cell tile
    assert spans[0][0] == 0 and spans[-1][1] == n_cells
    assert all(a[1] == b[0] for a, b in zip(spans[:-1], spans[1:]))
    assert all(lo % 16 == 0 for lo, _ in spans)


def test_cell_ranges_partition():
    sys.path.insert(0, ROOT)
    import quantized_paged_kv_q8_gb300 as k8
    for n in (0, 1, 15, 16, 17, 237568, 237605):
        for world in (1, 2, 3, 8):
            r = k8.cell_ranges(n, world)
            assert len(r) == world and r[0][0] == 0 and r[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(r[:-1], r[1:]))
            assert all(lo % 16 == 0 and lo <= hi for lo, hi in r)
            assert all(hi % 16 == 0 for _, hi in r[:-1])
