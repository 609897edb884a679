"""The seeded input generators (synth/): the counter-based SplitMix64 stream is
the published generator, and the generators' documented properties hold (a
slice of a sequence draws the same numbers as the whole, seeds and streams are
independent, page tables are permutations)."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402


def test_splitmix64_published_sequence():
    """Stream 0 of seed 1234567 is SplitMix64 seeded with 1234567: its first five
    outputs are the generator's published test values."""
    got = [int(x) for x in synth.raw_u64(1234567, 0, 0, 5)]
    assert got == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                   4593380528125082431, 16408922859458223821]
    # counter form: any window of the stream equals the same window of the whole
    whole = synth.raw_u64(99, 7, 0, 64)
    assert np.array_equal(synth.raw_u64(99, 7, 20, 10), whole[20:30])


def test_kv_slices_draw_the_same_numbers():
    """Cell c of a sequence has the same values whether it is drawn with its
    history or as part of a later chunk (cell0 offset)."""
    seed = synth.config_seed(5)
    full = synth.kv_values(seed, synth.T_K, 2, 300, 2, 3, "bf16")
    part = synth.kv_values(seed, synth.T_K, 2, 100, 2, 3, "bf16", cell0=200)
    assert np.array_equal(full.f32[200:300], part.f32)
    assert np.array_equal(full.dev[200:300], part.dev)
    other = synth.kv_values(seed, synth.T_V, 2, 300, 2, 3, "bf16")
    assert not np.array_equal(full.f32, other.f32)                 # K and V streams differ


def test_uniform_and_normal_ranges():
    u = synth.uniform(5, 1, 0, 100000)
    assert u.min() > 0.0 and u.max() <= 1.0 and abs(u.mean() - 0.5) < 0.01
    x = synth.normal(5, 2, 200000)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01


def test_page_tables_are_permutations():
    pt = synth.page_table_shuffled(3, synth.stream_id(synth.T_PT, 0), 50, 64)
    assert len(set(pt.tolist())) == 50 and pt.min() >= 0 and pt.max() < 64
    lens = np.array([700, 1333, 64], np.int32)
    table, n_pages = synth.interleaved_pool(11, lens, 64)
    used = [int(table[b, j]) for b in range(3) for j in range((int(lens[b]) + 63) // 64)]
    assert sorted(used) == list(range(n_pages))
