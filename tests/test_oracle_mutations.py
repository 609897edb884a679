"""The oracle's pins catch plausible mistakes: each case below plants one
mistake in a copy of the oracle's C source (on the CPU, in a temporary build)
or of its Python page-lookup function, puts it in place of the real one, and
runs the pins; at least one pin must fail.  The real oracle is restored
afterwards."""
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = open(oracle.SRC).read()

# (name, text in k8v4_oracle.c, replacement): one plausible mistake each
MUTATIONS = [
    ("int8 ties away from zero", "float r = rintf(x[i] / s);", "float r = roundf(x[i] / s);"),
    ("int8 divisor 128", "float s = a / 127.0f;", "float s = a / 128.0f;"),
    ("int8 reciprocal quotient", "float r = rintf(x[i] / s);", "float r = rintf(x[i] * (1.0f / s));"),
    ("int8 quotient by absmax", "float r = rintf(x[i] / s);", "float r = rintf((x[i] * 127.0f) / a);"),
    ("q4 reciprocal quotient", "float r = rintf(y[j] / d) + 8.0f;", "float r = rintf(y[j] * (1.0f / d)) + 8.0f;"),
    ("q4 last index on ties", "if (fabsf(y[j]) > fabsf(y[im])) im = j;", "if (fabsf(y[j]) >= fabsf(y[im])) im = j;"),
    ("q4 scale sign", "orc_f32_to_f16(m / -8.0f)", "orc_f32_to_f16(m / 8.0f)"),
    ("q4 ties away from zero", "float r = rintf(y[j] / d) + 8.0f;", "float r = roundf(y[j] / d) + 8.0f;"),
    ("nibble order", "nib[j] = (uint8_t)(q[j] | (q[j + 16] << 4));", "nib[j] = (uint8_t)((q[j] << 4) | q[j + 16]);"),
    ("hadamard index", "__builtin_popcount((unsigned)(i & j))", "__builtin_popcount((unsigned)(i | j))"),
    ("V run offset", "p.vq = base + 264 * H * P + r * 128;", "p.vq = base + 256 * H * P + r * 128;"),
    ("GQA map", "g = h / GQA;", "g = h % a->C.H;"),
    ("softmax scale dropped", "sc[j] = dot * sm_scale;", "sc[j] = dot;"),
    ("inverse rotation scale", "o[i] = s / 16.0;", "o[i] = s / 8.0;"),
    ("one cell short", "n = a->row_vis[r], g", "n = a->row_vis[r] - (a->row_vis[r] > 0), g"),
    ("q4 K left rotated", "orc_hadamard_rotate(kr, k_out + off);", "memcpy(k_out + off, kr, sizeof kr);"),
    ("q4 query rotation scale", "q[i] = s / 16.0;", "q[i] = s / 8.0;"),
]

PINS = [
    lambda o: pins.test_int8_hand_ties(o),
    lambda o: pins.test_int8_quotient_is_one_ieee_division(o),
    lambda o: pins.test_q4_quotient_is_one_ieee_division(o),
    lambda o: pins.test_int8_bound_and_extremes(o),
    lambda o: pins.test_q4_hand_ties_through_rotation(o),
    lambda o: pins.test_q4_error_bounds(o),
    lambda o: pins.test_hadamard_is_sylvester_and_orthogonal(o),
    lambda o: pins.test_rotate_equals_exact_rational_rounding(o, "normal"),
    lambda o: pins.test_page_layout_hand_offsets(o),
    lambda o: pins.test_attention_closed_forms(o),
    lambda o: pins.test_attention_matches_torch_sdpa(o, "k8v4"),
    lambda o: pins.test_head_count_separability(o, "k8v4"),
    lambda o: pins.test_q4_format_quantises_k_like_v(o),
    lambda o: pins.test_q4_format_dequant_and_attention(o),
]


def _build(tmp_path, text: str) -> str:
    src = os.path.join(tmp_path, "mutant.c")
    lib = os.path.join(tmp_path, "libmutant.so")
    with open(src, "w") as f:
        f.write(text)
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", lib, src, "-lm"], check=True)
    return lib


def test_unmutated_oracle_passes_the_pins():
    oracle.build()
    for pin in PINS:
        pin(oracle)


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_the_mutation(tmp_path, monkeypatch, name, old, new):
    assert SRC.count(old) == 1, f"mutation target not found once: {old}"
    lib = _build(str(tmp_path), SRC.replace(old, new))
    monkeypatch.setattr(oracle, "LIB", lib)
    monkeypatch.setattr(oracle, "build", lambda force=False: lib)
    monkeypatch.setattr(oracle, "_lib", None)
    caught = []
    for i, pin in enumerate(PINS):
        try:
            pin(oracle)
        except Exception:                     # an assertion, or an error the mistake provokes
            caught.append(i)
            break
    assert caught, f"no pin failed for the mutation '{name}'"


# ---------------------------------------------------------------- the lookup oracle (Python)
STREAM_SRC = None


def _stream_variant(old: str, new: str):
    """oracle.stream_resolve with one line of its source replaced."""
    import inspect
    import textwrap
    global STREAM_SRC
    if STREAM_SRC is None:
        STREAM_SRC = textwrap.dedent(inspect.getsource(oracle.stream_resolve))
    assert STREAM_SRC.count(old) == 1, old
    ns = {"np": __import__("numpy")}
    exec(STREAM_SRC.replace(old, new), ns)
    return ns["stream_resolve"]


STREAM_MUTATIONS = [
    ("pages rounded down", "for i in range((n + P - 1) // P):", "for i in range(n // P):"),
    ("lengths not clipped", "n = min(max(int(seq_lens[b]), 0), max_seq_len)", "n = max(int(seq_lens[b]), 0)"),
    ("staging from n_resident + 1", "slot = n_resident + rank", "slot = n_resident + rank + 1"),
]

STREAM_PINS = [
    lambda o: pins.test_stream_resolve_worked_example(o),
    lambda o: pins.test_stream_resolve_extremes_and_overflow(o),
    lambda o: pins.test_stream_resolve_reads_the_right_bytes(o),
]


@pytest.mark.parametrize("name,old,new", STREAM_MUTATIONS, ids=[m[0] for m in STREAM_MUTATIONS])
def test_stream_pins_catch_the_mutation(monkeypatch, name, old, new):
    monkeypatch.setattr(oracle, "stream_resolve", _stream_variant(old, new))
    caught = False
    for pin in STREAM_PINS:
        try:
            pin(oracle)
        except Exception:
            caught = True
            break
    assert caught, f"no pin failed for the mutation '{name}'"
