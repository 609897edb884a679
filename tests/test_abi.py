"""CPU checks of the C ABI: the library loads, exports every entry point that
include/k8v4.h declares, and rejects bad arguments on the host (no device call
is needed for a rejected call)."""
import ctypes
import os
import re

import pytest

import quantized_paged_kv_q8_gb300 as k8

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    k8.build()
    return k8.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "k8v4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^[a-z_0-9 \*]+?\b([a-z_0-9]+)\(", src, flags=re.M)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert "kv_append_k8v4" in names and "attn_k8v4_prefill" in names
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(k8.EXPORTED)


def test_bytes_per_cell(L):
    assert k8.k8v4_bytes_per_cell(k8.FORMAT_K8V4, 2) == 816
    assert k8.k8v4_bytes_per_cell(k8.FORMAT_INT8, 2) == 1056
    assert k8.k8v4_bytes_per_cell(k8.FORMAT_Q4, 2) == 576
    assert k8.k8v4_bytes_per_cell(k8.FORMAT_K8V4, 1) == 408
    assert k8.k8v4_bytes_per_cell(0, 2) == 0
    assert k8.k8v4_bytes_per_cell(4, 2) == 0
    assert k8.k8v4_bytes_per_cell(k8.FORMAT_K8V4, 0) == 0


def _desc(**kw):
    d = dict(pages=0x10000, n_pages=4, page_size=16, n_kv_heads=2, head_dim=256, format=k8.FORMAT_K8V4)
    d.update(kw)
    return k8.k8v4_cache(ctypes.c_void_p(d["pages"]), d["n_pages"], d["page_size"], d["n_kv_heads"],
                         d["head_dim"], d["format"])


FAKE = ctypes.c_void_p(0x20000)


@pytest.mark.parametrize("bad,code", [
    (dict(head_dim=128), k8.EINVAL), (dict(page_size=8), k8.EINVAL), (dict(page_size=24), k8.EINVAL),
    (dict(n_kv_heads=9), k8.EINVAL), (dict(format=0), k8.EINVAL), (dict(format=4), k8.EINVAL), (dict(n_pages=0), k8.EINVAL),
    (dict(pages=0), k8.EINVAL), (dict(pages=0x10010), k8.EALIGN),
])
def test_bad_cache_descriptor_rejected(L, bad, code):
    d = _desc(**bad)
    rc = L.kv_append_k8v4(ctypes.byref(d), FAKE, 4, 1, FAKE, 1, FAKE, FAKE, k8.BF16, None)
    assert rc == code


def test_bad_arguments_rejected(L):
    d = ctypes.byref(_desc())
    assert L.kv_append_k8v4(d, FAKE, 4, 1, FAKE, 1, FAKE, FAKE, 7, None) == k8.EINVAL          # dtype
    assert L.kv_append_k8v4(d, None, 4, 1, FAKE, 1, FAKE, FAKE, k8.BF16, None) == k8.EINVAL    # table
    assert L.kv_append_k8v4(d, FAKE, 4, 1, FAKE, 1, ctypes.c_void_p(0x20004), FAKE, k8.BF16, None) == k8.EALIGN
    assert L.kv_append_k8v4(d, FAKE, 4, 0, FAKE, 1, FAKE, FAKE, k8.BF16, None) == k8.OK        # nothing to do
    # decode: n_q, lengths beyond the table, scale
    assert L.attn_k8v4_decode(d, FAKE, k8.BF16, FAKE, 4, FAKE, 1, 65, 0.0625, FAKE, FAKE, 1 << 20, None) == k8.EINVAL
    assert L.attn_k8v4_decode(d, FAKE, k8.BF16, FAKE, 4, FAKE, 1, 64, -1.0, FAKE, FAKE, 1 << 20, None) == k8.EINVAL
    assert L.attn_k8v4_verify(d, FAKE, k8.BF16, FAKE, 4, FAKE, 1, 9, 64, 0.0625, FAKE, FAKE, 1 << 20, None) == k8.EINVAL
    # prefill: bf16 only, k8v4 only
    assert L.attn_k8v4_prefill(d, FAKE, k8.F32, FAKE, 4, 64, 8, None, 0.0625, FAKE, None) == k8.EINVAL
    d8 = ctypes.byref(_desc(format=k8.FORMAT_INT8))
    assert L.attn_k8v4_prefill(d8, FAKE, k8.BF16, FAKE, 4, 64, 8, None, 0.0625, FAKE, None) == k8.EINVAL
    d4 = ctypes.byref(_desc(format=k8.FORMAT_Q4))
    assert L.attn_k8v4_prefill(d4, FAKE, k8.BF16, FAKE, 4, 64, 8, None, 0.0625, FAKE, None) == k8.EINVAL
    assert L.attn_k8v4_prefill(d, FAKE, k8.BF16, FAKE, 4, 64, 65, None, 0.0625, FAKE, None) == k8.EINVAL
    # dequant range
    assert L.kv_dequant_k8v4(d, FAKE, 4, 60, 5, FAKE, FAKE, None, None) == k8.EINVAL


def test_stream_arguments_rejected(L):
    """The streaming calls check geometry, counts, pointers and sizes on the host."""
    d, h = ctypes.byref(_desc()), ctypes.byref(_desc(pages=0x30000))
    q4 = ctypes.byref(_desc(pages=0x30000, format=k8.FORMAT_Q4))
    p32 = ctypes.byref(_desc(pages=0x30000, page_size=32))
    assert L.kv_stream_workspace_bytes(2, 10) == 16 + 8 * 20
    assert L.kv_stream_workspace_bytes(1, 1 << 29) == 0
    args = (FAKE, 0, FAKE, 4, FAKE, 1, 64, FAKE, FAKE, 1 << 20, None)
    assert L.kv_stream_resolve(q4, d, *args) == k8.EINVAL                # format differs
    assert L.kv_stream_resolve(p32, d, *args) == k8.EINVAL               # page size differs
    assert L.kv_stream_resolve(h, d, FAKE, 5, FAKE, 4, FAKE, 1, 64, FAKE, FAKE, 1 << 20, None) == k8.EINVAL
    assert L.kv_stream_resolve(h, d, FAKE, 0, FAKE, 4, FAKE, 1, 65, FAKE, FAKE, 1 << 20, None) == k8.EINVAL
    assert L.kv_stream_resolve(h, d, None, 0, FAKE, 4, FAKE, 1, 64, FAKE, FAKE, 1 << 20, None) == k8.EINVAL
    assert L.kv_stream_resolve(h, d, FAKE, 0, FAKE, 4, FAKE, 1, 64, FAKE, FAKE, 47, None) == k8.ENOSPACE
    assert L.kv_stream_resolve(h, d, FAKE, 0, FAKE, 4, FAKE, 1, 64, FAKE, ctypes.c_void_p(0x20008), 1 << 20,
                               None) == k8.EALIGN
    assert L.kv_stream_resolve(h, d, FAKE, 0, FAKE, 4, FAKE, 0, 64, FAKE, FAKE, 0, None) == k8.OK
    assert L.kv_append_k8v4_mirrored(h, d, None, FAKE, 4, 1, FAKE, 1, FAKE, FAKE, k8.BF16, None) == k8.EINVAL
    assert L.kv_append_k8v4_mirrored(q4, d, FAKE, FAKE, 4, 1, FAKE, 1, FAKE, FAKE, k8.BF16, None) == k8.EINVAL
    assert L.kv_stream_copy(h, d, FAKE, -1, None) == k8.EINVAL
    assert L.kv_stream_copy(h, d, ctypes.c_void_p(0x20004), 3, None) == k8.EALIGN
    assert L.kv_stream_copy(h, d, FAKE, 0, None) == k8.OK


def test_workspace_size_is_positive_and_monotone(L):
    d = ctypes.byref(_desc(n_pages=4096, page_size=64))
    a = L.attn_k8v4_workspace_bytes(d, 1, 1, 32768)
    b = L.attn_k8v4_workspace_bytes(d, 8, 5, 65536)
    assert a > 0 and b > 0
    assert L.attn_k8v4_workspace_bytes(d, 1, 9, 100) == 0


def test_valid_call_without_gpu_reports_device(L):
    """With valid arguments and no sm_103 device the call reports EDEVICE (on a
    GB300 this test is skipped)."""
    if k8.k8v4_device_check() == k8.OK:
        pytest.skip("a GB300 is present")
    d = ctypes.byref(_desc())
    assert L.kv_append_k8v4(d, FAKE, 4, 1, FAKE, 1, FAKE, FAKE, k8.BF16, None) in (k8.EDEVICE, k8.ECUDA)
    assert k8.status_string(k8.ERANGE).startswith("position")


def test_header_is_plain_c(tmp_path):
    """include/k8v4.h compiles as C99 with warnings as errors, and every entry
    point the binding exports is declared there with a C prototype."""
    import subprocess
    names = k8.EXPORTED
    src = tmp_path / "use_header.c"
    body = "\n".join(f"  (void)&{n};" for n in names)
    src.write_text(f'#include "k8v4.h"\nint main(void) {{\n{body}\n  return 0;\n}}\n')
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", inc, "-c", str(src),
                        "-o", str(tmp_path / "use_header.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
