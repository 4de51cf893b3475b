"""Host-side checks of the C ABI: the library builds, loads, exports every function that
include/osf.h declares, and rejects invalid arguments before touching a device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "osf.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(osf_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("osf_attn_fwd", "osf_attn_fwd_gqa", "osf_softmax_rows", "osf_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(osf):
    lib = ctypes.CDLL(osf.library_path)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared in osf.h but not exported: {missing}"


def test_status_strings(osf):
    for code in range(6):
        s = osf.osf_status_string(code)
        assert s.startswith("OSF_")
    assert osf.osf_status_string(99) == "unknown osf status"
    assert osf.osf_version() >= 100


def test_invalid_arguments_rejected_on_host(osf):
    lib = osf.lib()
    p = ctypes.c_void_p(1 << 40)
    o = ctypes.c_void_p(1 << 44)
    # negative sizes / bad head dim
    assert lib.osf_attn_fwd(p, p, p, o, -1, 4, 4, None) == osf.OSF_ERR_INVALID
    assert lib.osf_attn_fwd(p, p, p, o, 4, 4, 0, None) == osf.OSF_ERR_INVALID
    # empty problems are a no-op (the pages return early on N == 0)
    assert lib.osf_attn_fwd(None, None, None, None, 0, 4, 4, None) == osf.OSF_OK
    assert lib.osf_attn_fwd(None, None, None, None, 4, 0, 4, None) == osf.OSF_OK
    # Hq not divisible by Hkv, unknown dtype, causal with 1 < Sq != Sk, D too large
    args = lambda dt, Hq, Hkv, Sq, Sk, D, causal: (p, p, p, o, dt, 1, Hq, Hkv, Sq, Sk, D, causal,
                                                    0.0, None, None, 0, None)
    assert lib.osf_attn_fwd_gqa(*args(1, 6, 4, 8, 8, 64, 0)) == osf.OSF_ERR_INVALID
    assert lib.osf_attn_fwd_gqa(*args(7, 4, 4, 8, 8, 64, 0)) == osf.OSF_ERR_INVALID
    assert lib.osf_attn_fwd_gqa(*args(1, 4, 4, 8, 9, 64, 1)) == osf.OSF_ERR_INVALID
    assert lib.osf_attn_fwd_gqa(*args(1, 4, 4, 8, 8, 257, 0)) == osf.OSF_ERR_UNSUPPORTED
    assert lib.osf_attn_fwd_gqa(*args(1, 4, 4, 0, 8, 64, 0)) == osf.OSF_OK
    # NULL with non-zero size
    assert lib.osf_attn_fwd_gqa(None, p, p, o, 1, 1, 4, 4, 8, 8, 64, 0, 0.0, None, None, 0,
                                None) == osf.OSF_ERR_INVALID
    # output overlapping an input
    assert lib.osf_attn_fwd_gqa(p, p, p, p, 1, 1, 4, 4, 8, 8, 64, 0, 0.0, None, None, 0,
                                None) == osf.OSF_ERR_INVALID
    # softmax: negative sizes, NULL, partial overlap; z == x is allowed (checked on GPU)
    assert lib.osf_softmax_rows(p, o, -1, 4, None, 0, None) == osf.OSF_ERR_INVALID
    assert lib.osf_softmax_rows(None, o, 2, 4, None, 0, None) == osf.OSF_ERR_INVALID
    assert lib.osf_softmax_rows(p, ctypes.c_void_p((1 << 40) + 4), 2, 4, None, 0, None) == osf.OSF_ERR_INVALID
    assert lib.osf_softmax_rows(None, None, 0, 4, None, 0, None) == osf.OSF_OK
    n = ctypes.c_size_t(123)
    assert lib.osf_softmax_workspace_bytes(-1, 4, ctypes.byref(n)) == osf.OSF_ERR_INVALID
    assert lib.osf_attn_workspace_bytes(1, 1, 3, 2, 1, 8, 64, ctypes.byref(n)) == osf.OSF_ERR_INVALID


def test_host_buffer_entry_point_rejects_invalid_arguments_on_host(osf):
    """osf_attn_fwd_gqa_host checks sizes, host pointers and its device buffer before any copy."""
    lib = osf.lib()
    p = ctypes.c_void_p(1 << 40)
    o = ctypes.c_void_p(1 << 44)
    buf = ctypes.c_void_p(1 << 45)
    f = lib.osf_attn_fwd_gqa_host
    args = lambda Hq, Hkv, Sq, Sk, causal, b: (p, p, p, o, 1, 1, Hq, Hkv, Sq, Sk, 64, causal, 0.0, b, 1 << 30, None)
    assert f(*args(6, 4, 8, 8, 0, buf)) == osf.OSF_ERR_INVALID         # Hq % Hkv != 0
    assert f(*args(4, 4, 8, 9, 1, buf)) == osf.OSF_ERR_INVALID         # causal with 1 < Sq != Sk
    assert f(*args(4, 4, 0, 8, 0, None)) == osf.OSF_OK                 # empty: nothing to do
    assert f(*args(4, 2, 8, 8, 0, None)) == osf.OSF_ERR_WORKSPACE      # no device buffer
    assert f(p, p, p, p, 1, 1, 4, 4, 8, 8, 64, 0, 0.0, buf, 1 << 30, None) == osf.OSF_ERR_INVALID   # O overlaps Q
    n = ctypes.c_size_t(7)
    assert lib.osf_attn_host_buffer_bytes(1, 1, 6, 4, 8, 8, 64, 0, ctypes.byref(n)) == osf.OSF_ERR_INVALID
    assert lib.osf_attn_host_buffer_bytes(1, 1, 4, 4, 8, 8, 64, 0, None) == osf.OSF_ERR_INVALID


def test_strided_entry_point_rejects_bad_layouts_on_host(osf):
    """osf_attn_fwd_gqa_ex validates strides and masks before touching the device."""
    lib = osf.lib()
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 8, 8, 64
    q, k, v, o = (ctypes.c_void_p(x << 40) for x in (1, 2, 3, 4))
    bshd_q = [Sq * Hq * D, D, Hq * D]
    bshd_kv = [Sk * Hkv * D, D, Hkv * D]

    def call(strides, mask=0, out=o, Sq_=Sq, Sk_=Sk):
        arr = None if strides is None else (ctypes.c_longlong * 12)(*strides)
        return lib.osf_attn_fwd_gqa_ex(q, k, v, out, osf.OSF_BF16, B, Hq, Hkv, Sq_, Sk_, D,
                                       None if arr is None else ctypes.cast(arr, ctypes.c_void_p), mask,
                                       0.0, None, None, 0, None)

    good = bshd_q + bshd_kv + bshd_kv + bshd_q
    assert call(good, mask=7) == osf.OSF_ERR_INVALID                       # unknown mask
    assert call(good[:2] + [-Hq * D] + good[3:]) == osf.OSF_ERR_INVALID    # negative stride
    overlapping_o = good[:9] + [Sq * Hq * D, D, D]                          # rows of O collide
    assert call(overlapping_o) == osf.OSF_ERR_INVALID
    broadcast_o = good[:9] + [0, Sq * D, D]                                  # O may not broadcast
    assert call(broadcast_o) == osf.OSF_ERR_INVALID
    assert call(good, out=q) == osf.OSF_ERR_INVALID                         # O over Q
    # inputs may broadcast (stride 0) and any mask is accepted for Sq != Sk; empty problems are no-ops
    assert call(good, Sq_=0) == osf.OSF_OK
    assert call(good[:3] + [0, 0, D] + [0, 0, D] + good[9:], Sq_=0) == osf.OSF_OK
    assert call(good, mask=2, Sk_=0) == osf.OSF_OK


def test_binding_refuses_cpu_tensors(osf):
    torch = pytest.importorskip("torch")
    x = torch.zeros(4, 8)
    with pytest.raises(ValueError):
        osf.osf_softmax_rows(x)
    with pytest.raises(ValueError):
        osf.osf_attn_fwd(x, x, x, x, 4, 4, 8)


def test_product_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "online_softmax_flash_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
                assert "seeded_inputs" not in src, f


def test_header_is_plain_c(tmp_path):
    """include/osf.h compiles as C99 on its own (no CUDA or torch headers needed by a caller)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_osf.c"
    src.write_text('#include <stdio.h>\n#include "osf.h"\n'
                   "int use(void *q, void *k, void *v, void *o, void *ws, size_t n, osf_stream s) {\n"
                   "    int st = osf_attn_fwd_gqa(q, k, v, o, OSF_BF16, 2, 32, 8, 4096, 4096, 128, 1, 0.f,\n"
                   "                              NULL, ws, n, s);\n"
                   "    if (st != OSF_OK) fprintf(stderr, \"%s\\n\", osf_status_string(st));\n"
                   "    return st;\n}\n")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-I", os.path.dirname(HEADER), str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_backward_workspace_sizes(osf):
    """osf_attn_bwd_workspace_bytes: the row sums (one float per query row, 256-byte rounded),
    plus, for bf16 with D in {64, 128} while it stays within 16 GiB, bf16 dS^T over the key and
    query counts rounded up to 128; other dtypes, head dims and larger problems get the row sums
    alone (the path that recomputes S and dP for dQ)."""
    lib = osf.lib()
    n = ctypes.c_size_t(0)
    r256 = lambda x: (x + 255) // 256 * 256
    r128 = lambda x: (x + 127) // 128 * 128

    def bytes_for(dt, B, Hq, Hkv, Sq, Sk, D):
        assert lib.osf_attn_bwd_workspace_bytes(dt, B, Hq, Hkv, Sq, Sk, D, ctypes.byref(n)) == osf.OSF_OK
        return n.value

    for (B, Hq, Hkv, Sq, Sk, D) in [(2, 32, 8, 4096, 4096, 128), (1, 4, 2, 200, 333, 64), (3, 16, 4, 1100, 700, 128)]:
        rows = r256(B * Hq * Sq * 4)
        assert bytes_for(osf.OSF_BF16, B, Hq, Hkv, Sq, Sk, D) == rows + r256(B * Hq * r128(Sk) * r128(Sq) * 2)
        assert bytes_for(osf.OSF_F32, B, Hq, Hkv, Sq, Sk, D if D == 64 else 128) == rows
    assert bytes_for(osf.OSF_BF16, 1, 4, 2, 77, 77, 96) == r256(4 * 77 * 4)
    # dS^T past 16 GiB: the row sums alone
    B, Hq, S = 2, 64, 65536
    assert B * Hq * S * S * 2 > 16 << 30
    assert bytes_for(osf.OSF_BF16, B, Hq, 8, S, S, 128) == r256(B * Hq * S * 4)
    assert bytes_for(osf.OSF_BF16, 1, 1, 1, 0, 8, 128) == 0
