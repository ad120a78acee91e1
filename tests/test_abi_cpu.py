"""The C-ABI library loads without a GPU and exports every symbol that
include/k3moe.h declares; host-only arithmetic and argument refusals."""
import ctypes
import os
import re

import pytest

from conftest import ROOT
from mxfp4_routed_expert_select_gb300 import k3moe as k


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "k3moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = set(re.findall(r"\b(k3moe_[a-z0-9_]+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol():
    lib = k.lib()
    names = _declared_functions()
    assert len(names) >= 25
    missing = [n for n in sorted(names) if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding knows every one of them
    assert names <= set(k.SIGNATURES), sorted(names - set(k.SIGNATURES))


def test_header_is_plain_c():
    """include/k3moe.h is a C header: it compiles as strict C99 and C11 with
    every warning on, no C++ or CUDA types in it (checked by gcc reading the
    source from stdin, nothing written)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    src = '#include "k3moe.h"\nint main(void) { return (int)k3moe_expert_bytes(7168, 1536) & 0; }\n'
    for std in ("c99", "c11"):
        r = subprocess.run([gcc, "-std=" + std, "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                            "-I", os.path.join(ROOT, "include"), "-x", "c", "-"],
                           input=src, capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_byte_arithmetic_host():
    assert k.expert_bytes(7168, 1536) == 17547264
    assert k.matrix_bytes(1536, 7168) == 5849088
    assert k.expert_bytes(7168, 1500) == -1
    assert k.matrix_bytes(0, 32) == -1


def test_expert_view_offsets():
    d, f = 7168, 1536
    base = 1 << 20
    e = k.expert_view(base, d, f)
    assert e.gate.packed == base and e.gate.scales == base + f * d // 2
    assert e.up.packed == base + 5849088
    assert e.down.packed == base + 2 * 5849088
    assert e.down.scales == base + 2 * 5849088 + d * f // 2
    assert (e.gate.rows, e.gate.in_, e.down.rows, e.down.in_) == (f, d, d, f)
    for m in (e.gate, e.up, e.down):
        assert m.packed % 16 == 0 and m.scales % 16 == 0
    with pytest.raises(k.K3Error):
        k.expert_view(base + 8, d, f)  # misaligned blob


def test_refusals_before_any_cuda_call():
    lib = k.lib()
    m = k.Mat(0, 0, 4, 32)
    assert lib.k3moe_matmul_mxfp4(None, None, ctypes.byref(m), None) == k.K3MOE_EINVAL
    m = k.Mat(16, 16, 4, 33)
    assert lib.k3moe_matmul_mxfp4(16, 16, ctypes.byref(m), None) == k.K3MOE_EINVAL
    assert lib.k3moe_layer_create(None, None) == k.K3MOE_EINVAL
    desc = k.LayerDesc(0, 16, 7168, 1536, 16, None, 16, 1)
    h = ctypes.c_void_p()
    assert lib.k3moe_layer_create(ctypes.byref(h), ctypes.byref(desc)) == k.K3MOE_EINVAL
    assert lib.k3moe_expert_gemv_workspace(7168, 1536) == 1536 * 4
    assert lib.k3moe_expert_gemv_workspace(7168, 4096) == 0  # f beyond the batch-1 path
    assert k.strerror(k.K3MOE_EBUSY) == "no evictable cache slot"
