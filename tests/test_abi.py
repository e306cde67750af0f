"""The C-ABI library builds, loads and exports what include/marlin.h declares;
host-side argument checks (no GPU needed: these paths return before any CUDA
call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "marlin.h")


@pytest.fixture(scope="module")
def lib():
    from w4a16_mixed_precision_gb300 import _binding, build
    build.build()
    return _binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(marlin_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    from w4a16_mixed_precision_gb300 import _binding
    assert declared_functions() == sorted(_binding.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    from w4a16_mixed_precision_gb300 import _binding
    for code, name in [(0, "MARLIN_OK"), (1, "MARLIN_ERR_INVALID_ARG"), (3, "MARLIN_ERR_MISALIGNED"),
                       (4, "MARLIN_ERR_WORKSPACE_TOO_SMALL"), (6, "MARLIN_ERR_TIMEOUT"),
                       (7, "MARLIN_ERR_BOUNDS"), (2, "MARLIN_ERR_UNSUPPORTED")]:
        assert _binding.status_string(code) == name


def test_packed_layout(lib):
    from w4a16_mixed_precision_gb300 import _binding
    b, s, z = _binding.packed_layout(4096, 4096, 128, False)
    assert s == 4096 * 4096 // 2
    assert b == s + 32 * 4096 * 2 and z == b
    b, s, z = _binding.packed_layout(2048, 5632, 2048, True)
    assert s == 2048 * 5632 // 2 and z == s + 5632 * 2 and b == z + 5632 // 2
    assert s % 256 == 0 and z % 256 == 0
    b1, _, _ = _binding.packed_layout(2048, 5632, -1, True)
    assert b1 == b
    for bad in [(100, 128, 128), (128, 100, 128), (384, 128, 256), (0, 128, 128), (256, 128, 0),
                (256, 128, 96)]:
        with pytest.raises(_binding.MarlinError) as e:
            _binding.packed_layout(*bad, False)
        assert e.value.status == _binding.ERR_INVALID_ARG
    # groups of 32 or 64 divide K but are not served ("Marlin", section
    # "Group size 为什么是 128": 64 runs slower, 32 may not run)
    for small in [(256, 128, 64), (256, 128, 32)]:
        with pytest.raises(_binding.MarlinError) as e:
            _binding.packed_layout(*small, False)
        assert e.value.status == _binding.ERR_UNSUPPORTED


def test_gemm_host_checks(lib):
    """Shape, group and alignment errors come back before anything touches CUDA."""
    from w4a16_mixed_precision_gb300 import _binding as b
    good = 0x10000
    # M == 0 is a no-op
    assert b.gemm_raw(good, good, good, None, good, 0, 256, 256, 128, good, 1 << 20, 0) == b.OK
    assert b.gemm_raw(good, good, good, None, good, -1, 256, 256, 128, good, 1 << 20, 0) == b.ERR_INVALID_ARG
    assert b.gemm_raw(good, good, good, None, good, 4, 200, 256, 128, good, 1 << 20, 0) == b.ERR_INVALID_ARG
    assert b.gemm_raw(good, good, good, None, good, 4, 256, 200, 128, good, 1 << 20, 0) == b.ERR_INVALID_ARG
    assert b.gemm_raw(good, good, good, None, good, 4, 256, 256, 64, good, 1 << 20, 0) == b.ERR_UNSUPPORTED
    assert b.gemm_raw(good, good, good, None, good, 4, 256, 256, 0, good, 1 << 20, 0) == b.ERR_INVALID_ARG
    assert b.gemm_raw(0, good, good, None, good, 4, 256, 256, 128, good, 1 << 20, 0) == b.ERR_INVALID_ARG
    assert b.gemm_raw(good, good, good, None, good, 4, 256, 256, 128, 0, 1 << 20, 0) == b.ERR_INVALID_ARG
    assert b.gemm_raw(good + 8, good, good, None, good, 4, 256, 256, 128, good, 1 << 20, 0) == b.ERR_MISALIGNED
    assert b.gemm_raw(good, good + 4, good, None, good, 4, 256, 256, 128, good, 1 << 20, 0) == b.ERR_MISALIGNED
    assert b.gemm_raw(good, good, good, good + 2, good, 4, 256, 256, 128, good, 1 << 20, 0) == b.ERR_MISALIGNED
    assert b.gemm_raw(good, good, good, None, good + 1, 4, 256, 256, 128, good, 1 << 20, 0) == b.ERR_MISALIGNED


def test_repack_host_checks(lib):
    from w4a16_mixed_precision_gb300 import _binding as b
    good = 0x10000
    assert b.repack_raw(0, good, None, 256, 256, 128, good, 0) == b.ERR_INVALID_ARG
    assert b.repack_raw(good, good, None, 256, 256, 96, good, 0) == b.ERR_INVALID_ARG
    assert b.repack_raw(good, good, None, 256, 192, 128, good, 0) == b.ERR_INVALID_ARG
    assert b.repack_raw(good + 4, good, None, 256, 256, 128, good, 0) == b.ERR_MISALIGNED
    assert b.repack_raw(good, good, None, 256, 256, 128, good + 8, 0) == b.ERR_MISALIGNED


def test_product_path_does_not_import_the_oracle():
    """The package and the binding never reference the oracle."""
    pkg = os.path.join(ROOT, "w4a16_mixed_precision_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "oracle.c" not in src, f


def test_sparse_packed_layout(lib):
    from w4a16_mixed_precision_gb300 import _binding
    b, m, s, z = _binding.sparse_packed_layout(4096, 4096, 128, False)
    assert m == 4096 * 4096 // 4                       # kept codes: half of the dense codes
    assert s == m + 4096 * 4096 // 8                   # index pairs: 4 bits per four weights
    assert b == s + 32 * 4096 * 2 and z == b
    b, m, s, z = _binding.sparse_packed_layout(2048, 5632, -1, True)
    assert m % 256 == 0 and s % 256 == 0 and z % 256 == 0
    assert m >= 2048 * 5632 // 4 and s >= m + 2048 * 5632 // 8
    assert z == s + 5632 * 2 and b == z + 5632 // 2
    for bad in [(100, 128, 128), (0, 128, 128)]:
        with pytest.raises(_binding.MarlinError) as e:
            _binding.sparse_packed_layout(*bad, False)
        assert e.value.status == _binding.ERR_INVALID_ARG
    with pytest.raises(_binding.MarlinError) as e:
        _binding.sparse_packed_layout(256, 128, 64, False)
    assert e.value.status == _binding.ERR_UNSUPPORTED


def test_sparse_host_checks(lib):
    """The 2:4 entry points reject bad arguments before touching CUDA."""
    from w4a16_mixed_precision_gb300 import _binding as b
    g = 0x10000
    call = b.sparse_gemm_raw
    # meta is required; the dense warp-level kernel forced above 32 tokens is not served
    assert call(g, g, None, g, None, g, 4, 256, 256, 128, g, 1 << 20, 0) == b.ERR_INVALID_ARG
    assert b.gemm_ex_raw(g, g, g, None, g, 33, 256, 256, 128, g, 1 << 20, 1, 0) == b.ERR_UNSUPPORTED
    assert call(g, g, g, g, None, g, 0, 256, 256, 128, g, 1 << 20, 0) == b.OK
    assert call(g, g, g, g, None, g, 4, 256, 200, 128, g, 1 << 20, 0) == b.ERR_INVALID_ARG
    assert call(g, g, g + 8, g, None, g, 4, 256, 256, 128, g, 1 << 20, 0) == b.ERR_MISALIGNED
    assert call(g, g + 8, g, g, None, g, 4, 256, 256, 128, g, 1 << 20, 0) == b.ERR_MISALIGNED
    rp = b.sparse_repack_raw
    assert rp(0, g, None, 256, 256, 128, g, None, 0) == b.ERR_INVALID_ARG
    assert rp(g, g, None, 256, 256, 96, g, None, 0) == b.ERR_INVALID_ARG
    assert rp(g, g, None, 256, 256, 128, g + 8, None, 0) == b.ERR_MISALIGNED
    assert rp(g, g, None, 256, 256, 128, g, g + 2, 0) == b.ERR_MISALIGNED
