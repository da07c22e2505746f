"""The C-ABI library loads on a CPU host and exports every declared entry
point; argument errors are reported from the host before any CUDA work."""
import ctypes
import os
import subprocess

import pytest

import global_attention_sinks_swa_b300 as A


def test_every_declared_symbol_is_exported():
    declared = A.declared_symbols()
    assert len(declared) >= 12
    out = subprocess.run(["nm", "-D", "--defined-only", A.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [s for s in declared if s not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for s in declared:
        assert getattr(A._lib, s) is not None


def test_only_declared_symbols_are_public():
    out = subprocess.run(["nm", "-D", "--defined-only", A.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    extra = sorted(s for s in exported if s.startswith("attn_") and s not in A.declared_symbols())
    assert not extra, f"exported but not declared: {extra}"


def test_version_and_error_string():
    assert A.attn_version() >= 100
    assert isinstance(A._lib.attn_last_error(), bytes)


@pytest.mark.parametrize("fn,nargs", [("attn_swa_sink_prefill", 15), ("attn_ga_sink_prefill", 14)])
def test_null_pointers_rejected_on_host(fn, nargs):
    f = getattr(A._lib, fn)
    args = [None] * 6 + [1, 16, 8, 1, 128] + ([128] if fn.startswith("attn_swa") else []) + \
           [ctypes.c_float(0.1), 0, None]
    assert len(args) == nargs
    assert f(*args) == A.ATTN_ERR_INVALID_ARG
    assert b"null" in A._lib.attn_last_error()


def test_verify_workspace_size_formula():
    # one split (context <= 4096) needs no scratch; otherwise 32 rows x (D + 2) floats per unit
    assert A.attn_ga_sink_verify_workspace(64, 64, 8, 128, 4, 4096) == 0
    n = A.attn_ga_sink_verify_workspace(64, 64, 8, 128, 4, 65536)
    units = 64 * 8 * 16
    assert n >= units * 32 * 130 * 4


def test_new_entry_points_reject_null_pointers_on_host():
    L = A._lib
    f32 = ctypes.c_float
    # packed prefill: 7 pointers, then B, total, max_seqlen, Hq, Hkv, D, (window), scale, vscale
    assert L.attn_swa_sink_prefill_varlen(*([None] * 7), 1, 16, 16, 8, 1, 128, 128, f32(0.1),
                                          f32(1.0), 0, None) == A.ATTN_ERR_INVALID_ARG
    assert L.attn_ga_sink_prefill_varlen(*([None] * 7), 1, 16, 16, 8, 1, 128, f32(0.1), f32(1.0),
                                         0, None) == A.ATTN_ERR_INVALID_ARG
    # backward: 12 pointers, workspace bytes, B, T, Hq, Hkv, D, window, scale, dtype, stream
    assert L.attn_sink_prefill_backward(*([None] * 12), 0, 1, 16, 8, 1, 128, 128, f32(0.1), 0,
                                        None) == A.ATTN_ERR_INVALID_ARG
    # 8-bit append and verify
    assert L.attn_ga_paged_append_fp8(*([None] * 7), 4, 4, 64, None, None, 1, 8, 128, 4,
                                      None) == A.ATTN_ERR_INVALID_ARG
    assert L.attn_ga_sink_verify_fp8(*([None] * 5), 4, 4, 64, *([None] * 6), 0, 1, 64, 8, 128, 4,
                                     4096, f32(0.1), None) == A.ATTN_ERR_INVALID_ARG
    assert b"null" in L.attn_last_error()


def test_backward_workspace_size():
    # D = <dO, O> per (b, h, i) in fp32, rounded up to 256 bytes (no dq partials)
    assert A._lib.attn_sink_prefill_backward_workspace(1, 1024, 64, 128) == 64 * 1024 * 4
    assert A._lib.attn_sink_prefill_backward_workspace(2, 1000, 3, 128) == (2 * 3 * 1000 * 4 + 255) // 256 * 256
    assert A._lib.attn_sink_prefill_backward_workspace(1, 1024, 64, 64) == 0   # unsupported D


def test_package_refuses_to_import_without_its_library(tmp_path):
    """No CPU fallback: a copy of the binding with no library next to it fails
    at import with a message naming the build step."""
    import importlib.util
    import shutil

    import global_attention_sinks_swa_b300 as A
    pkg = tmp_path / "pkg_copy"
    pkg.mkdir()
    shutil.copy(os.path.join(os.path.dirname(A.__file__), "__init__.py"), pkg / "__init__.py")
    spec = importlib.util.spec_from_file_location("pkg_copy", pkg / "__init__.py",
                                                  submodule_search_locations=[str(pkg)])
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError, match="no CPU fallback"):
        spec.loader.exec_module(mod)
