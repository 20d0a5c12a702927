"""The C-ABI library loads without a GPU, exports every entry point that
include/pa.h declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")
LIB = os.path.join(ROOT, "paged_kv_cache_158_gb300", "_lib", "libpa.so")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["pa_decode", "pa_decode_workspace_size", "pa_reshape_and_cache", "pa_copy_blocks",
              "pa_slot_mapping", "pa_check_errors", "pa_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(LIB)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_constants_match_the_header():
    """Every status code, error bit and flag the header defines has the same
    value in the Python binding."""
    import paged_kv_cache_158_gb300 as pa
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    consts = {n: int(v, 0) for n, v in re.findall(r"#define\s+(PA_[A-Z_]+)\s+(0x[0-9a-fA-F]+|\d+)u?\b",
                                                  text)}
    consts.update({n: int(v) for n, v in re.findall(r"\b(PA_[A-Z_]+)\s*=\s*(\d+)", text)})
    assert {"PA_OK", "PA_ERR_TIMEOUT", "PA_ERRBIT_TIMEOUT", "PA_DECODE_ZEROED_WORKSPACE",
            "PA_DECODE_INPUTS_READY"} <= set(consts)
    for n, v in consts.items():
        assert getattr(pa, n) == v, n


def test_status_strings_and_sizes_on_host():
    lib = ctypes.CDLL(LIB)
    lib.pa_status_string.restype = ctypes.c_char_p
    assert lib.pa_status_string(0) == b"PA_OK"
    assert lib.pa_status_string(4) == b"PA_ERR_OUT_OF_RANGE"
    lib.pa_decode_workspace_size.restype = ctypes.c_size_t
    assert lib.pa_decode_workspace_size(32, 40, 128, 1024) > 0
    assert lib.pa_decode_workspace_size(32, 40, 96, 1024) == 0       # unsupported head_dim
    assert lib.pa_decode_workspace_size(-1, 40, 128, 1024) == 0


def test_bad_arguments_are_rejected_before_any_launch():
    lib = ctypes.CDLL(LIB)
    vp = ctypes.c_void_p
    f = lib.pa_decode
    f.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int, vp, ctypes.c_size_t, vp]
    good = 0x10000
    # unsupported head_dim / block_size
    assert f(good, good, good, good, good, 4, good, 2, 2, 96, 16, 8, 0.1, 64, good, 1 << 20, None) == 2
    assert f(good, good, good, good, good, 4, good, 2, 2, 128, 12, 8, 0.1, 64, good, 1 << 20, None) == 2
    # null / misaligned pointers, negative sizes, small workspace
    assert f(None, good, good, good, good, 4, good, 2, 2, 128, 16, 8, 0.1, 64, good, 1 << 20, None) == 1
    assert f(good + 2, good, good, good, good, 4, good, 2, 2, 128, 16, 8, 0.1, 64, good, 1 << 20, None) == 1
    assert f(good, good, good, good, good, 4, good, 2, -2, 128, 16, 8, 0.1, 64, good, 1 << 20, None) == 1
    assert f(good, good, good, good, good, 4, good, 2, 2, 128, 16, 8, 0.1, 64, good, 8, None) == 1
    # zero sequences is a no-op
    assert f(None, None, None, None, None, 4, None, 0, 2, 128, 16, 8, 0.1, 64, None, 0, None) == 0
    g = lib.pa_reshape_and_cache
    g.argtypes = [vp, vp, vp, vp, vp] + [ctypes.c_int] * 5 + [vp]
    assert g(good, good, good, good, good, 3, 2, 128, 5, 8, None) == 2
    assert g(good, good, good, good, good + 4, 3, 2, 128, 16, 8, None) == 1
    assert g(None, None, None, None, None, 0, 2, 128, 16, 8, None) == 0
    h = lib.pa_copy_blocks
    h.argtypes = [vp, vp, ctypes.c_int, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, vp]
    ptrs = (ctypes.c_void_p * 1)(good + 8)
    assert h(ptrs, ptrs, 1, good, 2, 2, 128, 16, 8, None) == 1        # misaligned cache pointer
    assert h(None, None, 0, None, 0, 2, 128, 16, 8, None) == 0
    s = lib.pa_slot_mapping
    s.argtypes = [vp, vp, ctypes.c_int, vp, vp] + [ctypes.c_int] * 4 + [vp]
    assert s(good, good, 4, good, good, 3, 2, 6, 8, None) == 2
    assert s(good + 4, good, 4, good, good, 3, 2, 16, 8, None) == 1


def test_python_binding_refuses_to_run_without_library(tmp_path, monkeypatch):
    """The product path has no fallback: with the library absent, the import fails."""
    import importlib.util
    import shutil
    pkg = tmp_path / "paged_kv_cache_158_gb300"
    shutil.copytree(os.path.join(ROOT, "paged_kv_cache_158_gb300"), pkg,
                    ignore=shutil.ignore_patterns("_lib", "_build", "__pycache__"))
    spec = importlib.util.spec_from_file_location("pa_copy_without_lib", pkg / "__init__.py",
                                                  submodule_search_locations=[str(pkg)])
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)


def test_fp8_calls_reject_bad_arguments_before_any_launch():
    lib = ctypes.CDLL(LIB)
    vp, i, fl = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    good = 0x10000
    d = lib.pa_decode_fp8
    d.argtypes = [vp, vp, vp, vp, vp, i, vp, i, i, i, i, i, fl, fl, fl, i, vp, ctypes.c_size_t, vp]
    for ks, vs in [(0.0, 1.0), (1.0, -1.0), (float("inf"), 1.0), (1.0, float("nan"))]:
        assert d(good, good, good, good, good, 4, good, 2, 2, 128, 16, 8, 0.1, ks, vs, 64, good,
                 1 << 20, None) == 1
    assert d(good, good, good, good, good, 4, good, 2, 2, 96, 16, 8, 0.1, 1.0, 1.0, 64, good,
             1 << 20, None) == 2
    assert d(good, good + 8, good, good, good, 4, good, 2, 2, 128, 16, 8, 0.1, 1.0, 1.0, 64, good,
             1 << 20, None) == 1
    assert d(None, None, None, None, None, 4, None, 0, 2, 128, 16, 8, 0.1, 1.0, 1.0, 64, None, 0,
             None) == 0
    r = lib.pa_reshape_and_cache_fp8
    r.argtypes = [vp, vp, vp, vp, vp] + [i] * 5 + [fl, fl, vp]
    assert r(good, good, good, good, good, 3, 2, 128, 16, 8, 0.0, 1.0, None) == 1
    assert r(good, good, good, good, good, 3, 2, 64, 12, 8, 1.0, 1.0, None) == 2
    assert r(good, good, good + 8, good, good, 3, 2, 64, 16, 8, 1.0, 1.0, None) == 1
    assert r(None, None, None, None, None, 0, 2, 128, 16, 8, 1.0, 1.0, None) == 0
    c = lib.pa_copy_blocks_fp8
    c.argtypes = [vp, vp, i, vp, i, i, i, i, i, vp]
    ptrs = (ctypes.c_void_p * 1)(good + 8)
    assert c(ptrs, ptrs, 1, good, 2, 2, 128, 16, 8, None) == 1
    assert c(None, None, 0, None, 0, 2, 128, 16, 8, None) == 0
    v = lib.pa_convert_cache_fp8
    v.argtypes = [vp, vp, ctypes.c_size_t, fl, vp]
    assert v(good, good, 24, 1.0, None) == 1                           # not a multiple of 16
    assert v(good, good, 32, -1.0, None) == 1
    assert v(good + 8, good, 32, 1.0, None) == 1
    assert v(None, None, 0, 1.0, None) == 0


def test_swap_rejects_bad_arguments_before_any_launch():
    lib = ctypes.CDLL(LIB)
    vp = ctypes.c_void_p
    f = lib.pa_swap_blocks
    f.argtypes = [vp, vp, ctypes.c_int, vp, ctypes.c_int, ctypes.c_size_t, ctypes.c_int64,
                  ctypes.c_int64, vp]
    good = 0x10000
    ptrs = (ctypes.c_void_p * 1)(good)
    assert f(ptrs, ptrs, 1, good, 2, 24, 8, 8, None) == 1            # block bytes not a multiple of 16
    assert f(ptrs, ptrs, 1, good, 2, 0, 8, 8, None) == 1
    assert f(ptrs, ptrs, 1, good, 2, 64, 0, 8, None) == 1           # empty pool
    assert f(ptrs, ptrs, 1, good + 4, 2, 64, 8, 8, None) == 1       # misaligned mapping
    assert f(None, None, 0, None, 0, 64, 8, 8, None) == 0           # nothing to do


def test_prefill_rejects_bad_arguments_before_any_launch():
    lib = ctypes.CDLL(LIB)
    vp, i = ctypes.c_void_p, ctypes.c_int
    f = lib.pa_prefill
    f.argtypes = [vp, vp, vp, vp, vp, i, vp, vp, i, i, i, i, i, i, ctypes.c_float, i, vp]
    g = 0x10000
    assert f(g, g, g, g, g, 4, g, g, 2, 10, 2, 96, 16, 8, 0.1, 8, None) == 2    # head_dim
    assert f(g, g, g, g, g, 4, g, g, 2, 10, 2, 128, 4, 8, 0.1, 8, None) == 2    # block_size 4
    assert f(g + 8, g, g, g, g, 4, g, g, 2, 10, 2, 128, 16, 8, 0.1, 8, None) == 1
    assert f(g, g, g, g, g, 4, g, g + 2, 2, 10, 2, 128, 16, 8, 0.1, 8, None) == 1
    assert f(g, g, g, g, g, 4, g, g, 2, 10, 2, 128, 16, 8, 0.1, -1, None) == 1
    assert f(None, None, None, None, None, 4, None, None, 0, 0, 2, 128, 16, 8, 0.1, 8, None) == 0
    assert f(g, g, g, g, g, 4, g, g, 2, 10, 2, 128, 16, 1 << 27, 0.1, 8, None) == 2   # rows >= 2^31
    f8 = lib.pa_prefill_fp8
    fl = ctypes.c_float
    f8.argtypes = [vp, vp, vp, vp, vp, i, vp, vp, i, i, i, i, i, i, fl, fl, fl, i, vp]
    assert f8(g, g, g, g, g, 4, g, g, 2, 10, 2, 96, 16, 8, 0.1, 1.0, 1.0, 8, None) == 2   # head_dim
    for ks, vs in ((0.0, 1.0), (1.0, -1.0), (float("inf"), 1.0), (1.0, float("nan"))):
        assert f8(g, g, g, g, g, 4, g, g, 2, 10, 2, 128, 16, 8, 0.1, ks, vs, 8, None) == 1
    assert f8(g + 4, g, g, g, g, 4, g, g, 2, 10, 2, 128, 16, 8, 0.1, 1.0, 1.0, 8, None) == 1
    assert f8(None, None, None, None, None, 4, None, None, 0, 0, 2, 128, 16, 8, 0.1, 1.0, 1.0, 8,
              None) == 0
    fx = lib.pa_prefill_ex
    u = ctypes.c_uint
    fx.argtypes = [vp, vp, vp, vp, vp, i, vp, vp, i, i, i, i, i, i, ctypes.c_float, i, i, u, vp]
    assert fx(g, g, g, g, g, 4, g, g, 2, 10, 2, 128, 16, 8, 0.1, 8, -1, 0x1, None) == 1  # unknown flag
    assert fx(g, g, g, g, g, 4, g, g, 2, 10, 2, 128, 16, 8, 0.1, 8, -1, 0x6, None) == 1
    assert fx(g + 8, g, g, g, g, 4, g, g, 2, 10, 2, 128, 16, 8, 0.1, 8, -1, 0x2, None) == 1
    assert fx(None, None, None, None, None, 4, None, None, 0, 0, 2, 128, 16, 8, 0.1, 8, -1, 0x2,
              None) == 0
    # The count of one-token sequences: -1 (unknown) or 0 .. min(num_seqs, num_query_tokens).
    assert fx(g, g, g, g, g, 4, g, g, 2, 10, 2, 128, 16, 8, 0.1, 8, -2, 0, None) == 1
    assert fx(g, g, g, g, g, 4, g, g, 2, 10, 2, 128, 16, 8, 0.1, 8, 3, 0, None) == 1
    assert fx(g, g, g, g, g, 4, g, g, 3, 2, 2, 128, 16, 8, 0.1, 8, 3, 0, None) == 1
    assert fx(None, None, None, None, None, 4, None, None, 0, 0, 2, 128, 16, 8, 0.1, 8, 0, 0,
              None) == 0
    f8x = lib.pa_prefill_fp8_ex
    f8x.argtypes = [vp, vp, vp, vp, vp, i, vp, vp, i, i, i, i, i, i, fl, fl, fl, i, i, u, vp]
    assert f8x(g, g, g, g, g, 4, g, g, 2, 10, 2, 128, 16, 8, 0.1, 1.0, 1.0, 8, -1, 0x4, None) == 1
    assert f8x(g, g, g, g, g, 4, g, g, 2, 10, 2, 128, 16, 8, 0.1, 0.0, 1.0, 8, -1, 0x2, None) == 1
    assert f8x(g, g, g, g, g, 4, g, g, 2, 10, 2, 128, 16, 8, 0.1, 1.0, 1.0, 8, 5, 0x2, None) == 1


def test_partition_size_follows_batch_size():
    """Small batches (fewer than 4096 items of 512 tokens) take 256-token partitions, larger
    ones 512; the override wins and is rounded up to a multiple of 32 (host-only logic)."""
    import paged_kv_cache_158_gb300 as pa
    try:
        assert pa.pa_decode_partition_tokens(32, 40, 1024) == 256       # 2560 items
        assert pa.pa_decode_partition_tokens(256, 32, 4096) == 512      # 65536 items
        assert pa.pa_decode_partition_tokens(64, 32, 2056) == 512       # 10240 items
        assert pa.pa_decode_partition_tokens(1, 1, 0) == 256            # empty contexts
        pa.pa_decode_set_partition_tokens(100)
        assert pa.pa_decode_partition_tokens(256, 32, 4096) == 128
    finally:
        pa.pa_decode_set_partition_tokens(0)


def test_plain_c_caller_links_and_gets_host_side_answers(tmp_path):
    """A C program (tests/c_abi/host_paths.c) compiled against include/pa.h and linked with
    libpa.so, no Python in between: status strings, workspace and partition sizes, and bad
    arguments refused before any CUDA call."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "host_paths"
    lib_dir = os.path.dirname(LIB)
    subprocess.run([gcc, "-std=c11", "-O1", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi", "host_paths.c"), "-L", lib_dir, "-lpa",
                    "-Wl,-rpath," + lib_dir, "-o", str(exe)], check=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert res.returncode == 0 and res.stdout.strip() == "ok", res.stdout + res.stderr
