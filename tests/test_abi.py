"""The C ABI library (CPU): it builds, loads, exports every function the
headers declare, and its host-side argument checks answer without a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib_path():
    from sparse_kv_offload_gb300 import build
    return build.build()


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(dd_[a-z0-9_]+)\s*\(", text))
    return names


def test_every_declared_function_is_exported(lib_path):
    declared = declared_functions()
    assert {"dd_create", "dd_step", "dd_gather_kv", "dd_sparse_attn_decode"} <= declared
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(dd_[a-z0-9_]+)$", out, flags=re.M))
    assert declared <= exported, declared - exported
    from sparse_kv_offload_gb300 import dd
    assert set(dd.EXPORTED) == declared


def test_library_is_built_for_sm_103a(lib_path):
    out = subprocess.run(["cuobjdump", "--list-elf", lib_path], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    assert "sm_103a" in out.stdout


def test_host_checks_answer_without_a_gpu(lib_path):
    from sparse_kv_offload_gb300 import dd
    assert dd.status_str(dd.DD_ERR_CAPACITY).startswith("more missing chunks")
    lib = ctypes.CDLL(lib_path)
    lib.dd_create.restype = ctypes.c_int32
    bad = dd.Dims(1, 8, 2, 64, 1024, 16, 8, 2)          # d = 64 is not supported
    h = ctypes.c_void_p()
    assert lib.dd_create(ctypes.byref(bad), ctypes.c_int64(4), ctypes.c_int64(0), ctypes.byref(h)) == dd.DD_ERR_INVALID_ARG
    bad = dd.Dims(1, 8, 2, 128, 1024, 16, 65, 2)        # k > C
    assert lib.dd_create(ctypes.byref(bad), ctypes.c_int64(4), ctypes.c_int64(0), ctypes.byref(h)) == dd.DD_ERR_INVALID_ARG
    import torch
    if not torch.cuda.is_available():
        good = dd.Dims(1, 8, 2, 128, 1024, 16, 8, 2)
        assert lib.dd_create(ctypes.byref(good), ctypes.c_int64(4), ctypes.c_int64(0), ctypes.byref(h)) == dd.DD_ERR_CUDA


# (B, Hq, Hkv, d, L, cs, k, n_q), max_misses, hot_slots: each breaks one rule dd_create checks on the host
BAD_SHAPES = {
    "negative_batch": ((-1, 8, 2, 128, 1024, 16, 8, 2), 4, 0),
    "heads_not_grouped": ((1, 6, 4, 128, 1024, 16, 8, 2), 4, 0),
    "no_kv_heads": ((1, 8, 0, 128, 1024, 16, 8, 2), 4, 0),
    "chunk_size_8": ((1, 8, 2, 128, 1024, 8, 8, 2), 4, 0),
    "chunk_size_128": ((1, 8, 2, 128, 1024, 128, 4, 2), 4, 0),
    "ragged_context": ((1, 8, 2, 128, 1000, 16, 8, 2), 4, 0),
    "k_zero": ((1, 8, 2, 128, 1024, 16, 0, 2), 4, 0),
    "more_chunks_than_supported": ((1, 8, 2, 128, 16384 * 16 + 16, 16, 8, 2), 4, 0),
    "no_query": ((1, 8, 2, 128, 1024, 16, 8, 0), 4, 0),
    "nine_queries": ((1, 8, 2, 128, 1024, 16, 8, 9), 4, 0),
    "65_query_vectors": ((1, 72, 8, 128, 1024, 16, 8, 8), 4, 0),     # n_q * G = 72
    "negative_staging": ((1, 8, 2, 128, 1024, 16, 8, 2), -1, 0),
    "staging_rows_overflow_int32": ((1, 8, 2, 128, 1024, 16, 8, 2), 1 << 27, 0),
    "hot_rows_overflow_int32": ((1, 8, 2, 128, 1024, 16, 8, 2), 4, 1 << 27),
}


@pytest.mark.parametrize("case", sorted(BAD_SHAPES))
def test_create_refuses_each_unsupported_shape(lib_path, case):
    from sparse_kv_offload_gb300 import dd
    dims, max_misses, hot_slots = BAD_SHAPES[case]
    lib = ctypes.CDLL(lib_path)
    lib.dd_create.restype = ctypes.c_int32
    h = ctypes.c_void_p(1)
    d = dd.Dims(*dims)
    r = lib.dd_create(ctypes.byref(d), ctypes.c_int64(max_misses), ctypes.c_int64(hot_slots), ctypes.byref(h))
    assert r == dd.DD_ERR_INVALID_ARG
    assert h.value is None                     # no context handed out
