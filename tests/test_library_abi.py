"""The C-ABI library builds, loads without a GPU and exports every function the headers in
include/ declare; host-side argument checks answer before any device is touched."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(kv_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_block_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("kv_compute_slot_mapping", "kv_reshape_and_cache", "kv_paged_attention_decode",
              "kv_paged_attention_workspace_size", "kv_status_string", "kv_decode_step",
              "kv_bm_create", "kv_bm_allocate", "kv_bm_flush", "kv_apply_block_updates"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} is declared in include/ but not exported"


def test_library_exports_nothing_undeclared():
    import subprocess
    from paged_kv_cache_block_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.build()], capture_output=True,
                         text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l and l.split()[-1].startswith("kv_")}
    assert exported == set(declared_functions())


def test_status_strings(lib):
    lib.kv_status_string.restype = ctypes.c_char_p
    assert lib.kv_status_string(0) == b"KV_OK"
    assert lib.kv_status_string(4) == b"KV_ERR_WORKSPACE"
    assert lib.kv_status_string(5) == b"KV_ERR_OUT_OF_BLOCKS"


def test_null_pointers_rejected_on_host(lib):
    lib.kv_last_error.restype = ctypes.c_char_p
    P = ctypes.c_void_p
    f = lib.kv_compute_slot_mapping
    f.argtypes = [P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, P, P, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_int32, P, P, P]
    assert f(None, 4, 1, 4, None, None, 3, 16, 10, None, None, None) == 1
    assert b"null" in lib.kv_last_error()
    # nothing to do is fine without any device
    assert f(None, 4, 1, 4, None, None, 0, 16, 10, None, None, None) == 0
