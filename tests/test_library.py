"""The C-ABI library builds for sm_103a, loads without a GPU and exports every
function that include/echo.h declares.  No compute calls (no GPU here)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "echo.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:echo_status_t|size_t|int32_t|void)\s+(echo_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for n in ["echo_index_prefetch", "echo_topk", "echo_cache_alloc", "echo_cache_evict", "echo_cache_recall",
              "echo_cache_writeback", "echo_cache_reserve", "echo_sparse_mla_decode", "echo_decode_layer_step",
              "echo_cache_metadata_bytes"]:
        assert n in names


def test_library_builds_and_exports_every_declared_symbol():
    from sparse_attention_kv_dsa_gb300 import build as B
    path = B.build()
    lib = ctypes.CDLL(path)
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} not exported"


def test_binding_signatures_cover_the_header():
    import sparse_attention_kv_dsa_gb300.echo as E
    assert set(E.SIGNATURES) == set(declared_functions())


def test_binding_struct_layouts_match_the_library():
    import ctypes as C
    import sparse_attention_kv_dsa_gb300.echo as E
    out = (C.c_size_t * 3)()
    E.lib().echo_abi_struct_sizes(out)
    assert list(out) == [C.sizeof(E.CacheLayerT), C.sizeof(E.StepArgsT), C.sizeof(E.HostPoolT)]


def test_metadata_closed_form_through_the_abi():
    import sparse_attention_kv_dsa_gb300.echo as E
    assert E.metadata_bytes(2_000_000, 200_000) == 10_600_000
    assert E.metadata_bytes(8192, 1024) == 46_080


def test_kernels_target_sm103a():
    # the object files carry sm_103a code only (checked through nvcc's own listing)
    import shutil
    import subprocess
    from sparse_attention_kv_dsa_gb300 import build as B
    B.build()
    tool = shutil.which("cuobjdump") or "/usr/local/cuda/bin/cuobjdump"
    if not os.path.exists(tool):
        pytest.skip("cuobjdump not available")
    out = subprocess.run([tool, "--list-elf", B.LIB], capture_output=True, text=True).stdout
    assert "sm_103a" in out and "sm_90" not in out


def test_binding_constants_match_the_header():
    import sparse_attention_kv_dsa_gb300.echo as E
    src = open(os.path.join(ROOT, "include", "echo.h")).read()

    def define(name):
        m = re.search(r"^#define\s+%s\s+(\S+)" % name, src, flags=re.M)
        assert m, name
        return int(m.group(1))

    assert define("ECHO_PF_DEFER_CAP") == E.PF_DEFER_CAP
    assert define("ECHO_PENDING_LIST_MIN_SLOTS") == E.PENDING_LIST_MIN_SLOTS
    m = re.search(r"ECHO_NUM_COUNTERS\s*=\s*(\d+)", src)
    assert m and int(m.group(1)) == E.NUM_COUNTERS
