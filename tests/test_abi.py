"""The C-ABI library loads without a GPU and exports every symbol its header declares."""
import ctypes
import os
import re
import subprocess

import pytest

import paged_kv_cache_80_gb300 as pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for required in ["pkv_pool_create", "pkv_append_kv", "pkv_decode_attention", "pkv_copy_blocks",
                     "pkv_swap_out", "pkv_swap_in", "pkv_plan_append", "pkv_seq_fork", "pkv_seq_free",
                     "pkv_check_device_error"]:
        assert required in names


def test_every_declared_symbol_is_exported():
    lib = ctypes.CDLL(pkv.library_path())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.library_path()], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (pkv_[a-z_0-9]+)$", out, flags=re.M))
    assert set(declared_functions()) <= exported


def test_library_is_built_for_sm103a_only():
    # the build compiles every source with exactly one -gencode: sm_103a machine code
    from paged_kv_cache_80_gb300 import build

    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


@pytest.mark.gpu
def test_loaded_device_code_is_sm103():
    # what the runtime loaded for this device: sm_103a machine code (binaryVersion 103)
    binary, ptx = pkv.pkv_device_code_version()
    assert binary == 103, binary


def test_version_and_status_names():
    assert pkv.pkv_version() == 1
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_pool_create(1, 3, 2, 8, 4, "bf16", 16)  # H_q not a multiple of H_kv
    assert e.value.name == "PKV_ERR_INVALID_ARG"
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_pool_create(1, 2, 2, 8, 4, 7, 16)
    assert e.value.name == "PKV_ERR_UNSUPPORTED"
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_pool_create(1, 2, 2, 8, 4, "bf16", 4, initial_free_order=[0, 1, 1, 2])
    assert e.value.name == "PKV_ERR_INVALID_ARG"
