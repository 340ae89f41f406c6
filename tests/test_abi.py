"""The C ABI library loads on a machine without a GPU and exports every
entry point include/pagedkv.h declares (no compute calls here)."""

import ctypes
import os
import re

import pytest

import paged_kv_cache_128_gb300 as pk
from paged_kv_cache_128_gb300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pagedkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_expected_calls():
    names = declared_functions()
    for must in ("paged_reshape_and_cache", "paged_decode_attention", "paged_decode_workspace_size",
                 "kvbm_create", "kvbm_allocate_for_prefill", "kvbm_append_slot_for_decode", "kvbm_free_sequence",
                 "kvbm_can_allocate", "kvbm_export", "kv_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(_lib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    assert set(declared_functions()) == set(_lib.SIGNATURES)


def test_status_strings():
    lib = pk.lib()
    for code in range(12):
        s = lib.kv_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.kv_status_string(99).decode() == "unknown status"


def test_plan_is_host_only_and_validates():
    # planning needs no GPU when it cannot query one: it must still validate
    from paged_kv_cache_128_gb300 import kernels
    import torch
    with pytest.raises(pk.KVError) as e:
        kernels.decode_plan(4, 6, 4, 64, 16, 100, torch.float16)   # Hq % Hkv != 0
    assert e.value.code == "INVALID_ARG"
    with pytest.raises(pk.KVError):
        kernels.decode_plan(4, 8, 4, 60, 16, 100, torch.float16)   # D not a multiple of 8
