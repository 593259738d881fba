"""CPU checks of the C ABI: the library loads, exports every function that
include/pkv.h declares, and rejects bad arguments on the host before any CUDA
call (no compute is launched here)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_kvh_gb300 as m
    return m


def test_every_declared_symbol_is_exported(pkv):
    names = _declared()
    assert {"pkv_store_kvcache", "pkv_prefill_varlen", "pkv_decode"} <= set(names)
    lib = ctypes.CDLL(pkv.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in pkv.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (pkv_\w+)", out))
    assert set(names) == exported, (set(names) ^ exported)
    assert set(pkv.EXPORTED) == exported       # the binding covers the whole ABI


def test_status_strings(pkv):
    for code in range(-9, 1):
        s = pkv.pkv_status_string(code)
        assert s and s != "unknown status"
    assert pkv.pkv_status_string(-1000) == "unknown status"


def test_host_side_rejections_before_any_cuda_call(pkv):
    lib = pkv._lib
    nul = None
    # negative token count, zero heads
    assert lib.pkv_store_kvcache(nul, 0, nul, 0, nul, nul, nul, -1, 8, 128, 0, nul) == -6
    assert lib.pkv_store_kvcache(nul, 0, nul, 0, nul, nul, nul, 4, 0, 128, 0, nul) == -6
    # empty call is a no-op
    assert lib.pkv_store_kvcache(nul, 0, nul, 0, nul, nul, nul, 0, 8, 128, 0, nul) == 0
    # missing pointers
    assert lib.pkv_store_kvcache(nul, 1024, nul, 1024, nul, nul, nul, 4, 8, 128, 256, nul) == -1
    # unsupported attention shapes
    args = [nul, 2048, nul, nul, 16, nul, 16, nul, 4]
    assert lib.pkv_decode(*args, 16, 8, 64, 256, 4096, 0.1, nul, nul, 0, nul) == -2     # head_dim 64
    assert lib.pkv_decode(*args, 16, 8, 128, 16, 4096, 0.1, nul, nul, 0, nul) == -2    # block_size 16
    assert lib.pkv_decode(*args, 32, 8, 128, 256, 4096, 0.1, nul, nul, 0, nul) == -2   # 32 q heads
    # nothing to do
    assert lib.pkv_decode(nul, 2048, nul, nul, 16, nul, 16, nul, 0, 16, 8, 128, 256, 4096, 0.1, nul, nul, 0,
                          nul) == 0
    # missing pointers, then bad scale
    assert lib.pkv_decode(*args, 16, 8, 128, 256, 4096, 0.1, nul, nul, 0, nul) == -1
    assert lib.pkv_decode(*args, 16, 8, 128, 256, 4096, -1.0, nul, nul, 0, nul) == -6
    # prefill: unsupported shape, empty, missing pointers
    assert lib.pkv_prefill_varlen(nul, 2048, 10, nul, nul, 1024, 10, nul, nul, 0, nul, nul, 10, 10, nul, 0, 1,
                                  16, 8, 96, 256, 0.1, nul, nul, 0, nul) == -2
    assert lib.pkv_prefill_varlen(nul, 2048, 0, nul, nul, 1024, 0, nul, nul, 0, nul, nul, 0, 0, nul, 0, 0,
                                  16, 8, 128, 256, 0.1, nul, nul, 0, nul) == 0
    assert lib.pkv_prefill_varlen(nul, 2048, 10, nul, nul, 1024, 10, nul, nul, 0, nul, nul, 10, 10, nul, 0, 1,
                                  16, 8, 128, 256, 0.1, nul, nul, 0, nul) == -1


@pytest.mark.parametrize("suffix", ["", "_f16"])
def test_typed_entry_points_share_host_checks(pkv, suffix):
    """The bf16 and fp16 entry points run the same host-side checks."""
    lib = pkv._lib
    nul = None
    dec = getattr(lib, "pkv_decode" + suffix)
    args = [nul, 2048, nul, nul, 16, nul, 16, nul, 4]
    assert dec(*args, 16, 8, 64, 256, 4096, 0.1, nul, nul, 0, nul) == -2
    assert dec(*args, 16, 8, 128, 256, 4096, 0.1, nul, nul, 0, nul) == -1
    assert dec(nul, 2048, nul, nul, 16, nul, 16, nul, 0, 16, 8, 128, 256, 4096, 0.1, nul, nul, 0, nul) == 0
    pre = getattr(lib, "pkv_prefill_varlen" + suffix)
    assert pre(nul, 2048, 10, nul, nul, 1024, 10, nul, nul, 0, nul, nul, 10, 10, nul, 0, 1,
               16, 8, 96, 256, 0.1, nul, nul, 0, nul) == -2
    assert pre(nul, 2048, 10, nul, nul, 1024, 10, nul, nul, 0, nul, nul, 10, 10, nul, 0, 1,
               16, 8, 128, 256, 0.1, nul, nul, 0, nul) == -1
    sd = getattr(lib, "pkv_store_decode" + suffix)
    # new-row pointers are checked before the decode arguments
    assert sd(nul, 2048, nul, 4096, nul, 4096, nul, nul, nul, 16, nul, 16, nul, 4, 16, 8, 128, 256, 4096, 0.1,
              nul, nul, 0, nul) == -1
    # a new-row stride shorter than the row
    one = ctypes.c_void_p(16)
    assert sd(nul, 2048, one, 512, one, 4096, one, nul, nul, 16, nul, 16, nul, 4, 16, 8, 128, 256, 4096, 0.1,
              nul, nul, 0, nul) == -3


def test_workspace_sizes(pkv):
    assert pkv.pkv_decode_workspace_bytes(0, 4096) == 0
    a = pkv.pkv_decode_workspace_bytes(256, 4096)
    b = pkv.pkv_decode_workspace_bytes(256, 2048)
    assert a > b > 0
    # partial (m, l) and o per (sequence, 256-token split, head) dominate
    assert a >= 256 * 16 * 16 * 128 * 4
    assert pkv.pkv_prefill_workspace_bytes(27, 1024) == 0
