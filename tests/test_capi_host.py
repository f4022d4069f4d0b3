"""The C-ABI library without a GPU: it loads, exports every function that
include/kv4mla.h declares, and rejects bad arguments on the host before any
device call.  Also checks the oracle library's exports."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared(header):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kv4(?:ref)?_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from bit_kv_cache_nvfp4_gb300 import build
    return ctypes.CDLL(build.build())


def test_exports_every_declared_symbol(lib):
    names = declared(os.path.join(ROOT, "include", "kv4mla.h"))
    assert "kv4_sparse_mla_decode" in names and "kv4_quantize_write" in names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_header_declares_every_exported_symbol(lib):
    """Every kv4_* function the library exports is declared in the header."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    from bit_kv_cache_nvfp4_gb300 import build
    out = subprocess.run([nm, "-D", "--defined-only", build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout.split()
    exported = sorted({w for w in out if re.fullmatch(r"kv4_[a-z0-9_]+", w)})
    names = set(declared(os.path.join(ROOT, "include", "kv4mla.h")))
    assert exported and not [n for n in exported if n not in names]


def test_oracle_exports_every_declared_symbol():
    import oracle
    olib = ctypes.CDLL(oracle.build())
    names = declared(os.path.join(ROOT, "oracle", "kv4ref.h"))
    assert not [n for n in names if not hasattr(olib, n)]


def test_status_strings_and_version(lib):
    lib.kv4_status_str.restype = ctypes.c_char_p
    assert lib.kv4_status_str(0) == b"ok"
    assert b"workspace" in lib.kv4_status_str(5)
    assert lib.kv4_version() >= 1


def test_host_side_validation_needs_no_device(lib):
    P, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.kv4_quantize_write.argtypes = [P, i64, P, i64, P, i64, P, i64, P, P]
    assert lib.kv4_quantize_write(None, 512, None, 64, None, -1, None, 10, None, None) == 1
    assert lib.kv4_quantize_write(None, 512, None, 64, None, 0, None, 10, None, None) == 0
    # 16 tokens with null pointers
    assert lib.kv4_quantize_write(None, 512, None, 64, None, 16, None, 10, None, None) == 1
    s, ws = ctypes.c_int(), ctypes.c_size_t()
    lib.kv4_decode_plan.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_int),
                                                         ctypes.POINTER(ctypes.c_size_t)]
    assert lib.kv4_decode_plan(1, 1, 48, 128, 0, ctypes.byref(s), ctypes.byref(ws)) == 2
    assert lib.kv4_decode_plan(1, 0, 64, 128, 0, ctypes.byref(s), ctypes.byref(ws)) == 1
    lib.kv4_set_wait_limit.argtypes = [i64, ctypes.c_int]
    assert lib.kv4_set_wait_limit(-1, 0) == 1
    assert lib.kv4_set_wait_limit(0, 5) == 1
    assert lib.kv4_set_wait_limit(0, 0) == 0
    f = ctypes.c_float
    lib.kv4_sparse_mla_decode.argtypes = [P, P, i64, P, i64, ctypes.c_int, P, ctypes.c_int, P,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int, f, P, P, P,
                                          ctypes.c_size_t, ctypes.c_int, P, P]
    # page size other than 64
    assert lib.kv4_sparse_mla_decode(None, None, 64, None, 1, 32, None, 8, None, 1, 1, 16, 0.1,
                                     None, None, None, 0, 0, None, None) == 2
    # empty batch is a no-op
    assert lib.kv4_sparse_mla_decode(None, None, 64, None, 1, 64, None, 8, None, 0, 1, 16, 0.1,
                                     None, None, None, 0, 0, None, None) == 0


def test_binding_fails_loudly_without_cuda_tensors():
    import torch
    import bit_kv_cache_nvfp4_gb300 as kv
    with pytest.raises(TypeError):
        kv.quantize_write(torch.zeros(1, 512, dtype=torch.bfloat16),
                          torch.zeros(1, 64, dtype=torch.bfloat16),
                          torch.zeros(1, dtype=torch.int64), torch.zeros(64, 352, dtype=torch.uint8))


def test_binding_constants_match_header():
    """The binding's layout constants are the header's enum values."""
    import bit_kv_cache_nvfp4_gb300 as kv
    text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "kv4mla.h")).read(), flags=re.S)
    values = {k: int(v) for k, v in re.findall(r"\bKV4_([A-Z0-9_]+)\s*=\s*(\d+)", text)}
    for name in ("ROW_BYTES", "LATENT", "ROPE", "QK_DIM", "PAGE", "TILE_KEYS", "ROW_BYTES_LATENT",
                 "ROW_BYTES_FP8"):
        assert getattr(kv, name) == values[name], name


def test_write_and_decode_checks_both_parts_first(lib):
    """kv4_quantize_write_and_decode refuses a bad decode argument before it
    launches the write, and a bad write argument before anything else."""
    P, i64, i32, f = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    fn = lib.kv4_quantize_write_and_decode
    fn.argtypes = [P, i64, P, i64, P, i64, P, i64,
                   P, P, i64, i32, P, i32, P, i32, i32, i32, f, P, P, P, ctypes.c_size_t, i32, P,
                   P]
    fn.restype = i32
    buf = ctypes.create_string_buffer(1 << 12)
    ptr = ctypes.cast(buf, P)
    # a page size other than 64 (decode) -> unsupported, with a valid-looking write
    assert fn(ptr, 512, ptr, 64, ptr, 4, ptr, 64,
              ptr, ptr, 1, 32, ptr, 8, ptr, 1, 1, 16, 0.1, ptr, ptr, None, 0, 0, None, None) == 2
    # an unsupported head count (decode) -> unsupported
    assert fn(ptr, 512, ptr, 64, ptr, 4, ptr, 64,
              ptr, ptr, 1, 64, ptr, 8, ptr, 1, 1, 48, 0.1, ptr, ptr, None, 0, 0, None, None) == 2
    # null decode outputs -> invalid argument
    assert fn(ptr, 512, ptr, 64, ptr, 4, ptr, 64,
              ptr, ptr, 1, 64, ptr, 8, ptr, 1, 1, 16, 0.1, None, None, None, 0, 0, None,
              None) == 1


def test_noalloc_checks_arguments_before_its_scratch_limit(lib):
    """kv4_sparse_mla_decode_noalloc reports bad pointers and unsupported
    shapes as such, before it looks at the size of its scratch array or at
    the device."""
    P, i64, i32, f = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    fn = lib.kv4_sparse_mla_decode_noalloc
    fn.argtypes = [P, P, i64, P, i64, i32, P, i32, P, i32, i32, i32, f, P, P, i32, P, P]
    fn.restype = i32
    buf = ctypes.create_string_buffer(1 << 12)
    a = (ctypes.addressof(buf) + 255) & ~255          # 256-byte aligned inside buf
    ok = ctypes.c_void_p(a)
    odd = ctypes.c_void_p(a + 4)                        # 4-byte aligned only
    # a large shape (16 splits of 16 x 64 heads would exceed the array) but a
    # null q: invalid argument, not a scratch-limit refusal
    assert fn(None, ok, 64, ok, 1, 64, ok, 2048, ok, 16, 1, 64, 0.1, ok, ok, 16, None,
              None) == 1
    # null out / lse
    assert fn(ok, ok, 64, ok, 1, 64, ok, 2048, ok, 16, 1, 64, 0.1, None, ok, 16, None,
              None) == 1
    assert fn(ok, ok, 64, ok, 1, 64, ok, 2048, ok, 16, 1, 64, 0.1, ok, None, 16, None,
              None) == 1
    # misaligned output
    assert fn(ok, ok, 64, ok, 1, 64, ok, 2048, ok, 16, 1, 64, 0.1, odd, ok, 16, None,
              None) == 1
    # unsupported page size and head count
    assert fn(ok, ok, 64, ok, 1, 32, ok, 2048, ok, 16, 1, 64, 0.1, ok, ok, 16, None,
              None) == 2
    assert fn(ok, ok, 64, ok, 1, 64, ok, 2048, ok, 16, 1, 48, 0.1, ok, ok, 16, None,
              None) == 2
    # an empty batch is a no-op
    assert fn(None, None, 64, None, 1, 64, None, 8, None, 0, 1, 16, 0.1, None, None, 0, None,
              None) == 0


def test_host_pipe_checks_arguments_without_a_device(lib):
    """The host-buffer pipe entry points refuse null handles and outputs and
    unsupported shapes before any device call."""
    P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    lib.kv4_host_pipe_bytes.argtypes = [i32, i32, i32, i32, i64, i32, ctypes.POINTER(sz)]
    lib.kv4_host_pipe_create.argtypes = [i32, i32, i32, i32, i64, i32, P, sz, P, P, P,
                                         ctypes.POINTER(P)]
    lib.kv4_host_pipe_step.argtypes = [P, P, P, P, i64, P, i64, P, i64, i32, P, P, P,
                                       ctypes.c_float, P, P, P]
    lib.kv4_host_pipe_destroy.argtypes = [P]
    n = sz()
    assert lib.kv4_host_pipe_bytes(1, 1, 64, 2048, 1, 0, None) == 1
    assert lib.kv4_host_pipe_bytes(1, 1, 48, 2048, 1, 0, ctypes.byref(n)) == 2
    assert lib.kv4_host_pipe_bytes(1, 0, 64, 2048, 1, 0, ctypes.byref(n)) == 1
    assert lib.kv4_host_pipe_bytes(0, 1, 64, 2048, 1, 0, ctypes.byref(n)) == 1
    assert lib.kv4_host_pipe_bytes(1, 1, 64, 2048, -1, 0, ctypes.byref(n)) == 1
    assert lib.kv4_host_pipe_create(1, 1, 64, 2048, 1, 0, None, 0, None, None, None, None) == 1
    assert lib.kv4_host_pipe_step(None, None, None, None, 0, None, 0, None, 1, 64, None, None,
                                  None, 0.1, None, None, None) == 1
    assert lib.kv4_host_pipe_destroy(None) == 1


def test_dcp_compaction_and_counted_decode_check_arguments(lib):
    """The compaction and the counted partial decode refuse bad arguments
    before any device call."""
    P, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    c = lib.kv4_dcp_compact_topk
    c.argtypes = [P, P, i64, P, i32, i32, i32, i32, i32, P, P, P]
    c.restype = i32
    buf = ctypes.create_string_buffer(1 << 12)
    ptr = ctypes.cast(buf, P)
    assert c(ptr, ptr, 1, ptr, 1, 1, 8, 2, 2, ptr, ptr, None) == 1     # rank >= world
    assert c(ptr, ptr, 1, ptr, 1, 1, 8, 2, 0, ptr, None, None) == 1    # no count output
    assert c(ptr, ptr, 1, ptr, 1, 1, 8, 2, 0, ptr, ptr, None) == 1     # output overlaps input
    assert c(None, None, 1, None, 0, 1, 8, 2, 0, None, None, None) == 0  # empty batch
    d = lib.kv4_sparse_mla_decode_partial_counted
    f = ctypes.c_float
    d.argtypes = [P, P, i64, P, i64, i32, P, i32, P, P, i32, i32, i32, f, P, P, P,
                  ctypes.c_size_t, i32, P, P]
    d.restype = i32
    # no count array
    assert d(ptr, ptr, 64, ptr, 1, 64, ptr, 8, None, ptr, 1, 1, 16, 0.1, ptr, ptr, None, 0, 0,
             None, None) == 1
