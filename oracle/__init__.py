"""CPU oracle for NVFP4 latent-KV sparse-MLA decode -- TEST INFRASTRUCTURE.

This package is the plain, single-threaded C++ definition of what the GPU
path computes (``kv4ref.h`` documents the byte layout, the quantizer and the
attention).  Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs may import it.  The product
library (``bit_kv_cache_nvfp4_gb300``) never imports it, and the two share
no source, header, table or helper.

``build()`` compiles ``libkv4ref.so`` next to this file with g++ (-O2, no
OpenMP, no SIMD intrinsics, ``-ffp-contract=off`` so that x86 and Arm hosts
round identically).  The wrappers below take numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SOURCES = ["kv4ref_codec.cpp", "kv4ref_attention.cpp"]
_LIB_PATH = os.path.join(_HERE, "libkv4ref.so")
_lock = threading.Lock()
_lib = None

OK = 0
ERR_ARG = 1
ERR_SLOT = 2
ERR_PAGE = 3


def build(force: bool = False) -> str:
    """Compile the oracle library in place; returns its path."""
    srcs = [os.path.join(_HERE, s) for s in _SOURCES]
    hdr = os.path.join(_HERE, "kv4ref.h")
    if not force and os.path.exists(_LIB_PATH):
        newest = max(os.path.getmtime(p) for p in srcs + [hdr])
        if os.path.getmtime(_LIB_PATH) >= newest:
            return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp] + srcs
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32, i64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_float
        lib.kv4ref_enc_e4m3.argtypes = [f32]
        lib.kv4ref_enc_e4m3.restype = ctypes.c_uint8
        lib.kv4ref_dec_e4m3.argtypes = [ctypes.c_uint8]
        lib.kv4ref_dec_e4m3.restype = f32
        lib.kv4ref_enc_e2m1.argtypes = [f32]
        lib.kv4ref_enc_e2m1.restype = ctypes.c_uint8
        lib.kv4ref_dec_e2m1.argtypes = [ctypes.c_uint8]
        lib.kv4ref_dec_e2m1.restype = f32
        lib.kv4ref_enc_e4m3_n.argtypes = [P, P, i64]
        lib.kv4ref_enc_e4m3_n.restype = None
        lib.kv4ref_enc_e2m1_n.argtypes = [P, P, i64]
        lib.kv4ref_enc_e2m1_n.restype = None
        lib.kv4ref_quantize_row.argtypes = [P, P, P]
        lib.kv4ref_quantize_row.restype = None
        lib.kv4ref_dequant_row.argtypes = [P, P]
        lib.kv4ref_dequant_row.restype = None
        lib.kv4ref_quantize_write.argtypes = [P, i64, P, i64, P, i64, P, i64]
        lib.kv4ref_quantize_write.restype = i32
        lib.kv4ref_quantize_write_fp8.argtypes = [P, i64, P, i64, P, i64, P, i64]
        lib.kv4ref_quantize_write_fp8.restype = i32
        lib.kv4ref_dequant_row_fp8.argtypes = [P, P]
        lib.kv4ref_dequant_row_fp8.restype = None
        lib.kv4ref_fp8_scratch.argtypes = [P, i64, P, i64, i32, P, i32, P, i32, i32, P]
        lib.kv4ref_fp8_scratch.restype = i32
        lib.kv4ref_quantize_row_mse.argtypes = [P, P, P]
        lib.kv4ref_quantize_row_mse.restype = None
        lib.kv4ref_quantize_write_mse.argtypes = [P, i64, P, i64, P, i64, P, i64]
        lib.kv4ref_quantize_write_mse.restype = i32
        lib.kv4ref_resolve_slots.argtypes = [P, i64, i32, P, i32, P, i32, i32, i64, P]
        lib.kv4ref_resolve_slots.restype = i32
        lib.kv4ref_gather_dequant.argtypes = [P, i64, P, i64, i32, P, i32, P, i32, i32, P, P]
        lib.kv4ref_gather_dequant.restype = i32
        lib.kv4ref_sparse_mla_decode.argtypes = [P, P, i64, P, i64, i32, P, i32, P,
                                                 i32, i32, i32, f32, i32, P, P]
        lib.kv4ref_sparse_mla_decode.restype = i32
        lib.kv4ref_sparse_mla_decode_fp8.argtypes = lib.kv4ref_sparse_mla_decode.argtypes
        lib.kv4ref_sparse_mla_decode_fp8.restype = i32
        lib.kv4ref_merge.argtypes = [P, P, i32, i32, i32, P, P]
        lib.kv4ref_merge.restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle wrappers need C-contiguous arrays"
    return a.ctypes.data_as(ctypes.c_void_p)


def _as(a, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == dtype, f"expected {dtype}, got {a.dtype}"
    return a


# ---- scalar codecs ---------------------------------------------------------
def enc_e4m3(x: float) -> int:
    return int(_load().kv4ref_enc_e4m3(float(x)))


def dec_e4m3(c: int) -> float:
    return float(_load().kv4ref_dec_e4m3(int(c)))


def enc_e2m1(x: float) -> int:
    return int(_load().kv4ref_enc_e2m1(float(x)))


def dec_e2m1(c: int) -> float:
    return float(_load().kv4ref_dec_e2m1(int(c)))


def enc_e4m3_array(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().kv4ref_enc_e4m3_n(_ptr(x), _ptr(out), x.size)
    return out


def enc_e2m1_array(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().kv4ref_enc_e2m1_n(_ptr(x), _ptr(out), x.size)
    return out


# ---- rows ------------------------------------------------------------------
def quantize_row(latent_bits: np.ndarray, rope_bits: np.ndarray) -> np.ndarray:
    """latent_bits uint16[512], rope_bits uint16[64] (bf16 bit patterns)."""
    lat = _as(latent_bits, np.uint16)
    rope = _as(rope_bits, np.uint16)
    assert lat.size == 512 and rope.size == 64
    row = np.zeros(352, dtype=np.uint8)
    _load().kv4ref_quantize_row(_ptr(lat), _ptr(rope), _ptr(row))
    return row


def quantize_row_mse(latent_bits: np.ndarray, rope_bits: np.ndarray) -> np.ndarray:
    """The row with MSE-searched block scales (see kv4ref.h)."""
    lat = _as(latent_bits, np.uint16)
    rope = _as(rope_bits, np.uint16)
    assert lat.size == 512 and rope.size == 64
    row = np.zeros(352, dtype=np.uint8)
    _load().kv4ref_quantize_row_mse(_ptr(lat), _ptr(rope), _ptr(row))
    return row


def dequant_row(row: np.ndarray) -> np.ndarray:
    row = _as(row, np.uint8)
    assert row.size == 352
    out = np.zeros(576, dtype=np.float32)
    _load().kv4ref_dequant_row(_ptr(row), _ptr(out))
    return out


def quantize_write(latent_bits, rope_bits, slot_mapping, pool) -> int:
    """latent_bits uint16[N,>=512], rope_bits uint16[N,>=64], slots int64[N];
    pool uint8[num_slots,352] is written in place.  Returns the status."""
    lat = _as(latent_bits, np.uint16)
    rope = _as(rope_bits, np.uint16)
    slots = _as(slot_mapping, np.int64)
    assert pool.dtype == np.uint8 and pool.flags["C_CONTIGUOUS"]
    n = slots.shape[0]
    return int(_load().kv4ref_quantize_write(
        _ptr(lat), lat.shape[1] if lat.ndim == 2 else 512,
        _ptr(rope), rope.shape[1] if rope.ndim == 2 else 64,
        _ptr(slots), n, _ptr(pool), pool.shape[0]))


def quantize_write_mse(latent_bits, rope_bits, slot_mapping, pool) -> int:
    """quantize_write with MSE-searched block scales."""
    lat = _as(latent_bits, np.uint16)
    rope = _as(rope_bits, np.uint16)
    slots = _as(slot_mapping, np.int64)
    assert pool.dtype == np.uint8 and pool.flags["C_CONTIGUOUS"]
    n = slots.shape[0]
    return int(_load().kv4ref_quantize_write_mse(
        _ptr(lat), lat.shape[1] if lat.ndim == 2 else 512,
        _ptr(rope), rope.shape[1] if rope.ndim == 2 else 64,
        _ptr(slots), n, _ptr(pool), pool.shape[0]))


def resolve_slots(page_table, topk_idx, seq_lens, num_slots, page_size=64):
    pt = _as(page_table, np.int32)
    topk = _as(topk_idx, np.int32)
    sl = _as(seq_lens, np.int32)
    B, Sq, K = topk.shape
    slots = np.empty((B, Sq, K), dtype=np.int64)
    st = _load().kv4ref_resolve_slots(_ptr(pt), pt.shape[1], page_size, _ptr(topk), K,
                                      _ptr(sl), B, Sq, int(num_slots), _ptr(slots))
    return st, slots


def gather_dequant(pool, page_table, topk_idx, seq_lens, page_size=64):
    pool = _as(pool, np.uint8)
    pt = _as(page_table, np.int32)
    topk = _as(topk_idx, np.int32)
    sl = _as(seq_lens, np.int32)
    B, Sq, K = topk.shape
    rows = np.empty((B, Sq, K, 576), dtype=np.float32)
    valid = np.empty((B, Sq, K), dtype=np.uint8)
    st = _load().kv4ref_gather_dequant(_ptr(pool), pool.shape[0], _ptr(pt), pt.shape[1],
                                       page_size, _ptr(topk), K, _ptr(sl), B, Sq,
                                       _ptr(rows), _ptr(valid))
    return st, rows, valid


def sparse_mla_decode(q_bits, pool, page_table, topk_idx, seq_lens, sm_scale,
                      splits=1, page_size=64, fp8_rows=False):
    """q_bits uint16[B,Sq,H,576] -> (status, out fp32[B,Sq,H,512], lse fp32[B,Sq,H]).
    pool rows: 352-byte NVFP4, or 576-byte FP8 with fp8_rows=True."""
    q = _as(q_bits, np.uint16)
    pool = _as(pool, np.uint8)
    pt = _as(page_table, np.int32)
    topk = _as(topk_idx, np.int32)
    sl = _as(seq_lens, np.int32)
    B, Sq, H, D = q.shape
    assert D == 576 and topk.shape[:2] == (B, Sq)
    K = topk.shape[2]
    out = np.empty((B, Sq, H, 512), dtype=np.float32)
    lse = np.empty((B, Sq, H), dtype=np.float32)
    fn = _load().kv4ref_sparse_mla_decode_fp8 if fp8_rows else _load().kv4ref_sparse_mla_decode
    st = fn(_ptr(q), _ptr(pool), pool.shape[0], _ptr(pt), pt.shape[1], page_size, _ptr(topk), K,
            _ptr(sl), B, Sq, H, float(sm_scale), int(splits), _ptr(out), _ptr(lse))
    return st, out, lse


def quantize_write_fp8(latent_bits, rope_bits, slot_mapping, pool) -> int:
    """576-byte FP8 rows (E4M3 of every latent and rope value) into pool
    uint8[num_slots,576]."""
    lat = _as(latent_bits, np.uint16)
    rope = _as(rope_bits, np.uint16)
    slots = _as(slot_mapping, np.int64)
    assert pool.dtype == np.uint8 and pool.flags["C_CONTIGUOUS"] and pool.shape[1] == 576
    return int(_load().kv4ref_quantize_write_fp8(
        _ptr(lat), lat.shape[1] if lat.ndim == 2 else 512,
        _ptr(rope), rope.shape[1] if rope.ndim == 2 else 64,
        _ptr(slots), slots.shape[0], _ptr(pool), pool.shape[0]))


def dequant_row_fp8(row: np.ndarray) -> np.ndarray:
    row = _as(row, np.uint8)
    assert row.size == 576
    out = np.zeros(576, dtype=np.float32)
    _load().kv4ref_dequant_row_fp8(_ptr(row), _ptr(out))
    return out


def fp8_scratch(pool, page_table, topk_idx, seq_lens, page_size=64):
    """(status, scratch uint8[B*Sq*K, 576]): the FP8 copy of the rows the keys
    select (zero rows for masked keys)."""
    pool = _as(pool, np.uint8)
    pt = _as(page_table, np.int32)
    topk = _as(topk_idx, np.int32)
    sl = _as(seq_lens, np.int32)
    B, Sq, K = topk.shape
    scratch = np.empty((B * Sq * K, 576), dtype=np.uint8)
    st = _load().kv4ref_fp8_scratch(_ptr(pool), pool.shape[0], _ptr(pt), pt.shape[1], page_size,
                                    _ptr(topk), K, _ptr(sl), B, Sq, _ptr(scratch))
    return st, scratch


def merge(o_parts, lse_parts):
    """o_parts fp32[S,n,D], lse_parts fp32[S,n] -> (out fp32[n,D], lse fp32[n])."""
    o = _as(o_parts, np.float32)
    l = _as(lse_parts, np.float32)
    S, n, D = o.shape
    out = np.empty((n, D), dtype=np.float32)
    lse = np.empty((n,), dtype=np.float32)
    _load().kv4ref_merge(_ptr(o), _ptr(l), S, n, D, _ptr(out), _ptr(lse))
    return out, lse
