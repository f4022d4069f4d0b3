"""NVFP4 latent-KV cache write and sparse MLA decode for GB300 (sm_103a).

A thin Python binding over ``libkv4mla.so`` (C ABI in ``include/kv4mla.h``).
Every step of the computation runs in the library's CUDA kernels; this
module only checks tensors, passes device pointers and the current CUDA
stream, allocates outputs and the split-K workspace with PyTorch, and turns
status codes into exceptions.  There is no CPU fallback: if the library
cannot be loaded, importing the functions raises.

Row format and method: numinousmuses "inference-optimizations" README,
sections "4-bit KV cache" (352-byte NVFP4 row, kv4mla decode; the 288-byte
rope-free row of the GLM-5.3-Flash bullet, served by the ``*_latent``
functions) and "Attention kernels" (split-K sparse decode).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "Kv4Error", "library_path", "load_library", "quantize_write", "decode_plan",
    "sparse_mla_decode", "debug_gather_dequant", "set_wait_limit", "set_timing_event",
    "quantize_write_mse", "quantize_write_fp8", "decode_plan_fp8", "sparse_mla_decode_fp8",
    "fp8_scratch", "scratch_index", "ROW_BYTES_FP8", "quantize_write_and_decode", "quantize_write_latent", "decode_plan_latent", "sparse_mla_decode_latent",
    "debug_gather_dequant_latent", "sparse_mla_decode_partial", "dcp_mask_topk",
    "merge_partials", "gather_partials", "dcp_sparse_mla_decode", "dcp_local_page_table",
    "dcp_local_slots", "dcp_local_pages", "dcp_compact_topk", "ROW_BYTES", "ROW_BYTES_LATENT", "LATENT", "ROPE", "QK_DIM", "PAGE", "DEV_BAD_SLOT", "DEV_BAD_PAGE",
    "DEV_TIMEOUT", "HostPipe",
]

ROW_BYTES, LATENT, ROPE, QK_DIM, PAGE, TILE_KEYS = 352, 512, 64, 576, 64, 128
ROW_BYTES_LATENT = 288
ROW_BYTES_FP8 = 576
DEV_BAD_SLOT, DEV_BAD_PAGE, DEV_TIMEOUT = 1, 2, 4
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape or page size",
           3: "device is not compute capability 10.3", 4: "kernel launch failed",
           5: "workspace missing or too small",
           6: "split-K partials exceed the library's static scratch"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None
_workspaces: dict = {}


class Kv4Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {_STATUS.get(status, 'unknown status')} (status {status})")
        self.status = status


def library_path() -> str:
    return os.path.join(_HERE, "libkv4mla.so")


def load_library():
    """Load libkv4mla.so (building it first if the sources are newer)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        from . import build as _build
        path = _build.build()
        lib = ctypes.CDLL(path)
        P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                ctypes.c_float, ctypes.c_size_t)
        lib.kv4_quantize_write.argtypes = [P, i64, P, i64, P, i64, P, i64, P, P]
        lib.kv4_quantize_write.restype = i32
        lib.kv4_decode_plan.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(i32),
                                        ctypes.POINTER(sz)]
        lib.kv4_decode_plan.restype = i32
        lib.kv4_sparse_mla_decode.argtypes = [P, P, i64, P, i64, i32, P, i32, P, i32, i32, i32,
                                              f32, P, P, P, sz, i32, P, P]
        lib.kv4_sparse_mla_decode.restype = i32
        lib.kv4_debug_gather_dequant.argtypes = [P, i64, P, i64, i32, P, i32, P, i32, i32, P, P,
                                                 P]
        lib.kv4_debug_gather_dequant.restype = i32
        lib.kv4_quantize_write_fp8.argtypes = lib.kv4_quantize_write.argtypes
        lib.kv4_quantize_write_fp8.restype = i32
        lib.kv4_decode_plan_fp8.argtypes = lib.kv4_decode_plan.argtypes
        lib.kv4_decode_plan_fp8.restype = i32
        lib.kv4_sparse_mla_decode_fp8.argtypes = lib.kv4_sparse_mla_decode.argtypes
        lib.kv4_sparse_mla_decode_fp8.restype = i32
        lib.kv4_fp8_scratch.argtypes = lib.kv4_debug_gather_dequant.argtypes
        lib.kv4_fp8_scratch.restype = i32
        lib.kv4_quantize_write_mse.argtypes = lib.kv4_quantize_write.argtypes
        lib.kv4_quantize_write_mse.restype = i32
        lib.kv4_sparse_mla_decode_partial.argtypes = lib.kv4_sparse_mla_decode.argtypes
        lib.kv4_sparse_mla_decode_partial.restype = i32
        lib.kv4_dcp_mask_topk.argtypes = [P, P, i64, P, i32, i32, i32, i32, i32, P, P]
        lib.kv4_dcp_mask_topk.restype = i32
        lib.kv4_dcp_compact_topk.argtypes = [P, P, i64, P, i32, i32, i32, i32, i32, P, P, P]
        lib.kv4_dcp_compact_topk.restype = i32
        lib.kv4_sparse_mla_decode_partial_counted.argtypes = (
            lib.kv4_sparse_mla_decode.argtypes[:8] + [P] + lib.kv4_sparse_mla_decode.argtypes[8:])
        lib.kv4_sparse_mla_decode_partial_counted.restype = i32
        lib.kv4_dcp_local_page_table.argtypes = [P, i64, i32, i32, i32, P, P]
        lib.kv4_dcp_local_page_table.restype = i32
        lib.kv4_dcp_local_slots.argtypes = [P, i64, i32, i32, P, P]
        lib.kv4_dcp_local_slots.restype = i32
        lib.kv4_fp8_scratch_index.argtypes = [P, i32, P, i32, i32, P, P, P, P]
        lib.kv4_fp8_scratch_index.restype = i32
        lib.kv4_merge_partials.argtypes = [P, P, i32, i64, P, P, P]
        lib.kv4_merge_partials.restype = i32
        lib.kv4_quantize_write_latent.argtypes = [P, i64, P, i64, P, i64, P, P]
        lib.kv4_quantize_write_latent.restype = i32
        lib.kv4_decode_plan_latent.argtypes = lib.kv4_decode_plan.argtypes
        lib.kv4_decode_plan_latent.restype = i32
        lib.kv4_sparse_mla_decode_latent.argtypes = lib.kv4_sparse_mla_decode.argtypes
        lib.kv4_sparse_mla_decode_latent.restype = i32
        lib.kv4_debug_gather_dequant_latent.argtypes = lib.kv4_debug_gather_dequant.argtypes
        lib.kv4_debug_gather_dequant_latent.restype = i32
        lib.kv4_quantize_write_and_decode.argtypes = (lib.kv4_quantize_write.argtypes[:8] +
                                                      lib.kv4_sparse_mla_decode.argtypes[:1] +
                                                      lib.kv4_sparse_mla_decode.argtypes[3:])
        lib.kv4_quantize_write_and_decode.restype = i32
        lib.kv4_host_pipe_bytes.argtypes = [i32, i32, i32, i32, i64, i32, ctypes.POINTER(sz)]
        lib.kv4_host_pipe_bytes.restype = i32
        lib.kv4_host_pipe_create.argtypes = [i32, i32, i32, i32, i64, i32, P, sz, P, P, P,
                                             ctypes.POINTER(P)]
        lib.kv4_host_pipe_create.restype = i32
        lib.kv4_host_pipe_step.argtypes = [P, P, P, P, i64, P, i64, P, i64, i32, P, P, P, f32, P,
                                           P, P]
        lib.kv4_host_pipe_step.restype = i32
        lib.kv4_host_pipe_destroy.argtypes = [P]
        lib.kv4_host_pipe_destroy.restype = i32
        lib.kv4_set_wait_limit.argtypes = [i64, i32]
        lib.kv4_set_wait_limit.restype = i32
        lib.kv4_set_timing_event.argtypes = [P]
        lib.kv4_set_timing_event.restype = i32
        lib.kv4_status_str.argtypes = [i32]
        lib.kv4_status_str.restype = ctypes.c_char_p
        lib.kv4_version.argtypes = []
        lib.kv4_version.restype = i32
        _lib = lib
        return lib


def _check(fn: str, status: int):
    if status != 0:
        raise Kv4Error(fn, status)


def _dev(t: torch.Tensor, name: str, dtype: torch.dtype, contiguous: bool = True):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _err_ptr(dev_err):
    if dev_err is None:
        return None
    return _dev(dev_err, "dev_err", torch.int32)


def quantize_write(latent: torch.Tensor, rope: torch.Tensor, slot_mapping: torch.Tensor,
                   pool: torch.Tensor, dev_err: torch.Tensor | None = None) -> None:
    """Quantize latent bf16 [N,512] and rope bf16 [N,64] into pool uint8
    [num_slots,352] at slot_mapping int64 [N] (negative = skip)."""
    _quantize("kv4_quantize_write", latent, rope, slot_mapping, pool, dev_err)


def quantize_write_mse(latent: torch.Tensor, rope: torch.Tensor, slot_mapping: torch.Tensor,
                       pool: torch.Tensor, dev_err: torch.Tensor | None = None) -> None:
    """quantize_write with MSE-searched block scales (kv4_quantize_write_mse);
    the rows decode with sparse_mla_decode unchanged."""
    _quantize("kv4_quantize_write_mse", latent, rope, slot_mapping, pool, dev_err)


def quantize_write_fp8(latent: torch.Tensor, rope: torch.Tensor, slot_mapping: torch.Tensor,
                       pool: torch.Tensor, dev_err: torch.Tensor | None = None) -> None:
    """576-byte FP8 rows (E4M3 of every latent and rope value) into pool
    uint8 [num_slots,576] -- the row the NVFP4 row replaces, for comparison."""
    if pool.dim() != 2 or pool.shape[1] != ROW_BYTES_FP8:
        raise ValueError("pool must be [num_slots, 576]")
    _quantize("kv4_quantize_write_fp8", latent, rope, slot_mapping, pool, dev_err)


def _quantize(fn, latent, rope, slot_mapping, pool, dev_err):
    lib = load_library()
    n = slot_mapping.shape[0]
    if latent.dim() != 2 or rope.dim() != 2 or latent.shape[0] != n or rope.shape[0] != n:
        raise ValueError("latent [N,512], rope [N,64] and slot_mapping [N] must agree")
    if latent.stride(1) != 1 or rope.stride(1) != 1:
        raise ValueError("latent and rope rows must be contiguous")
    _check(fn, getattr(lib, fn)(
        _dev(latent, "latent", torch.bfloat16, False), latent.stride(0),
        _dev(rope, "rope", torch.bfloat16, False), rope.stride(0),
        _dev(slot_mapping, "slot_mapping", torch.int64), n,
        _dev(pool, "pool", torch.uint8), pool.shape[0], _err_ptr(dev_err),
        _stream(pool.device)))


def quantize_write_latent(latent: torch.Tensor, slot_mapping: torch.Tensor, pool: torch.Tensor,
                          dev_err: torch.Tensor | None = None) -> None:
    """Latent-only rows: quantize latent bf16 [N,512] into pool uint8
    [num_slots,288] at slot_mapping int64 [N] (negative = skip)."""
    lib = load_library()
    n = slot_mapping.shape[0]
    if latent.dim() != 2 or latent.shape[0] != n:
        raise ValueError("latent [N,512] and slot_mapping [N] must agree")
    if latent.stride(1) != 1:
        raise ValueError("latent rows must be contiguous")
    if pool.dim() != 2 or pool.shape[1] != ROW_BYTES_LATENT:
        raise ValueError("pool must be [num_slots, 288]")
    _check("kv4_quantize_write_latent", lib.kv4_quantize_write_latent(
        _dev(latent, "latent", torch.bfloat16, False), latent.stride(0),
        _dev(slot_mapping, "slot_mapping", torch.int64), n,
        _dev(pool, "pool", torch.uint8), pool.shape[0], _err_ptr(dev_err),
        _stream(pool.device)))


def _plan(fn: str, B: int, Sq: int, H: int, K: int, force_splits: int):
    s = ctypes.c_int(0)
    ws = ctypes.c_size_t(0)
    _check(fn, getattr(load_library(), fn)(B, Sq, H, K, force_splits, ctypes.byref(s),
                                           ctypes.byref(ws)))
    return s.value, ws.value


def decode_plan(B: int, Sq: int, H: int, K: int, force_splits: int = 0):
    """(splits, workspace_bytes) the decode will use on the current device."""
    return _plan("kv4_decode_plan", B, Sq, H, K, force_splits)


def decode_plan_fp8(B: int, Sq: int, H: int, K: int, force_splits: int = 0):
    """(splits, workspace_bytes) of sparse_mla_decode_fp8 on the current device."""
    return _plan("kv4_decode_plan_fp8", B, Sq, H, K, force_splits)


def decode_plan_latent(B: int, Sq: int, H: int, K: int, force_splits: int = 0):
    """(splits, workspace_bytes) of sparse_mla_decode_latent on the current device."""
    return _plan("kv4_decode_plan_latent", B, Sq, H, K, force_splits)


def _workspace(device, nbytes: int):
    if nbytes == 0:
        return None
    key = (str(device), torch.cuda.current_stream(device).cuda_stream)
    buf = _workspaces.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _workspaces[key] = buf
    return buf


def sparse_mla_decode(q: torch.Tensor, pool: torch.Tensor, page_table: torch.Tensor,
                      topk_idx: torch.Tensor, seq_lens: torch.Tensor, sm_scale: float,
                      out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, force_splits: int = 0,
                      dev_err: torch.Tensor | None = None):
    """Sparse MLA decode over the NVFP4 pool.

    q bf16 [B,Sq,H,576]; pool uint8 [num_slots,352]; page_table int32
    [B,pt_stride]; topk_idx int32 [B,Sq,K] (logical positions, -1 = pad);
    seq_lens int32 [B].  Returns (out bf16 [B,Sq,H,512], lse fp32 [B,Sq,H]).
    """
    return _decode("nvfp4", q, pool, page_table, topk_idx, seq_lens, sm_scale, out, lse, workspace,
                   force_splits, dev_err)


def sparse_mla_decode_latent(q: torch.Tensor, pool: torch.Tensor, page_table: torch.Tensor,
                             topk_idx: torch.Tensor, seq_lens: torch.Tensor, sm_scale: float,
                             out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                             workspace: torch.Tensor | None = None, force_splits: int = 0,
                             dev_err: torch.Tensor | None = None):
    """The same decode over latent-only rows: q bf16 [B,Sq,H,512], pool uint8
    [num_slots,288]; QK^T over the 512 latent columns."""
    return _decode("latent", q, pool, page_table, topk_idx, seq_lens, sm_scale, out, lse,
                   workspace, force_splits, dev_err)


def sparse_mla_decode_fp8(q: torch.Tensor, pool: torch.Tensor, page_table: torch.Tensor,
                          topk_idx: torch.Tensor, seq_lens: torch.Tensor, sm_scale: float,
                          out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                          workspace: torch.Tensor | None = None, force_splits: int = 0,
                          dev_err: torch.Tensor | None = None):
    """The decode over 576-byte FP8 rows (q bf16 [B,Sq,H,576]; pool uint8
    [num_slots,576]) -- the comparison path of the NVFP4 decode."""
    return _decode("fp8", q, pool, page_table, topk_idx, seq_lens, sm_scale, out, lse, workspace,
                   force_splits, dev_err)


def fp8_scratch(pool: torch.Tensor, page_table: torch.Tensor, topk_idx: torch.Tensor,
                seq_lens: torch.Tensor, scratch: torch.Tensor | None = None,
                dev_err: torch.Tensor | None = None) -> torch.Tensor:
    """The FP8 scratch copy of the NVFP4 rows the keys select: uint8
    [B*Sq*K, 576] (E4M3 of the dequantized values; masked keys give zero rows)."""
    lib = load_library()
    B, Sq, K = topk_idx.shape
    if scratch is None:
        scratch = torch.empty((B * Sq * K, ROW_BYTES_FP8), dtype=torch.uint8, device=pool.device)
    _check("kv4_fp8_scratch", lib.kv4_fp8_scratch(
        _dev(pool, "pool", torch.uint8), pool.shape[0],
        _dev(page_table, "page_table", torch.int32), page_table.shape[1], PAGE,
        _dev(topk_idx, "topk_idx", torch.int32), K, _dev(seq_lens, "seq_lens", torch.int32),
        B, Sq, _dev(scratch, "scratch", torch.uint8), _err_ptr(dev_err), _stream(pool.device)))
    return scratch


def scratch_index(topk_idx: torch.Tensor, seq_lens: torch.Tensor):
    """Indexing that makes a scratch copy (row (b*Sq + s)*K + k for key k of
    token s of request b) look like a paged pool: (page_table, topk, seq_lens)
    for a decode of B*Sq one-token requests whose K positions are 0..K-1,
    masked where the original key is masked (kv4_fp8_scratch_index).  K must
    be a multiple of 64."""
    lib = load_library()
    B, Sq, K = topk_idx.shape
    if K % PAGE:
        raise ValueError("the scratch path needs K to be a multiple of 64")
    dev = topk_idx.device
    n = B * Sq
    page_table = torch.empty((n, max(1, K // PAGE)), dtype=torch.int32, device=dev)
    topk = torch.empty((n, 1, K), dtype=torch.int32, device=dev)
    lens = torch.empty((n,), dtype=torch.int32, device=dev)
    _check("kv4_fp8_scratch_index", lib.kv4_fp8_scratch_index(
        _dev(topk_idx, "topk_idx", torch.int32), K, _dev(seq_lens, "seq_lens", torch.int32), B,
        Sq, _dev(page_table, "pt_out", torch.int32), _dev(topk, "topk_out", torch.int32),
        _dev(lens, "lens_out", torch.int32), _stream(dev)))
    return page_table, topk, lens


def sparse_mla_decode_partial(q: torch.Tensor, pool: torch.Tensor, page_table: torch.Tensor,
                              topk_idx: torch.Tensor, seq_lens: torch.Tensor, sm_scale: float,
                              out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                              workspace: torch.Tensor | None = None, force_splits: int = 0,
                              dev_err: torch.Tensor | None = None,
                              k_count: torch.Tensor | None = None):
    """sparse_mla_decode with an fp32 output: one context-parallel rank's
    normalized partial (o fp32 [B,Sq,H,512], lse fp32 [B,Sq,H]).  With
    k_count (int32 [B*Sq], e.g. from dcp_compact_topk) each query walks only
    the first k_count entries of its list (kv4_sparse_mla_decode_partial_counted)."""
    B, Sq, H, _ = q.shape
    if out is None:
        out = torch.empty((B, Sq, H, LATENT), dtype=torch.float32, device=q.device)
    if k_count is None:
        return _decode("nvfp4", q, pool, page_table, topk_idx, seq_lens, sm_scale, out, lse,
                       workspace, force_splits, dev_err, partial=True)
    lib = load_library()
    if q.shape[3] != QK_DIM or pool.dim() != 2 or pool.shape[1] != ROW_BYTES:
        raise ValueError(f"q must be [B, Sq, H, {QK_DIM}] and pool [num_slots, {ROW_BYTES}]")
    K = topk_idx.shape[2]
    if (tuple(topk_idx.shape[:2]) != (B, Sq) or seq_lens.shape[0] != B or
            page_table.shape[0] != B or k_count.numel() != B * Sq):
        raise ValueError("topk_idx [B,Sq,K], seq_lens [B], page_table [B,*] and k_count [B*Sq] "
                         "must agree with q")
    if lse is None:
        lse = torch.empty((B, Sq, H), dtype=torch.float32, device=q.device)
    splits, ws_bytes = decode_plan(B, Sq, H, K, force_splits)
    if workspace is None:
        workspace = _workspace(q.device, ws_bytes)
    ws_ptr = None if workspace is None else _dev(workspace, "workspace", workspace.dtype)
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    fn = "kv4_sparse_mla_decode_partial_counted"
    _check(fn, lib.kv4_sparse_mla_decode_partial_counted(
        _dev(q, "q", torch.bfloat16), _dev(pool, "pool", torch.uint8), pool.shape[0],
        _dev(page_table, "page_table", torch.int32), page_table.shape[1], PAGE,
        _dev(topk_idx, "topk_idx", torch.int32), K, _dev(k_count, "k_count", torch.int32),
        _dev(seq_lens, "seq_lens", torch.int32), B, Sq, H, float(sm_scale),
        _dev(out, "out", torch.float32), _dev(lse, "lse", torch.float32), ws_ptr, ws_len,
        force_splits, _err_ptr(dev_err), _stream(q.device)))
    return out, lse


def dcp_mask_topk(topk_idx: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                  world: int, rank: int) -> torch.Tensor:
    """The top-k list of context-parallel rank ``rank`` of ``world``: the
    positions whose physical page p has p % world == rank, -1 elsewhere."""
    lib = load_library()
    B, Sq, K = topk_idx.shape
    out = torch.empty_like(topk_idx)
    _check("kv4_dcp_mask_topk", lib.kv4_dcp_mask_topk(
        _dev(topk_idx, "topk_idx", torch.int32), _dev(page_table, "page_table", torch.int32),
        page_table.shape[1], _dev(seq_lens, "seq_lens", torch.int32), B, Sq, K, int(world),
        int(rank), _dev(out, "topk_out", torch.int32), _stream(topk_idx.device)))
    return out


def dcp_compact_topk(topk_idx: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                     world: int, rank: int):
    """The positions dcp_mask_topk keeps for rank ``rank``, moved to the front
    of each query's list in their order (-1 after them), and their number per
    query: (topk int32 [B,Sq,K], count int32 [B*Sq])."""
    lib = load_library()
    B, Sq, K = topk_idx.shape
    out = torch.empty_like(topk_idx)
    count = torch.empty(B * Sq, dtype=torch.int32, device=topk_idx.device)
    _check("kv4_dcp_compact_topk", lib.kv4_dcp_compact_topk(
        _dev(topk_idx, "topk_idx", torch.int32), _dev(page_table, "page_table", torch.int32),
        page_table.shape[1], _dev(seq_lens, "seq_lens", torch.int32), B, Sq, K, int(world),
        int(rank), _dev(out, "topk_out", torch.int32), _dev(count, "count_out", torch.int32),
        _stream(topk_idx.device)))
    return out, count


def dcp_local_page_table(page_table: torch.Tensor, world: int, rank: int) -> torch.Tensor:
    """Rank ``rank``'s page table over its own pool: p // world where the
    rank owns physical page p (p % world == rank), -1 elsewhere."""
    lib = load_library()
    B, stride = page_table.shape
    out = torch.empty_like(page_table)
    _check("kv4_dcp_local_page_table", lib.kv4_dcp_local_page_table(
        _dev(page_table, "page_table", torch.int32), stride, B, int(world), int(rank),
        _dev(out, "pt_local", torch.int32), _stream(page_table.device)))
    return out


def dcp_local_slots(slot_mapping: torch.Tensor, world: int, rank: int) -> torch.Tensor:
    """Cache-write slots in rank ``rank``'s own pool: (page // world) * 64 +
    slot % 64 for the tokens on the rank's pages, -1 (no write) elsewhere."""
    lib = load_library()
    out = torch.empty_like(slot_mapping)
    _check("kv4_dcp_local_slots", lib.kv4_dcp_local_slots(
        _dev(slot_mapping, "slot_mapping", torch.int64), slot_mapping.numel(), int(world),
        int(rank), _dev(out, "slots_out", torch.int64), _stream(slot_mapping.device)))
    return out


def dcp_local_pages(num_pages: int, world: int, rank: int) -> int:
    """Pages of rank ``rank``'s own pool when the cache has ``num_pages``
    physical pages: those p < num_pages with p % world == rank."""
    return max(0, (num_pages - rank + world - 1) // world)


def merge_partials(o_parts: torch.Tensor, lse_parts: torch.Tensor):
    """Log-sum-exp merge of R partials: o_parts fp32 [R, ..., 512], lse_parts
    fp32 [R, ...] -> (out bf16 [..., 512], lse fp32 [...])."""
    lib = load_library()
    R = o_parts.shape[0]
    shape = tuple(lse_parts.shape[1:])
    n_rows = lse_parts[0].numel()
    if tuple(o_parts.shape[1:-1]) != shape or o_parts.shape[-1] != LATENT:
        raise ValueError("o_parts must be [R, ..., 512] and lse_parts [R, ...]")
    out = torch.empty(shape + (LATENT,), dtype=torch.bfloat16, device=o_parts.device)
    lse = torch.empty(shape, dtype=torch.float32, device=o_parts.device)
    _check("kv4_merge_partials", lib.kv4_merge_partials(
        _dev(o_parts, "o_parts", torch.float32), _dev(lse_parts, "lse_parts", torch.float32), R,
        n_rows, _dev(out, "out", torch.bfloat16), _dev(lse, "lse", torch.float32),
        _stream(o_parts.device)))
    return out, lse


def gather_partials(o: torch.Tensor, lse: torch.Tensor, group=None):
    """All-gather of every rank's (o, lse) over ``group`` (torch.distributed):
    returns o_parts [world, *o.shape] and lse_parts [world, *lse.shape]."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    o_list = [torch.empty_like(o) for _ in range(world)]
    lse_list = [torch.empty_like(lse) for _ in range(world)]
    dist.all_gather(o_list, o.contiguous(), group=group)
    dist.all_gather(lse_list, lse.contiguous(), group=group)
    return torch.stack(o_list), torch.stack(lse_list)


def dcp_sparse_mla_decode(q, local_pool, page_table, topk_idx, seq_lens, sm_scale, group=None,
                          dev_err=None):
    """One decode step with the context split over the ranks of ``group``:
    each rank decodes the keys on its pages from its own pool (``local_pool``:
    the rank's pages only, written through dcp_local_slots) via its local page
    table, the ranks all-gather their fp32 (o, lse), and every rank merges
    them into the full result (out bf16 [B,Sq,H,512], lse fp32 [B,Sq,H]).
    ``page_table`` is the global (physical) one."""
    import torch.distributed as dist
    world, rank = dist.get_world_size(group), dist.get_rank(group)
    mine, count = dcp_compact_topk(topk_idx, page_table, seq_lens, world, rank)
    pt_local = dcp_local_page_table(page_table, world, rank)
    o, lse = sparse_mla_decode_partial(q, local_pool, pt_local, mine, seq_lens, sm_scale,
                                       dev_err=dev_err, k_count=count)
    o_parts, lse_parts = gather_partials(o, lse, group)
    return merge_partials(o_parts, lse_parts)


def _decode(fmt, q, pool, page_table, topk_idx, seq_lens, sm_scale, out, lse, workspace,
            force_splits, dev_err, partial=False):
    """fmt: "nvfp4" (352-byte rows), "latent" (288-byte rows) or "fp8" (576)."""
    lib = load_library()
    B, Sq, H, D = q.shape
    fp8, latent_only = fmt == "fp8", fmt == "latent"
    qk, row = ((LATENT, ROW_BYTES_LATENT) if latent_only else
               (QK_DIM, ROW_BYTES_FP8) if fp8 else (QK_DIM, ROW_BYTES))
    if D != qk:
        raise ValueError(f"q must be [B, Sq, H, {qk}]")
    if pool.dim() != 2 or pool.shape[1] != row:
        raise ValueError(f"pool must be [num_slots, {row}]")
    K = topk_idx.shape[2]
    if tuple(topk_idx.shape[:2]) != (B, Sq) or seq_lens.shape[0] != B or page_table.shape[0] != B:
        raise ValueError("topk_idx [B,Sq,K], seq_lens [B] and page_table [B,*] must agree with q")
    dev = q.device
    if out is None:
        out = torch.empty((B, Sq, H, LATENT), dtype=torch.bfloat16, device=dev)
    out_dtype = torch.float32 if partial else torch.bfloat16
    if lse is None:
        lse = torch.empty((B, Sq, H), dtype=torch.float32, device=dev)
    fn = ("kv4_sparse_mla_decode_latent" if latent_only else
          "kv4_sparse_mla_decode_fp8" if fp8 else
          "kv4_sparse_mla_decode_partial" if partial else "kv4_sparse_mla_decode")
    plan = decode_plan_latent if latent_only else decode_plan_fp8 if fp8 else decode_plan
    splits, ws_bytes = plan(B, Sq, H, K, force_splits)
    if workspace is None:
        workspace = _workspace(dev, ws_bytes)
    ws_ptr = None if workspace is None else _dev(workspace, "workspace", workspace.dtype)
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(fn, getattr(lib, fn)(
        _dev(q, "q", torch.bfloat16), _dev(pool, "pool", torch.uint8), pool.shape[0],
        _dev(page_table, "page_table", torch.int32), page_table.shape[1], PAGE,
        _dev(topk_idx, "topk_idx", torch.int32), K, _dev(seq_lens, "seq_lens", torch.int32),
        B, Sq, H, float(sm_scale), _dev(out, "out", out_dtype),
        _dev(lse, "lse", torch.float32), ws_ptr, ws_len, force_splits, _err_ptr(dev_err),
        _stream(dev)))
    return out, lse


def quantize_write_and_decode(latent: torch.Tensor, rope: torch.Tensor,
                              slot_mapping: torch.Tensor, pool: torch.Tensor, q: torch.Tensor,
                              page_table: torch.Tensor, topk_idx: torch.Tensor,
                              seq_lens: torch.Tensor, sm_scale: float,
                              out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                              workspace: torch.Tensor | None = None, force_splits: int = 0,
                              dev_err: torch.Tensor | None = None):
    """One decode step (kv4_quantize_write_and_decode): quantize_write of the
    step's new tokens, then sparse_mla_decode, with the same results; the
    decode's reads of q, page_table, topk_idx and seq_lens overlap the write."""
    lib = load_library()
    n = slot_mapping.shape[0]
    if latent.dim() != 2 or rope.dim() != 2 or latent.shape[0] != n or rope.shape[0] != n:
        raise ValueError("latent [N,512], rope [N,64] and slot_mapping [N] must agree")
    if latent.stride(1) != 1 or rope.stride(1) != 1:
        raise ValueError("latent and rope rows must be contiguous")
    B, Sq, H, D = q.shape
    if D != QK_DIM:
        raise ValueError(f"q must be [B, Sq, H, {QK_DIM}]")
    if pool.dim() != 2 or pool.shape[1] != ROW_BYTES:
        raise ValueError(f"pool must be [num_slots, {ROW_BYTES}]")
    K = topk_idx.shape[2]
    if tuple(topk_idx.shape[:2]) != (B, Sq) or seq_lens.shape[0] != B or page_table.shape[0] != B:
        raise ValueError("topk_idx [B,Sq,K], seq_lens [B] and page_table [B,*] must agree with q")
    dev = q.device
    if out is None:
        out = torch.empty((B, Sq, H, LATENT), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, Sq, H), dtype=torch.float32, device=dev)
    splits, ws_bytes = decode_plan(B, Sq, H, K, force_splits)
    if workspace is None:
        workspace = _workspace(dev, ws_bytes)
    ws_ptr = None if workspace is None else _dev(workspace, "workspace", workspace.dtype)
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    fn = "kv4_quantize_write_and_decode"
    _check(fn, lib.kv4_quantize_write_and_decode(
        _dev(latent, "latent", torch.bfloat16, False), latent.stride(0),
        _dev(rope, "rope", torch.bfloat16, False), rope.stride(0),
        _dev(slot_mapping, "slot_mapping", torch.int64), n,
        _dev(pool, "pool", torch.uint8), pool.shape[0],
        _dev(q, "q", torch.bfloat16),
        _dev(page_table, "page_table", torch.int32), page_table.shape[1], PAGE,
        _dev(topk_idx, "topk_idx", torch.int32), K, _dev(seq_lens, "seq_lens", torch.int32),
        B, Sq, H, float(sm_scale), _dev(out, "out", torch.bfloat16),
        _dev(lse, "lse", torch.float32), ws_ptr, ws_len, force_splits, _err_ptr(dev_err),
        _stream(dev)))
    return out, lse


def _host(t: torch.Tensor, name: str, dtype: torch.dtype):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


class HostPipe:
    """Decode steps fed from host memory (kv4_host_pipe_*): each step copies
    its inputs from host tensors into device staging on a copy-in stream, runs
    the write and the decode on the current stream, and copies out and lse
    back into host tensors on a copy-out stream; two steps are in flight.

    The staging memory (two areas and the split-K workspace) is allocated here
    with PyTorch on `device`.  Host tensors should be pinned.  A step's host
    inputs must stay unchanged, and its host outputs unread, until
    ``synchronize()`` (or a later ``synchronize`` of the copy-out stream)."""

    def __init__(self, B: int, Sq: int, H: int, K: int, max_new: int, device=None,
                 force_splits: int = 0):
        lib = load_library()
        self._lib = lib
        self.device = torch.device("cuda") if device is None else torch.device(device)
        self.shape = (B, Sq, H, K)
        self.max_new = max_new
        nbytes = ctypes.c_size_t(0)
        _check("kv4_host_pipe_bytes", lib.kv4_host_pipe_bytes(B, Sq, H, K, max_new, force_splits,
                                                              ctypes.byref(nbytes)))
        self._staging = torch.empty(max(nbytes.value, 256), dtype=torch.uint8, device=self.device)
        self.copy_in = torch.cuda.Stream(self.device)
        self.copy_out = torch.cuda.Stream(self.device)
        self.compute = torch.cuda.current_stream(self.device)
        handle = ctypes.c_void_p(None)
        _check("kv4_host_pipe_create", lib.kv4_host_pipe_create(
            B, Sq, H, K, max_new, force_splits, ctypes.c_void_p(self._staging.data_ptr()),
            self._staging.numel(), ctypes.c_void_p(self.copy_in.cuda_stream),
            ctypes.c_void_p(self.compute.cuda_stream),
            ctypes.c_void_p(self.copy_out.cuda_stream), ctypes.byref(handle)))
        self._handle = handle

    def step(self, latent: torch.Tensor, rope: torch.Tensor, slot_mapping: torch.Tensor,
             pool: torch.Tensor, q: torch.Tensor, page_table: torch.Tensor,
             topk_idx: torch.Tensor, seq_lens: torch.Tensor, sm_scale: float,
             out: torch.Tensor, lse: torch.Tensor, dev_err: torch.Tensor | None = None) -> None:
        """Enqueue one step.  Host tensors: latent bf16 [N, 512], rope bf16
        [N, 64], slot_mapping int64 [N], q bf16 [B, Sq, H, 576], topk_idx int32
        [B, Sq, K], seq_lens int32 [B], out bf16 [B, Sq, H, 512], lse fp32
        [B, Sq, H].  Device tensors: pool, page_table (and dev_err)."""
        if self._handle is None:
            raise RuntimeError("HostPipe is closed")
        B, Sq, H, K = self.shape
        n = slot_mapping.shape[0]
        if (tuple(q.shape) != (B, Sq, H, QK_DIM) or tuple(topk_idx.shape) != (B, Sq, K) or
                tuple(seq_lens.shape) != (B,) or tuple(out.shape) != (B, Sq, H, LATENT) or
                tuple(lse.shape) != (B, Sq, H) or tuple(latent.shape) != (n, LATENT) or
                tuple(rope.shape) != (n, ROPE)):
            raise ValueError("host tensors must match the pipe's shape")
        if pool.dim() != 2 or pool.shape[1] != ROW_BYTES or page_table.shape[0] != B:
            raise ValueError(f"pool must be [num_slots, {ROW_BYTES}] and page_table [B, *]")
        _check("kv4_host_pipe_step", self._lib.kv4_host_pipe_step(
            self._handle, _host(latent, "latent", torch.bfloat16),
            _host(rope, "rope", torch.bfloat16), _host(slot_mapping, "slot_mapping", torch.int64),
            n, _dev(pool, "pool", torch.uint8), pool.shape[0],
            _dev(page_table, "page_table", torch.int32), page_table.shape[1], PAGE,
            _host(q, "q", torch.bfloat16), _host(topk_idx, "topk_idx", torch.int32),
            _host(seq_lens, "seq_lens", torch.int32), float(sm_scale),
            _host(out, "out", torch.bfloat16), _host(lse, "lse", torch.float32),
            _err_ptr(dev_err)))

    def synchronize(self) -> None:
        """Wait until every enqueued step's results are in host memory."""
        self.copy_out.synchronize()
        self.compute.synchronize()

    def close(self) -> None:
        """Wait for the enqueued steps, then release the pipe (its staging
        memory returns to PyTorch only after that)."""
        if self._handle is not None:
            self.synchronize()
            self.copy_in.synchronize()
            _check("kv4_host_pipe_destroy", self._lib.kv4_host_pipe_destroy(self._handle))
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def debug_gather_dequant(pool: torch.Tensor, page_table: torch.Tensor, topk_idx: torch.Tensor,
                         seq_lens: torch.Tensor, dev_err: torch.Tensor | None = None):
    """The decode's gather + dequantization: f16 [B,Sq,K,576] (masked rows 0)."""
    return _gather(False, pool, page_table, topk_idx, seq_lens, dev_err)


def debug_gather_dequant_latent(pool: torch.Tensor, page_table: torch.Tensor,
                                topk_idx: torch.Tensor, seq_lens: torch.Tensor,
                                dev_err: torch.Tensor | None = None):
    """The same over latent-only rows: f16 [B,Sq,K,512] (masked rows 0)."""
    return _gather(True, pool, page_table, topk_idx, seq_lens, dev_err)


def _gather(latent_only, pool, page_table, topk_idx, seq_lens, dev_err):
    lib = load_library()
    B, Sq, K = topk_idx.shape
    fn = "kv4_debug_gather_dequant_latent" if latent_only else "kv4_debug_gather_dequant"
    rows = torch.empty((B, Sq, K, LATENT if latent_only else QK_DIM), dtype=torch.float16,
                       device=pool.device)
    _check(fn, getattr(lib, fn)(
        _dev(pool, "pool", torch.uint8), pool.shape[0],
        _dev(page_table, "page_table", torch.int32), page_table.shape[1], PAGE,
        _dev(topk_idx, "topk_idx", torch.int32), K, _dev(seq_lens, "seq_lens", torch.int32),
        B, Sq, _dev(rows, "rows", torch.float16), _err_ptr(dev_err), _stream(pool.device)))
    return rows


def set_timing_event(event: "torch.cuda.Event | None") -> None:
    """Measurement hook: record ``event`` between the decode and merge kernels
    of every later sparse_mla_decode call (None turns it off)."""
    handle = None if event is None else ctypes.c_void_p(event.cuda_event)
    _check("kv4_set_timing_event", load_library().kv4_set_timing_event(handle))


def set_wait_limit(timeout_ns: int = 0, fault_site: int = 0) -> None:
    """Test hook: bounded-wait limit for the next launches and an optional
    injected wait on a barrier nothing arrives on (fault_site=1)."""
    _check("kv4_set_wait_limit", load_library().kv4_set_wait_limit(int(timeout_ns),
                                                                   int(fault_site)))
