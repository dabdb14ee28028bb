"""Thin Python binding of libnvfp4kv.so (argument marshalling only).

Every function mirrors one C-ABI entry point of include/nvfp4kv.h and takes
torch tensors that already live on the current CUDA device; the work runs in
the library's kernels.  There is no fallback: if the compiled library is
missing the import of this module raises.  PyTorch provides device memory and
the current stream, nothing else.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

NVFP4KV_OK = 0
NVFP4KV_ERR_ARG = -1
NVFP4KV_ERR_SHAPE = -2
NVFP4KV_ERR_WORKSPACE = -3
NVFP4KV_ERR_CUDA = -4
NVFP4KV_ERR_TIMEOUT = -5
NVFP4KV_ERR_DEVICE_INDEX = -6
NVFP4KV_ERR_UNSUPPORTED = -7
ERR_NAMES = {-1: "ERR_ARG", -2: "ERR_SHAPE", -3: "ERR_WORKSPACE", -4: "ERR_CUDA", -5: "ERR_TIMEOUT",
             -6: "ERR_DEVICE_INDEX", -7: "ERR_UNSUPPORTED"}
VARIANT_A4Q = 0
VARIANT_DQ_AHEAD = 1
VARIANT_A4Q_FP4PV = 2
QUANT_GLOBAL = 0
QUANT_PER_ROW = 1
OP_PREFILL = 0
OP_DECODE = 1
HEAD_DIM = 128
PAGE_SIZE = 16

EXPORTED = ["nvfp4_kv_append", "nvfp4_paged_prefill", "nvfp4_paged_decode", "nvfp4_workspace_bytes",
            "nvfp4_cache_bytes", "nvfp4_quantize_rows", "nvfp4_dequantize_rows", "nvfp4kv_get_device_status",
            "nvfp4kv_status_string", "nvfp4kv_version", "nvfp4kv_debug_wait_timeout",
            "nvfp4_paged_prefill_noalloc", "nvfp4_paged_prefill_noalloc_max_bytes",
            "nvfp4_paged_prefill_plan", "nvfp4_paged_prefill_run", "nvfp4_v_token_major",
            "fp8_kv_append", "fp8_paged_prefill", "fp8_paged_decode", "fp8_workspace_bytes", "fp8_cache_bytes"]


class CacheDesc(ctypes.Structure):
    _fields_ = [("k_data", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("v_data", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("k_global_scale", ctypes.c_float), ("v_global_scale", ctypes.c_float)]


class Fp8CacheDesc(ctypes.Structure):
    _fields_ = [("k_data", ctypes.c_void_p), ("v_data", ctypes.c_void_p), ("num_pages", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


class NvFp4Error(RuntimeError):
    def __init__(self, where: str, code: int):
        super().__init__(f"{where}: {ERR_NAMES.get(code, code)} ({status_string(code)})")
        self.code = code


def _load() -> ctypes.CDLL:
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"libnvfp4kv.so has not been built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    D = ctypes.POINTER(CacheDesc)
    lib.nvfp4_kv_append.argtypes = [P, P, P, i64, D, P]
    lib.nvfp4_paged_prefill.argtypes = [P, i64, i32, D, P, i32, P, P, i32, i32, f32, i32, f32, P, P, P, sz, P]
    lib.nvfp4_paged_decode.argtypes = [P, i32, D, P, i32, P, i32, f32, P, P, P, sz, P]
    lib.nvfp4_paged_prefill_plan.argtypes = [i64, i32, D, P, i32, P, P, i32, i32, i32, P, sz, P]
    lib.nvfp4_paged_prefill_run.argtypes = [P, i64, i32, D, P, i32, P, P, i32, i32, f32, i32, f32, P, P, P, sz, P]
    lib.nvfp4_paged_prefill_noalloc.argtypes = [P, i64, i32, D, P, i32, P, P, i32, i32, f32, i32, f32, P, P, P]
    lib.nvfp4_paged_prefill_noalloc_max_bytes.argtypes = []
    lib.nvfp4_paged_prefill_noalloc_max_bytes.restype = sz
    lib.nvfp4_workspace_bytes.argtypes = [i32, i32, i32, i32, i64, i32]
    lib.nvfp4_workspace_bytes.restype = sz
    lib.nvfp4_cache_bytes.argtypes = [i32, i32, i32, i32]
    lib.nvfp4_cache_bytes.restype = sz
    lib.nvfp4_quantize_rows.argtypes = [P, i64, i32, f32, P, P, P, P]
    lib.nvfp4_dequantize_rows.argtypes = [P, P, i64, P, f32, P, P]
    lib.nvfp4_v_token_major.argtypes = [D, P, i32, P, P, P]
    lib.nvfp4kv_get_device_status.argtypes = [P]
    lib.nvfp4kv_status_string.argtypes = [ctypes.c_int]
    lib.nvfp4kv_status_string.restype = ctypes.c_char_p
    lib.nvfp4kv_version.restype = ctypes.c_char_p
    F = ctypes.POINTER(Fp8CacheDesc)
    lib.fp8_kv_append.argtypes = [P, P, P, i64, F, P]
    lib.fp8_paged_prefill.argtypes = [P, i64, i32, F, P, i32, P, P, i32, i32, f32, P, P, P, sz, P]
    lib.fp8_paged_decode.argtypes = [P, i32, F, P, i32, P, i32, f32, P, P, P, sz, P]
    lib.fp8_workspace_bytes.argtypes = [i32, i32, i32, i32, i64, i32]
    lib.fp8_workspace_bytes.restype = sz
    lib.fp8_cache_bytes.argtypes = [i32, i32, i32, i32]
    lib.fp8_cache_bytes.restype = sz
    lib.nvfp4kv_debug_wait_timeout.argtypes = [ctypes.c_uint32, P]
    lib.nvfp4kv_debug_wait_timeout.restype = ctypes.c_int
    for name in ("nvfp4_kv_append", "nvfp4_paged_prefill", "nvfp4_paged_prefill_noalloc", "nvfp4_paged_decode",
                 "nvfp4_paged_prefill_plan", "nvfp4_paged_prefill_run", "nvfp4_v_token_major",
                 "nvfp4_quantize_rows",
                 "nvfp4_dequantize_rows", "nvfp4kv_get_device_status", "fp8_kv_append", "fp8_paged_prefill",
                 "fp8_paged_decode"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


lib = _load()


def status_string(code: int) -> str:
    return lib.nvfp4kv_status_string(int(code)).decode()


def _check(where: str, rc: int) -> None:
    if rc != NVFP4KV_OK:
        raise NvFp4Error(where, rc)


def _ptr(t: Optional[torch.Tensor]):
    """Device pointer of a contiguous CUDA tensor.  Every pointer of the ABI
    except the cache descriptor is a device pointer, so a host tensor is
    refused here rather than handed to a kernel."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to nvfp4kv must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors passed to nvfp4kv must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _require(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _check_dtype(t: Optional[torch.Tensor], dtype, name: str) -> None:
    if t is not None:
        _require(t.dtype == dtype, f"{name} must be {dtype}, got {t.dtype}")


def _check_rows(q: torch.Tensor, name: str = "q") -> None:
    _check_dtype(q, torch.bfloat16, name)
    _require(q.dim() == 3 and q.shape[2] == HEAD_DIM, f"{name} must be [tokens][heads][{HEAD_DIM}]")


def _check_tables(page_table: torch.Tensor, kv_lens: torch.Tensor, qo_indptr: Optional[torch.Tensor]) -> int:
    """Dtypes and shapes of the request metadata; returns the batch size."""
    _check_dtype(page_table, torch.int32, "page_table")
    _check_dtype(kv_lens, torch.int32, "kv_lens")
    _require(kv_lens.dim() == 1, "kv_lens must be [batch]")
    batch = kv_lens.shape[0]
    _require(page_table.dim() == 2 and page_table.shape[0] == batch, "page_table must be [batch][max_pages]")
    if qo_indptr is not None:
        _check_dtype(qo_indptr, torch.int32, "qo_indptr")
        _require(qo_indptr.dim() == 1 and qo_indptr.shape[0] == batch + 1, "qo_indptr must be [batch + 1]")
    return batch


def _check_out(out: Optional[torch.Tensor], lse: Optional[torch.Tensor], rows: int, heads: int) -> None:
    if out is not None:
        _check_rows(out, "out")
        _require(tuple(out.shape) == (rows, heads, HEAD_DIM), "out must have the shape of q")
    if lse is not None:
        _check_dtype(lse, torch.float32, "lse")
        _require(tuple(lse.shape) == (rows, heads), "lse must be [tokens][heads]")


def _device(*tensors) -> torch.device:
    """The one CUDA device every given tensor lives on.  The library launches
    on the current device with pointers that must belong to it, so a host
    tensor or tensors spread over several devices are refused here."""
    dev = None
    for t in tensors:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensors passed to nvfp4kv must live on a CUDA device")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"tensors passed to nvfp4kv must share one device ({dev} and {t.device})")
    if dev is None:
        raise ValueError("tensors passed to nvfp4kv must live on a CUDA device")
    return dev


def _stream(stream, dev: torch.device) -> ctypes.c_void_p:
    """The caller's stream (or the current stream of `dev`); it must belong to
    the device the tensors live on."""
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    if s.device != dev:
        raise ValueError(f"stream is on {s.device} but the tensors are on {dev}")
    return ctypes.c_void_p(s.cuda_stream)


class Cache:
    """One layer's NVFP4 cache: four caller-owned device pools (uint8 tensors)
    in the documented layout, plus the two per-tensor scales."""

    def __init__(self, num_pages: int, num_kv_heads: int, k_global_scale: float, v_global_scale: float,
                 device=None, fill: Optional[int] = 0):
        dev = device or torch.device("cuda")
        shp_d = (num_pages, num_kv_heads, PAGE_SIZE, HEAD_DIM // 2)
        shp_s = (num_pages, num_kv_heads, PAGE_SIZE, HEAD_DIM // 16)
        mk = (lambda s: torch.zeros(s, dtype=torch.uint8, device=dev)) if fill == 0 else \
            (lambda s: torch.full(s, int(fill), dtype=torch.uint8, device=dev))
        self.k_data, self.k_scale = mk(shp_d), mk(shp_s)
        self.v_data, self.v_scale = mk(shp_d), mk(shp_s)
        self.num_pages, self.num_kv_heads = num_pages, num_kv_heads
        self.k_global_scale, self.v_global_scale = float(k_global_scale), float(v_global_scale)

    def pools(self):
        return (self.k_data, self.k_scale, self.v_data, self.v_scale)

    def desc(self) -> CacheDesc:
        """Host descriptor of the four pools.  The pools are device memory that
        the kernels read and write, so a host-memory cache is refused."""
        for t in self.pools():
            if not t.is_cuda:
                raise ValueError("cache pools must live on a CUDA device")
            if not t.is_contiguous() or t.dtype != torch.uint8:
                raise ValueError("cache pools must be contiguous uint8 tensors")
        return CacheDesc(self.k_data.data_ptr(), self.k_scale.data_ptr(), self.v_data.data_ptr(),
                         self.v_scale.data_ptr(), self.num_pages, PAGE_SIZE, self.num_kv_heads, HEAD_DIM,
                         self.k_global_scale, self.v_global_scale)


class Fp8Cache:
    """One layer's FP8 (E4M3) comparison cache: two caller-owned device pools
    [pages][kv heads][16][128] of codes, plus the two per-tensor scales."""

    def __init__(self, num_pages: int, num_kv_heads: int, k_scale: float, v_scale: float, device=None,
                 fill: Optional[int] = 0):
        dev = device or torch.device("cuda")
        shp = (num_pages, num_kv_heads, PAGE_SIZE, HEAD_DIM)
        self.k_data = torch.full(shp, int(fill or 0), dtype=torch.uint8, device=dev)
        self.v_data = torch.full(shp, int(fill or 0), dtype=torch.uint8, device=dev)
        self.num_pages, self.num_kv_heads = num_pages, num_kv_heads
        self.k_scale, self.v_scale = float(k_scale), float(v_scale)

    def pools(self):
        return (self.k_data, self.v_data)

    def desc(self) -> Fp8CacheDesc:
        """Host descriptor of the two pools (which must be device memory)."""
        for t in self.pools():
            if not t.is_cuda:
                raise ValueError("cache pools must live on a CUDA device")
            if not t.is_contiguous() or t.dtype != torch.uint8:
                raise ValueError("cache pools must be contiguous uint8 tensors")
        return Fp8CacheDesc(self.k_data.data_ptr(), self.v_data.data_ptr(), self.num_pages, PAGE_SIZE,
                            self.num_kv_heads, HEAD_DIM, self.k_scale, self.v_scale)


def fp8_cache_bytes(num_pages: int, page_size: int, num_kv_heads: int, head_dim: int) -> int:
    return int(lib.fp8_cache_bytes(num_pages, page_size, num_kv_heads, head_dim))


def fp8_workspace_bytes(op: int, batch: int, num_q_heads: int, num_kv_heads: int, total_q: int = 0,
                        max_kv_len: int = 0) -> int:
    return int(lib.fp8_workspace_bytes(op, batch, num_q_heads, num_kv_heads, total_q, max_kv_len))


def fp8_kv_append(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, cache: Fp8Cache, stream=None) -> None:
    _check_rows(k, "k")
    _check_rows(v, "v")
    _require(k.shape == v.shape and k.shape[1] == cache.num_kv_heads, "k and v must be [tokens][kv heads][128]")
    _check_dtype(slot_mapping, torch.int64, "slot_mapping")
    _require(slot_mapping.dim() == 1 and slot_mapping.shape[0] == k.shape[0], "slot_mapping must be [tokens]")
    d = cache.desc()  # a host-memory cache is refused before the other tensors
    dev = _device(*cache.pools(), k, v, slot_mapping)
    with torch.cuda.device(dev):
        _check("fp8_kv_append", lib.fp8_kv_append(_ptr(k), _ptr(v), _ptr(slot_mapping), k.shape[0], ctypes.byref(d),
                                                  _stream(stream, dev)))


def fp8_paged_prefill(q: torch.Tensor, cache: Fp8Cache, page_table: torch.Tensor, kv_lens: torch.Tensor,
                      qo_indptr: torch.Tensor, causal: bool = True, sm_scale: Optional[float] = None,
                      out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Paged prefill over the FP8 cache (BF16 query; K/V converted once per
    KV tile, BF16 QK and FP16 PV on the tensor cores)."""
    _check_rows(q)
    batch = _check_tables(page_table, kv_lens, qo_indptr)
    total_q, hq, _ = q.shape
    _check_out(out, lse, total_q, hq)
    d = cache.desc()  # a host-memory cache is refused before the other tensors
    dev = _device(*cache.pools(), q, page_table, kv_lens, qo_indptr, out, lse, workspace)
    if out is None:
        out = torch.empty_like(q)
    if sm_scale is None:
        sm_scale = HEAD_DIM ** -0.5
    if workspace is None:
        need = fp8_workspace_bytes(OP_PREFILL, batch, hq, cache.num_kv_heads, total_q, page_table.shape[1] * PAGE_SIZE)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _check("fp8_paged_prefill", lib.fp8_paged_prefill(
            _ptr(q), total_q, hq, ctypes.byref(d), _ptr(page_table), page_table.shape[1], _ptr(kv_lens),
            _ptr(qo_indptr), batch, int(bool(causal)), float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream, dev)))
    return out


def fp8_paged_decode(q: torch.Tensor, cache: Fp8Cache, page_table: torch.Tensor, kv_lens: torch.Tensor,
                     sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                     lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
    _check_rows(q)
    batch = _check_tables(page_table, kv_lens, None)
    _require(q.shape[0] == batch, "q must be [batch][heads][128] (one query token per request)")
    _, hq, _ = q.shape
    _check_out(out, lse, batch, hq)
    d = cache.desc()  # a host-memory cache is refused before the other tensors
    dev = _device(*cache.pools(), q, page_table, kv_lens, out, lse, workspace)
    if out is None:
        out = torch.empty_like(q)
    if sm_scale is None:
        sm_scale = HEAD_DIM ** -0.5
    need = fp8_workspace_bytes(OP_DECODE, batch, hq, cache.num_kv_heads, 0, page_table.shape[1] * PAGE_SIZE)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _check("fp8_paged_decode", lib.fp8_paged_decode(
            _ptr(q), hq, ctypes.byref(d), _ptr(page_table), page_table.shape[1], _ptr(kv_lens), batch,
            float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream(stream, dev)))
    return out


def nvfp4_cache_bytes(num_pages: int, page_size: int, num_kv_heads: int, head_dim: int) -> int:
    return int(lib.nvfp4_cache_bytes(num_pages, page_size, num_kv_heads, head_dim))


def nvfp4_workspace_bytes(op: int, batch: int, num_q_heads: int, num_kv_heads: int, total_q: int = 0,
                          max_kv_len: int = 0) -> int:
    return int(lib.nvfp4_workspace_bytes(op, batch, num_q_heads, num_kv_heads, total_q, max_kv_len))


def nvfp4_kv_append(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, cache: Cache, stream=None) -> None:
    _check_rows(k, "k")
    _check_rows(v, "v")
    _require(k.shape == v.shape and k.shape[1] == cache.num_kv_heads, "k and v must be [tokens][kv heads][128]")
    _check_dtype(slot_mapping, torch.int64, "slot_mapping")
    _require(slot_mapping.dim() == 1 and slot_mapping.shape[0] == k.shape[0], "slot_mapping must be [tokens]")
    d = cache.desc()  # a host-memory cache is refused before the other tensors
    dev = _device(*cache.pools(), k, v, slot_mapping)
    with torch.cuda.device(dev):
        _check("nvfp4_kv_append", lib.nvfp4_kv_append(_ptr(k), _ptr(v), _ptr(slot_mapping), k.shape[0],
                                                      ctypes.byref(d), _stream(stream, dev)))


def nvfp4_paged_prefill(q: torch.Tensor, cache: Cache, page_table: torch.Tensor, kv_lens: torch.Tensor,
                        qo_indptr: torch.Tensor, causal: bool = True, sm_scale: Optional[float] = None,
                        variant: int = VARIANT_A4Q, out: Optional[torch.Tensor] = None,
                        lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                        stream=None, q_global_scale: float = 0.0) -> torch.Tensor:
    """A4Q (or dequant-ahead) paged prefill.  q_global_scale selects the A4Q
    query scale scheme: 0 = per (token, head) row, amax/2688; > 0 = that one
    scale for every row (per-tensor, or 1 for single level)."""
    _check_rows(q)
    batch = _check_tables(page_table, kv_lens, qo_indptr)
    total_q, hq, _ = q.shape
    _check_out(out, lse, total_q, hq)
    d = cache.desc()  # a host-memory cache is refused before the other tensors
    dev = _device(*cache.pools(), q, page_table, kv_lens, qo_indptr, out, lse, workspace)
    if out is None:
        out = torch.empty_like(q)
    if sm_scale is None:
        sm_scale = HEAD_DIM ** -0.5
    if workspace is None:
        need = nvfp4_workspace_bytes(OP_PREFILL, batch, hq, cache.num_kv_heads, total_q,
                                     page_table.shape[1] * PAGE_SIZE)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _check("nvfp4_paged_prefill", lib.nvfp4_paged_prefill(
            _ptr(q), total_q, hq, ctypes.byref(d), _ptr(page_table), page_table.shape[1], _ptr(kv_lens),
            _ptr(qo_indptr), batch, int(bool(causal)), float(sm_scale), int(variant), float(q_global_scale),
            _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream(stream, dev)))
    return out


def nvfp4_paged_prefill_plan(cache: Cache, total_q: int, num_q_heads: int, page_table: torch.Tensor,
                             kv_lens: torch.Tensor, qo_indptr: torch.Tensor, workspace: torch.Tensor,
                             causal: bool = True, variant: int = VARIANT_A4Q, stream=None) -> None:
    """Schedule (and, in repack mode, the repacked tile records) into the workspace."""
    _check_tables(page_table, kv_lens, qo_indptr)
    _check_dtype(workspace, torch.uint8, "workspace")
    d = cache.desc()  # a host-memory cache is refused before the other tensors
    dev = _device(*cache.pools(), page_table, kv_lens, qo_indptr, workspace)
    with torch.cuda.device(dev):
        _check("nvfp4_paged_prefill_plan", lib.nvfp4_paged_prefill_plan(
            total_q, num_q_heads, ctypes.byref(d), _ptr(page_table), page_table.shape[1], _ptr(kv_lens),
            _ptr(qo_indptr), kv_lens.shape[0], int(bool(causal)), int(variant), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream, dev)))


def nvfp4_paged_prefill_run(q: torch.Tensor, cache: Cache, page_table: torch.Tensor, kv_lens: torch.Tensor,
                            qo_indptr: torch.Tensor, workspace: torch.Tensor, causal: bool = True,
                            sm_scale: Optional[float] = None, variant: int = VARIANT_A4Q,
                            out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                            stream=None, q_global_scale: float = 0.0) -> torch.Tensor:
    """The attention kernel alone, reading the schedule a matching plan call wrote."""
    _check_rows(q)
    _check_tables(page_table, kv_lens, qo_indptr)
    _check_dtype(workspace, torch.uint8, "workspace")
    total_q, hq, _ = q.shape
    _check_out(out, lse, total_q, hq)
    d = cache.desc()  # a host-memory cache is refused before the other tensors
    dev = _device(*cache.pools(), q, page_table, kv_lens, qo_indptr, workspace, out, lse)
    if out is None:
        out = torch.empty_like(q)
    if sm_scale is None:
        sm_scale = HEAD_DIM ** -0.5
    with torch.cuda.device(dev):
        _check("nvfp4_paged_prefill_run", lib.nvfp4_paged_prefill_run(
            _ptr(q), total_q, hq, ctypes.byref(d), _ptr(page_table), page_table.shape[1], _ptr(kv_lens),
            _ptr(qo_indptr), kv_lens.shape[0], int(bool(causal)), float(sm_scale), int(variant),
            float(q_global_scale), _ptr(out), _ptr(lse), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream, dev)))
    return out


def nvfp4_paged_prefill_noalloc_max_bytes() -> int:
    return int(lib.nvfp4_paged_prefill_noalloc_max_bytes())


def nvfp4_paged_prefill_noalloc(q: torch.Tensor, cache: Cache, page_table: torch.Tensor, kv_lens: torch.Tensor,
                                qo_indptr: torch.Tensor, causal: bool = True, sm_scale: Optional[float] = None,
                                variant: int = VARIANT_A4Q, out: Optional[torch.Tensor] = None,
                                lse: Optional[torch.Tensor] = None, stream=None,
                                q_global_scale: float = 0.0) -> torch.Tensor:
    """Same as nvfp4_paged_prefill but with the work schedule in the
    library's static device array: for callers that cannot allocate device
    memory at call time.  Always runs in-kernel mode.  Calls that overlap on
    the GPU race on that array."""
    _check_rows(q)
    _check_tables(page_table, kv_lens, qo_indptr)
    total_q, hq, _ = q.shape
    _check_out(out, lse, total_q, hq)
    d = cache.desc()  # a host-memory cache is refused before the other tensors
    dev = _device(*cache.pools(), q, page_table, kv_lens, qo_indptr, out, lse)
    if out is None:
        out = torch.empty_like(q)
    if sm_scale is None:
        sm_scale = HEAD_DIM ** -0.5
    with torch.cuda.device(dev):
        _check("nvfp4_paged_prefill_noalloc", lib.nvfp4_paged_prefill_noalloc(
            _ptr(q), total_q, hq, ctypes.byref(d), _ptr(page_table), page_table.shape[1], _ptr(kv_lens),
            _ptr(qo_indptr), kv_lens.shape[0], int(bool(causal)), float(sm_scale), int(variant),
            float(q_global_scale), _ptr(out), _ptr(lse), _stream(stream, dev)))
    return out


def nvfp4_paged_decode(q: torch.Tensor, cache: Cache, page_table: torch.Tensor, kv_lens: torch.Tensor,
                       sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                       lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
    _check_rows(q)
    batch = _check_tables(page_table, kv_lens, None)
    _require(q.shape[0] == batch, "q must be [batch][heads][128] (one query token per request)")
    _, hq, _ = q.shape
    _check_out(out, lse, batch, hq)
    d = cache.desc()  # a host-memory cache is refused before the other tensors
    dev = _device(*cache.pools(), q, page_table, kv_lens, out, lse, workspace)
    if out is None:
        out = torch.empty_like(q)
    if sm_scale is None:
        sm_scale = HEAD_DIM ** -0.5
    need = nvfp4_workspace_bytes(OP_DECODE, batch, hq, cache.num_kv_heads, 0, page_table.shape[1] * PAGE_SIZE)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _check("nvfp4_paged_decode", lib.nvfp4_paged_decode(
            _ptr(q), hq, ctypes.byref(d), _ptr(page_table), page_table.shape[1], _ptr(kv_lens), batch,
            float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream(stream, dev)))
    return out


def nvfp4_quantize_rows(x: torch.Tensor, mode: int = QUANT_GLOBAL, global_scale: float = 1.0, stream=None):
    _check_dtype(x, torch.bfloat16, "x")
    _require(x.shape[-1] == HEAD_DIM, f"x must be [...][{HEAD_DIM}]")
    dev = _device(x)
    rows = x.numel() // HEAD_DIM
    packed = torch.empty(rows, HEAD_DIM // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(rows, HEAD_DIM // 16, dtype=torch.uint8, device=dev)
    row_scales = torch.empty(rows, dtype=torch.float32, device=dev) if mode == QUANT_PER_ROW else None
    with torch.cuda.device(dev):
        _check("nvfp4_quantize_rows", lib.nvfp4_quantize_rows(_ptr(x), rows, mode, float(global_scale),
                                                              _ptr(packed), _ptr(scales), _ptr(row_scales),
                                                              _stream(stream, dev)))
    return packed, scales, row_scales


def nvfp4_dequantize_rows(packed: torch.Tensor, scales: torch.Tensor, row_scales: Optional[torch.Tensor] = None,
                          global_scale: float = 1.0, stream=None) -> torch.Tensor:
    _check_dtype(packed, torch.uint8, "packed")
    _check_dtype(scales, torch.uint8, "scales")
    _check_dtype(row_scales, torch.float32, "row_scales")
    rows = packed.shape[0]
    _require(tuple(packed.shape) == (rows, HEAD_DIM // 2) and tuple(scales.shape) == (rows, HEAD_DIM // 16),
             "packed must be [rows][64] and scales [rows][8]")
    _require(row_scales is None or tuple(row_scales.shape) == (rows,), "row_scales must be [rows]")
    dev = _device(packed, scales, row_scales)
    out = torch.empty(rows, HEAD_DIM, dtype=torch.bfloat16, device=dev)
    with torch.cuda.device(dev):
        _check("nvfp4_dequantize_rows", lib.nvfp4_dequantize_rows(_ptr(packed), _ptr(scales), rows,
                                                                  _ptr(row_scales), float(global_scale), _ptr(out),
                                                                  _stream(stream, dev)))
    return out


def nvfp4_v_token_major(cache: Cache, page_ids: torch.Tensor, stream=None):
    """The token-major V blocks of the listed pages (the re-layout the FP4 PV
    prefill variant reads): codes uint8 [n][kv heads][128][8] and scales uint8
    [n][kv heads][128]."""
    _check_dtype(page_ids, torch.int32, "page_ids")
    _require(page_ids.dim() == 1 and page_ids.is_contiguous(), "page_ids must be a contiguous [n] tensor")
    d = cache.desc()  # a host-memory cache is refused before the other tensors
    dev = _device(*cache.pools(), page_ids)
    n, h = page_ids.shape[0], cache.num_kv_heads
    codes = torch.empty(n, h, HEAD_DIM, 8, dtype=torch.uint8, device=dev)
    scales = torch.empty(n, h, HEAD_DIM, dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _check("nvfp4_v_token_major", lib.nvfp4_v_token_major(ctypes.byref(d), _ptr(page_ids), n, _ptr(codes),
                                                              _ptr(scales), _stream(stream, dev)))
    return codes, scales


def _current_device() -> torch.device:
    return torch.device("cuda", torch.cuda.current_device())


def nvfp4kv_debug_wait_timeout(limit_ns: int, stream=None) -> None:
    dev = stream.device if stream is not None else _current_device()
    with torch.cuda.device(dev):
        _check("nvfp4kv_debug_wait_timeout", lib.nvfp4kv_debug_wait_timeout(int(limit_ns), _stream(stream, dev)))


def nvfp4kv_get_device_status(stream=None) -> int:
    dev = stream.device if stream is not None else _current_device()
    with torch.cuda.device(dev):
        return int(lib.nvfp4kv_get_device_status(_stream(stream, dev)))
