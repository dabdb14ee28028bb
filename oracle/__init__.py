"""CPU oracle for the NVFP4 paged KV-cache path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and bench.py's ``cpu_baseline`` /
``--impl reference`` legs may import this package.  The product path (the CUDA
library ``libnvfp4kv.so`` and its Python binding) never imports, links or
calls anything here, and this package shares no code with it: the arithmetic
lives in ``nvfp4_oracle.c`` (plain C, fp64 attention, stated fp32 codec
steps), and this module only marshals numpy arrays into it.

The readings the oracle takes where the source pages are silent (scale
formula, rounding, division by the quantized scale, zero blocks, nibble order,
Q scheme, causal alignment, cache layout) are listed in ``nvfp4_oracle.h``.

Parity status per function:
  e2m1/e4m3 codec, block quantizer, append, gather/decode, attention,
  cache_bytes -- pinned by tests/test_oracle_*.py (format definitions, a
  library cast, brute force, closed forms, the pages' worked byte counts).
  FP8 comparison cache (fp8_* and FP8Pools) -- the element codec pinned
  against torch's float8_e4m3fn cast, the byte count against the pages'
  131,072 B per token, attention through the same pinned definition.
  dense_attention (attention on the unquantized values, the reference of the
  accuracy report) -- pinned against scipy softmax on a ragged batch.
  decode_q_a4q with a single caller-given scale (per-tensor or single-level
  query scheme) -- the GLOBAL mode of the cache's block codec, pinned by the
  codec pins and an exact round trip.
  FP4 PV experiment (v_token_major_page, gather_v_token_major,
  fp4pv_attention_rows, paged_attention(pv="fp4")) -- the pages define no
  FP4 PV, so its readings X1..X5 are this oracle's own; pinned by the
  re-layout's axis against numpy reductions, closed forms (uniform and
  one-hot attention), its distance to the exact attention, and the
  reference-independence that X3 promises (tile size and threshold change
  nothing but rounding).
  quantize_rows(mode=PER_ROW), the per-row A4Q Q scheme -- the pages leave
  the scheme open, so it is pinned only to its stated reading (round trip and
  error bound), not to any external value: parity unpinned against the pages.
"""
from __future__ import annotations

import concurrent.futures as cf
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

GLOBAL = 0
PER_ROW = 1

_lib = None

# Independent (request, head) problems and disjoint token ranges of the append
# run on a thread pool: ctypes releases the GIL inside the C calls, and no two
# tasks write the same output.  Nothing about the arithmetic changes.
WORKERS = max(1, min(32, os.cpu_count() or 1))


def _pmap(fn, items):
    items = list(items)
    if WORKERS == 1 or len(items) <= 1:
        return [fn(x) for x in items]
    with cf.ThreadPoolExecutor(max_workers=WORKERS) as ex:
        return list(ex.map(fn, items))


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, no fused multiply-add)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or force or (
        os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                           os.path.getmtime(os.path.join(_HERE, "nvfp4_oracle.h"))))
    if stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, f32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_double
        lib.orc_e2m1_value.restype = f64
        lib.orc_e2m1_value.argtypes = [ctypes.c_uint]
        lib.orc_e4m3_value.restype = f64
        lib.orc_e4m3_value.argtypes = [ctypes.c_uint]
        lib.orc_e4m3_encode.restype = ctypes.c_uint
        lib.orc_e4m3_encode.argtypes = [f32]
        lib.orc_e2m1_encode.restype = ctypes.c_uint
        lib.orc_e2m1_encode.argtypes = [f32]
        lib.orc_e2m1_encode_n.argtypes = [P, i64, P]
        lib.orc_quantize_block16.argtypes = [P, f32, P, P]
        lib.orc_quantize_rows.argtypes = [P, i64, i32, i32, f32, P, P, P]
        lib.orc_dequantize_rows.argtypes = [P, P, i64, i32, P, f32, P]
        lib.orc_kv_append.restype = i32
        lib.orc_kv_append.argtypes = [P, P, P, i64, i32, i32, i32, i64, f32, f32, P, P, P, P]
        lib.orc_gather_decode.restype = i32
        lib.orc_gather_decode.argtypes = [P, P, P, i32, i32, i32, i32, i32, i64, f32, P]
        lib.orc_attention_rows.argtypes = [P, P, i32, i32, P, P, i32, i32, i32, f64, P, P]
        lib.orc_cache_bytes.restype = i64
        lib.orc_cache_bytes.argtypes = [i64, i32, i32, i32]
        lib.orc_fp8_encode.restype = ctypes.c_uint
        lib.orc_fp8_encode.argtypes = [f32]
        lib.orc_fp8_quantize_rows.argtypes = [P, i64, f32, P]
        lib.orc_fp8_kv_append.restype = i32
        lib.orc_fp8_kv_append.argtypes = [P, P, P, i64, i32, i32, i32, i64, f32, f32, P, P]
        lib.orc_fp8_gather_decode.restype = i32
        lib.orc_fp8_gather_decode.argtypes = [P, P, i32, i32, i32, i32, i32, i64, f32, P]
        lib.orc_fp8_cache_bytes.restype = i64
        lib.orc_fp8_cache_bytes.argtypes = [i64, i32, i32, i32]
        lib.orc_v_token_major_page.argtypes = [P, i32, P, P]
        lib.orc_fp4pv_attention_rows.argtypes = [P, P, i32, i32, P, P, i32, i32, i32, f64, i32, i32, f32, f64,
                                                 P, P, P]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _f32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


# --- formats -----------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return _load().orc_e2m1_value(int(code))


def e4m3_value(byte: int) -> float:
    return _load().orc_e4m3_value(int(byte))


def e4m3_encode(x: float) -> int:
    return int(_load().orc_e4m3_encode(float(np.float32(x))))


def e2m1_encode(q: float) -> int:
    return int(_load().orc_e2m1_encode(float(np.float32(q))))


def e4m3_encode_array(x) -> np.ndarray:
    lib = _load()
    return np.array([lib.orc_e4m3_encode(float(v)) for v in _f32(x).ravel()], dtype=np.uint8)


def e2m1_encode_array(q) -> np.ndarray:
    q = _f32(q).ravel()
    codes = np.empty(q.size, dtype=np.uint8)
    _load().orc_e2m1_encode_n(_ptr(q), q.size, _ptr(codes))
    return codes


# --- codec -------------------------------------------------------------------

def quantize_block16(x, g: float):
    x = _f32(x)
    assert x.shape == (16,)
    packed = np.zeros(8, np.uint8)
    scale = np.zeros(1, np.uint8)
    _load().orc_quantize_block16(_ptr(x), float(np.float32(g)), _ptr(packed), _ptr(scale))
    return packed, int(scale[0])


def quantize_rows(x, mode: int = GLOBAL, g: float = 1.0):
    """x: [rows, D] float32 -> (packed [rows, D/2] u8, scales [rows, D/16] u8,
    row_g [rows] f32 or None)."""
    x = _f32(x)
    rows, D = x.shape
    packed = np.zeros((rows, D // 2), np.uint8)
    scales = np.zeros((rows, D // 16), np.uint8)
    row_g = np.zeros(rows, np.float32) if mode == PER_ROW else None
    _load().orc_quantize_rows(_ptr(x), rows, D, mode, float(np.float32(g)), _ptr(packed),
                              _ptr(scales), _ptr(row_g) if row_g is not None else None)
    return packed, scales, row_g


def dequantize_rows(packed, scales, row_g=None, g: float = 1.0) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, half = packed.shape
    D = half * 2
    out = np.zeros((rows, D), np.float64)
    rg = _f32(row_g) if row_g is not None else None
    _load().orc_dequantize_rows(_ptr(packed), _ptr(scales), rows, D,
                                _ptr(rg) if rg is not None else None,
                                float(np.float32(g)), _ptr(out))
    return out


# --- paged cache -------------------------------------------------------------

class Pools:
    """The four byte pools of one layer's cache, in the stated layout:
    data [pages][Hkv][page_size][D/2], scales [pages][Hkv][page_size][D/16]."""

    def __init__(self, num_pages: int, Hkv: int, D: int = 128, page_size: int = 16,
                 fill: int = 0):
        self.num_pages, self.Hkv, self.D, self.page_size = num_pages, Hkv, D, page_size
        shp_d = (num_pages, Hkv, page_size, D // 2)
        shp_s = (num_pages, Hkv, page_size, D // 16)
        self.k_data = np.full(shp_d, fill, np.uint8)
        self.k_scale = np.full(shp_s, fill, np.uint8)
        self.v_data = np.full(shp_d, fill, np.uint8)
        self.v_scale = np.full(shp_s, fill, np.uint8)


def kv_append(pools: Pools, k, v, slot_mapping, k_g: float, v_g: float) -> None:
    """k, v: [T, Hkv, D] float32 (bf16 values); slot_mapping: [T] int64."""
    k = _f32(k)
    v = _f32(v)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, Hkv, D = k.shape
    assert Hkv == pools.Hkv and D == pools.D and slots.shape == (T,)
    lib = _load()
    step = max(1024, (T + WORKERS - 1) // WORKERS)

    def run(t0):
        n = min(step, T - t0)
        return lib.orc_kv_append(
            ctypes.c_void_p(k.ctypes.data + t0 * k.strides[0]), ctypes.c_void_p(v.ctypes.data + t0 * v.strides[0]),
            ctypes.c_void_p(slots.ctypes.data + t0 * 8), n, Hkv, D, pools.page_size, pools.num_pages,
            float(np.float32(k_g)), float(np.float32(v_g)), _ptr(pools.k_data), _ptr(pools.k_scale),
            _ptr(pools.v_data), _ptr(pools.v_scale))

    if T > 0 and any(rc != 0 for rc in _pmap(run, range(0, T, step))):
        raise ValueError("slot out of range")


# --- FP8 (E4M3) comparison cache (readings F1..F3 of nvfp4_oracle.h) -------

def fp8_encode_array(x) -> np.ndarray:
    lib = _load()
    return np.array([lib.orc_fp8_encode(float(v)) for v in _f32(x).ravel()], dtype=np.uint8)


def fp8_quantize(x, g: float) -> np.ndarray:
    """Any-shape float32 array -> uint8 codes with per-tensor scale g (F1, F2)."""
    x = _f32(x)
    out = np.zeros(x.shape, np.uint8)
    _load().orc_fp8_quantize_rows(_ptr(x), x.size, float(np.float32(g)), _ptr(out))
    return out


class FP8Pools:
    """The two byte pools of one layer's FP8 cache (F3):
    data [pages][Hkv][page_size][D], one E4M3 code per value."""

    def __init__(self, num_pages: int, Hkv: int, D: int = 128, page_size: int = 16, fill: int = 0):
        self.num_pages, self.Hkv, self.D, self.page_size = num_pages, Hkv, D, page_size
        shp = (num_pages, Hkv, page_size, D)
        self.k_data = np.full(shp, fill, np.uint8)
        self.v_data = np.full(shp, fill, np.uint8)


def fp8_kv_append(pools: FP8Pools, k, v, slot_mapping, k_g: float, v_g: float) -> None:
    """k, v: [T, Hkv, D] float32 (bf16 values); slot_mapping: [T] int64."""
    k = _f32(k)
    v = _f32(v)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, Hkv, D = k.shape
    assert Hkv == pools.Hkv and D == pools.D and slots.shape == (T,)
    lib = _load()
    step = max(1024, (T + WORKERS - 1) // WORKERS)

    def run(t0):
        n = min(step, T - t0)
        return lib.orc_fp8_kv_append(
            ctypes.c_void_p(k.ctypes.data + t0 * k.strides[0]), ctypes.c_void_p(v.ctypes.data + t0 * v.strides[0]),
            ctypes.c_void_p(slots.ctypes.data + t0 * 8), n, Hkv, D, pools.page_size, pools.num_pages,
            float(np.float32(k_g)), float(np.float32(v_g)), _ptr(pools.k_data), _ptr(pools.v_data))

    if T > 0 and any(rc != 0 for rc in _pmap(run, range(0, T, step))):
        raise ValueError("slot out of range")


def fp8_gather_decode(pools: FP8Pools, which: str, page_row, kv_len: int, head: int, g: float) -> np.ndarray:
    data = pools.k_data if which == "k" else pools.v_data
    row = np.ascontiguousarray(page_row, dtype=np.int32)
    out = np.zeros((kv_len, pools.D), np.float64)
    rc = _load().orc_fp8_gather_decode(_ptr(data), _ptr(row), kv_len, head, pools.Hkv, pools.D, pools.page_size,
                                       pools.num_pages, float(np.float32(g)), _ptr(out))
    if rc != 0:
        raise ValueError("page id out of range")
    return out


def fp8_cache_bytes(num_pages: int, page_size: int, Hkv: int, D: int) -> int:
    return int(_load().orc_fp8_cache_bytes(num_pages, page_size, Hkv, D))


def gather_decode(pools: Pools, which: str, page_row, kv_len: int, head: int, g: float) -> np.ndarray:
    data = pools.k_data if which == "k" else pools.v_data
    scale = pools.k_scale if which == "k" else pools.v_scale
    row = np.ascontiguousarray(page_row, dtype=np.int32)
    out = np.zeros((kv_len, pools.D), np.float64)
    rc = _load().orc_gather_decode(_ptr(data), _ptr(scale), _ptr(row), kv_len, head, pools.Hkv,
                                   pools.D, pools.page_size, pools.num_pages,
                                   float(np.float32(g)), _ptr(out))
    if rc != 0:
        raise ValueError("page id out of range")
    return out


# --- attention ---------------------------------------------------------------

def attention_rows(q, pos, q_len: int, k, v, causal: bool, sm_scale: float):
    """q: [n, D] float64 decoded queries at positions pos (within the request);
    k, v: [kv_len, D] float64.  Returns (o [n, D] f64, lse [n] f64)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    n, D = q.shape
    out = np.zeros((n, D), np.float64)
    lse = np.zeros(n, np.float64)
    _load().orc_attention_rows(_ptr(q), _ptr(pos), n, q_len, _ptr(k), _ptr(v), k.shape[0], D,
                               int(bool(causal)), float(sm_scale), _ptr(out), _ptr(lse))
    return out, lse


def cache_bytes(num_pages: int, page_size: int, Hkv: int, D: int) -> int:
    return int(_load().orc_cache_bytes(num_pages, page_size, Hkv, D))


# --- FP4 PV experiment (readings X1..X5 in nvfp4_oracle.h) ---------------------

FP4PV_TILE = 128
FP4PV_TAU = 4


def fp4pv_p_scale(tau: int = FP4PV_TAU) -> float:
    """X4: g_p = fl32(2^tau / 2688)."""
    return float(np.float32(2.0 ** tau) / np.float32(2688.0))


def v_token_major_page(x16):
    """X1 for one page: x16 [16, D] values (decoded without g) -> codes
    [D, 8] uint8 (slot 2i in the low nibble of byte i) and scales [D] uint8."""
    x = _f32(x16)
    assert x.shape[0] == 16
    D = x.shape[1]
    codes = np.zeros((D, 8), np.uint8)
    scales = np.zeros(D, np.uint8)
    _load().orc_v_token_major_page(_ptr(x), D, _ptr(codes), _ptr(scales))
    return codes, scales


def decode_token_major(codes, scales, g: float) -> np.ndarray:
    """Decode one page's token-major blocks: [D, 8] codes and [D] scales ->
    [16, D] float64 values e2m1 * e4m3 * g (X1, R5)."""
    codes = np.asarray(codes, np.uint8)
    e2m1 = np.array([e2m1_value(c) for c in range(16)])
    e4m3 = np.array([e4m3_value(b) for b in range(256)])
    nib = np.stack([codes & 15, codes >> 4], axis=2).reshape(codes.shape[0], 16)  # [D, slot]
    return (e2m1[nib] * e4m3[np.asarray(scales, np.uint8)][:, None] * float(np.float32(g))).T


def gather_v_token_major(pools: Pools, page_row, kv_len: int, head: int, v_g: float) -> np.ndarray:
    """X1 over a request: the first kv_len tokens of V for one kv head,
    re-coded page by page along tokens (slots past kv_len taken as 0) and
    decoded.  Returns [kv_len, D] float64."""
    raw = gather_decode(pools, "v", page_row, kv_len, head, 1.0)  # e2m1 * e4m3, exact
    n_pages = -(-kv_len // 16)
    buf = np.zeros((n_pages * 16, pools.D), np.float32)
    buf[:kv_len] = raw
    out = np.zeros((n_pages * 16, pools.D), np.float64)
    for p in range(n_pages):
        codes, scales = v_token_major_page(buf[16 * p:16 * p + 16])
        out[16 * p:16 * p + 16] = decode_token_major(codes, scales, v_g)
    return out[:kv_len]


def fp4pv_attention_rows(q, pos, q_len: int, k, vhat, causal: bool, sm_scale: float,
                         tile: int = FP4PV_TILE, tau: int = FP4PV_TAU, eps=None):
    """X2..X5 for rows of one (request, q-head): q [n, D] decoded queries,
    k [kv_len, D] decoded keys, vhat [kv_len, D] token-major V decoded by X1.
    Returns (o [n, D] f64, lse [n] f64), and with eps given also the slack
    [n, D]: how far o can move when P decisions within relative eps of a
    rounding boundary go the other way."""
    assert tile > 0 and tile % 16 == 0
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    vhat = np.ascontiguousarray(vhat, dtype=np.float64)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    n, D = q.shape
    out = np.zeros((n, D), np.float64)
    lse = np.zeros(n, np.float64)
    slack = np.zeros((n, D), np.float64) if eps is not None else None
    _load().orc_fp4pv_attention_rows(_ptr(q), _ptr(pos), n, q_len, _ptr(k), _ptr(vhat), k.shape[0], D,
                                     int(bool(causal)), float(sm_scale), int(tile), int(tau),
                                     fp4pv_p_scale(tau), float(eps or 0.0), _ptr(out), _ptr(lse),
                                     _ptr(slack) if slack is not None else None)
    return (out, lse) if eps is None else (out, lse, slack)


def decode_q_a4q(q_rows, q_scale: float = 0.0) -> np.ndarray:
    """A4Q query as the kernel sees it, quantized then decoded (R6, R5).
    q_scale 0: per-row dual-level scale (R6); q_scale > 0: that one scale for
    every row (the GLOBAL mode of the same block codec -- a per-tensor scale,
    or 1 for a single-level scheme).  q_rows: [n, D] float32 -> [n, D]
    float64."""
    if q_scale > 0:
        packed, scales, _ = quantize_rows(q_rows, GLOBAL, q_scale)
        return dequantize_rows(packed, scales, g=q_scale)
    packed, scales, row_g = quantize_rows(q_rows, PER_ROW)
    return dequantize_rows(packed, scales, row_g=row_g)


def paged_attention(pools: Pools, q, qo_indptr, kv_lens, page_table, Hq: int, k_g: float,
                    v_g: float, causal: bool, sm_scale: float, q_mode: str = "bf16",
                    rows=None, q_scale: float = 0.0, pv: str = "wide", slack_eps=None):
    """Attention of a ragged batch over the paged cache (an NVFP4 `Pools` or
    an FP8 `FP8Pools`, decoded by R5 or F3).

    q: [total_q, Hq, D] float32 (bf16 values); q_mode "bf16" uses q as is,
    "a4q" uses the quantized-then-decoded query (per-row scale, or the single
    scale q_scale when it is > 0).  rows: optional list of (request, position)
    pairs to evaluate (all rows of every request if None).  pv "wide" is the
    definition (P and V exact); "fp4" is the FP4 PV experiment (X1..X5, NVFP4
    pools only), and with slack_eps given each value also carries the slack
    [Hq, D] of fp4pv_attention_rows.
    Returns dict {(request, position): (o [Hq, D], lse [Hq])}.
    """
    assert slack_eps is None or pv == "fp4"
    assert pv in ("wide", "fp4") and (pv == "wide" or isinstance(pools, Pools))
    q = _f32(q)
    qo = np.asarray(qo_indptr, dtype=np.int64)
    kvl = np.asarray(kv_lens, dtype=np.int64)
    pt = np.asarray(page_table, dtype=np.int32)
    Hkv = pools.Hkv
    G = Hq // Hkv
    B = len(kvl)
    want = {}
    if rows is None:
        for b in range(B):
            for i in range(int(qo[b + 1] - qo[b])):
                want.setdefault(b, []).append(i)
    else:
        for b, i in rows:
            want.setdefault(int(b), []).append(int(i))
    result = {}

    # One request at a time: decode its K and V once per kv head, then run
    # the rows in chunks so that every worker thread has work even when a
    # request has few kv heads and many sampled rows.
    for b, positions in want.items():
        q_len, kv_len = int(qo[b + 1] - qo[b]), int(kvl[b])
        pos_all = np.array(sorted(set(positions)), np.int32)
        gather = fp8_gather_decode if isinstance(pools, FP8Pools) else gather_decode
        gather_v = (lambda h: gather_v_token_major(pools, pt[b], kv_len, h, v_g)) if pv == "fp4" else \
            (lambda h: gather(pools, "v", pt[b], kv_len, h, v_g))
        attend = (lambda *a: fp4pv_attention_rows(*a, eps=slack_eps)) if pv == "fp4" else attention_rows
        dec = dict(zip(range(Hkv), _pmap(
            lambda h: (gather(pools, "k", pt[b], kv_len, h, k_g), gather_v(h)), range(Hkv))))
        n_chunks = max(1, min(len(pos_all), -(-2 * WORKERS // Hkv)))
        chunks = [c for c in np.array_split(pos_all, n_chunks) if len(c)]

        def one(task):
            h, pos = task
            kd, vd = dec[h]
            res = []
            for gq in range(G):
                hq = h * G + gq
                qr = q[qo[b] + pos, hq, :]
                qd = decode_q_a4q(qr, q_scale) if q_mode == "a4q" else qr.astype(np.float64)
                res.append((hq,) + attend(qd, pos, q_len, kd, vd, causal, sm_scale))
            return pos, res

        for i in pos_all:
            result[(b, int(i))] = (np.zeros((Hq, pools.D)), np.zeros(Hq)) + \
                ((np.zeros((Hq, pools.D)),) if slack_eps is not None else ())
        for pos, res in _pmap(one, [(h, c) for h in range(Hkv) for c in chunks]):
            for hq, *vals in res:
                for r, i in enumerate(pos):
                    for slot, val in enumerate(vals):
                        result[(b, int(i))][slot][hq] = val[r]
        del dec
    return result


def dense_attention(q, qo_indptr, k, v, kv_indptr, Hq: int, causal: bool, sm_scale: float, rows):
    """Attention of the given (request, position) rows on the UNQUANTIZED
    values: q [total_q, Hq, D], k and v [total_kv, Hkv, D] float32 (bf16
    values), request b's keys are rows kv_indptr[b] .. kv_indptr[b+1]-1.  No
    cache codec is involved: this is the fp64 reference the quantization error
    is measured against.  Returns {(request, position): (o [Hq, D], lse [Hq])}."""
    q = _f32(q)
    k = _f32(k)
    v = _f32(v)
    qo = np.asarray(qo_indptr, dtype=np.int64)
    kvi = np.asarray(kv_indptr, dtype=np.int64)
    Hkv = k.shape[1]
    G = Hq // Hkv
    want = {}
    for b, i in rows:
        want.setdefault(int(b), set()).add(int(i))
    result = {}
    for b, positions in want.items():
        pos_all = np.array(sorted(positions), np.int32)
        q_len = int(qo[b + 1] - qo[b])
        k0, k1 = int(kvi[b]), int(kvi[b + 1])

        def one(h):
            kd = np.ascontiguousarray(k[k0:k1, h, :], dtype=np.float64)
            vd = np.ascontiguousarray(v[k0:k1, h, :], dtype=np.float64)
            res = []
            for gq in range(G):
                hq = h * G + gq
                qr = q[qo[b] + pos_all, hq, :].astype(np.float64)
                res.append((hq,) + attention_rows(qr, pos_all, q_len, kd, vd, causal, sm_scale))
            return res

        for i in pos_all:
            result[(b, int(i))] = (np.zeros((Hq, k.shape[2])), np.zeros(Hq))
        for res in _pmap(one, range(Hkv)):
            for hq, o, lse in res:
                for r, i in enumerate(pos_all):
                    result[(b, int(i))][0][hq] = o[r]
                    result[(b, int(i))][1][hq] = lse[r]
    return result
