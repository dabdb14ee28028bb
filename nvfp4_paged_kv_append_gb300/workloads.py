"""Seeded synthetic inputs shaped like the workloads the NVFP4 KV-cache pages
benchmark.  This module generates numbers only: it holds none of the
quantization or attention arithmetic, and both the CUDA path's tests/bench and
the CPU oracle draw their inputs from it.

Shapes follow the benchmark matrix of "NVFP4 KV cache A4Q prefill explained"
(section "Build the benchmark matrix": full prefills, a 128-token query over 2K
KV, 8-16 query tails over 16K KV) and the repack case of section "Compare A4Q
with dequantize-ahead repacking" (batch 4, q 128, KV 2,048, head dim 128).

Every tensor is drawn on the CPU from ``torch.Generator().manual_seed(seed)``.
Values are bf16.  The per-tensor global scale is the recipe's
``amax / (6 * 448)`` -- a caller-chosen input of the cache format, computed
here so that every consumer sees the same float32 value.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

HEAD_DIM = 128
PAGE_SIZE = 16


@dataclasses.dataclass
class Workload:
    """One batch: requests with (q_len, kv_len), heads, and the value recipe."""
    name: str
    q_lens: List[int]
    kv_lens: List[int]
    num_q_heads: int
    num_kv_heads: int
    causal: bool = True
    dist: str = "normal"          # normal | outliers | logu_channels
    seed: int = 0
    head_dim: int = HEAD_DIM
    page_size: int = PAGE_SIZE
    extra_pages: int = 3          # unused pages in the pool (never referenced)

    @property
    def batch(self) -> int:
        return len(self.q_lens)

    @property
    def total_q(self) -> int:
        return sum(self.q_lens)

    @property
    def total_kv(self) -> int:
        return sum(self.kv_lens)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def visible_pairs(self) -> int:
        """(query, key) pairs attended, per q-head (causal bound bottom-right)."""
        n = 0
        for ql, kl in zip(self.q_lens, self.kv_lens):
            if self.causal:
                first = kl - ql + 1      # keys visible to the first query
                n += ql * first + ql * (ql - 1) // 2
            else:
                n += ql * kl
        return n

    def flops(self) -> float:
        """QK + PV: 2*D multiply-adds each per visible pair per q-head."""
        return 4.0 * self.head_dim * self.visible_pairs() * self.num_q_heads


# The five configurations (sizes as stated; names say what they are).
def tiny_causal() -> Workload:
    return Workload("tiny_causal_b1_s256_h4x2", [256], [256], 4, 2, dist="outliers")


def short_q_long_kv() -> Workload:
    return Workload("shortq_b4_q128_kv2048_h32x8", [128] * 4, [2048] * 4, 32, 8)


def full_prefill_16k() -> Workload:
    return Workload("prefill_b1_s16384_h32x8", [16384], [16384], 32, 8, dist="logu_channels")


def chunked_tails() -> Workload:
    return Workload("tails_b8_q16_kv16400_h32x8", [16] * 8, [16400] * 8, 32, 8)


def decode_batch(seed: int = 0) -> Workload:
    g = torch.Generator().manual_seed(seed)
    kv = torch.randint(1024, 32769, (32,), generator=g).tolist()
    return Workload("decode_b32_kvU1K-32K_h32x8", [1] * 32, kv, 32, 8, seed=seed)


def long_prefill_ragged() -> Workload:
    return Workload("prefill_b2_s32768+7001_h64x8", [32768, 7001], [32768, 7001], 64, 8)


def small_ragged(seed: int = 1) -> Workload:
    """A ragged mixed batch small enough for full oracle comparison: several
    q tiles, a ragged tail, a q_len < kv_len request and a one-token request."""
    return Workload("small_ragged_h8x2", [200, 37, 1, 96], [200, 301, 17, 96], 8, 2, seed=seed)


CONFIGS = {
    "tiny": tiny_causal,
    "shortq": short_q_long_kv,
    "prefill16k": full_prefill_16k,
    "tails": chunked_tails,
    "decode": decode_batch,
    "prefill32k": long_prefill_ragged,
    "small_ragged": small_ragged,
}


def _values(shape, dist: str, gen: torch.Generator) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    D = shape[-1]
    if dist == "outliers":
        # 2% of the channels of this tensor (at least one) scaled by 8.
        n = max(1, round(0.02 * D))
        ch = torch.randperm(D, generator=gen)[:n]
        x[..., ch] *= 8.0
    elif dist == "logu_channels":
        # per-channel scale ~ LogUniform(0.25, 4)
        u = torch.rand(D, generator=gen, dtype=torch.float32)
        s = torch.exp(math.log(0.25) + u * (math.log(4.0) - math.log(0.25)))
        x = x * s
    elif dist != "normal":
        raise ValueError(dist)
    return x.to(torch.bfloat16)


def global_scale(x: torch.Tensor) -> float:
    """Recipe value of the per-tensor scale: amax / (6 * 448) in float32."""
    amax = x.float().abs().max()
    g = (amax / torch.tensor(2688.0, dtype=torch.float32)).item()
    return float(g) if g > 0 else 1.0


def fp8_scale(x: torch.Tensor) -> float:
    """Per-tensor scale of the FP8 comparison cache: amax / 448 in float32,
    so that the largest value lands on the largest finite E4M3 value."""
    amax = x.float().abs().max()
    g = (amax / torch.tensor(448.0, dtype=torch.float32)).item()
    return float(g) if g > 0 else 1.0


@dataclasses.dataclass
class Inputs:
    wl: Workload
    q: torch.Tensor            # [total_q, Hq, D] bf16
    k: torch.Tensor            # [total_kv, Hkv, D] bf16 (every cached token)
    v: torch.Tensor
    qo_indptr: torch.Tensor    # [B+1] int32
    kv_indptr: torch.Tensor    # [B+1] int64 (row offsets into k/v)
    kv_lens: torch.Tensor      # [B] int32
    page_table: torch.Tensor   # [B, max_pages] int32 (unused entries = -1)
    slot_mapping: torch.Tensor  # [total_kv] int64, slot of every k/v row
    num_pages: int
    k_global: float
    v_global: float
    sm_scale: float


def make_inputs(wl: Workload, with_q: bool = True) -> Inputs:
    gen = torch.Generator().manual_seed(wl.seed)
    D, P = wl.head_dim, wl.page_size
    Hq, Hkv = wl.num_q_heads, wl.num_kv_heads
    k = _values((wl.total_kv, Hkv, D), wl.dist, gen)
    v = _values((wl.total_kv, Hkv, D), wl.dist, gen)
    q = _values((wl.total_q, Hq, D), wl.dist, gen) if with_q else torch.empty(0, Hq, D, dtype=torch.bfloat16)
    pages_per = [(kl + P - 1) // P for kl in wl.kv_lens]
    num_pages = sum(pages_per) + wl.extra_pages
    perm = torch.randperm(num_pages, generator=gen).to(torch.int32)
    max_pages = max(pages_per) if pages_per else 1
    page_table = torch.full((wl.batch, max(1, max_pages)), -1, dtype=torch.int32)
    slots = []
    off = 0
    for b, kl in enumerate(wl.kv_lens):
        n = pages_per[b]
        page_table[b, :n] = perm[off:off + n]
        off += n
        j = torch.arange(kl, dtype=torch.int64)
        slots.append(page_table[b, (j // P)].to(torch.int64) * P + j % P)
    slot_mapping = torch.cat(slots) if slots else torch.empty(0, dtype=torch.int64)
    qo = torch.zeros(wl.batch + 1, dtype=torch.int32)
    qo[1:] = torch.cumsum(torch.tensor(wl.q_lens, dtype=torch.int64), 0).to(torch.int32)
    kvi = torch.zeros(wl.batch + 1, dtype=torch.int64)
    kvi[1:] = torch.cumsum(torch.tensor(wl.kv_lens, dtype=torch.int64), 0)
    return Inputs(wl, q, k, v, qo, kvi, torch.tensor(wl.kv_lens, dtype=torch.int32), page_table,
                  slot_mapping, num_pages, global_scale(k), global_scale(v), 1.0 / math.sqrt(D))


def shuffled_append_order(n: int, seed: int = 0) -> torch.Tensor:
    """A permutation used to append tokens out of order."""
    return torch.randperm(n, generator=torch.Generator().manual_seed(seed + 7))


def sample_rows(wl: Workload, per_request: int, seed: int = 0):
    """(request, position) pairs: the first and last query of every request
    plus `per_request` seeded random positions."""
    gen = torch.Generator().manual_seed(seed + 11)
    rows = []
    for b, ql in enumerate(wl.q_lens):
        if ql == 0:
            continue
        pos = {0, ql - 1}
        if ql > 2 and per_request > 0:
            pos.update(torch.randint(0, ql, (per_request,), generator=gen).tolist())
        rows.extend((b, int(i)) for i in sorted(pos))
    return rows


def tile_rows(wl: Workload, rows_per_tile: int = 128, seed: int = 0):
    """(request, position) pairs with one seeded query position inside every
    block of rows_per_tile // group consecutive query tokens of every request
    (a block of 128 rows = tokens x grouped heads), plus the first and last
    query of every request.  Used to reach every (request, q block) of a large
    batch with an affordable number of rows."""
    gen = torch.Generator().manual_seed(seed + 13)
    tpq = max(1, rows_per_tile // wl.group)
    rows = []
    for b, ql in enumerate(wl.q_lens):
        if ql == 0:
            continue
        pos = {0, ql - 1}
        n_blocks = (ql + tpq - 1) // tpq
        off = torch.randint(0, tpq, (n_blocks,), generator=gen).tolist()
        for t in range(n_blocks):
            pos.add(min(ql - 1, t * tpq + off[t]))
        rows.extend((b, int(i)) for i in sorted(pos))
    return rows
