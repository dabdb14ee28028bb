"""Pins of the cache byte accounting against the figures printed on the pages
(tests/golden/accounting.json, each entry with its page and section)."""
import json
import os

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "accounting.json")
GIB = 1024 ** 3


def g():
    return json.load(open(GOLDEN))


def test_bits_per_value(orc):
    b = g()["bits_per_value"]
    # one (token, head) row of D=128 values: bytes for K alone
    per_row = orc.cache_bytes(1, 1, 1, 128) // 2
    bits = 8 * per_row / 128
    assert bits == b["bits_per_value"]
    assert b["data_bits_per_16"] + b["scale_bits_per_16"] == b["bits_per_16"] == 16 * bits
    assert 100 * bits / 8 == b["ratio_vs_fp8_percent"]
    assert round(8 / bits, 2) == b["capacity_multiplier_approx"]


def test_worked_example_L64(orc):
    w = g()["worked_per_token_L64"]
    L, H, D = w["layers"], w["kv_heads"], w["head_dim"]
    fp8 = 2 * L * H * D
    nv = L * orc.cache_bytes(1, 1, H, D)
    assert fp8 == w["fp8_bytes_per_token"] and fp8 // 1024 == w["fp8_kib_per_token"]
    assert nv == w["nvfp4_bytes_per_token"] and nv // 1024 == w["nvfp4_kib_per_token"]
    assert fp8 * w["tokens"] == w["fp8_gib"] * GIB
    assert nv * w["tokens"] == w["nvfp4_gib"] * GIB
    assert (fp8 - nv) * w["tokens"] == w["difference_gib"] * GIB


def test_worked_example_L80(orc):
    w = g()["worked_per_token_L80"]
    L, H, D = w["layers"], w["kv_heads"], w["head_dim"]
    vals = 2 * L * H * D
    assert vals == w["values_per_token"]
    assert 2 * vals == w["bf16_bytes_per_token"] and 2 * vals // 1024 == w["bf16_kib_per_token"]
    assert vals // 1024 == w["fp8_kib_per_token"]
    nv = L * orc.cache_bytes(1, 1, H, D)
    assert nv == w["nvfp4_bytes_per_token"] and nv // 1024 == w["nvfp4_kib_per_token"]
    seq = nv * w["seq_tokens"] / GIB
    assert round(seq, 2) == w["nvfp4_gib_per_seq_approx"]
    assert 2 * vals * w["seq_tokens"] == w["bf16_gib_per_seq"] * GIB
    assert vals * w["seq_tokens"] == w["fp8_gib_per_seq"] * GIB
    assert nv * w["seq_tokens"] * w["num_seqs"] == w["nvfp4_gib_all_seqs"] * GIB
    assert 2 * vals * w["seq_tokens"] * w["num_seqs"] == w["bf16_gib_all_seqs"] * GIB


def test_pool_bytes_scale_with_pages(orc):
    # pages of 16 tokens: the pool is pages * 16 token rows of 144 B per head
    assert orc.cache_bytes(10, 16, 8, 128) == 10 * 16 * 8 * 144
