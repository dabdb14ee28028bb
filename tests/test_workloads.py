"""The seeded input recipe: the shapes and sizes the parity tests and the
bench rely on are what the recipe states, and the generator is
deterministic (inputs follow the benchmark matrix of "NVFP4 KV cache prefill
vs decode performance", section "Build the benchmark matrix")."""
import numpy as np
import torch

from nvfp4_paged_kv_append_gb300 import workloads as W


def test_decode_batch_lengths():
    wl = W.decode_batch()
    kv = np.array(wl.kv_lens)
    assert wl.batch == 32 and wl.num_q_heads == 32 and wl.num_kv_heads == 8
    assert kv.min() >= 1024 and kv.max() <= 32768
    assert int(kv.sum()) == 429_798  # the decode bytes quoted in the docs: 144 B x 8 heads x this
    assert 144 * 8 * int(kv.sum()) == 495_127_296


def test_prefill_16k_shape():
    wl = W.full_prefill_16k()
    assert wl.batch == 1 and wl.q_lens == [16384] and wl.kv_lens == [16384]
    assert (wl.num_q_heads, wl.num_kv_heads, wl.causal) == (32, 8, True)
    # QK and PV FLOPs of the causal 16K case: 2 x D per visible pair per q head each
    pairs = 16384 * 16385 // 2
    assert wl.flops() == 2 * (2 * 128 * pairs * 32)


def test_inputs_are_deterministic_and_paged():
    wl = W.Workload("det", [5, 0, 17], [40, 3, 17], 4, 2, seed=11)
    a, b = W.make_inputs(wl), W.make_inputs(wl)
    for x, y in ((a.q, b.q), (a.k, b.k), (a.v, b.v), (a.page_table, b.page_table), (a.slot_mapping, b.slot_mapping)):
        assert torch.equal(x, y)
    # every token gets a distinct slot inside its request's pages
    slots = a.slot_mapping.numpy()
    assert len(set(slots.tolist())) == len(slots) == sum(wl.kv_lens)
    off = 0
    for r, kl in enumerate(wl.kv_lens):
        pages = set(a.page_table[r, : (kl + 15) // 16].tolist())
        assert all(int(s) // 16 in pages for s in slots[off:off + kl])
        assert [int(s) % 16 for s in slots[off:off + kl]] == [j % 16 for j in range(kl)]
        off += kl
    assert a.qo_indptr.tolist() == [0, 5, 5, 22]


def test_global_scale_recipe():
    x = torch.tensor([[0.5, -1344.0, 3.0]], dtype=torch.bfloat16)
    assert W.global_scale(x) == 0.5  # amax / (6 * 448) = 1344 / 2688
    assert W.global_scale(torch.zeros(4)) == 1.0


def test_shuffled_order_is_a_permutation():
    p = W.shuffled_append_order(1000)
    assert sorted(p.tolist()) == list(range(1000))
    assert not torch.equal(p, torch.arange(1000))
