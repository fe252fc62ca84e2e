"""CPU tests of the seeded input generators (layout only; no method arithmetic lives there)."""
import numpy as np

import mla_workloads as W


def test_bf16_rounding_is_rne_and_roundtrips():
    import torch
    r = np.random.default_rng(0)
    a = r.standard_normal(10000).astype(np.float32) * 100
    bits = W.to_bf16_bits(a)
    back = W.bf16_bits_to_f32(bits)
    ref = torch.from_numpy(a).to(torch.bfloat16).float().numpy()
    assert np.array_equal(back, ref)
    # ties go to even: 1 + 2^-8 sits halfway between 1 and 1 + 2^-7
    assert W.bf16_bits_to_f32(W.to_bf16_bits(np.array([1.0 + 2.0 ** -8], np.float32)))[0] == 1.0
    assert W.bf16_bits_to_f32(W.to_bf16_bits(np.array([W.SENTINEL], np.float32)))[0] == W.SENTINEL


def test_page_table_is_a_permutation_prefix():
    r = np.random.default_rng(1)
    pt, n = W.make_page_table(r, [1, 64, 65, 200], 64, 5, True)
    need = [1, 1, 2, 4]
    used = np.concatenate([pt[b, :k] for b, k in enumerate(need)])
    assert len(set(used.tolist())) == len(used) == sum(need)
    assert used.min() >= 0 and used.max() < n == sum(need) + 5
    for b, k in enumerate(need):
        assert np.all(pt[b, k:] == -1)


def test_scatter_gather_roundtrip_and_untouched_slots():
    s = W.replace_shape(W.TINY, page_size=4)
    case = W.make_decode_case(s, "bf16", [9, 4, 1], seed=3, spare_pages=2)
    pool, pt = case["pool"], case["page_table"]
    sentinel = W.sentinel_rows(1, s.width, "bf16")[0]
    owned = set()
    for b, L in enumerate([9, 4, 1]):
        rows = W.gather_rows(pool, pt[b], L)
        assert rows.shape == (L, s.width)
        for t in range(L):
            owned.add((int(pt[b, t // 4]), t % 4))
    for p in range(pool.shape[0]):
        for slot in range(4):
            if (p, slot) not in owned:
                assert np.array_equal(pool[p, slot], sentinel)


def test_generators_are_deterministic():
    a = W.make_decode_case(W.TINY, "bf16", [70, 3], seed=9)
    b = W.make_decode_case(W.TINY, "bf16", [70, 3], seed=9)
    for k in ("pool", "page_table", "q_nope", "q_rope", "w_uk", "w_uv", "w_o"):
        assert np.array_equal(a[k], b[k])


def test_append_case_reserves_the_new_slot():
    case = W.make_decode_case(W.TINY, "bf16", [64, 10], seed=4, append=True)
    assert list(case["seq_lens"]) == [65, 11]
    assert list(case["append_pos"]) == [64, 10]
    # position 64 of sequence 0 needs a second page
    assert case["page_table"][0, 1] >= 0


def test_named_workloads_shapes():
    w = W.WORKLOADS["decode_b16_l4096"]
    assert w.shape.width == 576 and w.batch == 16 and w.lens == (4096,) * 16
    r = np.random.default_rng(W.WORKLOADS["decode_ragged_b256"].seed)
    lens = W.draw_lens(W.WORKLOADS["decode_ragged_b256"], r)
    assert lens.shape == (256,) and lens.min() >= 256 and lens.max() <= 8192
    tiny = W.make_workload("tiny_f32")
    assert tiny["pool"].dtype == np.float32 and tiny["pool"].shape == (1, 64, 40)
