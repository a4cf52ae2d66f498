"""The seeded input generator: deterministic, the workloads' shapes and structure."""
import math

import torch

from gva_inputs import WORKLOADS, make_case, make_gqa_keys, workload


def test_deterministic():
    a = make_case(workload("tiny"))
    b = make_case(workload("tiny"))
    for k in ("V", "Kr", "q_nope", "q_rope", "M", "seq_len", "v_new", "k_new"):
        assert torch.equal(getattr(a, k), getattr(b, k))


def test_workload_table():
    w = WORKLOADS["350m"]
    assert (w.B, w.H, w.G, w.d_h, w.d_n, w.d_r, w.T) == (8, 16, 4, 64, 64, 16, 4096)
    assert abs(w.scale - 1 / math.sqrt(80)) < 1e-15
    assert WORKLOADS["tiny"].cache_dtype == "f32"
    assert WORKLOADS["long"].T == 131072 and WORKLOADS["long"].spike_frac == 0.01
    assert WORKLOADS["paged"].page_size == 64


def test_shapes_and_dtypes_small_350m():
    c = make_case(workload("350m", T=100))
    assert c.V.shape == (8 * 100, 4, 64) and c.V.dtype == torch.bfloat16
    assert c.Kr.shape == (800, 16) and c.q_nope.dtype == torch.bfloat16
    assert c.M.dtype == torch.float32 and c.seq_len.tolist() == [100] * 8
    # M ~ N(0, 1/d_h)
    assert abs(c.M.std().item() - 1 / 8) < 0.01


def test_ragged_lengths_and_offsets():
    c = make_case(workload("ragged", B=32, len_range=(1, 50)))
    L = c.seq_len.long()
    assert int(L.min()) >= 1 and int(L.max()) <= 50
    assert c.offsets[0] == 0 and torch.equal(c.offsets[1:] - c.offsets[:-1], c.seq_len)
    assert c.num_rows == int(L.sum())


def test_paged_block_table_is_a_permutation():
    c = make_case(workload("paged", B=6, len_range=(10, 300), extra_slots=5))
    bt = c.block_table.long()
    used = bt[bt >= 0]
    assert sorted(used.tolist()) == list(range(c.num_pages))
    for b in range(6):
        need = (int(c.seq_len[b]) + 5 + 63) // 64
        assert int((bt[b] >= 0).sum()) == need


def test_long_spikes_scale_one_percent():
    c = make_case(workload("long", T=3000, B=2))
    for b, pos in enumerate(c.extras["spikes"]):
        assert len(pos) == 30 and len(set(pos.tolist())) == 30
    big = c.V.float().abs().amax(dim=(1, 2)).view(2, 3000)
    spiked = big[0, c.extras["spikes"][0]]
    assert spiked.mean() > 4 * big[0].median()


def test_gqa_keys_match_value_layout():
    c = make_case(workload("350m", T=10))
    K = make_gqa_keys(c)
    assert K.shape == c.V.shape and K.dtype == c.V.dtype and not torch.equal(K, c.V)
