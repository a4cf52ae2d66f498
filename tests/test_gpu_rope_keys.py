"""GPU parity of the decode with ordinary RoPE on the reconstructed key
(gva_rope_keys_decode_attention, through the C ABI) against the oracle's
od_gva_decode_rope_keys on the same seeded inputs.  bf16 cache: max-abs 2e-2 and relative
L2 1e-3 on out and lse, the bound of every bf16-cache decode here.

The variant follows the agihunt summary (results discussion: the scale-matched row
rotates the rebuilt key itself) and the analysis page (关键技巧二: the rotation then sits
between q and M_h^T, so M_h cannot be absorbed)."""
import numpy as np
import pytest
import torch

import oracle
from gva_inputs import make_case, workload
from helpers import assert_close, gva, oracle_rows

pytestmark = pytest.mark.gpu


def _rows(c, dev):
    g = gva()
    w = c.w
    offs = c.offsets.to(dev) if c.offsets is not None else None
    bt = c.block_table.to(dev) if c.block_table is not None else None
    return g.Rows(w.layout, c.num_rows, T_cap=c.T_cap, offsets=offs, block_table=bt,
                  page_size=w.page_size)


def _table(c):
    """(cos, sin) over d_n, from the oracle's table routine (fp64 values rounded once)."""
    rows = max(128, int(c.seq_len.max()) + 1 if c.w.B else 1)
    return torch.from_numpy(oracle.rope_table_f32(rows, c.w.d_n, c.w.base))


def _run(c):
    g = gva()
    w = c.w
    dev = torch.device("cuda")
    dims = g.Dims(w.B, w.H, w.G, w.d_h, w.d_n, 0, g.GVA_BF16,
                  g.GVA_F32 if w.q_dtype == "f32" else g.GVA_BF16)
    cache = g.Cache(_rows(c, dev), c.V.to(dev), None)
    out = torch.full((w.B, w.H, w.d_h), float("nan"), device=dev)
    lse = torch.full((w.B, w.H), float("nan"), device=dev)
    ws = g.rope_keys_workspace(dims, dev)
    g.gva_rope_keys_decode_attention(dims, c.q_nope.to(dev), c.M.to(dev), c.seq_len.to(dev),
                                     cache, _table(c).to(dev), w.scale, out, lse, ws)
    torch.cuda.synchronize()
    assert g.gva_get_device_status() == 0
    return out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _oracle(c):
    w = c.w
    return oracle.gva_decode_rope_keys(c.q_nope, c.M, c.seq_len, oracle_rows(c), c.V, w.scale,
                                       w.base, w.G)


def _oracle_heads(c, b, heads):
    """The oracle on sequence b and some heads of one value group (that group's value
    columns passed as a one-group cache)."""
    w = c.w
    r = w.H // w.G
    g = heads[0] // r
    assert all(h // r == g for h in heads)
    hs = torch.tensor(heads)
    V1 = c.V[:, g:g + 1, :].contiguous()
    return oracle.gva_decode_rope_keys(c.q_nope[b:b + 1][:, hs], c.M[hs], c.seq_len[b:b + 1],
                                       oracle_rows(c, [b]), V1, w.scale, w.base, 1)


CASES = [
    ("350m", dict(T=300, B=3)),                                   # d_h 64, d_n 64, 4 heads / slice
    ("350m", dict(T=1000, B=2, G=2)),                             # r = 8: two slices per group
    ("350m", dict(T=129, B=3, H=8, G=8)),                         # r = 1: 64 accumulator columns
    ("350m", dict(T=300, B=2, d_n=128)),                          # d_h 64, d_n 128
    ("long", dict(T=700, B=2)),                                   # d_h 128, d_n 128, 2 heads / slice
    ("long", dict(T=200, B=2, H=8, G=4, d_n=64)),                 # d_h 128, d_n 64
    ("350m", dict(T=257, B=2, q_dtype="f32")),                    # fp32 queries
    ("ragged", dict(B=7, len_range=(0, 600))),                    # ragged tails, empty rows
    ("paged", dict(B=5, len_range=(1, 700))),                     # 64-token pages
    ("paged", dict(B=4, len_range=(50, 400), page_size=16, H=16, G=4, d_h=64, d_n=64)),
]


@pytest.mark.parametrize("name,over", CASES)
def test_rope_keys_decode_matches_oracle(name, over):
    c = make_case(workload(name, **over))
    out, lse = _run(c)
    ref, ref_lse = _oracle(c)
    assert_close(out, ref, "bf16", f"rope-keys {name} {over} out")
    assert_close(lse, ref_lse, "bf16", f"rope-keys {name} {over} lse")


@pytest.mark.parametrize("lengths", [[1, 127, 128, 256], [0, 5, 0, 129]])
def test_rope_keys_tile_edges_and_empty(lengths):
    """Lengths on and around the 128-token tile edge, and empty sequences (out = 0,
    lse = -inf)."""
    c = make_case(workload("350m", B=4, T=256), lengths=lengths)
    out, lse = _run(c)
    ref, ref_lse = _oracle(c)
    for b, L in enumerate(lengths):
        if L == 0:
            assert np.all(out[b] == 0.0) and np.all(np.isneginf(lse[b]))
    keep = [b for b, L in enumerate(lengths) if L > 0]
    assert_close(out[keep], ref[keep], "bf16", f"rope-keys edges {lengths} out")
    assert_close(lse[keep], ref_lse[keep], "bf16", f"rope-keys edges {lengths} lse")


def test_rope_keys_full_size_350m():
    """The 350M-class layer (B = 8, T = 4096, H = 16, G = 4, d_h = d_n = 64), every output
    against the oracle."""
    c = make_case(workload("350m"))
    out, lse = _run(c)
    ref, ref_lse = _oracle(c)
    assert_close(out, ref, "bf16", "rope-keys 350m out")
    assert_close(lse, ref_lse, "bf16", "rope-keys 350m lse")


def test_rope_keys_full_size_long_sampled():
    """The long-context layer (B = 2, T = 131072, H = 32, G = 8, d_h = d_n = 128) in its
    launch configuration; the oracle (d_h d_n multiply-adds per token and head) on sampled
    (sequence, heads) pairs."""
    c = make_case(workload("long"))
    out, lse = _run(c)
    for b, heads in ((0, [0, 3]), (1, [29])):
        ref, ref_lse = _oracle_heads(c, b, heads)
        assert_close(out[b, heads], ref[0], "bf16", f"rope-keys long b={b} out")
        assert_close(lse[b, heads], ref_lse[0], "bf16", f"rope-keys long b={b} lse")


def test_rope_keys_refuses_unsupported_shapes():
    g = gva()
    assert g.gva_rope_keys_workspace_size(g.Dims(2, 16, 4, 64, 64, 16)) == 0   # d_r != 0
    assert g.gva_rope_keys_workspace_size(g.Dims(2, 16, 4, 64, 64, 0)) > 0
    c = make_case(workload("350m", T=200, B=2, d_h=32, d_n=32))
    dev = torch.device("cuda")
    w = c.w
    dims = g.Dims(w.B, w.H, w.G, w.d_h, w.d_n, 0)
    cache = g.Cache(_rows(c, dev), c.V.to(dev), None)
    out = torch.empty((w.B, w.H, w.d_h), device=dev)
    with pytest.raises(g.GvaError) as e:
        g.gva_rope_keys_decode_attention(dims, c.q_nope.to(dev), c.M.to(dev),
                                         c.seq_len.to(dev), cache, _table(c).to(dev), w.scale,
                                         out, None, g.rope_keys_workspace(dims, dev))
    assert e.value.status == g.GVA_ERR_UNSUPPORTED
