"""GPU parity of the MLA-shaped comparator (gva_mla_decode_attention, through the C ABI)
against the oracle's explicit MLA decode (keys c_j W_uk_h with the shared positional key,
values c_j W_uv_h), on the same seeded inputs: bf16 cache, max-abs 2e-2 and relative L2
1e-3 on out and lse."""
import numpy as np
import pytest
import torch

import oracle
from gva_inputs import make_case, make_mla_case, workload
from helpers import assert_close, gva, oracle_rows, rope_tab

pytestmark = pytest.mark.gpu


def _run(c, m, sample=None):
    g = gva()
    w = c.w
    dev = torch.device("cuda")
    dims = g.MlaDims(w.B, w.H, m.d_c, w.d_n, w.d_r, w.d_h, g.GVA_BF16, g.GVA_BF16)
    offs = c.offsets.to(dev) if c.offsets is not None else None
    bt = c.block_table.to(dev) if c.block_table is not None else None
    rows = g.Rows(w.layout, c.num_rows, T_cap=c.T_cap, offsets=offs, block_table=bt,
                  page_size=w.page_size)
    cache = g.Cache(rows, m.C.to(dev), c.Kr.to(dev))
    tab = rope_tab(c).to(dev)
    out = torch.full((w.B, w.H, w.d_h), float("nan"), device=dev)
    lse = torch.full((w.B, w.H), float("nan"), device=dev)
    ws = g.mla_workspace(dims, dev)
    g.gva_mla_decode_attention(dims, c.q_nope.to(dev), c.q_rope.to(dev), m.W_uk.to(dev),
                               m.W_uv.to(dev), c.seq_len.to(dev), cache, tab, w.scale, out, lse,
                               ws)
    torch.cuda.synchronize()
    assert g.gva_get_device_status() == 0
    got = out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)
    idx = list(range(w.B)) if sample is None else list(sample)
    t = torch.tensor(idx)
    ref = oracle.mla_decode(c.q_nope[t], c.q_rope[t], m.W_uk, m.W_uv, c.seq_len[t],
                            oracle_rows(c, None if sample is None else idx), m.C, c.Kr,
                            w.scale, w.base)
    return got[0][idx], got[1][idx], ref


@pytest.mark.parametrize("name,over", [
    ("350m", dict(T=300, B=3)),                                      # d_c = 256, H = 16
    ("350m", dict(T=200, B=2, G=2)),                                 # d_c = 128
    ("350m", dict(T=97, B=3, H=8, G=2, d_r=24)),                     # H = 8, d_r with a k8 step
    ("350m", dict(T=150, B=2, H=32, G=4, d_r=0)),                    # H = 32, no positional slice
    ("ragged", dict(B=5, len_range=(1, 400))),
    ("paged", dict(B=4, len_range=(64, 500), H=16, G=2, d_h=128, d_n=128)),  # d_c = 256, d_h 128
])
def test_mla_decode_matches_oracle(name, over):
    c = make_case(workload(name, **over))
    m = make_mla_case(c)
    out, lse, (ref, ref_lse) = _run(c, m)
    assert_close(out, ref, "bf16", f"mla {name} {over} out")
    assert_close(lse, ref_lse, "bf16", f"mla {name} {over} lse")


def test_mla_decode_full_size_350m():
    """The bench's comparator workload (350M-class layer, B = 8, T = 4096, latent width
    256 = G d_h, the same cache bytes per token as GVA), in its launch configuration;
    the oracle's explicit MLA (16 K multiply-adds per token and head) on every sequence
    and head."""
    c = make_case(workload("350m"))
    m = make_mla_case(c)
    out, lse, (ref, ref_lse) = _run(c, m)
    assert_close(out, ref, "bf16", "mla 350m out")
    assert_close(lse, ref_lse, "bf16", "mla 350m lse")


def test_mla_refuses_unsupported_shapes():
    g = gva()
    assert g.gva_mla_workspace_size(g.MlaDims(2, 16, 192, 64, 16, 64)) == 0   # d_c
    assert g.gva_mla_workspace_size(g.MlaDims(2, 36, 256, 64, 16, 64)) == 0   # H / 4 > 8
    assert g.gva_mla_workspace_size(g.MlaDims(2, 6, 256, 64, 16, 64)) == 0    # H % 4
    assert g.gva_mla_workspace_size(g.MlaDims(2, 16, 256, 64, 16, 64)) > 0
