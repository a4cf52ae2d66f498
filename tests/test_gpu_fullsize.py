"""GPU parity at the workloads' full sizes, in the launch configuration the benchmark
times (default grid, automatic path: the tensor-core decode for these bf16 caches).

The whole batch is appended and decoded on the GPU; the fp64 oracle then recomputes
every sequence and every head (out and lse), and every appended cache row is compared
bit for bit.  The 350M-class layer is also decoded at grid sizes whose split-K shares
cut through sequences at different places (a share that spans the end of one sequence
and the start of the next is the path where partials from two sequences meet)."""
import numpy as np
import pytest
import torch

import oracle
from gva_inputs import make_case, make_gqa_keys, make_gqa_query, workload
from helpers import Dev, assert_close, gva, oracle_append, oracle_decode, oracle_rows

pytestmark = pytest.mark.gpu

FULL = ["350m", "ragged", "long", "paged"]


def _row(c, b, j):
    w = c.w
    if w.layout == "contiguous":
        return b * c.T_cap + j
    if w.layout == "ragged":
        return int(c.offsets[b]) + j
    return int(c.block_table[b, j // w.page_size]) * w.page_size + j % w.page_size


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("via", ["calls", "step"])
@pytest.mark.parametrize("name", FULL)
def test_full_size_parity(name, via):
    """`calls`: gva_append_cache then gva_decode_attention.  `step`: one gva_decode_step
    layer, the call the benchmark's step makes (the append inside the absorption's grid)."""
    c = make_case(workload(name))
    D = Dev(c)
    pos = (c.seq_len - 1).to(torch.int32)
    if via == "calls":
        D.append(pos)
        out, lse = D.decode(path="auto")
    else:
        w = c.w
        o = torch.full((w.B, w.H, w.d_h), float("nan"), device="cuda")
        l = torch.full((w.B, w.H), float("nan"), device="cuda")
        layer = dict(v_new=D.v_new, k_rope_new=D.k_new, q_nope=D.q_nope, q_rope=D.q_rope,
                     M=D.M, cache=D.cache, out=o, lse=l)
        gva().gva_decode_step(D.dims, [layer], pos.cuda(), D.seq_len, D.tab, w.scale, D.ws)
        torch.cuda.synchronize()
        out = o.cpu().numpy().astype(np.float64)
        lse = l.cpu().numpy().astype(np.float64)
    assert gva().gva_get_device_status() == 0
    V, K = oracle_append(c, pos, D.tab_h)
    ref, ref_lse = oracle_decode(c, V, K)           # every sequence, every head
    assert_close(out, ref, c.w.cache_dtype, f"{name} full-size out")
    assert_close(lse, ref_lse, c.w.cache_dtype, f"{name} full-size lse")
    # every appended row, bit for bit
    idx = [_row(c, b, int(pos[b])) for b in range(c.w.B)]
    rows = torch.tensor(idx, device=D.V.device)
    gv = D.V.index_select(0, rows).cpu()
    gk = D.Kr.index_select(0, rows).cpu()
    ov = torch.from_numpy(V[idx].view(np.int16)).view(torch.bfloat16)
    ok = torch.from_numpy(K[idx].view(np.int16)).view(torch.bfloat16)
    assert torch.equal(_bits(gv), _bits(ov)), f"{name}: appended V differs"
    assert torch.equal(_bits(gk), _bits(ok)), f"{name}: appended K_rope differs"


@pytest.mark.parametrize("num_ctas", [37, 100, 148, 150, 300, 1000])
def test_full_size_350m_share_boundaries(num_ctas):
    """2048 slabs over 8 sequences of 256 slabs: none of these grid sizes puts every
    share boundary on a sequence boundary."""
    c = make_case(workload("350m"))
    D = Dev(c)
    out, lse = D.decode(path="auto", num_ctas=num_ctas)
    assert gva().gva_get_device_status() == 0
    ref, ref_lse = oracle_decode(c)
    assert_close(out, ref, "bf16", f"350m n_ctas={num_ctas} out")
    assert_close(lse, ref_lse, "bf16", f"350m n_ctas={num_ctas} lse")


@pytest.mark.parametrize("name", ["ragged", "350m"])
def test_full_size_gqa_comparator_repeated(name):
    """The GQA comparator at full size in the bench's launch configuration, five calls in a
    row, every sequence and head against the oracle each time.  Both batches give each CTA
    more slabs than its ring has stages (the ragged batch about five rounds), so the
    consumer warps wait on stages whose previous round another warp of the group took."""
    c = make_case(workload(name))
    D = Dev(c)
    g = gva()
    K = make_gqa_keys(c)
    q = make_gqa_query(c)
    kv = g.KVCache(D.rows, K.cuda(), D.V)
    w = c.w
    scale = 1.0 / np.sqrt(w.d_h)
    ref, ref_lse = oracle.gqa_decode(q, c.seq_len, oracle_rows(c), K, c.V, scale, w.G)
    qd = q.cuda()
    for it in range(5):
        out = torch.full((w.B, w.H, w.d_h), float("nan"), device="cuda")
        lse = torch.full((w.B, w.H), float("nan"), device="cuda")
        g.gva_gqa_decode_attention(D.dims, qd, D.seq_len, kv, scale, out, lse, D.ws, path="auto")
        torch.cuda.synchronize()
        assert g.gva_get_device_status() == 0
        assert_close(out.cpu().numpy(), ref, "bf16", f"gqa {name} call {it} out")
        assert_close(lse.cpu().numpy(), ref_lse, "bf16", f"gqa {name} call {it} lse")
