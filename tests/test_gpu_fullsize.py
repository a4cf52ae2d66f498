"""GPU parity at the workloads' full sizes, in the launch configuration the benchmark
times (default grid, automatic path: the tensor-core decode for these bf16 caches).

The whole batch is appended and decoded on the GPU; the fp64 oracle then recomputes a
sample of the sequences (the longest, the shortest and a seeded random one; all heads
of each) and the appended cache rows of the sample are compared bit for bit."""
import numpy as np
import pytest
import torch

from gva_inputs import make_case, workload
from helpers import Dev, assert_close, oracle_append, oracle_decode

pytestmark = pytest.mark.gpu

FULL = ["350m", "ragged", "long", "paged"]


def _sample(c, k=3):
    lens = c.seq_len.tolist()
    order = sorted(range(len(lens)), key=lambda b: lens[b])
    rng = np.random.default_rng(c.w.seed)
    pick = [order[-1], order[0], int(rng.integers(len(lens)))]
    return sorted(set(pick))[:k]


def _row(c, b, j):
    w = c.w
    if w.layout == "contiguous":
        return b * c.T_cap + j
    if w.layout == "ragged":
        return int(c.offsets[b]) + j
    return int(c.block_table[b, j // w.page_size]) * w.page_size + j % w.page_size


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_parity(name):
    c = make_case(workload(name))
    D = Dev(c)
    pos = (c.seq_len - 1).to(torch.int32)
    D.append(pos)
    out, lse = D.decode(path="auto")
    assert gva_status() == 0
    sample = _sample(c)
    V, K = oracle_append(c, pos, D.tab_h)
    ref, ref_lse = oracle_decode(c, V, K, sample=sample)
    assert_close(out[sample], ref, c.w.cache_dtype, f"{name} full-size out {sample}")
    assert_close(lse[sample], ref_lse, c.w.cache_dtype, f"{name} full-size lse {sample}")
    # the appended rows of the sample, bit for bit
    rows = torch.tensor([_row(c, b, int(pos[b])) for b in sample], device=D.V.device)
    gv = D.V.index_select(0, rows).cpu()
    gk = D.Kr.index_select(0, rows).cpu()
    ov = torch.from_numpy(V[[int(r) for r in rows.cpu()]].view(np.int16)).view(torch.bfloat16)
    ok = torch.from_numpy(K[[int(r) for r in rows.cpu()]].view(np.int16)).view(torch.bfloat16)
    assert torch.equal(gv.view(torch.int16), ov.view(torch.int16)), f"{name}: appended V differs"
    assert torch.equal(gk.view(torch.int16), ok.view(torch.int16)), f"{name}: appended K_rope differs"


def gva_status():
    from helpers import gva
    return gva().gva_get_device_status()
