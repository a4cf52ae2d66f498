"""gva_decode_attention_static: the decode for callers that cannot allocate device
memory (graph capture, allocator-less plugins, latency-critical loops).  Its scratch
is the library's fixed device array; its results must match the workspace-taking
entry point.  Collected last so that a failure here comes after every other test."""
import ctypes

import numpy as np
import pytest
import torch

from gva_inputs import make_case, workload
from helpers import Dev, TOL, errors, gva

pytestmark = pytest.mark.gpu


def _static_call(D, out, lse):
    """Through the C ABI directly (the binding adds only pointer marshalling)."""
    g = gva()
    w = D.c.w
    d = D.dims.c()
    cc = D.cache.c()
    st = g._lib.gva_decode_attention_static(
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), ctypes.byref(d),
        ctypes.c_void_p(D.q_nope.data_ptr()), ctypes.c_void_p(D.q_rope.data_ptr()),
        ctypes.c_void_p(D.M.data_ptr()), ctypes.c_void_p(D.seq_len.data_ptr()),
        ctypes.byref(cc), ctypes.c_void_p(D.tab.data_ptr()), int(D.tab.shape[0]),
        ctypes.c_float(w.scale), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()))
    assert st == g.GVA_OK, g.gva_status_string(st)


@pytest.mark.parametrize("name,over", [("350m", dict(T=700, B=3)),
                                       ("paged", dict(B=6, len_range=(100, 1500)))])
def test_static_scratch_matches_workspace_entry(name, over):
    c = make_case(workload(name, **over))
    D = Dev(c)
    w = c.w
    ref_out, ref_lse = D.decode()              # existing entry point, caller workspace
    for _ in range(2):                        # two calls in a row share the array
        out = torch.full((w.B, w.H, w.d_h), float("nan"), device="cuda")
        lse = torch.full((w.B, w.H), float("nan"), device="cuda")
        _static_call(D, out, lse)
        torch.cuda.synchronize()
        assert gva().gva_get_device_status() == 0
        o = out.cpu().numpy().astype(np.float64)
        l = lse.cpu().numpy().astype(np.float64)
        for got, ref in ((o, ref_out), (l, ref_lse)):
            max_abs, rel = errors(got, ref)
            assert max_abs <= TOL["bf16"]["max_abs"] and rel <= TOL["bf16"]["rel_l2"]


def test_static_scratch_rejects_oversize():
    g = gva()
    big = g.Dims(4096, 32, 8, 128, 128, 16)   # valid shape, workspace beyond the fixed array
    assert g.gva_decode_workspace_size(big) > (24 << 20)
    fake = torch.empty(16, device="cuda")
    rows = g.Rows("contiguous", 4096, T_cap=1)
    cache = g.Cache(rows, fake, fake)
    with pytest.raises(g.GvaError) as e:
        g.gva_decode_attention_static(big, fake, fake, fake, fake.int(), cache, fake, 0.1,
                                      fake, None)
    assert e.value.status == g.GVA_ERR_WORKSPACE
