"""gva_decode_attention_static: the decode for callers that cannot allocate device
memory where they decode (plugins handed no allocator, engines whose memory is planned
once at start-up, loops that forbid allocator calls).  Its scratch is the library's
fixed device array.  On two calls in a row it must give the workspace-taking entry
point's results (the same kernels on the same plan: bit for bit, so within any
tolerance) and match the fp64 oracle within the bf16 tolerance.  Collected last so
that a failure here comes after every other test."""
import ctypes

import numpy as np
import pytest
import torch

from gva_inputs import make_case, workload
from helpers import Dev, assert_close, gva, oracle_decode

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
    o_ref, l_ref = oracle_decode(c)
    for _ in range(2):                         # two calls in a row share the array
        out = torch.full((w.B, w.H, w.d_h), float("nan"), device="cuda")
        lse = torch.full((w.B, w.H), float("nan"), device="cuda")
        _static_call(D, out, lse)
        torch.cuda.synchronize()
        assert gva().gva_get_device_status() == 0
        o = out.cpu().numpy().astype(np.float64)
        l = lse.cpu().numpy().astype(np.float64)
        assert np.array_equal(o, ref_out), "static out differs from the workspace entry's"
        assert np.array_equal(l, ref_lse), "static lse differs from the workspace entry's"
        assert_close(o, o_ref, "bf16", f"{name} static out vs oracle")
        assert_close(l, l_ref, "bf16", f"{name} static lse vs oracle")


def test_static_scratch_rejects_oversize():
    """Checked by the library before anything touches memory, so dummy pointers do."""
    g = gva()
    big = g.Dims(4096, 32, 8, 128, 128, 16)   # valid shape, workspace beyond the fixed array
    assert g.gva_decode_workspace_size(big) > (24 << 20)
    fake = torch.empty(16, device="cuda")
    p = ctypes.c_void_p(fake.data_ptr())
    d = big.c()
    cc = g.Cache(g.Rows("contiguous", 4096, T_cap=1), fake, fake).c()
    st = g._lib.gva_decode_attention_static(
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), ctypes.byref(d), p, p, p, p,
        ctypes.byref(cc), p, 1, ctypes.c_float(0.1), p, None)
    assert st == g.GVA_ERR_WORKSPACE


def test_static_scratch_in_a_graph():
    """The reason the entry exists: a warm call, then the static call recorded into a CUDA
    graph and replayed twice, with new query contents written in place before the second
    replay; each replay equals the workspace entry on the same contents bit for bit."""
    c = make_case(workload("350m", T=500, B=4))
    D = Dev(c)
    w = c.w
    out = torch.full((w.B, w.H, w.d_h), float("nan"), device="cuda")
    lse = torch.full((w.B, w.H), float("nan"), device="cuda")
    _static_call(D, out, lse)                  # the one-time set-up, outside the capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            _static_call(D, out, lse)
    for it in range(2):
        if it == 1:
            D.q_nope.mul_(-0.5)                # new contents, same storage
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert gva().gva_get_device_status() == 0
        ref_out, ref_lse = D.decode()
        assert np.array_equal(out.cpu().numpy().astype(np.float64), ref_out), f"replay {it}"
        assert np.array_equal(lse.cpu().numpy().astype(np.float64), ref_lse), f"replay {it}"
    q = c.q_nope.clone()
    c.q_nope.mul_(-0.5)                        # the oracle on the second replay's queries
    o_ref, l_ref = oracle_decode(c)
    c.q_nope.copy_(q)
    assert_close(out.cpu().numpy().astype(np.float64), o_ref, "bf16", "graph replay out vs oracle")
    assert_close(lse.cpu().numpy().astype(np.float64), l_ref, "bf16", "graph replay lse vs oracle")
