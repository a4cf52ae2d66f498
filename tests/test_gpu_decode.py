"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same
seeded inputs.  Decode within the workloads' tolerances (bf16 cache: max-abs 2e-2 and
relative L2 1e-3; fp32 cache: 1e-5 for both); append and paged gather bit-exact."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gva_inputs import make_case, make_gqa_keys, make_gqa_query, workload
from helpers import Dev, assert_close, gva, oracle_append, oracle_decode, oracle_rows

pytestmark = pytest.mark.gpu


def _mma_ok(c):
    """The tensor-core path's support matrix (include/gva.h: bf16 cache, d_h 64 or 128,
    at most 8 value groups)."""
    w = c.w
    return w.cache_dtype == "bf16" and w.d_h in (64, 128) and w.G <= 8


def paths_for(c):
    return ["simt"] + (["mma"] if _mma_ok(c) else [])


# small variants of the five workloads: several slabs and CTAs, ragged tails
SMALL = {
    "tiny": {},
    "350m": dict(T=300, B=3),
    "ragged": dict(B=7, len_range=(1, 700)),
    "long": dict(B=2, T=3001),
    "paged": dict(B=5, len_range=(64, 900)),
}


def _step(c, path, num_ctas=0):
    """append at t = L - 1 then decode over 0..t, on both sides"""
    D = Dev(c)
    pos = (c.seq_len - 1).to(torch.int32)
    D.append(pos)
    out, lse = D.decode(path=path, num_ctas=num_ctas)
    assert gva().gva_get_device_status() == 0
    V, K = oracle_append(c, pos, D.tab_h)
    ref, ref_lse = oracle_decode(c, V, K)
    return out, lse, ref, ref_lse, D


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("path", ["simt", "mma", "auto"])
def test_step_small_workloads(name, path):
    c = make_case(workload(name, **SMALL[name]))
    if path == "mma" and not _mma_ok(c):
        pytest.skip("tensor-core path needs a bf16 cache")
    out, lse, ref, ref_lse, _ = _step(c, path)
    assert_close(out, ref, c.w.cache_dtype, f"{name}/{path} out")
    assert_close(lse, ref_lse, c.w.cache_dtype, f"{name}/{path} lse")


@pytest.mark.parametrize("num_ctas", [1, 2, 7, 148, 1000])
def test_split_counts(num_ctas):
    c = make_case(workload("350m", T=257, B=3))
    for path in paths_for(c):
        D = Dev(c)
        out, lse = D.decode(path=path, num_ctas=num_ctas)
        ref, ref_lse = oracle_decode(c)
        assert_close(out, ref, "bf16", f"{path} n={num_ctas}")
        assert_close(lse, ref_lse, "bf16", f"{path} n={num_ctas} lse")


@pytest.mark.parametrize("lengths", [[1, 1, 1], [15, 16, 17], [0, 33, 0], [0, 0, 0],
                                     [100, 1, 31]])
def test_edge_lengths(lengths):
    c = make_case(workload("350m", T=100, B=3), lengths=lengths)
    for path in paths_for(c):
        D = Dev(c)
        out, lse = D.decode(path=path)
        ref, ref_lse = oracle_decode(c)
        assert_close(out, ref, "bf16", f"{path} {lengths}")
        assert_close(lse, ref_lse, "bf16", f"{path} {lengths} lse")
        for b, L in enumerate(lengths):
            if L == 0:
                assert np.all(out[b] == 0) and np.all(np.isneginf(lse[b]))
            if L == 1:   # a single cached token returns its value (rounding only)
                v = oracle.f64(c.V)[b * c.T_cap, :, :]
                r = c.w.H // c.w.G
                for h in range(c.w.H):
                    assert np.max(np.abs(out[b, h] - v[h // r])) <= 1e-6


@pytest.mark.parametrize("H,G,d_h,d_n,d_r", [
    (8, 8, 64, 64, 16), (8, 4, 64, 32, 8), (8, 2, 128, 128, 24), (8, 1, 64, 64, 32),
    (16, 2, 32, 32, 0), (4, 4, 128, 64, 16), (32, 4, 64, 128, 16), (3, 3, 64, 64, 16),
])
@pytest.mark.parametrize("cache", ["bf16", "f32"])
def test_shapes(H, G, d_h, d_n, d_r, cache):
    w = workload("350m", B=2, T=133, H=H, G=G, d_h=d_h, d_n=d_n, d_r=d_r, cache_dtype=cache,
                 q_dtype="f32" if cache == "f32" else "bf16")
    c = make_case(w)
    for path in paths_for(c):
        out, lse, ref, ref_lse, _ = _step(c, path)
        assert_close(out, ref, cache, f"{path} out")
        assert_close(lse, ref_lse, cache, f"{path} lse")


def test_garbage_beyond_length_is_ignored():
    """Slots past a sequence's end may hold anything, NaN included."""
    c = make_case(workload("350m", T=160, B=3), lengths=[150, 37, 1])
    ref, ref_lse = oracle_decode(c)
    V = c.V.clone()
    K = c.Kr.clone()
    for b, L in enumerate(c.seq_len.tolist()):
        V[b * c.T_cap + L:(b + 1) * c.T_cap] = float("nan")
        K[b * c.T_cap + L:(b + 1) * c.T_cap] = float("inf")
    c.V, c.Kr = V, K
    for path in paths_for(c):
        out, lse = Dev(c).decode(path=path)
        assert_close(out, ref, "bf16", path)
        assert_close(lse, ref_lse, "bf16", path)


def test_paged_nan_slack():
    c = make_case(workload("paged", B=4, len_range=(70, 300), extra_slots=40))
    ref, ref_lse = oracle_decode(c)
    V = c.V.clone()
    bt = c.block_table
    for b, L in enumerate(c.seq_len.tolist()):
        for j in range(L, (L + 40 + 63) // 64 * 64):
            if j // 64 < bt.shape[1] and bt[b, j // 64] >= 0:
                V[int(bt[b, j // 64]) * 64 + j % 64] = float("nan")
    c.V = V
    for path in paths_for(c):
        out, lse = Dev(c).decode(path=path)
        assert_close(out, ref, "bf16", path)


# --------------------------------------------------------------------------- #
# append: bit-exact against the oracle's fp32-decided rounding
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("layout", ["contiguous", "ragged", "paged"])
@pytest.mark.parametrize("cache", ["bf16", "f32"])
@pytest.mark.parametrize("mode", ["overwrite", "extend"])
def test_append_bit_exact(layout, cache, mode):
    name = {"contiguous": "350m", "ragged": "ragged", "paged": "paged"}[layout]
    over = dict(B=6, cache_dtype=cache, extra_slots=3 if mode == "extend" else 0)
    if layout == "contiguous":
        over["T"] = 200
    else:
        over["len_range"] = (1, 500)
    c = make_case(workload(name, **over))
    D = Dev(c)
    if mode == "overwrite":
        pos = (c.seq_len - 1).to(torch.int32)
        D.append(pos)
        new_len = c.seq_len
    else:
        pos = c.seq_len.clone()
        lens = D.seq_len.clone()
        D.append(lens, seq_len_out=lens)   # pos and seq_len_out alias
        new_len = lens.cpu()
        assert torch.equal(new_len, c.seq_len + 1)
    torch.cuda.synchronize()
    assert gva().gva_get_device_status() == 0
    V, K = oracle_append(c, pos, D.tab_h)
    gv = oracle._np(D.V.cpu())
    gk = oracle._np(D.Kr.cpu())
    assert np.array_equal(gv.view(np.uint8), V.view(np.uint8))
    assert np.array_equal(gk.view(np.uint8), K.view(np.uint8))
    # and the decode over the extended cache matches
    if mode == "extend":
        out, lse = D.decode(seq_len=lens)
        ref, ref_lse = oracle_decode(c, V, K, seq_len=new_len)
        assert_close(out, ref, cache, "decode after extend")


@pytest.mark.parametrize("over", [
    dict(B=5),
    # several 8-sequence groups per CTA and a partial last chunk (300 = 9 x 32 + 12)
    dict(B=300, H=16, G=4, d_h=64, d_n=64, d_r=16),
    # d_n = 256 (chunks of 32), fp32 queries: the per-CTA sequence cap of the staging
    dict(B=400, H=8, G=2, d_h=32, d_n=256, d_r=8, cache_dtype="f32", q_dtype="f32"),
    dict(B=70, H=4, G=2, d_h=128, d_n=256, d_r=32),
    # chunk sizes that are not a multiple of 4 (padded chunks, per-element scatter)
    dict(B=33, H=3, G=3, d_h=32, d_n=24, d_r=8, cache_dtype="f32", q_dtype="f32"),
    dict(B=50, H=6, G=2, d_h=64, d_n=40, d_r=24),
    dict(B=9, H=2, G=1, d_h=32, d_n=8, d_r=16),
], ids=lambda o: "-".join(f"{k}{v}" for k, v in o.items()))
def test_absorb_matches_oracle(over):
    c = make_case(workload("350m", T=50, **over))
    D = Dev(c)
    w = c.w
    qt = torch.empty((w.B, w.H, w.d_h), device="cuda")
    qh = torch.empty((w.B, w.H, w.d_r), device="cuda")
    gva().gva_absorb_query(D.dims, D.q_nope, D.q_rope, D.M, D.seq_len, D.tab, w.scale, qt, qh)
    torch.cuda.synchronize()
    rt, rh = oracle.absorb(c.q_nope, c.q_rope, c.M, c.seq_len, w.scale, w.base)
    for got, ref in ((qt, rt), (qh, rh)):
        g = got.cpu().numpy().astype(np.float64)
        assert np.max(np.abs(g - ref)) <= 2e-6 * max(1.0, np.max(np.abs(ref)))


# --------------------------------------------------------------------------- #
# device-side checks: no trap, a status code, the other sequences still right
# --------------------------------------------------------------------------- #
def test_length_beyond_capacity_is_reported():
    c = make_case(workload("350m", T=64, B=3), lengths=[64, 20, 10])
    D = Dev(c)
    bad = torch.tensor([64, 9999, 10], dtype=torch.int32, device="cuda")
    out, lse = D.decode(seq_len=bad)
    assert gva().gva_get_device_status() == gva().GVA_DEV_BAD_LENGTH
    ref, ref_lse = oracle_decode(c)
    for b in (0, 2):
        assert_close(out[b], ref[b], "bf16", f"b={b}")
    assert np.all(out[1] == 0) and np.isneginf(lse[1]).all()
    assert gva().gva_get_device_status() == 0


def test_bad_page_is_reported():
    c = make_case(workload("paged", B=3, len_range=(100, 200)))
    D = Dev(c)
    D.block_table[1, 0] = 10 ** 6
    D.decode()
    assert gva().gva_get_device_status() == gva().GVA_DEV_BAD_PAGE


def test_append_bad_position_is_reported():
    c = make_case(workload("350m", T=32, B=2))
    D = Dev(c)
    D.append(torch.tensor([5, 32], dtype=torch.int32))
    torch.cuda.synchronize()
    assert gva().gva_get_device_status() == gva().GVA_DEV_BAD_POSITION


def test_host_argument_errors():
    c = make_case(workload("350m", T=32, B=2))
    D = Dev(c)
    g = gva()
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    out = torch.empty((2, 16, 64), device="cuda")
    with pytest.raises(g.GvaError) as e:
        g.gva_decode_attention(D.dims, D.q_nope, D.q_rope, D.M, D.seq_len, D.cache, D.tab,
                               0.1, out, None, small)
    assert e.value.status == g.GVA_ERR_WORKSPACE
    bad = g.Dims(2, 16, 5, 64, 64, 16)
    with pytest.raises(g.GvaError) as e:
        g.gva_decode_attention(bad, D.q_nope, D.q_rope, D.M, D.seq_len, D.cache, D.tab, 0.1,
                               out, None, D.ws)
    assert e.value.status == g.GVA_ERR_ARG
    f32 = workload("tiny")
    cf = make_case(f32)
    Df = Dev(cf)
    with pytest.raises(g.GvaError) as e:
        Df.decode(path="mma")
    assert e.value.status == g.GVA_ERR_UNSUPPORTED


def test_binding_refuses_undersized_tensors():
    """The binding checks every tensor against what the C call touches and raises
    GVA_ERR_ARG before any launch (the C ABI sees plain pointers, not sizes)."""
    c = make_case(workload("350m", T=32, B=2))
    D = Dev(c)
    g = gva()
    w = c.w
    out = torch.empty((w.B, w.H, w.d_h), device="cuda")
    cases = {
        "out": dict(out=out[:, :, :8].contiguous()),
        "q_nope": dict(q_nope=D.q_nope[:1].contiguous()),
        "M": dict(M=D.M[:3].contiguous()),
        "seq_len": dict(seq_len=D.seq_len[:1].contiguous()),
        "V": dict(cache=g.Cache(D.rows, D.V[:5].contiguous(), D.Kr)),
        "K_rope dtype": dict(cache=g.Cache(D.rows, D.V, D.Kr.float())),
    }
    for what, over in cases.items():
        a = dict(q_nope=D.q_nope, M=D.M, seq_len=D.seq_len, cache=D.cache, out=out)
        a.update(over)
        with pytest.raises(g.GvaError) as e:
            g.gva_decode_attention(D.dims, a["q_nope"], D.q_rope, a["M"], a["seq_len"],
                                   a["cache"], D.tab, w.scale, a["out"], None, D.ws)
        assert e.value.status == g.GVA_ERR_ARG, what
    with pytest.raises(g.GvaError) as e:
        g.gva_append_cache(D.dims, D.v_new[:1].contiguous(), D.k_new,
                           torch.zeros(2, dtype=torch.int32, device="cuda"), None, D.cache, D.tab)
    assert e.value.status == g.GVA_ERR_ARG
    torch.cuda.synchronize()
    assert g.gva_get_device_status() == 0


# --------------------------------------------------------------------------- #
# GQA comparator
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("name", ["350m", "ragged", "paged"])
def test_gqa_comparator(name):
    c = make_case(workload(name, **SMALL[name]))
    K = make_gqa_keys(c)
    q = make_gqa_query(c)
    D = Dev(c)
    g = gva()
    kv = g.KVCache(D.rows, K.cuda(), D.V)
    w = c.w
    scale = 1.0 / np.sqrt(w.d_h)
    ref, ref_lse = oracle.gqa_decode(q, c.seq_len, oracle_rows(c), K, c.V, scale, w.G)
    for path in paths_for(c):
        out = torch.empty((w.B, w.H, w.d_h), device="cuda")
        lse = torch.empty((w.B, w.H), device="cuda")
        g.gva_gqa_decode_attention(D.dims, q.cuda(), D.seq_len, kv, scale, out, lse, D.ws,
                                   path=path)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), ref, "bf16", f"gqa {path}")
        assert_close(lse.cpu().numpy(), ref_lse, "bf16", f"gqa {path} lse")


# --------------------------------------------------------------------------- #
# CUDA graphs: the calls can be captured (torch's default global capture mode)
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("path", ["simt", "mma"])
def test_graph_capture_and_replay(path):
    c = make_case(workload("350m", T=200, B=3))
    D = Dev(c)
    w = c.w
    g = gva()
    pos = (c.seq_len - 1).to(torch.int32).cuda()
    out = torch.empty((w.B, w.H, w.d_h), device="cuda")
    lse = torch.empty((w.B, w.H), device="cuda")

    def step():
        g.gva_append_cache(D.dims, D.v_new, D.k_new, pos, None, D.cache, D.tab)
        g.gva_decode_attention(D.dims, D.q_nope, D.q_rope, D.M, D.seq_len, D.cache, D.tab,
                               w.scale, out, lse, D.ws, path=path)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step()                      # first call eagerly (per-device set-up)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            step()
            step()                  # second call follows a kernel node (programmatic edge)
    out.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert gva().gva_get_device_status() == 0
    V, K = oracle_append(c, pos.cpu(), D.tab_h)
    ref, ref_lse = oracle_decode(c, V, K)
    assert_close(out.cpu().numpy(), ref, "bf16", f"graph {path}")
    assert_close(lse.cpu().numpy(), ref_lse, "bf16", f"graph {path} lse")


def test_read_probe_reads_every_word():
    """The bandwidth probe folds every 32-bit word of its buffer: its XOR matches the
    host's (odd size: the unrolled part and the tail both run)."""
    g = gva()
    n = 37 * 1024 * 1024 // 4 + 12   # words (a multiple of 4 words: 16-byte vectors)
    gen = torch.Generator().manual_seed(7)
    host = torch.randint(-2**31, 2**31 - 1, (n,), generator=gen, dtype=torch.int64).to(torch.int32)
    buf = host.cuda()
    sink = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    g.gva_read_probe(buf, sink)
    torch.cuda.synchronize()
    ref = int(np.bitwise_xor.reduce(host.numpy().view(np.uint32)))
    assert int(sink.cpu().numpy().view(np.uint32)[0]) == ref


def test_prepared_calls_match_the_oracle():
    """Prepared append + decode calls (arguments marshalled once, called twice) give the
    oracle's result, like the plain entry points."""
    c = make_case(workload("350m", T=200, B=3))
    D = Dev(c)
    w = c.w
    g = gva()
    pos = (c.seq_len - 1).to(torch.int32).cuda()
    out = torch.empty((w.B, w.H, w.d_h), device="cuda")
    lse = torch.empty((w.B, w.H), device="cuda")
    app = g.prepare_append_cache(D.dims, D.v_new, D.k_new, pos, None, D.cache, D.tab)
    dec = g.prepare_decode_attention(D.dims, D.q_nope, D.q_rope, D.M, D.seq_len, D.cache, D.tab,
                                     w.scale, out, lse, D.ws)
    for _ in range(2):
        out.zero_()
        app()
        dec()
    torch.cuda.synchronize()
    assert g.gva_get_device_status() == 0
    V, K = oracle_append(c, pos.cpu(), D.tab_h)
    ref, ref_lse = oracle_decode(c, V, K)
    assert_close(out.cpu().numpy(), ref, "bf16", "prepared")
    assert_close(lse.cpu().numpy(), ref_lse, "bf16", "prepared lse")


# --------------------------------------------------------------------------- #
# query RMSNorm variant (normalise each head's content query, then absorb)
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("name", ["350m", "ragged", "tiny", "paged"])
@pytest.mark.parametrize("with_gain", [False, True])
def test_query_rmsnorm_decode(name, with_gain):
    c = make_case(workload(name, **SMALL[name]))
    w = c.w
    eps = 1e-5
    gen = torch.Generator().manual_seed(99)
    gain = torch.rand(w.d_n, generator=gen) * 2 + 0.25 if with_gain else None
    qn = oracle.query_rmsnorm(c.q_nope, None if gain is None else gain.numpy(), eps)
    for path in paths_for(c):
        D = Dev(c)
        out = torch.empty((w.B, w.H, w.d_h), device="cuda")
        lse = torch.empty((w.B, w.H), device="cuda")
        gva().gva_decode_attention(D.dims, D.q_nope, D.q_rope, D.M, D.seq_len, D.cache, D.tab,
                                   w.scale, out, lse, D.ws, path=path,
                                   q_norm=(None if gain is None else gain.cuda(), eps))
        torch.cuda.synchronize()
        assert gva().gva_get_device_status() == 0
        ref, ref_lse = oracle.gva_decode(qn, c.q_rope, c.M, c.seq_len, oracle_rows(c),
                                         oracle._np(c.V), oracle._np(c.Kr), w.scale, w.base, w.G)
        assert_close(out.cpu().numpy(), ref, w.cache_dtype, f"{name}/{path} q-norm out")
        assert_close(lse.cpu().numpy(), ref_lse, w.cache_dtype, f"{name}/{path} q-norm lse")


def test_query_rmsnorm_absorb():
    c = make_case(workload("350m", T=50, B=37, d_n=128))
    D = Dev(c)
    w = c.w
    gain = torch.linspace(0.5, 1.5, w.d_n)
    qt = torch.empty((w.B, w.H, w.d_h), device="cuda")
    qh = torch.empty((w.B, w.H, w.d_r), device="cuda")
    gva().gva_absorb_query(D.dims, D.q_nope, D.q_rope, D.M, D.seq_len, D.tab, w.scale, qt, qh,
                           q_norm=(gain.cuda(), 1e-6))
    torch.cuda.synchronize()
    qn = oracle.query_rmsnorm(c.q_nope, gain.numpy(), 1e-6)
    rt, rh = oracle.absorb(qn, c.q_rope, c.M, c.seq_len, w.scale, w.base)
    for got, ref in ((qt, rt), (qh, rh)):
        g = got.cpu().numpy().astype(np.float64)
        assert np.max(np.abs(g - ref)) <= 2e-6 * max(1.0, np.max(np.abs(ref)))


def test_gqa_refuses_query_rmsnorm():
    c = make_case(workload("350m", **SMALL["350m"]))
    D = Dev(c)
    g = gva()
    kv = g.KVCache(D.rows, make_gqa_keys(c).cuda(), D.V)
    w = c.w
    out = torch.empty((w.B, w.H, w.d_h), device="cuda")
    o = g.gva_decode_opts(0, 0, g.GVA_FLAG_QUERY_RMSNORM, 1e-6, None)
    st = g._lib.gva_gqa_decode_attention(None, ctypes.byref(D.dims.c()), ctypes.c_void_p(make_gqa_query(c).cuda().data_ptr()),
                                         ctypes.c_void_p(D.seq_len.data_ptr()), ctypes.byref(kv.c()),
                                         ctypes.c_float(0.125), ctypes.c_void_p(out.data_ptr()), None,
                                         ctypes.c_void_p(D.ws.data_ptr()),
                                         ctypes.c_size_t(D.ws.numel()), ctypes.byref(o))
    assert st == g.GVA_ERR_UNSUPPORTED


@pytest.mark.parametrize("per_sm,long_len,shape", [
    (2, (2600, 3201), {}), (3, (4000, 4601), {}),
    (3, (4000, 4601), dict(H=8, G=2)),   # GQA's smaller stages take three CTAs per SM too
])
def test_several_ctas_per_sm_ragged(per_sm, long_len, shape):
    """Ragged caches long enough for the two- and three-CTAs-per-SM plans (the row capacity
    gives every CTA of that many times the SM count at least 16 slabs; below the next
    plan's threshold for two): half the sequences of 1-40 tokens, half long, so that shares
    cross many short sequences and partial slabs.  GVA and the GQA comparator (whose larger
    stages take the two-CTA plan in both cases) against the oracle, every sequence and
    head.  With G = 2 the GQA comparator's stages are small enough for three per SM."""
    g = gva()
    gen = np.random.default_rng(11)
    B = 64
    lengths = [int(x) for x in gen.integers(1, 41, B // 2)] + \
              [int(x) for x in gen.integers(long_len[0], long_len[1], B // 2)]
    gen.shuffle(lengths)
    c = make_case(workload("ragged", B=B, **shape), lengths=lengths)
    slabs, sms = c.num_rows // 16, g.gva_num_sms()
    assert slabs >= per_sm * sms * 16 and (per_sm == 3 or slabs < 3 * sms * 16)
    D = Dev(c)
    out, lse = D.decode(path="auto")
    assert g.gva_get_device_status() == 0
    ref, ref_lse = oracle_decode(c)
    assert_close(out, ref, "bf16", f"{per_sm} CTAs per SM out")
    assert_close(lse, ref_lse, "bf16", f"{per_sm} CTAs per SM lse")
    w = c.w
    K = make_gqa_keys(c)
    q = make_gqa_query(c)
    kv = g.KVCache(D.rows, K.cuda(), D.V)
    scale = 1.0 / np.sqrt(w.d_h)
    gref, gref_lse = oracle.gqa_decode(q, c.seq_len, oracle_rows(c), K, c.V, scale, w.G)
    gout = torch.full((w.B, w.H, w.d_h), float("nan"), device="cuda")
    glse = torch.full((w.B, w.H), float("nan"), device="cuda")
    g.gva_gqa_decode_attention(D.dims, q.cuda(), D.seq_len, kv, scale, gout, glse, D.ws, path="auto")
    torch.cuda.synchronize()
    assert g.gva_get_device_status() == 0
    assert_close(gout.cpu().numpy(), gref, "bf16", f"{per_sm} CTAs per SM gqa out")
    assert_close(glse.cpu().numpy(), gref_lse, "bf16", f"{per_sm} CTAs per SM gqa lse")


def test_largest_batch():
    """B = 4096, the largest batch the in-kernel prefix handles (its lengths and slab
    offsets take 32 KB of shared memory, shrinking the ring): every path, mixed lengths
    0..33 over a capacity of 40."""
    B = 4096
    gen = np.random.default_rng(5)
    lengths = [int(x) for x in gen.integers(0, 34, B)]
    c = make_case(workload("350m", B=B, T=40, H=4, G=2, d_h=64, d_n=64, d_r=16), lengths=lengths)
    ref, ref_lse = oracle_decode(c)
    for path in paths_for(c):
        D = Dev(c)
        out, lse = D.decode(path=path)
        assert gva().gva_get_device_status() == 0
        assert_close(out, ref, "bf16", f"B=4096 {path}")
        assert_close(lse, ref_lse, "bf16", f"B=4096 {path} lse")


STEP_CASES = {
    "350m": ("350m", {}), "paged": ("paged", {}), "tiny": ("tiny", {}),
    "ragged": ("ragged", {}), "long": ("long", {}),
    "350m_f32_query": ("350m", dict(q_dtype="f32")),
    "350m_dn32": ("350m", dict(d_n=32)),      # tensor-core path, separate append kernel
    # the largest batch: the held slabs' indices take another 16 KB of shared memory
    "350m_b4096": ("350m", dict(B=4096, T=40, H=4, G=2, d_h=64, d_n=64, d_r=16)),
}


@pytest.mark.parametrize("case", list(STEP_CASES))
def test_decode_step_matches_per_layer_calls(case):
    """gva_decode_step over three layers (one C call: each layer's append, then its decode,
    the layers sharing one workspace) equals the per-layer gva_append_cache and
    gva_decode_attention calls bit for bit, outputs and appended rows, and the oracle.
    On the tensor-core path with a bf16 cache the step runs each layer's append inside
    the absorption's grid (bf16 and fp32 queries), on the others as its own kernel."""
    g = gva()
    name, extra = STEP_CASES[case]
    c = make_case(workload(name, **{**SMALL[name], **extra}))
    pos = (c.seq_len - 1).to(torch.int32).cuda()
    a = [Dev(c) for _ in range(3)]          # per-layer calls
    s = [Dev(c) for _ in range(3)]          # one step call
    w = c.w
    outs_a, outs_s = [], []
    for D in a:
        D.append(pos)
        outs_a.append(D.decode())
    layers = []
    for D in s:
        out = torch.full((w.B, w.H, w.d_h), float("nan"), device="cuda")
        lse = torch.full((w.B, w.H), float("nan"), device="cuda")
        layers.append(dict(v_new=D.v_new, k_rope_new=D.k_new, q_nope=D.q_nope, q_rope=D.q_rope,
                           M=D.M, cache=D.cache, out=out, lse=lse))
    g.gva_decode_step(s[0].dims, layers, pos, s[0].seq_len, s[0].tab, w.scale, s[0].ws)
    torch.cuda.synchronize()
    assert g.gva_get_device_status() == 0
    for (oa, la), L, Da, Ds in zip(outs_a, layers, a, s):
        assert np.array_equal(oa, L["out"].cpu().numpy().astype(np.float64))
        assert np.array_equal(la, L["lse"].cpu().numpy().astype(np.float64))
        assert torch.equal(Da.V, Ds.V) and torch.equal(Da.Kr, Ds.Kr)
    V, K = oracle_append(c, pos.cpu(), s[0].tab_h)
    ref, ref_lse = oracle_decode(c, V, K)
    assert_close(outs_a[0][0], ref, w.cache_dtype, f"{case} step out")
    assert_close(outs_a[0][1], ref_lse, w.cache_dtype, f"{case} step lse")


@pytest.mark.parametrize("name", ["350m", "ragged", "paged"])
def test_decode_step_rows_inside_the_sequences(name):
    """gva_decode_step whose appends overwrite rows inside the sequences (positions in the
    first slab, in a middle slab, in the last slab, and past the length, which the decode
    does not read): the decode holds back exactly the slab each new row falls in, so the
    outputs and rows equal those of the per-layer calls bit for bit, and the oracle."""
    g = gva()
    c = make_case(workload(name, **SMALL[name], extra_slots=2))
    w = c.w
    L = c.seq_len.tolist()
    pos_l = []
    for b, Lb in enumerate(L):
        choice = b % 4
        if choice == 0:
            p = min(3, Lb - 1)
        elif choice == 1:
            p = Lb // 2
        elif choice == 2:
            p = Lb - 1
        else:
            p = Lb if w.extra_slots > 0 else Lb - 1     # every capacity is L_b + extra_slots
        pos_l.append(max(p, 0))
    pos = torch.tensor(pos_l, dtype=torch.int32).cuda()
    a, s = Dev(c), Dev(c)
    a.append(pos)
    oa, la = a.decode()
    out = torch.full((w.B, w.H, w.d_h), float("nan"), device="cuda")
    lse = torch.full((w.B, w.H), float("nan"), device="cuda")
    layer = dict(v_new=s.v_new, k_rope_new=s.k_new, q_nope=s.q_nope, q_rope=s.q_rope, M=s.M,
                 cache=s.cache, out=out, lse=lse)
    g.gva_decode_step(s.dims, [layer], pos, s.seq_len, s.tab, w.scale, s.ws)
    torch.cuda.synchronize()
    assert g.gva_get_device_status() == 0
    assert np.array_equal(oa, out.cpu().numpy().astype(np.float64))
    assert np.array_equal(la, lse.cpu().numpy().astype(np.float64))
    assert torch.equal(a.V, s.V) and torch.equal(a.Kr, s.Kr)
    V, K = oracle_append(c, pos.cpu(), s.tab_h)
    ref, ref_lse = oracle_decode(c, V, K)
    assert_close(oa, ref, w.cache_dtype, f"{name} overwrite step out")
    assert_close(la, ref_lse, w.cache_dtype, f"{name} overwrite step lse")


@pytest.mark.parametrize("name", ["350m", "paged", "tiny"])
def test_step_plan_replays_the_step(name):
    """A step recorded by gva_step_plan_create and launched twice, with new queries written
    in place between the launches, gives what the per-layer calls give on the same
    contents, bit for bit: outputs and appended rows of three layers."""
    g = gva()
    c = make_case(workload(name, **SMALL[name]))
    pos = (c.seq_len - 1).to(torch.int32).cuda()
    a = [Dev(c) for _ in range(3)]          # per-layer calls
    s = [Dev(c) for _ in range(3)]          # the recorded step
    w = c.w
    layers = []
    for D in s:
        out = torch.full((w.B, w.H, w.d_h), float("nan"), device="cuda")
        lse = torch.full((w.B, w.H), float("nan"), device="cuda")
        layers.append(dict(v_new=D.v_new, k_rope_new=D.k_new, q_nope=D.q_nope, q_rope=D.q_rope,
                           M=D.M, cache=D.cache, out=out, lse=lse))
    plan = g.create_step_plan(s[0].dims, layers, pos, s[0].seq_len, s[0].tab, w.scale, s[0].ws)
    for it in range(2):
        if it == 1:
            for D in a + s:
                D.q_nope.mul_(-0.5)             # new contents, same storage
        plan.launch()
        refs = []
        for D in a:
            D.append(pos)
            refs.append(D.decode())
        torch.cuda.synchronize()
        assert g.gva_get_device_status() == 0
        for (oa, la), L, Da, Ds in zip(refs, layers, a, s):
            assert np.array_equal(oa, L["out"].cpu().numpy().astype(np.float64)), f"launch {it}"
            assert np.array_equal(la, L["lse"].cpu().numpy().astype(np.float64)), f"launch {it}"
            assert torch.equal(Da.V, Ds.V) and torch.equal(Da.Kr, Ds.Kr)
    plan.close()
