"""GPU parity of the causal chunked prefill (gva_prefill_attention, through the C ABI)
against the fp64 oracle on the same seeded inputs: the appended rows bit-exact, the
outputs within the decode tolerances (bf16 cache: max-abs 2e-2 and relative L2 1e-3;
fp32 cache: 1e-5)."""
import numpy as np
import pytest
import torch

import oracle
from gva_inputs import make_case, make_prefill_chunk, workload
from helpers import assert_close, dims_of, gva, oracle_rows, oracle_table, rope_tab

pytestmark = pytest.mark.gpu


def _supported(c, path):
    w = c.w
    if path == "mma":
        return w.cache_dtype == "bf16" and w.d_h in (64, 128) and w.G <= 8
    return True


class Run:
    """One prefill call on the GPU and the oracle's answer for the same chunk."""

    def __init__(self, c, n, path="auto", q_norm=None, L0=None):
        g = gva()
        w = c.w
        d = torch.device("cuda")
        ch = make_prefill_chunk(c, n)
        if L0 is not None:
            ch.L0 = torch.tensor(L0, dtype=torch.int32)
        self.c, self.ch = c, ch
        self.V, self.Kr = c.V.to(d), c.Kr.to(d)
        rows = g.Rows(w.layout, c.num_rows, T_cap=c.T_cap,
                      offsets=c.offsets.to(d) if c.offsets is not None else None,
                      block_table=c.block_table.to(d) if c.block_table is not None else None,
                      page_size=w.page_size)
        cache = g.Cache(rows, self.V, self.Kr)
        dims = dims_of(c)
        self.tab_h = rope_tab(c)
        ws = g.prefill_workspace(dims, n, rows, d)
        self.out = torch.full((w.B, n, w.H, w.d_h), float("nan"), device=d)
        self.lse = torch.full((w.B, n, w.H), float("nan"), device=d)
        gq = None
        if q_norm is not None:
            gq = (None if q_norm[0] is None else q_norm[0].to(d), q_norm[1])
        g.gva_prefill_attention(dims, ch.q_nope.to(d), ch.q_rope.to(d), c.M.to(d),
                                ch.L0.to(d), ch.v_new.to(d), ch.k_new.to(d), cache,
                                self.tab_h.to(d), w.scale, self.out, self.lse, ws, path=path,
                                q_norm=gq)
        torch.cuda.synchronize()
        self.status = g.gva_get_device_status()

    def oracle_cache(self, n=None):
        """Host storage with the oracle's append of the chunk's first n tokens."""
        c, ch = self.c, self.ch
        n = ch.n if n is None else n
        Vh, Kh = oracle._np(c.V).copy(), oracle._np(c.Kr).copy()
        R = oracle_rows(c)
        for i in range(n):
            oracle.append(ch.v_new[:, i], ch.k_new[:, i], ch.L0.to(torch.int64) + i, R, Vh, Kh,
                          oracle_table(c, int(self.tab_h.shape[0])))
        return Vh, Kh

    def oracle_out(self, Vh, Kh, q_nope=None, n=None):
        c, ch, w = self.c, self.ch, self.c.w
        n = ch.n if n is None else n
        qn = ch.q_nope if q_nope is None else q_nope
        return oracle.gva_prefill(qn[:, :n], ch.q_rope[:, :n], c.M, ch.L0, oracle_rows(c), Vh,
                                  Kh, w.scale, w.base, w.G)

    def got(self):
        return (self.out.cpu().numpy().astype(np.float64),
                self.lse.cpu().numpy().astype(np.float64))


def _check_cache(r, Vh, Kh):
    assert np.array_equal(oracle._np(r.V.cpu()), Vh), "appended values differ"
    assert np.array_equal(oracle._np(r.Kr.cpu()), Kh), "appended positional keys differ"


# small variants: several slabs and CTAs, ragged tails, chunks crossing slab and page
# boundaries
SMALL = {
    "tiny": (dict(), 5),
    "350m": (dict(T=320, B=3), 9),
    "long": (dict(B=2, T=1200), 3),
    "paged": (dict(B=5, len_range=(64, 900)), 17),
}


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("path", ["simt", "mma", "auto"])
def test_prefill_small_workloads(name, path):
    over, n = SMALL[name]
    c = make_case(workload(name, **over))
    if not _supported(c, path):
        pytest.skip(f"{path} path needs a bf16 cache")
    r = Run(c, n, path)
    assert r.status == 0
    Vh, Kh = r.oracle_cache()
    _check_cache(r, Vh, Kh)
    ref, ref_lse = r.oracle_out(Vh, Kh)
    out, lse = r.got()
    assert_close(out, ref, c.w.cache_dtype, f"{name}/{path} out")
    assert_close(lse, ref_lse, c.w.cache_dtype, f"{name}/{path} lse")


@pytest.mark.parametrize("n", [1, 16, 33])
def test_prefill_chunk_lengths(n):
    """One token (a decode step), one slab, and a chunk with a ragged tail, from an
    empty history for one sequence."""
    c = make_case(workload("350m", T=128, B=3), lengths=[128, 100, n])
    r = Run(c, n)
    assert r.status == 0
    Vh, Kh = r.oracle_cache()
    _check_cache(r, Vh, Kh)
    ref, ref_lse = r.oracle_out(Vh, Kh)
    out, lse = r.got()
    assert_close(out, ref, "bf16", f"n={n}")
    assert_close(lse, ref_lse, "bf16", f"n={n} lse")


@pytest.mark.parametrize("n", [20, 32])
def test_prefill_128_row_groups(n):
    """Chunks whose group rows (n r = 80 and 128) fill the tensor-core prefill kernel's
    128-row products (d_h = 64), over histories that end mid-tile and in permuted pages."""
    for name, over, lengths in (("350m", dict(T=400, B=3), [400, 231, n]),
                                ("paged", dict(B=3, len_range=(64, 600), H=16, G=4, d_h=64, d_n=64),
                                 None)):
        c = make_case(workload(name, **over), lengths=lengths)
        r = Run(c, n)
        assert r.status == 0
        Vh, Kh = r.oracle_cache()
        _check_cache(r, Vh, Kh)
        ref, ref_lse = r.oracle_out(Vh, Kh)
        out, lse = r.got()
        assert_close(out, ref, "bf16", f"{name} n={n}")
        assert_close(lse, ref_lse, "bf16", f"{name} n={n} lse")


def test_prefill_largest_batch():
    """B * n = 4096 decode entries, the largest the library takes."""
    c = make_case(workload("350m", T=160, B=64))
    r = Run(c, 64)
    assert r.status == 0
    Vh, Kh = r.oracle_cache()
    _check_cache(r, Vh, Kh)
    ref, ref_lse = r.oracle_out(Vh, Kh)
    out, lse = r.got()
    assert_close(out, ref, "bf16", "B*n=4096")
    assert_close(lse, ref_lse, "bf16", "B*n=4096 lse")


@pytest.mark.parametrize("cache", ["bf16", "f32"])
def test_prefill_query_rmsnorm(cache):
    w = workload("350m", T=192, B=2, cache_dtype=cache,
                 q_dtype="f32" if cache == "f32" else "bf16")
    c = make_case(w)
    gain = torch.randn(w.d_n, generator=torch.Generator().manual_seed(9)) * 0.5 + 1.0
    r = Run(c, 6, q_norm=(gain, 1e-6))
    assert r.status == 0
    Vh, Kh = r.oracle_cache()
    n = r.ch.n
    qn = oracle.query_rmsnorm(r.ch.q_nope.reshape(w.B * n, w.H, w.d_n), gain.numpy(), 1e-6)
    ref, ref_lse = r.oracle_out(Vh, Kh, q_nope=qn.reshape(w.B, n, w.H, w.d_n))
    out, lse = r.got()
    assert_close(out, ref, cache, "q-norm out")
    assert_close(lse, ref_lse, cache, "q-norm lse")


def test_prefill_past_capacity_is_reported():
    """A chunk running past the capacity: its tokens beyond it are skipped with a status
    code, their queries return out = 0 and lse = -inf, and the queries that fit are
    right."""
    c = make_case(workload("350m", T=64, B=2), lengths=[64, 30])
    r = Run(c, 8, L0=[60, 22])
    assert r.status == gva().GVA_DEV_BAD_POSITION
    Vh, Kh = r.oracle_cache(n=4)          # sequence 0 keeps 4 tokens, sequence 1 all 8
    seq1 = oracle.Rows("ragged", offsets=np.array([c.T_cap, 2 * c.T_cap]))
    for i in range(4, 8):
        oracle.append(r.ch.v_new[1:, i], r.ch.k_new[1:, i], [22 + i], seq1, Vh, Kh,
                      oracle_table(c, int(r.tab_h.shape[0])))
    _check_cache(r, Vh, Kh)
    out, lse = r.got()
    ref, ref_lse = r.oracle_out(Vh, Kh, n=4)
    assert_close(out[0, :4], ref[0], "bf16", "b=0 fitting queries")
    assert np.all(out[0, 4:] == 0) and np.isneginf(lse[0, 4:]).all()
    ref1, _ = oracle.gva_prefill(r.ch.q_nope[1:], r.ch.q_rope[1:], c.M, r.ch.L0[1:], seq1, Vh,
                                 Kh, c.w.scale, c.w.base, c.w.G)
    assert_close(out[1], ref1[0], "bf16", "b=1")
    assert gva().gva_get_device_status() == 0


@pytest.mark.parametrize("B,lens,n", [(3, (20, 60), 4), (5, (30, 900), 16), (4, (129, 700), 20)])
def test_prefill_ragged_layout(B, lens, n):
    """Ragged rows (sequences packed at arbitrary offsets): the tcgen05 prefill reads the
    caller's rows (64 query rows per group at n = 16, 128 at n = 20), appended rows
    bit-exact and outputs against the oracle; the view paths refuse the layout."""
    c = make_case(workload("ragged", B=B, len_range=lens))
    r = Run(c, n)
    assert r.status == 0
    Vh, Kh = r.oracle_cache()
    _check_cache(r, Vh, Kh)
    ref, ref_lse = r.oracle_out(Vh, Kh)
    out, lse = r.got()
    assert_close(out, ref, "bf16", f"ragged B={B} n={n} out")
    assert_close(lse, ref_lse, "bf16", f"ragged B={B} n={n} lse")
    g = gva()
    for path in ("simt", "mma"):
        with pytest.raises(g.GvaError) as e:
            Run(c, n, path)
        assert e.value.status == g.GVA_ERR_UNSUPPORTED


@pytest.mark.parametrize("H,G,d_h,d_n,d_r", [
    (8, 8, 64, 64, 16), (8, 4, 64, 32, 8), (8, 2, 128, 128, 24), (8, 1, 64, 64, 32),
    (16, 2, 64, 32, 0), (4, 4, 128, 64, 16), (32, 4, 64, 128, 16), (3, 3, 64, 64, 16),
    (16, 8, 128, 128, 32),
])
@pytest.mark.parametrize("n", [3, 21])
def test_prefill_shapes(H, G, d_h, d_n, d_r, n):
    """The default path (the tensor-core prefill kernel for bf16 caches) over head
    groupings r = 1..8, every positional width, both value widths."""
    w = workload("350m", B=2, T=160, H=H, G=G, d_h=d_h, d_n=d_n, d_r=d_r)
    c = make_case(w, lengths=[160, 45])
    r = Run(c, n)
    assert r.status == 0
    Vh, Kh = r.oracle_cache()
    _check_cache(r, Vh, Kh)
    ref, ref_lse = r.oracle_out(Vh, Kh)
    out, lse = r.got()
    assert_close(out, ref, "bf16", f"{H},{G},{d_h},{d_n},{d_r} n={n}")
    assert_close(lse, ref_lse, "bf16", f"{H},{G},{d_h},{d_n},{d_r} n={n} lse")


def test_prefill_paths_agree_on_a_paged_batch():
    """Every path on the same paged chunk: the tensor-core prefill kernel (auto) and the
    decode-entry compositions (simt, mma), each against the oracle."""
    c = make_case(workload("paged", B=3, len_range=(100, 700)))
    refs = None
    for path in ("auto", "simt", "mma"):
        r = Run(c, 12, path)
        assert r.status == 0
        if refs is None:
            Vh, Kh = r.oracle_cache()
            refs = r.oracle_out(Vh, Kh), (Vh, Kh)
        _check_cache(r, *refs[1])
        out, lse = r.got()
        assert_close(out, refs[0][0], "bf16", f"{path} out")
        assert_close(lse, refs[0][1], "bf16", f"{path} lse")


def test_prefill_full_size_350m():
    """The bench's prefill workload in its launch configuration (350M layer, B = 8,
    T = 4096, the last 16 tokens of every sequence as the chunk, default path), every
    output against the oracle."""
    c = make_case(workload("350m"))
    r = Run(c, 16)
    assert r.status == 0
    Vh, Kh = r.oracle_cache()
    _check_cache(r, Vh, Kh)
    ref, ref_lse = r.oracle_out(Vh, Kh)
    out, lse = r.got()
    assert_close(out, ref, "bf16", "350m full size")
    assert_close(lse, ref_lse, "bf16", "350m full size lse")


@pytest.mark.parametrize("B,H,G,n", [(1, 4, 1, 16), (1, 8, 2, 8), (2, 8, 1, 4)])
def test_prefill_range_merge_paths(B, H, G, n):
    """The tcgen05 prefill splits each (value group, sequence) over 148 / (B G) history
    ranges, most of them empty at this length.  Their log-sum-exp merge runs in the
    kernel's last CTA per (group, sequence) when the ranges' (max, sum) of the group's rows
    fit its P buffers (32 rows over 74 ranges), else in the merge kernel (64 rows over 148
    ranges)."""
    w = workload("350m", B=B, T=3008, H=H, G=G)
    c = make_case(w, lengths=[3008, 1777][:B])
    r = Run(c, n)
    assert r.status == 0
    Vh, Kh = r.oracle_cache()
    _check_cache(r, Vh, Kh)
    ref, ref_lse = r.oracle_out(Vh, Kh)
    out, lse = r.got()
    assert_close(out, ref, "bf16", f"B={B} H={H} G={G} n={n} out")
    assert_close(lse, ref_lse, "bf16", f"B={B} H={H} G={G} n={n} lse")


def test_prefill_plan_replays_the_chunk():
    """A chunk through two layers recorded by gva_prefill_plan_create and launched twice,
    with new queries written in place between the launches, gives what the per-layer
    gva_prefill_attention calls give on the same contents, bit for bit."""
    g = gva()
    c = make_case(workload("350m", **SMALL["350m"][0]))
    n = 9
    w = c.w
    d = torch.device("cuda")
    ch = make_prefill_chunk(c, n)
    rows = g.Rows(w.layout, c.num_rows, T_cap=c.T_cap)
    dims = dims_of(c)
    tab = rope_tab(c).to(d)
    L0 = ch.L0.to(d)

    def layer():
        return dict(q_nope=ch.q_nope.to(d), q_rope=ch.q_rope.to(d), M=c.M.to(d),
                    v_new=ch.v_new.to(d), k_rope_new=ch.k_new.to(d),
                    cache=g.Cache(rows, c.V.to(d), c.Kr.to(d)),
                    out=torch.full((w.B, n, w.H, w.d_h), float("nan"), device=d),
                    lse=torch.full((w.B, n, w.H), float("nan"), device=d))
    ref_layers, plan_layers = [layer(), layer()], [layer(), layer()]
    ws_ref = g.prefill_workspace(dims, n, rows, d)
    ws = g.prefill_workspace(dims, n, rows, d)
    plan = g.create_prefill_plan(dims, n, plan_layers, L0, tab, w.scale, ws)
    for it in range(2):
        if it == 1:
            for L in ref_layers + plan_layers:
                L["q_nope"].mul_(-0.5)
        plan.launch()
        for L in ref_layers:
            g.gva_prefill_attention(dims, L["q_nope"], L["q_rope"], L["M"], L0, L["v_new"],
                                    L["k_rope_new"], L["cache"], tab, w.scale, L["out"],
                                    L["lse"], ws_ref)
        torch.cuda.synchronize()
        assert g.gva_get_device_status() == 0
        for R, P in zip(ref_layers, plan_layers):
            assert torch.equal(R["out"], P["out"]), f"launch {it} out"
            assert torch.equal(R["lse"], P["lse"]), f"launch {it} lse"
            assert torch.equal(R["cache"].V.view(torch.int16), P["cache"].V.view(torch.int16))
            assert torch.equal(R["cache"].K_rope.view(torch.int16), P["cache"].K_rope.view(torch.int16))
    plan.close()
