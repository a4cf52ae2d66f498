"""Test helpers: move a seeded case to the GPU, run the library through its Python
binding (the C ABI), run the oracle on the same inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from gva_inputs import Case

# tolerances the decode must meet against the fp64 oracle
TOL = {"bf16": dict(max_abs=2e-2, rel_l2=1e-3), "f32": dict(max_abs=1e-5, rel_l2=1e-5)}


def gva():
    import value_only_kv_gva_b300 as m
    return m


def dims_of(c: Case):
    g = gva()
    w = c.w
    return g.Dims(w.B, w.H, w.G, w.d_h, w.d_n, w.d_r,
                  g.GVA_F32 if w.cache_dtype == "f32" else g.GVA_BF16,
                  g.GVA_F32 if w.q_dtype == "f32" else g.GVA_BF16)


def rope_tab(c: Case, extra: int = 1) -> torch.Tensor:
    cap = c.T_cap if c.w.layout == "contiguous" else int(c.seq_len.max()) + c.w.extra_slots
    return gva().gva_rope_table_fill(max(cap, int(c.seq_len.max())) + extra, c.w.d_r, c.w.base)


def oracle_rows(c: Case, sample=None) -> oracle.Rows:
    """Row map of the whole batch, or of the sub-batch `sample` (list of b)."""
    w = c.w
    if sample is None:
        if w.layout == "contiguous":
            return oracle.Rows("contiguous", T_cap=c.T_cap)
        if w.layout == "ragged":
            return oracle.Rows("ragged", offsets=c.offsets.numpy())
        return oracle.Rows("paged", block_table=c.block_table.numpy(), page_size=w.page_size)
    sample = list(sample)
    if w.layout == "contiguous":
        return oracle.Rows("ragged", offsets=np.array([b * c.T_cap for b in sample] + [0]))
    if w.layout == "ragged":
        return oracle.Rows("ragged", offsets=np.array([int(c.offsets[b]) for b in sample] + [0]))
    return oracle.Rows("paged", block_table=c.block_table.numpy()[sample], page_size=w.page_size)


class Dev:
    """A case's tensors on the GPU plus the binding's cache descriptors."""

    def __init__(self, c: Case, device="cuda"):
        g = gva()
        self.c = c
        self.d = torch.device(device)
        d = self.d
        self.V = c.V.to(d)
        self.Kr = c.Kr.to(d)
        self.q_nope = c.q_nope.to(d)
        self.q_rope = c.q_rope.to(d)
        self.M = c.M.to(d)
        self.seq_len = c.seq_len.to(d)
        self.v_new = c.v_new.to(d)
        self.k_new = c.k_new.to(d)
        self.offsets = c.offsets.to(d) if c.offsets is not None else None
        self.block_table = c.block_table.to(d) if c.block_table is not None else None
        w = c.w
        self.rows = g.Rows(w.layout, c.num_rows, T_cap=c.T_cap, offsets=self.offsets,
                           block_table=self.block_table, page_size=w.page_size)
        self.cache = g.Cache(self.rows, self.V, self.Kr)
        self.dims = dims_of(c)
        self.tab_h = rope_tab(c)
        self.tab = self.tab_h.to(d)
        self.ws = g.workspace(self.dims, d)

    def append(self, pos: torch.Tensor, seq_len_out=None):
        gva().gva_append_cache(self.dims, self.v_new, self.k_new, pos.to(self.d), seq_len_out,
                               self.cache, self.tab)

    def decode(self, path="auto", num_ctas=0, seq_len=None):
        w = self.c.w
        out = torch.full((w.B, w.H, w.d_h), float("nan"), device=self.d)
        lse = torch.full((w.B, w.H), float("nan"), device=self.d)
        gva().gva_decode_attention(self.dims, self.q_nope, self.q_rope, self.M,
                                   self.seq_len if seq_len is None else seq_len, self.cache,
                                   self.tab, w.scale, out, lse, self.ws, path=path,
                                   num_ctas=num_ctas)
        torch.cuda.synchronize()
        return out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def oracle_table(c: Case, max_pos: int) -> np.ndarray:
    """The oracle's own fp32 (cos, sin) table, built by the oracle (not the library)."""
    return oracle.rope_table_f32(int(max_pos), c.w.d_r, c.w.base)


def oracle_append(c: Case, pos, tab_h: torch.Tensor):
    """Host copies of the cache storage with the oracle's append applied.  The oracle
    builds its own rotation table (as many positions as the library's table `tab_h`,
    whose length only bounds which positions are valid)."""
    V = oracle._np(c.V).copy()
    K = oracle._np(c.Kr).copy()
    oracle.append(c.v_new, c.k_new, pos, oracle_rows(c), V, K,
                  oracle_table(c, int(tab_h.shape[0])))
    return V, K


def oracle_decode(c: Case, V=None, K=None, seq_len=None, sample=None):
    """fp64 reference outputs for all sequences, or for the sub-batch `sample`."""
    w = c.w
    V = oracle._np(c.V) if V is None else V
    K = oracle._np(c.Kr) if K is None else K
    sl = (c.seq_len if seq_len is None else seq_len).numpy().astype(np.int64)
    qn, qr = c.q_nope, c.q_rope
    if sample is not None:
        idx = torch.tensor(list(sample))
        qn, qr, sl = qn[idx], qr[idx], sl[list(sample)]
    return oracle.gva_decode(qn, qr, c.M, sl, oracle_rows(c, sample), V, K, w.scale, w.base, w.G)


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), "non-finite pattern differs"
    d = np.abs(got[fin] - ref[fin])
    max_abs = float(d.max()) if d.size else 0.0
    den = float(np.linalg.norm(ref[fin]))
    rel = float(np.linalg.norm(got[fin] - ref[fin]) / den) if den > 0 else max_abs
    return max_abs, rel


def assert_close(got, ref, dtype: str, what=""):
    t = TOL[dtype]
    max_abs, rel = errors(got, ref)
    assert max_abs <= t["max_abs"] and rel <= t["rel_l2"], \
        f"{what}: max_abs {max_abs:.3e} (<= {t['max_abs']}), rel_l2 {rel:.3e} (<= {t['rel_l2']})"
    return max_abs, rel
