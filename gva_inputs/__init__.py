"""Seeded synthetic inputs for GVA decode: the one module both the CUDA path's tests
and the fp64 oracle take their inputs from.

It holds none of the method's arithmetic: it only draws numbers, rounds storage
dtypes, builds layouts (lengths, offsets, block tables) and packs them.  Every
draw comes from one CPU ``torch.Generator`` per case, in a fixed order:

  1. lengths       (ragged / paged workloads only: integers, inclusive range)
  2. V             N(0, 1), fp32, whole storage (slots past a sequence's end too)
  3. K_rope        N(0, 1), fp32 -- the positional keys are "cached already
                   rotated"; a rotated standard normal vector is again standard
                   normal, so the stored keys are drawn directly in that
                   distribution and no rotation happens here
  4. q_nope        N(0, 1)
  5. q_rope        N(0, 1)
  6. M             N(0, 1/d_h)   (the scale-matched init with sigma_Q = sigma_V = 1,
                                  d_in = d_h)
  7. extras        spike positions (long workload), page permutation (paged),
                   new-token v / k for the append step

then a single round-to-nearest-even cast to bf16 where the workload stores bf16.
The five workloads are the ones the decode path is measured and checked on:
tiny, 350m, ragged, long, paged.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

ROPE_BASE = 10000.0
PAGE_SIZE = 64


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    G: int
    d_h: int
    d_n: int
    d_r: int
    T: int = 0                      # contiguous capacity = length of every sequence
    len_range: tuple | None = None  # ragged / paged: lengths uniform in [lo, hi]
    layout: str = "contiguous"      # contiguous | ragged | paged
    cache_dtype: str = "bf16"       # bf16 | f32
    q_dtype: str = "bf16"
    seed: int = 0
    spike_frac: float = 0.0         # fraction of positions whose V is scaled
    spike_scale: float = 1.0
    page_size: int = PAGE_SIZE
    extra_slots: int = 0            # free capacity after each sequence (appends)
    base: float = ROPE_BASE

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d_n + self.d_r)

    @property
    def r(self) -> int:
        return self.H // self.G


WORKLOADS = {
    "tiny": Workload("tiny", B=1, H=4, G=2, d_h=32, d_n=32, d_r=8, T=64,
                     cache_dtype="f32", q_dtype="f32", seed=0),
    "350m": Workload("350m", B=8, H=16, G=4, d_h=64, d_n=64, d_r=16, T=4096, seed=1),
    "ragged": Workload("ragged", B=32, H=16, G=4, d_h=64, d_n=64, d_r=24,
                       len_range=(1, 8192), layout="ragged", seed=2),
    "long": Workload("long", B=2, H=32, G=8, d_h=128, d_n=128, d_r=16, T=131072,
                     seed=3, spike_frac=0.01, spike_scale=8.0),
    "paged": Workload("paged", B=64, H=32, G=8, d_h=128, d_n=128, d_r=16,
                      len_range=(1024, 16384), layout="paged", seed=4),
}


def workload(name: str, **over) -> Workload:
    return replace(WORKLOADS[name], **over)


@dataclass
class Case:
    """All tensors on the CPU.  V: [rows, G, d_h], Kr: [rows, d_r] in the cache dtype;
    q_nope [B,H,d_n], q_rope [B,H,d_r] in the query dtype; M [H,d_h,d_n] fp32;
    seq_len [B] int32; offsets [B+1] int32 (ragged); block_table [B,max_pages] int32
    (paged, unused entries -1); v_new [B,G,d_h] and k_new [B,d_r] fp32 (unrotated)."""
    w: Workload
    V: torch.Tensor
    Kr: torch.Tensor
    q_nope: torch.Tensor
    q_rope: torch.Tensor
    M: torch.Tensor
    seq_len: torch.Tensor
    v_new: torch.Tensor
    k_new: torch.Tensor
    T_cap: int = 0
    offsets: torch.Tensor | None = None
    block_table: torch.Tensor | None = None
    num_pages: int = 0
    extras: dict = field(default_factory=dict)

    @property
    def num_rows(self) -> int:
        return int(self.V.shape[0])


def _dt(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def make_case(w: Workload, lengths=None) -> Case:
    """Draw one case.  ``lengths`` (a list) overrides the drawn / fixed lengths."""
    g = torch.Generator().manual_seed(w.seed)
    B = w.B
    # 1. lengths
    if lengths is not None:
        lens = torch.tensor(list(lengths), dtype=torch.int64)
        assert lens.numel() == B
    elif w.len_range is not None:
        lo, hi = w.len_range
        lens = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64)
    else:
        lens = torch.full((B,), w.T, dtype=torch.int64)
    cap = lens + w.extra_slots
    offsets = block_table = None
    num_pages = 0
    T_cap = 0
    if w.layout == "contiguous":
        T_cap = int(max(int(cap.max()), w.T + w.extra_slots)) if B else 0
        rows = B * T_cap
    elif w.layout == "ragged":
        offsets = torch.zeros(B + 1, dtype=torch.int64)
        offsets[1:] = torch.cumsum(cap, 0)
        rows = int(offsets[-1])
    elif w.layout == "paged":
        pages_per = (cap + w.page_size - 1) // w.page_size
        num_pages = int(pages_per.sum())
        rows = num_pages * w.page_size
    else:
        raise ValueError(w.layout)
    # 2.-6.
    V = torch.randn((rows, w.G, w.d_h), generator=g, dtype=torch.float32)
    Kr = torch.randn((rows, w.d_r), generator=g, dtype=torch.float32)
    q_nope = torch.randn((B, w.H, w.d_n), generator=g, dtype=torch.float32)
    q_rope = torch.randn((B, w.H, w.d_r), generator=g, dtype=torch.float32)
    M = torch.randn((w.H, w.d_h, w.d_n), generator=g, dtype=torch.float32) / math.sqrt(w.d_h)
    # 7. extras
    extras = {}
    if w.layout == "paged":
        perm = torch.randperm(num_pages, generator=g)
        max_pages = int(pages_per.max()) if B else 0
        block_table = torch.full((B, max(max_pages, 1)), -1, dtype=torch.int64)
        k = 0
        for b in range(B):
            for p in range(int(pages_per[b])):
                block_table[b, p] = perm[k]
                k += 1
        extras["perm"] = perm
    if w.spike_frac > 0:
        # per sequence: floor(frac * L_b) positions without replacement, V scaled
        # at every group, before the storage cast (K_rope untouched)
        spikes = []
        for b in range(B):
            L = int(lens[b])
            n = int(math.floor(w.spike_frac * L))
            pos = torch.randperm(L, generator=g)[:n]
            spikes.append(pos)
            if w.layout == "contiguous":
                V[b * T_cap + pos] *= w.spike_scale
            elif w.layout == "ragged":
                V[int(offsets[b]) + pos] *= w.spike_scale
            else:
                pg = block_table[b, pos // w.page_size]
                V[pg * w.page_size + pos % w.page_size] *= w.spike_scale
        extras["spikes"] = spikes
    v_new = torch.randn((B, w.G, w.d_h), generator=g, dtype=torch.float32)
    k_new = torch.randn((B, w.d_r), generator=g, dtype=torch.float32)
    cd, qd = _dt(w.cache_dtype), _dt(w.q_dtype)
    return Case(
        w=w, V=V.to(cd), Kr=Kr.to(cd), q_nope=q_nope.to(qd), q_rope=q_rope.to(qd), M=M,
        seq_len=lens.to(torch.int32), v_new=v_new, k_new=k_new, T_cap=T_cap,
        offsets=None if offsets is None else offsets.to(torch.int32),
        block_table=None if block_table is None else block_table.to(torch.int32),
        num_pages=num_pages, extras=extras)


def make_gqa_keys(case: Case) -> torch.Tensor:
    """Explicit keys for the matched GQA comparator: same rows/layout as V, drawn
    N(0, 1) from a second generator (seed + 1000), cast to the cache dtype."""
    g = torch.Generator().manual_seed(case.w.seed + 1000)
    K = torch.randn(tuple(case.V.shape), generator=g, dtype=torch.float32)
    return K.to(case.V.dtype)


def make_gqa_query(case: Case) -> torch.Tensor:
    """GQA query [B, H, d_h] N(0, 1) (seed + 2000), in the workload's query dtype."""
    g = torch.Generator().manual_seed(case.w.seed + 2000)
    q = torch.randn((case.w.B, case.w.H, case.w.d_h), generator=g, dtype=torch.float32)
    return q.to(_dt(case.w.q_dtype))


@dataclass
class MlaCase:
    """Inputs of the MLA-shaped comparator at matched cache bytes (latent width
    d_c = G d_h, so a latent row plus the positional key has the size of a GVA row):
    latent rows C [rows, d_c] N(0, 1) in the cache dtype (the case's row layout), up-
    projections W_uk [H, d_c, d_n] and W_uv [H, d_c, d_h] N(0, 1/d_c) fp32.  The queries,
    positional keys and lengths are the case's own."""
    d_c: int
    C: torch.Tensor
    W_uk: torch.Tensor
    W_uv: torch.Tensor


def make_mla_case(case: Case) -> MlaCase:
    """Drawn from a fourth generator (seed + 4000) in the order C, W_uk, W_uv."""
    w = case.w
    d_c = w.G * w.d_h
    g = torch.Generator().manual_seed(w.seed + 4000)
    C = torch.randn((case.num_rows, d_c), generator=g, dtype=torch.float32)
    Wuk = torch.randn((w.H, d_c, w.d_n), generator=g, dtype=torch.float32) / math.sqrt(d_c)
    Wuv = torch.randn((w.H, d_c, w.d_h), generator=g, dtype=torch.float32) / math.sqrt(d_c)
    return MlaCase(d_c=d_c, C=C.to(case.V.dtype), W_uk=Wuk, W_uv=Wuv)


@dataclass
class Chunk:
    """A prefill chunk of n new tokens per sequence, all on the CPU: the history L0
    [B] int32, queries q_nope [B,n,H,d_n] and q_rope [B,n,H,d_r] (query dtype), new
    values v_new [B,n,G,d_h] and unrotated positional keys k_new [B,n,d_r] (fp32)."""
    n: int
    L0: torch.Tensor
    q_nope: torch.Tensor
    q_rope: torch.Tensor
    v_new: torch.Tensor
    k_new: torch.Tensor


def make_prefill_chunk(case: Case, n: int) -> Chunk:
    """The chunk that ends at the case's lengths: L0[b] = L_b - n (every L_b >= n), drawn
    N(0, 1) from a third generator (seed + 3000) in the order q_nope, q_rope, v_new,
    k_new."""
    w = case.w
    L0 = case.seq_len.to(torch.int64) - n
    assert bool((L0 >= 0).all()), "every sequence must hold at least n tokens"
    g = torch.Generator().manual_seed(w.seed + 3000)
    qd = _dt(w.q_dtype)
    q_nope = torch.randn((w.B, n, w.H, w.d_n), generator=g, dtype=torch.float32).to(qd)
    q_rope = torch.randn((w.B, n, w.H, w.d_r), generator=g, dtype=torch.float32).to(qd)
    v_new = torch.randn((w.B, n, w.G, w.d_h), generator=g, dtype=torch.float32)
    k_new = torch.randn((w.B, n, w.d_r), generator=g, dtype=torch.float32)
    return Chunk(n=n, L0=L0.to(torch.int32), q_nope=q_nope, q_rope=q_rope, v_new=v_new,
                 k_new=k_new)
