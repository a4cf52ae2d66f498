"""Plain fp64 CPU oracle for Grouped Value Attention (GVA) decode.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code with
the CUDA library in ``value_only_kv_gva_b300`` and never imports it.

The arithmetic lives in ``gva_oracle.c`` (plain C, fp64, OpenMP over (b, h)); this
module compiles it with gcc, loads it with ctypes and widens every input to fp64
exactly.  Function docstrings cite the page and section each one follows:

  [A] "GVA：KV 缓存里的 Key 其实可以不存——从 Value 里"现算"出来就行" (analysis page)
  [S] "Grouped Value Attention: Efficient KV Caching via On-Demand Key Reconstruction"
  [K] "KV Cache 优化（一）：从 MHA 到 MQA 与 GQA"
  [C] KV-cache compression survey, MHA -> MQA -> GQA -> MLA -> CSA/HCA
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gva_oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

GCC_FLAGS = ["-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile gva_oracle.c into liboracle.so next to it (no-op when up to date)."""
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _SO)
    return _SO


class _Rows(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int),
        ("T_cap", ctypes.c_longlong),
        ("offsets", ctypes.POINTER(ctypes.c_longlong)),
        ("block_table", ctypes.POINTER(ctypes.c_longlong)),
        ("max_pages", ctypes.c_int),
        ("page_size", ctypes.c_int),
    ]


_P = ctypes.c_void_p
_I = ctypes.c_int
_LL = ctypes.c_longlong
_D = ctypes.c_double


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            L.od_set_threads.argtypes = [_I]
            L.od_get_threads.restype = _I
            L.od_row.argtypes = [ctypes.POINTER(_Rows), _I, _LL]
            L.od_row.restype = _LL
            L.od_rope_theta.argtypes = [_I, _I, _D]
            L.od_rope_theta.restype = _D
            L.od_rotate.argtypes = [_P, _P, _I, _LL, _D]
            L.od_rope_table_f32.argtypes = [_P, _I, _I, _D]
            L.od_bf16_rne_array.argtypes = [_P, _P, _LL]
            L.od_absorb.argtypes = [_I] * 5 + [_P, _P, _P, _P, _D, _D, _P, _P]
            L.od_gva_decode.argtypes = ([_I] * 6 + [_P, _P, _P, _P, ctypes.POINTER(_Rows)]
                                        + [_P, _P, _I, _D, _D, _P, _P])
            L.od_gva_decode_explicit.argtypes = L.od_gva_decode.argtypes
            L.od_gqa_decode.argtypes = ([_I] * 4 + [_P, _P, ctypes.POINTER(_Rows)]
                                        + [_P, _P, _I, _D, _P, _P])
            L.od_append.argtypes = ([_I] * 4 + [_P, _P, _P, ctypes.POINTER(_Rows), _I,
                                                _P, _P, _P])
            L.od_rotate_keys_f64.argtypes = [_I, _I, _P, _P, _D, _P]
            L.od_query_rmsnorm.argtypes = [_I, _I, _I, _P, _P, _D, _P]
            L.od_gva_decode_rope_keys.argtypes = ([_I] * 5 + [_P, _P, _P, ctypes.POINTER(_Rows)]
                                                  + [_P, _I, _D, _D, _LL, _P, _P])
            L.od_mla_decode.argtypes = ([_I] * 6 + [_P, _P, _P, _P, _P, ctypes.POINTER(_Rows)]
                                        + [_P, _P, _I, _D, _D, _P, _P])
            _lib = L
        return _lib


def set_threads(n: int) -> None:
    lib().od_set_threads(int(n))


def get_threads() -> int:
    return int(lib().od_get_threads())


# --------------------------------------------------------------------------- #
# exact widening of inputs
# --------------------------------------------------------------------------- #
def _np(x):
    """torch tensor or array -> numpy (CPU); bf16 tensors come back as uint16 bits."""
    if hasattr(x, "detach"):
        import torch  # local: only to read tensors handed in
        t = x.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()
    return np.ascontiguousarray(x)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit pattern -> float64, exactly (the 16 bits are the top half of an fp32)."""
    u = bits.astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def f64(x) -> np.ndarray:
    """Any stored tensor (bf16 bits, fp32, fp64, int) -> contiguous float64, exactly."""
    a = _np(x)
    if a.dtype == np.uint16:
        return np.ascontiguousarray(bf16_bits_to_f64(a))
    return np.ascontiguousarray(a.astype(np.float64))


def _storage(x):
    """Cache storage for the C side: (array, is_bf16) without widening."""
    a = _np(x)
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a), 1
    if a.dtype == np.float32:
        return np.ascontiguousarray(a), 0
    raise TypeError(f"cache storage must be bf16 or fp32, got {a.dtype}")


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------------------- #
# storage-row descriptors
# --------------------------------------------------------------------------- #
@dataclass
class Rows:
    """Where logical token (b, j) lives in the row arrays ([K] §7: paging moves bytes,
    not maths).  kind: 'contiguous' (row = b*T_cap + j), 'ragged' (offsets[b] + j),
    'paged' (block_table[b][j // page_size] * page_size + j % page_size)."""
    kind: str
    T_cap: int = 0
    offsets: np.ndarray | None = None
    block_table: np.ndarray | None = None
    page_size: int = 0
    _keep: list = field(default_factory=list, repr=False)

    def c(self) -> _Rows:
        kinds = {"contiguous": 0, "ragged": 1, "paged": 2}
        r = _Rows()
        r.kind = kinds[self.kind]
        r.T_cap = int(self.T_cap)
        r.max_pages = 0
        r.page_size = int(self.page_size)
        if self.offsets is not None:
            off = np.ascontiguousarray(_np(self.offsets).astype(np.int64))
            self._keep.append(off)
            r.offsets = off.ctypes.data_as(ctypes.POINTER(_LL))
        if self.block_table is not None:
            bt = np.ascontiguousarray(_np(self.block_table).astype(np.int64))
            self._keep.append(bt)
            r.block_table = bt.ctypes.data_as(ctypes.POINTER(_LL))
            r.max_pages = int(bt.shape[1])
        return r

    def row(self, b: int, j: int) -> int:
        return int(lib().od_row(ctypes.byref(self.c()), int(b), int(j)))


# --------------------------------------------------------------------------- #
# RoPE and rounding
# --------------------------------------------------------------------------- #
def rope_theta(i: int, d_r: int, base: float) -> float:
    """theta_i = base^(-2i/d_r)  (reading of [A] "关键技巧二"; interleaved pairs)."""
    return float(lib().od_rope_theta(int(i), int(d_r), float(base)))


def rotate(x, p: int, base: float) -> np.ndarray:
    """Rot(p) x in fp64 on interleaved pairs (the relative rotation R_{j-t} of [A])."""
    xv = f64(x).reshape(-1)
    y = np.empty_like(xv)
    lib().od_rotate(_ptr(xv), _ptr(y), int(xv.size), int(p), float(base))
    return y


def rope_table_f32(max_pos: int, d_r: int, base: float) -> np.ndarray:
    """[max_pos, d_r/2, 2] fp32 table of (cos, sin)(p * theta_i), each rounded once."""
    tab = np.empty((max_pos, d_r // 2, 2), dtype=np.float32)
    if max_pos > 0 and d_r > 0:
        lib().od_rope_table_f32(_ptr(tab), int(max_pos), int(d_r), float(base))
    return tab


def bf16_rne(x) -> np.ndarray:
    """fp32 -> bf16 bits, round to nearest, ties to even."""
    a = np.ascontiguousarray(_np(x).astype(np.float32))
    out = np.empty(a.shape, dtype=np.uint16)
    lib().od_bf16_rne_array(_ptr(a), _ptr(out), int(a.size))
    return out


# --------------------------------------------------------------------------- #
# the method
# --------------------------------------------------------------------------- #
def query_rmsnorm(q_nope, gain=None, eps: float = 1e-6):
    """Per-head RMSNorm of the content query, fp64 ([A] 实验 / [S] results table,
    "scale-matched + query RMSNorm"; the formula is a reading, see od_query_rmsnorm):
    y = gain * x / sqrt(mean(x^2) + eps) over each head's d_n values."""
    x = f64(q_nope)
    B, H, d_n = x.shape
    y = np.empty_like(x)
    g = None if gain is None else np.ascontiguousarray(f64(gain).reshape(d_n))
    lib().od_query_rmsnorm(B, H, d_n, _ptr(x), _ptr(g) if g is not None else None,
                           float(eps), _ptr(y))
    return y


def absorb(q_nope, q_rope, M, seq_len, scale: float, base: float):
    """q~_h = scale * q_h^nope M_h^T and q^_h = scale * Rot(L_b - 1) q_h^rope
    ([A] "关键技巧一" eq. q_h k_{j,h}^T = q~_h v_{j,g(h)}^T; [S] "absorption")."""
    qn, qr, Mm = f64(q_nope), f64(q_rope), f64(M)
    B, H, d_n = qn.shape
    d_r = qr.shape[2]
    d_h = Mm.shape[1]
    sl = np.ascontiguousarray(_np(seq_len).astype(np.int64))
    qt = np.zeros((B, H, d_h))
    qh = np.zeros((B, H, max(d_r, 1)))
    lib().od_absorb(B, H, d_h, d_n, d_r, _ptr(qn), _ptr(qr), _ptr(Mm), _ptr(sl),
                    float(scale), float(base), _ptr(qt), _ptr(qh))
    return qt, qh[:, :, :d_r]


def _decode(fn, q_nope, q_rope, M, seq_len, rows: Rows, V, Kr, scale, base, G):
    qn, qr, Mm = f64(q_nope), f64(q_rope), f64(M)
    B, H, d_n = qn.shape
    d_r = qr.shape[2]
    d_h = Mm.shape[1]
    sl = np.ascontiguousarray(_np(seq_len).astype(np.int64))
    Vs, vb = _storage(V)
    if d_r > 0:
        Ks, kb = _storage(Kr)
        assert kb == vb, "V and K_rope share the cache dtype"
    else:
        Ks = np.zeros(1, dtype=Vs.dtype)
    out = np.zeros((B, H, d_h))
    lse = np.zeros((B, H))
    rc = rows.c()
    fn(B, H, G, d_h, d_n, d_r, _ptr(qn), _ptr(qr), _ptr(Mm), _ptr(sl), ctypes.byref(rc),
       _ptr(Vs), _ptr(Ks), vb, float(scale), float(base), _ptr(out), _ptr(lse))
    return out, lse


def gva_decode(q_nope, q_rope, M, seq_len, rows: Rows, V, Kr, scale: float,
               base: float, G: int):
    """GVA decode, absorbed path: z_j = scale*(q~.v_{j,g} + Rot(t)q_rope . k_rope_j),
    out = softmax(z) V_g, lse = logsumexp(z), t = L_b - 1
    ([A] "关键技巧一/二"; [S]; [K] §1 for append-then-attend).
    V rows are [G, d_h], K_rope rows are [d_r]; storage bf16 or fp32."""
    return _decode(lib().od_gva_decode, q_nope, q_rope, M, seq_len, rows, V, Kr,
                   scale, base, G)


def gva_decode_explicit(q_nope, q_rope, M, seq_len, rows: Rows, V, Kr, scale: float,
                        base: float, G: int):
    """GVA decode with the content key materialised, K_h = V_{g(h)} M_h ([A] eq.),
    concatenated with the rotated positional key, then ordinary softmax attention."""
    return _decode(lib().od_gva_decode_explicit, q_nope, q_rope, M, seq_len, rows, V,
                   Kr, scale, base, G)


def gva_decode_rope_keys(q, M, seq_len, rows: Rows, V, scale: float, base: float, G: int,
                         pos_offset: int = 0):
    """GVA with ordinary RoPE on the reconstructed key (the non-absorbable variant; [S]
    results discussion, [A] 关键技巧二; formula is a reading, see od_gva_decode_rope_keys):
    z_j = scale * (Rot(t) q_h) . (Rot(j) v_{j,g} M_h), out = softmax(z) V_g."""
    qq, Mm = f64(q), f64(M)
    B, H, d_n = qq.shape
    d_h = Mm.shape[1]
    sl = np.ascontiguousarray(_np(seq_len).astype(np.int64))
    Vs, vb = _storage(V)
    out = np.zeros((B, H, d_h))
    lse = np.zeros((B, H))
    rc = rows.c()
    lib().od_gva_decode_rope_keys(B, H, G, d_h, d_n, _ptr(qq), _ptr(Mm), _ptr(sl),
                                  ctypes.byref(rc), _ptr(Vs), vb, float(scale), float(base),
                                  int(pos_offset), _ptr(out), _ptr(lse))
    return out, lse


def mla_decode(q_nope, q_rope, Wuk, Wuv, seq_len, rows: Rows, C, Kr, scale: float,
               base: float):
    """MLA-shaped decode, explicit path ([A] 问题 / 对 MLA 的优势: T(d_c + d_r) cache;
    [C] 3.1.2-3.1.3): keys [c_j Wuk_h ; k_rope_j], values c_j Wuv_h, query
    [q_nope ; Rot(t) q_rope].  C rows [d_c], K_rope rows [d_r] (shared); Wuk [H, d_c, d_n],
    Wuv [H, d_c, d_h]."""
    qn, qr = f64(q_nope), f64(q_rope)
    Wk, Wv = f64(Wuk), f64(Wuv)
    B, H, d_n = qn.shape
    d_r = qr.shape[2]
    d_c, d_h = Wk.shape[1], Wv.shape[2]
    sl = np.ascontiguousarray(_np(seq_len).astype(np.int64))
    Cs, cb = _storage(C)
    if d_r > 0:
        Ks, kb = _storage(Kr)
        assert kb == cb, "C and K_rope share the cache dtype"
    else:
        Ks = np.zeros(1, dtype=Cs.dtype)
    out = np.zeros((B, H, d_h))
    lse = np.zeros((B, H))
    rc = rows.c()
    lib().od_mla_decode(B, H, d_c, d_n, d_h, d_r, _ptr(qn), _ptr(qr), _ptr(Wk), _ptr(Wv),
                        _ptr(sl), ctypes.byref(rc), _ptr(Cs), _ptr(Ks), cb, float(scale),
                        float(base), _ptr(out), _ptr(lse))
    return out, lse


def gva_prefill(q_nope, q_rope, M, L0, rows, V, Kr, scale: float, base: float, G: int):
    """Chunked prefill, causal ([K] §1: every new token attends to all history up to and
    including itself; [S] notes that prefill stays matrix-heavy).  The cache already
    holds the chunk: sequence b's n new tokens sit at positions L0[b] .. L0[b] + n - 1.
    `rows` is the cache's row map: an int T_cap (contiguous), or a Rows of any kind.
    Query i of sequence b (position p = L0[b] + i) is scored exactly as a decode query
    of a sequence of length p + 1 (absorbed content part, positional query rotated by
    p).  q_nope [B, n, H, d_n], q_rope [B, n, H, d_r]; returns out [B, n, H, d_h],
    lse [B, n, H].  Each query is one entry of a decode over a view of the same
    storage (one entry per (b, i), all reading sequence b's rows)."""
    qn, qr = f64(q_nope), f64(q_rope)
    B, n, H, d_n = qn.shape
    d_r = qr.shape[3]
    L0 = np.asarray(_np(L0), dtype=np.int64)
    lens = (L0[:, None] + np.arange(n)[None, :] + 1).reshape(-1)
    if isinstance(rows, Rows) and rows.kind == "paged":
        bt = np.asarray(_np(rows.block_table), dtype=np.int64)
        assert np.all(L0 + n <= bt.shape[1] * rows.page_size), "the chunk must fit the capacity"
        R = Rows("paged", block_table=np.repeat(bt[:B], n, axis=0), page_size=rows.page_size)
    elif isinstance(rows, Rows) and rows.kind == "ragged":
        offs = np.asarray(_np(rows.offsets), dtype=np.int64)
        assert np.all(L0 + n <= offs[1:B + 1] - offs[:B]), "the chunk must fit the capacity"
        R = Rows("ragged", offsets=np.append(np.repeat(offs[:B], n), 0))
    else:
        T_cap = rows.T_cap if isinstance(rows, Rows) else int(rows)
        assert np.all(L0 + n <= T_cap), "the chunk must fit the capacity"
        R = Rows("ragged", offsets=np.append(np.repeat(np.arange(B, dtype=np.int64) * T_cap, n), 0))
    out, lse = gva_decode(qn.reshape(B * n, H, d_n), qr.reshape(B * n, H, d_r), M, lens, R, V,
                          Kr, scale, base, G)
    return out.reshape(B, n, H, -1), lse.reshape(B, n, H)


def gqa_decode(q, seq_len, rows: Rows, K, V, scale: float, G: int):
    """GQA decode, head_h = softmax(scale * q_h K_g^T) V_g ([K] §4; [C] §2.2)."""
    qq = f64(q)
    B, H, d_h = qq.shape
    sl = np.ascontiguousarray(_np(seq_len).astype(np.int64))
    Ks, kb = _storage(K)
    Vs, vb = _storage(V)
    assert kb == vb
    out = np.zeros((B, H, d_h))
    lse = np.zeros((B, H))
    rc = rows.c()
    lib().od_gqa_decode(B, H, G, d_h, _ptr(qq), _ptr(sl), ctypes.byref(rc), _ptr(Ks),
                        _ptr(Vs), vb, float(scale), _ptr(out), _ptr(lse))
    return out, lse


def append(v_new, k_new, pos, rows: Rows, V, Kr, rope_tab):
    """Write token b at logical position pos[b]: V[row] = v_new[b] (one rounding to the
    cache dtype), K_rope[row] = Rot(pos[b]) k_new[b] decided in fp32 with a fixed
    operation order and no FMA, then rounded once ([S]: cached already rotated).
    V/Kr are numpy storage arrays (uint16 bf16 bits or float32), updated in place."""
    vn = np.ascontiguousarray(_np(v_new).astype(np.float32))
    kn = np.ascontiguousarray(_np(k_new).astype(np.float32))
    B, G, d_h = vn.shape
    d_r = kn.shape[1] if kn.ndim == 2 else 0
    ps = np.ascontiguousarray(_np(pos).astype(np.int64))
    assert V.flags["C_CONTIGUOUS"] and (d_r == 0 or Kr.flags["C_CONTIGUOUS"])
    is_bf16 = 1 if V.dtype == np.uint16 else 0
    tab = np.ascontiguousarray(np.asarray(rope_tab, dtype=np.float32))
    rc = rows.c()
    lib().od_append(B, G, d_h, d_r, _ptr(vn), _ptr(kn), _ptr(ps), ctypes.byref(rc),
                    is_bf16, _ptr(V), _ptr(Kr) if d_r > 0 else None, _ptr(tab))


def rotate_keys_f64(k_new, pos, base: float) -> np.ndarray:
    """Rot(pos[b]) k_new[b] in fp64 (no fp32 rounding), shape [B, d_r]."""
    kn = f64(k_new)
    B, d_r = kn.shape
    ps = np.ascontiguousarray(_np(pos).astype(np.int64))
    out = np.zeros_like(kn)
    lib().od_rotate_keys_f64(B, d_r, _ptr(kn), _ptr(ps), float(base), _ptr(out))
    return out


# --------------------------------------------------------------------------- #
# cache accounting  ([A] "缓存账本"; [K] §2, §3, §5)
# --------------------------------------------------------------------------- #
def n_gva(T: int, G: int, d_h: int, d_r: int) -> int:
    """Persistent GVA cache scalars per layer and sequence: N = T G d_h + T d_r."""
    return T * G * d_h + T * d_r


def n_gqa(T: int, G: int, d_h: int) -> int:
    """Matched GQA cache scalars: N = 2 T G d_h."""
    return 2 * T * G * d_h


def n_mha(T: int, H: int, d_h: int) -> int:
    """MHA cache scalars: N = 2 T H d_h."""
    return 2 * T * H * d_h


def gva_over_gqa(G: int, d_h: int, d_r: int) -> float:
    """N_GVA / N_GQA = 1/2 + d_r / (2 G d_h)."""
    return 0.5 + d_r / (2.0 * G * d_h)


def kv_bytes(L: int, B: int, T: int, n_kv: int, d_h: int, elem_bytes: int) -> int:
    """M_KV = 2 L B T N_KV D_h x bytes ([K] opening formula)."""
    return 2 * L * B * T * n_kv * d_h * elem_bytes
