"""Python binding of libgva.so -- Grouped Value Attention decode on a B300 (sm_103a).

Argument marshalling only: every function here has the name of a C entry point in
``include/gva.h``, checks that the torch tensors it is handed have the device,
dtype and layout the C ABI documents, and passes their data pointers and the
current CUDA stream.  All arithmetic runs in the library's CUDA kernels; there is
no CPU or PyTorch fallback.  Importing fails when ``libgva.so`` is missing.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgva.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'` "
        "or `python -m value_only_kv_gva_b300._build`")

_lib = ctypes.CDLL(LIB_PATH)

# --------------------------------------------------------------------------- #
# C structs
# --------------------------------------------------------------------------- #
GVA_OK, GVA_ERR_ARG, GVA_ERR_UNSUPPORTED, GVA_ERR_CUDA, GVA_ERR_WORKSPACE, \
    GVA_ERR_DEVICE_CHECK = 0, -1, -2, -3, -4, -5
GVA_DEV_OK, GVA_DEV_BAD_LENGTH, GVA_DEV_BAD_PAGE, GVA_DEV_BAD_POSITION, \
    GVA_DEV_TIMEOUT = 0, 1, 2, 3, 4
GVA_F32, GVA_BF16 = 0, 1
LAYOUTS = {"contiguous": 0, "ragged": 1, "paged": 2}
PATHS = {"auto": 0, "simt": 1, "mma": 2}


class gva_dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("G", ctypes.c_int),
                ("d_h", ctypes.c_int), ("d_n", ctypes.c_int), ("d_r", ctypes.c_int),
                ("cache_dtype", ctypes.c_int), ("q_dtype", ctypes.c_int)]


class gva_rows(ctypes.Structure):
    _fields_ = [("layout", ctypes.c_int), ("num_rows", ctypes.c_longlong),
                ("T_cap", ctypes.c_longlong), ("offsets", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("max_pages", ctypes.c_int),
                ("page_size", ctypes.c_int)]


class gva_cache(ctypes.Structure):
    _fields_ = [("rows", gva_rows), ("V", ctypes.c_void_p), ("K_rope", ctypes.c_void_p)]


class gva_kv_cache(ctypes.Structure):
    _fields_ = [("rows", gva_rows), ("K", ctypes.c_void_p), ("V", ctypes.c_void_p)]


class gva_mla_dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("d_c", ctypes.c_int),
                ("d_n", ctypes.c_int), ("d_r", ctypes.c_int), ("d_h", ctypes.c_int),
                ("cache_dtype", ctypes.c_int), ("q_dtype", ctypes.c_int)]


class gva_layer_args(ctypes.Structure):
    _fields_ = [("v_new", ctypes.c_void_p), ("k_rope_new", ctypes.c_void_p),
                ("q_nope", ctypes.c_void_p), ("q_rope", ctypes.c_void_p), ("M", ctypes.c_void_p),
                ("cache", gva_cache), ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p)]


class gva_prefill_layer_args(ctypes.Structure):
    _fields_ = [("q_nope", ctypes.c_void_p), ("q_rope", ctypes.c_void_p), ("M", ctypes.c_void_p),
                ("v_new", ctypes.c_void_p), ("k_rope_new", ctypes.c_void_p),
                ("cache", gva_cache), ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p)]


class gva_decode_opts(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("num_ctas", ctypes.c_int), ("flags", ctypes.c_int),
                ("q_norm_eps", ctypes.c_float), ("q_norm_gain", ctypes.c_void_p)]


GVA_FLAG_QUERY_RMSNORM = 1


_P, _I, _F, _D, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_size_t
_PD, _PC = ctypes.POINTER(gva_dims), ctypes.POINTER(gva_cache)
_PKV, _PO = ctypes.POINTER(gva_kv_cache), ctypes.POINTER(gva_decode_opts)

_lib.gva_status_string.restype = ctypes.c_char_p
_lib.gva_status_string.argtypes = [_I]
_lib.gva_abi_version.restype = _I
_lib.gva_num_sms.restype = _I
_lib.gva_rope_table_fill.argtypes = [_P, _I, _I, _D]
_lib.gva_absorb_query.argtypes = [_P, _PD, _P, _P, _P, _P, _P, _I, _F, _P, _P]
_lib.gva_absorb_query_ex.argtypes = _lib.gva_absorb_query.argtypes + [ctypes.c_void_p]
_lib.gva_append_cache.argtypes = [_P, _PD, _P, _P, _P, _P, _PC, _P, _I]
_lib.gva_decode_workspace_size.restype = _Z
_lib.gva_decode_workspace_size.argtypes = [_PD]
_lib.gva_decode_attention.argtypes = [_P, _PD, _P, _P, _P, _P, _PC, _P, _I, _F, _P, _P, _P, _Z]
_lib.gva_decode_attention_ex.argtypes = _lib.gva_decode_attention.argtypes + [_PO]
_lib.gva_gqa_decode_attention.argtypes = [_P, _PD, _P, _P, _PKV, _F, _P, _P, _P, _Z, _PO]
_lib.gva_get_device_status.argtypes = [ctypes.POINTER(_I)]
_lib.gva_last_cuda_error.restype = _I
_lib.gva_decode_attention_static.argtypes = [_P, _PD, _P, _P, _P, _P, _PC, _P, _I, _F, _P, _P]
_lib.gva_read_probe.argtypes = [_P, _P, _Z, _P]
_lib.gva_selftest_bounded_wait.argtypes = [_P, ctypes.c_uint]
_lib.gva_prefill_workspace_size.restype = _Z
_lib.gva_prefill_workspace_size.argtypes = [_PD, _I, ctypes.POINTER(gva_rows)]
_lib.gva_mla_workspace_size.restype = _Z
_lib.gva_mla_workspace_size.argtypes = [ctypes.POINTER(gva_mla_dims)]
_lib.gva_mla_decode_attention.argtypes = [_P, ctypes.POINTER(gva_mla_dims), _P, _P, _P, _P, _P,
                                          _PC, _P, _I, _F, _P, _P, _P, _Z]
_lib.gva_rope_keys_workspace_size.restype = _Z
_lib.gva_rope_keys_workspace_size.argtypes = [_PD]
_lib.gva_rope_keys_decode_attention.argtypes = [_P, _PD, _P, _P, _P, _PC, _P, _I, _F, _P, _P,
                                                _P, _Z]
_lib.gva_decode_step.argtypes = [_P, _PD, _I, ctypes.POINTER(gva_layer_args), _P, _P, _P, _I,
                                 _F, _P, _Z, _PO]
_lib.gva_step_plan_create.argtypes = [_PD, _I, ctypes.POINTER(gva_layer_args), _P, _P, _P, _I,
                                      _F, _P, _Z, _PO, ctypes.POINTER(ctypes.c_void_p)]
_lib.gva_step_plan_launch.argtypes = [_P, _P]
_lib.gva_prefill_plan_create.argtypes = [_PD, _I, _I, ctypes.POINTER(gva_prefill_layer_args), _P,
                                         _P, _I, _F, _P, _Z, _PO, ctypes.POINTER(ctypes.c_void_p)]
_lib.gva_step_plan_destroy.argtypes = [_P]
_lib.gva_prefill_attention.argtypes = [_P, _PD, _I, _P, _P, _P, _P, _P, _P, _PC, _P, _I, _F,
                                       _P, _P, _P, _Z, _PO]

EXPORTS = ["gva_status_string", "gva_abi_version", "gva_num_sms", "gva_rope_table_fill",
           "gva_absorb_query", "gva_append_cache", "gva_decode_workspace_size",
           "gva_decode_attention", "gva_decode_attention_ex", "gva_gqa_decode_attention",
           "gva_get_device_status", "gva_last_cuda_error", "gva_decode_attention_static",
           "gva_read_probe", "gva_absorb_query_ex", "gva_prefill_workspace_size",
           "gva_prefill_attention", "gva_mla_workspace_size", "gva_mla_decode_attention",
           "gva_rope_keys_workspace_size", "gva_rope_keys_decode_attention",
           "gva_selftest_bounded_wait", "gva_decode_step", "gva_step_plan_create",
           "gva_step_plan_launch", "gva_step_plan_destroy", "gva_prefill_plan_create"]


class GvaError(RuntimeError):
    def __init__(self, status: int, what: str):
        extra = ""
        if status == GVA_ERR_CUDA:
            extra = f", cudaError {int(_lib.gva_last_cuda_error())}"
        super().__init__(f"{what}: {gva_status_string(status)} ({status}{extra})")
        self.status = status


def _check(status: int, what: str) -> None:
    if status != GVA_OK:
        raise GvaError(status, what)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return GVA_F32
    if t.dtype == torch.bfloat16:
        return GVA_BF16
    raise TypeError(f"dtype {t.dtype} is not fp32 or bf16")


def _ptr(t, dtype=None, what="tensor"):
    """Device pointer of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


_ELEM_DT = {GVA_F32: torch.float32, GVA_BF16: torch.bfloat16}


def _need(t, n: int, what: str, dtype=None) -> None:
    """The C call reads or writes n elements of `t`: refuse a smaller tensor (or one of
    another dtype than the dims declare) before any device memory is touched."""
    if t is None:
        return
    if dtype is not None and t.dtype != dtype:
        raise GvaError(GVA_ERR_ARG, f"{what}: dtype {t.dtype}, the dims declare {dtype}")
    if t.numel() < n:
        raise GvaError(GVA_ERR_ARG, f"{what}: {t.numel()} elements, the call touches {n}")


def _check_rows(rows, B: int) -> None:
    if rows.offsets is not None:
        _need(rows.offsets, B + 1, "offsets")
    if rows.block_table is not None and rows.block_table.shape[0] < B:
        raise GvaError(GVA_ERR_ARG, f"block_table: {rows.block_table.shape[0]} rows < B = {B}")


def _check_cache(dims, cache) -> None:
    """V [num_rows, G, d_h] and K_rope [num_rows, d_r] in the cache dtype."""
    n = int(cache.rows.num_rows)
    _need(cache.V, n * dims.G * dims.d_h, "V", _ELEM_DT.get(dims.cache_dtype))
    if dims.d_r:
        _need(cache.K_rope, n * dims.d_r, "K_rope", _ELEM_DT.get(dims.cache_dtype))
    _check_rows(cache.rows, dims.B)


def _check_tab(rope_tab, d_r: int) -> None:
    if d_r and rope_tab is not None:
        _need(rope_tab, int(rope_tab.shape[0]) * d_r, "rope_tab")


def _check_decode(dims, q_nope, q_rope, M, seq_len, cache, rope_tab, out, lse, per=1) -> None:
    """Sizes a GVA decode (per = 1) or a prefill of `per` queries per sequence touches."""
    B, H, qd = dims.B, dims.H, _ELEM_DT.get(dims.q_dtype)
    _need(q_nope, B * per * H * dims.d_n, "q_nope", qd)
    if dims.d_r:
        _need(q_rope, B * per * H * dims.d_r, "q_rope", qd)
    _need(M, H * dims.d_h * dims.d_n, "M")
    _need(seq_len, B, "seq_len")
    _check_cache(dims, cache)
    _check_tab(rope_tab, dims.d_r)
    _need(out, B * per * H * dims.d_h, "out")
    _need(lse, B * per * H, "lse")


# --------------------------------------------------------------------------- #
# argument holders
# --------------------------------------------------------------------------- #
@dataclass
class Dims:
    B: int
    H: int
    G: int
    d_h: int
    d_n: int = 0
    d_r: int = 0
    cache_dtype: int = GVA_BF16
    q_dtype: int = GVA_BF16

    def c(self) -> gva_dims:
        return gva_dims(self.B, self.H, self.G, self.d_h, self.d_n, self.d_r,
                        self.cache_dtype, self.q_dtype)


@dataclass
class Rows:
    """Where token j of sequence b is stored (gva_rows)."""
    layout: str
    num_rows: int
    T_cap: int = 0
    offsets: torch.Tensor | None = None       # int32 [B+1] on the device (ragged)
    block_table: torch.Tensor | None = None   # int32 [B, max_pages] on the device (paged)
    page_size: int = 0

    def c(self) -> gva_rows:
        r = gva_rows()
        r.layout = LAYOUTS[self.layout]
        r.num_rows = int(self.num_rows)
        r.T_cap = int(self.T_cap)
        r.offsets = _ptr(self.offsets, torch.int32, "offsets")
        r.block_table = _ptr(self.block_table, torch.int32, "block_table")
        r.max_pages = int(self.block_table.shape[1]) if self.block_table is not None else 0
        r.page_size = int(self.page_size)
        return r


@dataclass
class Cache:
    """GVA cache: V rows [G, d_h] and K_rope rows [d_r] on the device (gva_cache)."""
    rows: Rows
    V: torch.Tensor
    K_rope: torch.Tensor | None

    def c(self) -> gva_cache:
        return gva_cache(self.rows.c(), _ptr(self.V, None, "V"),
                         _ptr(self.K_rope, None, "K_rope") if self.K_rope is not None
                         and self.K_rope.numel() > 0 else None)


@dataclass
class KVCache:
    """GQA comparator cache: explicit K and V rows [G, d_h] (gva_kv_cache)."""
    rows: Rows
    K: torch.Tensor
    V: torch.Tensor

    def c(self) -> gva_kv_cache:
        return gva_kv_cache(self.rows.c(), _ptr(self.K, None, "K"), _ptr(self.V, None, "V"))


def _opts(path: str, num_ctas: int, q_norm=None) -> gva_decode_opts:
    """q_norm: None, or (gain, eps) for the query RMSNorm (gain: fp32 device tensor
    [d_n] or None for ones)."""
    if q_norm is None:
        return gva_decode_opts(PATHS[path], int(num_ctas), 0, 0.0, None)
    gain, eps = q_norm
    return gva_decode_opts(PATHS[path], int(num_ctas), GVA_FLAG_QUERY_RMSNORM, float(eps),
                           _ptr(gain, torch.float32, "q_norm gain"))


# --------------------------------------------------------------------------- #
# entry points (same names as the C ABI)
# --------------------------------------------------------------------------- #
def gva_status_string(status: int) -> str:
    return _lib.gva_status_string(int(status)).decode()


def gva_abi_version() -> int:
    return int(_lib.gva_abi_version())


def gva_num_sms() -> int:
    return int(_lib.gva_num_sms())


def gva_read_probe(buf, sink, stream=None) -> None:
    """Read every byte of the device tensor `buf` once (pure read stream) and fold its
    32-bit words by XOR into the int32 device tensor `sink` (one element)."""
    _check(_lib.gva_read_probe(_stream(stream), _ptr(buf, None, "buf"),
                               buf.numel() * buf.element_size(), _ptr(sink, torch.int32, "sink")),
           "gva_read_probe")


def gva_rope_table_fill(max_pos: int, d_r: int, base: float = 10000.0) -> torch.Tensor:
    """Host fp32 table [max_pos, d_r/2, 2] of (cos, sin)(p * base^(-2i/d_r))."""
    tab = torch.empty((max_pos, max(d_r // 2, 0), 2), dtype=torch.float32)
    ptr = ctypes.c_void_p(tab.data_ptr()) if tab.numel() else None
    _check(_lib.gva_rope_table_fill(ptr, int(max_pos), int(d_r), float(base)),
           "gva_rope_table_fill")
    return tab


def gva_last_cuda_error() -> int:
    return int(_lib.gva_last_cuda_error())


def gva_absorb_query(dims: Dims, q_nope, q_rope, M, seq_len, rope_tab, scale: float,
                     q_tilde, q_rope_rot, stream=None, q_norm=None) -> None:
    """gva_absorb_query / gva_absorb_query_ex (q_norm as in _opts)."""
    d = dims.c()
    o = _opts("auto", 0, q_norm)
    B, H, qd = dims.B, dims.H, _ELEM_DT.get(dims.q_dtype)
    _need(q_nope, B * H * dims.d_n, "q_nope", qd)
    if dims.d_r:
        _need(q_rope, B * H * dims.d_r, "q_rope", qd)
        _need(q_rope_rot, B * H * dims.d_r, "q_rope_rot")
    _need(M, H * dims.d_h * dims.d_n, "M")
    _need(seq_len, B, "seq_len")
    _check_tab(rope_tab, dims.d_r)
    _need(q_tilde, B * H * dims.d_h, "q_tilde")
    _check(_lib.gva_absorb_query_ex(
        _stream(stream), ctypes.byref(d), _ptr(q_nope, None, "q_nope"),
        _ptr(q_rope, None, "q_rope") if dims.d_r else None, _ptr(M, torch.float32, "M"),
        _ptr(seq_len, torch.int32, "seq_len"),
        _ptr(rope_tab, torch.float32, "rope_tab") if dims.d_r else None,
        int(rope_tab.shape[0]) if rope_tab is not None else 0, float(scale),
        _ptr(q_tilde, torch.float32, "q_tilde"),
        _ptr(q_rope_rot, torch.float32, "q_rope_rot") if dims.d_r else None,
        ctypes.byref(o)), "gva_absorb_query")


def _check_append(dims, v_new, k_rope_new, pos, seq_len_out, cache, rope_tab) -> None:
    B = dims.B
    _need(v_new, B * dims.G * dims.d_h, "v_new")
    if dims.d_r:
        _need(k_rope_new, B * dims.d_r, "k_rope_new")
    _need(pos, B, "pos")
    _need(seq_len_out, B, "seq_len_out")
    _check_cache(dims, cache)
    _check_tab(rope_tab, dims.d_r)


def gva_append_cache(dims: Dims, v_new, k_rope_new, pos, seq_len_out, cache: Cache,
                     rope_tab, stream=None) -> None:
    d = dims.c()
    cc = cache.c()
    _check_append(dims, v_new, k_rope_new, pos, seq_len_out, cache, rope_tab)
    _check(_lib.gva_append_cache(
        _stream(stream), ctypes.byref(d), _ptr(v_new, torch.float32, "v_new"),
        _ptr(k_rope_new, torch.float32, "k_rope_new") if dims.d_r else None,
        _ptr(pos, torch.int32, "pos"), _ptr(seq_len_out, torch.int32, "seq_len_out"),
        ctypes.byref(cc), _ptr(rope_tab, torch.float32, "rope_tab") if dims.d_r else None,
        int(rope_tab.shape[0]) if rope_tab is not None else 0), "gva_append_cache")


def gva_decode_workspace_size(dims: Dims) -> int:
    d = dims.c()
    return int(_lib.gva_decode_workspace_size(ctypes.byref(d)))


def gva_decode_attention(dims: Dims, q_nope, q_rope, M, seq_len, cache: Cache, rope_tab,
                         scale: float, out, lse, workspace, path: str = "auto",
                         num_ctas: int = 0, stream=None, q_norm=None) -> None:
    """gva_decode_attention_ex (q_norm as in _opts: the query RMSNorm variant)."""
    d = dims.c()
    cc = cache.c()
    o = _opts(path, num_ctas, q_norm)
    _check_decode(dims, q_nope, q_rope, M, seq_len, cache, rope_tab, out, lse)
    _check(_lib.gva_decode_attention_ex(
        _stream(stream), ctypes.byref(d), _ptr(q_nope, None, "q_nope"),
        _ptr(q_rope, None, "q_rope") if dims.d_r else None, _ptr(M, torch.float32, "M"),
        _ptr(seq_len, torch.int32, "seq_len"), ctypes.byref(cc),
        _ptr(rope_tab, torch.float32, "rope_tab") if dims.d_r else None,
        int(rope_tab.shape[0]) if rope_tab is not None else 0, float(scale),
        _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(workspace, None, "workspace"), int(workspace.numel() * workspace.element_size()),
        ctypes.byref(o)), "gva_decode_attention")


def gva_prefill_workspace_size(dims: Dims, n: int, rows: Rows) -> int:
    d, r = dims.c(), rows.c()
    return int(_lib.gva_prefill_workspace_size(ctypes.byref(d), int(n), ctypes.byref(r)))


def gva_prefill_attention(dims: Dims, q_nope, q_rope, M, L0, v_new, k_rope_new, cache: Cache,
                          rope_tab, scale: float, out, lse, workspace, path: str = "auto",
                          num_ctas: int = 0, stream=None, q_norm=None) -> None:
    """gva_prefill_attention: append the chunk q_nope.shape[1] = n tokens per sequence
    after L0[b] cached ones, then causal attention of each new token (q_nope
    [B, n, H, d_n], v_new [B, n, G, d_h], k_rope_new [B, n, d_r], out [B, n, H, d_h],
    lse [B, n, H]; q_norm as in _opts).  path "auto" takes the tensor-core prefill
    kernel where it applies; "simt" and "mma" run each query as a decode
    entry."""
    d = dims.c()
    cc = cache.c()
    o = _opts(path, num_ctas, q_norm)
    n = int(q_nope.shape[1])
    _check_decode(dims, q_nope, q_rope, M, L0, cache, rope_tab, out, lse, per=n)
    _need(v_new, dims.B * n * dims.G * dims.d_h, "v_new")
    if dims.d_r:
        _need(k_rope_new, dims.B * n * dims.d_r, "k_rope_new")
    _check(_lib.gva_prefill_attention(
        _stream(stream), ctypes.byref(d), n, _ptr(q_nope, None, "q_nope"),
        _ptr(q_rope, None, "q_rope") if dims.d_r else None, _ptr(M, torch.float32, "M"),
        _ptr(L0, torch.int32, "L0"), _ptr(v_new, torch.float32, "v_new"),
        _ptr(k_rope_new, torch.float32, "k_rope_new") if dims.d_r else None, ctypes.byref(cc),
        _ptr(rope_tab, torch.float32, "rope_tab") if dims.d_r else None,
        int(rope_tab.shape[0]) if rope_tab is not None else 0, float(scale),
        _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(workspace, None, "workspace"), int(workspace.numel() * workspace.element_size()),
        ctypes.byref(o)), "gva_prefill_attention")


class PreparedCall:
    """One C-ABI call with its arguments validated and marshalled once, for loops that
    repeat the same call on the same buffers (a decode step per layer): calling the
    object issues the C function directly.  The tensors are kept alive by the object;
    their contents may change between calls, their storage may not."""

    def __init__(self, fn, args, what, keep):
        self._fn, self._args, self._what, self._keep = fn, args, what, keep

    def __call__(self) -> None:
        _check(self._fn(*self._args), self._what)


def prepare_append_cache(dims: Dims, v_new, k_rope_new, pos, seq_len_out, cache: Cache,
                         rope_tab, stream=None) -> PreparedCall:
    """gva_append_cache with fixed arguments (see PreparedCall)."""
    d, cc = dims.c(), cache.c()
    _check_append(dims, v_new, k_rope_new, pos, seq_len_out, cache, rope_tab)
    args = (_stream(stream), ctypes.byref(d), _ptr(v_new, torch.float32, "v_new"),
            _ptr(k_rope_new, torch.float32, "k_rope_new") if dims.d_r else None,
            _ptr(pos, torch.int32, "pos"), _ptr(seq_len_out, torch.int32, "seq_len_out"),
            ctypes.byref(cc), _ptr(rope_tab, torch.float32, "rope_tab") if dims.d_r else None,
            int(rope_tab.shape[0]) if rope_tab is not None else 0)
    return PreparedCall(_lib.gva_append_cache, args, "gva_append_cache",
                        (d, cc, v_new, k_rope_new, pos, seq_len_out, cache, rope_tab))


def prepare_decode_attention(dims: Dims, q_nope, q_rope, M, seq_len, cache: Cache, rope_tab,
                             scale: float, out, lse, workspace, path: str = "auto",
                             num_ctas: int = 0, stream=None, q_norm=None) -> PreparedCall:
    """gva_decode_attention(_ex) with fixed arguments (see PreparedCall)."""
    d, cc, o = dims.c(), cache.c(), _opts(path, num_ctas, q_norm)
    _check_decode(dims, q_nope, q_rope, M, seq_len, cache, rope_tab, out, lse)
    args = (_stream(stream), ctypes.byref(d), _ptr(q_nope, None, "q_nope"),
            _ptr(q_rope, None, "q_rope") if dims.d_r else None, _ptr(M, torch.float32, "M"),
            _ptr(seq_len, torch.int32, "seq_len"), ctypes.byref(cc),
            _ptr(rope_tab, torch.float32, "rope_tab") if dims.d_r else None,
            int(rope_tab.shape[0]) if rope_tab is not None else 0, float(scale),
            _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"),
            _ptr(workspace, None, "workspace"), int(workspace.numel() * workspace.element_size()),
            ctypes.byref(o))
    return PreparedCall(_lib.gva_decode_attention_ex, args, "gva_decode_attention",
                        (d, cc, o, q_nope, q_rope, M, seq_len, cache, rope_tab, out, lse, workspace,
                         q_norm))


def _addr(t, dtype=None, what="tensor"):
    """Device address of a contiguous CUDA tensor as an int (None -> NULL), for a field
    of a C structure."""
    p = _ptr(t, dtype, what)
    return None if p is None else p.value


def prepare_decode_step(dims: Dims, layers, pos, seq_len, rope_tab, scale: float, workspace,
                        path: str = "auto", num_ctas: int = 0, stream=None,
                        q_norm=None) -> PreparedCall:
    """gva_decode_step with fixed arguments (see PreparedCall): one C call per step runs
    every layer's append (when the layer has "v_new") and decode.  `layers` is a list of
    dicts with the keys v_new, k_rope_new (optional), q_nope, q_rope, M, cache (Cache),
    out and lse (optional), as in gva_append_cache and gva_decode_attention."""
    d, o, arr = _step_layers(dims, layers, pos, seq_len, rope_tab, path, num_ctas, q_norm)
    args = (_stream(stream), ctypes.byref(d), len(layers), arr,
            _ptr(pos, torch.int32, "pos"), _ptr(seq_len, torch.int32, "seq_len"),
            _ptr(rope_tab, torch.float32, "rope_tab") if dims.d_r else None,
            int(rope_tab.shape[0]) if rope_tab is not None else 0, float(scale),
            _ptr(workspace, None, "workspace"), int(workspace.numel() * workspace.element_size()),
            ctypes.byref(o))
    return PreparedCall(_lib.gva_decode_step, args, "gva_decode_step",
                        (d, o, arr, list(layers), pos, seq_len, rope_tab, workspace, q_norm))


def _step_layers(dims, layers, pos, seq_len, rope_tab, path, num_ctas, q_norm):
    """Checked gva_dims, options and the gva_layer_args array of a decode step."""
    d, o = dims.c(), _opts(path, num_ctas, q_norm)
    arr = (gva_layer_args * len(layers))()
    for i, L in enumerate(layers):
        cache = L["cache"]
        _check_decode(dims, L["q_nope"], L.get("q_rope"), L["M"], seq_len, cache, rope_tab,
                      L["out"], L.get("lse"))
        if L.get("v_new") is not None:
            _check_append(dims, L["v_new"], L.get("k_rope_new"), pos, None, cache, rope_tab)
        a = arr[i]
        a.v_new = _addr(L.get("v_new"), torch.float32, "v_new")
        a.k_rope_new = _addr(L.get("k_rope_new"), torch.float32, "k_rope_new") if dims.d_r else None
        a.q_nope = _addr(L["q_nope"], None, "q_nope")
        a.q_rope = _addr(L.get("q_rope"), None, "q_rope") if dims.d_r else None
        a.M = _addr(L["M"], torch.float32, "M")
        a.cache = cache.c()
        a.out = _addr(L["out"], torch.float32, "out")
        a.lse = _addr(L.get("lse"), torch.float32, "lse")
    return d, o, arr


class StepPlan:
    """A decode step recorded once by gva_step_plan_create and replayed by launch(): the
    buffers given at creation stay in place (kept alive here); refresh their contents in
    place between launches."""

    def __init__(self, handle, keep):
        self._h, self._keep = handle, keep

    def launch(self, stream=None) -> None:
        if self._h is None:
            raise GvaError(GVA_ERR_ARG, "gva_step_plan_launch: the plan was closed")
        _check(_lib.gva_step_plan_launch(self._h, _stream(stream)), "gva_step_plan_launch")

    def close(self) -> None:
        """Release the plan (after its last launch has completed)."""
        if self._h is not None:
            _lib.gva_step_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def create_prefill_plan(dims: Dims, n: int, layers, L0, rope_tab, scale: float, workspace,
                        path: str = "auto", num_ctas: int = 0, q_norm=None) -> StepPlan:
    """gva_prefill_plan_create: a chunk of n tokens per sequence through every layer,
    recorded once.  `layers` is a list of dicts with the keys q_nope, q_rope, M, v_new,
    k_rope_new, cache (Cache), out and lse (optional), as in gva_prefill_attention."""
    d, o = dims.c(), _opts(path, num_ctas, q_norm)
    arr = (gva_prefill_layer_args * len(layers))()
    for i, L in enumerate(layers):
        cache = L["cache"]
        _check_decode(dims, L["q_nope"], L.get("q_rope"), L["M"], L0, cache, rope_tab,
                      L["out"], L.get("lse"), per=n)
        _need(L["v_new"], dims.B * n * dims.G * dims.d_h, "v_new")
        if dims.d_r:
            _need(L.get("k_rope_new"), dims.B * n * dims.d_r, "k_rope_new")
        a = arr[i]
        a.q_nope = _addr(L["q_nope"], None, "q_nope")
        a.q_rope = _addr(L.get("q_rope"), None, "q_rope") if dims.d_r else None
        a.M = _addr(L["M"], torch.float32, "M")
        a.v_new = _addr(L["v_new"], torch.float32, "v_new")
        a.k_rope_new = _addr(L.get("k_rope_new"), torch.float32, "k_rope_new") if dims.d_r else None
        a.cache = cache.c()
        a.out = _addr(L["out"], torch.float32, "out")
        a.lse = _addr(L.get("lse"), torch.float32, "lse")
    h = ctypes.c_void_p()
    _check(_lib.gva_prefill_plan_create(
        ctypes.byref(d), int(n), len(layers), arr, _ptr(L0, torch.int32, "L0"),
        _ptr(rope_tab, torch.float32, "rope_tab") if dims.d_r else None,
        int(rope_tab.shape[0]) if rope_tab is not None else 0, float(scale),
        _ptr(workspace, None, "workspace"), int(workspace.numel() * workspace.element_size()),
        ctypes.byref(o), ctypes.byref(h)), "gva_prefill_plan_create")
    return StepPlan(h, (list(layers), L0, rope_tab, workspace, q_norm))


def create_step_plan(dims: Dims, layers, pos, seq_len, rope_tab, scale: float, workspace,
                     path: str = "auto", num_ctas: int = 0, q_norm=None) -> StepPlan:
    """gva_step_plan_create (layers as in prepare_decode_step)."""
    d, o, arr = _step_layers(dims, layers, pos, seq_len, rope_tab, path, num_ctas, q_norm)
    h = ctypes.c_void_p()
    _check(_lib.gva_step_plan_create(
        ctypes.byref(d), len(layers), arr, _ptr(pos, torch.int32, "pos"),
        _ptr(seq_len, torch.int32, "seq_len"),
        _ptr(rope_tab, torch.float32, "rope_tab") if dims.d_r else None,
        int(rope_tab.shape[0]) if rope_tab is not None else 0, float(scale),
        _ptr(workspace, None, "workspace"), int(workspace.numel() * workspace.element_size()),
        ctypes.byref(o), ctypes.byref(h)), "gva_step_plan_create")
    return StepPlan(h, (list(layers), pos, seq_len, rope_tab, workspace, q_norm))


def gva_decode_step(dims: Dims, layers, pos, seq_len, rope_tab, scale: float, workspace,
                    path: str = "auto", num_ctas: int = 0, stream=None, q_norm=None) -> None:
    """gva_decode_step: every layer's append and decode from one C call (see
    prepare_decode_step for `layers`)."""
    prepare_decode_step(dims, layers, pos, seq_len, rope_tab, scale, workspace, path,
                        num_ctas, stream, q_norm)()


def gva_gqa_decode_attention(dims: Dims, q, seq_len, cache: KVCache, scale: float, out, lse,
                             workspace, path: str = "auto", num_ctas: int = 0,
                             stream=None) -> None:
    d = dims.c()
    cc = cache.c()
    o = _opts(path, num_ctas)
    B, H, n = dims.B, dims.H, int(cache.rows.num_rows)
    _need(q, B * H * dims.d_h, "q", _ELEM_DT.get(dims.q_dtype))
    _need(seq_len, B, "seq_len")
    _need(cache.K, n * dims.G * dims.d_h, "K", _ELEM_DT.get(dims.cache_dtype))
    _need(cache.V, n * dims.G * dims.d_h, "V", _ELEM_DT.get(dims.cache_dtype))
    _check_rows(cache.rows, B)
    _need(out, B * H * dims.d_h, "out")
    _need(lse, B * H, "lse")
    _check(_lib.gva_gqa_decode_attention(
        _stream(stream), ctypes.byref(d), _ptr(q, None, "q"),
        _ptr(seq_len, torch.int32, "seq_len"), ctypes.byref(cc), float(scale),
        _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(workspace, None, "workspace"), int(workspace.numel() * workspace.element_size()),
        ctypes.byref(o)), "gva_gqa_decode_attention")


@dataclass
class MlaDims:
    """gva_mla_dims: the MLA-shaped comparator (latent width d_c, output width d_h)."""
    B: int
    H: int
    d_c: int
    d_n: int
    d_r: int
    d_h: int
    cache_dtype: int = GVA_BF16
    q_dtype: int = GVA_BF16

    def c(self) -> gva_mla_dims:
        return gva_mla_dims(self.B, self.H, self.d_c, self.d_n, self.d_r, self.d_h,
                            self.cache_dtype, self.q_dtype)


def gva_mla_workspace_size(dims: MlaDims) -> int:
    d = dims.c()
    return int(_lib.gva_mla_workspace_size(ctypes.byref(d)))


def gva_mla_decode_attention(dims: MlaDims, q_nope, q_rope, W_uk, W_uv, seq_len, cache: Cache,
                             rope_tab, scale: float, out, lse, workspace, stream=None) -> None:
    """gva_mla_decode_attention: cache.V holds the latent rows [rows, d_c], cache.K_rope the
    shared positional keys; W_uk [H, d_c, d_n], W_uv [H, d_c, d_h] fp32; out [B, H, d_h]."""
    d = dims.c()
    cc = cache.c()
    B, H, qd = dims.B, dims.H, _ELEM_DT.get(dims.q_dtype)
    _need(q_nope, B * H * dims.d_n, "q_nope", qd)
    if dims.d_r:
        _need(q_rope, B * H * dims.d_r, "q_rope", qd)
        _need(cache.K_rope, int(cache.rows.num_rows) * dims.d_r, "K_rope",
              _ELEM_DT.get(dims.cache_dtype))
    _need(cache.V, int(cache.rows.num_rows) * dims.d_c, "latent rows", _ELEM_DT.get(dims.cache_dtype))
    _check_rows(cache.rows, B)
    _need(W_uk, H * dims.d_c * dims.d_n, "W_uk")
    _need(W_uv, H * dims.d_c * dims.d_h, "W_uv")
    _need(seq_len, B, "seq_len")
    _check_tab(rope_tab, dims.d_r)
    _need(out, B * H * dims.d_h, "out")
    _need(lse, B * H, "lse")
    _check(_lib.gva_mla_decode_attention(
        _stream(stream), ctypes.byref(d), _ptr(q_nope, None, "q_nope"),
        _ptr(q_rope, None, "q_rope") if dims.d_r else None, _ptr(W_uk, torch.float32, "W_uk"),
        _ptr(W_uv, torch.float32, "W_uv"), _ptr(seq_len, torch.int32, "seq_len"),
        ctypes.byref(cc), _ptr(rope_tab, torch.float32, "rope_tab") if dims.d_r else None,
        int(rope_tab.shape[0]) if rope_tab is not None else 0, float(scale),
        _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(workspace, None, "workspace"), int(workspace.numel() * workspace.element_size())),
        "gva_mla_decode_attention")


def mla_workspace(dims: MlaDims, device=None) -> torch.Tensor:
    n = gva_mla_workspace_size(dims)
    if n == 0:
        raise GvaError(GVA_ERR_ARG, "gva_mla_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def gva_selftest_bounded_wait(limit_us: int, stream=None) -> None:
    """One warp waits on an mbarrier nothing arrives on; after `limit_us` the wait gives
    up and the device status reads GVA_DEV_TIMEOUT (see gva.h)."""
    _check(_lib.gva_selftest_bounded_wait(_stream(stream), int(limit_us)),
           "gva_selftest_bounded_wait")


def gva_rope_keys_workspace_size(dims: Dims) -> int:
    d = dims.c()
    return int(_lib.gva_rope_keys_workspace_size(ctypes.byref(d)))


def gva_rope_keys_decode_attention(dims: Dims, q, M, seq_len, cache: Cache, rope_tab,
                                   scale: float, out, lse, workspace, stream=None) -> None:
    """gva_rope_keys_decode_attention: the variant with ordinary RoPE on the reconstructed
    key.  q [B, H, d_n] (the whole query), M [H, d_h, d_n] fp32, cache.V the value rows
    [rows, G, d_h] (cache.K_rope unused), rope_tab [max_pos, d_n/2, 2] over d_n (max_pos
    >= 128 and >= every length), dims.d_r = 0; out [B, H, d_h], lse [B, H] or None."""
    d = dims.c()
    cc = cache.c()
    B, H, qd = dims.B, dims.H, _ELEM_DT.get(dims.q_dtype)
    _need(q, B * H * dims.d_n, "q", qd)
    _need(M, H * dims.d_h * dims.d_n, "M")
    _need(seq_len, B, "seq_len")
    _check_rows(cache.rows, B)
    _need(cache.V, int(cache.rows.num_rows) * dims.G * dims.d_h, "V",
          _ELEM_DT.get(dims.cache_dtype))
    _check_tab(rope_tab, dims.d_n)
    _need(out, B * H * dims.d_h, "out")
    if lse is not None:
        _need(lse, B * H, "lse")
    _check(_lib.gva_rope_keys_decode_attention(
        _stream(stream), ctypes.byref(d), _ptr(q, None, "q"), _ptr(M, torch.float32, "M"),
        _ptr(seq_len, torch.int32, "seq_len"), ctypes.byref(cc),
        _ptr(rope_tab, torch.float32, "rope_tab"), int(rope_tab.shape[0]), float(scale),
        _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(workspace, None, "workspace"), int(workspace.numel() * workspace.element_size())),
        "gva_rope_keys_decode_attention")


def rope_keys_workspace(dims: Dims, device=None) -> torch.Tensor:
    n = gva_rope_keys_workspace_size(dims)
    if n == 0:
        raise GvaError(GVA_ERR_ARG, "gva_rope_keys_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def gva_decode_attention_static(dims: Dims, q_nope, q_rope, M, seq_len, cache: Cache, rope_tab,
                                scale: float, out, lse, stream=None) -> None:
    """gva_decode_attention for callers that cannot allocate device memory: the
    library's fixed device scratch array stands in for the workspace (see gva.h)."""
    d = dims.c()
    cc = cache.c()
    _check_decode(dims, q_nope, q_rope, M, seq_len, cache, rope_tab, out, lse)
    _check(_lib.gva_decode_attention_static(
        _stream(stream), ctypes.byref(d), _ptr(q_nope, None, "q_nope"),
        _ptr(q_rope, None, "q_rope") if dims.d_r else None, _ptr(M, torch.float32, "M"),
        _ptr(seq_len, torch.int32, "seq_len"), ctypes.byref(cc),
        _ptr(rope_tab, torch.float32, "rope_tab") if dims.d_r else None,
        int(rope_tab.shape[0]) if rope_tab is not None else 0, float(scale),
        _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse")),
        "gva_decode_attention_static")


def gva_get_device_status() -> int:
    """Read and clear the device status word (synchronises the device)."""
    code = ctypes.c_int(0)
    st = _lib.gva_get_device_status(ctypes.byref(code))
    if st not in (GVA_OK, GVA_ERR_DEVICE_CHECK):
        raise GvaError(st, "gva_get_device_status")
    return int(code.value)


def workspace(dims: Dims, device=None) -> torch.Tensor:
    """Allocate a decode workspace (uint8, 256-byte aligned by the caching allocator;
    scratch only, zero-filled for determinism of unused bytes)."""
    n = gva_decode_workspace_size(dims)
    if n == 0:
        raise GvaError(GVA_ERR_ARG, "gva_decode_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def prefill_workspace(dims: Dims, n: int, rows: Rows, device=None) -> torch.Tensor:
    """Allocate a zero-filled prefill workspace for chunks of n tokens per sequence."""
    size = gva_prefill_workspace_size(dims, n, rows)
    if size == 0:
        raise GvaError(GVA_ERR_ARG, "gva_prefill_workspace_size")
    return torch.zeros(size, dtype=torch.uint8, device=device or "cuda")
