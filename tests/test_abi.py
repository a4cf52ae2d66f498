"""The C ABI without a GPU: libgva.so loads, exports every entry point that
include/gva.h declares, and its host-only paths behave (RoPE table, status strings,
argument validation that returns before any CUDA call)."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gva.h")


@pytest.fixture(scope="module")
def gva():
    import __graft_entry__
    __graft_entry__.build()
    import value_only_kv_gva_b300 as m
    return m


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gva_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("gva_absorb_query", "gva_append_cache", "gva_decode_attention",
              "gva_gqa_decode_attention", "gva_decode_workspace_size", "gva_rope_table_fill",
              "gva_status_string", "gva_get_device_status"):
        assert n in names


def test_every_declared_symbol_is_exported(gva):
    out = subprocess.run(["nm", "-D", "--defined-only", gva.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (gva_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in declared_functions():
        assert hasattr(gva._lib, n)
    assert set(gva.EXPORTS) <= exported


def test_abi_version_and_status_strings(gva):
    assert gva.gva_abi_version() == 6
    for code in (0, -1, -2, -3, -4, -5, 1, 2, 3, 4):
        s = gva.gva_status_string(code)
        assert s and "unknown" not in s
    assert "unknown" in gva.gva_status_string(12345)


@pytest.mark.parametrize("max_pos,d_r", [(1, 2), (4096, 16), (300, 24), (8192, 8), (17, 32)])
def test_rope_table_matches_oracle_bitwise(gva, max_pos, d_r):
    """Two independent fills of the same definition (libm cos/sin in double, one fp32
    rounding) agree bit for bit."""
    tab = gva.gva_rope_table_fill(max_pos, d_r, 10000.0).numpy()
    ref = oracle.rope_table_f32(max_pos, d_r, 10000.0)
    assert tab.shape == ref.shape and np.array_equal(tab.view(np.uint32), ref.view(np.uint32))


def test_rope_table_rejects_bad_args(gva):
    lib = gva._lib
    buf = (ctypes.c_float * 64)()
    assert lib.gva_rope_table_fill(None, 4, 8, 10000.0) == gva.GVA_ERR_ARG
    assert lib.gva_rope_table_fill(buf, 0, 8, 10000.0) == gva.GVA_ERR_ARG
    assert lib.gva_rope_table_fill(buf, 4, 7, 10000.0) == gva.GVA_ERR_ARG
    assert lib.gva_rope_table_fill(buf, 4, 8, -1.0) == gva.GVA_ERR_ARG


def test_path_values_beyond_mma_rejected(gva):
    """Paths are AUTO, SIMT and MMA; any other value is an argument error."""
    lib = gva._lib
    d = _dims(gva)
    fake = ctypes.c_void_p(0x10000)
    cache = gva.gva_cache(gva.gva_rows(0, 1 << 20, 1024, None, None, 0, 0), fake, fake)
    for path in (3, -1):
        o = gva.gva_decode_opts(path, 0, 0, 0.0, None)
        st = lib.gva_decode_attention_ex(None, ctypes.byref(d), fake, fake, fake, fake,
                                         ctypes.byref(cache), fake, 100, ctypes.c_float(0.1),
                                         fake, None, fake, ctypes.c_size_t(1 << 30),
                                         ctypes.byref(o))
        assert st == gva.GVA_ERR_ARG


def test_wait_selftest_rejects_bad_limits(gva):
    assert gva._lib.gva_selftest_bounded_wait(None, 0) == gva.GVA_ERR_ARG
    assert gva._lib.gva_selftest_bounded_wait(None, 2000000) == gva.GVA_ERR_ARG


@pytest.mark.parametrize("bad", [dict(d_r=16), dict(d_n=3), dict(B=0), dict(H=16, G=3),
                                 dict(cache_dtype=7), dict(d_h=12)])
def test_rope_keys_invalid_dims_rejected_before_cuda(gva, bad):
    """The rotated-key decode checks its arguments before any CUDA call."""
    lib = gva._lib
    base = dict(d_r=0)
    base.update(bad)
    d = _dims(gva, **base)
    fake = ctypes.c_void_p(0x10000)
    cache = gva.gva_cache(gva.gva_rows(0, 1 << 20, 1024, None, None, 0, 0), fake, None)
    assert lib.gva_rope_keys_workspace_size(ctypes.byref(d)) == 0
    st = lib.gva_rope_keys_decode_attention(None, ctypes.byref(d), fake, fake, fake,
                                            ctypes.byref(cache), fake, 4096, ctypes.c_float(0.1),
                                            fake, None, fake, ctypes.c_size_t(1 << 30))
    assert st == gva.GVA_ERR_ARG


def _dims(gva, **kw):
    base = dict(B=2, H=16, G=4, d_h=64, d_n=64, d_r=16, cache_dtype=1, q_dtype=1)
    base.update(kw)
    return gva.gva_dims(**base)


@pytest.mark.parametrize("bad", [dict(G=5), dict(H=64, G=4), dict(d_h=48), dict(d_r=12),
                                 dict(d_n=4), dict(B=0), dict(cache_dtype=7), dict(B=5000)])
def test_invalid_dims_rejected_before_cuda(gva, bad):
    lib = gva._lib
    d = _dims(gva, **bad)
    fake = ctypes.c_void_p(0x10000)
    cache = gva.gva_cache(gva.gva_rows(0, 1 << 20, 1024, None, None, 0, 0), fake, fake)
    assert lib.gva_decode_workspace_size(ctypes.byref(d)) == 0
    st = lib.gva_decode_attention(None, ctypes.byref(d), fake, fake, fake, fake,
                                  ctypes.byref(cache), fake, 100, ctypes.c_float(0.1), fake,
                                  None, fake, ctypes.c_size_t(1 << 30))
    assert st == gva.GVA_ERR_ARG
    st = lib.gva_append_cache(None, ctypes.byref(d), fake, fake, fake, None,
                              ctypes.byref(cache), fake, 100)
    assert st == gva.GVA_ERR_ARG


def test_null_and_misaligned_pointers_rejected(gva):
    lib = gva._lib
    d = _dims(gva)
    fake = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10004)
    rows = gva.gva_rows(0, 2 * 1024, 1024, None, None, 0, 0)
    good = gva.gva_cache(rows, fake, fake)
    # NULL output
    assert lib.gva_decode_attention(None, ctypes.byref(d), fake, fake, fake, fake,
                                    ctypes.byref(good), fake, 100, ctypes.c_float(0.1), None,
                                    None, fake, ctypes.c_size_t(1 << 30)) == gva.GVA_ERR_ARG
    # misaligned output
    assert lib.gva_decode_attention(None, ctypes.byref(d), fake, fake, fake, fake,
                                    ctypes.byref(good), fake, 100, ctypes.c_float(0.1), odd,
                                    None, fake, ctypes.c_size_t(1 << 30)) == gva.GVA_ERR_ARG
    # contiguous rows smaller than B * T_cap
    short = gva.gva_cache(gva.gva_rows(0, 100, 1024, None, None, 0, 0), fake, fake)
    assert lib.gva_append_cache(None, ctypes.byref(d), fake, fake, fake, None,
                                ctypes.byref(short), fake, 100) == gva.GVA_ERR_ARG
    # paged with a page size that is not a multiple of 16
    paged = gva.gva_cache(gva.gva_rows(2, 640, 0, None, fake, 4, 40), fake, fake)
    assert lib.gva_append_cache(None, ctypes.byref(d), fake, fake, fake, None,
                                ctypes.byref(paged), fake, 100) == gva.GVA_ERR_ARG
    # ragged without offsets
    rag = gva.gva_cache(gva.gva_rows(1, 640, 0, None, None, 0, 0), fake, fake)
    assert lib.gva_append_cache(None, ctypes.byref(d), fake, fake, fake, None,
                                ctypes.byref(rag), fake, 100) == gva.GVA_ERR_ARG
    # positional key missing while d_r > 0
    nokr = gva.gva_cache(rows, fake, None)
    assert lib.gva_append_cache(None, ctypes.byref(d), fake, fake, fake, None,
                                ctypes.byref(nokr), fake, 100) == gva.GVA_ERR_ARG


@pytest.mark.parametrize("flags,eps", [(2, 0.0), (1 | 4, 0.0), (1, -1.0), (1, float("inf")),
                                       (1, float("nan"))])
def test_bad_option_flags_rejected_before_cuda(gva, flags, eps):
    """Only GVA_FLAG_QUERY_RMSNORM is a valid flag, and its eps is finite and >= 0."""
    lib = gva._lib
    d = _dims(gva)
    fake = ctypes.c_void_p(0x10000)
    cache = gva.gva_cache(gva.gva_rows(0, 2 * 1024, 1024, None, None, 0, 0), fake, fake)
    o = gva.gva_decode_opts(0, 0, flags, eps, None)
    st = lib.gva_decode_attention_ex(None, ctypes.byref(d), fake, fake, fake, fake,
                                     ctypes.byref(cache), fake, 100, ctypes.c_float(0.1), fake,
                                     None, fake, ctypes.c_size_t(1 << 30), ctypes.byref(o))
    assert st == gva.GVA_ERR_ARG
    st = lib.gva_absorb_query_ex(None, ctypes.byref(d), fake, fake, fake, fake, fake, 100,
                                 ctypes.c_float(0.1), fake, fake, ctypes.byref(o))
    assert st == gva.GVA_ERR_ARG


def test_prefill_arguments_rejected_before_cuda(gva):
    """Contiguous capacities that are not a multiple of 16, and ragged caches on a path
    other than the automatic one (the view paths), are not taken (GVA_ERR_UNSUPPORTED);
    an empty chunk or more than 4096 decode entries is an argument error.  (Whether the
    automatic path takes a ragged cache depends on the device's plan: GPU tests.)"""
    lib = gva._lib
    d = _dims(gva)
    fake = ctypes.c_void_p(0x10000)

    def call(rows, n, path=None):
        cache = gva.gva_cache(rows, fake, fake)
        o = None if path is None else ctypes.byref(gva.gva_decode_opts(path, 0, 0, 0.0, None))
        return lib.gva_prefill_attention(None, ctypes.byref(d), n, fake, fake, fake, fake, fake,
                                         fake, ctypes.byref(cache), fake, 100,
                                         ctypes.c_float(0.1), fake, None, fake,
                                         ctypes.c_size_t(1 << 30), o)

    contig = gva.gva_rows(0, 2 * 1024, 1024, None, None, 0, 0)
    ragged = gva.gva_rows(1, 640, 0, fake, None, 0, 0)
    for path in (gva.PATHS["simt"], gva.PATHS["mma"]):
        assert call(ragged, 4, path) == gva.GVA_ERR_UNSUPPORTED
    assert call(gva.gva_rows(0, 2 * 1000, 1000, None, None, 0, 0), 4) == gva.GVA_ERR_UNSUPPORTED
    assert call(contig, 0) == gva.GVA_ERR_ARG
    assert call(contig, 2049) == gva.GVA_ERR_ARG          # B = 2: 4098 entries
    for rows in (contig, gva.gva_rows(1, 640, 0, fake, None, 0, 0)):
        assert lib.gva_prefill_workspace_size(ctypes.byref(d), 0, ctypes.byref(rows)) == 0


def test_plain_c_consumer(gva, tmp_path):
    """libgva.so as a C library: a C program that includes only include/gva.h, compiled
    with gcc and linked against the library, runs its host-only checks."""
    src = os.path.join(ROOT, "tests", "c", "abi_host_check.c")
    exe = str(tmp_path / "abi_host_check")
    libdir = os.path.dirname(gva.LIB_PATH)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    src, "-o", exe, "-L", libdir, "-lgva", "-Wl,-rpath," + libdir, "-lm"],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def _documented_valid(B, H, G, d_h, d_n, d_r, cd, qd):
    """The support matrix include/gva.h states for gva_dims."""
    return (1 <= B <= 4096 and H >= 1 and G >= 1 and H % G == 0 and H // G <= 8
            and d_h in (32, 64, 128) and H * d_h <= 4096 and 8 <= d_n <= 256
            and d_n % 8 == 0 and d_r in (0, 8, 16, 24, 32) and cd in (0, 1) and qd in (0, 1))


def test_dims_validation_follows_the_header(gva):
    """Random shapes: the library refuses exactly those the header's support matrix
    excludes.  The probe is gva_prefill_attention on a ragged cache with the SIMT path,
    which returns before any CUDA call either way: GVA_ERR_ARG for unsupported dims,
    GVA_ERR_UNSUPPORTED (the view paths do not take ragged layouts) for supported ones."""
    from hypothesis import given, settings, strategies as st

    lib = gva._lib
    fake = ctypes.c_void_p(0x10000)
    rag = gva.gva_cache(gva.gva_rows(1, 640, 0, fake, None, 0, 0), fake, fake)
    simt = gva.gva_decode_opts(gva.PATHS["simt"], 0, 0, 0.0, None)

    seen = {gva.GVA_ERR_ARG: 0, gva.GVA_ERR_UNSUPPORTED: 0}

    # a supported shape, then zero, one or two fields replaced by values drawn from a
    # wider range (often unsupported), so that both outcomes are common
    wide = dict(B=st.sampled_from([-1, 0, 4097, 5000, 1, 4096]), G=st.integers(0, 20),
                r=st.sampled_from([0, 9, 10, 1, 8]), skew=st.just(1),
                d_h=st.sampled_from([16, 48, 96, 256, 32, 128]),
                d_n=st.sampled_from([-8, 0, 4, 12, 257, 264, 8, 256]),
                d_r=st.sampled_from([-8, 2, 12, 40, 0, 32]), cd=st.just(2), qd=st.just(2))

    @st.composite
    def shapes(draw):
        v = dict(B=draw(st.integers(1, 4096)), G=draw(st.integers(1, 8)),
                 r=draw(st.integers(1, 8)), skew=0,
                 d_h=draw(st.sampled_from([32, 64, 128])),
                 d_n=8 * draw(st.integers(1, 32)),
                 d_r=draw(st.sampled_from([0, 8, 16, 24, 32])),
                 cd=draw(st.sampled_from([0, 1])), qd=draw(st.sampled_from([0, 1])))
        for k in draw(st.lists(st.sampled_from(sorted(wide)), max_size=2)):
            v[k] = draw(wide[k])
        return v

    @settings(max_examples=600, deadline=None, derandomize=True)
    @given(v=shapes())
    def check(v):
        B, G, r, skew, d_h, d_n, d_r, cd, qd = (v[k] for k in ("B", "G", "r", "skew", "d_h",
                                                               "d_n", "d_r", "cd", "qd"))
        H = G * r + skew                  # skew 1 usually breaks H % G == 0
        d = gva.gva_dims(B, H, G, d_h, d_n, d_r, cd, qd)
        st_ = lib.gva_prefill_attention(None, ctypes.byref(d), 1, fake, fake, fake, fake, fake,
                                        fake, ctypes.byref(rag), fake, 100, ctypes.c_float(0.1),
                                        fake, None, fake, ctypes.c_size_t(1 << 30),
                                        ctypes.byref(simt))
        want = gva.GVA_ERR_UNSUPPORTED if _documented_valid(B, H, G, d_h, d_n, d_r, cd, qd) \
            else gva.GVA_ERR_ARG
        assert st_ == want, (B, H, G, d_h, d_n, d_r, cd, qd, st_)
        seen[want] += 1

    check()
    assert seen[gva.GVA_ERR_UNSUPPORTED] >= 20 and seen[gva.GVA_ERR_ARG] >= 20, seen


def test_decode_step_argument_checks(gva):
    """gva_decode_step refuses a negative layer count or a missing layer array before any
    CUDA call, and a step of no layers does nothing."""
    lib = gva._lib
    d = gva.Dims(2, 16, 4, 64, 64, 16).c()

    def step(n):
        return lib.gva_decode_step(None, ctypes.byref(d), n, None, None, None, None, 0, 1.0,
                                   None, 0, None)
    assert step(-1) == gva.GVA_ERR_ARG
    assert step(3) == gva.GVA_ERR_ARG
    assert step(0) == gva.GVA_OK


def test_step_plan_argument_checks(gva):
    """gva_step_plan_create refuses a missing output handle, an empty step or a missing
    layer array before any CUDA call; launch refuses a NULL plan; destroy accepts one."""
    lib = gva._lib
    d = gva.Dims(2, 16, 4, 64, 64, 16).c()
    h = ctypes.c_void_p()

    def create(n, out):
        return lib.gva_step_plan_create(ctypes.byref(d), n, None, None, None, None, 0, 1.0,
                                        None, 0, None, out)
    assert create(1, None) == gva.GVA_ERR_ARG
    assert create(0, ctypes.byref(h)) == gva.GVA_ERR_ARG and not h.value
    assert create(2, ctypes.byref(h)) == gva.GVA_ERR_ARG and not h.value
    assert lib.gva_step_plan_launch(None, None) == gva.GVA_ERR_ARG
    assert lib.gva_step_plan_destroy(None) == gva.GVA_OK

    def create_prefill(n, layers_n, out):
        return lib.gva_prefill_plan_create(ctypes.byref(d), n, layers_n, None, None, None, 0,
                                           1.0, None, 0, None, out)
    assert create_prefill(16, 1, None) == gva.GVA_ERR_ARG
    assert create_prefill(0, 1, ctypes.byref(h)) == gva.GVA_ERR_ARG and not h.value
    assert create_prefill(16, 0, ctypes.byref(h)) == gva.GVA_ERR_ARG and not h.value
    assert create_prefill(16, 1, ctypes.byref(h)) == gva.GVA_ERR_ARG and not h.value
