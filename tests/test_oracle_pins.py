"""Pins of the fp64 oracle to things other than itself: values printed on the pages,
closed forms, invariants, and special cases that reduce to a library routine
(torch's scaled_dot_product_attention / logsumexp in fp64, torch's bf16 cast,
numpy's complex exponential).  CPU only."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from gva_inputs import make_case, workload

BASE = 10000.0


def _contig(B, T):
    return oracle.Rows("contiguous", T_cap=T)


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _rot_complex(x, p, base=BASE):
    """Rotation through complex multiplication by exp(i p theta_k): an independent
    route to the interleaved-pair RoPE reading."""
    x = np.asarray(x, dtype=np.float64)
    d_r = x.shape[-1]
    z = x[..., 0::2] + 1j * x[..., 1::2]
    theta = base ** (-(2.0 * np.arange(d_r // 2)) / d_r)
    w = z * np.exp(1j * p * theta)
    y = np.empty_like(x)
    y[..., 0::2] = w.real
    y[..., 1::2] = w.imag
    return y


# --------------------------------------------------------------------------- #
# absorption identity (GVA analysis page, 关键技巧一: exact, not an approximation)
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("shape", [
    dict(B=1, H=4, G=2, d_h=32, d_n=32, d_r=8, T=64),      # the tiny workload's shape
    dict(B=2, H=16, G=4, d_h=64, d_n=64, d_r=16, T=150),    # 350M-class head shape
    dict(B=3, H=6, G=3, d_h=16, d_n=24, d_r=0, T=33),       # d_n != d_h, no RoPE
    dict(B=2, H=8, G=1, d_h=8, d_n=4, d_r=24, T=17),        # MQA-like grouping
])
def test_absorbed_equals_explicit(shape):
    B, H, G, d_h, d_n, d_r, T = (shape[k] for k in ("B", "H", "G", "d_h", "d_n", "d_r", "T"))
    s = 1 / math.sqrt(d_n + d_r)
    V = _f32(_rand((B * T, G, d_h), 1))
    Kr = _f32(_rand((B * T, d_r), 2))
    qn = _rand((B, H, d_n), 3)
    qr = _rand((B, H, d_r), 4)
    M = _rand((H, d_h, d_n), 5, 1 / math.sqrt(d_h))
    lens = np.array([T - b for b in range(B)])
    rows = _contig(B, T)
    o1, l1 = oracle.gva_decode(qn, qr, M, lens, rows, V, Kr, s, BASE, G)
    o2, l2 = oracle.gva_decode_explicit(qn, qr, M, lens, rows, V, Kr, s, BASE, G)
    assert np.max(np.abs(o1 - o2)) <= 1e-12
    assert np.max(np.abs(l1 - l2)) <= 1e-12


def test_absorbed_equals_explicit_on_tiny_workload():
    c = make_case(workload("tiny"))
    w = c.w
    rows = oracle.Rows("contiguous", T_cap=c.T_cap)
    o1, l1 = oracle.gva_decode(c.q_nope, c.q_rope, c.M, c.seq_len, rows, c.V, c.Kr,
                               w.scale, w.base, w.G)
    o2, l2 = oracle.gva_decode_explicit(c.q_nope, c.q_rope, c.M, c.seq_len, rows, c.V,
                                        c.Kr, w.scale, w.base, w.G)
    assert np.max(np.abs(o1 - o2)) <= 1e-12 and np.max(np.abs(l1 - l2)) <= 1e-12


def test_absorb_matches_decode_scores():
    """q~ from od_absorb dotted with the cache gives the same output as the decode."""
    B, H, G, d_h, d_n, d_r, T = 2, 4, 2, 8, 6, 4, 9
    s = 0.3
    qn, qr = _rand((B, H, d_n), 1), _rand((B, H, d_r), 2)
    M = _rand((H, d_h, d_n), 3)
    lens = np.array([T, 5])
    qt, qh = oracle.absorb(qn, qr, M, lens, s, BASE)
    # library matmul route to q~ = s * q_nope M_h^T and q^ = s * Rot(t) q_rope
    for b in range(B):
        for h in range(H):
            ref = s * (M[h] @ qn[b, h])
            assert np.allclose(qt[b, h], ref, rtol=0, atol=1e-13)
            assert np.allclose(qh[b, h], s * _rot_complex(qr[b, h], lens[b] - 1),
                               rtol=0, atol=1e-13)


# --------------------------------------------------------------------------- #
# degenerate cases that reduce to a textbook attention
# --------------------------------------------------------------------------- #
def _sdpa(q, k, v, scale):
    """q [H, d], k/v [H, L, d] -> [H, d] via torch's fp64 scaled_dot_product_attention."""
    out = F.scaled_dot_product_attention(
        torch.from_numpy(q)[:, None, :], torch.from_numpy(k), torch.from_numpy(v),
        scale=scale)
    return out[:, 0, :].numpy()


def test_shared_kv_degenerate_case():
    """d_r = 0 and M_h = I make K = V (the failed first cut on the GVA analysis page,
    第一次尝试): the result is ordinary softmax attention with keys equal to values."""
    B, H, G, d, T = 2, 6, 3, 16, 40
    s = 0.25
    V = _f32(_rand((B * T, G, d), 7))
    qn = _rand((B, H, d), 8)
    M = np.broadcast_to(np.eye(d), (H, d, d)).copy()
    lens = np.array([T, 23])
    out, lse = oracle.gva_decode(qn, np.zeros((B, H, 0)), M, lens, _contig(B, T), V,
                                 np.zeros((B * T, 0), np.float32), s, BASE, G)
    Vd = V.astype(np.float64).reshape(B, T, G, d)
    r = H // G
    for b in range(B):
        L = lens[b]
        kv = np.stack([Vd[b, :L, h // r] for h in range(H)])     # [H, L, d]
        ref = _sdpa(qn[b], kv, kv, s)
        assert np.max(np.abs(out[b] - ref)) <= 1e-12
        z = s * torch.einsum("hd,hld->hl", torch.from_numpy(qn[b]), torch.from_numpy(kv))
        assert np.max(np.abs(lse[b] - torch.logsumexp(z, dim=1).numpy())) <= 1e-12


def test_identity_map_with_positional_slice():
    """M_h = I with d_r > 0: keys are [v_j ; k_rope_j], queries [q_nope ; Rot(t) q_rope]
    (the decoupled score of 关键技巧二), rotation taken through complex numbers."""
    B, H, G, d, d_r, T = 2, 4, 2, 8, 8, 30
    s = 1 / math.sqrt(d + d_r)
    V = _f32(_rand((B * T, G, d), 11))
    Kr = _f32(_rand((B * T, d_r), 12))
    qn, qr = _rand((B, H, d), 13), _rand((B, H, d_r), 14)
    M = np.broadcast_to(np.eye(d), (H, d, d)).copy()
    lens = np.array([T, 11])
    out, _ = oracle.gva_decode(qn, qr, M, lens, _contig(B, T), V, Kr, s, BASE, G)
    Vd = V.astype(np.float64).reshape(B, T, G, d)
    Kd = Kr.astype(np.float64).reshape(B, T, d_r)
    r = H // G
    for b in range(B):
        L = lens[b]
        q = np.concatenate([qn[b], _rot_complex(qr[b], L - 1)], axis=1)
        k = np.stack([np.concatenate([Vd[b, :L, h // r], Kd[b, :L]], axis=1) for h in range(H)])
        v = np.stack([Vd[b, :L, h // r] for h in range(H)])
        assert np.max(np.abs(out[b] - _sdpa(q, k, v, s))) <= 1e-12


def test_one_position_returns_value_exactly():
    B, H, G, d_h, d_n, d_r = 3, 8, 2, 16, 12, 8
    V = _f32(_rand((B * 5, G, d_h), 21))
    Kr = _f32(_rand((B * 5, d_r), 22))
    qn, qr = _rand((B, H, d_n), 23, 10.0), _rand((B, H, d_r), 24, 10.0)
    M = _rand((H, d_h, d_n), 25)
    out, lse = oracle.gva_decode(qn, qr, M, np.ones(B, np.int64), _contig(B, 5), V, Kr,
                                 0.7, BASE, G)
    Vd = V.astype(np.float64).reshape(B, 5, G, d_h)
    for b in range(B):
        for h in range(H):
            assert np.array_equal(out[b, h], Vd[b, 0, h // (H // G)])


def test_zero_query_gives_mean_of_values():
    B, H, G, d_h, d_n, d_r, T = 2, 4, 4, 8, 8, 8, 37
    V = _f32(_rand((B * T, G, d_h), 31))
    Kr = _f32(_rand((B * T, d_r), 32))
    lens = np.array([T, 19])
    out, lse = oracle.gva_decode(np.zeros((B, H, d_n)), np.zeros((B, H, d_r)),
                                 _rand((H, d_h, d_n), 33), lens, _contig(B, T), V, Kr,
                                 0.5, BASE, G)
    Vd = V.astype(np.float64).reshape(B, T, G, d_h)
    for b in range(B):
        for h in range(H):
            assert np.allclose(out[b, h], Vd[b, :lens[b], h].mean(axis=0), rtol=0,
                               atol=1e-13)
            assert abs(lse[b, h] - math.log(lens[b])) <= 1e-13


def test_empty_sequence():
    V = np.zeros((4, 1, 4), np.float32)
    out, lse = oracle.gva_decode(np.ones((1, 2, 4)), np.ones((1, 2, 2)),
                                 np.ones((2, 4, 4)), np.array([0]), _contig(1, 4), V,
                                 np.zeros((4, 2), np.float32), 1.0, BASE, 1)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_worked_example_from_mqa_section(golden):
    """GVA with d_h = d_n = 2, d_r = 0, M = 0.1 I turns the values [10,0], [0,10] into the
    keys [1,0], [0,1] of the page's two-position example; scale 1 as on the page."""
    gx = golden("mqa_worked_example.txt")
    V = _f32(np.array([gx["value0"], gx["value1"]])[:, None, :])       # rows [2, G=1, 2]
    M = 0.1 * np.eye(2)[None]
    keys = (V[:, 0, :].astype(np.float64) @ M[0])
    assert np.allclose(keys, [gx["key0"], gx["key1"]], atol=1e-15)
    for q, scores, wts, outp in (("q1", "q1_scores", "q1_weights", "q1_output"),
                                 ("q2", "q2_scores", "q2_weights", "q2_output")):
        qn = np.array(gx[q], dtype=np.float64)[None, None, :]
        out, lse = oracle.gva_decode(qn, np.zeros((1, 1, 0)), M, np.array([2]),
                                     _contig(1, 2), V, np.zeros((2, 0), np.float32),
                                     1.0, BASE, 1)
        z = keys @ qn[0, 0]
        assert np.allclose(z, gx[scores])
        weights = out[0, 0] / 10.0                    # values are 10 * unit vectors
        assert np.allclose(np.round(weights, int(gx["weights_decimals"])), gx[wts])
        assert np.allclose(np.round(out[0, 0], int(gx["output_decimals"])), gx[outp])
        # closed form: 10 * logistic(2) = 8.807970779778824...
        hi = 10.0 / (1.0 + math.exp(-2.0))
        assert abs(max(out[0, 0]) - hi) <= 1e-14 and abs(min(out[0, 0]) - (10 - hi)) <= 1e-14
        assert abs(lse[0, 0] - math.log(math.exp(2) + 1)) <= 1e-14


# --------------------------------------------------------------------------- #
# RoPE reading: interleaved pairs, theta_i = base^(-2i/d_r)
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("d_r", [2, 8, 16, 24, 32])
def test_rotation_matches_complex_exponential(d_r):
    x = _rand((d_r,), 41)
    for p in (0, 1, 7, 4095, 131071):
        # theta_i from two pow implementations may differ by an ulp; the angle error
        # grows with the position, so the bound does too (sign or pairing errors are O(1))
        tol = 1e-12 * max(1.0, p / 100.0)
        assert np.allclose(oracle.rotate(x, p, BASE), _rot_complex(x, p), rtol=0, atol=tol)


def test_rotation_group_properties():
    d_r = 16
    x, y = _rand((d_r,), 51), _rand((d_r,), 52)
    assert np.array_equal(oracle.rotate(x, 0, BASE), x)
    for a, b in ((3, 5), (100, 4000), (65536, 65535)):
        ab = oracle.rotate(oracle.rotate(x, a, BASE), b, BASE)
        assert np.allclose(ab, oracle.rotate(x, a + b, BASE), atol=1e-10)
        assert abs(np.linalg.norm(oracle.rotate(x, a, BASE)) - np.linalg.norm(x)) <= 1e-12
    # relative property: (Rot(t+D) q).(Rot(j+D) k) does not depend on D
    t, j = 4095, 17
    ref = oracle.rotate(x, t, BASE) @ oracle.rotate(y, j, BASE)
    for D in (1, 1000, 100000):
        got = oracle.rotate(x, t + D, BASE) @ oracle.rotate(y, j + D, BASE)
        assert abs(got - ref) <= 1e-9
    # pair 0 has theta_0 = 1: angle equals the position
    e = np.zeros(d_r)
    e[0] = 1.0
    r = oracle.rotate(e, 3, BASE)
    assert abs(r[0] - math.cos(3)) <= 1e-15 and abs(r[1] - math.sin(3)) <= 1e-15


def test_rope_table_matches_numpy():
    tab = oracle.rope_table_f32(4096, 16, BASE)
    p = np.arange(4096)[:, None]
    theta = BASE ** (-(2.0 * np.arange(8)) / 16)
    ang = p * theta
    ref = np.stack([np.cos(ang), np.sin(ang)], axis=-1).astype(np.float32)
    diff = np.abs(tab.astype(np.float64) - ref.astype(np.float64))
    ulp = np.spacing(np.abs(ref)).astype(np.float64)
    assert np.all(diff <= ulp)
    assert np.mean(tab == ref) > 0.999


def test_decode_rope_score_uses_relative_position():
    """A cache whose keys were rotated to their own positions and a query rotated to t
    score like an unrotated query against keys rotated by j - t."""
    B, H, G, d_h, d_n, d_r, T = 1, 2, 1, 4, 4, 8, 12
    s = 0.9
    k_unrot = _rand((T, d_r), 61)
    Kr = _f32(np.stack([_rot_complex(k_unrot[j], j) for j in range(T)]))
    V = _f32(_rand((T, G, d_h), 62))
    qr = _rand((B, H, d_r), 63)
    M = np.zeros((H, d_h, d_n))                          # content score 0
    out, lse = oracle.gva_decode(np.zeros((B, H, d_n)), qr, M, np.array([T]),
                                 _contig(1, T), V, Kr, s, BASE, G)
    Kd = Kr.astype(np.float64)
    for h in range(H):
        z = s * np.array([_rot_complex(qr[0, h], T - 1) @ Kd[j] for j in range(T)])
        p = np.exp(z - z.max())
        p /= p.sum()
        assert np.allclose(out[0, h], p @ V[:, 0, :].astype(np.float64), atol=1e-13)


# --------------------------------------------------------------------------- #
# permutation invariance and layouts
# --------------------------------------------------------------------------- #
def test_permutation_invariance():
    B, H, G, d_h, d_n, d_r, T = 2, 4, 2, 8, 8, 8, 50
    V = _f32(_rand((B * T, G, d_h), 71))
    Kr = _f32(_rand((B * T, d_r), 72))
    qn, qr, M = _rand((B, H, d_n), 73), _rand((B, H, d_r), 74), _rand((H, d_h, d_n), 75)
    lens = np.array([T, 31])
    o1, l1 = oracle.gva_decode(qn, qr, M, lens, _contig(B, T), V, Kr, 0.3, BASE, G)
    rng = np.random.default_rng(76)
    Vp, Kp = V.copy(), Kr.copy()
    for b in range(B):
        perm = rng.permutation(lens[b])
        Vp[b * T: b * T + lens[b]] = V[b * T + perm]
        Kp[b * T: b * T + lens[b]] = Kr[b * T + perm]
    o2, l2 = oracle.gva_decode(qn, qr, M, lens, _contig(B, T), Vp, Kp, 0.3, BASE, G)
    assert np.max(np.abs(o1 - o2)) <= 1e-12 and np.max(np.abs(l1 - l2)) <= 1e-12


def _to_paged(V, Kr, lens, T, page, seed):
    """Scatter a contiguous cache into a permuted page pool."""
    B = len(lens)
    npg = [(int(L) + page - 1) // page for L in lens]
    P = sum(npg)
    perm = np.random.default_rng(seed).permutation(P)
    bt = -np.ones((B, max(npg)), np.int64)
    Vp = np.full((P * page,) + V.shape[1:], np.nan, V.dtype)
    Kp = np.full((P * page,) + Kr.shape[1:], np.nan, Kr.dtype)
    k = 0
    for b in range(B):
        for p in range(npg[b]):
            bt[b, p] = perm[k]
            k += 1
        for j in range(int(lens[b])):
            row = bt[b, j // page] * page + j % page
            Vp[row] = V[b * T + j]
            Kp[row] = Kr[b * T + j]
    return Vp, Kp, bt


def test_paged_and_ragged_equal_contiguous_bitwise():
    """Paging moves bytes, not maths (section 7 of the MQA/GQA page): the same logical
    tokens give bit-identical results through any layout."""
    B, H, G, d_h, d_n, d_r, T = 3, 4, 2, 8, 8, 8, 70
    V = _f32(_rand((B * T, G, d_h), 81))
    Kr = _f32(_rand((B * T, d_r), 82))
    qn, qr, M = _rand((B, H, d_n), 83), _rand((B, H, d_r), 84), _rand((H, d_h, d_n), 85)
    lens = np.array([70, 1, 64])
    o1, l1 = oracle.gva_decode(qn, qr, M, lens, _contig(B, T), V, Kr, 0.3, BASE, G)
    Vp, Kp, bt = _to_paged(V, Kr, lens, T, 16, 86)
    o2, l2 = oracle.gva_decode(qn, qr, M, lens, oracle.Rows("paged", block_table=bt,
                                                             page_size=16), Vp, Kp, 0.3, BASE, G)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    off = np.concatenate([[0], np.cumsum(lens)])
    Vr = np.concatenate([V[b * T: b * T + lens[b]] for b in range(B)])
    Kr2 = np.concatenate([Kr[b * T: b * T + lens[b]] for b in range(B)])
    o3, l3 = oracle.gva_decode(qn, qr, M, lens, oracle.Rows("ragged", offsets=off), Vr,
                               Kr2, 0.3, BASE, G)
    assert np.array_equal(o1, o3) and np.array_equal(l1, l3)


def test_row_map():
    bt = np.array([[5, 2], [0, 7]])
    R = oracle.Rows("paged", block_table=bt, page_size=64)
    assert R.row(0, 0) == 320 and R.row(0, 65) == 129 and R.row(1, 127) == 7 * 64 + 63
    assert oracle.Rows("contiguous", T_cap=100).row(3, 7) == 307
    assert oracle.Rows("ragged", offsets=np.array([0, 10, 30])).row(1, 4) == 14


# --------------------------------------------------------------------------- #
# GQA comparator
# --------------------------------------------------------------------------- #
def test_gqa_matches_sdpa_enable_gqa():
    B, H, G, d, T = 2, 8, 2, 16, 45
    K = _f32(_rand((B * T, G, d), 91))
    V = _f32(_rand((B * T, G, d), 92))
    q = _rand((B, H, d), 93)
    lens = np.array([T, 30])
    out, lse = oracle.gqa_decode(q, lens, _contig(B, T), K, V, 1 / math.sqrt(d), G)
    for b in range(B):
        L = lens[b]
        k = torch.from_numpy(K.astype(np.float64).reshape(B, T, G, d)[b, :L].transpose(1, 0, 2).copy())
        v = torch.from_numpy(V.astype(np.float64).reshape(B, T, G, d)[b, :L].transpose(1, 0, 2).copy())
        ref = F.scaled_dot_product_attention(torch.from_numpy(q[b])[:, None, :], k, v,
                                             scale=1 / math.sqrt(d), enable_gqa=True)
        assert np.max(np.abs(out[b] - ref[:, 0].numpy())) <= 1e-12


def test_gva_equals_gqa_on_reconstructed_keys():
    """With one head per group and no positional slice, GVA over V equals GQA whose
    explicit keys are the reconstructed K_g = V_g M_g."""
    B, H, d, T = 2, 3, 8, 20
    V = _f32(_rand((B * T, H, d), 95))
    M = _rand((H, d, d), 96)
    qn = _rand((B, H, d), 97)
    lens = np.array([T, 9])
    o1, l1 = oracle.gva_decode(qn, np.zeros((B, H, 0)), M, lens, _contig(B, T), V,
                               np.zeros((B * T, 0), np.float32), 0.4, BASE, H)
    Vd = V.astype(np.float64)
    Kd = np.einsum("rhi,hik->rhk", Vd, M)                 # [rows, H, d]
    o2, l2 = oracle.gqa_decode(qn, lens, _contig(B, T), Kd.astype(np.float32),
                               V, 0.4, H)
    # keys were rounded to fp32 for storage: compare loosely, through the fp32 keys
    assert np.max(np.abs(o1 - o2)) <= 1e-5


# --------------------------------------------------------------------------- #
# rounding and append
# --------------------------------------------------------------------------- #
def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(101)
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * 1e3,
        np.array([0.0, -0.0, 1.0, np.inf, -np.inf, 1e-40, -1e-40, 3.4e38, 65504.0],
                 np.float32),
        # exact ties: mantissa halfway between two bf16 values
        (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
    ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_rne(x), ref)
    nan = oracle.bf16_rne(np.array([np.nan], np.float32))
    assert (nan[0] & 0x7f80) == 0x7f80 and (nan[0] & 0x7f) != 0


@pytest.mark.parametrize("bf16", [True, False])
def test_append_writes_value_and_rotated_key(bf16):
    B, G, d_h, d_r, T = 4, 2, 8, 16, 300
    rows = _contig(B, T)
    dt = np.uint16 if bf16 else np.float32
    V = np.zeros((B * T, G, d_h), dt)
    Kr = np.zeros((B * T, d_r), dt)
    vn = _f32(_rand((B, G, d_h), 111))
    kn = _f32(_rand((B, d_r), 112))
    pos = np.array([0, 1, 257, 299])
    tab = oracle.rope_table_f32(T, d_r, BASE)
    oracle.append(vn, kn, pos, rows, V, Kr, tab)
    kd = oracle.rotate_keys_f64(kn, pos, BASE)
    for b in range(B):
        row = b * T + pos[b]
        if bf16:
            assert np.array_equal(V[row], oracle.bf16_rne(vn[b]))
            tv = torch.from_numpy(vn[b]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(V[row], tv)
            got = oracle.bf16_bits_to_f64(Kr[row])
            ref = oracle.bf16_bits_to_f64(oracle.bf16_rne(kd[b].astype(np.float32)))
            ulp = 2.0 ** (np.floor(np.log2(np.abs(ref) + 1e-300)) - 7)
            assert np.all(np.abs(got - ref) <= ulp)
        else:
            assert np.array_equal(V[row], vn[b])
            assert np.allclose(Kr[row], kd[b], rtol=2e-7, atol=1e-7)
        # position 0 is the identity rotation
        if pos[b] == 0:
            exp = oracle.bf16_rne(kn[b]) if bf16 else kn[b]
            assert np.array_equal(Kr[row], exp)
    # untouched slots stay untouched
    touched = {b * T + pos[b] for b in range(B)}
    others = [i for i in range(B * T) if i not in touched]
    assert not np.any(V[others]) and not np.any(Kr[others])


def test_append_paged_row():
    G, d_h, d_r = 1, 4, 2
    bt = np.array([[3, 1]])
    rows = oracle.Rows("paged", block_table=bt, page_size=64)
    V = np.zeros((4 * 64, G, d_h), np.float32)
    Kr = np.zeros((4 * 64, d_r), np.float32)
    oracle.append(np.ones((1, G, d_h), np.float32), np.ones((1, d_r), np.float32),
                  np.array([70]), rows, V, Kr, oracle.rope_table_f32(128, d_r, BASE))
    assert np.all(V[1 * 64 + 6] == 1) and np.count_nonzero(V) == d_h


# --------------------------------------------------------------------------- #
# cache accounting (analysis page 缓存账本; summary page; MQA/GQA page §2, §3, §5)
# --------------------------------------------------------------------------- #
def test_cache_counts(golden):
    gx = golden("cache_counts.txt")
    G, d_h = int(gx["gva_G"]), int(gx["gva_d_h"])
    T = 4096
    for d_r, key in ((16, "reduction_pct_d_r16"), (24, "reduction_pct_d_r24")):
        red = 1 - oracle.n_gva(T, G, d_h, d_r) / oracle.n_gqa(T, G, d_h)
        assert round(100 * red) == gx[key]
        assert gx["reduction_range_pct"][0] <= 100 * red <= gx["reduction_range_pct"][1] + 0.5
        assert abs(oracle.gva_over_gqa(G, d_h, d_r) - (1 - red)) < 1e-15
    assert 1 - oracle.n_gva(T, 4, 64, 16) / oracle.n_gqa(T, 4, 64) == 0.46875
    assert 1 - oracle.n_gva(T, 4, 64, 24) / oracle.n_gqa(T, 4, 64) == 0.453125
    assert oracle.n_gva(T, G, d_h, 0) * 2 == oracle.n_gqa(T, G, d_h)
    # bytes per token and layer, FP16
    assert oracle.kv_bytes(1, 1, 1, 8, 128, 2) == gx["mha8_bytes_per_token_layer"]
    assert oracle.kv_bytes(1, 1, 1, 1, 128, 2) == gx["mqa8_bytes_per_token_layer"]
    L, Tt, Dh = int(gx["table_L"]), int(gx["table_T"]), int(gx["table_Dh"])
    for nkv, kib, mib in ((32, "table_mha_kib_per_token_layer", "table_mha_mib"),
                          (8, "table_gqa_kib_per_token_layer", "table_gqa_mib"),
                          (1, "table_mqa_kib_per_token_layer", "table_mqa_mib")):
        assert oracle.kv_bytes(1, 1, 1, nkv, Dh, 2) / 1024 == gx[kib]
        assert oracle.kv_bytes(L, 1, Tt, nkv, Dh, 2) / 2 ** 20 == gx[mib]
    assert oracle.n_mha(1, 8, 128) == 2 * 8 * 128


# --------------------------------------------------------------------------- #
# query RMSNorm (the "scale-matched + query RMSNorm" variant; formula is a reading)
# --------------------------------------------------------------------------- #
def test_query_rmsnorm_unit_rms_and_direction():
    """With unit gain and eps = 0 each head's normalised query keeps its direction
    (a positive multiple of the input) and has mean square exactly 1: together these
    fix it uniquely (a wrong axis, a missing square root or a sum instead of a mean
    each fails one of them)."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((3, 5, 24)) * rng.uniform(0.1, 30, (3, 5, 1))
    y = oracle.query_rmsnorm(x, None, 0.0)
    assert np.allclose(np.mean(y ** 2, axis=-1), 1.0, rtol=0, atol=1e-12)
    ratio = y / x
    assert np.all(ratio > 0)
    assert np.allclose(ratio, ratio[..., :1], rtol=1e-12, atol=0)


def test_query_rmsnorm_scale_invariance_gain_and_eps():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((2, 4, 32))
    # eps = 0: invariant to a positive rescaling of the query
    for c in (1e-3, 0.5, 7.0, 1e4):
        assert np.allclose(oracle.query_rmsnorm(c * x, None, 0.0),
                           oracle.query_rmsnorm(x, None, 0.0), rtol=0, atol=1e-12)
    # the gain multiplies each dimension of the unit-gain result
    g = rng.uniform(-2, 2, 32)
    assert np.allclose(oracle.query_rmsnorm(x, g, 0.0) / oracle.query_rmsnorm(x, None, 0.0),
                       np.broadcast_to(g, x.shape), rtol=1e-12, atol=0)
    # eps: mean square of the output is ms / (ms + eps); a zero query stays zero
    eps = 0.25
    ms = np.mean(x ** 2, axis=-1)
    y = oracle.query_rmsnorm(x, None, eps)
    assert np.allclose(np.mean(y ** 2, axis=-1), ms / (ms + eps), rtol=1e-12, atol=0)
    z = oracle.query_rmsnorm(np.zeros((1, 2, 8)), None, 1e-6)
    assert np.all(z == 0.0)


def test_query_rmsnorm_decode_reduces_to_plain_for_unit_rms_queries():
    """A query that already has unit mean square (unit gain, eps = 0) decodes exactly as
    the plain path."""
    w = workload("350m", B=2, T=40, H=4, G=2, d_h=32, d_n=32, d_r=8)
    c = make_case(w)
    q = oracle.f64(c.q_nope)
    q = q / np.sqrt(np.mean(q ** 2, axis=-1, keepdims=True))
    qn = oracle.query_rmsnorm(q, None, 0.0)
    R = oracle.Rows("contiguous", T_cap=c.T_cap)
    a, la = oracle.gva_decode(q, c.q_rope, c.M, c.seq_len, R, oracle._np(c.V), oracle._np(c.Kr),
                              w.scale, w.base, w.G)
    b, lb = oracle.gva_decode(qn, c.q_rope, c.M, c.seq_len, R, oracle._np(c.V), oracle._np(c.Kr),
                              w.scale, w.base, w.G)
    assert np.max(np.abs(a - b)) < 1e-12 and np.max(np.abs(la - lb)) < 1e-12


# --------------------------------------------------------------------------- #
# the non-absorbable variant: ordinary RoPE on the reconstructed key (a reading)
# --------------------------------------------------------------------------- #
def _rope_complex(x: torch.Tensor, pos: torch.Tensor, base: float) -> torch.Tensor:
    """RoPE as complex multiplication: pair (x[2i], x[2i+1]) -> (x0 + i x1) e^{i p theta_i},
    theta_i = base^(-2i/d) -- an independent formulation of the rotation."""
    d = x.shape[-1]
    theta = base ** (-2.0 * torch.arange(d // 2, dtype=torch.float64) / d)
    ang = pos.to(torch.float64)[..., None] * theta
    xc = torch.view_as_complex(x.reshape(*x.shape[:-1], d // 2, 2).contiguous())
    return torch.view_as_real(xc * torch.polar(torch.ones_like(ang), ang)).reshape(x.shape)


@pytest.mark.parametrize("shape", [dict(B=2, H=4, G=2, d_h=16, d_n=24, T=29),
                                   dict(B=3, H=6, G=3, d_h=32, d_n=16, T=41)])
def test_rope_keys_variant_equals_explicit_torch_attention(shape):
    """Explicit keys K = V_g M_h (torch einsum), rotated by complex multiplication, the
    whole query rotated to t = L - 1, then fp64 scaled-dot-product attention."""
    T = shape.pop("T")
    w = workload("350m", d_r=0, T=T, cache_dtype="f32", q_dtype="f32", **shape)
    c = make_case(w, lengths=[T - 3 * b for b in range(w.B)])
    q = torch.randn(w.B, w.H, w.d_n, generator=torch.Generator().manual_seed(31),
                    dtype=torch.float64)
    scale = 1.0 / math.sqrt(w.d_n)
    R = oracle.Rows("contiguous", T_cap=c.T_cap)
    out, lse = oracle.gva_decode_rope_keys(q, c.M, c.seq_len, R, c.V, scale, w.base, w.G)
    V = c.V.to(torch.float64).reshape(w.B, c.T_cap, w.G, w.d_h)
    M = c.M.to(torch.float64)
    r = w.H // w.G
    for b in range(w.B):
        L = int(c.seq_len[b])
        pos = torch.arange(L)
        for h in range(w.H):
            g = h // r
            K = _rope_complex(V[b, :L, g] @ M[h], pos, w.base)               # [L, d_n]
            qr = _rope_complex(q[b, h][None], torch.tensor([L - 1]), w.base)  # [1, d_n]
            ref = F.scaled_dot_product_attention(qr[None], K[None], V[b, :L, g][None],
                                                 scale=scale)[0, 0]
            assert np.max(np.abs(out[b, h] - ref.numpy())) < 1e-12
            z = scale * (K @ qr[0])
            assert abs(lse[b, h] - torch.logsumexp(z, 0).item()) < 1e-12


def test_rope_keys_variant_relative_position_and_one_token():
    """Shifting every position by a constant leaves the output unchanged (the score
    depends on j - t only); a one-token cache returns that token's value."""
    w = workload("350m", d_r=0, T=33, B=2, H=4, G=2, d_h=32, d_n=32, cache_dtype="f32",
                 q_dtype="f32")
    c = make_case(w)
    q = oracle.f64(c.q_nope)
    R = oracle.Rows("contiguous", T_cap=c.T_cap)
    a, la = oracle.gva_decode_rope_keys(q, c.M, c.seq_len, R, c.V, 0.2, w.base, w.G)
    b_, lb = oracle.gva_decode_rope_keys(q, c.M, c.seq_len, R, c.V, 0.2, w.base, w.G,
                                         pos_offset=77)
    assert np.max(np.abs(a - b_)) < 1e-12 and np.max(np.abs(la - lb)) < 1e-12
    one = np.ones(w.B, dtype=np.int64)
    o1, _ = oracle.gva_decode_rope_keys(q, c.M, one, R, c.V, 0.2, w.base, w.G)
    V = oracle.f64(c.V).reshape(w.B, c.T_cap, w.G, w.d_h)
    for b in range(w.B):
        for h in range(w.H):
            assert np.array_equal(o1[b, h], V[b, 0, h // 2])


# --------------------------------------------------------------------------- #
# the MLA-shaped comparator: latent cache c [d_c] + shared positional key [d_r]
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("dims", [dict(B=2, H=4, d_c=32, d_n=16, d_h=24, d_r=8, T=37),
                                  dict(B=3, H=2, d_c=48, d_n=32, d_h=32, d_r=0, T=20)])
def test_mla_decode_equals_absorbed_gva_then_up_projection(dims):
    """MLA's attention weights are GVA's with one value group (G = 1), values the latent
    (d_h = d_c) and M_h = Wuk_h; its output is that result times Wuv_h.  The MLA oracle
    materialises every key and value explicitly, the GVA oracle absorbs: they must agree
    (the absorption identity for MLA, with the up-projection moved past the sum)."""
    T = dims.pop("T")
    B, H, d_c, d_n, d_h, d_r = (dims[k] for k in ("B", "H", "d_c", "d_n", "d_h", "d_r"))
    gen = torch.Generator().manual_seed(41)
    Cc = torch.randn(B * T, d_c, generator=gen)
    Kr = torch.randn(B * T, max(d_r, 1), generator=gen)[:, :d_r].contiguous()
    qn = torch.randn(B, H, d_n, generator=gen)
    qr = torch.randn(B, H, d_r, generator=gen)
    Wuk = torch.randn(H, d_c, d_n, generator=gen) / math.sqrt(d_c)
    Wuv = torch.randn(H, d_c, d_h, generator=gen) / math.sqrt(d_c)
    L = torch.tensor([T - 5 * b for b in range(B)])
    R = oracle.Rows("contiguous", T_cap=T)
    scale = 1.0 / math.sqrt(d_n + d_r)
    out, lse = oracle.mla_decode(qn, qr, Wuk, Wuv, L, R, Cc, Kr, scale, 10000.0)
    # GVA with one group: cache rows [1][d_c], M_h = Wuk_h (d_h := d_c, d_n)
    o_lat, lse_g = oracle.gva_decode(qn, qr, Wuk, L, R, Cc.reshape(B * T, 1, d_c), Kr, scale,
                                     10000.0, 1)
    ref = np.einsum("bhc,hcd->bhd", o_lat, oracle.f64(Wuv))
    assert np.max(np.abs(out - ref)) < 1e-12
    assert np.max(np.abs(lse - lse_g)) < 1e-12


def test_mla_decode_equals_explicit_torch_attention():
    """An independent construction: torch einsum keys and values from the latent, the
    positional query rotated by complex multiplication, fp64 SDPA."""
    B, H, d_c, d_n, d_h, d_r, T = 2, 3, 24, 16, 8, 8, 19
    gen = torch.Generator().manual_seed(43)
    Cc = torch.randn(B * T, d_c, generator=gen, dtype=torch.float64).to(torch.float32)
    Kr = torch.randn(B * T, d_r, generator=gen, dtype=torch.float64).to(torch.float32)
    qn = torch.randn(B, H, d_n, generator=gen, dtype=torch.float64)
    qr = torch.randn(B, H, d_r, generator=gen, dtype=torch.float64)
    Wuk = torch.randn(H, d_c, d_n, generator=gen, dtype=torch.float64)
    Wuv = torch.randn(H, d_c, d_h, generator=gen, dtype=torch.float64)
    L = torch.tensor([T, T - 6])
    scale = 0.3
    out, lse = oracle.mla_decode(qn, qr, Wuk, Wuv, L, oracle.Rows("contiguous", T_cap=T), Cc, Kr,
                                 scale, 10000.0)
    C64 = Cc.to(torch.float64).reshape(B, T, d_c)
    K64 = Kr.to(torch.float64).reshape(B, T, d_r)
    for b in range(B):
        n = int(L[b])
        for h in range(H):
            keys = torch.cat([C64[b, :n] @ Wuk[h], K64[b, :n]], dim=1)
            vals = C64[b, :n] @ Wuv[h]
            q = torch.cat([qn[b, h], _rope_complex(qr[b, h][None], torch.tensor([n - 1]),
                                                   10000.0)[0]])
            ref = F.scaled_dot_product_attention(q[None, None], keys[None], vals[None],
                                                 scale=scale)[0, 0]
            assert np.max(np.abs(out[b, h] - ref.numpy())) < 1e-12
            assert abs(lse[b, h] - torch.logsumexp(scale * (keys @ q), 0).item()) < 1e-12


# --------------------------------------------------------------------------- #
# chunked prefill (causal), composed from the decode oracle
# --------------------------------------------------------------------------- #
def test_prefill_equals_causal_torch_attention():
    """Each new token attends causally to the history and the chunk up to itself:
    compared with fp64 SDPA over explicitly materialised keys [V_g M_h ; k_rope] and a
    boolean causal mask offset by the history length."""
    w = workload("350m", B=2, H=4, G=2, d_h=32, d_n=16, d_r=8, T=40, cache_dtype="f32",
                 q_dtype="f32")
    c = make_case(w)
    n = 5
    L0 = torch.tensor([30, 17])
    gen = torch.Generator().manual_seed(53)
    qn = torch.randn(w.B, n, w.H, w.d_n, generator=gen, dtype=torch.float64)
    qr = torch.randn(w.B, n, w.H, w.d_r, generator=gen, dtype=torch.float64)
    out, lse = oracle.gva_prefill(qn, qr, c.M, L0, c.T_cap, c.V, c.Kr, w.scale, w.base, w.G)
    V = c.V.to(torch.float64).reshape(w.B, c.T_cap, w.G, w.d_h)
    Kr = c.Kr.to(torch.float64).reshape(w.B, c.T_cap, w.d_r)
    M = c.M.to(torch.float64)
    r = w.H // w.G
    for b in range(w.B):
        P = int(L0[b]) + n                        # positions 0 .. P-1 hold history + chunk
        pos_q = torch.arange(int(L0[b]), P)
        mask = torch.arange(P)[None, :] <= pos_q[:, None]          # [n, P] causal
        for h in range(w.H):
            g = h // r
            keys = torch.cat([V[b, :P, g] @ M[h], Kr[b, :P]], dim=1)   # K_h = V_g M_h
            q = torch.cat([qn[b, :, h], _rope_complex(qr[b, :, h], pos_q, w.base)], dim=1)
            ref = F.scaled_dot_product_attention(q[None], keys[None], V[b, :P, g][None],
                                                 attn_mask=mask[None], scale=w.scale)[0]
            assert np.max(np.abs(out[b, :, h] - ref.numpy())) < 1e-12
            z = w.scale * (q @ keys.T)
            z = z.masked_fill(~mask, float("-inf"))
            assert np.max(np.abs(lse[b, :, h] - torch.logsumexp(z, 1).numpy())) < 1e-12


def test_prefill_views_of_paged_and_ragged_storage_match_contiguous():
    """Where rows live moves bytes, not maths ([K] §7): the same history and chunk stored
    in permuted pages, or at ragged offsets with gaps, give the contiguous prefill bit
    for bit."""
    w = workload("350m", B=3, H=4, G=2, d_h=32, d_n=16, d_r=8, T=64, cache_dtype="f32",
                 q_dtype="f32")
    c = make_case(w)
    n = 7
    L0 = np.array([40, 9, 57])
    gen = torch.Generator().manual_seed(71)
    qn = torch.randn(w.B, n, w.H, w.d_n, generator=gen, dtype=torch.float64)
    qr = torch.randn(w.B, n, w.H, w.d_r, generator=gen, dtype=torch.float64)
    T = c.T_cap
    Vc = c.V.numpy().reshape(w.B, T, w.G, w.d_h)
    Kc = c.Kr.numpy().reshape(w.B, T, w.d_r)
    ref, ref_lse = oracle.gva_prefill(qn, qr, c.M, L0, T, c.V, c.Kr, w.scale, w.base, w.G)
    # paged: 16-row pages at a random permutation of physical pages
    ps, mp = 16, T // 16
    bt = np.random.default_rng(5).permutation(w.B * mp).reshape(w.B, mp)
    Vp = np.zeros((w.B * mp * ps, w.G, w.d_h), dtype=np.float32)
    Kp = np.zeros((w.B * mp * ps, w.d_r), dtype=np.float32)
    for b in range(w.B):
        for p in range(mp):
            Vp[bt[b, p] * ps:(bt[b, p] + 1) * ps] = Vc[b, p * ps:(p + 1) * ps]
            Kp[bt[b, p] * ps:(bt[b, p] + 1) * ps] = Kc[b, p * ps:(p + 1) * ps]
    out, lse = oracle.gva_prefill(qn, qr, c.M, L0, oracle.Rows("paged", block_table=bt,
                                                                page_size=ps),
                                  Vp, Kp, w.scale, w.base, w.G)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)
    # ragged: sequences at offsets with unused rows between them
    offs = np.array([3, 3 + T + 5, 3 + 2 * T + 11, 3 + 3 * T + 11])
    Vr = np.full((int(offs[-1]), w.G, w.d_h), np.nan, dtype=np.float32)
    Kr = np.full((int(offs[-1]), w.d_r), np.nan, dtype=np.float32)
    for b in range(w.B):
        Vr[offs[b]:offs[b] + T] = Vc[b]
        Kr[offs[b]:offs[b] + T] = Kc[b]
    out, lse = oracle.gva_prefill(qn, qr, c.M, L0, oracle.Rows("ragged", offsets=offs),
                                  Vr, Kr, w.scale, w.base, w.G)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)
