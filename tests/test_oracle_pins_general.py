"""Pins for the oracle's general problems: query and key lengths that differ,
grouped key/value heads, packed variable-length sequences and dropout of the
attention weights.  Each is tied to something other than the oracle itself:
a library routine (torch's float64 SDPA with autograd, on key/value heads
expanded with repeat_interleave, whose backward sums the group), the
generator's published known-answer vectors, finite differences of the
oracle's own forward with the dropout mask held fixed, and consistency
between the packed and the batched numbering of the dropout mask.
"""

from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def sdpa_ref(q, k, v, do, causal, scale):
    """torch float64 SDPA (top-left causal mask for Nq != Nk) with autograd;
    k, v repeated over the query heads of their group."""
    G = q.shape[1] // k.shape[1]
    qt, kt, vt = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    ke, ve = kt.repeat_interleave(G, dim=1), vt.repeat_interleave(G, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, ke, ve, is_causal=causal,
                                                         scale=scale)
    o.backward(torch.tensor(do, dtype=torch.float64))
    s = scale * (qt @ ke.transpose(-1, -2))
    if causal:
        Nq, Nk = s.shape[-2:]
        s = s.masked_fill(~torch.ones(Nq, Nk, dtype=torch.bool).tril(), float("-inf"))
    L = torch.logsumexp(s, dim=-1)
    return dict(o=o.detach().numpy(), lse=L.detach().numpy(), dq=qt.grad.numpy(),
                dk=kt.grad.numpy(), dv=vt.grad.numpy())


def test_philox_known_answers():
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        w = [int(x, 16) for x in r]
        assert oracle.philox4x32_10(w[0:4], w[4:6]) == tuple(w[6:10])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(37, 53), (200, 96), (64, 1), (1, 70)])
def test_non_square_matches_library(Nq, Nk, causal):
    """The Triton page's test shapes include Nq != Nk, with the mask the lower
    triangle of the Nq x Nk score matrix."""
    q, do = rnd((1, 2, Nq, 32), 1), rnd((1, 2, Nq, 32), 2)
    k, v = rnd((1, 2, Nk, 32), 3), rnd((1, 2, Nk, 32), 4)
    g = oracle.fwd_bwd(q, k, v, do, causal, 0.3)
    r = sdpa_ref(q, k, v, do, causal, 0.3)
    for key in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_allclose(g[key], r[key], rtol=1e-10, atol=1e-11, err_msg=key)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (6, 1), (4, 4)])
def test_grouped_heads_match_library(Hq, Hkv, causal):
    q, do = rnd((2, Hq, 45, 16), 5), rnd((2, Hq, 45, 16), 6)
    k, v = rnd((2, Hkv, 60, 16), 7), rnd((2, Hkv, 60, 16), 8)
    g = oracle.fwd_bwd(q, k, v, do, causal, 0.25)
    r = sdpa_ref(q, k, v, do, causal, 0.25)
    for key in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_allclose(g[key], r[key], rtol=1e-10, atol=1e-11, err_msg=key)


def test_grouped_rows_match_full():
    q, do = rnd((2, 6, 50, 16), 9), rnd((2, 6, 50, 16), 10)
    k, v = rnd((2, 2, 40, 16), 11), rnd((2, 2, 40, 16), 12)
    dr = oracle.dropout_params(0.2, seed=77, offset=5)
    g = oracle.fwd_bwd(q, k, v, do, True, 0.25, dr)
    qrows = np.array([[0, 0], [5, 49], [7, 20], [11, 3]])
    krows = np.array([[0, 0], [1, 39], [3, 17]])
    qr = oracle.query_rows(q, k, v, do, True, qrows, 0.25, dropout=dr)
    kr = oracle.key_rows(q, k, v, do, True, krows, 0.25, dropout=dr)
    b, h, i = qrows[:, 0] // 6, qrows[:, 0] % 6, qrows[:, 1]
    for key in ("o", "lse", "delta", "dq"):
        np.testing.assert_allclose(qr[key], g[key][b, h, i], rtol=1e-13, atol=1e-14)
    b, h, j = krows[:, 0] // 2, krows[:, 0] % 2, krows[:, 1]
    for key in ("dk", "dv"):
        np.testing.assert_allclose(kr[key], g[key][b, h, j], rtol=1e-13, atol=1e-14)


def test_dropout_zero_is_no_dropout():
    q, k, v, do = (rnd((1, 2, 33, 16), s) for s in (13, 14, 15, 16))
    a = oracle.fwd_bwd(q, k, v, do, True, 0.25)
    b = oracle.fwd_bwd(q, k, v, do, True, 0.25, oracle.dropout_params(0.0, seed=3))
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])


def _mask(p, seed, offset, bh, Nq, Nk):
    """Z built here from the generator (pinned above) and the stated counter
    layout: 16-bit half j%2 of word (j%8)/2 of philox((j/8, i, bh, offset),
    (seed lo, seed hi)) against floor(p * 65536)."""
    thr = min(int(np.floor(float(np.float32(p)) * 65536.0)), 65535)
    z = np.zeros((Nq, Nk))
    for i in range(Nq):
        for jg in range((Nk + 7) // 8):
            w = oracle.philox4x32_10([jg, i, bh, offset], [seed & 0xFFFFFFFF, seed >> 32])
            halves = [h for word in w for h in (word & 0xFFFF, word >> 16)]
            for e in range(8):
                j = 8 * jg + e
                if j < Nk:
                    z[i, j] = 1.0 / (1.0 - float(np.float32(p))) if halves[e] >= thr else 0.0
    return z


def test_dropout_output_is_masked_probabilities_times_v():
    """O = (P o Z) V with P the dense path's probabilities and Z assembled
    from the generator; L is unchanged by dropout."""
    B, H, N, D = 1, 2, 30, 8
    q, k, v = (rnd((B, H, N, D), s) for s in (17, 18, 19))
    seed, off, p = 0x1234_5678_9ABC, 9, 0.3
    o, L = oracle.fwd(q, k, v, True, 0.4, oracle.dropout_params(p, seed, off))
    dn = oracle.dense(q, k, v, None, True, 0.4, want_probs=True)
    for h in range(H):
        z = _mask(p, seed, off, h, N, N)
        np.testing.assert_allclose(o[0, h], (dn["p"][0, h] * z) @ v[0, h], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L, dn["lse"], rtol=1e-13, atol=1e-13)


def test_dropout_z_matches_the_generator_layout():
    """oracle.dropout_z (the factor the oracle's passes apply) equals Z
    assembled here from the pinned generator, for several flat heads, a ragged
    key count and a 64-bit seed; without dropout it is 1 everywhere."""
    seed, off, p = 0xFEDC_BA98_7654_3210, 4, 0.23
    dr = oracle.dropout_params(p, seed, off)
    for bh in (0, 3, 70001):
        z = _mask(p, seed, off, bh, 19, 45)
        np.testing.assert_array_equal(oracle.dropout_z(dr, bh, 19, 45), z)
        np.testing.assert_array_equal(oracle.dropout_z(dr, bh, 7, 45, i0=12), z[12:])
    np.testing.assert_array_equal(oracle.dropout_z(oracle.dropout_params(0.0), 1, 5, 9),
                                  np.ones((5, 9)))


def test_dropout_keep_fraction():
    """About 1 - p of the weights survive (binomial, 6 standard deviations)."""
    p, n = 0.17, 0
    z = _mask(p, 99, 0, 0, 64, 256)
    n = z.size
    kept = (z > 0).mean()
    sd = np.sqrt(p * (1 - p) / n)
    assert abs(kept - (1 - p)) < 6 * sd


def test_dropout_gradients_match_finite_differences():
    """With the mask fixed by (seed, offset) the forward is a smooth function
    of Q, K, V; central differences of sum(dO o O) pin dQ, dK, dV, including
    dS = P o (Z o dP - Delta) and dV = (P o Z)^T dO."""
    B, Hq, Hkv, Nq, Nk, D = 1, 2, 1, 9, 11, 4
    q, do = rnd((B, Hq, Nq, D), 20), rnd((B, Hq, Nq, D), 21)
    k, v = rnd((B, Hkv, Nk, D), 22), rnd((B, Hkv, Nk, D), 23)
    dr = oracle.dropout_params(0.35, seed=2024, offset=1)
    g = oracle.fwd_bwd(q, k, v, do, True, 0.5, dr)

    def f(qq, kk, vv):
        return float((oracle.fwd(qq, kk, vv, True, 0.5, dr)[0] * do).sum())

    eps = 1e-6
    for name, arr in (("dq", q), ("dk", k), ("dv", v)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a1, a2 = arr.copy(), arr.copy()
            a1[idx] += eps
            a2[idx] -= eps
            args1 = {"dq": (a1, k, v), "dk": (q, a1, v), "dv": (q, k, a1)}[name]
            args2 = {"dq": (a2, k, v), "dk": (q, a2, v), "dv": (q, k, a2)}[name]
            num[idx] = (f(*args1) - f(*args2)) / (2 * eps)
        np.testing.assert_allclose(g[name], num, rtol=1e-6, atol=1e-7, err_msg=name)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_library_per_sequence(causal):
    """Each packed sequence is its own attention problem."""
    lens_q, lens_k = [5, 0, 40, 17], [9, 3, 40, 1]
    cu_q, cu_k = np.cumsum([0] + lens_q), np.cumsum([0] + lens_k)
    Hq, Hkv, D = 4, 2, 16
    q, do = rnd((cu_q[-1], Hq, D), 24), rnd((cu_q[-1], Hq, D), 25)
    k, v = rnd((cu_k[-1], Hkv, D), 26), rnd((cu_k[-1], Hkv, D), 27)
    g = oracle.varlen_fwd_bwd(q, k, v, do, cu_q, cu_k, causal, 0.25)
    for b in range(4):
        qs, qe, ks, ke = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        if qe == qs:
            np.testing.assert_array_equal(g["dk"][ks:ke], 0.0)
            continue
        t = lambda a, s, e: a[s:e].transpose(1, 0, 2)[None]
        r = sdpa_ref(t(q, qs, qe), t(k, ks, ke), t(v, ks, ke), t(do, qs, qe), causal, 0.25)
        np.testing.assert_allclose(g["o"][qs:qe], r["o"][0].transpose(1, 0, 2), rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(g["lse"][:, qs:qe], r["lse"][0], rtol=1e-10, atol=1e-11)
        for key in ("dq",):
            np.testing.assert_allclose(g[key][qs:qe], r[key][0].transpose(1, 0, 2), rtol=1e-10, atol=1e-11)
        for key in ("dk", "dv"):
            np.testing.assert_allclose(g[key][ks:ke], r[key][0].transpose(1, 0, 2), rtol=1e-10, atol=1e-11)


def test_varlen_empty_keys_give_zero_output_and_minus_inf():
    cu_q, cu_k = np.array([0, 3]), np.array([0, 0])
    q, do = rnd((3, 2, 8), 28), rnd((3, 2, 8), 29)
    k = np.zeros((0, 2, 8)); v = np.zeros((0, 2, 8))
    g = oracle.varlen_fwd_bwd(q, k, v, do, cu_q, cu_k, False, 0.3)
    assert (g["o"] == 0).all() and (g["dq"] == 0).all() and np.isneginf(g["lse"]).all()


def test_varlen_equal_lengths_match_batched_including_dropout_numbering():
    """Packed sequence b numbers its heads b*Hq + h, as the batched layout does."""
    B, Hq, Hkv, N, D = 3, 4, 2, 21, 8
    q, do = rnd((B, Hq, N, D), 30), rnd((B, Hq, N, D), 31)
    k, v = rnd((B, Hkv, N, D), 32), rnd((B, Hkv, N, D), 33)
    dr = oracle.dropout_params(0.25, seed=5, offset=7)
    g = oracle.fwd_bwd(q, k, v, do, True, 0.35, dr)
    pack = lambda a: a.transpose(0, 2, 1, 3).reshape(B * N, a.shape[1], D)
    cu = np.arange(B + 1) * N
    r = oracle.varlen_fwd_bwd(pack(q), pack(k), pack(v), pack(do), cu, cu, True, 0.35,
                              p=0.25, seed=5, offset=7)
    for key in ("o", "dq", "dk", "dv"):
        np.testing.assert_allclose(r[key], pack(g[key]), rtol=1e-13, atol=1e-14, err_msg=key)
    np.testing.assert_allclose(r["lse"], g["lse"].transpose(1, 0, 2).reshape(Hq, B * N),
                               rtol=1e-13, atol=1e-14)


def test_magnitudes_bound_values_with_groups_and_dropout():
    q, do = rnd((1, 4, 30, 8), 34, 2.0), rnd((1, 4, 30, 8), 35)
    k, v = rnd((1, 2, 41, 8), 36, 2.0), rnd((1, 2, 41, 8), 37, 2.0)
    dr = oracle.dropout_params(0.3, seed=11)
    g = oracle.fwd_bwd(q, k, v, do, True, 0.3, dr)
    m = oracle.magnitudes(q, k, v, do, True, 0.3, dr)
    for key in ("o", "dq", "dk", "dv"):
        assert m[key].shape == g[key].shape
        assert (m[key] >= np.abs(g[key]) - 1e-12).all(), key
    vp = np.abs(v)
    g2 = oracle.fwd_bwd(q, k, vp, do, True, 0.3, dr)
    m2 = oracle.magnitudes(q, k, vp, do, True, 0.3, dr)
    np.testing.assert_allclose(m2["o"], g2["o"], rtol=1e-13, atol=0)
