"""Pins for the fp64 oracle, each against something other than the oracle itself.

Every check below ties the oracle to a fact fixed by the pages or by the
mathematics: a hand-derived closed-form example, invariants of softmax
attention, special cases with a closed form, finite differences of the
forward, tile-size invariance of the FlashAttention-2 recurrences, and a
library routine (torch's float64 SDPA with autograd).
"""

from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed, scale=1.0):
    r = np.random.default_rng(seed)
    return r.standard_normal(shape) * scale


# ---------------------------------------------------------------- golden file
def _parse_golden(path):
    env = {"ln": math.log, "__builtins__": {}}
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            name, *toks = line.split()
            vals[name] = np.array([float(eval(t, env)) for t in toks])
    return vals


@pytest.mark.parametrize("causal", [False, True])
def test_golden_hand_example(causal):
    """Hand-derived closed-form example (tests/golden/hand_n2_d2.txt)."""
    g = _parse_golden(os.path.join(GOLDEN, "hand_n2_d2.txt"))
    N, D = 2, 2
    t = {k: g[k].reshape(1, 1, N, D) for k in ("q", "k", "v", "do")}
    out = oracle.fwd_bwd(t["q"], t["k"], t["v"], t["do"], causal, scale=g["scale"][0])
    pre = "causal." if causal else "full."
    for key, ref in (("o", "o"), ("lse", "lse"), ("delta", "delta"), ("dq", "dq"),
                     ("dk", "dk"), ("dv", "dv")):
        np.testing.assert_allclose(out[key].ravel(), g[pre + ref], rtol=0, atol=1e-14,
                                   err_msg=key)


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("causal", [False, True])
def test_p1_rows_sum_to_one_and_mask(causal):
    q, k, v = (rnd((2, 3, 45, 16), s) for s in (1, 2, 3))
    out = oracle.dense(q, k, v, None, causal, want_probs=True)
    p = out["p"]
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-12)
    assert (p >= 0).all()
    if causal:
        upper = np.triu(np.ones((45, 45), dtype=bool), 1)
        assert (p[..., upper] == 0).all()
        assert (p[..., ~upper] > 0).all()


def test_p2_lse_direct_sum():
    """L_i = ln sum_j exp(S_ij), recomputed with math.fsum, no max shift."""
    q, k, v = (rnd((1, 2, 20, 8), s, 0.5) for s in (4, 5, 6))
    scale = 0.37
    for causal in (False, True):
        _, L = oracle.fwd(q, k, v, causal, scale)
        for h in range(2):
            for i in range(20):
                nk = i + 1 if causal else 20
                terms = [math.exp(scale * math.fsum(q[0, h, i] * k[0, h, j])) for j in range(nk)]
                ref = math.log(math.fsum(terms))
                assert abs(L[0, h, i] - ref) <= 1e-12 * max(1.0, abs(ref))


@pytest.mark.parametrize("causal", [False, True])
def test_p3_constant_v(causal):
    q, k = rnd((2, 2, 33, 8), 7, 3.0), rnd((2, 2, 33, 8), 8, 3.0)
    vrow = rnd((8,), 9)
    v = np.broadcast_to(vrow, (2, 2, 33, 8)).copy()
    o, _ = oracle.fwd(q, k, v, causal)
    np.testing.assert_allclose(o, np.broadcast_to(vrow, o.shape), rtol=0, atol=1e-14 * 33)


def test_p4_causal_row0():
    q, k, v = (rnd((1, 3, 17, 8), s) for s in (10, 11, 12))
    o, L = oracle.fwd(q, k, v, True, 0.5)
    np.testing.assert_array_equal(o[:, :, 0], v[:, :, 0])
    np.testing.assert_allclose(L[:, :, 0], 0.5 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]),
                               rtol=0, atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_p5_zero_q_uniform(causal):
    N = 29
    q = np.zeros((1, 2, N, 8))
    k, v = rnd((1, 2, N, 8), 13), rnd((1, 2, N, 8), 14)
    o, L = oracle.fwd(q, k, v, causal)
    for i in range(N):
        n = i + 1 if causal else N
        np.testing.assert_allclose(o[:, :, i], v[:, :, :n].mean(axis=2), rtol=0, atol=1e-14)
        np.testing.assert_allclose(L[:, :, i], math.log(n), rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_p6_single_key(causal):
    q, k, v, do = (rnd((2, 2, 1, 8), s) for s in (15, 16, 17, 18))
    out = oracle.fwd_bwd(q, k, v, do, causal, 0.3)
    np.testing.assert_array_equal(out["o"], v)
    np.testing.assert_allclose(out["lse"][..., 0], 0.3 * (q * k).sum(-1)[..., 0], rtol=0, atol=1e-15)
    np.testing.assert_array_equal(out["dq"], 0)
    np.testing.assert_array_equal(out["dk"], 0)
    np.testing.assert_array_equal(out["dv"], do)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,D", [(7, 4), (16, 8)])
def test_p7_finite_differences(causal, N, D):
    """Central differences of f = sum(dO o O) w.r.t. every element of Q, K, V."""
    q, k, v, do = (rnd((1, 1, N, D), s) for s in (20 + N, 21 + N, 22 + N, 23 + N))
    scale = 1.0 / math.sqrt(D)
    g = oracle.fwd_bwd(q, k, v, do, causal, scale)
    h = 1e-6

    def f(q_, k_, v_):
        o, _ = oracle.fwd(q_, k_, v_, causal, scale)
        return float((o * do).sum())

    for name, grad in (("q", g["dq"]), ("k", g["dk"]), ("v", g["dv"])):
        fd = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            args = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
            args[name][idx] += h
            fp = f(args["q"], args["k"], args["v"])
            args[name][idx] -= 2 * h
            fm = f(args["q"], args["k"], args["v"])
            fd[idx] = (fp - fm) / (2 * h)
        err = np.abs(fd - grad).max() / max(np.abs(grad).max(), 1e-3)
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("causal", [False, True])
def test_p8_p9_gradient_sums(causal):
    q, k, v, do = (rnd((2, 3, 50, 16), s, 2.0) for s in (30, 31, 32, 33))
    g = oracle.fwd_bwd(q, k, v, do, causal)
    # each row of dS sums to 0 (softmax shift invariance) -> sum_j dK_j = 0
    np.testing.assert_allclose(g["dk"].sum(axis=2), 0, rtol=0, atol=1e-11)
    # P rows sum to 1 -> sum_j dV_j = sum_i dO_i
    np.testing.assert_allclose(g["dv"].sum(axis=2), do.sum(axis=2), rtol=0, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_delta_is_rowsum_do_o(causal):
    q, k, v, do = (rnd((1, 2, 40, 8), s) for s in (34, 35, 36, 37))
    g = oracle.fwd_bwd(q, k, v, do, causal)
    np.testing.assert_allclose(g["delta"], (do * g["o"]).sum(-1), rtol=0, atol=1e-13)


# ---------------------------------------------------------------- tile invariance
@pytest.mark.parametrize("causal", [False, True])
def test_p10_tile_invariance(causal):
    N, D = 37, 8
    q, k, v, do = (rnd((1, 2, N, D), s, 2.0) for s in (40, 41, 42, 43))
    ref = oracle.fwd_bwd(q, k, v, do, causal)
    for bq in (1, 3, 16, 64, N):
        for bk in (1, 5, 16, 128, N):
            t = oracle.tiled(q, k, v, do, causal, bq, bk)
            for key in ("o", "lse", "dq", "dk", "dv"):
                np.testing.assert_allclose(t[key], ref[key], rtol=0, atol=1e-12,
                                           err_msg=f"{key} bq={bq} bk={bk}")


@pytest.mark.parametrize("causal", [False, True])
def test_p10_tile_invariance_multi_tile(causal):
    N, D = 300, 16
    q, k, v, do = (rnd((1, 1, N, D), s, 4.0) for s in (44, 45, 46, 47))
    ref = oracle.fwd_bwd(q, k, v, do, causal)
    for bq, bk in ((128, 128), (64, 128), (128, 64), (96, 80)):
        t = oracle.tiled(q, k, v, do, causal, bq, bk)
        for key in ("o", "lse", "dq", "dk", "dv"):
            # scores have sigma ~ 16 here, so gradients reach ~1e2: compare
            # relative to the tensor's magnitude
            tol = 1e-12 * max(1.0, float(np.abs(ref[key]).max()))
            np.testing.assert_allclose(t[key], ref[key], rtol=0, atol=tol,
                                       err_msg=f"{key} bq={bq} bk={bk}")


# ---------------------------------------------------------------- other paths
@pytest.mark.parametrize("causal", [False, True])
def test_dense_matches_row_mode(causal):
    q, k, v, do = (rnd((2, 2, 70, 16), s) for s in (50, 51, 52, 53))
    a = oracle.fwd_bwd(q, k, v, do, causal)
    b = oracle.dense(q, k, v, do, causal)
    for key in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_allclose(a[key], b[key], rtol=0, atol=1e-12, err_msg=key)


def test_fwd_rows_matches_fwd():
    q, k, v = (rnd((2, 3, 64, 8), s) for s in (54, 55, 56))
    for causal in (False, True):
        o, L = oracle.fwd(q, k, v, causal)
        rows = np.array([[0, 0], [5, 63], [3, 17], [1, 40]])
        orows, Lrows = oracle.fwd_rows(q, k, v, causal, rows)
        for t, (bh, i) in enumerate(rows):
            b, h = divmod(bh, 3)
            np.testing.assert_array_equal(orows[t], o[b, h, i])
            assert Lrows[t] == L[b, h, i]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,D", [(33, 16), (128, 64)])
def test_p11_torch_sdpa_float64(causal, N, D):
    """torch's float64 scaled_dot_product_attention (math backend on CPU) and
    autograd, plus torch.logsumexp of the masked float64 scores."""
    q, k, v, do = (torch.from_numpy(rnd((2, 2, N, D), s)) for s in (60, 61, 62, 63))
    qt, kt, vt = (x.clone().requires_grad_(True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal)
    o.backward(do)
    s = (q @ k.transpose(-1, -2)) / math.sqrt(D)
    if causal:
        s = s.masked_fill(~torch.ones(N, N, dtype=torch.bool).tril(), float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    g = oracle.fwd_bwd(q.numpy(), k.numpy(), v.numpy(), do.numpy(), causal)
    np.testing.assert_allclose(g["o"], o.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(g["lse"], lse.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(g["dq"], qt.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(g["dk"], kt.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(g["dv"], vt.grad.numpy(), rtol=0, atol=1e-11)


def test_strided_input_is_read_as_logical_bhnd():
    """A permuted [B,N,H,D] -> [B,H,N,D] view gives the same result as its
    contiguous copy (the wrapper converts views exactly)."""
    base = torch.from_numpy(rnd((2, 20, 3, 8), 70))
    view = base.permute(0, 2, 1, 3)
    a = oracle.fwd(view, view, view, True)
    b = oracle.fwd(view.contiguous().numpy(), view.contiguous().numpy(),
                   view.contiguous().numpy(), True)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_rows_match_full(causal):
    """The sampled-row entry points give exactly the rows of the full result."""
    q, k, v, do = (rnd((2, 3, 90, 16), s) for s in (80, 81, 82, 83))
    full = oracle.fwd_bwd(q, k, v, do, causal)
    rows = np.array([[0, 0], [5, 89], [3, 17], [1, 40], [5, 0], [2, 64]])
    qr = oracle.query_rows(q, k, v, do, causal, rows)
    kr = oracle.key_rows(q, k, v, do, causal, rows)
    for t, (bh, i) in enumerate(rows):
        b, h = divmod(bh, 3)
        np.testing.assert_allclose(qr["o"][t], full["o"][b, h, i], rtol=0, atol=1e-14)
        np.testing.assert_allclose(qr["lse"][t], full["lse"][b, h, i], rtol=0, atol=1e-14)
        np.testing.assert_allclose(qr["delta"][t], full["delta"][b, h, i], rtol=0, atol=1e-13)
        np.testing.assert_allclose(qr["dq"][t], full["dq"][b, h, i], rtol=0, atol=1e-13)
        np.testing.assert_allclose(kr["dk"][t], full["dk"][b, h, i], rtol=0, atol=1e-13)
        np.testing.assert_allclose(kr["dv"][t], full["dv"][b, h, i], rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_magnitudes_bound_the_values_and_match_them_for_one_signed_terms(causal):
    """sum |terms| >= |sum of terms| everywhere, with equality when every term
    has the same sign (V >= 0 for O, dO >= 0 for dV)."""
    q, k, v, do = (rnd((2, 2, 60, 8), s, 2.0) for s in (90, 91, 92, 93))
    g = oracle.fwd_bwd(q, k, v, do, causal)
    m = oracle.magnitudes(q, k, v, do, causal)
    for key in ("o", "dq", "dk", "dv"):
        assert (m[key] >= np.abs(g[key]) - 1e-12).all(), key
    vp, dop = np.abs(v), np.abs(do)
    g2 = oracle.fwd_bwd(q, k, vp, dop, causal)
    m2 = oracle.magnitudes(q, k, vp, dop, causal)
    np.testing.assert_allclose(m2["o"], g2["o"], rtol=1e-13, atol=0)
    np.testing.assert_allclose(m2["dv"], g2["dv"], rtol=1e-13, atol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_row_magnitudes_equal_full_magnitudes(causal):
    q, k, v, do = (rnd((2, 3, 70, 16), s, 4.0) for s in (94, 95, 96, 97))
    m = oracle.magnitudes(q, k, v, do, causal)
    rows = np.array([[0, 0], [1, 69], [4, 33], [5, 1]])
    qr = oracle.query_rows(q, k, v, do, causal, rows, magnitudes=True)
    kr = oracle.key_rows(q, k, v, do, causal, rows, magnitudes=True)
    b, h, i = rows[:, 0] // 3, rows[:, 0] % 3, rows[:, 1]
    for key, src in (("o", qr), ("dq", qr), ("dk", kr), ("dv", kr)):
        np.testing.assert_allclose(src[key + "_abs"], m[key][b, h, i], rtol=1e-12, atol=1e-300)
