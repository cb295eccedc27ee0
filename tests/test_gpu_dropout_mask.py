"""GPU tests of the dropout keep mask (fa_problem.dropout_mask): stored by
the forward as it draws the decisions (or by fa_dropout_mask without a
forward) and read by the dK/dV and dQ kernels instead of drawing them again.

* The mask bytes, from fa_dropout_mask and from the forward: every entry the
  kernels read holds the oracle's keep decisions (Philox4x32-10 at
  (key / 8, row, flat head, offset), the 16-bit half against
  floor(p * 65536)), bit for bit, in the layout fa.h states:
  [Bt][Hq][key tiles of 128][rows][16 bytes], bit (key mod 8) of byte
  ((key / 8) mod 16).  Fixed and packed lengths, causal and not, ragged tails.
* The passes: O, L, dQ, dK, dV with the mask stored and read are bitwise those
  with the decisions drawn again (tensor-core D = 128 and D <= 64 kernels,
  grouped heads, Nq != Nk, packed sequences with an empty one, the FFMA
  kernels for fp32, and the single-pass backward), and they match the oracle
  within the general problems' tolerance.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from exact_attention_83_gb300 import fa
from exact_attention_83_gb300.inputs import GeneralWorkload, make_general_inputs
from general import DEV, _kw, compare, run_general

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.load_library()
    fa.set_path(fa.FA_PATH_AUTO)
    yield
    fa.set_path(fa.FA_PATH_AUTO)


def _mask_bits(mask: torch.Tensor, Bt: int, Hq: int, rows: int, Nk: int) -> np.ndarray:
    """[Bt, Hq, rows, KT * 128] keep bits decoded from the documented layout."""
    kt = (Nk + 127) // 128
    m = mask.cpu().numpy()[: Bt * Hq * kt * rows * 16].reshape(Bt, Hq, kt, rows, 16)
    bits = np.unpackbits(m, axis=-1, bitorder="little")          # [Bt, Hq, kt, rows, 128]
    return bits.transpose(0, 1, 3, 2, 4).reshape(Bt, Hq, rows, kt * 128)


def _check_sequence(bits, w, bb, r0, nq, nk, bh):
    """Entries of one (sequence, head): rows r0 .. r0+nq-1 of the decoded bits
    against the oracle's Z for flat head bh, on the key tiles the kernels read."""
    kt = (nk + 127) // 128
    if nq == 0 or kt == 0:
        return 0
    dr = oracle.dropout_params(w.dropout_p, w.drop_seed, w.drop_offset)
    ref = oracle.dropout_z(dr, bh, nq, kt * 128) > 0
    got = bits[bb, bh % w.Hq, r0:r0 + nq, : kt * 128].astype(bool)
    rows = np.arange(nq)[:, None]
    tiles = np.arange(kt * 128)[None, :] // 128
    read = np.ones((nq, kt * 128), dtype=bool)
    if w.causal:
        read = tiles <= rows // 128
    bad = np.argwhere((got != ref) & read)
    assert bad.size == 0, f"head {bh}: first mismatch at (row, key) {tuple(bad[0])}"
    return int(read.sum())


MASK_CASES = [
    GeneralWorkload("mask-fixed", 2, 3, 1, 300, 333, 64, "bf16", False, dropout_p=0.17,
                    drop_seed=0xDEADBEEF12345, drop_offset=3),
    GeneralWorkload("mask-fixed-causal", 2, 3, 3, 385, 260, 128, "fp16", True, dropout_p=0.5,
                    drop_seed=77, drop_offset=0),
    GeneralWorkload("mask-packed-causal", 5, 4, 2, 260, 300, 64, "bf16", True,
                    seqlens_q=(100, 1, 260, 0, 64), seqlens_k=(130, 7, 300, 5, 0),
                    dropout_p=0.3, drop_seed=6, drop_offset=11),
]


@pytest.mark.parametrize("by", ["dropout_mask", "forward"])
@pytest.mark.parametrize("w", MASK_CASES, ids=[w.name for w in MASK_CASES])
def test_mask_bytes_hold_the_oracle_decisions(w, by):
    q, k, v, _, cu_q, cu_k = make_general_inputs(w, DEV)
    kw = _kw(w, cu_q, cu_k)
    nbytes = fa.dropout_mask_bytes(q, k, w.causal, w.scale, **kw)
    rows = q.shape[0] if w.packed else w.Nq
    Bt = 1 if w.packed else w.B
    assert nbytes == Bt * w.Hq * ((w.Nk + 127) // 128) * rows * 16
    if by == "dropout_mask":
        mask = fa.make_dropout_mask(q, k, w.causal, w.scale, **kw)
    else:
        mask = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device=DEV)
        fa.attention_ex_fwd(q, k, v, w.causal, w.scale, **dict(kw, dropout_mask=mask))
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    bits = _mask_bits(mask, Bt, w.Hq, rows, w.Nk)
    checked = 0
    for b in range(w.B):
        if w.packed:
            r0, r1 = int(cu_q[b]), int(cu_q[b + 1])
            nq, nk = r1 - r0, int(cu_k[b + 1]) - int(cu_k[b])
            bb = 0
        else:
            r0, nq, nk, bb = 0, w.Nq, w.Nk, b
        for h in range(w.Hq):
            checked += _check_sequence(bits, w, bb, r0, nq, nk, b * w.Hq + h)
    assert checked > 0


PASS_CASES = [
    GeneralWorkload("pass-d128-causal", 2, 4, 2, 333, 517, 128, "bf16", True, dropout_p=0.17,
                    seed=5, drop_seed=0xDEADBEEF12345, drop_offset=3),
    GeneralWorkload("pass-d128-cross", 1, 4, 4, 1000, 300, 128, "fp16", False, dropout_p=0.1,
                    seed=6),
    GeneralWorkload("pass-d64-causal-gqa", 2, 8, 2, 640, 641, 64, "fp16", True, dropout_p=0.25,
                    seed=7, drop_offset=9),
    GeneralWorkload("pass-d32", 2, 4, 1, 129, 257, 32, "bf16", False, dropout_p=0.4, seed=8),
    GeneralWorkload("pass-packed-causal", 5, 4, 1, 260, 260, 64, "bf16", True,
                    seqlens_q=(100, 1, 260, 0, 64), seqlens_k=(100, 1, 260, 0, 64),
                    dropout_p=0.3, seed=9, drop_offset=11),
    GeneralWorkload("pass-packed-cross-d128", 3, 4, 2, 300, 390, 128, "bf16", False,
                    seqlens_q=(300, 77, 129), seqlens_k=(390, 5, 200), dropout_p=0.2, seed=10),
    GeneralWorkload("pass-fp32", 2, 2, 2, 200, 150, 64, "fp32", True, dropout_p=0.2, seed=11),
]


@pytest.mark.parametrize("w", PASS_CASES, ids=[w.name for w in PASS_CASES])
def test_passes_reading_the_mask_equal_drawing_it(w):
    inputs, drawn = run_general(w)
    _, read = run_general(w, keep_mask=True)
    for key in ("o", "lse", "delta", "dq", "dk", "dv"):
        np.testing.assert_array_equal(read[key], drawn[key], err_msg=f"{w.name}:{key}")
    compare(w, inputs, read)


def test_single_pass_backward_with_the_mask():
    """fa_bwd_fused draws its own decisions: with a forward that read the
    mask, dK and dV are bitwise those of a forward that drew them."""
    w = GeneralWorkload("pass-fused", 2, 4, 2, 300, 300, 128, "bf16", True, dropout_p=0.1,
                        seed=12)
    _, drawn = run_general(w, fused=True)
    inputs, read = run_general(w, fused=True, keep_mask=True)
    for key in ("o", "lse", "dk", "dv"):
        np.testing.assert_array_equal(read[key], drawn[key], err_msg=key)
    compare(w, inputs, read)


def test_autograd_keep_mask_policy():
    """attention_gqa with keep_mask True / False / None (auto) gives the same
    bits; the auto policy keeps a mask for a problem this small."""
    w = GeneralWorkload("autograd-mask", 1, 4, 2, 200, 260, 128, "bf16", True, dropout_p=0.1,
                        seed=13)
    q, k, v, do, _, _ = make_general_inputs(w, DEV)
    res = []
    for km in (True, False, None):
        qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
        o = fa.attention_gqa(qa, ka, va, True, None, 0.1, w.drop_seed, 0, keep_mask=km)
        o.backward(do)
        res.append((o.detach(), qa.grad, ka.grad, va.grad))
    for other in res[1:]:
        for a, b in zip(res[0], other):
            assert torch.equal(a, b)
    kw = dict(dropout_p=0.1, seed=w.drop_seed, offset=0)
    assert 0 < fa.dropout_mask_bytes(q, k, True, None, **kw) <= fa.DROPOUT_MASK_AUTO_BYTES


def test_backward_trusts_the_mask_it_is_given():
    """The backward reads whatever the buffer holds: given a mask drawn for
    another seed it computes that mask's gradients (no error), which is why
    the buffer must come from this problem's forward or fa_dropout_mask."""
    w = GeneralWorkload("mask-other", 1, 2, 2, 256, 256, 64, "bf16", False, dropout_p=0.2,
                        seed=14, drop_seed=1)
    q, k, v, do, _, _ = make_general_inputs(w, DEV)
    kw = _kw(w, None, None)
    own = torch.empty(fa.dropout_mask_bytes(q, k, False, w.scale, **kw), dtype=torch.uint8,
                      device=DEV)
    o, lse = fa.attention_ex_fwd(q, k, v, False, w.scale, **dict(kw, dropout_mask=own))
    other = fa.make_dropout_mask(q, k, False, w.scale, **dict(kw, seed=2))
    g_own = fa.attention_ex_bwd(q, k, v, o, lse, do, False, w.scale, **dict(kw, dropout_mask=own))
    g_drawn = fa.attention_ex_bwd(q, k, v, o, lse, do, False, w.scale, **kw)
    g_other = fa.attention_ex_bwd(q, k, v, o, lse, do, False, w.scale,
                                  **dict(kw, dropout_mask=other))
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    for a, b in zip(g_own, g_drawn):
        assert torch.equal(a, b)
    assert (g_own[2].float() - g_other[2].float()).abs().max() > 0.05     # dV


def test_mask_at_bench_size_sampled_rows():
    """The keep mask of the benchmark's dropout workload (32 heads of 16384 x
    16384, causal, p = 0.1): sampled rows (tile edges, the last row) of the
    first and last head, every key tile the kernels read, against the oracle."""
    from exact_attention_83_gb300.inputs import BENCH_GENERAL
    w = next(x for x in BENCH_GENERAL if x.dropout_p > 0)
    q, k, _, _, _, _ = make_general_inputs(w, DEV)
    kw = _kw(w, None, None)
    mask = fa.make_dropout_mask(q, k, w.causal, w.scale, **kw)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    kt = (w.Nk + 127) // 128
    entries = mask.view(w.B * w.Hq * kt, w.Nq, 16)
    dr = oracle.dropout_params(w.dropout_p, w.drop_seed, w.drop_offset)
    for bh in (0, w.B * w.Hq - 1):
        for row in (0, 127, 128, 4095, 9000, w.Nq - 1):
            tiles = row // 128 + 1 if w.causal else kt
            got = entries[bh * kt: bh * kt + tiles, row].cpu().numpy()       # [tiles, 16]
            bits = np.unpackbits(got, axis=-1, bitorder="little").reshape(-1)
            ref = oracle.dropout_z(dr, bh, 1, tiles * 128, i0=row)[0] > 0
            np.testing.assert_array_equal(bits.astype(bool), ref, err_msg=f"head {bh} row {row}")
