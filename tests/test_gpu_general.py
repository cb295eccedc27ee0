"""GPU parity for the general problems (fa_fwd_ex / fa_bwd_ex) against the
fp64 oracle: query and key lengths that differ (the Triton page's test shapes),
grouped and multi-query key/value heads, packed variable-length sequences
(empty ones included) and dropout of the attention weights, on the
tensor-core kernels (fp16/bf16) and the FFMA kernels (fp32).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from exact_attention_83_gb300 import fa
from exact_attention_83_gb300.inputs import GeneralWorkload, make_general_inputs
from general import PAGE_SHAPES, compare, random_general, run_general

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.load_library()
    fa.set_path(fa.FA_PATH_AUTO)
    yield
    fa.set_path(fa.FA_PATH_AUTO)


# --------------------------------------------------------------- Nq != Nk
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
@pytest.mark.parametrize("shape", PAGE_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_page_shapes(shape, dtype, causal):
    B, Nq, Nk, D = shape
    w = GeneralWorkload(f"shape-{dtype}-{B}x{Nq}x{Nk}x{D}-{causal}", B, 2, 2, Nq, Nk, D, dtype,
                        causal, seed=Nq + Nk)
    compare(w, *run_general(w))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(300, 1000), (1000, 300), (129, 1), (1, 257), (640, 641)])
def test_non_square_lengths(Nq, Nk, causal):
    w = GeneralWorkload(f"nonsq-bf16-{Nq}x{Nk}-{causal}", 2, 4, 4, Nq, Nk, 128, "bf16", causal,
                        seed=7)
    compare(w, *run_general(w))


# --------------------------------------------------------------- grouped heads
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("Hq,Hkv,D", [(8, 2, 128), (8, 1, 64), (6, 3, 32), (4, 4, 16)])
def test_grouped_heads(Hq, Hkv, D, dtype, causal):
    w = GeneralWorkload(f"gqa-{dtype}-Hq{Hq}-Hkv{Hkv}-D{D}-{causal}", 2, Hq, Hkv, 777, 901, D,
                        dtype, causal, seed=Hq * 10 + Hkv)
    compare(w, *run_general(w))


# --------------------------------------------------------------- packed sequences
VARLEN = [
    (1, 127, 128, 129, 700, 0, 1500, 3),
    (256, 1, 511),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("lens", VARLEN, ids=["mix", "short"])
def test_packed_sequences(lens, dtype, causal):
    lk = tuple(reversed(lens))          # key lengths differ from query lengths
    w = GeneralWorkload(f"varlen-{dtype}-{len(lens)}seq-{causal}", len(lens), 8, 2, max(lens),
                        max(lk), 128 if dtype != "fp32" else 64, dtype, causal,
                        seqlens_q=lens, seqlens_k=lk, seed=3)
    compare(w, *run_general(w))


def test_packed_sequence_with_no_keys():
    """An empty key sequence: O = 0, L = -inf, dQ = 0; keys nobody attends:
    dK = dV = 0."""
    w = GeneralWorkload("varlen-nokeys-bf16", 3, 4, 4, 200, 130, 64, "bf16", False,
                        seqlens_q=(200, 5, 0), seqlens_k=(0, 9, 130), seed=4)
    inputs, got = run_general(w)
    assert (got["o"][:200] == 0).all() and np.isneginf(got["lse"][:, :200]).all()
    assert (got["dk"][9:] == 0).all() and (got["dv"][9:] == 0).all()
    compare(w, inputs, got)


def test_inconsistent_offsets_are_reported_not_followed():
    """Decreasing offsets: the kernels skip that sequence and record
    FA_ERR_SEQLENS; nothing outside the tensors is touched."""
    q = torch.zeros(64, 2, 64, dtype=torch.bfloat16, device=DEV)
    o = torch.zeros_like(q)
    lse = torch.zeros(2, 64, dtype=torch.float32, device=DEV)
    cu = torch.tensor([0, 40, 30, 64], dtype=torch.int32, device=DEV)
    fa.fwd_ex(q, q, q, o, lse, False, 0.125, cu_seqlens_q=cu, cu_seqlens_k=cu,
              max_seqlen_q=40, max_seqlen_k=40)
    torch.cuda.synchronize()
    assert fa.device_status() == 13
    assert fa.device_status() == 0          # read and cleared


# --------------------------------------------------------------- dropout
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp16", 64), ("bf16", 32), ("fp32", 64)])
def test_dropout(dtype, D, causal):
    w = GeneralWorkload(f"drop-{dtype}-D{D}-{causal}", 2, 4, 2, 333, 517, D, dtype, causal,
                        dropout_p=0.17, seed=5, drop_seed=0xDEADBEEF12345, drop_offset=3)
    compare(w, *run_general(w))


def test_dropout_packed():
    lens = (100, 1, 260, 0, 64)
    w = GeneralWorkload("drop-varlen-bf16", 5, 4, 1, 260, 260, 64, "bf16", True,
                        seqlens_q=lens, seqlens_k=lens, dropout_p=0.3, seed=6, drop_offset=11)
    compare(w, *run_general(w))


def test_dropout_mask_follows_seed_and_offset():
    base = GeneralWorkload("drop-det", 1, 2, 2, 300, 300, 64, "bf16", False, dropout_p=0.2, seed=8)
    _, a = run_general(base)
    _, b = run_general(base)
    np.testing.assert_array_equal(a["o"], b["o"])
    _, c = run_general(GeneralWorkload("drop-det2", 1, 2, 2, 300, 300, 64, "bf16", False,
                                       dropout_p=0.2, seed=8, drop_offset=1))
    assert np.abs(a["o"] - c["o"]).max() > 0.05


def test_autograd_general():
    w = GeneralWorkload("autograd-gqa", 1, 4, 2, 200, 260, 64, "bf16", True, dropout_p=0.1,
                        seed=9)
    q, k, v, do, _, _ = make_general_inputs(w, DEV)
    qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = fa.attention_gqa(qa, ka, va, True, None, 0.1, w.drop_seed, 0)
    o.backward(do)
    o2, lse = fa.attention_ex_fwd(q, k, v, True, None, dropout_p=0.1, seed=w.drop_seed)
    grads = fa.attention_ex_bwd(q, k, v, o2, lse, do, True, None, dropout_p=0.1,
                                seed=w.drop_seed)
    assert torch.equal(o, o2)
    for a, b in zip((qa.grad, ka.grad, va.grad), grads):
        assert torch.equal(a, b)


@pytest.mark.parametrize("seed", range(40))
def test_random_general_problems(seed):
    w = random_general(seed)
    compare(w, *run_general(w))
