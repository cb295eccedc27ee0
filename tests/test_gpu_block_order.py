"""The grouped block order of the forward, dK/dV and dQ grids.

The grids take heads in groups whose shared operand fits in part of L2, and
run each group longest tile first (include/fa.h, fa_test_set_l2_bytes).  On a
real problem a partial last group only appears at large sizes, which the
full-size tests check on sampled rows.  Here fa_test_set_l2_bytes forces small
groups on small problems.  The order only decides which CTAs run together, never
what a CTA computes, so O, L, dQ, dK and dV must be bitwise those of the
default order.

Group sizes below follow the library's rule, all heads when they fit in 3/4
of L2, else floor(L2 * 3/8 / per_head_bytes).  Here per_head_bytes is
2 * Nk * D * element size for the forward and dQ (per query head), and
2 * Nq * D * element size * (Hq / Hkv) for dK/dV (per key/value head).
"""

from __future__ import annotations

import numpy as np
import pytest

from exact_attention_83_gb300 import fa
from exact_attention_83_gb300.inputs import GeneralWorkload
from general import run_general

pytestmark = pytest.mark.gpu


def _group(bh: int, per_head: int, l2: int) -> int:
    if bh * per_head <= l2 * 3 // 4:
        return bh
    return max(1, min(bh, l2 * 3 // 8 // per_head))


CASES = [
    # 16 query heads of 512000 bytes: groups of 3 (3,3,3,3,3,1) in the
    # two-tile forward, the per-tile dK/dV kernel (D = 128) and dQ
    (GeneralWorkload("order-d128-causal", 2, 8, 8, 1000, 1000, 128, "bf16", True, seed=31),
     4_200_000, (3, 3)),
    # 24 query heads of 230400 bytes: groups of 5 (5,5,5,5,4) in the D = 64
    # forward and dQ; 6 key/value heads of 716800 bytes: groups of 1 in the
    # clustered dK/dV kernel (four query heads per key/value head)
    (GeneralWorkload("order-gqa-d64-causal", 3, 8, 2, 700, 900, 64, "fp16", True, seed=32),
     3_100_000, (5, 1)),
    # packed sequences, not causal: the grids count (sequence, head) pairs and
    # the longest sequence's tiles; 12 heads of 76800 bytes, groups of 5
    # (5, 5, 2) in every kernel
    (GeneralWorkload("order-packed-d64", 3, 4, 4, 300, 300, 64, "bf16", False,
                     seqlens_q=(300, 17, 129), seqlens_k=(280, 300, 5), seed=33),
     1_100_000, (5, 5)),
]


@pytest.mark.parametrize("w, l2, groups", CASES, ids=[c[0].name for c in CASES])
def test_forced_head_groups_give_the_same_bits(w, l2, groups):
    esz = 2
    fwd_group = _group(w.B * w.Hq, 2 * w.Nk * w.D * esz, l2)
    dkdv_group = _group(w.B * w.Hkv, 2 * w.Nq * w.D * esz * (w.Hq // w.Hkv), l2)
    assert (fwd_group, dkdv_group) == groups
    fa.load_library()
    _, ref = run_general(w)
    fa.test_set_l2_bytes(l2)
    try:
        _, got = run_general(w)
    finally:
        fa.test_set_l2_bytes(0)
    for key in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=f"{w.name}:{key}")
