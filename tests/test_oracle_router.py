"""Pins for the oracle's router, top-k and permutation.

* canonical-order logits: hand-derived values on inputs where the order of
  the FP32 additions decides the result, and the FP32 error bound against an
  exact FP64 dot product on random inputs;
* top-k: hand examples with ties, and a plain sort with an explicit key;
* permutation: a hand example, inverse / stability / histogram invariants.
"""

import numpy as np
import pytest

from oracle import moe, nvfp4


def _bf16(a):
    return nvfp4.bf16_to_f32(nvfp4.bf16_round(np.asarray(a, dtype=np.float32)))


def test_logits_tree_order_by_hand():
    # H = 256: chunk c (8 elements) feeds partial c.  Put 2^24 in partial 0,
    # 1 in partial 16, -2^24 in partial 1.  The pairwise tree first forms
    # 2^24 + 1 -> 2^24 (tie, even), then 2^24 - 2^24 = 0.  A left-to-right sum
    # would give 1.
    H = 256
    x = np.zeros((1, H), np.float32)
    w = np.ones((H, 1), np.float32)
    x[0, 8 * 0] = 2.0 ** 24
    x[0, 8 * 16] = 1.0
    x[0, 8 * 1] = -(2.0 ** 24)
    assert moe.router_logits(x, w)[0, 0] == 0.0


def test_logits_chunk_order_by_hand():
    # H = 512: partial 0 takes chunk 0 (h 0..7) then chunk 32 (h 256..263).
    # 2^24 at h=0, then +1 at h=256 and +1 at h=257: each +1 ties to even and is
    # lost, so the logit is 2^24.  Summing the two ones first would give 2^24+2.
    H = 512
    x = np.zeros((1, H), np.float32)
    w = np.ones((H, 1), np.float32)
    x[0, 0] = 2.0 ** 24
    x[0, 256] = 1.0
    x[0, 257] = 1.0
    assert moe.router_logits(x, w)[0, 0] == np.float32(2.0 ** 24)
    # the same three values inside one chunk, smaller ones first: 1+1 = 2,
    # then 2 + 2^24 is exact
    x2 = np.zeros((1, H), np.float32)
    x2[0, 0], x2[0, 1], x2[0, 2] = 1.0, 1.0, 2.0 ** 24
    assert moe.router_logits(x2, w)[0, 0] == np.float32(2.0 ** 24 + 2)


def test_logits_bias_is_one_add():
    H = 256
    x = np.zeros((2, H), np.float32)
    x[0, 3] = 1.5
    w = np.zeros((H, 3), np.float32)
    w[3, 1] = 2.0
    b = np.float32([0.25, -1.0, 3.0])
    got = moe.router_logits(x, w, b)
    assert got.tolist() == [[0.25, 2.0, 3.0], [0.25, -1.0, 3.0]]


def test_logits_within_fp32_error_bound():
    rng = np.random.default_rng(11)
    T, H, E = 8, 1024, 16
    x = _bf16(rng.standard_normal((T, H)))
    w = _bf16(rng.standard_normal((H, E)) * 0.02)
    got = moe.router_logits(x, w).astype(np.float64)
    exact = x.astype(np.float64) @ w.astype(np.float64)       # products exact, fp64 sum
    absum = np.abs(x.astype(np.float64)) @ np.abs(w.astype(np.float64))
    n = H // 32 + 5                                            # chain length + tree depth
    bound = n * 2.0 ** -24 * absum * 1.01
    assert np.all(np.abs(got - exact) <= bound)
    # and the order is not a no-op: fp32 sums differ from fp64 somewhere
    assert np.any(got != exact)


def test_topk_ties_by_hand():
    logits = np.float32([[1.0, 3.0, 3.0, 2.0], [0.0, 0.0, 0.0, 0.0]])
    ids, w = moe.topk_route(logits, 2)
    assert ids.tolist() == [[1, 2], [0, 1]]
    assert w.tolist() == [[0.5, 0.5], [0.5, 0.5]]


def test_topk_weights_by_hand():
    # logits ln 1, ln 2, ln 3 (approximately): softmax ~ 1/6, 2/6, 3/6; top-2 = {2, 1}
    l = np.float32([[0.0, np.log(2.0), np.log(3.0)]])
    ids, w = moe.topk_route(l, 2)
    assert ids.tolist() == [[2, 1]]
    np.testing.assert_allclose(w[0], [0.6, 0.4], rtol=1e-6)


def test_topk_against_plain_sort():
    rng = np.random.default_rng(12)
    T, E, K = 40, 32, 6
    logits = np.round(rng.standard_normal((T, E)), 1).astype(np.float32)   # many ties
    ids, w = moe.topk_route(logits, K)
    for t in range(T):
        plain = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:K]
        assert ids[t].tolist() == plain
        assert abs(float(np.sum(w[t], dtype=np.float64)) - 1.0) < 1e-6
        assert np.all(np.diff(w[t]) <= 0)          # weights follow the logit order


def test_bias_forces_expert():
    rng = np.random.default_rng(13)
    T, H, E = 6, 256, 8
    x = _bf16(rng.standard_normal((T, H)))
    w = _bf16(rng.standard_normal((H, E)) * 0.02)
    b = np.zeros(E, np.float32)
    b[5] = 100.0
    ids, _ = moe.topk_route(moe.router_logits(x, w, b), 2)
    assert (ids[:, 0] == 5).all()


def test_permute_by_hand():
    ids = np.int32([[1, 0], [0, 2], [1, 2]])
    off, src_of_row, row_of_src = moe.permute(ids, 3)
    assert off.tolist() == [0, 2, 4, 6]
    # expert 0: (t0,j1)=1, (t1,j0)=2; expert 1: (t0,j0)=0, (t2,j0)=4; expert 2: 3, 5
    assert src_of_row.tolist() == [1, 2, 0, 4, 3, 5]
    assert row_of_src.tolist() == [2, 0, 1, 4, 3, 5]


@pytest.mark.parametrize("T,E,K", [(1, 4, 1), (17, 8, 2), (64, 128, 8), (300, 16, 3)])
def test_permute_invariants(T, E, K):
    rng = np.random.default_rng(T * 31 + E)
    ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    off, src_of_row, row_of_src = moe.permute(ids, E)
    R = T * K
    assert off[0] == 0 and off[-1] == R
    assert np.array_equal(np.diff(off), np.bincount(ids.reshape(-1), minlength=E))
    assert np.array_equal(row_of_src[src_of_row], np.arange(R))
    assert np.array_equal(src_of_row[row_of_src], np.arange(R))
    for e in range(E):
        seg = src_of_row[off[e]:off[e + 1]]
        assert (ids.reshape(-1)[seg] == e).all()
        assert np.all(np.diff(seg // K) > 0)             # token order, no repeats
    # expand then unpermute is the identity on a [T*K, D] tensor
    Y = rng.standard_normal((R, 5))
    expanded = Y[src_of_row]
    assert np.array_equal(expanded[row_of_src], Y)
    # same as Python's stable sort on the expert id
    plain = sorted(range(R), key=lambda s: ids.reshape(-1)[s])
    assert src_of_row.tolist() == plain
