"""Pins of the oracle's block scorer and top-k selection (CPU only).

The pages name the scorer but not its score; the oracle follows the reading
stated in its module (mean-pooled index vectors, an fp32 dot product summed in
index-dim order, the diagonal block first, then the top scores with ties to the
lower block).  These tests tie each step to something other than the oracle:
exact arithmetic where fp32 is exact, a hand-worked case where the summation
order decides the value, an independent ranking by numpy lexsort, and a
hand-worked golden selection."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import msa_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))


def _bits(x):
    """Exact bf16 bit patterns of float values that bf16 represents exactly."""
    t = torch.tensor(np.asarray(x, np.float64), dtype=torch.float64)
    b = t.to(torch.bfloat16)
    assert torch.equal(b.double(), t), "test value not exact in bf16"
    return b.view(torch.int16).numpy().view(np.uint16)


def test_pooling_equals_exact_means_on_dyadic_inputs():
    rng = np.random.default_rng(0)
    lengths = [64 * 3, 64, 128]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    T = int(cu[-1])
    x = rng.integers(-1, 2, size=(T, 2, 8)) / 4.0            # sums over 64 stay exact in bf16 and fp32
    bits = _bits(x)
    for size in (8, 64):
        got = O.bf16_to_f64(O.pool_index(bits, cu, size))  # [Hi, G, D]
        exp = np.concatenate([x[cu[d]:cu[d + 1]].reshape(-1, size, 2, 8).mean(axis=1)
                              for d in range(len(lengths))]).transpose(1, 0, 2)
        np.testing.assert_array_equal(got, exp)


def test_pooling_of_partial_groups_averages_the_tokens_present():
    # documents of 5 and 11 tokens: groups of 8 -> sizes 5 | 8, 3; every token of a
    # group holds the same value, so the mean is that value for any group size
    cu = np.array([0, 5, 16])
    vals = np.array([0.75] * 5 + [1.5] * 8 + [-3.0] * 3)
    x = np.repeat(vals[:, None, None], 4, axis=2)
    got = O.bf16_to_f64(O.pool_index(_bits(x), cu, 8))[0]
    np.testing.assert_array_equal(got[:, 0], [0.75, 1.5, -3.0])


def test_scores_equal_exact_dot_products_where_fp32_is_exact():
    rng = np.random.default_rng(1)
    qp = rng.integers(-8, 9, size=(2, 7, 128)) / 8.0
    kp = rng.integers(-8, 9, size=(2, 5, 128)) / 8.0
    got = O.block_scores(_bits(qp), _bits(kp))
    np.testing.assert_array_equal(got.astype(np.float64), np.einsum("hqd,hkd->hqk", qp, kp))


def test_scores_accumulate_in_fp32_in_index_dim_order():
    # q = (1, 1, 1), k = (2**24, 1, -2**24): in fp32, (2**24 + 1) rounds back to
    # 2**24, so accumulating dims 0, 1, 2 in that order gives 0; the exact dot
    # product (and any order that adds dims 0 and 2 first) gives 1
    q = np.zeros((1, 128))
    k = np.zeros((1, 128))
    q[0, :3] = 1.0
    k[0, :3] = [2.0 ** 24, 1.0, -2.0 ** 24]
    assert float(O.block_scores(_bits(q), _bits(k))[0, 0]) == 0.0
    k[0, :3] = [2.0 ** 24, -2.0 ** 24, 1.0]
    assert float(O.block_scores(_bits(q), _bits(k))[0, 0]) == 1.0


def _rank_independently(scores, diag, k):
    """Selection rule restated with numpy lexsort: key (-score, block)."""
    b = np.arange(diag)
    order = np.lexsort((b, -scores[:diag].astype(np.float64)))
    return [diag] + [int(x) for x in order[:k - 1]]


@pytest.mark.parametrize("seed", range(4))
def test_selection_matches_an_independent_ranking(seed):
    rng = np.random.default_rng(seed)
    lengths = [int(n) for n in rng.integers(1, 300, size=3)]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    T, Hi, B, C, K = int(cu[-1]), 2, 16, 4, 5
    qi = rng.integers(-3, 4, size=(T, Hi, 16)) / 2.0       # coarse values: many exact ties between blocks
    ki = rng.integers(-3, 4, size=(T, Hi, 16)) / 2.0
    qb, kb = _bits(qi), _bits(ki)
    sel = O.select_topk(qb, kb, cu, B, C, K)
    lay = O.DocLayout(cu, B, C)
    qpool, kpool = O.pool_index(qb, cu, C), O.pool_index(kb, cu, B)
    ties = 0
    for d in range(len(lengths)):
        g0, r0 = int(lay.chunk_off[d]), int(lay.blk_off[d])
        for hi in range(Hi):
            sc = O.block_scores(qpool[hi, g0:g0 + lay.nc[d]], kpool[hi, r0:r0 + lay.nb[d]])
            for c in range(int(lay.nc[d])):
                diag = c * C // B
                row = _rank_independently(sc[c], diag, K)
                exp = row + [-1] * (K - len(row))
                assert list(sel[hi, g0 + c]) == exp
                ties += diag - len(np.unique(sc[c, :diag]))
    assert ties > 0, "the case should exercise the tie rule"
    O.validate_selection(sel, lay)                         # distinct and causal: a valid sel


def test_hand_worked_selection():
    with open(os.path.join(HERE, "golden", "scorer_hand.json")) as f:
        g = json.load(f)
    qi = _bits(np.array(g["q_index"], np.float64)[:, None, :])
    ki = _bits(np.array(g["k_index"], np.float64)[:, None, :])
    for k, key in ((3, "sel_k3"), (2, "sel_k2")):
        sel = O.select_topk(qi, ki, np.array(g["cu_seqlens"]), g["block"], g["chunk"], k)
        assert sel[0].tolist() == g[key]
