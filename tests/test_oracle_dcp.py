"""Pins of the oracle's decode-context-parallel steps ("Serving GLM-5.2-504B on 8x RTX PRO 6000
GPUs", "Reaching 240K context with DCP": the KV is sharded along the sequence across the ranks).

The exchange must be exact: the top-k of the union of every rank's local top-k is the top-k of the
whole row, and the LSE merge of the ranks' partial attention is the attention over the whole
selection.  Both are checked against the single-device definitions, including rows whose top
scores all sit on one rank, ties across ranks and rows shorter than k.
"""
import numpy as np
import pytest

from oracle import dsa_oracle as o


@pytest.mark.parametrize("world", [1, 2, 3, 8])
@pytest.mark.parametrize("n,k", [(1, 4), (7, 4), (100, 8), (513, 64), (40, 100)])
def test_dcp_selection_is_the_single_device_topk(world, n, k):
    rng = np.random.default_rng(world * 1000 + n + k)
    scores = rng.standard_normal(n)
    scores[rng.integers(0, n, max(1, n // 4))] = 0.25         # ties, also across ranks
    sel, cand = o.dcp_select(scores, k, world)
    assert np.array_equal(sel, o.topk_select(scores, k))
    assert len(cand) == world and all(len(c) <= k for c in cand)


def test_top_scores_on_one_rank():
    """Every top-k position lies on rank 0: a per-rank share of k / world would lose most of them."""
    world, k, n = 4, 16, 400
    scores = np.random.default_rng(5).uniform(0, 1, n)
    scores[np.arange(0, 4 * k, world)] += 10.0                # positions 0, 4, 8, ...: rank 0
    sel, cand = o.dcp_select(scores, k, world)
    assert np.array_equal(sel, o.topk_select(scores, k))
    assert all(s % world == 0 for s in sel)


def test_interleave_partitions_the_positions():
    for L, world in [(1, 2), (10, 3), (257, 8)]:
        parts = [o.dcp_local_positions(L, r, world) for r in range(world)]
        allp = np.sort(np.concatenate(parts))
        assert np.array_equal(allp, np.arange(L))
        assert all(np.all(p % world == r) for r, p in enumerate(parts))


@pytest.mark.parametrize("world", [1, 2, 5])
def test_dcp_attention_is_the_attention_over_the_selection(world):
    rng = np.random.default_rng(11 + world)
    L, H, dl, dr, k = 90, 3, 6, 2, 20
    rows = rng.standard_normal((L, dl + dr))
    q = rng.standard_normal((H, dl + dr))
    scores = rng.standard_normal(L)
    sel, _ = o.dcp_select(scores, k, world)
    out, lse = o.dcp_attend(q, lambda pos: rows[pos], sel, world, 0.3, dl)
    ref_out, ref_lse = o.attend(q, rows[sel[sel >= 0]], 0.3, dl)
    assert np.allclose(out, ref_out, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_a_rank_without_selected_positions_contributes_nothing():
    rng = np.random.default_rng(3)
    rows = rng.standard_normal((12, 5))
    q = rng.standard_normal((2, 5))
    sel = np.array([0, 2, 4, 6, -1, -1])                      # world 2: all on rank 0
    out, lse = o.dcp_attend(q, lambda pos: rows[pos], sel, 2, 0.5, 4)
    ref_out, ref_lse = o.attend(q, rows[[0, 2, 4, 6]], 0.5, 4)
    assert np.allclose(out, ref_out) and np.allclose(lse, ref_lse)
