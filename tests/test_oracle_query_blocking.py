"""Pins of the oracle's query-blocked union reuse ("Making GLM-5.2 Sparse on TPUs", "Reuse pages across
queries").

The page's ratios (29.7x fewer page loads for 2.16x more score work at QB 64, Kp 32, U about 69) and its
uniform-random union (about 795 of 880 pages) are stored with their citation in
tests/golden/query_blocking_ratios.txt: the first pins the two ratio formulas, the second is met by the
closed form of the expected union size and by seeded draws.  Membership is pinned against loops; the
blocked attention (the union loaded once, each row masked back to its own pages, causality applied) must
equal each row's attention over its own pages, since the union is never truncated.
"""
import os

import numpy as np
import pytest

from oracle import brute
from oracle import dsa_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "query_blocking_ratios.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    return vals


def test_the_pages_ratios():
    g = _golden()
    qb, kp, u = int(g["qb"]), int(g["kp"]), int(g["union"])
    assert round(o.page_load_reduction(qb, kp, u), 1) == g["page_load_reduction"]
    assert round(o.score_work_expansion(u, kp), 2) == g["score_work_expansion"]


def test_uniform_random_selections_fill_most_of_the_pages():
    """Expected union of QB draws of Kp distinct pages out of N: N (1 - (1 - Kp/N)^QB)."""
    g = _golden()
    qb, kp, n = int(g["qb"]), int(g["kp"]), int(g["random_pages"])
    expected = n * (1 - (1 - kp / n) ** qb)
    assert abs(expected - g["random_union"]) <= 0.01 * g["random_union"]
    rng = np.random.default_rng(880)
    sizes = [len(o.page_union([rng.choice(n, kp, replace=False) for _ in range(qb)])) for _ in range(50)]
    assert abs(np.mean(sizes) - expected) <= 0.01 * expected
    assert max(sizes) <= o.union_capacity(qb, kp, n)


def test_union_and_membership_against_loops():
    rng = np.random.default_rng(3)
    for qb, kp, units in [(1, 3, 10), (4, 5, 12), (8, 2, 100), (3, 7, 7)]:
        lists = []
        for _ in range(qb):
            p = rng.choice(units, min(kp, units), replace=False)
            p = np.concatenate([p, -np.ones(kp - len(p), dtype=np.int64)])
            lists.append(p)
        u = o.page_union(lists)
        assert list(u) == sorted({int(x) for p in lists for x in p if x >= 0})
        assert len(u) <= o.union_capacity(qb, kp, units)
        m = o.union_membership(lists, u)
        assert m.tolist() == brute.membership([[int(x) for x in p] for p in lists], [int(x) for x in u])
        assert np.all(m.sum(axis=1) == [(np.asarray(p) >= 0).sum() for p in lists])


def test_locality_shaped_selections_reach_the_pages_regime():
    """Nearby rows whose page preferences mostly agree (workloads.locality_page_scores) select their top
    Kp pages with the oracle's page budget: at the calibrated noise the union is about the page's 69 of
    880 and the ratios about its 29.7x and 2.16x; no noise gives one shared selection (QB x fewer loads);
    very large noise tends to the uniform-random closed form; the union never exceeds its capacity."""
    import workloads as wlm
    g = _golden()
    qb, kp, n = int(g["qb"]), int(g["kp"]), int(g["random_pages"])

    def unions(noise, seeds):
        out = []
        for seed in seeds:
            sc = wlm.locality_page_scores(qb, n, noise, seed)
            u = o.page_union([o.page_topk_select(sc[q], kp) for q in range(qb)])
            assert len(u) <= o.union_capacity(qb, kp, n)
            out.append(len(u))
        return np.asarray(out, dtype=float)

    u = unions(0.17, range(30)).mean()
    assert abs(u - g["union"]) <= 0.1 * g["union"]
    assert abs(o.page_load_reduction(qb, kp, u) - g["page_load_reduction"]) <= 0.1 * g["page_load_reduction"]
    assert abs(o.score_work_expansion(u, kp) - g["score_work_expansion"]) <= 0.1 * g["score_work_expansion"]
    assert np.all(unions(0.0, range(3)) == kp) and o.page_load_reduction(qb, kp, kp) == qb
    means = [unions(s, range(10)).mean() for s in (0.05, 0.17, 1.0)]
    assert means[0] < means[1] < means[2]
    closed = n * (1 - (1 - kp / n) ** qb)
    assert abs(unions(50.0, range(10)).mean() - closed) <= 0.02 * closed


def test_identical_and_disjoint_selections_bound_the_ratios():
    kp, qb = 6, 5
    same = [np.arange(kp)] * qb
    assert len(o.page_union(same)) == kp and o.page_load_reduction(qb, kp, kp) == qb
    apart = [np.arange(kp) + kp * q for q in range(qb)]
    u = len(o.page_union(apart))
    assert u == qb * kp and o.page_load_reduction(qb, kp, u) == 1.0
    assert o.score_work_expansion(u, kp) == qb


@pytest.mark.parametrize("qb,kp,P", [(4, 3, 4), (6, 2, 8), (3, 5, 2)])
def test_blocked_attention_equals_each_rows_own_pages(qb, kp, P):
    """Rows of one request at positions base + i (prefill / verify rows), each with its own page
    selection among the visible pages; the blocked form over the union with membership and causal
    masks equals every row's attention over its own pages' visible tokens."""
    rng = np.random.default_rng(qb * 100 + kp * 10 + P)
    H, dl, dr = 2, 5, 2
    L = 60
    rows = rng.standard_normal((L, dl + dr))
    base = L - qb
    q_rows = rng.standard_normal((qb, H, dl + dr))
    row_pos = np.array([base + i for i in range(qb)])
    lists = []
    for i in range(qb):
        visible_pages = row_pos[i] // P + 1
        lists.append(np.sort(rng.choice(visible_pages, min(kp, visible_pages), replace=False)))
    u = o.page_union(lists)
    union_pos = np.concatenate([np.arange(pg * P, min(pg * P + P, L)) for pg in u])
    slot_of_token = np.concatenate([np.full(min(pg * P + P, L) - pg * P, j) for j, pg in enumerate(u)])
    member = o.union_membership(lists, u)[:, slot_of_token]
    out, lse = o.blocked_attend(q_rows, rows[union_pos], union_pos, member, row_pos, 0.3, dl)
    for i in range(qb):
        own = o.pages_to_positions(lists[i], P, int(row_pos[i]))
        own = own[own >= 0]
        ref_out, ref_lse = o.attend(q_rows[i], rows[own], 0.3, dl)
        assert np.allclose(out[i], ref_out, rtol=1e-12, atol=1e-12)
        assert np.allclose(lse[i], ref_lse, rtol=1e-12, atol=1e-12)


def test_a_dropped_mask_is_detected():
    """Without the membership mask the blocked form attends to other rows' pages: it must differ."""
    rng = np.random.default_rng(9)
    rows = rng.standard_normal((32, 6))
    q = rng.standard_normal((2, 2, 6))
    lists = [np.array([0, 1]), np.array([5, 6])]
    u = o.page_union(lists)
    pos = np.concatenate([np.arange(pg * 4, pg * 4 + 4) for pg in u])
    slot = np.repeat(np.arange(len(u)), 4)
    member = o.union_membership(lists, u)[:, slot]
    good, _ = o.blocked_attend(q, rows[pos], pos, member, np.array([31, 31]), 0.5, 4)
    bad, _ = o.blocked_attend(q, rows[pos], pos, np.ones_like(member), np.array([31, 31]), 0.5, 4)
    assert not np.allclose(good, bad)
