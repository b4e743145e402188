"""Pins of the oracle's page-granular selection ("Making GLM-5.2 Sparse on TPUs", "Make the
sparsity unit match the memory unit" and "Stream indexer scores over live context").

The page's worked example (four top tokens in four four-token pages: 4 / 16 / 8 positions) and its
score-size arithmetic (4.125 GiB of token scores, 33 MiB of 128-token page scores) are stored with
their citation in tests/golden/page_budget_example.txt.  Brute force over loops pins the page
maximum and the ranking; closed forms pin the special cases (page size 1 is token top-k, a budget
of every page is dense attention), and a planted invisible score checks that masks precede the
maximum.
"""
import os

import numpy as np
import pytest

from oracle import brute
from oracle import dsa_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_budget_example.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    return vals


def test_worked_example_four_pages_of_four_tokens():
    g = _golden()
    P, n_pages, k = int(g["page_size"]), int(g["pages"]), int(g["top_tokens"])
    rng = np.random.default_rng(7)
    scores = rng.uniform(0.0, 1.0, P * n_pages)
    top = [1, 6, 11, 12]                        # one top-scoring token in each page
    scores[top] = [10.0, 11.0, 12.0, 13.0]
    pos = P * n_pages - 1
    tok = o.topk_select(scores, k)
    assert sorted(int(x) for x in tok if x >= 0) == top
    assert len(top) == g["token_topk_positions"]
    # expanding the k tokens to their pages reads every token of those pages
    touched = sorted({t // P for t in top})
    expanded = o.pages_to_positions(np.array(touched), P, pos)
    assert int((expanded >= 0).sum()) == g["page_expansion_positions"]
    # a two-page budget reads two pages' tokens: the pages of the two best tokens
    pages = o.page_topk_select(o.page_scores(scores, P), 2)
    assert list(pages) == [2, 3]
    kept = o.pages_to_positions(pages, P, pos)
    assert int((kept >= 0).sum()) == g["two_page_budget_positions"]
    assert list(kept) == list(range(8, 16))


def test_page_scores_shrink_the_score_output_by_the_page_size():
    g = _golden()
    Q, L, P = int(g["queries"]), int(g["positions"]), int(g["pool_page"])
    token_bytes = Q * L * 4
    assert token_bytes / 2 ** 30 == g["token_score_gib"]
    n_pages = len(o.page_scores(np.zeros(L), P))
    assert n_pages == L // P
    assert round(Q * n_pages * 4 / 2 ** 20) == g["page_score_mib"]


@pytest.mark.parametrize("n,P,budget", [(1, 1, 1), (5, 2, 1), (17, 4, 2), (64, 8, 3), (100, 16, 7), (33, 64, 1),
                                        (40, 4, 100)])
def test_page_selection_matches_brute_force(n, P, budget):
    rng = np.random.default_rng(n * 131 + P)
    scores = rng.standard_normal(n)
    scores[rng.integers(0, n, max(1, n // 5))] = 0.5        # ties between pages
    pos = n - 1
    pages = o.page_topk_select(o.page_scores(scores, P), budget)
    positions = o.pages_to_positions(pages, P, pos)
    want_pages, want_pos = brute.page_select([float(x) for x in scores], P, budget)
    assert [int(x) for x in pages if x >= 0] == want_pages
    assert all(x == -1 for x in pages[len(want_pages):])
    assert [int(x) for x in positions if x >= 0] == want_pos
    assert len(positions) == budget * P


def test_page_size_one_is_token_topk():
    rng = np.random.default_rng(3)
    scores = rng.standard_normal(50)
    for k in (1, 7, 50, 60):
        assert np.array_equal(o.page_topk_select(o.page_scores(scores, 1), k), o.topk_select(scores, k))


def test_a_budget_of_every_page_is_dense():
    scores = np.random.default_rng(4).standard_normal(37)
    pages = o.page_topk_select(o.page_scores(scores, 8), 5)     # 37 positions -> 5 pages
    assert list(pages) == [0, 1, 2, 3, 4]
    assert list(o.pages_to_positions(pages, 8, 36)[:37]) == list(range(37))


def test_masks_precede_the_page_maximum(tiny_case):
    """A huge score just beyond the row's position, inside the row's last page, must not promote
    that page: the page score only sees visible tokens."""
    case = tiny_case(22, [29], [1], 8, "bf16")    # both head weights positive
    b, pos = case.rows()[0]
    assert pos == 28                                  # page 3 holds 24..31, visible 24..28
    # plant at position 30 (invisible, same page) the strongest of a few large candidate keys
    import workloads as wlm
    q, w = o.bf16_to_f64(case.q_idx[0]), case.w[0].astype(np.float64)
    cands = [30.0 * v for v in list(np.eye(case.d_index)) + list(-np.eye(case.d_index)) + list(q) + list(-q)]
    row30 = max((wlm.bf16_bits(np.asarray(c, dtype=np.float32)) for c in cands),
                key=lambda bits: o.index_scores(q, w, o.bf16_to_f64(bits[None, :]))[0])
    zeros = np.zeros((1, case.d_latent + case.d_rope), dtype=np.uint16)
    case.cache.append(zeros[:, :case.d_latent], zeros[:, case.d_latent:], case.slots(0, [30]),
                      k_idx_bits=row30[None, :])
    pages, positions, ps, ts = o.page_indexer_topk(case.cache, case.block_table, case.seq_lens, case.qsl,
                                                   case.q_idx, case.w, 1)
    assert len(ps[0]) == 4 and len(ts[0]) == pos + 1
    planted = o.index_scores(q, w, o.bf16_to_f64(row30[None, :]))[0]
    assert planted > ts[0].max()                      # it would win page 3 the budget if it were seen
    assert ps[0][3] == ts[0][24:29].max()             # the last page scores only its visible tokens
    want_pages, _ = brute.page_select([float(x) for x in ts[0]], 8, 1)
    assert list(pages[0]) == want_pages
    if want_pages != [3]:
        assert 3 not in list(pages[0])
    assert all(int(x) <= pos for x in positions[0] if x >= 0)


def test_page_indexer_matches_brute_force(tiny_case):
    case = tiny_case(33, [37, 20], [2, 1], 4, "fp8")
    pages, positions, ps, ts = o.page_indexer_topk(case.cache, case.block_table, case.seq_lens, case.qsl,
                                                   case.q_idx, case.w, 3)
    for r, (b, pos) in enumerate(case.rows()):
        want_pages, want_pos = brute.page_select([float(x) for x in ts[r]], case.P, 3)
        assert [int(x) for x in pages[r] if x >= 0] == want_pages
        assert [int(x) for x in positions[r] if x >= 0] == want_pos
