"""Pins of the oracle's lightning indexer and top-k selection."""
import numpy as np
import pytest

from oracle import brute
from oracle import dsa_oracle as o


def _brute_row(case, r, b, pos, codes_scales=None):
    """Pure-Python scores over positions 0..pos from the raw generated data."""
    q = [[brute.bf16(x) for x in h] for h in case.q_idx[r]]
    w = [float(x) for x in case.w[r]]
    out = []
    for s in range(pos + 1):
        if case.key_format == "bf16":
            key = [brute.bf16(x) for x in case.keys[b][s]]
        else:
            codes, scale = brute.quantize_key([brute.bf16(x) for x in case.keys[b][s]])
            key = [brute.e4m3_value(c) * scale for c in codes]
        out.append(brute.score(q, w, key))
    return out


def check_indexer_vs_brute(case, topks):
    idx_all = {}
    for k in topks:
        idx, scores = o.indexer_topk(case.cache, case.block_table, case.seq_lens, case.qsl, case.q_idx, case.w, k)
        idx_all[k] = idx
        for r, (b, pos) in enumerate(case.rows()):
            ref = _brute_row(case, r, b, pos)
            if len(ref) != len(scores[r]) or not np.allclose(scores[r], ref, rtol=1e-12, atol=1e-12):
                return False
            want = brute.topk(ref, k)
            got = [int(x) for x in idx[r] if x >= 0]
            if got != want or any(x != -1 for x in idx[r][len(got):]):
                return False
    return True


CASES = [
    # (seq_lens, q_lens, page size, key format)
    ([5, 9], [1, 1], 1, "bf16"),
    ([7, 12, 4], [1, 3, 2], 3, "bf16"),
    ([70, 65], [2, 1], 64, "bf16"),
    ([13, 17], [4, 1], 3, "fp8"),
    ([64, 129], [1, 2], 64, "fp8"),
]


@pytest.mark.parametrize("seq_lens,q_lens,P,fmt", CASES)
def test_indexer_and_topk_match_brute_force(tiny_case, seq_lens, q_lens, P, fmt):
    case = tiny_case(100 + P, seq_lens, q_lens, P, fmt)
    L = max(seq_lens)
    assert check_indexer_vs_brute(case, topks=[1, 3, L - 1, L, L + 5])


def test_fp8_score_factors_the_token_scale(tiny_case):
    """I(s) with dequantised keys equals sum_h w_h * scale_s * ReLU(q_h . code_s)."""
    case = tiny_case(9, [40], [1], 8, "fp8", n_idx_heads=3, d_index=5)
    _, scores = o.indexer_topk(case.cache, case.block_table, case.seq_lens, case.qsl, case.q_idx, case.w, 4)
    q = o.bf16_to_f64(case.q_idx[0])
    for s in range(40):
        pg, off = case.block_table[0, s // 8], s % 8
        k8 = o.e4m3_to_f64(case.cache.index_keys[pg, off])
        scale = float(case.cache.index_scales[pg, off])
        ref = sum(float(case.w[0, h]) * scale * max(0.0, float(q[h] @ k8)) for h in range(3))
        assert scores[0][s] == pytest.approx(ref, rel=1e-12, abs=1e-14)


def test_top1_with_one_head_is_the_relu_argmax(tiny_case):
    case = tiny_case(21, [50], [1], 4, "bf16", n_idx_heads=1)
    case.w[:] = 1.0
    idx, scores = o.indexer_topk(case.cache, case.block_table, case.seq_lens, case.qsl, case.q_idx, case.w, 1)
    keys = case.cache.index_key_rows(case.block_table[0], np.arange(50))
    dots = np.maximum(keys @ o.bf16_to_f64(case.q_idx[0, 0]), 0)
    assert idx[0, 0] == int(np.argmax(dots))


def test_mask_precedes_selection(tiny_case):
    """A huge score planted beyond the row's position is never selected and changes nothing."""
    case = tiny_case(33, [30], [3], 4, "bf16")
    idx0, _ = o.indexer_topk(case.cache, case.block_table, case.seq_lens, case.qsl, case.q_idx, case.w, 5)
    # key at the last position aligned with every query head -> huge positive score for all rows
    q = o.bf16_to_f64(case.q_idx).sum(axis=(0, 1))
    import workloads as wlm
    big = wlm.bf16_bits((1e3 * np.sign(q)).astype(np.float32))
    pg, off = case.block_table[0, 29 // 4], 29 % 4
    case.cache.index_keys[pg, off] = big
    idx1, _ = o.indexer_topk(case.cache, case.block_table, case.seq_lens, case.qsl, case.q_idx, case.w, 5)
    # rows at positions 27 and 28 cannot see position 29
    assert np.array_equal(idx0[:2], idx1[:2])
    assert 29 not in idx1[0] and 29 not in idx1[1]


def test_ties_prefer_smaller_positions():
    s = np.array([1.0, 3.0, 2.0, 3.0, 3.0, 0.5, 3.0])
    assert o.topk_select(s, 3).tolist() == [1, 3, 4]
    assert o.topk_select(s, 5).tolist() == [1, 2, 3, 4, 6]
    assert o.topk_select(np.array([-0.0, 0.0, 0.0]), 2).tolist() == [0, 1]


def test_short_context_selects_everything_and_pads():
    assert o.topk_select(np.array([0.3, -2.0, 1.0]), 5).tolist() == [0, 1, 2, -1, -1]
    assert o.topk_select(np.array([0.3, -2.0, 1.0]), 3).tolist() == [0, 1, 2]


def test_scores_invariant_under_page_permutation(tiny_case):
    a = tiny_case(44, [37, 20], [2, 1], 4, "fp8")
    b = tiny_case(44, [37, 20], [2, 1], 4, "fp8")
    # same logical data, different physical placement
    rng = np.random.default_rng(1)
    perm = rng.permutation(b.num_pages)
    b.block_table = np.where(a.block_table >= 0, perm[np.maximum(a.block_table, 0)], -1).astype(np.int32)
    from oracle import dsa_oracle as o2
    b.cache = o2.PagedCache(b.num_pages, 4, "fp8", b.d_latent, b.d_rope, b.d_index)
    for r, L in enumerate(b.seq_lens):
        b.cache.append(b.latent[r][:, :b.d_latent], b.latent[r][:, b.d_latent:], b.slots(r, np.arange(L)),
                       k_idx_bits=b.keys[r])
    ia, sa = o.indexer_topk(a.cache, a.block_table, a.seq_lens, a.qsl, a.q_idx, a.w, 6)
    ib, sb = o.indexer_topk(b.cache, b.block_table, b.seq_lens, b.qsl, b.q_idx, b.w, 6)
    assert np.array_equal(ia, ib)
    for x, y in zip(sa, sb):
        assert np.array_equal(x, y)


def test_rows_invariant_under_request_permutation(tiny_case):
    case = tiny_case(55, [23, 31, 17], [1, 2, 1], 4, "bf16")
    idx, scores = o.indexer_topk(case.cache, case.block_table, case.seq_lens, case.qsl, case.q_idx, case.w, 7)
    order = [2, 0, 1]
    rows_of = {0: [0], 1: [1, 2], 2: [3]}
    new_rows = sum((rows_of[b] for b in order), [])
    qsl = np.concatenate([[0], np.cumsum([case.q_lens[b] for b in order])]).astype(np.int32)
    idx2, scores2 = o.indexer_topk(case.cache, case.block_table[order], [case.seq_lens[b] for b in order], qsl,
                                   case.q_idx[new_rows], case.w[new_rows], 7)
    assert np.array_equal(idx2, idx[new_rows])


def test_chunked_rows_equal_one_shot_and_decode_is_a_one_row_extend(tiny_case):
    """Rows of a 6-token chunk scored in one call equal the same rows split into 2+4, and a
    decode row equals the last row of an extend (positions follow L - q_len + i)."""
    case = tiny_case(66, [40], [6], 4, "bf16")
    idx_all, s_all = o.indexer_topk(case.cache, case.block_table, [40], np.array([0, 6]), case.q_idx, case.w, 9)
    idx_a, s_a = o.indexer_topk(case.cache, case.block_table, [36], np.array([0, 2]), case.q_idx[:2], case.w[:2], 9)
    idx_b, s_b = o.indexer_topk(case.cache, case.block_table, [40], np.array([0, 4]), case.q_idx[2:], case.w[2:], 9)
    assert np.array_equal(np.concatenate([idx_a, idx_b]), idx_all)
    idx_d, s_d = o.indexer_topk(case.cache, case.block_table, [40], np.array([0, 1]), case.q_idx[5:], case.w[5:], 9)
    assert np.array_equal(idx_d[0], idx_all[5]) and np.array_equal(s_d[0], s_all[5])


def test_shared_layer_cache_cannot_score():
    c = o.PagedCache(4, 4, None, 6, 3, 4)
    with pytest.raises(ValueError):
        o.indexer_topk(c, np.zeros((1, 4), np.int32), [3], np.array([0, 1]), np.zeros((1, 2, 4), np.uint16),
                       np.zeros((1, 2), np.float32), 2)
