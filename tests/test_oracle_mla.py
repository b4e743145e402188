"""Pins of the oracle's sparse absorbed MLA and split merge."""
import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle import brute
from oracle import dsa_oracle as o


def check_attention_vs_brute(case, idx, scale):
    out, lse = o.sparse_mla(case.cache, case.block_table, case.seq_lens, case.qsl, case.q, idx, scale)
    for r, (b, pos) in enumerate(case.rows()):
        sel = [int(s) for s in idx[r] if 0 <= s <= pos]
        rows = [[brute.bf16(x) for x in case.latent[b][s]] for s in sel]
        qh = [[brute.bf16(x) for x in h] for h in case.q[r]]
        ref_o, ref_l = brute.attention(qh, rows, scale, case.d_latent)
        if not (np.allclose(out[r], ref_o, rtol=1e-11, atol=1e-13) and np.allclose(lse[r], ref_l, rtol=1e-12)):
            return False
    return True


@pytest.mark.parametrize("seq_lens,q_lens,P", [([9, 14], [1, 3], 1), ([30, 70], [2, 1], 64), ([17], [5], 3)])
def test_attention_matches_brute_force(tiny_case, seq_lens, q_lens, P):
    case = tiny_case(200 + P, seq_lens, q_lens, P)
    idx, _ = o.indexer_topk(case.cache, case.block_table, case.seq_lens, case.qsl, case.q_idx, case.w, 5)
    assert check_attention_vs_brute(case, idx, 0.37)


def test_sparse_with_k_at_least_context_equals_dense(tiny_case):
    """Selecting every visible position reproduces dense attention over 0..pos."""
    case = tiny_case(7, [25, 40], [3, 1], 4)
    idx, _ = o.indexer_topk(case.cache, case.block_table, case.seq_lens, case.qsl, case.q_idx, case.w, 64)
    out, lse = o.sparse_mla(case.cache, case.block_table, case.seq_lens, case.qsl, case.q, idx, 0.25)
    for r, (b, pos) in enumerate(case.rows()):
        kv = o.bf16_to_f64(case.latent[b][:pos + 1])
        q = o.bf16_to_f64(case.q[r])
        z = 0.25 * q @ kv.T
        np.testing.assert_allclose(out[r], softmax(z, axis=1) @ kv[:, :case.d_latent], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse[r], logsumexp(z, axis=1), rtol=1e-13)


def test_absorbed_equals_explicit_per_head_up_projection():
    """W_UK absorbed into q and W_UV applied after the latent sum equals explicit per-head K/V.

    Explicit: K_h[s] = W_UK_h c[s] (192), V_h[s] = W_UV_h c[s] (256), q_h = [q_nope (192) | q_R (64)],
    score = (q_nope . K_h[s] + q_R . k_R[s]) / sqrt(192 + 64).  Absorbed: q_lat = W_UK_h^T q_nope (512),
    score = (q_lat . c[s] + q_R . k_R[s]) / 16 and out_h = W_UV_h (sum_s p_s c[s])."""
    rng = np.random.default_rng(3)
    Hh, m, dl, dn, dr, dv = 4, 23, 512, 192, 64, 256
    c = rng.standard_normal((m, dl))
    kr = rng.standard_normal((m, dr))
    W_UK = rng.standard_normal((Hh, dn, dl)) / np.sqrt(dl)
    W_UV = rng.standard_normal((Hh, dv, dl)) / np.sqrt(dl)
    q_nope = rng.standard_normal((Hh, dn))
    q_r = rng.standard_normal((Hh, dr))
    scale = 1.0 / np.sqrt(dn + dr)
    assert scale == 1.0 / 16
    q_lat = np.einsum("hnl,hn->hl", W_UK, q_nope)
    out_lat, lse_abs = o.attend(np.concatenate([q_lat, q_r], axis=1), np.concatenate([c, kr], axis=1), scale, dl)
    for h in range(Hh):
        K = c @ W_UK[h].T
        V = c @ W_UV[h].T
        z = (K @ q_nope[h] + kr @ q_r[h]) * scale
        np.testing.assert_allclose(W_UV[h] @ out_lat[h], softmax(z) @ V, rtol=1e-10, atol=1e-12)
        assert lse_abs[h] == pytest.approx(logsumexp(z), rel=1e-12)


def test_closed_forms():
    rng = np.random.default_rng(4)
    rows = rng.standard_normal((9, 10))
    q = rng.standard_normal((3, 10))
    # one selected token: out = c[s], lse = z_s
    out, lse = o.attend(q, rows[4:5], 0.5, 7)
    np.testing.assert_allclose(out, np.repeat(rows[4:5, :7], 3, axis=0), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, 0.5 * q @ rows[4], rtol=1e-14)
    # q = 0: uniform weights -> the mean of the selected latents, lse = ln |T|
    out, lse = o.attend(np.zeros((2, 10)), rows, 0.5, 7)
    np.testing.assert_allclose(out, np.repeat(rows[:, :7].mean(axis=0, keepdims=True), 2, axis=0), atol=1e-15)
    np.testing.assert_allclose(lse, np.log(9.0), rtol=1e-15)
    # identical latents: out equals that latent whatever the weights
    same = np.repeat(rows[2:3], 6, axis=0)
    same[:, 7:] = rng.standard_normal((6, 3))
    out, _ = o.attend(q, same, 0.5, 7)
    np.testing.assert_allclose(out, np.repeat(rows[2:3, :7], 3, axis=0), atol=1e-14)
    # nothing selected: out 0, lse -inf
    out, lse = o.attend(q, rows[:0], 0.5, 7)
    assert not out.any() and np.all(np.isneginf(lse))


def test_lse_merge_of_any_partition_equals_the_whole():
    rng = np.random.default_rng(5)
    rows = rng.standard_normal((40, 12)) * 3
    q = rng.standard_normal((4, 12))
    whole = o.attend(q, rows, 0.7, 9)
    for trial in range(5):
        cuts = np.sort(rng.choice(np.arange(1, 40), size=trial + 1, replace=False))
        parts = [o.attend(q, piece, 0.7, 9) for piece in np.split(rows, cuts)]
        out, lse = o.lse_merge(parts + [o.attend(q, rows[:0], 0.7, 9)])   # an empty piece merges as nothing
        np.testing.assert_allclose(out, whole[0], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse, whole[1], rtol=1e-13)


def test_padding_and_out_of_range_entries_are_skipped(tiny_case):
    case = tiny_case(8, [20], [2], 4)
    good = np.array([[3, 7, 11, -1, -1], [0, 18, 19, -1, -1]])
    noisy = np.array([[3, 7, 11, 19, -1], [0, 18, 19, 25, -7]])     # 19 > pos 18 for row 0; 25 beyond context
    a = o.sparse_mla(case.cache, case.block_table, [20], np.array([0, 2]), case.q, good, 0.3)
    b = o.sparse_mla(case.cache, case.block_table, [20], np.array([0, 2]), case.q, noisy, 0.3)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_outputs_invariant_under_page_permutation(tiny_case):
    a = tiny_case(12, [33, 9], [1, 2], 4)
    b = tiny_case(12, [33, 9], [1, 2], 4)
    perm = np.random.default_rng(9).permutation(b.num_pages)
    b.block_table = np.where(a.block_table >= 0, perm[np.maximum(a.block_table, 0)], -1).astype(np.int32)
    b.cache = o.PagedCache(b.num_pages, 4, "bf16", b.d_latent, b.d_rope, b.d_index)
    for r, L in enumerate(b.seq_lens):
        b.cache.append(b.latent[r][:, :b.d_latent], b.latent[r][:, b.d_latent:], b.slots(r, np.arange(L)),
                       k_idx_bits=b.keys[r])
    idx, _ = o.indexer_topk(a.cache, a.block_table, a.seq_lens, a.qsl, a.q_idx, a.w, 6)
    ra = o.sparse_mla(a.cache, a.block_table, a.seq_lens, a.qsl, a.q, idx, 0.2)
    rb = o.sparse_mla(b.cache, b.block_table, b.seq_lens, b.qsl, b.q, idx, 0.2)
    np.testing.assert_array_equal(ra[0], rb[0])
    np.testing.assert_array_equal(ra[1], rb[1])


def test_global_page_ids_in_place_of_local_ones_change_the_output(tiny_case):
    """Fault injection from the pages' data-parallel test proposal: a page table holding another
    request's page ids must change the result (the check that would catch it is not blind)."""
    case = tiny_case(13, [24, 24], [1, 1], 4)
    idx, _ = o.indexer_topk(case.cache, case.block_table, case.seq_lens, case.qsl, case.q_idx, case.w, 8)
    good = o.sparse_mla(case.cache, case.block_table, case.seq_lens, case.qsl, case.q, idx, 0.2)
    bad_bt = case.block_table.copy()
    bad_bt[1] = case.block_table[0]
    bad = o.sparse_mla(case.cache, bad_bt, case.seq_lens, case.qsl, case.q, idx, 0.2)
    assert np.abs(bad[0][1] - good[0][1]).max() > 1e-3
    np.testing.assert_array_equal(bad[0][0], good[0][0])
