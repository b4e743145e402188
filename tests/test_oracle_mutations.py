"""Test the tests: plausible mistakes planted in the oracle (on the CPU) must fail a pin.

Each mutant replaces one oracle function with a wrong variant (a dropped term,
a wrong sign, index or scale, a transposed operand, a wrong rounding rule) and
the corresponding pin check must reject it.
"""
import numpy as np
import pytest

from oracle import brute
from oracle import dsa_oracle as o
from test_oracle_indexer import check_indexer_vs_brute
from test_oracle_mla import check_attention_vs_brute


def _indexer_ok(tiny_case, fmt="bf16", P=3):
    case = tiny_case(501, [11, 7], [2, 1], P, fmt)
    return check_indexer_vs_brute(case, topks=[2, 5, 20])


def _attention_ok(tiny_case):
    case = tiny_case(502, [13, 9], [2, 1], 3)
    idx, _ = o.indexer_topk(case.cache, case.block_table, case.seq_lens, case.qsl, case.q_idx, case.w, 4)
    return check_attention_vs_brute(case, idx, 0.3)


def _e4m3_ok():
    vals = np.array([1.0625, 1.1875, 0.7, -3.3, 0.004, 300.0, 1e5], dtype=np.float32)
    return all(int(c) == brute.e4m3_encode(float(v)) for v, c in zip(vals, o.f32_to_e4m3(vals)))


def test_unmutated_oracle_passes(tiny_case):
    assert _indexer_ok(tiny_case) and _indexer_ok(tiny_case, "fp8") and _attention_ok(tiny_case) and _e4m3_ok()


INDEXER_MUTANTS = {
    "relu_dropped": lambda q, w, k: (k @ np.asarray(q, float).T) @ np.asarray(w, float),
    "weight_inside_relu": lambda q, w, k: np.maximum((k @ np.asarray(q, float).T) * np.asarray(w, float), 0).sum(1),
    "relu_sign_flipped": lambda q, w, k: np.minimum(k @ np.asarray(q, float).T, 0) @ np.asarray(w, float),
    "head_weights_reversed": lambda q, w, k: np.maximum(k @ np.asarray(q, float).T, 0) @ np.asarray(w, float)[::-1],
}


@pytest.mark.parametrize("name", sorted(INDEXER_MUTANTS))
def test_indexer_mutants_are_caught(tiny_case, monkeypatch, name):
    monkeypatch.setattr(o, "index_scores", INDEXER_MUTANTS[name])
    assert not _indexer_ok(tiny_case)


def test_tie_break_mutant_is_caught(monkeypatch):
    def larger_position_first(scores, k):
        scores = np.asarray(scores, float)
        n = len(scores)
        if n <= k:
            chosen = np.arange(n)
        else:
            chosen = np.sort(np.lexsort((-np.arange(n), -scores))[:k])
        out = np.full(k, -1, np.int32)
        out[:len(chosen)] = chosen
        return out
    monkeypatch.setattr(o, "topk_select", larger_position_first)
    s = [1.0, 2.0, 2.0, 0.0, 2.0]
    assert o.topk_select(np.array(s), 2).tolist() != brute.topk(s, 2)


def test_off_by_one_position_mutant_is_caught(tiny_case, monkeypatch):
    real = o.row_positions

    def shifted(seq_lens, qsl):
        req, pos = real(seq_lens, qsl)
        return req, pos - 1
    monkeypatch.setattr(o, "row_positions", shifted)
    assert not _indexer_ok(tiny_case)


def test_fp8_scale_mutant_is_caught(tiny_case, monkeypatch):
    real = o.quantize_index_keys

    def wrong_scale(bits):
        codes, scale = real(bits)
        return codes, (scale * np.float32(448.0 / 240.0)).astype(np.float32)
    monkeypatch.setattr(o, "quantize_index_keys", wrong_scale)
    assert not _indexer_ok(tiny_case, "fp8")


def test_rounding_mutant_is_caught(monkeypatch):
    real = o.f32_to_e4m3

    def half_away(x):
        x = np.asarray(x, np.float32)
        nudged = np.nextafter(x, np.copysign(np.float32(np.inf), x))            # ties move away from zero
        return real(nudged)
    monkeypatch.setattr(o, "f32_to_e4m3", half_away)
    assert not _e4m3_ok()


ATTEND_MUTANTS = {
    "rope_term_dropped": lambda q, rows, scale, dl=512: _attend_variant(q, rows, scale, dl, rope=False),
    "scale_of_576": lambda q, rows, scale, dl=512: _attend_variant(q, rows, scale * 16 / 24, dl),
    "latent_offset_wrong": lambda q, rows, scale, dl=512: _attend_variant(q, rows, scale, dl, shift=1),
    "weights_transposed": lambda q, rows, scale, dl=512: _attend_variant(q, rows, scale, dl, transpose=True),
}


def _attend_variant(q, rows, scale, dl, rope=True, shift=0, transpose=False):
    q = np.asarray(q, float)
    if rows.shape[0] == 0:
        return np.zeros((q.shape[0], dl)), np.full(q.shape[0], -np.inf)
    z = scale * (q[:, :dl] @ rows[:, :dl].T + (q[:, dl:] @ rows[:, dl:].T if rope else 0))
    m = z.max(1, keepdims=True)
    p = np.exp(z - m)
    l = p.sum(1, keepdims=True)
    pn = p / l
    if transpose:   # softmax taken over heads instead of over selected tokens
        pn = np.exp(z - z.max(0, keepdims=True))
        pn = pn / pn.sum(0, keepdims=True)
    out = pn @ rows[:, shift:shift + dl]
    return out, (m + np.log(l))[:, 0]


@pytest.mark.parametrize("name", sorted(ATTEND_MUTANTS))
def test_attention_mutants_are_caught(tiny_case, monkeypatch, name):
    monkeypatch.setattr(o, "attend", ATTEND_MUTANTS[name])
    assert not _attention_ok(tiny_case)


def _pages_ok():
    """The page-selection pins: brute force over a few shapes with ties between pages."""
    for n, P, budget in [(17, 4, 2), (64, 8, 3), (100, 16, 7), (37, 8, 2)]:
        rng = np.random.default_rng(n * 7 + P)
        scores = rng.standard_normal(n)
        scores[rng.integers(0, n, max(1, n // 5))] = 0.5
        pages = o.page_topk_select(o.page_scores(scores, P), budget)
        positions = o.pages_to_positions(pages, P, n - 1)
        want_pages, want_pos = brute.page_select([float(x) for x in scores], P, budget)
        if [int(x) for x in pages if x >= 0] != want_pages or [int(x) for x in positions if x >= 0] != want_pos:
            return False
    return True


PAGE_MUTANTS = {
    # the page score as the sum, the mean or the first token of the page instead of the maximum
    "page_sum": ("page_scores", lambda s, P: np.array([np.sum(s[i:i + P]) for i in range(0, len(s), P)])),
    "page_mean": ("page_scores", lambda s, P: np.array([np.mean(s[i:i + P]) for i in range(0, len(s), P)])),
    "page_first": ("page_scores", lambda s, P: np.asarray(s, float)[::P].copy()),
    # a page index off by one when expanding to positions
    "expand_shifted": ("pages_to_positions", lambda pages, P, pos: np.array(
        [s for pg in sorted(int(x) for x in pages if x >= 0) for s in range((pg + 1) * P, (pg + 2) * P) if s <= pos]
        + [-1] * len(pages) * P, dtype=np.int32)[:len(pages) * P]),
}


def test_unmutated_page_selection_passes():
    assert _pages_ok()


@pytest.mark.parametrize("name", sorted(PAGE_MUTANTS))
def test_page_mutants_are_caught(monkeypatch, name):
    fn, bad = PAGE_MUTANTS[name]
    monkeypatch.setattr(o, fn, bad)
    assert not _pages_ok()


def test_dcp_share_of_k_mutant_is_caught(monkeypatch):
    """Keeping only k / world candidates per rank (a plausible shortcut) loses selections whenever the
    top scores cluster on one rank: the DCP pin against the single-device top-k must fail."""
    def share_of_k(scores, k, world):
        scores = np.asarray(scores, float)
        union = []
        for rank in range(world):
            pos = o.dcp_local_positions(len(scores), rank, world)
            local = o.topk_select(scores[pos], max(1, k // world))
            union += [(scores[pos[i]], int(pos[i])) for i in local if i >= 0]
        union.sort(key=lambda c: (-c[0], c[1]))
        out = np.full(k, -1, np.int32)
        chosen = sorted(p for _, p in union[:k])
        out[:len(chosen)] = chosen
        return out, None
    monkeypatch.setattr(o, "dcp_select", share_of_k)
    world, k, n = 4, 16, 400
    scores = np.random.default_rng(5).uniform(0, 1, n)
    scores[np.arange(0, 4 * k, world)] += 10.0
    assert not np.array_equal(o.dcp_select(scores, k, world)[0], o.topk_select(scores, k))


C8_MUTANTS = {
    # an int8-style scale, the scale applied twice, k_R quantised along with c_KV
    "scale_amax_over_127": lambda bits: (lambda x, s: (o.f32_to_e4m3((x / s[:, None]).astype(np.float32)), s))(
        o.bf16_to_f64(bits).astype(np.float32),
        np.where(np.abs(o.bf16_to_f64(bits)).max(-1) > 0, np.abs(o.bf16_to_f64(bits)).max(-1) / 127.0, 1.0).astype(np.float32)),
    "no_scale": lambda bits: (o.f32_to_e4m3(o.bf16_to_f64(bits).astype(np.float32)),
                              np.ones(bits.shape[0], np.float32)),
}


@pytest.mark.parametrize("name", sorted(C8_MUTANTS))
def test_c8_quantizer_mutants_are_caught(monkeypatch, name):
    import test_oracle_c8 as pins
    monkeypatch.setattr(o, "quantize_latent", C8_MUTANTS[name])
    with pytest.raises(AssertionError):
        pins.test_latent_quantizer_matches_exhaustive_nearest_code()
    with pytest.raises(AssertionError):
        pins.test_c8_attention_matches_brute_force()


def test_c8_rope_quantised_mutant_is_caught(monkeypatch):
    """k_R pushed through the c_KV quantizer as well: the stored rope columns change."""
    import test_oracle_c8 as pins
    real_append = o.PagedCache.append

    def append(self, c_kv_bits, k_rope_bits, slot_mapping, **kw):
        if self.latent_format == "e4m3":
            codes, scales = o.quantize_latent(k_rope_bits)
            k_rope_bits = wlm_bits(o.e4m3_to_f64(codes) * scales.astype(np.float64)[:, None])
        return real_append(self, c_kv_bits, k_rope_bits, slot_mapping, **kw)

    def wlm_bits(v):
        import workloads as wlm
        return wlm.bf16_bits(v.astype(np.float32))

    monkeypatch.setattr(o.PagedCache, "append", append)
    with pytest.raises(AssertionError):
        pins.test_rope_columns_are_stored_untouched()
