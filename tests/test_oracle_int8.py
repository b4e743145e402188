"""Pins of the oracle's int8 index keys with binary16 scales ("GLM-5.2 on vLLM Ascend", section 7
"GLM-5.2 shared-indexer construction" and "Quantization and Hardware Branches": one hardware family
keeps its indexer cache as INT8 keys with FP16 scales, beside e4m3 keys with FP32 scales).

The binary16 codec is pinned against a pure-Python decoder written from the IEEE format and an
exhaustive nearest-value search; the quantizer element by element against an exhaustive
nearest-code search; integer-valued rows must come back exactly; the round trip obeys half a
code step; scores over an int8 cache match the pure-Python brute force and factor the token's
scale; and planted mistakes in the quantizer (the e4m3 scale rule, an unrounded scale, truncation,
an amax / 128 scale with the code -128) are each caught.
"""
import numpy as np
import pytest

import workloads as wlm
from oracle import brute
from oracle import dsa_oracle as o


def _key_rows(seed, n, width=128):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, width)).astype(np.float32)
    x[0] = 0.0                                              # amax 0: scale 1, codes 0
    x[1] *= np.float32(2.0 ** -30)                          # amax / 127 below half's subnormal range
    x[2, :] = np.float32(-0.75)                             # constant row: every code is -127
    x[3] *= np.float32(2.0 ** 24)                           # amax / 127 beyond 65504: the scale is held there
    x[4] *= np.float32(2.0 ** -17)                          # scale in half's subnormal range
    x[5, 3] = 127.0                                         # scale exactly 1
    return wlm.bf16_bits(x)


def test_f16_decoder_matches_the_ieee_definition_for_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint16)
    got = o.f16_to_f64(bits)
    want = np.array([brute.f16_value(int(b)) for b in bits])
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all()
    assert o.f16_to_f64(np.uint16(0x7BFF)) == 65504.0 and o.f16_to_f64(np.uint16(0x0001)) == 2.0 ** -24


def test_f16_rounding_matches_exhaustive_nearest_search():
    rng = np.random.default_rng(3)
    vals = [float(v) for v in (np.exp2(rng.uniform(-26, 17, 300))).astype(np.float32)]
    # exact midpoints between neighbouring halves (ties) in the normal and subnormal ranges
    for b in (0x3C00, 0x3C01, 0x0001, 0x0002, 0x03FF, 0x0400, 0x7BFE, 0x2E66):
        lo, hi = brute.f16_value(b), brute.f16_value(b + 1)
        vals.append((lo + hi) / 2)
    vals += [0.0, 65504.0, 65519.0, 65520.0, 1e9, 2.0 ** -25, 2.0 ** -25 * 1.0001]
    got = o.f32_to_f16(np.array(vals, dtype=np.float32))
    for v, g in zip(vals, got):
        assert int(g) == brute.f16_nearest(float(np.float32(v))), v


def test_int8_quantizer_matches_exhaustive_nearest_code():
    bits = _key_rows(1, 8, width=32)
    codes, scales = o.quantize_index_keys_int8(bits)
    assert codes.dtype == np.int8 and scales.dtype == np.uint16
    for t in range(bits.shape[0]):
        want_codes, want_scale = brute.quantize_key_int8([brute.bf16(b) for b in bits[t]])
        assert int(scales[t]) == want_scale, f"row {t}"
        assert [int(c) for c in codes[t]] == want_codes, f"row {t}"


def test_edge_rows():
    bits = _key_rows(2, 8)
    codes, scales = o.quantize_index_keys_int8(bits)
    s = o.f16_to_f64(scales)
    assert s[0] == 1.0 and np.all(codes[0] == 0)
    assert scales[1] == 1 and s[1] == 2.0 ** -24                  # the smallest positive half
    assert np.all(codes[2] == -127)
    assert s[3] == 65504.0 and np.abs(codes[3]).max() == 127       # held at the largest finite half
    assert 0 < s[4] < 2.0 ** -14                                   # a subnormal half
    assert s[5] == 1.0 and codes[5, 3] == 127
    assert codes.min() >= -127


def test_integer_rows_come_back_exactly():
    rng = np.random.default_rng(4)
    ints = rng.integers(-127, 128, (6, 128)).astype(np.float32)
    ints[:, 0] = 127.0                                            # amax 127: scale 127/127 = 1
    for shift in (0, -5, 3):                                       # power-of-two scales are exact halves
        x = ints * np.float32(2.0 ** shift)
        codes, scales = o.quantize_index_keys_int8(wlm.bf16_bits(x))
        assert np.all(o.f16_to_f64(scales) == 2.0 ** shift)
        assert np.array_equal(codes.astype(np.float32), ints)


def test_round_trip_is_within_half_a_code_step():
    bits = _key_rows(5, 64)
    codes, scales = o.quantize_index_keys_int8(bits)
    x = o.bf16_to_f64(bits)
    s = o.f16_to_f64(scales)[:, None]
    deq = codes.astype(np.float64) * s
    amax = np.abs(x).max(axis=1, keepdims=True)
    # half a step, the float32 quotient's own rounding, and what the clamp at 127 costs when the
    # half-rounded scale sits below amax / 127 (at most 2^-11 relative, so at most 127 * 2^-11 steps)
    bound = s / 2 + np.abs(x) * 2.0 ** -23 + np.maximum(amax - 127 * s, 0)
    ok = np.abs(deq - x) <= bound * (1 + 2.0 ** -20)
    ok[1] = True                                                    # scale held at 2^-24: codes only bounded
    ok[3] = True                                                    # scale held at 65504: codes saturate
    assert ok.all()
    assert codes.min() >= -127


def test_every_int8_code_splits_into_two_exact_e4m3_terms():
    """The GPU reads int8 keys as hi + lo with hi = e4m3(v) (nearest-even) and lo = v - hi: for every code
    both terms are exact e4m3 values, so the two MMA chains sum to v exactly; int8 values are also bf16 values."""
    v = np.arange(-127, 128, dtype=np.float32)
    hi = o.e4m3_to_f64(o.f32_to_e4m3(v))
    lo = v - hi
    assert np.array_equal(o.e4m3_to_f64(o.f32_to_e4m3(lo.astype(np.float32))), lo)
    assert np.array_equal(hi + lo, v) and np.abs(lo).max() == 4.0
    assert all(brute.e4m3_value(brute.e4m3_encode(float(x))) == x for x in hi)      # hi exact by exhaustive search
    assert np.array_equal(o.bf16_to_f64(wlm.bf16_bits(v)), v)


def _brute_row_int8(case, r, b, pos):
    q = [[brute.bf16(x) for x in h] for h in case.q_idx[r]]
    w = [float(x) for x in case.w[r]]
    out = []
    for s in range(pos + 1):
        codes, sbits = brute.quantize_key_int8([brute.bf16(x) for x in case.keys[b][s]])
        scale = brute.f16_value(sbits)
        out.append(brute.score(q, w, [c * scale for c in codes]))
    return out


def _int8_indexer_ok(case, topks):
    for k in topks:
        idx, scores = o.indexer_topk(case.cache, case.block_table, case.seq_lens, case.qsl, case.q_idx, case.w, k)
        for r, (b, pos) in enumerate(case.rows()):
            ref = _brute_row_int8(case, r, b, pos)
            if len(ref) != len(scores[r]) or not np.allclose(scores[r], ref, rtol=1e-12, atol=1e-12):
                return False
            got = [int(x) for x in idx[r] if x >= 0]
            if got != brute.topk(ref, k):
                return False
    return True


@pytest.mark.parametrize("seq_lens,q_lens,P", [([13, 17], [4, 1], 3), ([64, 129], [1, 2], 64), ([9], [9], 1)])
def test_int8_indexer_matches_brute_force(tiny_case, seq_lens, q_lens, P):
    case = tiny_case(700 + P, seq_lens, q_lens, P, "int8")
    L = max(seq_lens)
    assert _int8_indexer_ok(case, [1, 3, L - 1, L, L + 5])


def test_int8_score_factors_the_token_scale(tiny_case):
    """I(s) over dequantised keys equals sum_h w_h * scale_s * ReLU(q_h . code_s)."""
    case = tiny_case(11, [40], [1], 8, "int8", n_idx_heads=3, d_index=5)
    _, scores = o.indexer_topk(case.cache, case.block_table, case.seq_lens, case.qsl, case.q_idx, case.w, 4)
    q = o.bf16_to_f64(case.q_idx[0])
    w = case.w[0].astype(np.float64)
    pg, off = case.cache.slots(case.block_table[0], np.arange(40))
    codes = case.cache.index_keys[pg, off].astype(np.float64)
    scale = o.f16_to_f64(case.cache.index_scales[pg, off])
    factored = scale * (np.maximum(codes @ q.T, 0) @ w)
    assert np.allclose(scores[0], factored, rtol=1e-13, atol=1e-13)


def test_prequantised_int8_keys_are_stored_as_given(tiny_case):
    case = tiny_case(12, [10], [1], 4, "int8")
    codes, scales = o.quantize_index_keys_int8(case.keys[0])
    c = o.PagedCache(case.num_pages, 4, "int8", case.d_latent, case.d_rope, case.d_index)
    c.append(case.latent[0][:, :case.d_latent], case.latent[0][:, case.d_latent:], case.slots(0, np.arange(10)),
             k_idx_codes=codes, k_idx_scales=scales)
    assert np.array_equal(c.index_keys, case.cache.index_keys)
    assert np.array_equal(c.index_scales, case.cache.index_scales)


# ---------------------------------------------------------------------------
# planted mistakes in the quantizer must fail the exhaustive nearest-code pin
# ---------------------------------------------------------------------------
_quantize = o.quantize_index_keys_int8          # the unmutated quantizer, for the mutants' other half
def _quantizer_ok():
    bits = _key_rows(6, 8, width=32)
    codes, scales = o.quantize_index_keys_int8(bits)
    for t in range(bits.shape[0]):
        want_codes, want_scale = brute.quantize_key_int8([brute.bf16(b) for b in bits[t]])
        if int(scales[t]) != want_scale or [int(c) for c in codes[t]] != want_codes:
            return False
    return True


def _e4m3_scale_rule(bits):
    x = o.bf16_to_f64(bits).astype(np.float32)
    s16 = o.f32_to_f16(np.max(np.abs(x), axis=-1) / np.float32(448.0))
    s16 = np.where(s16 == 0, np.uint16(0x3C00), s16).astype(np.uint16)
    s = o.f16_to_f64(s16).astype(np.float32)
    return np.clip(np.rint(x / s[:, None]), -127, 127).astype(np.int8), s16


def _unrounded_scale(bits):
    _, s16 = _quantize(bits)
    x = o.bf16_to_f64(bits).astype(np.float32)
    s32 = np.max(np.abs(x), axis=-1) / np.float32(127.0)
    s32 = np.where(s32 > 0, s32, np.float32(1.0)).astype(np.float32)
    return np.clip(np.rint(x / s32[:, None]), -127, 127).astype(np.int8), s16


def _truncation(bits):
    _, s16 = _quantize(bits)
    x = o.bf16_to_f64(bits).astype(np.float32)
    s = o.f16_to_f64(s16).astype(np.float32)
    return np.clip(np.trunc(x / s[:, None]), -127, 127).astype(np.int8), s16


def _divisor_128(bits):
    x = o.bf16_to_f64(bits).astype(np.float32)
    s16 = o.f32_to_f16(np.max(np.abs(x), axis=-1) / np.float32(128.0))
    s16 = np.where(np.max(np.abs(x), axis=-1) > 0, np.where(s16 == 0, 1, s16), 0x3C00).astype(np.uint16)
    s = o.f16_to_f64(s16).astype(np.float32)
    return np.clip(np.rint(x / s[:, None]), -128, 127).astype(np.int8), s16


MUTANTS = {"e4m3_scale_rule": _e4m3_scale_rule, "unrounded_scale": _unrounded_scale,
           "truncation": _truncation, "divisor_128": _divisor_128}


def test_unmutated_quantizer_passes():
    assert _quantizer_ok()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_quantizer_mutants_are_caught(monkeypatch, name):
    monkeypatch.setattr(o, "quantize_index_keys_int8", MUTANTS[name])
    assert not _quantizer_ok()
