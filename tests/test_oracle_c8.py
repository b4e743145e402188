"""Pins of the oracle's packed 8-bit latent cache (SFA C8: "GLM-5.2 on vLLM Ascend", "Quantization
and Hardware Branches"; "vLLM Inference Path", "MLA Projections and KV State": an FP8 KV setting
narrows the main MLA cache).

The quantizer is pinned element by element against an exhaustive nearest-code search (brute
force over every E4M3 code, whose values are pinned to the OCP table elsewhere); attention over a
C8 cache against the pure-Python brute force over the dequantised rows; rows that are exactly
representable must reproduce the bf16 result exactly; the round trip obeys E4M3's error bound;
and k_R is stored untouched.
"""
import numpy as np
import pytest

import workloads as wlm
from oracle import brute
from oracle import dsa_oracle as o


def _rows(seed, n, width=512):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, width)).astype(np.float32)
    x[0] = 0.0                                              # amax 0: scale 1, codes 0
    if n > 1:
        x[1] *= np.float32(2.0 ** -12)                      # values deep in e4m3's subnormal range after scaling
        x[1, 7] = 3.0                                       # one large value sets the scale
    if n > 2:
        x[2, :] = np.float32(0.75)                          # constant row: every code is 448
    return wlm.bf16_bits(x)


def test_latent_quantizer_matches_exhaustive_nearest_code():
    bits = _rows(1, 5, width=64)
    codes, scales = o.quantize_latent(bits)
    for t in range(bits.shape[0]):
        vals = [brute.bf16(b) for b in bits[t]]
        want_codes, want_scale = brute.quantize_key(vals)
        assert scales[t] == np.float32(want_scale)
        assert [int(c) for c in codes[t]] == want_codes, f"row {t}"


def test_round_trip_error_is_within_half_an_e4m3_step():
    bits = _rows(2, 64)
    codes, scales = o.quantize_latent(bits)
    x = o.bf16_to_f64(bits)
    deq = o.e4m3_to_f64(codes) * scales.astype(np.float64)[:, None]
    s = scales.astype(np.float64)[:, None]
    # half a step: 2^-4 relative in the normal range, 2^-10 x scale in the subnormal range,
    # plus the float32 division's own rounding
    bound = np.maximum(np.abs(x) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 2.0 ** -20) + np.abs(x) * 2.0 ** -23
    assert np.all(np.abs(deq - x) <= bound)
    assert np.all(np.abs(deq) <= 448.0 * s * (1 + 2.0 ** -20))
    assert scales[0] == 1.0 and np.all(codes[0] == 0)


def test_rope_columns_are_stored_untouched():
    case_bf16 = _case(5, "bf16")
    case_c8 = _case(5, "e4m3")
    lat_b, lat_c = case_bf16.cache.latent, case_c8.cache.latent
    assert np.array_equal(lat_b[..., case_bf16.d_latent:], lat_c[..., case_c8.d_latent:])
    assert np.all(lat_c[..., :case_c8.d_latent] == 0)


def _case(seed, latent_format, d_latent=6, d_rope=3):
    from conftest import TinyCase
    return TinyCase(seed, [13, 9], [2, 1], 4, "bf16", d_latent=d_latent, d_rope=d_rope, latent_format=latent_format)


def test_c8_attention_matches_brute_force():
    case = _case(7, "e4m3")
    idx = np.array([[0, 3, 5, 11, -1, 12], [1, 2, 4, 6, 8, 10], [0, 1, 2, 3, 4, 5]], dtype=np.int32)
    out, lse = o.sparse_mla(case.cache, case.block_table, case.seq_lens, case.qsl, case.q, idx, 0.37)
    for r, (b, pos) in enumerate(case.rows()):
        sel = [int(s) for s in idx[r] if 0 <= s <= pos]
        rows = []
        for s in sel:
            lat = case.latent[b][s]
            codes, scale = brute.quantize_key([brute.bf16(v) for v in lat[:case.d_latent]])
            rows.append([brute.e4m3_value(c) * scale for c in codes] + [brute.bf16(v) for v in lat[case.d_latent:]])
        q = [[brute.bf16(v) for v in case.q[r, h]] for h in range(case.q.shape[1])]
        want_out, want_lse = brute.attention(q, rows, 0.37, case.d_latent)
        assert np.allclose(out[r], np.array(want_out), rtol=1e-12, atol=1e-12)
        assert np.allclose(lse[r], np.array(want_lse), rtol=1e-12, atol=1e-12)


def test_exactly_representable_rows_reproduce_the_bf16_attention():
    """c_KV rows made of e4m3 values times 2^-3 with amax 56 (= 448 / 8): the scale is exactly 1/8,
    every quotient is a code, and the C8 cache's attention equals the bf16 cache's bit for bit."""
    rng = np.random.default_rng(9)
    from oracle.dsa_oracle import PagedCache
    d_latent, d_rope, P, L = 8, 2, 4, 10
    codes = rng.integers(0, 0x7F, size=(L, d_latent)).astype(np.uint8)
    codes[codes == 0x7F] = 0x7E
    codes |= (rng.integers(0, 2, size=(L, d_latent)) << 7).astype(np.uint8)
    vals = o.e4m3_to_f64(codes) / 8.0
    vals[:, 0] = 56.0                                       # amax 448 / 8 in every row
    c_bits = wlm.bf16_bits(vals.astype(np.float32))
    assert np.array_equal(o.bf16_to_f64(c_bits), vals)      # bf16 holds these values exactly
    r_bits = wlm.bf16_bits(rng.standard_normal((L, d_rope)).astype(np.float32))
    bt = np.arange(3, dtype=np.int32)[None, :]
    q = wlm.bf16_bits(rng.standard_normal((1, 3, d_latent + d_rope)).astype(np.float32))
    idx = np.array([[0, 2, 3, 7, 9, -1]], dtype=np.int32)
    res = []
    for fmt in ("bf16", "e4m3"):
        c = PagedCache(3, P, None, d_latent, d_rope, 4, latent_format=fmt)
        c.append(c_bits, r_bits, np.arange(L))
        res.append(o.sparse_mla(c, bt, [L], np.array([0, 1], dtype=np.int32), q, idx, 0.25))
    assert np.array_equal(res[0][0], res[1][0]) and np.array_equal(res[0][1], res[1][1])


def test_unknown_latent_format_is_rejected():
    from oracle.dsa_oracle import PagedCache
    with pytest.raises(ValueError):
        PagedCache(2, 4, None, latent_format="int8")
