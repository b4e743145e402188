"""Pins of the oracle's number formats: bf16 widening, OCP E4M3 decode/encode, fp8 key quantisation."""
import math
import os

import numpy as np
import pytest

from oracle import brute
from oracle import dsa_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_e4m3():
    rows = []
    with open(os.path.join(GOLDEN, "ocp_e4m3_values.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            code, val = line.split()
            rows.append((int(code, 16), float(val)))
    return rows


def test_e4m3_decode_matches_ocp_table():
    for code, val in _golden_e4m3():
        got = o.e4m3_to_f64(np.array([code], np.uint8))[0]
        if math.isnan(val):
            assert math.isnan(got)
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), (hex(code), got, val)


def test_e4m3_decode_matches_brute_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    got = o.e4m3_to_f64(codes)
    for c in range(256):
        ref = brute.e4m3_value(c)
        assert (math.isnan(ref) and math.isnan(got[c])) or got[c] == ref, hex(c)


def test_e4m3_decode_matches_torch_float8():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = o.e4m3_to_f64(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


def test_e4m3_every_finite_code_reencodes_to_itself():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = o.e4m3_to_f64(codes).astype(np.float32)
    back = o.f32_to_e4m3(vals)
    assert np.array_equal(back, codes)


def _midpoints():
    pos = sorted({brute.e4m3_value(c) for c in range(0x7F)})
    mids = [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])]
    return np.array(mids + [-m for m in mids], dtype=np.float64)


def test_e4m3_encode_matches_brute_on_midpoints_and_random():
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        _midpoints(),                                   # exact ties: must go to the even code
        rng.standard_normal(400) * 40,
        rng.standard_normal(200) * 0.01,                # subnormal range
        np.array([0.0, -0.0, 448.0, 460.0, 464.0, 470.0, 1e4, -1e6, 2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11]),
    ]).astype(np.float32)
    got = o.f32_to_e4m3(vals)
    for v, g in zip(vals.tolist(), got.tolist()):
        assert g == brute.e4m3_encode(v), (v, hex(g), hex(brute.e4m3_encode(v)))


def test_e4m3_ties_round_to_even_mantissa():
    # 1.0625 lies halfway between 1.0 (mantissa 0) and 1.125 (mantissa 1): even wins
    assert o.f32_to_e4m3(np.float32([1.0625]))[0] == 0x38
    # 1.1875 lies halfway between 1.125 (m=1) and 1.25 (m=2): even (m=2) wins
    assert o.f32_to_e4m3(np.float32([1.1875]))[0] == 0x3A
    # saturation instead of NaN above the largest finite value
    assert o.f32_to_e4m3(np.float32([1e9]))[0] == 0x7E
    assert o.f32_to_e4m3(np.float32([-1e9]))[0] == 0xFE


def test_e4m3_encode_matches_torch_cast_in_range():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    vals = np.concatenate([_midpoints(), rng.standard_normal(5000) * 60, rng.standard_normal(2000) * 0.02])
    vals = np.clip(vals, -464, 464).astype(np.float32)        # torch's cast turns (464, 480) into NaN
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(o.f32_to_e4m3(vals), ref)


def test_quantize_index_keys_matches_brute():
    import workloads as wlm
    rng = np.random.default_rng(3)
    x = rng.standard_normal((12, 16)).astype(np.float32) * rng.uniform(0.01, 10, (12, 1)).astype(np.float32)
    x[5] = 0.0                                                  # amax = 0 -> scale 1, all codes 0
    bits = wlm.bf16_bits(x)
    codes, scales = o.quantize_index_keys(bits)
    for t in range(x.shape[0]):
        vals = [brute.bf16(b) for b in bits[t]]
        bc, bs = brute.quantize_key(vals)
        assert scales[t] == np.float32(bs)
        assert codes[t].tolist() == bc
    assert scales[5] == 1.0 and not codes[5].any()


def test_quantised_key_reconstruction_error_bound():
    """Dequantised keys stay within half an e4m3 step of the input (relative 2^-4 of amax-scaled value)."""
    import workloads as wlm
    rng = np.random.default_rng(5)
    bits = wlm.bf16_bits(rng.standard_normal((64, 128)).astype(np.float32))
    codes, scales = o.quantize_index_keys(bits)
    x = o.bf16_to_f64(bits)
    rec = o.e4m3_to_f64(codes) * scales[:, None].astype(np.float64)
    amax = np.abs(x).max(axis=1, keepdims=True)
    # normal range: |err| <= 2^-4 * |x|; subnormal range (|x|/scale < 2^-6): |err| <= 2^-10 * scale
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * amax / 448) * (1 + 1e-6)
    assert np.all(np.abs(rec - x) <= bound)
    assert np.all(np.abs(o.e4m3_to_f64(codes)).max(axis=1) <= 448)


def test_bf16_widening_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(2)
    bits = rng.integers(0, 2 ** 16, 4096, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]                         # drop inf/nan patterns
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(o.bf16_to_f64(bits), ref)
