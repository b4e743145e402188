"""Pure-Python brute force of the DSA step for tiny inputs.  TEST INFRASTRUCTURE ONLY.

Independent of ``dsa_oracle``: no numpy arithmetic, plain loops over Python
floats (IEEE double), written straight from the definitions, so that the
float64 oracle can be pinned against something other than itself.
"""
from __future__ import annotations

import math
import struct


def bf16(bits: int) -> float:
    """Value of a bf16 bit pattern: it is the upper half of a float32."""
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def e4m3_value(code: int) -> float:
    """Value of an OCP E4M3 code (sign, 4-bit exponent with bias 7, 3-bit mantissa)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (8 + m) * 2.0 ** (e - 10)


def e4m3_encode(x: float) -> int:
    """Nearest finite E4M3 code by exhaustive search; ties go to the even mantissa; clamp at 448."""
    best, best_d = None, None
    for code in range(0x80):
        if code == 0x7F:
            continue
        d = abs(abs(x) - e4m3_value(code))
        if best is None or d < best_d or (d == best_d and (code & 1) == 0 and (best & 1) == 1):
            best, best_d = code, d
    if x < 0 or (x == 0 and math.copysign(1.0, x) < 0):
        best |= 0x80
    return best


def f32(x: float) -> float:
    """Round a double to float32."""
    return struct.unpack("<f", struct.pack("<f", x))[0]


def quantize_key(values_f32: list) -> tuple[list, float]:
    amax = max(abs(v) for v in values_f32)
    scale = f32(amax / 448.0) if amax > 0 else 1.0
    return [e4m3_encode(f32(v / scale)) for v in values_f32], scale


def f16_value(bits: int) -> float:
    """Value of an IEEE binary16 pattern (sign, 5-bit exponent with bias 15, 10-bit mantissa)."""
    bits = int(bits) & 0xFFFF
    sign = -1.0 if bits & 0x8000 else 1.0
    e = (bits >> 10) & 0x1F
    m = bits & 0x3FF
    if e == 0x1F:
        return sign * math.inf if m == 0 else math.nan
    if e == 0:
        return sign * m * 2.0 ** -24
    return sign * (1024 + m) * 2.0 ** (e - 25)


_F16_POSITIVE = None


def f16_nearest(x: float) -> int:
    """Bits of the finite binary16 value nearest to x >= 0, found by searching every positive finite
    pattern; ties go to the even pattern; values beyond the largest finite half give 65504."""
    global _F16_POSITIVE
    if _F16_POSITIVE is None:
        _F16_POSITIVE = [(f16_value(b), b) for b in range(0x7C00)]     # increasing with the bits
    best, best_d = None, None
    for v, b in _F16_POSITIVE:
        d = abs(x - v)
        if best is None or d < best_d or (d == best_d and (b & 1) == 0):
            best, best_d = b, d
        elif v > x:
            break
    return best


def nearest_int8(x: float) -> int:
    """Integer code in [-127, 127] nearest to x by search over all of them; ties go to the even code."""
    best, best_d = None, None
    for c in range(-127, 128):
        d = abs(x - c)
        if best is None or d < best_d or (d == best_d and c % 2 == 0):
            best, best_d = c, d
    return best


def quantize_key_int8(values_f32: list) -> tuple[list, int]:
    """(int8 codes, binary16 scale bits) of one key: scale = half(amax / 127) (1 if amax = 0, the
    smallest positive half if it would round to 0), code = nearest integer to the float32 x / scale."""
    amax = max(abs(v) for v in values_f32)
    if amax == 0:
        sbits = f16_nearest(1.0)
    else:
        sbits = f16_nearest(f32(amax / 127.0)) or 1
    scale = f16_value(sbits)
    return [nearest_int8(f32(v / scale)) for v in values_f32], sbits


def score(q_heads: list, w: list, key: list) -> float:
    """sum over heads of w[h] * ReLU(sum_d q[h][d] * key[d])."""
    total = 0.0
    for h in range(len(q_heads)):
        dot = 0.0
        for d in range(len(key)):
            dot += q_heads[h][d] * key[d]
        total += w[h] * (dot if dot > 0 else 0.0)
    return total


def topk(scores: list, k: int) -> list:
    """Sorted positions of the k best (score desc, position asc), or all positions if <= k."""
    n = len(scores)
    if n <= k:
        return list(range(n))
    ranked = sorted(range(n), key=lambda s: (-scores[s], s))
    return sorted(ranked[:k])


def attention(q_heads: list, rows: list, scale: float, d_latent: int) -> tuple[list, list]:
    """Per head: softmax over rows of scale * (q . row), output sum p * row[:d_latent], and lse."""
    outs, lses = [], []
    for qh in q_heads:
        z = []
        for row in rows:
            acc = 0.0
            for d in range(len(row)):
                acc += qh[d] * row[d]
            z.append(scale * acc)
        m = max(z)
        e = [math.exp(v - m) for v in z]
        l = sum(e)
        out = [0.0] * d_latent
        for j, row in enumerate(rows):
            p = e[j] / l
            for d in range(d_latent):
                out[d] += p * row[d]
        outs.append(out)
        lses.append(m + math.log(l))
    return outs, lses


def page_select(scores: list, page_size: int, budget: int) -> tuple[list, list]:
    """Page-granular selection by loops over the visible scores of one row (index = position).

    A page's score is the largest score among its positions; pages are ranked by (score descending,
    page ascending) and the first `budget` kept (all when fewer).  Returns (kept pages ascending,
    their positions ascending)."""
    n = len(scores)
    pages = []
    for pg in range((n + page_size - 1) // page_size):
        best = None
        for s in range(pg * page_size, min(n, (pg + 1) * page_size)):
            if best is None or scores[s] > best:
                best = scores[s]
        pages.append((best, pg))
    ranked = sorted(pages, key=lambda t: (-t[0], t[1]))
    kept = sorted(pg for _, pg in ranked[:budget])
    positions = [s for pg in kept for s in range(pg * page_size, min(n, (pg + 1) * page_size))]
    return kept, positions


def membership(page_lists: list, union: list) -> list:
    """Row-by-slot membership by loops: [[union[j] in row's pages for j] for row]."""
    out = []
    for pages in page_lists:
        row = []
        for u in union:
            hit = False
            for p in pages:
                if p >= 0 and p == u:
                    hit = True
            row.append(hit)
        out.append(row)
    return out
