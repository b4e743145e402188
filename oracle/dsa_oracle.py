"""Float64 CPU oracle of the GLM-5.2 DSA step.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline``
leg and ``--impl reference``) may import this module.  The product path in
``deepseek_sparse_mla_gb300`` never imports, links or runs it, and this module
shares no code with it.

Every value is widened exactly to float64 from its stored format (bf16, OCP
e4m3, float32) and every step below is the plain definition, in the order the
pages give it, with numpy's matmul / sort as library primitives and no
blocking, fusion or reordering.

Definitions (R query rows, B requests, P page size):

* addressing -- token s of request b lives at slot
  ``block_table[b, s // P] * P + s % P`` ("GLM-5.2 on vLLM Ascend:
  Request-to-Backend Inference Path", section 8 "The SFA backend, step by
  step": the slot mapping scatters new latent KV and indexer keys into their
  physical pages, the kernels receive block tables);
* position of a row -- row i of request b sits at ``L_b - q_len_b + i`` and
  sees positions ``0 .. pos`` inclusive ("Making GLM-5.2 Sparse on TPUs",
  "Pack requests and reuse prefixes": causality uses P + i; the row's own token
  is written before selection, per the SFA backend steps);
* indexer -- ``I(r, s) = sum_h w[r,h] * max(0, q_idx[r,h] . K[s])`` over 32
  heads of width 128 ("vLLM Inference Path: GLM-5.2 as an Example", "DSA
  Indexer" and the Model Shape table; "Making GLM-5.2 Sparse on TPUs",
  "Separate the indexer from the attention it controls": a weighted sum of
  ReLU-transformed query-key dot products);  K[s] is the bf16 key, or the e4m3
  code times the token's float32 scale;
* top-k -- the k highest-scoring visible positions, larger score first and the
  smaller position on ties; every visible position when there are at most k
  ("vLLM Inference Path", "DSA Indexer": Top-2048, contexts shorter than 2,048
  keep nearly every position);  emitted sorted ascending, padded with -1;
* sparse absorbed MLA -- for each head h and selected s:
  ``z = scale * (q_lat[h] . c_KV[s] + q_rope[h] . k_R[s])``, softmax over the
  selection, ``out[h] = sum_s p_s c_KV[s]`` (512-wide latent, before the
  value-up projection) and ``lse[h] = m + ln(sum exp(z - m))``, scale
  1/sqrt(192 + 64) ("Making GLM-5.2 Sparse on TPUs", "Separate the indexer
  ..." : absorbed MLA, scale tied to the original 192 + 64 q/k width; "vLLM
  Inference Path", "MLA Projections and KV State" and "Sparse MLA Attention");
  entries outside ``0 .. pos`` (including -1 padding) are skipped, and a row
  with no valid entry gets out = 0, lse = -inf;
* page-granular selection -- a page's score is the largest I over its visible
  tokens (masks before the maximum), the page budget keeps the best pages
  (ties: smaller page), and attention reads every visible token of a kept page
  ("Making GLM-5.2 Sparse on TPUs", "Make the sparsity unit match the memory
  unit": a page ranked by its highest legal token score; "Stream indexer scores
  over live context": only page scores reach HBM);
* decode context parallelism -- a request's tokens are interleaved over the
  ranks (token s on rank s mod N); each rank selects the top-k of its own
  positions, the candidates are exchanged, the top-k of their union is the
  selection, each rank attends over its share of it and the pieces are
  LSE-merged ("Serving GLM-5.2-504B on 8x RTX PRO 6000 GPUs", "Reaching 240K
  context with DCP": KV sharded along the sequence, each rank's indexer scores
  1/N of the keys; the interleave is the reading taken here);
* IndexShare -- layers marked shared reuse the index buffer of the nearest
  preceding full (owner) layer ("vLLM Inference Path", "DSA Indexer";
  "Serving GLM-5.2-504B on 8x RTX PRO 6000 GPUs", "Root cause: a missing
  index_topk_pattern": full -> F, shared -> S);
* fp8 index-key append -- per token, ``scale = amax / 448`` in float32 (1 if
  amax = 0) and ``code = e4m3_rne_satfinite(x / scale)`` with IEEE float32
  division.  The pages name "FP8 e4m3 keys with FP32 scales" ("GLM-5.2 on
  vLLM Ascend", section 7) without fixing the scale rule: amax/448 is the
  reading taken here.  The e4m3 format is the OCP 8-bit floating point
  specification's E4M3 (bias 7, no infinities, S.1111.111 = NaN, max 448);
* query-blocked union reuse -- a block of QB query rows loads the sorted,
  compacted union of the pages they selected once; each row keeps its own
  support through a membership mask indexed by union slot, before the online
  softmax, and causality and valid lengths still apply; the union is never
  truncated (its capacity is min(QB x Kp, units)), so the operation equals each
  row's attention over its own pages ("Making GLM-5.2 Sparse on TPUs", "Reuse
  pages across queries"); the page-load reduction is QB x Kp / U and the score
  work grows by U / Kp;
* packed 8-bit latent cache (SFA C8) -- the 512 c_KV values of a token are
  stored as e4m3 codes with one float32 scale per token, by the same rule as
  the fp8 index keys (``scale = amax / 448``, 1 if amax = 0, ``code =
  e4m3(x / scale)``); k_R stays bf16; attention runs over ``code * scale``
  exactly ("GLM-5.2 on vLLM Ascend", "Quantization and Hardware Branches": SFA
  C8 packs the main latent KV and uses the quantized sparse-attention operator,
  while the non-RoPE / RoPE split is preserved; "vLLM Inference Path", "MLA
  Projections and KV State": an explicit FP8 KV setting narrows the main MLA
  cache).  The per-token amax / 448 rule and bf16 k_R are the readings taken;
* int8 index-key append -- per token, ``scale = fp16(amax / 127)`` (the float32
  quotient rounded to IEEE binary16, nearest-even, held at the largest finite
  half 65504 above it and at the smallest positive half 2^-24 below it; 1 if
  amax = 0) and ``code = clamp(rne(x / scale), -127, 127)`` with the IEEE
  float32 quotient by the stored scale; the key is ``code * scale``.  The pages
  give "INT8 keys with FP16 scales" as the indexer cache of one hardware
  family beside e4m3 keys with float32 scales ("GLM-5.2 on vLLM Ascend",
  section 7 and "Quantization and Hardware Branches") without the rule: the
  symmetric amax / 127 scale, held to its half-precision value before the
  division so that ``code * scale`` reproduces the key, is the reading taken.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
INT8_MAX = 127
F16_MAX = 65504.0            # largest finite IEEE binary16 value
F16_MIN_SUBNORMAL = 2.0 ** -24


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------
def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact: bf16 is the top half of a float32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def e4m3_to_f64(codes) -> np.ndarray:
    """OCP E4M3 codes -> float64.

    Field layout s.eeee.mmm, exponent bias 7.  Exponent field 0 is subnormal:
    (m/8) * 2^-6.  Otherwise (1 + m/8) * 2^(e-7).  S.1111.111 is NaN; there
    are no infinities, so S.1111.110 = 448 is the largest finite value.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c & 0x80) != 0, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    out = sign * mag
    return np.where((c & 0x7F) == 0x7F, np.nan, out)


def f32_to_e4m3(x) -> np.ndarray:
    """float32 -> OCP E4M3 code, round to nearest (ties to even), saturating to +-448.

    For |x| in [2^e, 2^(e+1)) with e >= -6 the representable spacing is 2^(e-3);
    below 2^-6 (the subnormal range) it is 2^-9.  Dividing by the spacing is
    exact in float64, np.rint rounds half to even, and a magnitude that rounds
    up into the next binade is still representable.
    """
    v = np.asarray(x, dtype=np.float32).astype(np.float64)
    neg = np.signbit(v)
    a = np.abs(v)
    _, ex = np.frexp(a)                       # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)                # floor(log2 a), clamped to the subnormal binade
    step = np.ldexp(1.0, e - 3)
    q = np.minimum(np.rint(a / step) * step, E4M3_MAX)
    # encode the (exactly representable) magnitude q
    _, qex = np.frexp(np.where(q > 0, q, 1.0))
    qe = qex - 1
    normal = q >= 2.0 ** -6
    exp_field = np.where(normal, qe + 7, 0)
    mant = np.where(normal, q / np.ldexp(1.0, qe) - 1.0, q / 2.0 ** -9) * np.where(normal, 8.0, 1.0)
    code = (exp_field.astype(np.int64) << 3) | np.rint(mant).astype(np.int64)
    code = np.where(q == 0, 0, code)
    code = code | np.where(neg, 0x80, 0)
    return code.astype(np.uint8)


def quantize_latent(c_kv_bits) -> tuple[np.ndarray, np.ndarray]:
    """bf16 c_KV rows [T, 512] -> (e4m3 codes [T, 512], float32 scales [T]): the packed 8-bit latent
    cache, one scale per token by the same amax / 448 rule as the fp8 index keys."""
    return quantize_index_keys(c_kv_bits)


def quantize_index_keys(bits) -> tuple[np.ndarray, np.ndarray]:
    """bf16 index keys [T, 128] -> (e4m3 codes [T, 128], float32 scales [T]).

    scale = amax / 448 in float32 (1 when amax = 0); code = e4m3(x / scale) with
    the division done in IEEE float32, as the append step does.
    """
    x = bf16_to_f64(bits).astype(np.float32)          # exact: bf16 values are float32 values
    amax = np.max(np.abs(x), axis=-1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    codes = f32_to_e4m3((x / scale[..., None]).astype(np.float32))
    return codes, scale


def f16_to_f64(bits) -> np.ndarray:
    """IEEE binary16 bit patterns -> float64 (exact).

    Field layout s.eeeee.mmmmmmmmmm, exponent bias 15.  Exponent field 0 is
    subnormal: (m/1024) * 2^-14.  Otherwise (1 + m/1024) * 2^(e-15); field 31
    is infinity (m = 0) or NaN.
    """
    c = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where((c & 0x8000) != 0, -1.0, 1.0)
    e = (c >> 10) & 0x1F
    m = (c & 0x3FF).astype(np.float64)
    mag = np.where(e == 0, (m / 1024.0) * 2.0 ** -14, (1.0 + m / 1024.0) * np.exp2(e.astype(np.float64) - 15.0))
    mag = np.where(e == 0x1F, np.where(m == 0, np.inf, np.nan), mag)
    return sign * mag


def f32_to_f16(x) -> np.ndarray:
    """float32 -> IEEE binary16 bits, round to nearest (ties to even), held at +-65504.

    For |x| in [2^e, 2^(e+1)) with e >= -14 the spacing of binary16 is 2^(e-10);
    below 2^-14 (the subnormal range) it is 2^-24.  Same construction as the
    e4m3 encoder: divide by the spacing (exact in float64), np.rint, rebuild.
    """
    v = np.asarray(x, dtype=np.float32).astype(np.float64)
    neg = np.signbit(v)
    a = np.abs(v)
    _, ex = np.frexp(a)
    e = np.maximum(ex - 1, -14)
    step = np.ldexp(1.0, e - 10)
    q = np.minimum(np.rint(a / step) * step, F16_MAX)
    _, qex = np.frexp(np.where(q > 0, q, 1.0))
    qe = qex - 1
    normal = q >= 2.0 ** -14
    exp_field = np.where(normal, qe + 15, 0)
    mant = np.where(normal, (q / np.ldexp(1.0, qe) - 1.0) * 1024.0, q / F16_MIN_SUBNORMAL)
    code = (exp_field.astype(np.int64) << 10) | np.rint(mant).astype(np.int64)
    code = np.where(q == 0, 0, code) | np.where(neg, 0x8000, 0)
    return code.astype(np.uint16)


def quantize_index_keys_int8(bits) -> tuple[np.ndarray, np.ndarray]:
    """bf16 index keys [T, 128] -> (int8 codes [T, 128], binary16 scale bits [T]).

    scale = fp16(amax / 127): the float32 quotient rounded to binary16 (nearest,
    ties to even), at most 65504 and at least 2^-24; 1 when amax = 0.  code =
    rne(x / scale) with the float32 quotient by that stored scale, clamped to
    [-127, 127] (the rounded scale can sit a hair below amax / 127).
    """
    x = bf16_to_f64(bits).astype(np.float32)
    amax = np.max(np.abs(x), axis=-1)
    s16 = f32_to_f16((amax / np.float32(INT8_MAX)).astype(np.float32))
    s16 = np.where(s16 == 0, np.uint16(1), s16)                 # below 2^-25: the smallest positive half
    s16 = np.where(amax > 0, s16, f32_to_f16(np.float32(1.0))).astype(np.uint16)
    scale = f16_to_f64(s16).astype(np.float32)                  # exact: every half is a float32
    quot = (x / scale[..., None]).astype(np.float32)
    codes = np.clip(np.rint(quot.astype(np.float64)), -INT8_MAX, INT8_MAX).astype(np.int8)
    return codes, s16


# ---------------------------------------------------------------------------
# the paged caches
# ---------------------------------------------------------------------------
class PagedCache:
    """One layer's caches: latent pages [N_pg, P, 576] bf16 and, for an
    indexer-owning layer, index-key pages [N_pg, P, 128] (bf16, e4m3 codes
    with float32 scales [N_pg, P], or int8 codes with binary16 scale bits
    [N_pg, P]).  Unwritten slots hold 0."""

    def __init__(self, num_pages: int, page_size: int, key_format: str | None, d_latent=512, d_rope=64, d_index=128,
                 latent_format: str = "bf16"):
        self.num_pages, self.page_size, self.key_format = num_pages, page_size, key_format
        self.d_latent, self.d_rope, self.d_index = d_latent, d_rope, d_index
        self.latent_format = latent_format
        self.latent = np.zeros((num_pages, page_size, d_latent + d_rope), dtype=np.uint16)
        self.latent_codes = self.latent_scales = None
        if latent_format == "e4m3":
            # packed 8-bit latent: c_KV as e4m3 codes + a float32 scale per token; k_R stays in
            # the bf16 array's last 64 columns (its c_KV columns stay 0)
            self.latent_codes = np.zeros((num_pages, page_size, d_latent), dtype=np.uint8)
            self.latent_scales = np.zeros((num_pages, page_size), dtype=np.float32)
        elif latent_format != "bf16":
            raise ValueError(latent_format)
        self.index_keys = None
        self.index_scales = None
        if key_format == "bf16":
            self.index_keys = np.zeros((num_pages, page_size, d_index), dtype=np.uint16)
        elif key_format == "fp8":
            self.index_keys = np.zeros((num_pages, page_size, d_index), dtype=np.uint8)
            self.index_scales = np.zeros((num_pages, page_size), dtype=np.float32)
        elif key_format == "int8":
            self.index_keys = np.zeros((num_pages, page_size, d_index), dtype=np.int8)
            self.index_scales = np.zeros((num_pages, page_size), dtype=np.uint16)
        elif key_format is not None:
            raise ValueError(key_format)

    def append(self, c_kv_bits, k_rope_bits, slot_mapping, k_idx_bits=None, k_idx_codes=None, k_idx_scales=None):
        """Write new tokens at their slots (page = slot // P, offset = slot % P).

        The latent row is the bit-exact concatenation [c_KV | k_R].  Index keys
        are stored as given (bf16), quantised here (bf16 given, fp8 or int8 cache), or
        stored as given codes + scales (pre-quantised input)."""
        slot = np.asarray(slot_mapping, dtype=np.int64)
        pg, off = slot // self.page_size, slot % self.page_size
        if self.latent_format == "e4m3":
            codes, scales = quantize_latent(c_kv_bits)
            self.latent_codes[pg, off] = codes
            self.latent_scales[pg, off] = scales
        else:
            self.latent[pg, off, :self.d_latent] = c_kv_bits
        self.latent[pg, off, self.d_latent:] = k_rope_bits
        if self.key_format is None:
            return
        if self.key_format == "bf16":
            self.index_keys[pg, off] = k_idx_bits
        elif k_idx_codes is not None:
            self.index_keys[pg, off] = k_idx_codes
            self.index_scales[pg, off] = k_idx_scales
        else:
            quantize = quantize_index_keys_int8 if self.key_format == "int8" else quantize_index_keys
            codes, scales = quantize(k_idx_bits)
            self.index_keys[pg, off] = codes
            self.index_scales[pg, off] = scales

    def slots(self, block_row, positions) -> tuple[np.ndarray, np.ndarray]:
        positions = np.asarray(positions, dtype=np.int64)
        pages = np.asarray(block_row, dtype=np.int64)[positions // self.page_size]
        return pages, positions % self.page_size

    def latent_rows(self, block_row, positions) -> np.ndarray:
        """[n, 576] float64 cached rows [c_KV | k_R] at logical positions of one request (an e4m3
        c_KV is its code times the token's scale)."""
        pg, off = self.slots(block_row, positions)
        rows = bf16_to_f64(self.latent[pg, off])
        if self.latent_format == "e4m3":
            rows[:, :self.d_latent] = (e4m3_to_f64(self.latent_codes[pg, off]) *
                                       self.latent_scales[pg, off].astype(np.float64)[:, None])
        return rows

    def index_key_rows(self, block_row, positions) -> np.ndarray:
        """[n, 128] float64 index keys: the bf16 value, or the e4m3 / int8 code times the token's scale."""
        pg, off = self.slots(block_row, positions)
        if self.key_format == "bf16":
            return bf16_to_f64(self.index_keys[pg, off])
        if self.key_format == "int8":
            return self.index_keys[pg, off].astype(np.float64) * f16_to_f64(self.index_scales[pg, off])[:, None]
        return e4m3_to_f64(self.index_keys[pg, off]) * self.index_scales[pg, off].astype(np.float64)[:, None]


# ---------------------------------------------------------------------------
# batch metadata
# ---------------------------------------------------------------------------
def row_positions(seq_lens, query_start_loc) -> tuple[np.ndarray, np.ndarray]:
    """(request of each row, absolute position of each row = L_b - q_len_b + i)."""
    req, pos = [], []
    for b in range(len(seq_lens)):
        q_len = int(query_start_loc[b + 1]) - int(query_start_loc[b])
        for i in range(q_len):
            req.append(b)
            pos.append(int(seq_lens[b]) - q_len + i)
    return np.asarray(req, dtype=np.int64), np.asarray(pos, dtype=np.int64)


# ---------------------------------------------------------------------------
# the lightning indexer and top-k selection
# ---------------------------------------------------------------------------
def index_scores(q_idx_row, w_row, keys) -> np.ndarray:
    """I[s] = sum_h w[h] * max(0, q_idx[h] . K[s]) for the given keys [n, d].

    q_idx_row [H_I, d] and w_row [H_I] float64."""
    dots = keys @ np.asarray(q_idx_row, dtype=np.float64).T          # [n, H_I]
    return np.maximum(dots, 0.0) @ np.asarray(w_row, dtype=np.float64)


def topk_select(scores, k: int) -> np.ndarray:
    """k positions with the largest score (ties: smaller position first), or all
    positions when len(scores) <= k; sorted ascending, padded with -1 to k."""
    scores = np.asarray(scores, dtype=np.float64)
    n = scores.shape[0]
    if n <= k:
        chosen = np.arange(n)
    else:
        order = np.lexsort((np.arange(n), -scores))   # primary: score descending, then position ascending
        chosen = np.sort(order[:k])
    out = np.full(k, -1, dtype=np.int32)
    out[:chosen.shape[0]] = chosen
    return out


def indexer_topk(cache: PagedCache, block_table, seq_lens, query_start_loc, q_idx_bits, w, topk: int,
                 rows=None):
    """Scores and top-k for every query row (or the listed rows).

    Returns (idx [n_rows, topk] int32, scores: list of float64 arrays over 0..pos)."""
    if cache.index_keys is None:
        raise ValueError("layer holds no index keys: a shared layer must reuse an owner's index buffer")
    req, pos = row_positions(seq_lens, query_start_loc)
    rows = range(len(req)) if rows is None else rows
    q = bf16_to_f64(q_idx_bits)
    w = np.asarray(w, dtype=np.float64)
    idx, all_scores = [], []
    key_cache = {}
    for r in rows:
        b, p = int(req[r]), int(pos[r])
        if b not in key_cache:
            key_cache = {b: cache.index_key_rows(block_table[b], np.arange(int(seq_lens[b])))}
        keys = key_cache[b][:p + 1]                        # visible positions 0..pos only
        s = index_scores(q[r], w[r], keys)
        all_scores.append(s)
        idx.append(topk_select(s, topk))
    return np.stack(idx), all_scores


# ---------------------------------------------------------------------------
# page-granular selection ("Making GLM-5.2 Sparse on TPUs", "Make the sparsity unit match the
# memory unit" and "Stream indexer scores over live context")
# ---------------------------------------------------------------------------
def page_scores(scores, page_size: int) -> np.ndarray:
    """Score of each logical page of a row: the largest I over the page's visible tokens.

    `scores` holds I over the visible positions 0..pos only, so the causal / valid-length mask is
    applied before the maximum (an invisible token cannot promote its page).  Returns one value per
    page 0 .. pos // P (the pages holding at least one visible token)."""
    scores = np.asarray(scores, dtype=np.float64)
    n_pages = -(-scores.shape[0] // page_size)
    out = np.empty(n_pages, dtype=np.float64)
    for pg in range(n_pages):
        out[pg] = scores[pg * page_size:(pg + 1) * page_size].max()
    return out


def page_topk_select(pscores, page_budget: int) -> np.ndarray:
    """The page_budget pages with the largest page score (ties: smaller page first), or every page
    when there are at most page_budget; sorted ascending, padded with -1 (the token rule of
    topk_select, applied to pages)."""
    return topk_select(pscores, page_budget)


def pages_to_positions(pages, page_size: int, pos: int) -> np.ndarray:
    """The visible positions (<= pos) of the selected pages, ascending, padded with -1 to
    len(pages) * page_size: attention reads every visible token of a selected page."""
    out = np.full(len(pages) * page_size, -1, dtype=np.int32)
    at = 0
    for pg in sorted(int(x) for x in pages if x >= 0):
        for s in range(pg * page_size, (pg + 1) * page_size):
            if s <= pos:
                out[at] = s
                at += 1
    return out


def page_indexer_topk(cache: PagedCache, block_table, seq_lens, query_start_loc, q_idx_bits, w,
                      page_budget: int, rows=None):
    """Page-granular selection for every (or the listed) query row: token scores, page scores
    (maximum over visible tokens), the page_budget best pages and their visible positions.

    Returns (pages [n_rows, page_budget] int32, positions [n_rows, page_budget * P] int32,
    page scores: list of float64 arrays, token scores: list of float64 arrays)."""
    P = cache.page_size
    idx, t_scores = indexer_topk(cache, block_table, seq_lens, query_start_loc, q_idx_bits, w, 1, rows)
    _, pos = row_positions(seq_lens, query_start_loc)
    rows = range(len(pos)) if rows is None else rows
    pages, positions, p_scores = [], [], []
    for r, s in zip(rows, t_scores):
        ps = page_scores(s, P)
        sel = page_topk_select(ps, page_budget)
        p_scores.append(ps)
        pages.append(sel)
        positions.append(pages_to_positions(sel, P, int(pos[r])))
    return np.stack(pages), np.stack(positions), p_scores, t_scores


# ---------------------------------------------------------------------------
# decode context parallelism ("Serving GLM-5.2-504B on 8x RTX PRO 6000 GPUs", "Reaching 240K
# context with DCP": the KV is sharded along the sequence across the ranks, so each rank's indexer
# scores only its share of the keys)
# ---------------------------------------------------------------------------
def dcp_local_positions(L: int, rank: int, world: int) -> np.ndarray:
    """Global positions of a request's first L tokens held by `rank`: s = rank, rank + world, ...
    (interleaved by token; local position s // world)."""
    return np.arange(rank, L, world, dtype=np.int64)


def dcp_select(scores, k: int, world: int):
    """The DCP selection of one decode row from its token scores over 0..pos, step by step:
    each rank keeps the top-k of its own positions (local order = global order restricted to the
    rank), the ranks exchange their (score, position) candidates, and every rank takes the top-k of
    the union (larger score first, smaller position on ties).  Returns (global selection ascending,
    -1 padded, as topk_select; per-rank candidate lists)."""
    scores = np.asarray(scores, dtype=np.float64)
    cand = []
    for rank in range(world):
        pos = dcp_local_positions(len(scores), rank, world)
        local = topk_select(scores[pos], k)
        cand.append([(scores[pos[i]], int(pos[i])) for i in local if i >= 0])
    union = [c for lst in cand for c in lst]
    union.sort(key=lambda c: (-c[0], c[1]))
    chosen = sorted(p for _, p in union[:k])
    out = np.full(k, -1, dtype=np.int32)
    out[:len(chosen)] = chosen
    return out, cand


def dcp_attend(q_row, rows_of, selection, world: int, scale: float, d_latent: int = 512):
    """Attention of one decode row over a selection whose positions are split between the ranks
    that hold them: each rank attends over its own positions, and the partial results are combined
    by the LSE merge.  rows_of(positions) returns the cached rows of global positions."""
    sel = np.asarray([s for s in selection if s >= 0], dtype=np.int64)
    parts = []
    for rank in range(world):
        mine = sel[sel % world == rank]
        parts.append(attend(q_row, rows_of(mine), scale, d_latent))
    return lse_merge(parts)


# ---------------------------------------------------------------------------
# sparse absorbed MLA
# ---------------------------------------------------------------------------
def attend(q_row, rows, scale: float, d_latent: int = 512) -> tuple[np.ndarray, np.ndarray]:
    """Softmax attention of every head of one query row over the given cached rows.

    q_row [H, d_latent + d_rope] = [q_latent | q_rope] per head, rows [m, d_latent + d_rope]
    = [c_KV | k_R].  Returns (out [H, d_latent] = sum_s p_s c_KV[s], lse [H])."""
    q_row = np.asarray(q_row, dtype=np.float64)
    n_heads = q_row.shape[0]
    if rows.shape[0] == 0:
        return np.zeros((n_heads, d_latent)), np.full(n_heads, -np.inf)
    c_kv, k_r = rows[:, :d_latent], rows[:, d_latent:]
    q_lat, q_rope = q_row[:, :d_latent], q_row[:, d_latent:]
    z = scale * (q_lat @ c_kv.T + q_rope @ k_r.T)           # [H, m]
    m = z.max(axis=1, keepdims=True)
    p = np.exp(z - m)
    l = p.sum(axis=1, keepdims=True)
    out = (p / l) @ c_kv
    return out, (m + np.log(l))[:, 0]


def valid_selection(idx_row, pos: int) -> np.ndarray:
    """Entries of an index-buffer row that name a visible position (0 <= s <= pos)."""
    idx_row = np.asarray(idx_row, dtype=np.int64)
    return idx_row[(idx_row >= 0) & (idx_row <= pos)]


def sparse_mla(cache: PagedCache, block_table, seq_lens, query_start_loc, q_bits, topk_idx, scale: float,
               rows=None):
    """Absorbed sparse MLA of every (or the listed) query row over its selected positions.

    Returns (out [n_rows, H, 512] float64, lse [n_rows, H] float64)."""
    req, pos = row_positions(seq_lens, query_start_loc)
    rows = range(len(req)) if rows is None else rows
    outs, lses = [], []
    for r in rows:
        b, p = int(req[r]), int(pos[r])
        sel = valid_selection(topk_idx[r], p)
        cached = cache.latent_rows(block_table[b], sel)
        o, l = attend(bf16_to_f64(q_bits[r]), cached, scale, cache.d_latent)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def lse_merge(parts) -> tuple[np.ndarray, np.ndarray]:
    """Combine attention results over disjoint pieces of one selection.

    parts: list of (out [H, d], lse [H]) where out is the softmax-weighted mean
    of its piece.  The whole is sum_j exp(lse_j - lse) out_j with
    lse = ln sum_j exp(lse_j)."""
    lse = np.stack([p[1] for p in parts])                    # [J, H]
    mx = np.max(lse, axis=0)
    safe = np.where(np.isfinite(mx), mx, 0.0)
    wts = np.exp(lse - safe)                                 # [J, H]
    tot = wts.sum(axis=0)
    out = sum(wts[j][:, None] * parts[j][0] for j in range(len(parts)))
    with np.errstate(divide="ignore", invalid="ignore"):
        out = np.where(tot[:, None] > 0, out / tot[:, None], 0.0)
        merged = np.where(tot > 0, safe + np.log(tot), -np.inf)
    return out, merged


# ---------------------------------------------------------------------------
# query-blocked union reuse
# ---------------------------------------------------------------------------
def page_union(page_lists) -> np.ndarray:
    """The sorted, compacted union of a query block's selected pages (page ids, -1 padding ignored)."""
    pages = np.concatenate([np.asarray(p, dtype=np.int64).ravel() for p in page_lists])
    return np.unique(pages[pages >= 0])


def union_membership(page_lists, union) -> np.ndarray:
    """[QB, U] bool: row q selected the page in union slot j (indexed by slot, not by page id)."""
    union = np.asarray(union, dtype=np.int64)
    return np.stack([np.isin(union, np.asarray(p, dtype=np.int64)) for p in page_lists])


def union_capacity(qb: int, kp: int, units: int) -> int:
    """Lossless capacity of the union buffer: min(QB x Kp, number of units)."""
    return min(qb * kp, units)


def page_load_reduction(qb: int, kp: int, u: int) -> float:
    return qb * kp / u


def score_work_expansion(u: int, kp: int) -> float:
    return u / kp


def blocked_attend(q_rows, union_rows, union_pos, member_tokens, row_pos, scale: float, d_latent: int = 512):
    """Attention of a block of query rows over the tokens of their page union, loaded once.

    q_rows [QB, H, D]; union_rows [n, D] the cached rows of every token of the union's pages, at
    logical positions union_pos [n]; member_tokens [QB, n] each row's membership (its own pages);
    row_pos [QB] each row's position.  A token takes part in row q's softmax only if it is a member
    and visible (position <= row_pos[q]).  Returns (out [QB, H, d_latent], lse [QB, H])."""
    outs, lses = [], []
    union_pos = np.asarray(union_pos)
    for q in range(len(q_rows)):
        keep = np.asarray(member_tokens[q], dtype=bool) & (union_pos <= row_pos[q])
        o, l = attend(q_rows[q], np.asarray(union_rows)[keep], scale, d_latent)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


# ---------------------------------------------------------------------------
# IndexShare layer schedule
# ---------------------------------------------------------------------------
def indexshare_pattern(indexer_types) -> str:
    """Per-layer F/S string from a checkpoint's indexer_types: full -> F, shared -> S."""
    table = {"full": "F", "shared": "S"}
    return "".join(table[t] for t in indexer_types)


def owner_of_layer(pattern: str) -> list[int]:
    """For each layer, the index of the nearest full layer at or before it."""
    owners, last = [], None
    for i, c in enumerate(pattern):
        if c == "F":
            last = i
        if last is None:
            raise ValueError("layer %d is shared but no full layer precedes it" % i)
        owners.append(last)
    return owners
