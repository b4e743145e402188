// Top-k selection over one row's indexer scores.
//
// T(r) = the k visible positions with the largest score, ties broken towards
// the smaller position; every visible position when there are at most k
// ("vLLM Inference Path: GLM-5.2 as an Example", "DSA Indexer": Top-2048,
// short contexts keep nearly every position).  Output is sorted ascending and
// padded with -1.
//
// Scores are compared as order-preserving 32-bit keys.  Per row (one CTA of
// 32 warps):
//   1. radix select over a strided sample of 4096 keys (read once into shared
//      memory) gives the key a safety
//      margin below the sample's k-th rank: a threshold that the true k-th
//      key clears with high probability;
//   2. each warp scans its contiguous share of the row (sixteen coalesced loads
//      in flight per lane) and keeps the positions at or above the
//      threshold, in order, in its own shared-memory segment;
//   3. if the segments hold at least k entries and none overflowed they hold
//      the answer: radix select over the candidates finds the k-th key T and
//      how many keys equal to T are taken (the smallest positions first), and
//      the warps emit their kept positions in order through two 32-entry
//      prefix sums.  Otherwise (an unlucky sample) the same radix select runs
//      over the whole row followed by an ordered pass.
// Radix selects use MSB-first digits of 11, 11 and 10 bits and warp-aggregated
// shared-memory histograms.  Both paths give the same unique result.
#include "dsa_internal.cuh"

namespace dsa {

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);   // -0 becomes +0: equal scores compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The float whose order_key is k (k from order_key of a non-NaN float).
__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

constexpr int kTopkThreads = 1024;
constexpr int kWarps = kTopkThreads / 32;
constexpr int kSample = 4096;
constexpr int kSeg = 256;                                   // candidate capacity of one warp
constexpr int kScanUnroll = 16;                            // loads in flight per lane in the candidate scan
constexpr int kSampleBins = 4096;                           // the sample threshold's histogram: top 12 key bits
// (key, position) segments + histogram + the sample's keys
constexpr size_t kTopkSmem = (size_t)kWarps * kSeg * 8 + kSampleBins * 4 + (size_t)kSample * 4;

// Block-wide exclusive scan of a 32-bit value; returns the exclusive prefix and the block total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_tot, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    uint32_t x = warp_tot[lane];
    uint32_t xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, xi, o);
      if (lane >= o) xi += t;
    }
    warp_tot[lane] = xi - x;           // exclusive prefix of each warp
    if (lane == 31) warp_tot[32] = xi;  // block total
  }
  __syncthreads();
  const uint32_t ex = warp_tot[warp] + inc - v;
  total = warp_tot[32];
  __syncthreads();
  return ex;
}

// Histogram increment (shared-memory atomic; the inputs here spread over many bins).
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin, bool active) {
  if (active) atomicAdd(&hist[bin], 1u);
}

// The bin where the count from the top of hist[0..nb) reaches krem (1 <= krem <= total), in three
// short steps: every warp sums its slice of bins (warp 0 owns the highest), warp 0 finds the slice,
// and that slice's warp finds the bin.  Leaves the bin in sh[0] and krem minus the count above it in
// sh[1]; ends with a block barrier.  nb is 1024, 2048 or 4096.
template <int NW>
__device__ void find_bin_from_top(const uint32_t* hist, int nb, uint32_t krem, uint32_t* sh) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int per = nb / NW, per_lane = per / 32;              // bins per warp slice and per lane
  const int top = nb - 1 - warp * per - lane * per_lane;      // this lane's highest bin
  uint32_t mine = 0;
  for (int j = 0; j < per_lane; ++j) mine += hist[top - j];
  uint32_t wsum = mine;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  if (lane == 0) sh[8 + warp] = wsum;
  __syncthreads();
  if (warp == 0) {
    const uint32_t c = lane < NW ? sh[8 + lane] : 0u;
    uint32_t inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    const uint32_t ex = inc - c;
    if (ex < krem && krem <= inc) {
      sh[2] = (uint32_t)lane;
      sh[3] = krem - ex;
    }
  }
  __syncthreads();
  if (warp == (int)sh[2]) {
    const uint32_t kw = sh[3];
    uint32_t inc = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    const uint32_t ex = inc - mine;
    if (ex < kw && kw <= inc) {
      uint32_t c = ex;
      for (int j = 0; j < per_lane; ++j) {
        const uint32_t h = hist[top - j];
        if (c + h >= kw) {
          sh[0] = (uint32_t)(top - j);
          sh[1] = kw - c;
          break;
        }
        c += h;
      }
    }
  }
  __syncthreads();
}

// Radix select: the k-th largest of the keys produced by get(i), i < n (k <= n).  Returns T and
// the number of keys equal to T that belong to the top k.  The whole block calls it.
template <typename Get>
__device__ void radix_select(Get get, int n, uint32_t k, uint32_t* hist, uint32_t* sh, uint32_t& T,
                             uint32_t& need_eq) {
  const int tid = threadIdx.x;
  uint32_t prefix = 0, mask = 0, krem = k;
  const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = shifts[pass], nb = 1 << widths[pass];
    for (int i = tid; i < nb; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += kTopkThreads) {
      const int i = i0 + tid;
      const uint32_t key = i < n ? get(i) : 0u;
      hist_add(hist, (key >> shift) & (nb - 1), i < n && (key & mask) == prefix);
    }
    __syncthreads();
    find_bin_from_top<kWarps>(hist, nb, krem, sh);
    prefix |= sh[0] << shift;
    mask |= (uint32_t)(nb - 1) << shift;
    krem = sh[1];
    __syncthreads();
  }
  T = prefix;
  need_eq = krem;
}

// Sample threshold of one row (scores sc[0..n), n > k): a key at or below the (rank + margin + 1)-th
// largest key of a sample of S = min(n, 4096) scores, rank = k S / n (so the row's true k-th key
// clears it with high probability): the lower edge of the 12-bit bin that holds that sample key.
// A long row is sampled as 512 runs of 8 consecutive scores spread evenly over the row (one 32-byte
// sector each, so the sample costs 16 KB of reads instead of a sector per score).
// 0 when the sample is too small to cut anything.  Every CTA that asks for the same row gets the
// same value.  The whole block calls it (NT threads); ends with a block barrier.
template <int NT>
__device__ uint32_t row_threshold(const float* sc, int n, int k, uint32_t* samp, uint32_t* hist, uint32_t* sh) {
  const int tid = threadIdx.x;
  const int S = n < kSample ? n : kSample;
  const int rank = (int)(((int64_t)k * S) / n);
  const int margin = 3 * (int)sqrtf((float)rank + 1.f) + 8;
  if (rank + margin >= S) return 0u;
  // the sample is read once (all loads in flight together); S is either n (every position) or
  // kSample = 2^12: run i >> 3 starts at the 8-aligned position below (i >> 3) n / 2^9, and since
  // n >= 2^12 the runs are disjoint and end inside the row
#pragma unroll
  for (int j = 0; j < kSample / NT; ++j) {
    const int i = tid + j * NT;
    if (i < S) samp[i] = order_key(sc[S == kSample ? (int)((((int64_t)(i >> 3) * n) >> 9) & ~7ll) + (i & 7) : i]);
  }
  for (int i = tid; i < kSampleBins; i += NT) hist[i] = 0;
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kSample / NT; ++j) {
    const int i = tid + j * NT;
    hist_add(hist, (i < S ? samp[i] : 0u) >> 20, i < S);
  }
  __syncthreads();
  find_bin_from_top<NT / 32>(hist, kSampleBins, (uint32_t)(rank + margin + 1), sh);
  const uint32_t t = sh[0] << 20;
  __syncthreads();
  return t;
}

// Scan positions [w0, w1) of sc and keep, in order, those whose score is at least the threshold
// (compared as floats: the same order as the keys for non-NaN scores) in the warp's segment seg[0..cap):
// (key << 32 | position).  Returns the number kept (more than cap means overflow).  One warp calls it.
__device__ uint32_t scan_share(const float* sc, int w0, int w1, uint32_t t_low, uint64_t* seg, uint32_t cap) {
  const int lane = threadIdx.x & 31;
  float t_low_f = t_low == 0u ? -INFINITY : key_to_float(t_low);   // no threshold: every position
  if (t_low_f != t_low_f) t_low_f = -INFINITY;                        // a key below every finite score
  const float thr = t_low_f;
  uint32_t kept = 0;
  for (int c0 = w0; c0 < w1; c0 += 32 * kScanUnroll) {
    float v[kScanUnroll];
#pragma unroll
    for (int j = 0; j < kScanUnroll; ++j) {
      const int s = c0 + 32 * j + lane;
      v[j] = s < w1 ? sc[s] : -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < kScanUnroll; ++j) {
      const bool take = v[j] >= thr && c0 + 32 * j + lane < w1;
      const uint32_t ballot = __ballot_sync(0xffffffffu, take);
      if (ballot) {
        if (take) {
          const uint32_t slot = kept + __popc(ballot & ((1u << lane) - 1u));
          if (slot < cap) seg[slot] = ((uint64_t)order_key(v[j]) << 32) | (uint32_t)(c0 + 32 * j + lane);
        }
        kept += __popc(ballot);
      }
    }
  }
  return kept;
}

// Rows longer than `chunk` are scanned by one CTA per chunk of positions: each computes the row's
// threshold (the same in every chunk) and writes its candidates, in position order, to its slot of
// cand (at most cap) with their count in cand_cnt (0xFFFFFFFF on overflow).  Shorter rows are left
// to topk_kernel.
constexpr int kChunkThreads = 512;
constexpr int kChunkWarps = kChunkThreads / 32;
constexpr size_t kChunkSmem = (size_t)kChunkWarps * kSeg * 8 + kSampleBins * 4 + (size_t)kSample * 4;
static_assert(kChunkWarps * kSeg == kTopkChunkCap, "a chunk CTA holds exactly one candidate list");

__global__ void __launch_bounds__(kChunkThreads) topk_chunk_kernel(RowMeta m, int row0, const float* __restrict__ scores,
                                                                   int64_t stride, int max_seq_len, int k, int chunk,
                                                                   int chunks, int cap, uint64_t* __restrict__ cand,
                                                                   uint32_t* __restrict__ cand_cnt, int unit_shift) {
  extern __shared__ uint64_t chunk_smem[];
  uint64_t* seg = chunk_smem;                                                       // [16][kSeg]
  uint32_t* hist = reinterpret_cast<uint32_t*>(chunk_smem + kChunkWarps * kSeg);   // [kSampleBins]
  uint32_t* samp = hist + kSampleBins;                                              // [kSample]
  __shared__ uint32_t sh[8 + 32], wcnt[kChunkWarps];
  pdl_wait();
  pdl_trigger();   // the select kernel may start: it waits for this grid before reading its lists
  const int rl = blockIdx.y, r = row0 + rl, c = blockIdx.x;
  int b, pos;
  row_info(m, r, b, pos);
  int n = pos >= 0 ? (pos >> unit_shift) + 1 : 0;          // visible units (positions, or pages)
  if (n > max_seq_len) n = max_seq_len;
  if (n <= chunk) return;                                     // whole row in topk_kernel
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* my_cnt = cand_cnt + (int64_t)rl * chunks + c;
  const int c0 = c * chunk, c1 = min(n, c0 + chunk);
  if (c0 >= n) {
    if (tid == 0) *my_cnt = 0;
    return;
  }
  const float* sc = scores + (int64_t)rl * stride;
  const uint32_t t_low = row_threshold<kChunkThreads>(sc, n, k, samp, hist, sh);
  const int per_warp = (chunk + kChunkWarps - 1) / kChunkWarps;
  const int w0 = min(c1, c0 + warp * per_warp), w1 = min(c1, w0 + per_warp);
  const uint32_t kept = scan_share(sc, w0, w1, t_low, seg + warp * kSeg, kSeg);
  if (lane == 0) wcnt[warp] = kept;
  __syncthreads();
  if (warp == 0) {
    const uint32_t x = lane < kChunkWarps ? wcnt[lane] : 0u;
    const bool bad = __any_sync(0xffffffffu, x > (uint32_t)kSeg);
    uint32_t inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane < kChunkWarps) sh[8 + lane] = inc - x;            // first output index of each warp
    const uint32_t tot = __shfl_sync(0xffffffffu, inc, 31);
    if (lane == 0) sh[0] = (bad || tot > (uint32_t)cap) ? 0xFFFFFFFFu : tot;
  }
  __syncthreads();
  const uint32_t total = sh[0];
  if (total != 0xFFFFFFFFu) {
    uint64_t* dst = cand + ((int64_t)rl * chunks + c) * cap + sh[8 + warp];
    for (uint32_t j = lane; j < kept; j += 32) dst[j] = seg[warp * kSeg + j];
  }
  if (tid == 0) *my_cnt = total;
}

// Units are positions (unit_shift 0) or pages of 2^unit_shift positions, ranked by their page score.
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(RowMeta m, int row0, const float* __restrict__ scores,
                                                            int64_t stride, int max_seq_len, int k,
                                                            int32_t* __restrict__ topk_idx, int chunk, int chunks,
                                                            int cap, const uint64_t* __restrict__ cand,
                                                            const uint32_t* __restrict__ cand_cnt, int unit_shift) {
  extern __shared__ uint64_t topk_smem[];
  uint64_t* seg = topk_smem;                                                  // [kWarps][kSeg] key << 32 | position
  uint32_t* hist = reinterpret_cast<uint32_t*>(topk_smem + kWarps * kSeg);    // [kSampleBins]
  uint32_t* samp = hist + kSampleBins;                                        // [kSample]
  __shared__ uint32_t warp_tot[33];
  __shared__ uint32_t cnt[kWarps], eq_before[kWarps], sel_before[kWarps];
  __shared__ uint32_t sh[8 + kWarps];
  const int r = row0 + blockIdx.x;
  int b, pos;
  row_info(m, r, b, pos);
  int n = pos >= 0 ? (pos >> unit_shift) + 1 : 0;   // visible units (positions, or pages)
  if (n > max_seq_len) n = max_seq_len;   // never read past the row's scores, whatever seq_lens says
  // A programmatic dependent of the chunk kernel (or, when no row is split, of the indexer), this
  // grid may start before that one ends.  Rows the chunk kernel scans wait for its results before
  // reading them.  With a chunk kernel, the other rows read only the scores, which are complete
  // once it has started (it waits for the indexer before it triggers this launch), and wait just
  // before they exit, so that this grid never completes ahead of its predecessor.  Without one,
  // every row waits first.  Every CTA triggers the next launch after its wait.
  const auto wait_chunks = [] {
    pdl_wait();
    pdl_trigger();
  };
  if (chunks == 0) wait_chunks();
  int32_t* out = topk_idx + (int64_t)r * k;
  const float* sc = scores + (int64_t)blockIdx.x * stride;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (n <= k) {
    for (int i = tid; i < k; i += kTopkThreads) out[i] = i < n ? i : -1;
    wait_chunks();
    return;
  }

  uint32_t kept = 0, total = 0;
  if (chunks > 0 && n > chunk) {
    // ---- 1-2 (long rows). The chunk CTAs' candidate lists, concatenated in chunk (= position)
    // order and dealt to the warps in equal contiguous shares.
    const int nch = (n + chunk - 1) / chunk;                 // <= chunks <= 32
    const uint32_t* rc = cand_cnt + (int64_t)blockIdx.x * chunks;
    wait_chunks();
    if (warp == 0) {
      const uint32_t c = lane < nch ? rc[lane] : 0u;
      const bool bad = __any_sync(0xffffffffu, c == 0xFFFFFFFFu);
      uint32_t inc = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
      }
      eq_before[lane] = bad ? 0u : inc - c;                  // first concatenated index of each chunk
      const uint32_t tot = __shfl_sync(0xffffffffu, inc, 31);
      if (lane == 0) sh[2] = (bad || tot > (uint32_t)(kWarps * kSeg)) ? 0u : tot;
    }
    __syncthreads();
    total = sh[2];
    if (total >= (uint32_t)k) {
      const uint32_t per = (total + kWarps - 1) / kWarps;
      const uint32_t i0 = min(total, warp * per), i1 = min(total, i0 + per);
      kept = i1 - i0;
      const uint64_t* rcand = cand + (int64_t)blockIdx.x * chunks * cap;
      // per <= kSeg = 8 x 32: every lane issues its (at most 8) loads before storing any
      uint64_t v[kSeg / 32];
#pragma unroll
      for (int j = 0; j < kSeg / 32; ++j) {
        const uint32_t i = i0 + lane + 32 * j;
        if (i < i1) {
          int c = 0;
          while (c + 1 < nch && eq_before[c + 1] <= i) ++c;
          v[j] = rcand[(int64_t)c * cap + (i - eq_before[c])];
        }
      }
#pragma unroll
      for (int j = 0; j < kSeg / 32; ++j)
        if (i0 + lane + 32 * j < i1) seg[warp * kSeg + lane + 32 * j] = v[j];
      if (lane == 0) cnt[warp] = kept;
    }
    __syncthreads();
  } else {
    // ---- 1. threshold: a key ranked a margin below k * S / n in a strided sample
    const uint32_t t_low = row_threshold<kTopkThreads>(sc, n, k, samp, hist, sh);

    // ---- 2. each warp keeps its share's positions at or above the threshold, in order
    // each warp scans a contiguous share with kScanUnroll coalesced loads in flight per lane; a score
    // is kept when it is at least the threshold, and its key is formed only then
    const int per_warp = (n + kWarps - 1) / kWarps;
    const int w0 = min(n, warp * per_warp), w1 = min(n, w0 + per_warp);
    kept = scan_share(sc, w0, w1, t_low, seg + warp * kSeg, kSeg);
    if (lane == 0) {
      cnt[warp] = kept > (uint32_t)kSeg ? 0xFFFFFFFFu : kept;
      if (warp == 0) sh[2] = 0;
    }
    __syncthreads();
    if (tid < 32) {
      const uint32_t c = cnt[tid];
      const bool bad = __any_sync(0xffffffffu, c == 0xFFFFFFFFu);
      uint32_t tot = bad ? 0 : c;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
      if (tid == 0) sh[2] = bad ? 0u : tot;
    }
    __syncthreads();
    total = sh[2];
  }

  if (total >= (uint32_t)k) {
    // ---- 3a. exact k-th key among the candidates, then an ordered emission
    // candidate i of the concatenated segments: warp w holds indices [sum_{v<w} cnt_v, ...)
    if (tid < 32) {
      uint32_t c = cnt[tid], inc = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
        if (tid >= o) inc += t;
      }
      warp_tot[tid] = inc - c;          // first candidate index of each warp
    }
    __syncthreads();
    uint32_t T, need_eq;
    if (total <= (uint32_t)kSample) {
      // the candidates' keys, packed into the (now free) sample array: one word per candidate per pass
      for (uint32_t j = lane; j < kept; j += 32) samp[warp_tot[warp] + j] = (uint32_t)(seg[warp * kSeg + j] >> 32);
      __syncthreads();
      radix_select([&](int i) { return samp[i]; }, (int)total, (uint32_t)k, hist, sh, T, need_eq);
    } else {
      radix_select(
          [&](int i) {
            int lo = 0, hi = kWarps - 1;   // warp whose segment holds candidate i
            while (lo < hi) {
              const int mid = (lo + hi + 1) >> 1;
              if (warp_tot[mid] <= (uint32_t)i) lo = mid; else hi = mid - 1;
            }
            return (uint32_t)(seg[lo * kSeg + (i - warp_tot[lo])] >> 32);
          },
          (int)total, (uint32_t)k, hist, sh, T, need_eq);
    }
    // per-warp counts of keys > T and == T, then exclusive prefixes in warp (= position) order
    uint32_t gt = 0, eq = 0;
    for (uint32_t j = lane; j < kept; j += 32) {
      const uint32_t key = (uint32_t)(seg[warp * kSeg + j] >> 32);
      gt += key > T;
      eq += key == T;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      gt += __shfl_xor_sync(0xffffffffu, gt, o);
      eq += __shfl_xor_sync(0xffffffffu, eq, o);
    }
    if (lane == 0) {
      cnt[warp] = gt;
      eq_before[warp] = eq;
    }
    __syncthreads();
    if (tid < 32) {
      // selected entries of warp w: all of its keys > T plus its share of the first need_eq keys == T
      uint32_t e = eq_before[tid], einc = e;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, einc, o);
        if (tid >= o) einc += t;
      }
      const uint32_t e_ex = einc - e;
      const uint32_t take_eq = e_ex >= need_eq ? 0u : min(e, need_eq - e_ex);
      uint32_t sel = cnt[tid] + take_eq, sinc = sel;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, sinc, o);
        if (tid >= o) sinc += t;
      }
      sel_before[tid] = sinc - sel;
      eq_before[tid] = e_ex;
    }
    __syncthreads();
    uint32_t out_at = sel_before[warp], eq_seen = eq_before[warp];
    for (uint32_t j0 = 0; j0 < kept; j0 += 32) {
      const uint32_t j = j0 + lane;
      const uint64_t v = j < kept ? seg[warp * kSeg + j] : 0ull;
      const uint32_t key = (uint32_t)(v >> 32);
      const bool is_eq = j < kept && key == T;
      const uint32_t eq_ballot = __ballot_sync(0xffffffffu, is_eq);
      const uint32_t my_eq = eq_seen + __popc(eq_ballot & ((1u << lane) - 1u));
      const bool sel = j < kept && (key > T || (is_eq && my_eq < need_eq));
      const uint32_t sel_ballot = __ballot_sync(0xffffffffu, sel);
      if (sel) {
        const uint32_t o = out_at + __popc(sel_ballot & ((1u << lane) - 1u));
        if (o < (uint32_t)k) out[o] = (int32_t)(uint32_t)v;
      }
      out_at += __popc(sel_ballot);
      eq_seen += __popc(eq_ballot);
    }
    wait_chunks();
    return;
  }

  // ---- 3b. radix select over the whole row, then an ordered pass
  uint32_t T, need_eq;
  radix_select([&](int i) { return order_key(sc[i]); }, n, (uint32_t)k, hist, sh, T, need_eq);
  uint32_t base_gt = 0, base_eq = 0;
  for (int c0 = 0; c0 < n; c0 += 4 * kTopkThreads) {
    const int s0 = c0 + 4 * tid;
    uint32_t key[4];
    uint32_t c = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      key[j] = s0 + j < n ? order_key(sc[s0 + j]) : 0u;
      if (s0 + j < n) c += (key[j] > T ? 1u : 0u) + (key[j] == T ? 0x10000u : 0u);
    }
    uint32_t tot;
    const uint32_t ex = block_exclusive_scan(c, warp_tot, tot);
    uint32_t gt_before = base_gt + (ex & 0xFFFFu), eqb = base_eq + (ex >> 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (s0 + j >= n) break;
      // slots are < k by construction; the guard only keeps inconsistent input inside the row
      if (key[j] > T) {
        const uint32_t slot = gt_before + (eqb < need_eq ? eqb : need_eq);
        if (slot < (uint32_t)k) out[slot] = s0 + j;
        ++gt_before;
      } else if (key[j] == T) {
        if (eqb < need_eq && gt_before + eqb < (uint32_t)k) out[gt_before + eqb] = s0 + j;
        ++eqb;
      }
    }
    base_gt += tot & 0xFFFFu;
    base_eq += tot >> 16;
  }
  wait_chunks();
}

cudaError_t launch_topk(const RowMeta& m, int row0, int nrows, const float* scores, int64_t score_stride,
                        int max_seq_len, int topk, int32_t* topk_idx, const TopkChunks& ch, cudaStream_t s,
                        int unit_shift) {
  static std::atomic<uint64_t> configured{0};
  cudaError_t set = once_per_device(configured, [] {
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTopkSmem);
    return e != cudaSuccess ? e
                            : cudaFuncSetAttribute(topk_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)kChunkSmem);
  });
  if (set != cudaSuccess) return set;
  if (ch.chunks > 0) {
    cudaError_t e = launch_pdl(topk_chunk_kernel, dim3(ch.chunks, nrows), dim3(kChunkThreads), kChunkSmem, s, m, row0,
                               scores, score_stride, max_seq_len, topk, ch.chunk, ch.chunks, (int)kTopkChunkCap,
                               ch.cand, ch.cnt, unit_shift);
    count_launches(1);
    if (e != cudaSuccess) return e;
  }
  // after the chunk kernel the select kernel is a programmatic dependent, so its launch and
  // prologue overlap the chunk kernel's tail
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nrows);
  cfg.blockDim = dim3(kTopkThreads);
  cfg.dynamicSmemBytes = kTopkSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, topk_kernel, m, row0, scores, score_stride, max_seq_len, topk, topk_idx,
                                     ch.chunk, ch.chunks, (int)kTopkChunkCap, (const uint64_t*)ch.cand,
                                     (const uint32_t*)ch.cnt, unit_shift);
  count_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The positions of the selected pages ("Make the sparsity unit match the memory unit": attention
// reads every visible token of a kept page): token_idx[r][j P + t] = page_idx[r][j] P + t when that
// is a visible position, else -1.  Pages are ascending and only a row's last page can be partly
// visible, so the result is ascending with its -1 entries at the end.
__global__ void __launch_bounds__(256) page_expand_kernel(RowMeta m, int row0, const int32_t* __restrict__ page_idx,
                                                          int kp, int page_log2, int32_t* __restrict__ token_idx) {
  pdl_wait();
  pdl_trigger();
  const int r = row0 + blockIdx.x;
  int b, pos;
  row_info(m, r, b, pos);
  const int n = kp << page_log2;
  const int32_t* pr = page_idx + (int64_t)r * kp;
  int32_t* out = token_idx + (int64_t)r * n;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int pg = pr[i >> page_log2];
    const int s = (pg << page_log2) + (i & ((1 << page_log2) - 1));
    out[i] = (pg >= 0 && s <= pos) ? s : -1;
  }
}

cudaError_t launch_page_expand(const RowMeta& m, int row0, int nrows, const int32_t* page_idx, int kp, int page_log2,
                               int32_t* token_idx, cudaStream_t s) {
  cudaError_t e = launch_pdl(page_expand_kernel, dim3(nrows), dim3(256), 0, s, m, row0, page_idx, kp, page_log2,
                             token_idx);
  count_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dsa
