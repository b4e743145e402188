// Decode context parallelism: the device steps around the two exchanges.
// ("Serving GLM-5.2-504B on 8x RTX PRO 6000 GPUs", "Reaching 240K context with DCP": the KV is
// sharded along the sequence across the ranks, so each rank's indexer scores only its share of the
// keys.)  A request's tokens are interleaved over the ranks: token s lives on rank s mod N at local
// position s / N.  Each rank runs the indexer and top-k over its own keys; then
//   dcp_candidates_kernel  its local top-k as (score, global position) candidates,
//   (exchange 1: the caller all-gathers the candidates of every rank)
//   dcp_select_kernel      the top-k of the union, larger score first and the smaller position on
//                          ties (every rank computes the same), as global positions and as this
//                          rank's local index buffer (-1 where another rank holds the position),
//   (local sparse MLA over that buffer; exchange 2: the caller all-gathers out and lse)
//   dcp_merge_kernel       the LSE merge of the ranks' partial attention.
// The union of the local top-k lists holds the whole row's top-k, so the result is the
// single-device one.
#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kMaxCand = 16384;                 // world x topk per row that dcp_select handles
constexpr int kPerThread = kMaxCand / kSelThreads;
constexpr int kBitmapWords = kMaxCand / 2;      // the bitmap shares the sort buffer: 262,144 positions

__device__ __forceinline__ uint32_t dcp_order_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);  // -0 becomes +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(256) dcp_candidates_kernel(const float* __restrict__ local_scores, int64_t stride,
                                                             const int32_t* __restrict__ local_idx, int k, int rank,
                                                             int world, float* __restrict__ cand_score,
                                                             int32_t* __restrict__ cand_pos) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x, j = blockIdx.y * blockDim.x + threadIdx.x;   // one entry per thread
  if (j < k) {
    const int li = local_idx[(int64_t)r * k + j];
    cand_score[(int64_t)r * k + j] = li >= 0 ? local_scores[(int64_t)r * stride + li] : -INFINITY;
    cand_pos[(int64_t)r * k + j] = li >= 0 ? li * world + rank : -1;
  }
}

// Exclusive prefix sum over the block of one value per thread (kSelThreads threads); returns the
// prefix and writes the block total to *total.  wsum: kSelThreads / 32 words of shared memory.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* wsum, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const uint32_t w = wsum[lane];
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    wsum[lane] = wi - w;                                 // exclusive prefix of the warp totals
    if (lane == 31) wsum[32] = wi;
  }
  __syncthreads();
  const uint32_t r = wsum[warp] + inc - v;
  *total = wsum[32];
  __syncthreads();                                       // wsum may be reused right after
  return r;
}

// One radix pass of the select over 32-bit values: histogram of the digit (v >> shift) & (2^bits - 1)
// over the values v[i] whose bit i of `live` is set and that match prefix under mask, then the digit
// (from the top) holding the krem-th largest.  Updates prefix / mask / krem and returns the number of
// values in the chosen digit.
template <int KPT>
__device__ __forceinline__ uint32_t radix_pass32(const uint32_t (&v)[KPT], uint32_t live, int shift, int bits,
                                                 uint32_t& prefix, uint32_t& mask, uint32_t& krem, uint32_t* hist,
                                                 uint32_t* wsum, uint32_t* sh) {
  const int tid = threadIdx.x;
  const int nb = 1 << bits;
  for (int i = tid; i < nb; i += kSelThreads) hist[i] = 0;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < KPT; ++i)
    if (((live >> i) & 1u) && (v[i] & mask) == prefix) atomicAdd(&hist[(v[i] >> shift) & (uint32_t)(nb - 1)], 1u);
  __syncthreads();
  // thread t holds digits nb-1-2t and nb-2-2t (descending)
  const int b0 = nb - 1 - 2 * tid, b1 = b0 - 1;
  const uint32_t c0 = b0 >= 0 ? hist[b0] : 0u, c1 = b1 >= 0 ? hist[b1] : 0u;
  uint32_t total;
  const uint32_t ex = block_excl_scan(c0 + c1, wsum, &total);
  if (ex < krem && krem <= ex + c0) {
    sh[0] = (uint32_t)b0;
    sh[1] = krem - ex;
    sh[2] = c0;
  } else if (ex + c0 < krem && krem <= ex + c0 + c1) {
    sh[0] = (uint32_t)b1;
    sh[1] = krem - ex - c0;
    sh[2] = c1;
  }
  __syncthreads();
  prefix |= sh[0] << shift;
  mask |= (uint32_t)(nb - 1) << shift;
  krem = sh[1];
  const uint32_t cnt = sh[2];
  __syncthreads();
  return cnt;
}

// Top-k of one row's candidates [world][rows][k] (score, global position; position -1 = empty).
// A candidate is the pair (order_key(score), ~position), unique, ranking larger score first, then the
// smaller position.  Three radix passes (11/11/10 bits) over the score half find the k-th largest
// score; only when that score is shared by more candidates than still needed do three more passes
// over the position half pick the smaller positions.  The selection is put in ascending order
// through a bitmap over the positions when they are below 262,144 (each thread emits its words' set
// bits at its prefix), else compacted and bitonic-sorted; it is written with this rank's share (local
// positions, compacted) and the share's size.
__global__ void __launch_bounds__(kSelThreads) dcp_select_kernel(const float* __restrict__ cand_score,
                                                                 const int32_t* __restrict__ cand_pos, int world,
                                                                 int rows, int k, int rank,
                                                                 int32_t* __restrict__ global_idx,
                                                                 int32_t* __restrict__ local_idx,
                                                                 int32_t* __restrict__ local_count) {
  __shared__ uint32_t hist[2048];
  __shared__ int32_t spos[kMaxCand / 2];               // bitmap or sort buffer (k <= DSA_MAX_TOPK = 8192)
  __shared__ uint32_t wsum[33];
  __shared__ uint32_t sh[4];
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x, tid = threadIdx.x;
  uint32_t hi[kPerThread], lo[kPerThread];             // order key of the score (0: empty), ~position
  uint32_t nvalid = 0, live = 0;
  {
    // thread t takes candidates t + i kSelThreads, walked as (rank w, entry j) without divisions;
    // every load is issued before any is used
    int32_t pos[kPerThread];
    float sc[kPerThread];
    int w = tid / k, j = tid - w * k;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
      pos[i] = -1;
      sc[i] = 0.f;
      if (w < world) {
        const int64_t at = ((int64_t)w * rows + r) * k + j;
        pos[i] = __ldg(cand_pos + at);
        sc[i] = __ldg(cand_score + at);
      }
      j += kSelThreads;
      while (j >= k && w < world) {
        j -= k;
        ++w;
      }
    }
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
      const bool v = pos[i] >= 0;
      hi[i] = v ? dcp_order_key(sc[i]) : 0u;
      lo[i] = v ? ~(uint32_t)pos[i] : 0u;
      nvalid += v ? 1u : 0u;
      live |= (v ? 1u : 0u) << i;
    }
  }
  uint32_t V;
  block_excl_scan(nvalid, wsum, &V);
  uint32_t t_hi = 1, t_lo = 0;                         // select every valid candidate
  if (V > (uint32_t)k) {
    uint32_t prefix = 0, mask = 0, krem = (uint32_t)k;
    radix_pass32(hi, live, 21, 11, prefix, mask, krem, hist, wsum, sh);
    radix_pass32(hi, live, 10, 11, prefix, mask, krem, hist, wsum, sh);
    const uint32_t tied = radix_pass32(hi, live, 0, 10, prefix, mask, krem, hist, wsum, sh);
    t_hi = prefix;
    if (tied > krem) {                                 // uniform across the block
      uint32_t live_lo = 0;
#pragma unroll
      for (int i = 0; i < kPerThread; ++i) live_lo |= (hi[i] == t_hi ? 1u : 0u) << i;
      uint32_t p2 = 0, m2 = 0;
      radix_pass32(lo, live_lo, 21, 11, p2, m2, krem, hist, wsum, sh);
      radix_pass32(lo, live_lo, 10, 11, p2, m2, krem, hist, wsum, sh);
      radix_pass32(lo, live_lo, 0, 10, p2, m2, krem, hist, wsum, sh);
      t_lo = p2;
    }
  }
  // exactly k candidates (or every valid one) satisfy this
  auto selected = [&](int i) { return hi[i] != 0u && (hi[i] > t_hi || (hi[i] == t_hi && lo[i] >= t_lo)); };
  // the largest selected position decides how the selection is put in order
  uint32_t pmax = 0;
#pragma unroll
  for (int i = 0; i < kPerThread; ++i)
    if (selected(i)) pmax = max(pmax, ~lo[i]);
  if (tid == 0) sh[3] = 0;
  __syncthreads();
  pmax = __reduce_max_sync(0xffffffffu, pmax);
  if ((tid & 31) == 0) atomicMax(&sh[3], pmax);
  __syncthreads();
  const uint32_t max_pos = sh[3];
  __syncthreads();
  uint32_t nlocal;
  int cnt;
  if (max_pos < 32u * kBitmapWords) {
    // a bitmap over the positions: set the selected bits, then each thread emits its 8 words' set
    // bits in order at its prefix (no sort)
    uint32_t* bm = reinterpret_cast<uint32_t*>(spos);
    const int words = (int)(max_pos >> 5) + 1;
    for (int i = tid; i < words; i += kSelThreads) bm[i] = 0;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kPerThread; ++i)
      if (selected(i)) {
        const uint32_t p = ~lo[i];
        atomicOr(&bm[p >> 5], 1u << (p & 31));
      }
    __syncthreads();
    constexpr int WPT = kBitmapWords / kSelThreads;
    // this rank's positions in word wi are the bits b with (32 wi + b) mod world == rank: every
    // world-th bit from s = (rank - 32 wi) mod world
    uint32_t base = 0;
    for (int bit = 0; bit < 32; bit += world) base |= 1u << bit;
    const uint32_t step = 32u % (uint32_t)world;
    uint32_t off = (32u * (uint32_t)(tid * WPT)) % (uint32_t)world;
    uint32_t w[WPT], mine_bits[WPT], c_all = 0, c_mine = 0;
#pragma unroll
    for (int e = 0; e < WPT; ++e) {
      const int wi = tid * WPT + e;
      w[e] = wi < words ? bm[wi] : 0u;
      const uint32_t sft = (uint32_t)rank >= off ? (uint32_t)rank - off : (uint32_t)rank + (uint32_t)world - off;
      mine_bits[e] = base << sft;
      off += step;
      if (off >= (uint32_t)world) off -= (uint32_t)world;
      c_all += __popc(w[e]);
      c_mine += __popc(w[e] & mine_bits[e]);
    }
    uint32_t total;
    uint32_t at_all = block_excl_scan(c_all, wsum, &total);
    uint32_t at_mine = block_excl_scan(c_mine, wsum, &nlocal);
    cnt = min((int)total, k);
#pragma unroll
    for (int e = 0; e < WPT; ++e) {
      const int wi = tid * WPT + e;
      for (uint32_t x = w[e]; x; x &= x - 1) {
        const uint32_t b = (uint32_t)(__ffs(x) - 1), p = (uint32_t)wi * 32u + b;
        if (at_all < (uint32_t)k) global_idx[(int64_t)r * k + at_all] = (int32_t)p;
        ++at_all;
        if ((mine_bits[e] >> b) & 1u) local_idx[(int64_t)r * k + at_mine++] = (int32_t)(p / (uint32_t)world);
      }
    }
  } else {
    // compact the selected positions, then sort them ascending
    if (tid == 0) sh[3] = 0;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kPerThread; ++i)
      if (selected(i)) {
        const uint32_t slot = atomicAdd(&sh[3], 1u);
        if (slot < (uint32_t)k) spos[slot] = (int32_t)~lo[i];   // more only if a position repeats
      }
    __syncthreads();
    cnt = min((int)sh[3], k);
    int n2 = 1;
    while (n2 < cnt) n2 <<= 1;
    for (int i = cnt + tid; i < n2; i += kSelThreads) spos[i] = INT32_MAX;
    __syncthreads();
    for (int size = 2; size <= n2; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < n2; i += kSelThreads) {
          const int partner = i ^ stride;
          if (partner > i) {
            const bool up = (i & size) == 0;
            const int32_t x = spos[i], y = spos[partner];
            if ((x > y) == up) {
              spos[i] = y;
              spos[partner] = x;
            }
          }
        }
        __syncthreads();
      }
    }
    // this rank's share, in order: thread t takes the contiguous entries [t E, t E + E)
    constexpr int E = (kMaxCand / 2) / kSelThreads;
    uint32_t mine = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = tid * E + e;
      mine += (i < cnt && spos[i] % world == rank) ? 1u : 0u;
    }
    uint32_t at = block_excl_scan(mine, wsum, &nlocal);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = tid * E + e;
      if (i < cnt && spos[i] % world == rank) local_idx[(int64_t)r * k + at++] = spos[i] / world;
    }
    for (int i = tid; i < cnt; i += kSelThreads) global_idx[(int64_t)r * k + i] = spos[i];
  }
  for (int i = tid; i < k; i += kSelThreads) {
    if (i >= cnt) global_idx[(int64_t)r * k + i] = -1;
    if (i >= (int)nlocal) local_idx[(int64_t)r * k + i] = -1;
  }
  if (local_count && tid == 0) local_count[r] = (int32_t)nlocal;
}

// LSE merge of the ranks' attention outputs [world][rows][64][512] bf16 and lse [world][rows][64]:
//   out = sum_w e^{lse_w - M} out_w / sum_w e^{lse_w - M},  lse = M + ln sum_w e^{lse_w - M}.
// CTA (row, 8 heads), thread (head, 16 dims).
__global__ void __launch_bounds__(256) dcp_merge_kernel(const __nv_bfloat16* __restrict__ outs,
                                                        const float* __restrict__ lses, int world, int rows,
                                                        __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x, h = blockIdx.y * 8 + (threadIdx.x >> 5), d0 = (threadIdx.x & 31) * 16;
  // every rank's lse and 16 dims are loaded before any is used (world <= 8)
  float lw[8];
  uint4 v[8][2];
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    lw[w] = -INFINITY;
    if (w < world) {
      lw[w] = lses[((int64_t)w * rows + r) * kHeads + h];
      const uint4* src = reinterpret_cast<const uint4*>(outs + (((int64_t)w * rows + r) * kHeads + h) * kLatent + d0);
      v[w][0] = src[0];
      v[w][1] = src[1];
    }
  }
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < 8; ++w) M = fmaxf(M, lw[w]);
  float acc[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0.f;
  float L = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    if (lw[w] == -INFINITY) continue;                  // nothing selected there (or beyond world)
    const float wt = expf(lw[w] - M);
    L += wt;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&v[w][q]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(b2[e]);
        acc[8 * q + 2 * e] = fmaf(wt, f.x, acc[8 * q + 2 * e]);
        acc[8 * q + 2 * e + 1] = fmaf(wt, f.y, acc[8 * q + 2 * e + 1]);
      }
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  uint4 res[2];
  __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(res);
#pragma unroll
  for (int e = 0; e < 8; ++e) o2[e] = __floats2bfloat162_rn(acc[2 * e] * inv, acc[2 * e + 1] * inv);
  uint4* dst = reinterpret_cast<uint4*>(out + ((int64_t)r * kHeads + h) * kLatent + d0);
  dst[0] = res[0];
  dst[1] = res[1];
  if (lse && (threadIdx.x & 31) == 0) lse[(int64_t)r * kHeads + h] = L > 0.f ? M + logf(L) : -INFINITY;
}

}  // namespace

cudaError_t launch_dcp_candidates(const float* local_scores, int64_t stride, const int32_t* local_idx, int k, int rows,
                                  int rank, int world, float* cand_score, int32_t* cand_pos, cudaStream_t s) {
  cudaError_t e = launch_pdl(dcp_candidates_kernel, dim3(rows, (k + 255) / 256), dim3(256), 0, s, local_scores, stride,
                             local_idx, k,
                             rank, world, cand_score, cand_pos);
  count_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_dcp_select(const float* cand_score, const int32_t* cand_pos, int world, int rows, int k, int rank,
                              int32_t* global_idx, int32_t* local_idx, int32_t* local_count, cudaStream_t s) {
  cudaError_t e = launch_pdl(dcp_select_kernel, dim3(rows), dim3(kSelThreads), 0, s, cand_score, cand_pos, world, rows,
                             k, rank, global_idx, local_idx, local_count);
  count_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_dcp_merge(const void* outs, const float* lses, int world, int rows, void* out, float* lse,
                             cudaStream_t s) {
  cudaError_t e = launch_pdl(dcp_merge_kernel, dim3(rows, kHeads / 8), dim3(256), 0, s,
                             static_cast<const __nv_bfloat16*>(outs), lses, world, rows,
                             static_cast<__nv_bfloat16*>(out), lse);
  count_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dsa
