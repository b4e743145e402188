// Top-k selection over one row's indexer scores.
//
// T(r) = the k visible positions with the largest score, ties broken towards
// the smaller position; every visible position when there are at most k
// ("vLLM Inference Path: GLM-5.2 as an Example", "DSA Indexer": Top-2048,
// short contexts keep nearly every position).  Output is sorted ascending and
// padded with -1.
//
// Radix select on order-preserving 32-bit keys (MSB-first digits of 11, 11 and
// 10 bits, shared-memory histograms) finds the k-th largest key T; a final
// ordered pass writes every position with key > T and the first (in position
// order) of those with key == T until k are taken.  The result is unique and
// deterministic.
#include "dsa_internal.cuh"

namespace dsa {

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);   // -0 becomes +0: equal scores compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kTopkThreads = 1024;

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

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(RowMeta m, int row0, const float* __restrict__ scores,
                                                            int64_t stride, int max_seq_len, int k,
                                                            int32_t* __restrict__ topk_idx) {
  __shared__ uint32_t hist[2048];
  __shared__ uint32_t warp_tot[33];
  __shared__ uint32_t sh_bin, sh_krem;
  const int r = row0 + blockIdx.x;
  int b, pos;
  row_info(m, r, b, pos);
  int n = pos + 1 > 0 ? pos + 1 : 0;
  if (n > max_seq_len) n = max_seq_len;   // never read past the row's scores, whatever seq_lens says
  int32_t* out = topk_idx + (int64_t)r * k;
  const float* sc = scores + (int64_t)blockIdx.x * stride;
  const int tid = threadIdx.x;
  if (n <= k) {
    for (int i = tid; i < k; i += kTopkThreads) out[i] = i < n ? i : -1;
    return;
  }

  uint32_t prefix = 0, mask = 0;
  uint32_t krem = (uint32_t)k;
  const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = shifts[pass], nb = 1 << widths[pass];
    for (int i = tid; i < nb; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int s = tid; s < n; s += kTopkThreads) {
      const uint32_t key = order_key(sc[s]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & (nb - 1)], 1u);
    }
    __syncthreads();
    if (tid < 32) {
      // lane 0 owns the highest bins; find the bin where the count from the top reaches krem
      const int per = nb / 32;
      const int top = nb - 1 - tid * per;
      uint32_t sum = 0;
      for (int j = 0; j < per; ++j) sum += hist[top - j];
      uint32_t inc = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
        if (tid >= o) inc += t;
      }
      const uint32_t ex = inc - sum;
      if (ex < krem && krem <= inc) {
        uint32_t c = ex;
        for (int j = 0; j < per; ++j) {
          const uint32_t h = hist[top - j];
          if (c + h >= krem) {
            sh_bin = (uint32_t)(top - j);
            sh_krem = krem - c;
            break;
          }
          c += h;
        }
      }
    }
    __syncthreads();
    prefix |= sh_bin << shift;
    mask |= (uint32_t)(nb - 1) << shift;
    krem = sh_krem;
    __syncthreads();
  }
  const uint32_t T = prefix;       // key of the k-th largest score
  const uint32_t need_eq = krem;   // how many entries equal to T are taken (smallest positions first)

  uint32_t base_gt = 0, base_eq = 0;
  for (int c0 = 0; c0 < n; c0 += 4 * kTopkThreads) {
    const int s0 = c0 + 4 * tid;
    uint32_t key[4];
    uint32_t cnt = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      key[j] = s0 + j < n ? order_key(sc[s0 + j]) : 0u;
      if (s0 + j < n) cnt += (key[j] > T ? 1u : 0u) + (key[j] == T ? 0x10000u : 0u);
    }
    uint32_t total;
    const uint32_t ex = block_exclusive_scan(cnt, warp_tot, total);
    uint32_t gt_before = base_gt + (ex & 0xFFFFu), eq_before = base_eq + (ex >> 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (s0 + j >= n) break;
      // slots are < k by construction; the guard only keeps inconsistent input inside the row
      if (key[j] > T) {
        const uint32_t slot = gt_before + (eq_before < need_eq ? eq_before : need_eq);
        if (slot < (uint32_t)k) out[slot] = s0 + j;
        ++gt_before;
      } else if (key[j] == T) {
        if (eq_before < need_eq && gt_before + eq_before < (uint32_t)k) out[gt_before + eq_before] = s0 + j;
        ++eq_before;
      }
    }
    base_gt += total & 0xFFFFu;
    base_eq += total >> 16;
  }
}

cudaError_t launch_topk(const RowMeta& m, int row0, int nrows, const float* scores, int64_t score_stride,
                        int max_seq_len, int topk, int32_t* topk_idx, cudaStream_t s) {
  topk_kernel<<<nrows, kTopkThreads, 0, s>>>(m, row0, scores, score_stride, max_seq_len, topk, topk_idx);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace dsa
