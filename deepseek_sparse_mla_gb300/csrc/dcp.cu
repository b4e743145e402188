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
  const int r = blockIdx.x;
  for (int j = threadIdx.x; j < k; j += blockDim.x) {
    const int li = local_idx[(int64_t)r * k + j];
    cand_score[(int64_t)r * k + j] = li >= 0 ? local_scores[(int64_t)r * stride + li] : -INFINITY;
    cand_pos[(int64_t)r * k + j] = li >= 0 ? li * world + rank : -1;
  }
}

// Top-k of one row's candidates [world][rows][k] (score, global position; position -1 = empty).
// Candidate keys (order_key(score) << 32 | ~position) are unique and rank larger score first, then
// the smaller position; an MSB-first radix select of 8 passes of 8 bits finds the k-th largest key,
// the selected positions are compacted and bitonic-sorted ascending.
__global__ void __launch_bounds__(kSelThreads) dcp_select_kernel(const float* __restrict__ cand_score,
                                                                 const int32_t* __restrict__ cand_pos, int world,
                                                                 int rows, int k, int rank,
                                                                 int32_t* __restrict__ global_idx,
                                                                 int32_t* __restrict__ local_idx) {
  __shared__ uint32_t hist[256];
  __shared__ int32_t spos[kMaxCand / 2];               // the selection (k <= DSA_MAX_TOPK = 8192)
  __shared__ uint32_t sh[4];
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = world * k;
  uint64_t key[kPerThread];
  uint32_t nvalid = 0;
#pragma unroll
  for (int i = 0; i < kPerThread; ++i) {
    const int c = tid + i * kSelThreads;
    key[i] = 0;
    if (c < n) {
      const int w = c / k, j = c - w * k;
      const int64_t at = ((int64_t)w * rows + r) * k + j;
      const int32_t pos = cand_pos[at];
      if (pos >= 0) {
        key[i] = ((uint64_t)dcp_order_key(cand_score[at]) << 32) | (uint32_t)~(uint32_t)pos;
        ++nvalid;
      }
    }
  }
  if (tid == 0) sh[0] = 0;
  __syncthreads();
  atomicAdd(&sh[0], nvalid);
  __syncthreads();
  const uint32_t V = sh[0];
  uint64_t T = 1;                                      // select every valid candidate
  if (V > (uint32_t)k) {
    uint64_t prefix = 0, mask = 0;
    uint32_t krem = (uint32_t)k;
    for (int pass = 0; pass < 8; ++pass) {
      const int shift = 56 - 8 * pass;
      for (int b = tid; b < 256; b += kSelThreads) hist[b] = 0;
      __syncthreads();
#pragma unroll
      for (int i = 0; i < kPerThread; ++i)
        if (key[i] != 0 && (key[i] & mask) == prefix) atomicAdd(&hist[(key[i] >> shift) & 255u], 1u);
      __syncthreads();
      if (warp == 0) {
        // lane l holds bins 255 - 8l .. 248 - 8l (from the top); find the bin holding the krem-th key
        uint32_t c[8], tot = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          c[q] = hist[255 - 8 * lane - q];
          tot += c[q];
        }
        uint32_t inc = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += t;
        }
        const uint32_t ex = inc - tot;
        if (ex < krem && krem <= inc) {
          uint32_t cum = ex;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (cum + c[q] >= krem) {
              sh[1] = 255 - 8 * lane - q;
              sh[2] = krem - cum;
              break;
            }
            cum += c[q];
          }
        }
      }
      __syncthreads();
      prefix |= (uint64_t)sh[1] << shift;
      mask |= (uint64_t)0xFFu << shift;
      krem = sh[2];
      __syncthreads();
    }
    T = prefix;                                        // keys are unique: exactly k are >= T
  }
  // compact the selected positions, then sort them ascending
  if (tid == 0) sh[3] = 0;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kPerThread; ++i)
    if (key[i] != 0 && key[i] >= T) {
      const uint32_t slot = atomicAdd(&sh[3], 1u);
      if (slot < (uint32_t)k) spos[slot] = (int32_t)~(uint32_t)key[i];  // more only if a position repeats
    }
  __syncthreads();
  const int cnt = min((int)sh[3], k);
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
  for (int i = tid; i < k; i += kSelThreads) {
    const int32_t p = i < cnt ? spos[i] : -1;
    global_idx[(int64_t)r * k + i] = p;
    local_idx[(int64_t)r * k + i] = (p >= 0 && p % world == rank) ? p / world : -1;
  }
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
  float M = -INFINITY;
  for (int w = 0; w < world; ++w) M = fmaxf(M, lses[((int64_t)w * rows + r) * kHeads + h]);
  float acc[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0.f;
  float L = 0.f;
  if (M > -INFINITY) {
    for (int w = 0; w < world; ++w) {
      const float lw = lses[((int64_t)w * rows + r) * kHeads + h];
      if (lw == -INFINITY) continue;
      const float wt = expf(lw - M);
      L += wt;
      const uint4* src = reinterpret_cast<const uint4*>(outs + (((int64_t)w * rows + r) * kHeads + h) * kLatent + d0);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint4 v = src[q];
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(b2[e]);
          acc[8 * q + 2 * e] = fmaf(wt, f.x, acc[8 * q + 2 * e]);
          acc[8 * q + 2 * e + 1] = fmaf(wt, f.y, acc[8 * q + 2 * e + 1]);
        }
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
  cudaError_t e = launch_pdl(dcp_candidates_kernel, dim3(rows), dim3(256), 0, s, local_scores, stride, local_idx, k,
                             rank, world, cand_score, cand_pos);
  count_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_dcp_select(const float* cand_score, const int32_t* cand_pos, int world, int rows, int k, int rank,
                              int32_t* global_idx, int32_t* local_idx, cudaStream_t s) {
  cudaError_t e = launch_pdl(dcp_select_kernel, dim3(rows), dim3(kSelThreads), 0, s, cand_score, cand_pos, world, rows,
                             k, rank, global_idx, local_idx);
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
