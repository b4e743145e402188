// Lightning-indexer scoring:
//   I(r, s) = sum_{h<32} w[r,h] * max(0, q_idx[r,h,:] . K[s,:])   for 0 <= s <= pos(r)
// ("vLLM Inference Path: GLM-5.2 as an Example", "DSA Indexer"; "Making GLM-5.2
// Sparse on TPUs", "Separate the indexer from the attention it controls").
//
// One thread scores one key; the row's 32 x 128 query and its head weights sit
// in shared memory as fp32.  For e4m3 keys the per-token scale is positive, so
// it commutes with the ReLU and is applied once to the head-weighted sum.
// Positions beyond pos(r) get -inf, so the score buffer is masked before any
// selection ("Making GLM-5.2 Sparse on TPUs", "Make the sparsity unit match the
// memory unit": masks must precede the reduction).
#include "dsa_internal.cuh"

namespace dsa {

__device__ __forceinline__ void unpack_bf16x8(const uint4 raw, float* k) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    k[2 * i] = __low2float(p[i]);
    k[2 * i + 1] = __high2float(p[i]);
  }
}

__device__ __forceinline__ void unpack_e4m3x8(const uint2 raw, float* k) {
  const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu);
    const __half2 h = __half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3));
    const float2 f = __half22float2(h);
    k[2 * i] = f.x;
    k[2 * i + 1] = f.y;
  }
}

template <bool kFp8>
__global__ void __launch_bounds__(256) indexer_scores_kernel(
    const uint8_t* __restrict__ keys, const float* __restrict__ scales, int log2_page, int num_pages, RowMeta m,
    int row0, int max_seq_len, const __nv_bfloat16* __restrict__ q_idx, const float* __restrict__ w,
    float* __restrict__ scores, int64_t stride) {
  __shared__ float4 qs[kIndexHeads][kIndexDim / 4];
  __shared__ float ws[kIndexHeads];
  const int r = row0 + blockIdx.y;
  int b, pos;
  row_info(m, r, b, pos);
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  float* out = scores + (int64_t)blockIdx.y * stride;
  if ((int)(blockIdx.x * blockDim.x) > pos) {
    if (s < max_seq_len) out[s] = -INFINITY;
    return;
  }
  const __nv_bfloat162* qr = reinterpret_cast<const __nv_bfloat162*>(q_idx + (int64_t)r * kIndexHeads * kIndexDim);
  float* qf = reinterpret_cast<float*>(&qs[0][0]);
  for (int i = threadIdx.x; i < kIndexHeads * kIndexDim / 2; i += blockDim.x) {
    const __nv_bfloat162 v = qr[i];
    qf[2 * i] = __low2float(v);
    qf[2 * i + 1] = __high2float(v);
  }
  if (threadIdx.x < kIndexHeads) ws[threadIdx.x] = w[(int64_t)r * kIndexHeads + threadIdx.x];
  __syncthreads();
  if (s >= max_seq_len) return;
  const int64_t slot = s <= pos ? token_slot(m, b, s, log2_page, num_pages) : -1;
  if (slot < 0) {
    out[s] = -INFINITY;
    return;
  }
  float acc[kIndexHeads];
#pragma unroll
  for (int h = 0; h < kIndexHeads; ++h) acc[h] = 0.f;
#pragma unroll 2
  for (int d0 = 0; d0 < kIndexDim; d0 += 8) {
    float k[8];
    if (kFp8) unpack_e4m3x8(*reinterpret_cast<const uint2*>(keys + slot * kIndexDim + d0), k);
    else unpack_bf16x8(*reinterpret_cast<const uint4*>(keys + (slot * kIndexDim + d0) * 2), k);
#pragma unroll
    for (int h = 0; h < kIndexHeads; ++h) {
      const float4 a = qs[h][d0 / 4], c = qs[h][d0 / 4 + 1];
      acc[h] = fmaf(a.x, k[0], fmaf(a.y, k[1], fmaf(a.z, k[2], fmaf(a.w, k[3], acc[h]))));
      acc[h] = fmaf(c.x, k[4], fmaf(c.y, k[5], fmaf(c.z, k[6], fmaf(c.w, k[7], acc[h]))));
    }
  }
  float sc = 0.f;
#pragma unroll
  for (int h = 0; h < kIndexHeads; ++h) sc = fmaf(ws[h], fmaxf(acc[h], 0.f), sc);
  if (kFp8) sc *= scales[slot];
  out[s] = sc;
}

cudaError_t launch_indexer_scores(const dsa_cache& c, const RowMeta& m, int row0, int nrows, int max_seq_len,
                                  const void* q_idx, const float* w, float* scores, int64_t score_stride,
                                  cudaStream_t s) {
  const int threads = 256;
  dim3 grid((max_seq_len + threads - 1) / threads, nrows);
  const int lp = ilog2(c.page_size);
  const auto* keys = static_cast<const uint8_t*>(c.index_keys);
  const auto* q = static_cast<const __nv_bfloat16*>(q_idx);
  if (c.key_format == DSA_KEY_FP8_E4M3)
    indexer_scores_kernel<true><<<grid, threads, 0, s>>>(keys, c.index_scales, lp, c.num_pages, m, row0, max_seq_len,
                                                         q, w, scores, score_stride);
  else
    indexer_scores_kernel<false><<<grid, threads, 0, s>>>(keys, nullptr, lp, c.num_pages, m, row0, max_seq_len, q, w,
                                                          scores, score_stride);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace dsa
