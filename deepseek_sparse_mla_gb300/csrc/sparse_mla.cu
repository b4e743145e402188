// Sparse absorbed MLA over the selected positions, with split-k over the
// selection and a log-sum-exp merge.
//
// For row r, head h and valid selected s (0 <= s <= pos(r)):
//   z_s = scale * (q[r,h,:512] . c_KV[s] + q[r,h,512:] . k_R[s])
//   out[r,h,:] = sum_s softmax(z)_s c_KV[s],  lse[r,h] = ln sum_s exp(z_s)
// ("vLLM Inference Path: GLM-5.2 as an Example", "MLA Projections and KV State"
// and "Sparse MLA Attention"; "Making GLM-5.2 Sparse on TPUs", "Separate the
// indexer from the attention it controls": absorbed MLA with the scale tied to
// the unabsorbed 192 + 64 width, and "Carry sparse reads through prefill":
// online softmax over the selected entries).
//
// Grid = (split, row).  A CTA streams its slice of the row's index buffer in
// tiles of 32 cached rows gathered through the page table, keeps a running
// max / sum per head (online softmax) and the 64 x 512 output accumulator in
// registers.  With one split it writes the bf16 output directly; otherwise it
// writes (acc, m, l) partials that the merge kernel combines by LSE.
#include "dsa_internal.cuh"

namespace dsa {

constexpr int kTileTokens = 32;
constexpr int kThreadsMla = 512;           // thread = (head h = tid / 8, lane-in-head j = tid % 8)
constexpr int kRowPad = kRow + 8;          // padded smem row: 1168 bytes, keeps 8 rows on distinct banks
constexpr int kChunksRow = kRow / 8;       // 72 chunks of 8 bf16 per cached row

__device__ __forceinline__ float dot8(const uint4 a, const uint4 b, float acc) {
  const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fx = __bfloat1622float2(x[i]), fy = __bfloat1622float2(y[i]);
    acc = fmaf(fx.x, fy.x, fmaf(fx.y, fy.y, acc));
  }
  return acc;
}

__global__ void __launch_bounds__(kThreadsMla) sparse_mla_kernel(
    const uint4* __restrict__ latent, int log2_page, int num_pages, RowMeta m, const uint4* __restrict__ q,
    const int32_t* __restrict__ topk_idx, int topk, float scale, int tokens_per_split, int splits,
    __nv_bfloat16* __restrict__ out, float* __restrict__ lse, float* __restrict__ part_o, float* __restrict__ part_ml) {
  extern __shared__ uint4 smem[];
  uint4* qs = smem;                                   // [64][kRowPad/8] chunks
  uint4* kv = qs + kHeads * (kRowPad / 8);            // [32][kRowPad/8]
  float* ps = reinterpret_cast<float*>(kv + kTileTokens * (kRowPad / 8));   // [64][32]
  __shared__ int64_t tok_slot[kTileTokens];

  const int r = blockIdx.y, split = blockIdx.x;
  const int tid = threadIdx.x, h = tid >> 3, j = tid & 7;
  int b, pos;
  row_info(m, r, b, pos);

  const uint4* qg = q + (int64_t)r * kHeads * kChunksRow;
  for (int i = tid; i < kHeads * kChunksRow; i += kThreadsMla) qs[(i / kChunksRow) * (kRowPad / 8) + i % kChunksRow] = qg[i];

  float m_run = -INFINITY, l_run = 0.f;
  float acc[64];   // dims (c * 8 + j) * 8 + e for c, e in 0..7
#pragma unroll
  for (int i = 0; i < 64; ++i) acc[i] = 0.f;

  const int t_begin = split * tokens_per_split;
  const int t_end = min(topk, t_begin + tokens_per_split);
  const int32_t* idx_row = topk_idx + (int64_t)r * topk;
  for (int t0 = t_begin; t0 < t_end; t0 += kTileTokens) {
    __syncthreads();
    if (tid < kTileTokens) {
      const int t = t0 + tid;
      int64_t sl = -1;
      if (t < t_end) {
        const int s = idx_row[t];
        if (s >= 0 && s <= pos) sl = token_slot(m, b, s, log2_page, num_pages);
      }
      tok_slot[tid] = sl;
    }
    __syncthreads();
    for (int i = tid; i < kTileTokens * kChunksRow; i += kThreadsMla) {
      const int tt = i / kChunksRow, c = i % kChunksRow;
      const int64_t sl = tok_slot[tt];
      kv[tt * (kRowPad / 8) + c] = sl >= 0 ? latent[sl * kChunksRow + c] : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();

    float sc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int tt = j + 8 * u;
      const uint4* qrow = qs + h * (kRowPad / 8);
      const uint4* krow = kv + tt * (kRowPad / 8);
      float d = 0.f;
#pragma unroll 8
      for (int c = 0; c < kChunksRow; ++c) d = dot8(qrow[c], krow[c], d);
      sc[u] = tok_slot[tt] >= 0 ? d * scale : -INFINITY;
    }
    float tmax = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
    const float m_new = fmaxf(m_run, tmax);
    const float alpha = m_new == -INFINITY ? 1.f : expf(m_run - m_new);
    float psum = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float p = sc[u] == -INFINITY ? 0.f : expf(sc[u] - m_new);
      ps[h * kTileTokens + j + 8 * u] = p;
      psum += p;
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
    l_run = l_run * alpha + psum;
    m_run = m_new;
    __syncthreads();

#pragma unroll
    for (int i = 0; i < 64; ++i) acc[i] *= alpha;
    for (int tt = 0; tt < kTileTokens; ++tt) {
      const float p = ps[h * kTileTokens + tt];
      if (p == 0.f) continue;
      const uint4* krow = kv + tt * (kRowPad / 8);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = krow[c * 8 + j];
        const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(x[e]);
          acc[c * 8 + 2 * e] = fmaf(p, f.x, acc[c * 8 + 2 * e]);
          acc[c * 8 + 2 * e + 1] = fmaf(p, f.y, acc[c * 8 + 2 * e + 1]);
        }
      }
    }
  }

  if (splits == 1) {
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    __nv_bfloat16* o = out + ((int64_t)r * kHeads + h) * kLatent;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 v;
      __nv_bfloat162* x = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = __floats2bfloat162_rn(acc[c * 8 + 2 * e] * inv, acc[c * 8 + 2 * e + 1] * inv);
      reinterpret_cast<uint4*>(o)[c * 8 + j] = v;
    }
    if (lse && j == 0) lse[(int64_t)r * kHeads + h] = l_run > 0.f ? m_run + logf(l_run) : -INFINITY;
  } else {
    const int64_t base = ((int64_t)r * splits + split) * kHeads + h;
    float4* o = reinterpret_cast<float4*>(part_o + base * kLatent);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      o[(c * 8 + j) * 2] = make_float4(acc[c * 8], acc[c * 8 + 1], acc[c * 8 + 2], acc[c * 8 + 3]);
      o[(c * 8 + j) * 2 + 1] = make_float4(acc[c * 8 + 4], acc[c * 8 + 5], acc[c * 8 + 6], acc[c * 8 + 7]);
    }
    if (j == 0) {
      part_ml[base * 2] = m_run;
      part_ml[base * 2 + 1] = l_run;
    }
  }
}

// LSE merge of split partials: O = sum_j e^{m_j - M} acc_j / sum_j e^{m_j - M} l_j, lse = M + ln L.
__global__ void __launch_bounds__(kThreadsMla) mla_merge_kernel(const float* __restrict__ part_o,
                                                                const float* __restrict__ part_ml, int splits,
                                                                __nv_bfloat16* __restrict__ out,
                                                                float* __restrict__ lse) {
  const int r = blockIdx.x, tid = threadIdx.x, h = tid >> 3, j = tid & 7;
  float M = -INFINITY;
  for (int sp = 0; sp < splits; ++sp) M = fmaxf(M, part_ml[(((int64_t)r * splits + sp) * kHeads + h) * 2]);
  float L = 0.f;
  float acc[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) acc[i] = 0.f;
  for (int sp = 0; sp < splits; ++sp) {
    const int64_t base = ((int64_t)r * splits + sp) * kHeads + h;
    const float mj = part_ml[base * 2], lj = part_ml[base * 2 + 1];
    if (!(lj > 0.f)) continue;
    const float wgt = expf(mj - M);
    L = fmaf(wgt, lj, L);
    const float4* o = reinterpret_cast<const float4*>(part_o + base * kLatent);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float4 a = o[(c * 8 + j) * 2], bq = o[(c * 8 + j) * 2 + 1];
      acc[c * 8 + 0] = fmaf(wgt, a.x, acc[c * 8 + 0]);
      acc[c * 8 + 1] = fmaf(wgt, a.y, acc[c * 8 + 1]);
      acc[c * 8 + 2] = fmaf(wgt, a.z, acc[c * 8 + 2]);
      acc[c * 8 + 3] = fmaf(wgt, a.w, acc[c * 8 + 3]);
      acc[c * 8 + 4] = fmaf(wgt, bq.x, acc[c * 8 + 4]);
      acc[c * 8 + 5] = fmaf(wgt, bq.y, acc[c * 8 + 5]);
      acc[c * 8 + 6] = fmaf(wgt, bq.z, acc[c * 8 + 6]);
      acc[c * 8 + 7] = fmaf(wgt, bq.w, acc[c * 8 + 7]);
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16* o = out + ((int64_t)r * kHeads + h) * kLatent;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint4 v;
    __nv_bfloat162* x = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
    for (int e = 0; e < 4; ++e) x[e] = __floats2bfloat162_rn(acc[c * 8 + 2 * e] * inv, acc[c * 8 + 2 * e + 1] * inv);
    reinterpret_cast<uint4*>(o)[c * 8 + j] = v;
  }
  if (lse && j == 0) lse[(int64_t)r * kHeads + h] = L > 0.f ? M + logf(L) : -INFINITY;
}

cudaError_t launch_sparse_mla(const dsa_cache& c, const RowMeta& m, int num_rows, const void* q,
                              const int32_t* topk_idx, int topk, float scale, void* out, float* lse,
                              void* workspace, const MlaPlan& plan, cudaStream_t s) {
  const size_t smem = (size_t)(kHeads + kTileTokens) * kRowPad * 2 + (size_t)kHeads * kTileTokens * 4;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(sparse_mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  float* part_o = nullptr;
  float* part_ml = nullptr;
  if (plan.splits > 1) {
    part_o = reinterpret_cast<float*>(static_cast<char*>(workspace) + kWorkspaceHeader);
    part_ml = part_o + (size_t)num_rows * plan.splits * kHeads * kLatent;
  }
  dim3 grid(plan.splits, num_rows);
  sparse_mla_kernel<<<grid, kThreadsMla, smem, s>>>(
      static_cast<const uint4*>(c.latent), ilog2(c.page_size), c.num_pages, m, static_cast<const uint4*>(q), topk_idx,
      topk, scale, plan.tokens_per_split, plan.splits, static_cast<__nv_bfloat16*>(out), lse, part_o, part_ml);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || plan.splits == 1) return e;
  mla_merge_kernel<<<num_rows, kThreadsMla, 0, s>>>(part_o, part_ml, plan.splits, static_cast<__nv_bfloat16*>(out), lse);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace dsa
