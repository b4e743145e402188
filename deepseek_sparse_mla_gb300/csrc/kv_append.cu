// Paged KV append: scatter this step's tokens into one layer's latent pages and,
// for an indexer-owning layer, its index-key pages.
//
// "Making GLM-5.2 Sparse on TPUs", "Append new KV without moving the resident
// cache": the cost must scale with the new rows, never with the resident pool,
// and every other slot keeps its contents.  Here one warp owns one new token
// and moves its 1152-byte latent row (or its packed 8-bit 640-byte row and
// scale) with 16-byte stores straight into its slot; nothing else in the pool
// is read or written.
#include <cuda_fp16.h>

#include "dsa_internal.cuh"

namespace dsa {

// blockIdx.y = layer: one launch appends the step's tokens to every layer's caches (the tokens and
// their slots are the same in every layer of a step; each layer brings its own rows and keys)
__global__ void __launch_bounds__(256) kv_append_kernel(const AppendArgs a) {
  const AppendLayer& L = a.layer[blockIdx.y];
  const int t = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  if (t >= a.num_tokens) return;
  const int64_t slot = a.slot_mapping[t];
  if (slot < 0 || slot >= L.total_slots) return;

  constexpr int kChunksC = kLatent * 2 / 16, kChunksR = kRope * 2 / 16;
  const uint4* src_c = L.c_kv + (int64_t)t * kChunksC;
  const uint4* src_r = L.k_rope + (int64_t)t * kChunksR;
  if (L.latent_format == DSA_LATENT_BF16) {
    // latent row [c_KV(512) | k_R(64)] bf16 = 64 + 8 chunks of 16 bytes, copied bit-exactly
    uint4* dst = L.latent + slot * (kChunksC + kChunksR);
    for (int i = lane; i < kChunksC + kChunksR; i += 32) dst[i] = i < kChunksC ? src_c[i] : src_r[i - kChunksC];
  } else {
    // packed 8-bit row [c_KV as 512 e4m3 codes | k_R as 64 bf16] = 32 + 8 chunks of 16 bytes; the
    // codes by the index keys' rule (scale = amax / 448, or 1 if amax = 0; rne_satfinite(x / scale))
    uint4* dst = L.latent + slot * (kLatent / 16 + kChunksR);
    float x[16];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint4 v = src_c[2 * lane + q];
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[8 * q + 2 * e] = __low2float(b2[e]);
        x[8 * q + 2 * e + 1] = __high2float(b2[e]);
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    uint32_t packed[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(__fdiv_rn(x[i], scale), __NV_SATFINITE, __NV_E4M3);
      packed[i >> 2] |= (uint32_t)c << (8 * (i & 3));
    }
    dst[lane] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    if (lane < kChunksR) dst[kLatent / 16 + lane] = src_r[lane];
    if (lane == 0) L.latent_scales[slot] = scale;
  }

  if (L.index_keys == nullptr) return;
  if (L.key_format == DSA_KEY_BF16) {                 // 256 bytes per key, copied
    if (lane < 16)
      reinterpret_cast<uint4*>(L.index_keys)[slot * 16 + lane] = reinterpret_cast<const uint4*>(L.k_idx)[(int64_t)t * 16 + lane];
    return;
  }
  if (L.k_idx_format != DSA_KEY_BF16) {                // pre-quantised: 128 code bytes + scale, copied
    if (lane < 8)
      reinterpret_cast<uint4*>(L.index_keys)[slot * 8 + lane] = reinterpret_cast<const uint4*>(L.k_idx)[(int64_t)t * 8 + lane];
    if (lane == 0) {
      if (L.key_format == DSA_KEY_INT8)                // binary16 scales
        reinterpret_cast<uint16_t*>(L.index_scales)[slot] = reinterpret_cast<const uint16_t*>(L.k_idx_scales)[t];
      else
        L.index_scales[slot] = L.k_idx_scales[t];
    }
    return;
  }
  const uint2 raw = reinterpret_cast<const uint2*>(L.k_idx)[(int64_t)t * 32 + lane];   // 4 bf16 per lane
  float x[4];
  {
    const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
    const __nv_bfloat162 q = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
    x[0] = __low2float(p); x[1] = __high2float(p); x[2] = __low2float(q); x[3] = __high2float(q);
  }
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (L.key_format == DSA_KEY_INT8) {
    // quantise into int8 with a binary16 scale: scale = half(amax / 127) (nearest-even, held at
    // 65504 above and at the smallest positive half 2^-24 below; 1 if amax = 0), code =
    // rne(x / scale) with the stored scale, clamped to [-127, 127]
    uint16_t hb = __half_as_ushort(__float2half_rn(fminf(__fdiv_rn(amax, 127.0f), 65504.0f)));
    if (!(amax > 0.f)) hb = 0x3C00;
    else if (hb == 0) hb = 1;
    const float scale = __half2float(__ushort_as_half(hb));
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float c = fminf(fmaxf(rintf(__fdiv_rn(x[i], scale)), -127.0f), 127.0f);
      packed |= ((uint32_t)(int)c & 0xFFu) << (8 * i);
    }
    reinterpret_cast<uint32_t*>(L.index_keys)[slot * 32 + lane] = packed;
    if (lane == 0) reinterpret_cast<uint16_t*>(L.index_scales)[slot] = hb;
    return;
  }
  // quantise a bf16 key into e4m3: scale = amax / 448 (1 if amax = 0), code = rne_satfinite(x / scale)
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(__fdiv_rn(x[i], scale), __NV_SATFINITE, __NV_E4M3);
    packed |= (uint32_t)c << (8 * i);
  }
  reinterpret_cast<uint32_t*>(L.index_keys)[slot * 32 + lane] = packed;
  if (lane == 0) L.index_scales[slot] = scale;
}

AppendLayer append_layer(const dsa_cache& c, const void* c_kv, const void* k_rope, const void* k_idx, int k_idx_format,
                         const float* k_idx_scales) {
  AppendLayer L;
  L.latent = static_cast<uint4*>(c.latent);
  L.total_slots = (int64_t)c.num_pages * c.page_size;
  L.index_keys = static_cast<uint8_t*>(c.index_keys);
  L.index_scales = c.index_scales;
  L.latent_scales = c.latent_scales;
  L.key_format = c.key_format;
  L.latent_format = c.latent_format;
  L.c_kv = static_cast<const uint4*>(c_kv);
  L.k_rope = static_cast<const uint4*>(k_rope);
  L.k_idx = static_cast<const uint8_t*>(k_idx);
  L.k_idx_format = k_idx_format;
  L.k_idx_scales = k_idx_scales;
  return L;
}

cudaError_t launch_kv_append(const AppendArgs& a, int num_layers, cudaStream_t s) {
  const int threads = 256, per_block = threads / 32;
  const int blocks = (a.num_tokens + per_block - 1) / per_block;
  cudaError_t e = launch_pdl(kv_append_kernel, dim3(blocks, num_layers), dim3(threads), 0, s, a);
  count_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dsa
