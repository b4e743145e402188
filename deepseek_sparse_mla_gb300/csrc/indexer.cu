// Lightning-indexer scoring on tcgen05 tensor cores:
//   I(r, s) = sum_{h<32} w[r,h] * max(0, q_idx[r,h,:] . K[s,:])   for 0 <= s <= pos(r), -inf beyond
// ("vLLM Inference Path: GLM-5.2 as an Example", "DSA Indexer"; "Making GLM-5.2
// Sparse on TPUs", "Separate the indexer from the attention it controls").
//
// Rows are grouped by request (1 row in decode, up to 4 with e4m3 keys or 8
// with bf16 keys otherwise); every key read from HBM serves the whole group.
// One tile of 128 keys is one MMA chain D[key, (row, head, term)]:
//   M = 128 keys, N = 32 heads x terms x rows, K = 128, fp32 accumulators in TMEM,
// and the epilogue applies ReLU, the head weights, the key's scale and the
// causal mask (masks precede any selection: "Making GLM-5.2 Sparse on TPUs",
// "Make the sparsity unit match the memory unit").
//
// e4m3 keys run on the kind::f8f6f4 MMA with e4m3 on both sides: each (row,
// head) query vector is scaled by an exact power of two and split into two
// e4m3 terms q' = t1 + t2/16 that represent it exactly (query_exponent below),
// so the two accumulators give q . k exactly up to fp32 rounding; bf16 keys
// use kind::f16 with the bf16 queries as they are.  int8 keys (binary16
// scales) have no tensor path of their own on sm_103a (no integer MMA): three
// converter warps split each landed tile byte for byte into two e4m3 tiles,
// hi = e4m3(v) in place and lo = v - hi beside it (both exact, |lo| <= 4), and
// the issuer runs the e4m3 chain over both into the same accumulators.
//
// Per CTA (persistent, one per SM, 544 threads), over one contiguous range of
// the flattened (group, key tile) list:
//   warps 0-5  producers, tiles round-robin: page lookups from a register
//              window of the block table, TMA loads of the key pages into a
//              ring of 16 KB (e4m3) or 32 KB (bf16) stages, and bulk copies of
//              the keys' fp32 scales into a separate ring of scale slots;
//   warps 6-7  MMA issuers, even and odd tiles; a commit frees the key stage;
//   warp 8     B loader: each group's queries (split into e4m3 terms, or bf16)
//              into the B operand, 128-byte swizzled, K-major; the CTA's first
//              group together with the epilogue warps, which have no tile yet;
//   warps 9-16 two epilogue warpgroups, even and odd tiles (fed by the
//              matching issuer); the one that reads a tile's scales frees
//              its scale slot;
//   warps 17-19 (int8 keys only) converters, tile i by warp i % 3, each with
//              its own lo tile that the MMA of its previous tile releases.
// The key ring holds up to 8 stages (6 with int8 keys): enough bytes in flight
// to cover HBM latency, few enough not to congest the memory system.
#include <mutex>
#include <type_traits>

#include <cuda_fp16.h>

#include "dsa_internal.cuh"
#include "sm100.cuh"
#include "tmap.cuh"

namespace dsa {
using namespace sm100;

namespace idx {
constexpr int kTileKeys = 128;
constexpr int kProducers = 6;                      // warps issuing the key copies, tiles round-robin (at most the stages)
constexpr int kMmaWarps = 2;                       // MMA issuers: even and odd tiles
constexpr int kThreads = 32 * (kProducers + kMmaWarps + 1 + 8);  // producers, MMA, B loader, two epilogue warpgroups
constexpr int kConvWarps = 3;                      // int8 keys: tile converters (a divisor of the 6 key stages)
constexpr int kThreadsI8 = kThreads + 32 * kConvWarps;
constexpr int kI8Stages = 6;                       // int8 keys: always 6 stages (stage s is converted by warp s % 3)
constexpr int kI8MaxRows = 2;                      // int8 keys: rows per group, so that 6 stages and 3 lo tiles fit
constexpr int kBBytes = 65536;                      // B operand at most: 256 (row, head) query vectors
// Dynamic shared memory: [B buffers | key-scale ring | key ring].  The B buffers take only what the
// group size needs (16 KB in decode), and the key ring gets the rest, up to kMaxStages stages.
constexpr int kSmemBytes = 200 * 1024;
// Key stages in flight (16 KB e4m3 or 32 KB bf16).  With 6 producer warps, 8 stages of 16 KB
// measured 3.5 % faster than 3 producers over 6 stages, and 10 stages no faster than 8.
constexpr int kMaxStages = 8;
constexpr int kScStages = 16;                       // key-scale ring (e4m3): 16 tiles x 128 fp32
constexpr int kScRingBytes = kScStages * 128 * 4;   // fp32 scales (e4m3 keys); binary16 scales take half
static_assert((kScStages & (kScStages - 1)) == 0 && kScStages >= kMaxStages + 4, "scale ring: power of two, deep");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kPolls = 1u << 22;
constexpr int kMaxRows = 8;
constexpr int kGroupCache = 1024;                    // group descriptors staged in shared memory
}  // namespace idx

struct IdxArgs {
  RowMeta m;
  const int4* groups;            // [n][ (request, first row, rows, position of the first row) ]
  const int32_t* tile_start;     // [n + 1] exclusive prefix of each group's key tiles
  const int32_t* counts;         // [0] = groups, [1] = total key tiles
  int max_groups;
  int row0;                      // scores row = r - row0
  int rows_per_group;            // rows of one group at most (1 in decode)
  int log2_page, num_pages, box_rows;
  const float* key_scales;       // e4m3 keys only
  const __nv_bfloat16* q_idx;
  const float* w;
  float* scores;
  int64_t stride;
  int max_seq_len;
  int page_log2;                 // >= 0: page mode, write maxima over units of 2^min(page_log2, 5) visible keys
  int max_pages;                 // unit columns per row (page mode)
  uint32_t* err;
};

// Walks one CTA's contiguous range of the flattened (group, key tile) list.
struct TileCursor {
  int tau, tau_end;      // flattened tile index and end of this CTA's range
  int g, g_end_tile;     // current group and the flattened index where it ends
  int4 G;                // (request, first row, rows, first position) of group g
  int t;                 // key tile within the group
  __device__ bool valid() const { return tau < tau_end; }
};

__device__ __forceinline__ int4 group_at(const IdxArgs& a, const int4* gcache, int g) {
  return g < idx::kGroupCache ? gcache[g] : a.groups[g];
}

__device__ __forceinline__ int tile_start_at(const IdxArgs& a, const int* tcache, int g) {
  return g <= idx::kGroupCache ? tcache[g] : a.tile_start[g];
}

__device__ __forceinline__ void cursor_init(TileCursor& c, const IdxArgs& a, const int4* gcache, const int* tcache,
                                            int ngroups, int tau0, int tau1) {
  c.tau = tau0;
  c.tau_end = tau1;
  if (tau0 >= tau1) return;
  int lo = 0, hi = ngroups - 1;          // last group whose first tile is <= tau0
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start_at(a, tcache, mid) <= tau0) lo = mid; else hi = mid - 1;
  }
  c.g = lo;
  while (tile_start_at(a, tcache, c.g + 1) <= tau0) ++c.g;   // skip groups without tiles
  c.g_end_tile = tile_start_at(a, tcache, c.g + 1);
  c.G = group_at(a, gcache, c.g);
  c.t = tau0 - tile_start_at(a, tcache, c.g);
}

// Advance one tile; returns true when the next tile starts a new group.
__device__ __forceinline__ bool cursor_next(TileCursor& c, const IdxArgs& a, const int4* gcache, const int* tcache) {
  ++c.tau;
  ++c.t;
  if (c.tau < c.g_end_tile || c.tau >= c.tau_end) return false;
  do {
    ++c.g;
    c.g_end_tile = tile_start_at(a, tcache, c.g + 1);
  } while (c.g_end_tile <= c.tau);
  c.G = group_at(a, gcache, c.g);
  c.t = 0;
  return true;
}


// Exponent that moves a (row, head) query vector into the e4m3 split range: with q' = q * 2^(7-e),
// max |q'| lies in [128, 256).  q' = t1 + t2/16 with t1 = e4m3(q') and t2 = e4m3(16 (q' - t1)) is exact
// for every element above the e4m3 subnormal range (the rounding residual of a 4-bit mantissa has at
// most 4 significant bits), so the score needs no f16/bf16 operand.  Returns e; raw gets the query.
__device__ __forceinline__ int query_exponent(const IdxArgs& a, int row, int h, uint4 (&raw)[16]) {
  const __nv_bfloat16* qv = a.q_idx + ((int64_t)row * kIndexHeads + h) * kIndexDim;
#pragma unroll
  for (int c = 0; c < 16; ++c) raw[c] = reinterpret_cast<const uint4*>(qv)[c];
  float amax = 0.f;
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&raw[c]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(x[e]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
  return amax > 0.f ? ilogbf(amax) : 0;
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return (uint32_t)__nv_cvt_float_to_fp8(a, __NV_SATFINITE, __NV_E4M3) |
         ((uint32_t)__nv_cvt_float_to_fp8(b, __NV_SATFINITE, __NV_E4M3) << 8) |
         ((uint32_t)__nv_cvt_float_to_fp8(c, __NV_SATFINITE, __NV_E4M3) << 16) |
         ((uint32_t)__nv_cvt_float_to_fp8(d, __NV_SATFINITE, __NV_E4M3) << 24);
}

// The B operand of row group G: its 32 G.z (row, head) query vectors, for 8-bit keys each as the two
// exact e4m3 terms t1 (B row 64 rr + h) and t2 (B row 64 rr + 32 + h), for bf16 keys as they are
// (B row 32 rr + h, two 64-element K halves), all in the 128-byte swizzled layout.  This thread
// writes vectors p0, p0 + dp, ...
template <bool kFp8>
__device__ __forceinline__ void fill_group_queries(const IdxArgs& a, int4 G, uint8_t* bbuf, int p0, int dp) {
  const int N = 32 * (kFp8 ? 2 : 1) * G.z;
  for (int p = p0; p < 32 * G.z; p += dp) {
    const int rr = p >> 5, h = p & 31;
    uint4 raw[16];
    if (kFp8) {
      const int e = query_exponent(a, G.y + rr, h, raw);
      const float up = ldexpf(1.f, 7 - e);
      const int n_hi = rr * 64 + h, n_lo = rr * 64 + 32 + h;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {        // 16-byte units of the 128-byte e4m3 rows
        uint32_t t1[4], t2[4];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const __nv_bfloat162* v = reinterpret_cast<const __nv_bfloat162*>(&raw[2 * c + half]);
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const float2 f0 = __bfloat1622float2(v[2 * e2]), f1 = __bfloat1622float2(v[2 * e2 + 1]);
            const float x[4] = {f0.x * up, f0.y * up, f1.x * up, f1.y * up};
            float r[4];
#pragma unroll
            for (int z = 0; z < 4; ++z) {
              const float v1 = __half2float(__nv_cvt_fp8_to_halfraw(
                  __nv_cvt_float_to_fp8(x[z], __NV_SATFINITE, __NV_E4M3), __NV_E4M3));
              r[z] = (x[z] - v1) * 16.f;
            }
            t1[2 * half + e2] = e4m3x4(x[0], x[1], x[2], x[3]);
            t2[2 * half + e2] = e4m3x4(r[0], r[1], r[2], r[3]);
          }
        }
        *reinterpret_cast<uint4*>(bbuf + sw128_offset(n_hi, c)) = make_uint4(t1[0], t1[1], t1[2], t1[3]);
        *reinterpret_cast<uint4*>(bbuf + sw128_offset(n_lo, c)) = make_uint4(t2[0], t2[1], t2[2], t2[3]);
      }
    } else {
      const __nv_bfloat16* qv = a.q_idx + ((int64_t)(G.y + rr) * kIndexHeads + h) * kIndexDim;
#pragma unroll
      for (int c = 0; c < 16; ++c) raw[c] = reinterpret_cast<const uint4*>(qv)[c];
#pragma unroll
      for (int c = 0; c < 16; ++c)
        *reinterpret_cast<uint4*>(bbuf + (c >> 3) * (N * 128) + sw128_offset(p, c & 7)) = raw[c];
    }
  }
}

// Four int8 codes (one 32-bit word) -> the e4m3 codes of hi = e4m3(v) (nearest-even) and lo = v - hi,
// byte for byte.  For |v| <= 127 both are exact e4m3 values (|lo| <= 4), so hi + lo = v.  Each v is
// first made a half exactly: the bits 0x64XX with XX = v + 128 are the half 1024 + v + 128.
__device__ __forceinline__ void split_int8_e4m3(uint32_t w, uint32_t& hi, uint32_t& lo) {
  const uint32_t u = w ^ 0x80808080u;
  const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));     // 1152
  const uint32_t pairs[2] = {__byte_perm(u, 0x64646464u, 0x5140), __byte_perm(u, 0x64646464u, 0x5342)};
  uint32_t h[2], l[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&pairs[j]), bias);
    const __nv_fp8x2_storage_t hc = __nv_cvt_halfraw2_to_fp8x2(__half2_raw(v), __NV_SATFINITE, __NV_E4M3);
    const __half2 hv = __half2(__nv_cvt_fp8x2_to_halfraw2(hc, __NV_E4M3));
    const __nv_fp8x2_storage_t lc = __nv_cvt_halfraw2_to_fp8x2(__half2_raw(__hsub2(v, hv)), __NV_SATFINITE, __NV_E4M3);
    h[j] = hc;
    l[j] = lc;
  }
  hi = h[0] | (h[1] << 16);
  lo = l[0] | (l[1] << 16);
}

__device__ __forceinline__ float scale_value(float v) { return v; }
__device__ __forceinline__ float scale_value(uint16_t v) { return __half2float(__ushort_as_half(v)); }

// kKind: 0 bf16 keys, 1 e4m3 keys (fp32 scales), 2 int8 keys (binary16 scales).
template <int kKind>
__global__ void __launch_bounds__(kKind == 2 ? idx::kThreadsI8 : idx::kThreads, 1)
    indexer_tc_kernel(const __grid_constant__ CUtensorMap key_map, const IdxArgs a, int groups_share_keys) {
  using namespace idx;
  constexpr bool kFp8 = kKind != 0;                   // 8-bit keys: the e4m3 MMA path
  constexpr bool kI8 = kKind == 2;
  using ScaleT = std::conditional_t<kI8, uint16_t, float>;   // a key scale as stored
  constexpr int kStageBytes = kFp8 ? 16384 : 32768;
  constexpr int kRowsMax = kFp8 ? (kI8 ? kI8MaxRows : 4) : 8;
  constexpr int kTerms = kFp8 ? 2 : 1;               // B rows per (row, head): e4m3 split terms
  constexpr int kLoaderWarp = kProducers + kMmaWarps;
  constexpr int kEpiWarp0 = kLoaderWarp + 1;           // two epilogue warpgroups take alternate tiles
  // named barriers: 2 + eg within epilogue warpgroup eg; kPrologueBar for the loader and the
  // epilogue warps filling the first group's queries together
  constexpr int kPrologueBar = 6, kPrologueThreads = 32 * 9;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // carve-up (uniform across the CTA): B buffers sized for the group, then scales, then keys
  const int n_cap = 32 * kTerms * a.rows_per_group;                // D buffer width (columns)
  const int row_bytes = kFp8 ? 128 : 256;                           // one query vector in B
  const int nB = n_cap * row_bytes <= kBBytes / 2 ? 2 : 1;         // B buffers (queries of one group each)
  const int b_bytes = (n_cap * row_bytes + 1023) / 1024 * 1024;
  // an even stage count: a stage's consecutive tiles then have the same parity, i.e. the same issuer
  constexpr int kScBytes = kFp8 ? kScRingBytes * (int)sizeof(ScaleT) / 4 : 0;   // bf16 keys carry no scales
  constexpr int kLoBytes = kI8 ? kConvWarps * 16384 : 0;           // int8 keys: one lo tile per converter
  const int kStages = kI8 ? kI8Stages
                          : min(kMaxStages, (kSmemBytes - 1024 - nB * b_bytes - kScBytes) / kStageBytes) & ~1;
  uint8_t* sB = smem;
  ScaleT* sScale = reinterpret_cast<ScaleT*>(smem + nB * b_bytes);  // [kScStages][128], 8-bit keys only
  uint8_t* sRing = smem + nB * b_bytes + kScBytes;
  uint8_t* sLo = sRing + kStages * kStageBytes;                      // int8 keys: [kConvWarps][16 KB]
  if (kI8 && (a.rows_per_group > kI8MaxRows || 1024 + nB * b_bytes + kScBytes + kStages * kStageBytes + kLoBytes >
                                                   kSmemBytes)) {
    if (threadIdx.x == 0) atomicOr(a.err, kErrConfig);            // the host never launches this shape
    return;
  }

  __shared__ uint64_t st_full[kMaxStages], st_empty[kMaxStages], sc_full[kScStages], sc_empty[kScStages];
  __shared__ uint64_t d_full[4], d_empty[4], b_full[2], b_empty[2];
  __shared__ uint64_t mma_done[kMmaWarps];
  __shared__ uint64_t cv_full[kI8 ? kMaxStages : 1], lo_empty[kI8 ? kConvWarps : 1];   // int8 keys only
  __shared__ __align__(16) float wq_e[2][kMaxRows][32];   // each epilogue warpgroup's head weights for its group
  __shared__ int4 gcache[kGroupCache];
  __shared__ int tcache[kGroupCache + 1];
  __shared__ uint32_t tmem_base;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t box_bytes = (uint32_t)a.box_rows * 128u;
  const int loads_per_tile = kTileKeys / a.box_rows;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&st_full[s], 1);
      mbar_init(&st_empty[s], 1);                  // the MMA's commit frees a key stage
    }
    for (int s = 0; s < kScStages; ++s) {
      mbar_init(&sc_full[s], 1);
      mbar_init(&sc_empty[s], 4);                  // the epilogue frees a scale slot once it has read it
    }
    for (int b = 0; b < 4; ++b) {
      mbar_init(&d_full[b], 1);
      mbar_init(&d_empty[b], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&b_full[b], 1);
      mbar_init(&b_empty[b], kMmaWarps);         // every issuer commits when it leaves a group
    }
    for (int m = 0; m < kMmaWarps; ++m) mbar_init(&mma_done[m], 1);
    if (kI8) {
      for (int s = 0; s < kStages; ++s) mbar_init(&cv_full[s], 1);   // its converter, once converted
      for (int c = 0; c < kConvWarps; ++c) mbar_init(&lo_empty[c], 1);   // the MMA's commit frees a lo tile
    }
    fence_mbar_init();
  }
  if (warp == kProducers) {
    tmem_alloc(&tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&key_map);
  // the group table and every input are complete past this point (programmatic dependent launch)
  pdl_wait();
  pdl_trigger();
  const int ngroups = a.counts[0], total_tiles = a.counts[1];
  const int tau0 = (int)(((int64_t)blockIdx.x * total_tiles) / gridDim.x);
  const int tau1 = (int)(((int64_t)(blockIdx.x + 1) * total_tiles) / gridDim.x);
  for (int g = threadIdx.x; g <= kGroupCache; g += blockDim.x) {
    if (g < kGroupCache) gcache[g] = g < ngroups ? a.groups[g] : make_int4(0, 0, 0, 0);
    tcache[g] = g <= ngroups ? a.tile_start[g] : total_tiles;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const int DD = min(4, 512 / n_cap);                               // D ring depth

  // Barriers are waited on by phase parity, so every waiter must be at most one phase behind the
  // barrier it waits on.  Each stage is always refilled by the same producer warp (stage % nprod),
  // which waited for that stage's previous release itself; each stage's consumers are one issuer
  // (tile parity, stages even) that waits on its tiles in order; the D ring (depth 4 or 2) and the
  // scale ring (16) are used by one epilogue warpgroup per parity, also in order.
  const int nprod = min(kProducers, kStages);
  if (warp < kProducers) {
    // ------------------------------------------------------------------ producers (tiles round-robin)
    // Each warp keeps a register window of 32 page ids (one per lane) and loads the next window
    // ahead of use, so page-table reads never sit between a free stage and its copy.
    // scale rows are bulk-copied when a sub-box's scales make 16 bytes (4 fp32 or 8 binary16)
    const bool bulk_scales = kFp8 && a.box_rows * (int)sizeof(ScaleT) >= 16;
    const ScaleT* key_scales = reinterpret_cast<const ScaleT*>(a.key_scales);
    const uint32_t key_tx = (kFp8 ? 1u : 2u) * box_bytes;
    const bool windowed = loads_per_tile <= 32;
    TileCursor cur;
    cursor_init(cur, a, gcache, tcache, ngroups, tau0, tau1);
    // keys read by one row group only are evicted first (the score block stays in L2 for the top-k);
    // keys that a request's other row groups read again keep their normal priority
    const uint64_t key_policy = groups_share_keys ? l2_evict_normal() : l2_evict_first();
    int win_base = -1, win_req = -1, win_page = -1, nxt_page = -1;
    int last_tile = -1;
    // ring positions of tile i, stepped once per tile (no division on the issue path)
    int s = 0, n = 0, sci = 0, scn = 0;
    for (int i = 0; warp < nprod && cur.valid();
         ++i, cursor_next(cur, a, gcache, tcache), s = s + 1 == kStages ? 0 : s + 1, n += s == 0,
             sci = (sci + 1) & (kScStages - 1), scn += sci == 0) {
      if (s % nprod != warp) continue;
      const int req = cur.G.x, pos_last = cur.G.w + cur.G.z - 1;
      const int32_t* bt = a.m.block_table + (int64_t)req * a.m.block_table_stride;
      const int k0 = cur.t * kTileKeys;
      const int lp_first = k0 >> a.log2_page;
      if (windowed) {
        const int lp_last = (k0 + kTileKeys - 1) >> a.log2_page;
        if (req != win_req || lp_first < win_base || lp_last >= win_base + 64) {
          win_req = req;
          win_base = lp_first;
          const int l0 = win_base + lane, l1 = win_base + 32 + lane;
          win_page = l0 < a.m.block_table_stride ? bt[l0] : -1;
          nxt_page = l1 < a.m.block_table_stride ? bt[l1] : -1;
        } else if (lp_last >= win_base + 32) {
          // slide by one window: the next one was loaded a window ago
          win_base += 32;
          win_page = nxt_page;
          const int l1 = win_base + 32 + lane;
          nxt_page = l1 < a.m.block_table_stride ? bt[l1] : -1;
        }
      }
      // the next window is read only by tiles that reach into it (a warp-uniform test), so a window
      // that was just requested is not waited for by the tile that requested it
      const bool reach_next = windowed && (((k0 + kTileKeys - 1) >> a.log2_page) >= win_base + 32);
      auto page_of = [&](int lp) -> int {      // called by all 32 lanes together
        if (windowed) {
          const int off = lp - win_base;
          const int v0 = __shfl_sync(0xffffffffu, win_page, off & 31);
          int v1 = -1;
          if (reach_next) v1 = __shfl_sync(0xffffffffu, nxt_page, off & 31);
          if (lp >= a.m.block_table_stride) return -1;
          return off < 32 ? v0 : v1;
        }
        return lp < a.m.block_table_stride ? bt[lp] : -1;
      };
      if (n > 0 && !mbar_wait(&st_empty[s], (n - 1) & 1, a.err, kErrMmaTimeout, kPolls)) break;
      if (kFp8 && scn > 0 && !mbar_wait(&sc_empty[sci], (scn - 1) & 1, a.err, kErrMmaTimeout, kPolls)) break;
      uint8_t* stage = sRing + s * kStageBytes;
      ScaleT* sc = sScale + sci * kTileKeys;
      // sub-box j holds keys k0 + j*box_rows ..; it is loaded when it starts at a visible key of a valid page
      uint32_t nvalid = 0;
      int my_page[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        my_page[q] = -1;
        const int j0 = 32 * q;
        if (j0 < loads_per_tile) {
          const int j = j0 + lane;
          const int key = k0 + j * a.box_rows;
          const int page = page_of(key >> a.log2_page);     // every lane takes part in the shuffles
          bool v = false;
          if (j < loads_per_tile && key <= pos_last) {
            v = page >= 0 && page < a.num_pages;
            if (!v) atomicOr(a.err, kErrBadPage);
          }
          my_page[q] = v ? page : -1;
          nvalid += __popc(__ballot_sync(0xffffffffu, v));
        }
      }
      if (kFp8 && !bulk_scales) {        // small pages (under 16 bytes of scales): scales through registers
        for (int k = lane; k < kTileKeys; k += 32) {
          const int key = k0 + k;
          const int lp = key >> a.log2_page;
          ScaleT v = 0;
          if (key <= pos_last && lp < a.m.block_table_stride) {
            const int page = bt[lp];
            if (page >= 0 && page < a.num_pages)
              v = key_scales[((int64_t)page << a.log2_page) + (key & ((1 << a.log2_page) - 1))];
          }
          sc[k] = v;
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&st_full[s], nvalid * key_tx);
        if (kFp8)
          mbar_arrive_expect_tx(&sc_full[sci], bulk_scales ? nvalid * (uint32_t)a.box_rows * (uint32_t)sizeof(ScaleT) : 0u);
      }
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = 32 * q + lane;
        const int page = my_page[q];
        if (page < 0) continue;
        const int key = k0 + j * a.box_rows;
        const int y = (page << a.log2_page) + (key & ((1 << a.log2_page) - 1));
        tma_load_2d_hint(stage + j * box_bytes, &key_map, 0, y, &st_full[s], key_policy);
        if (!kFp8) tma_load_2d_hint(stage + 16384 + j * box_bytes, &key_map, 64, y, &st_full[s], key_policy);
        if (bulk_scales)
          bulk_load(sc + j * a.box_rows, key_scales + y, (uint32_t)a.box_rows * (uint32_t)sizeof(ScaleT), &sc_full[sci]);
      }
      last_tile = i;
    }
    // drain: no copy of this warp may still be in flight at exit
    if (last_tile >= 0) {
      mbar_wait(&st_full[last_tile % kStages], (last_tile / kStages) & 1, a.err, kErrTmaTimeout, kPolls);
      if (kFp8) mbar_wait(&sc_full[last_tile % kScStages], (last_tile / kScStages) & 1, a.err, kErrTmaTimeout, kPolls);
    }
  } else if (warp < kLoaderWarp) {
    // ------------------------------------------------------------------ MMA issuers: warp m takes tiles i % 2 == m
    // (one issuing thread cannot keep up with HBM at one small MMA chain per tile); each walks every
    // tile to keep the group and ring positions, and commits its own barriers
    const int mw = warp - kProducers;
    if (lane == 0) {
      TileCursor cur;
      cursor_init(cur, a, gcache, tcache, ngroups, tau0, tau1);
      int gcount = 0;
      bool ok = true, new_group = true;
      uint32_t b_addr = 0, idesc = 0;
      int N = 0, ub = 0;
      int s = 0, n = 0, db = 0, nd = 0, li = 0;    // li: lo tile of tile i (int8 keys), i % kConvWarps
      for (int i = 0; cur.valid() && ok; ++i) {
        if (new_group) {
          if (i > 0) {
            mma_commit(&b_empty[ub]);
            ++gcount;
          }
          N = 32 * kTerms * cur.G.z;
          idesc = kFp8 ? idesc_e4m3(128, N) : idesc_f16(128, N, true, true, false, false);
          ub = gcount % nB;
          if (!mbar_wait(&b_full[ub], (gcount / nB) & 1, a.err, kErrMmaTimeout, kPolls)) { ok = false; break; }
          b_addr = smem_u32(sB + ub * b_bytes);
        }
        if ((i & 1) == mw) {
          // int8 tiles are ready once their converter has split them.  A suspending wait: an issuer
          // that polls takes issue slots from the epilogue warps of its SM sub-partition (measured 5 %
          // slower in decode)
          if (!mbar_wait(kI8 ? &cv_full[s] : &st_full[s], n & 1, a.err, kErrTmaTimeout, kPolls)) { ok = false; break; }
          if (nd > 0 && !mbar_wait(&d_empty[db], (nd - 1) & 1, a.err, kErrMmaTimeout, kPolls)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + db * (uint32_t)n_cap;
          const uint32_t stage = smem_u32(sRing + s * kStageBytes);
          if (kFp8) {
            // one descriptor per operand and tile; K steps of 32 bytes advance the start address field
            const uint64_t da = smem_desc(stage, 16, 1024, kSwizzle128B), dbq = smem_desc(b_addr, 16, 1024, kSwizzle128B);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) mma_ss_f8(d, da + (uint64_t)(2 * kk), dbq + (uint64_t)(2 * kk), idesc, kk > 0);
            if (kI8) {        // the lo terms of int8 keys into the same accumulators
              const uint64_t dl = smem_desc(smem_u32(sLo + li * 16384), 16, 1024, kSwizzle128B);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) mma_ss_f8(d, dl + (uint64_t)(2 * kk), dbq + (uint64_t)(2 * kk), idesc, true);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(d, smem_desc(stage + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024, kSwizzle128B),
                     smem_desc(b_addr + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024, kSwizzle128B), idesc, kk > 0);
          }
          mma_commit(&d_full[db]);
          mma_commit(&st_empty[s]);
          if (kI8) mma_commit(&lo_empty[li]);
        }
        if (++s == kStages) { s = 0; ++n; }
        if (++db == DD) { db = 0; ++nd; }
        if (++li == kConvWarps) li = 0;
        new_group = cursor_next(cur, a, gcache, tcache);
      }
      mma_commit(&mma_done[mw]);
      mbar_wait(&mma_done[mw], 0, a.err, kErrMmaTimeout, kPolls);
    }
  } else if (warp == kLoaderWarp) {
    // ------------------------------------------------------------------ B loader: each group's queries
    TileCursor cur;
    cursor_init(cur, a, gcache, tcache, ngroups, tau0, tau1);
    int gcount = 0;
    bool new_group = true;
    for (int i = 0; cur.valid(); ++i) {
      if (new_group) {
        const int ub = gcount % nB;
        uint8_t* bbuf = sB + ub * b_bytes;
        if (gcount >= nB && !mbar_wait(&b_empty[ub], (gcount / nB - 1) & 1, a.err, kErrMmaTimeout, kPolls)) break;
        // the CTA's first group is filled together with the epilogue warps, idle until its first tile
        fill_group_queries<kFp8>(a, cur.G, bbuf, lane, gcount == 0 ? kPrologueThreads : 32);
        fence_proxy_async_smem();
        if (gcount == 0) named_bar_sync(kPrologueBar, kPrologueThreads);
        __syncwarp();
        if (lane == 0) mbar_arrive(&b_full[ub]);
        ++gcount;
      }
      new_group = cursor_next(cur, a, gcache, tcache);
    }
  } else if (kI8 && warp >= kEpiWarp0 + 8) {
    // ------------------------------------------------------------------ converters (int8 keys): tile i by warp i % 3
    // Stage s = i % 6 is always converted by warp s % 3, which waits on that stage's tiles in order; its
    // lo tile is rewritten only after the MMA of the warp's previous tile has committed.  A tile's
    // sub-boxes that were not loaded hold stale codes: any byte splits into finite terms, and the
    // epilogue masks those keys.
    const int cw = warp - (kEpiWarp0 + 8);
    const int ntiles = tau1 - tau0;
    int s = cw, n = 0;
    for (int i = cw, k = 0; i < ntiles; i += kConvWarps, ++k) {
      if (!mbar_wait(&st_full[s], n & 1, a.err, kErrTmaTimeout, kPolls)) break;
      if (k > 0 && !mbar_wait(&lo_empty[cw], (k - 1) & 1, a.err, kErrMmaTimeout, kPolls)) break;
      uint4* hi = reinterpret_cast<uint4*>(sRing + s * kStageBytes);
      uint4* lo = reinterpret_cast<uint4*>(sLo + cw * 16384);
#pragma unroll 2
      for (int c = lane; c < kStageBytes / 16; c += 32) {
        const uint4 v = hi[c];
        uint4 h, l;
        split_int8_e4m3(v.x, h.x, l.x);
        split_int8_e4m3(v.y, h.y, l.y);
        split_int8_e4m3(v.z, h.z, l.z);
        split_int8_e4m3(v.w, h.w, l.w);
        hi[c] = h;
        lo[c] = l;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&cv_full[s]);
      s += kConvWarps;
      if (s >= kStages) { s -= kStages; ++n; }
    }
  } else {
    // ------------------------------------------------------------------ epilogues: ReLU . w, scale, mask, store
    const int eg = (warp - kEpiWarp0) >> 2;          // warpgroup 0 takes even tiles, 1 odd tiles
    const int quarter = warp & 3;
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    const int key_local = 32 * quarter + lane;
    const int et = threadIdx.x - 32 * (kEpiWarp0 + 4 * eg);   // 0..127 within the warpgroup
    TileCursor cur;
    cursor_init(cur, a, gcache, tcache, ngroups, tau0, tau1);
    if (cur.valid()) {
      // the first group's queries, with the loader warp (B buffer 0; the loader signals it)
      fill_group_queries<kFp8>(a, cur.G, sB, threadIdx.x - 32 * kLoaderWarp, kPrologueThreads);
      fence_proxy_async_smem();
      named_bar_sync(kPrologueBar, kPrologueThreads);
    }
    bool new_group = true;
    int db = 0, nd = 0, sci = 0, scn = 0;
    for (int i = 0; cur.valid();
         ++i, db = db + 1 == DD ? 0 : db + 1, nd += db == 0, sci = (sci + 1) & (kScStages - 1), scn += sci == 0) {
      if (new_group) {
        named_bar_sync(2 + eg, 128);                 // the previous group's weights are no longer read
        for (int p = et; p < 32 * cur.G.z; p += 128) {
          const int rr = p >> 5, h = p & 31;
          float wgt = a.w[(int64_t)(cur.G.y + rr) * kIndexHeads + h];
          if (kFp8) {
            uint4 raw[16];
            wgt = ldexpf(wgt, query_exponent(a, cur.G.y + rr, h, raw) - 7);
          }
          wq_e[eg][rr][h] = wgt;
        }
        named_bar_sync(2 + eg, 128);
      }
      if ((i & 1) == eg) {
        if (!mbar_wait(&d_full[db], nd & 1, a.err, kErrMmaTimeout, kPolls)) break;
        tc_fence_after();
        float score[kRowsMax];
#pragma unroll
        for (int rr = 0; rr < kRowsMax; ++rr) {
          score[rr] = 0.f;
          if (rr < cur.G.z) {
            uint32_t v[32];
            float acc[4] = {0.f, 0.f, 0.f, 0.f};     // four partial sums: a short dependency chain
            const float4* wr = reinterpret_cast<const float4*>(wq_e[eg][rr]);
            const uint32_t col = tmem + lane_base + db * (uint32_t)n_cap + 32 * kTerms * rr;
            tmem_ld32(col, v);
            if (kFp8) {
              uint32_t lo[32];
              tmem_ld32(col + 32, lo);
              tmem_wait_ld();
#pragma unroll
              for (int h4 = 0; h4 < 8; ++h4) {
                const float4 w4 = wr[h4];
                const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const int h = 4 * h4 + j;
                  acc[j] = fmaf(wv[j], fmaxf(fmaf(__uint_as_float(lo[h]), 0.0625f, __uint_as_float(v[h])), 0.f), acc[j]);
                }
              }
            } else {
              tmem_wait_ld();
#pragma unroll
              for (int h4 = 0; h4 < 8; ++h4) {
                const float4 w4 = wr[h4];
                const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[j] = fmaf(wv[j], fmaxf(__uint_as_float(v[4 * h4 + j]), 0.f), acc[j]);
              }
            }
            score[rr] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&d_empty[db]);
        if (kFp8) {
          // the tile's key scales sit in their own ring slot, refilled only after this read (reading
          // them before the accumulators' wait measured slower)
          if (!mbar_wait(&sc_full[sci], scn & 1, a.err, kErrTmaTimeout, kPolls)) break;
          const float ks = scale_value(sScale[sci * kTileKeys + key_local]);
          __syncwarp();
          if (lane == 0) mbar_arrive(&sc_empty[sci]);
#pragma unroll
          for (int rr = 0; rr < kRowsMax; ++rr) score[rr] *= ks;
        }
        const int skey = cur.t * kTileKeys + key_local;
        if (a.page_log2 < 0) {
          if (skey < a.max_seq_len) {
#pragma unroll
            for (int rr = 0; rr < kRowsMax; ++rr)
              if (rr < cur.G.z)
                a.scores[(int64_t)(cur.G.y + rr - a.row0) * a.stride + skey] = skey <= cur.G.w + rr ? score[rr] : -INFINITY;
          }
        } else {
          // page mode ("Make the sparsity unit match the memory unit"; "Stream indexer scores over live
          // context"): the largest visible score (the mask comes first) of each unit of U = min(P, 32) keys,
          // reduced within the warp.  Pages of up to 32 keys are whole units; larger pages (at most 128
          // keys: one tile) are pooled from their units by a small kernel afterwards, since a page then
          // spans the keys of several warps and a barrier per tile to combine them costs more.
          const int lu = a.page_log2 < 5 ? a.page_log2 : 5, U = 1 << lu;
#pragma unroll
          for (int rr = 0; rr < kRowsMax; ++rr) {
            if (rr < cur.G.z) {                          // uniform across the warpgroup
              float v = skey <= cur.G.w + rr ? score[rr] : -INFINITY;
              for (int o = 1; o < U; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
              const int unit = skey >> lu;
              if ((lane & (U - 1)) == 0 && unit < a.max_pages)
                a.scores[(int64_t)(cur.G.y + rr - a.row0) * a.stride + unit] = v;
            }
          }
        }
      }
      new_group = cursor_next(cur, a, gcache, tcache);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kProducers) tmem_dealloc(tmem, kTmemCols);
}

// Row groups of rows [row0, row0 + nrows): consecutive rows of one request, at most `rg` per group,
// each with its count of 128-key tiles, and the exclusive prefix of those counts (one CTA).
__global__ void __launch_bounds__(1024) indexer_groups_kernel(RowMeta m, int row0, int nrows, int rg, int4* groups,
                                                              int32_t* tile_start, int32_t* counts, uint32_t* status) {
  __shared__ int carry, warp_tot[33];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  pdl_wait();
  pdl_trigger();
  // the workspace header starts clear: no call-wide bits yet (the indexer kernels set them only after
  // their own wait on this grid; status is null after the call's first row block) and no per-CTA words
  if (status != nullptr && tid == 0) {
    status[0] = 0u;
    status[1] = 0u;
  }
  // number of groups: in decode one per row; otherwise walk the requests
  int ngroups = 0;
  if (m.query_start_loc == nullptr) {
    ngroups = nrows;
    for (int g = tid; g < nrows; g += blockDim.x) {
      const int r = row0 + g;
      groups[g] = make_int4(r, r, 1, m.seq_lens[r] - 1);
    }
  } else {
    if (tid == 0) {
      int g = 0;
      for (int b = 0; b < m.num_requests; ++b) {
        const int q0 = m.query_start_loc[b], q1 = m.query_start_loc[b + 1];
        const int lo = max(q0, row0), hi = min(q1, row0 + nrows);
        for (int r = lo; r < hi; r += rg) {
          groups[g] = make_int4(b, r, min(rg, hi - r), m.seq_lens[b] - (q1 - q0) + (r - q0));
          ++g;
        }
      }
      carry = g;
    }
    __syncthreads();
    ngroups = carry;
  }
  __syncthreads();
  if (tid == 0) carry = 0;
  __syncthreads();
  // tiles per group and their exclusive prefix, 1024 groups per pass
  for (int base = 0; base < ngroups; base += blockDim.x) {
    const int g = base + tid;
    int tiles = 0;
    if (g < ngroups) {
      const int4 G = groups[g];
      const int pos_last = G.w + G.z - 1;
      tiles = pos_last < 0 ? 0 : pos_last / idx::kTileKeys + 1;
    }
    int inc = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane == 31) warp_tot[wid] = inc;
    __syncthreads();
    if (wid == 0) {
      const int x = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
      int xi = x;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, xi, o);
        if (lane >= o) xi += t;
      }
      warp_tot[lane] = xi - x;
      if (lane == 31) warp_tot[32] = xi;
    }
    __syncthreads();
    if (g < ngroups) tile_start[g] = carry + warp_tot[wid] + inc - tiles;
    __syncthreads();
    if (tid == 0) carry += warp_tot[32];
    __syncthreads();
  }
  if (tid == 0) {
    tile_start[ngroups] = carry;
    counts[0] = ngroups;
    counts[1] = carry;
  }
}

// -inf for the positions of a caller-visible score row that no tile covered (s beyond the row's last tile).
// -inf beyond what the indexer wrote for each row (its last 128-key tile), in units of 2^unit_log2
// keys (1: token scores; page mode: the units of at most 32 keys it pools), up to max_units columns.
__global__ void indexer_fill_tail_kernel(RowMeta m, int row0, float* scores, int64_t stride, int max_units,
                                         int unit_log2) {
  pdl_wait();
  pdl_trigger();
  const int r = row0 + blockIdx.y;
  int b, pos;
  row_info(m, r, b, pos);
  const int start = pos < 0 ? 0 : ((pos / 128 + 1) * 128) >> unit_log2;
  for (int s = start + blockIdx.x * blockDim.x + threadIdx.x; s < max_units; s += gridDim.x * blockDim.x)
    scores[(int64_t)blockIdx.y * stride + s] = -INFINITY;
}

// Page scores of pages larger than 32 keys from the indexer's 32-key unit maxima:
//   pages[r][p] = max_j units[r][p * pool + j] for the row's pages p <= pos / P, -inf for p < max_pages beyond.
__global__ void __launch_bounds__(256) page_pool_kernel(RowMeta m, int row0, const float* __restrict__ units,
                                                        int64_t unit_stride, int pool_log2, int page_log2,
                                                        float* __restrict__ pages, int64_t page_stride, int max_pages) {
  pdl_wait();
  pdl_trigger();
  const int r = row0 + blockIdx.y;
  int b, pos;
  row_info(m, r, b, pos);
  const int n = pos >= 0 ? (pos >> page_log2) + 1 : 0;
  const float* u = units + (int64_t)blockIdx.y * unit_stride;
  float* out = pages + (int64_t)blockIdx.y * page_stride;
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < max_pages; p += gridDim.x * blockDim.x) {
    float v = -INFINITY;
    if (p < n)
      for (int j = 0; j < (1 << pool_log2); ++j) v = fmaxf(v, u[((int64_t)p << pool_log2) + j]);
    out[p] = v;
  }
}

cudaError_t launch_page_pool(const RowMeta& m, int row0, int nrows, const float* units, int64_t unit_stride,
                             int page_log2, float* pages, int64_t page_stride, int max_pages, cudaStream_t s) {
  dim3 grid((max_pages + 255) / 256 < 16 ? (max_pages + 255) / 256 : 16, nrows);
  cudaError_t e = launch_pdl(page_pool_kernel, grid, dim3(256), 0, s, m, row0, units, unit_stride, page_log2 - 5,
                             page_log2, pages, page_stride, max_pages);
  count_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {
struct KeyMapCache {
  std::mutex mu;
  const void* ptr[8] = {};
  uint64_t rows[8] = {};
  int fmt[8] = {};
  uint32_t box[8] = {};
  CUtensorMap map[8];
  int next = 0;
  bool get(const void* p, uint64_t nrows, int format, uint32_t box_rows, CUtensorMap* out) {
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < 8; ++i)
      if (ptr[i] == p && p && rows[i] == nrows && fmt[i] == format && box[i] == box_rows) {
        *out = map[i];
        return true;
      }
    CUtensorMap m;
    const bool ok = format != DSA_KEY_BF16          // e4m3 and int8 keys: 128 bytes per key
                        ? encode_2d(&m, p, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kIndexDim, nrows, kIndexDim, 128, box_rows)
                        : encode_2d(&m, p, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kIndexDim, nrows, kIndexDim * 2, 64,
                                    box_rows);
    if (!ok) return false;
    ptr[next] = p;
    rows[next] = nrows;
    fmt[next] = format;
    box[next] = box_rows;
    map[next] = m;
    next = (next + 1) % 8;
    *out = m;
    return true;
  }
};
KeyMapCache g_key_maps;
}  // namespace

static int indexer_rows_per_group(const dsa_cache& c, bool decode) {
  if (decode) return 1;
  if (c.key_format == DSA_KEY_INT8) return idx::kI8MaxRows;
  return c.key_format == DSA_KEY_FP8_E4M3 ? 4 : idx::kMaxRows;
}

cudaError_t launch_indexer_scores(const dsa_cache& c, const RowMeta& m, int row0, int nrows, int max_seq_len,
                                  const void* q_idx, const float* w, float* scores, int64_t score_stride,
                                  bool fill_tail, int32_t* group_scratch, uint32_t* err, cudaStream_t s,
                                  int page_log2) {
  const int kind = c.key_format == DSA_KEY_FP8_E4M3 ? 1 : c.key_format == DSA_KEY_INT8 ? 2 : 0;
  const bool decode = m.query_start_loc == nullptr;
  static std::atomic<uint64_t> configured{0};
  const cudaError_t set = once_per_device(configured, [] {
    cudaError_t r = cudaFuncSetAttribute(indexer_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         idx::kSmemBytes);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(indexer_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, idx::kSmemBytes);
    return r != cudaSuccess ? r : cudaFuncSetAttribute(indexer_tc_kernel<0>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, idx::kSmemBytes);
  });
  if (set != cudaSuccess) return set;
  const uint32_t box_rows = (uint32_t)(c.page_size < idx::kTileKeys ? c.page_size : idx::kTileKeys);
  CUtensorMap map;
  if (!g_key_maps.get(c.index_keys, (uint64_t)c.num_pages * c.page_size, c.key_format, box_rows, &map))
    return cudaErrorInvalidValue;

  // group table: counts[4] | groups int4[nrows] | tile_start[nrows + 1]
  int32_t* counts = group_scratch;
  int4* groups = reinterpret_cast<int4*>(group_scratch + 4);
  int32_t* tile_start = group_scratch + 4 + 4 * nrows;
  const int rg = indexer_rows_per_group(c, decode);
  cudaError_t e = launch_pdl(indexer_groups_kernel, dim3(1), dim3(1024), 0, s, m, row0, nrows, rg, groups, tile_start,
                             counts, row0 == 0 ? err : (uint32_t*)nullptr);
  count_launches(1);
  if (e != cudaSuccess) return e;

  IdxArgs a;
  a.m = m;
  a.groups = groups;
  a.tile_start = tile_start;
  a.counts = counts;
  a.max_groups = nrows;
  a.row0 = row0;
  a.rows_per_group = rg;
  a.log2_page = ilog2(c.page_size);
  a.num_pages = c.num_pages;
  a.box_rows = (int)box_rows;
  a.key_scales = c.index_scales;
  a.q_idx = static_cast<const __nv_bfloat16*>(q_idx);
  a.w = w;
  a.scores = scores;
  a.stride = score_stride;
  a.max_seq_len = max_seq_len;
  a.page_log2 = page_log2;
  const int unit_log2 = page_log2 < 5 ? page_log2 : 5;
  a.max_pages = page_log2 >= 0 ? (max_seq_len + (1 << unit_log2) - 1) >> unit_log2 : 0;
  a.err = err;
  const int grid = device_sm_count();
  // more rows than row groups per request: some request's keys are read by several groups
  const int share = (int64_t)nrows > (int64_t)m.num_requests * rg ? 1 : 0;
  e = kind == 1   ? launch_pdl(indexer_tc_kernel<1>, dim3(grid), dim3(idx::kThreads), idx::kSmemBytes, s, map, a, share)
      : kind == 2 ? launch_pdl(indexer_tc_kernel<2>, dim3(grid), dim3(idx::kThreadsI8), idx::kSmemBytes, s, map, a, share)
                  : launch_pdl(indexer_tc_kernel<0>, dim3(grid), dim3(idx::kThreads), idx::kSmemBytes, s, map, a, share);
  count_launches(1);
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess || !fill_tail) return e;
  const int units = page_log2 >= 0 ? a.max_pages : max_seq_len;
  dim3 fgrid((units + 255) / 256 < 64 ? (units + 255) / 256 : 64, nrows);
  e = launch_pdl(indexer_fill_tail_kernel, fgrid, dim3(256), 0, s, m, row0, scores, score_stride, units,
                 page_log2 >= 0 ? unit_log2 : 0);
  count_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dsa
