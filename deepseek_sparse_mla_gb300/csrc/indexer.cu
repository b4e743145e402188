// Lightning-indexer scoring on tcgen05 tensor cores:
//   I(r, s) = sum_{h<32} w[r,h] * max(0, q_idx[r,h,:] . K[s,:])   for 0 <= s <= pos(r), -inf beyond
// ("vLLM Inference Path: GLM-5.2 as an Example", "DSA Indexer"; "Making GLM-5.2
// Sparse on TPUs", "Separate the indexer from the attention it controls").
//
// Rows are grouped by request (1 row in decode, up to 4 with e4m3 keys or 8
// with bf16 keys otherwise); every key read from HBM serves the whole group.
// One MMA computes D[key, (row, head)] for a tile of 128 keys:
//   M = 128 keys, N = 32 heads x rows, K = 128, fp32 accumulators in TMEM,
// and the epilogue applies ReLU, the head weights, the key's scale and the
// causal mask (masks precede any selection: "Making GLM-5.2 Sparse on TPUs",
// "Make the sparsity unit match the memory unit").
//
// Per CTA (persistent, one per SM, 192 threads):
//   warp 0     producer: looks up the key tile's pages and TMA-loads them into
//              a ring of shared-memory stages (8 x 16 KB e4m3, 4 x 32 KB bf16),
//              staging each key's fp32 scale beside it;
//   warp 1     MMA issuer;
//   warps 2-5  workers: per unit they load the group's queries into the B
//              operand (128-byte swizzled, K-major); for e4m3 keys they convert
//              each key row to f16 with cvt and store it straight into TMEM as
//              the A operand (the MMA then reads A from TMEM, B from shared
//              memory); and they run the epilogue of the previous tile.
// e4m3 keys need f16 operands on both sides (one MMA kind per instruction):
// every e4m3 value is exact in f16, and each (row, head) query vector is moved
// into f16 range by an exact power of two that is folded into its head weight.
#include <mutex>

#include "dsa_internal.cuh"
#include "sm100.cuh"
#include "tmap.cuh"

namespace dsa {
using namespace sm100;

namespace idx {
constexpr int kTileKeys = 128;
constexpr int kThreads = 192;
constexpr int kBBytes = 65536;                      // up to 256 (row, head) query vectors of 128 bf16/f16
constexpr int kRingBytes = 131072;                  // key stages
constexpr int kSmemBytes = kBBytes + kRingBytes + 8 * 512 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kPolls = 1u << 22;
constexpr int kMaxRows = 8;
constexpr int kGroupCache = 1024;                    // group descriptors staged in shared memory
}  // namespace idx

struct IdxArgs {
  RowMeta m;
  const int32_t* groups;         // [max_groups][3] = (request, first row, rows); nullptr in decode
  const int32_t* n_groups;       // device count of groups (nullptr in decode)
  int max_groups;
  int row0, nrows_block;         // rows this launch scores; scores row (r - row0)
  int block_tiles;               // key tiles per work unit
  int key_blocks;                // ceil(max_seq_len / (128 * block_tiles))
  int log2_page, num_pages, box_rows;
  const float* key_scales;       // e4m3 keys only
  const __nv_bfloat16* q_idx;
  const float* w;
  float* scores;
  int64_t stride;
  int max_seq_len;
  uint32_t* err;
};

struct GroupInfo {
  int req, row, nrows, pos_first;
};

__device__ __forceinline__ bool load_group_global(const IdxArgs& a, int g, GroupInfo& G) {
  if (a.groups == nullptr) {
    if (g >= a.nrows_block) return false;
    G.row = a.row0 + g;
    G.req = G.row;
    G.nrows = 1;
    G.pos_first = a.m.seq_lens[G.req] - 1;
    return true;
  }
  if (g >= *a.n_groups) return false;
  G.req = a.groups[3 * g];
  G.row = a.groups[3 * g + 1];
  G.nrows = a.groups[3 * g + 2];
  const int q0 = a.m.query_start_loc[G.req], q1 = a.m.query_start_loc[G.req + 1];
  G.pos_first = a.m.seq_lens[G.req] - (q1 - q0) + (G.row - q0);
  return true;
}

// Group g from the shared-memory copy (nrows == 0 marks a missing group) or from global memory.
__device__ __forceinline__ bool load_group(const IdxArgs& a, const int4* gcache, int g, GroupInfo& G) {
  if (g < idx::kGroupCache) {
    const int4 v = gcache[g];
    G.req = v.x;
    G.row = v.y;
    G.nrows = v.z;
    G.pos_first = v.w;
    return v.z > 0;
  }
  return load_group_global(a, g, G);
}

// Tiles [t_begin, t_end) of work unit u, or false when the unit has no visible key.
__device__ __forceinline__ bool unit_tiles(const IdxArgs& a, const int4* gcache, int u, GroupInfo& G, int& t_begin,
                                           int& t_end) {
  const int g = u / a.key_blocks, kb = u - g * a.key_blocks;
  if (!load_group(a, gcache, g, G)) return false;
  const int pos_last = G.pos_first + G.nrows - 1;
  if (pos_last < 0) return false;
  t_begin = kb * a.block_tiles;
  const int tiles_needed = pos_last / idx::kTileKeys + 1;
  t_end = min(t_begin + a.block_tiles, tiles_needed);
  return t_begin < t_end;
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

template <bool kFp8>
__global__ void __launch_bounds__(idx::kThreads, 1)
    indexer_tc_kernel(const __grid_constant__ CUtensorMap key_map, const IdxArgs a) {
  using namespace idx;
  constexpr int kStages = kFp8 ? 8 : 4;
  constexpr int kStageBytes = kFp8 ? 16384 : 32768;
  constexpr int kRowsMax = kFp8 ? 4 : 8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sB = smem;
  uint8_t* sRing = smem + kBBytes;
  float* sScale = reinterpret_cast<float*>(sRing + kRingBytes);        // [kStages][128] (e4m3 keys)

  __shared__ uint64_t st_full[kStages], st_empty[kStages];
  __shared__ uint64_t a_full[2], a_empty[2], d_full[2], d_empty[2], b_full, b_empty, mma_done;
  __shared__ float wq[2][kMaxRows][32];     // head weights (times the query prescale) per unit parity
  __shared__ int4 gcache[kGroupCache];
  __shared__ uint32_t tmem_base;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = a.max_groups * a.key_blocks;
  const uint32_t box_bytes = (uint32_t)a.box_rows * 128u;
  const int loads_per_tile = kTileKeys / a.box_rows;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&st_full[s], 1);
      mbar_init(&st_empty[s], kFp8 ? 4 : 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&a_full[b], 4);
      mbar_init(&a_empty[b], 1);
      mbar_init(&d_full[b], 1);
      mbar_init(&d_empty[b], 4);
    }
    mbar_init(&b_full, 1);
    mbar_init(&b_empty, 1);
    mbar_init(&mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&key_map);
  for (int g = threadIdx.x; g < kGroupCache; g += blockDim.x) {
    GroupInfo G;
    int4 v = make_int4(0, 0, 0, 0);
    if (g < a.max_groups && load_group_global(a, g, G)) v = make_int4(G.req, G.row, G.nrows, G.pos_first);
    gcache[g] = v;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  // TMEM: e4m3 -> A buffers at columns 0 / 64 and D buffers at 128 / 256; bf16 -> D at 0 / 256
  const uint32_t colA = 0;
  const uint32_t colD = kFp8 ? 128u : 0u, strideD = kFp8 ? 128u : 256u;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    int tiles = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      GroupInfo G;
      int tb, te;
      if (!unit_tiles(a, gcache, u, G, tb, te)) continue;
      const int pos_last = G.pos_first + G.nrows - 1;
      const int32_t* bt = a.m.block_table + (int64_t)G.req * a.m.block_table_stride;
      for (int t = tb; t < te; ++t, ++tiles) {
        const int s = tiles % kStages, n = tiles / kStages;
        if (n > 0 && !mbar_wait(&st_empty[s], (n - 1) & 1, a.err, kErrMmaTimeout, kPolls)) { ok = false; break; }
        const int k0 = t * kTileKeys;
        uint8_t* stage = sRing + s * kStageBytes;
        // page of each sub-box; a box past the row's last key, or on a bad page, is not loaded
        uint32_t nvalid = 0;
        for (int i0 = 0; i0 < loads_per_tile; i0 += 32) {
          const int i = i0 + lane;
          bool v = false;
          if (i < loads_per_tile) {
            const int key = k0 + i * a.box_rows;
            const int lp = key >> a.log2_page;
            if (key <= pos_last && lp < a.m.block_table_stride) {
              const int page = bt[lp];
              v = page >= 0 && page < a.num_pages;
              if (!v) atomicOr(a.err, kErrBadPage);
            }
          }
          nvalid += __popc(__ballot_sync(0xffffffffu, v));
        }
        if (kFp8) {
          float* sc = sScale + s * kTileKeys;
          for (int k = lane; k < kTileKeys; k += 32) {
            const int key = k0 + k;
            const int lp = key >> a.log2_page;
            float v = 0.f;
            if (key <= pos_last && lp < a.m.block_table_stride) {
              const int page = bt[lp];
              if (page >= 0 && page < a.num_pages)
                v = a.key_scales[((int64_t)page << a.log2_page) + (key & ((1 << a.log2_page) - 1))];
            }
            sc[k] = v;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(&st_full[s], nvalid * box_bytes * (kFp8 ? 1u : 2u));
        __syncwarp();
        for (int i = lane; i < loads_per_tile; i += 32) {
          const int key = k0 + i * a.box_rows;
          const int lp = key >> a.log2_page;
          if (key > pos_last || lp >= a.m.block_table_stride) continue;
          const int page = bt[lp];
          if (page < 0 || page >= a.num_pages) continue;
          const int y = (page << a.log2_page) + (key & ((1 << a.log2_page) - 1));
          tma_load_2d(stage + i * box_bytes, &key_map, 0, y, &st_full[s]);
          if (!kFp8) tma_load_2d(stage + 16384 + i * box_bytes, &key_map, 64, y, &st_full[s]);
        }
      }
    }
    // drain: no copy may still be in flight at exit
    for (int s = 0; s < kStages; ++s) {
      const int uses = tiles / kStages + (s < tiles % kStages ? 1 : 0);
      if (uses > 0) mbar_wait(&st_full[s], (uses - 1) & 1, a.err, kErrTmaTimeout, kPolls);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int tiles = 0, unit_count = 0;
      bool ok = true;
      const uint32_t b_addr = smem_u32(sB);
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        GroupInfo G;
        int tb, te;
        if (!unit_tiles(a, gcache, u, G, tb, te)) continue;
        const int N = 32 * G.nrows;
        const uint32_t idesc = idesc_f16(128, N, !kFp8, !kFp8, false, false);
        if (!mbar_wait(&b_full, unit_count & 1, a.err, kErrMmaTimeout, kPolls)) { ok = false; break; }
        for (int t = tb; t < te; ++t, ++tiles) {
          const int s = tiles % kStages, n = tiles / kStages, ab = tiles & 1, nb = tiles >> 1;
          if (kFp8) {
            if (!mbar_wait(&a_full[ab], nb & 1, a.err, kErrMmaTimeout, kPolls)) { ok = false; break; }
          } else {
            if (!mbar_wait(&st_full[s], n & 1, a.err, kErrTmaTimeout, kPolls)) { ok = false; break; }
          }
          if (nb > 0 && !mbar_wait(&d_empty[ab], (nb - 1) & 1, a.err, kErrMmaTimeout, kPolls)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + colD + ab * strideD;
          const uint32_t stage = smem_u32(sRing + s * kStageBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t bd = smem_desc(b_addr + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024, kSwizzle128B);
            if (kFp8) {
              mma_ts(d, tmem + colA + 64 * ab + 8 * kk, bd, idesc, kk > 0);
            } else {
              const uint64_t ad = smem_desc(stage + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024, kSwizzle128B);
              mma_ss(d, ad, bd, idesc, kk > 0);
            }
          }
          mma_commit(&d_full[ab]);
          if (kFp8) mma_commit(&a_empty[ab]);
          else mma_commit(&st_empty[s]);
        }
        if (!ok) break;
        mma_commit(&b_empty);
        ++unit_count;
      }
      mma_commit(&mma_done);
      mbar_wait(&mma_done, 0, a.err, kErrMmaTimeout, kPolls);
    }
  } else {
    // ------------------------------------------------------------------ workers: B operand, conversion, epilogue
    const int quarter = warp & 3;
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    const int key_local = 32 * quarter + lane;       // TMEM lane = key within the tile
    const int wt = threadIdx.x - 64;                 // 0..127
    int tiles = 0, unit_count = 0;
    bool ok = true;
    // epilogue state of the tile converted last
    bool have_prev = false;
    int prev_tile = 0, prev_k0 = 0, prev_row = 0, prev_rows = 0, prev_pos = 0, prev_par = 0;
    float prev_scale = 1.f, cur_scale = 1.f;

    auto epilogue = [&](int tile, int k0, int row, int rows, int pos_first, int par, float kscale) -> bool {
      const int ab = tile & 1, nb = tile >> 1;
      if (!mbar_wait(&d_full[ab], nb & 1, a.err, kErrMmaTimeout, kPolls)) return false;
      tc_fence_after();
      float score[kRowsMax];
#pragma unroll
      for (int rr = 0; rr < kRowsMax; ++rr) {
        score[rr] = 0.f;
        if (rr < rows) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + colD + ab * strideD + 32 * rr, v);
          tmem_wait_ld();
          float acc = 0.f;
#pragma unroll
          for (int h = 0; h < 32; ++h) acc = fmaf(wq[par][rr][h], fmaxf(__uint_as_float(v[h]), 0.f), acc);
          score[rr] = acc * kscale;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&d_empty[ab]);
      const int s = k0 + key_local;
      if (s < a.max_seq_len) {
#pragma unroll
        for (int rr = 0; rr < kRowsMax; ++rr)
          if (rr < rows)
            a.scores[(int64_t)(row + rr - a.row0) * a.stride + s] = s <= pos_first + rr ? score[rr] : -INFINITY;
      }
      return true;
    };

    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      GroupInfo G;
      int tb, te;
      if (!unit_tiles(a, gcache, u, G, tb, te)) continue;
      const int par = unit_count & 1;
      const int N = 32 * G.nrows;
      // ---- B operand and head weights for this group (after the previous unit's MMAs are done)
      if (unit_count > 0 && !mbar_wait(&b_empty, (unit_count - 1) & 1, a.err, kErrMmaTimeout, kPolls)) break;
      for (int p = wt; p < N; p += 128) {
        const int rr = p >> 5, h = p & 31;
        const __nv_bfloat16* qv = a.q_idx + ((int64_t)(G.row + rr) * kIndexHeads + h) * kIndexDim;
        float wgt = a.w[(int64_t)(G.row + rr) * kIndexHeads + h];
        uint4 raw[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) raw[c] = reinterpret_cast<const uint4*>(qv)[c];
        if (kFp8) {
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
          // exact power-of-two move into f16 range: max |q'| in [2^13, 2^14)
          const int ex = amax > 0.f ? ilogbf(amax) : 0;
          const float up = ldexpf(1.f, 13 - ex);
          wgt = ldexpf(wgt, ex - 13);
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&raw[c]);
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(x[e]);
              const __half2 hv = __floats2half2_rn(f.x * up, f.y * up);
              o[e] = *reinterpret_cast<const uint32_t*>(&hv);
            }
            raw[c] = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
#pragma unroll
        for (int c = 0; c < 16; ++c)
          *reinterpret_cast<uint4*>(sB + (c >> 3) * (N * 128) + sw128_offset(p, c & 7)) = raw[c];
        wq[par][rr][h] = wgt;
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (wt == 0) mbar_arrive(&b_full);

      for (int t = tb; t < te; ++t, ++tiles) {
        const int s = tiles % kStages, n = tiles / kStages, ab = tiles & 1, nb = tiles >> 1;
        if (kFp8) {
          // ---- convert this tile's e4m3 keys into the TMEM A operand
          if (!mbar_wait(&st_full[s], n & 1, a.err, kErrTmaTimeout, kPolls)) { ok = false; break; }
          const uint8_t* stage = sRing + s * kStageBytes;
          uint4 raw[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) raw[c] = *reinterpret_cast<const uint4*>(stage + sw128_offset(key_local, c));
          cur_scale = sScale[s * kTileKeys + key_local];
          __syncwarp();
          if (lane == 0) mbar_arrive(&st_empty[s]);
          if (nb > 0 && !mbar_wait(&a_empty[ab], (nb - 1) & 1, a.err, kErrMmaTimeout, kPolls)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t o[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint4 v = raw[half * 4 + c];
              o[8 * c + 0] = e4m3x2_to_f16x2(v.x);
              o[8 * c + 1] = e4m3x2_to_f16x2(v.x >> 16);
              o[8 * c + 2] = e4m3x2_to_f16x2(v.y);
              o[8 * c + 3] = e4m3x2_to_f16x2(v.y >> 16);
              o[8 * c + 4] = e4m3x2_to_f16x2(v.z);
              o[8 * c + 5] = e4m3x2_to_f16x2(v.z >> 16);
              o[8 * c + 6] = e4m3x2_to_f16x2(v.w);
              o[8 * c + 7] = e4m3x2_to_f16x2(v.w >> 16);
            }
            tmem_st32(tmem + lane_base + colA + 64 * ab + 32 * half, o);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_full[ab]);
        }
        if (have_prev && !epilogue(prev_tile, prev_k0, prev_row, prev_rows, prev_pos, prev_par, prev_scale)) {
          ok = false;
          break;
        }
        have_prev = true;
        prev_tile = tiles;
        prev_k0 = t * kTileKeys;
        prev_row = G.row;
        prev_rows = G.nrows;
        prev_pos = G.pos_first;
        prev_par = par;
        prev_scale = kFp8 ? cur_scale : 1.f;
      }
      ++unit_count;
    }
    if (ok && have_prev) epilogue(prev_tile, prev_k0, prev_row, prev_rows, prev_pos, prev_par, prev_scale);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Row groups of one launch: consecutive rows of one request, at most `rg` per group.
__global__ void indexer_groups_kernel(RowMeta m, int row0, int nrows, int rg, int32_t* groups, int32_t* n_groups) {
  if (threadIdx.x != 0) return;
  int g = 0;
  for (int b = 0; b < m.num_requests; ++b) {
    const int lo = max(m.query_start_loc[b], row0), hi = min(m.query_start_loc[b + 1], row0 + nrows);
    for (int r = lo; r < hi; r += rg) {
      groups[3 * g] = b;
      groups[3 * g + 1] = r;
      groups[3 * g + 2] = min(rg, hi - r);
      ++g;
    }
  }
  *n_groups = g;
}

// -inf for the positions of a caller-visible score row that no tile covered (s beyond the row's last tile).
__global__ void indexer_fill_tail_kernel(RowMeta m, int row0, float* scores, int64_t stride, int max_seq_len) {
  const int r = row0 + blockIdx.y;
  int b, pos;
  row_info(m, r, b, pos);
  const int start = pos < 0 ? 0 : (pos / 128 + 1) * 128;
  for (int s = start + blockIdx.x * blockDim.x + threadIdx.x; s < max_seq_len; s += gridDim.x * blockDim.x)
    scores[(int64_t)blockIdx.y * stride + s] = -INFINITY;
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
    const bool ok = format == DSA_KEY_FP8_E4M3
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
int g_sm_count = 0;
}  // namespace

static int indexer_rows_per_group(const dsa_cache& c, bool decode) {
  if (decode) return 1;
  return c.key_format == DSA_KEY_FP8_E4M3 ? 4 : idx::kMaxRows;
}

cudaError_t launch_indexer_scores(const dsa_cache& c, const RowMeta& m, int row0, int nrows, int max_seq_len,
                                  const void* q_idx, const float* w, float* scores, int64_t score_stride,
                                  bool fill_tail, int32_t* group_scratch, uint32_t* err, cudaStream_t s) {
  const bool fp8 = c.key_format == DSA_KEY_FP8_E4M3;
  const bool decode = m.query_start_loc == nullptr;
  static bool configured[2] = {false, false};
  if (!configured[fp8]) {
    cudaError_t e = fp8 ? cudaFuncSetAttribute(indexer_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               idx::kSmemBytes)
                        : cudaFuncSetAttribute(indexer_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               idx::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[fp8] = true;
  }
  if (g_sm_count == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (g_sm_count <= 0) g_sm_count = kMlaCtas;
  }
  const uint32_t box_rows = (uint32_t)(c.page_size < idx::kTileKeys ? c.page_size : idx::kTileKeys);
  CUtensorMap map;
  if (!g_key_maps.get(c.index_keys, (uint64_t)c.num_pages * c.page_size, c.key_format, box_rows, &map))
    return cudaErrorInvalidValue;

  IdxArgs a;
  a.m = m;
  const int rg = indexer_rows_per_group(c, decode);
  if (decode) {
    a.groups = nullptr;
    a.n_groups = nullptr;
    a.max_groups = nrows;
  } else {
    a.groups = group_scratch + 4;
    a.n_groups = group_scratch;
    a.max_groups = nrows;                        // every group holds at least one row
    indexer_groups_kernel<<<1, 32, 0, s>>>(m, row0, nrows, rg, group_scratch + 4, group_scratch);
    count_launches(1);
  }
  a.row0 = row0;
  a.nrows_block = nrows;
  // long key blocks amortise the group's query load when requests carry many rows (prefill)
  a.block_tiles = (!decode && nrows >= 8 * m.num_requests) ? 32 : 8;
  a.key_blocks = (max_seq_len + idx::kTileKeys * a.block_tiles - 1) / (idx::kTileKeys * a.block_tiles);
  a.log2_page = ilog2(c.page_size);
  a.num_pages = c.num_pages;
  a.box_rows = (int)box_rows;
  a.key_scales = c.index_scales;
  a.q_idx = static_cast<const __nv_bfloat16*>(q_idx);
  a.w = w;
  a.scores = scores;
  a.stride = score_stride;
  a.max_seq_len = max_seq_len;
  a.err = err;
  const int64_t units = (int64_t)a.max_groups * a.key_blocks;
  const int grid = (int)(units < g_sm_count ? units : g_sm_count);
  if (fp8)
    indexer_tc_kernel<true><<<grid, idx::kThreads, idx::kSmemBytes, s>>>(map, a);
  else
    indexer_tc_kernel<false><<<grid, idx::kThreads, idx::kSmemBytes, s>>>(map, a);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !fill_tail) return e;
  dim3 fgrid((max_seq_len + 255) / 256 < 64 ? (max_seq_len + 255) / 256 : 64, nrows);
  indexer_fill_tail_kernel<<<fgrid, 256, 0, s>>>(m, row0, scores, score_stride, max_seq_len);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace dsa
