// Sparse absorbed MLA over the selected positions, on tcgen05 tensor cores.
//
// For row r, head h and valid selected s (0 <= s <= pos(r)):
//   z_s = scale * (q[r,h,:512] . c_KV[s] + q[r,h,512:] . k_R[s])
//   out[r,h,:] = sum_s softmax(z)_s c_KV[s],  lse[r,h] = ln sum_s exp(z_s)
// ("vLLM Inference Path: GLM-5.2 as an Example", "MLA Projections and KV State"
// and "Sparse MLA Attention"; "Making GLM-5.2 Sparse on TPUs", "Separate the
// indexer from the attention it controls": absorbed MLA, scale tied to the
// unabsorbed 192 + 64 width; "Carry sparse reads through prefill": online
// softmax over the selected entries).
//
// Work: the rows' index buffers are cut into tiles of 64 entries.  With few
// rows (2 R <= 152) each row is cut into S = 2, 4 or 8 equal pieces taken by
// the S CTAs of one thread-block cluster: after a cluster barrier each CTA
// pushes its unnormalised O^T and (m, l) into the shared memory of the CTA
// that owns each head (distributed shared memory), and each CTA merges its
// 64 / S heads locally.  Otherwise the
// (row, tile) units are split into one contiguous range per CTA (persistent,
// one CTA per SM); a row cut between CTAs is finished by an LSE merge of the
// pieces in a second kernel, and a row inside one CTA is written directly.
//
// Per CTA (16 warps):
//   warps 0-6  producers: TMA-load the row's 64 x 576 query (9 boxes of 64
//              heads x 64 columns) and gather each tile's 64 cached rows
//              straight out of the paged pool with TMA gather4 (four 128-byte
//              row pieces per instruction, 128-byte swizzle), two stages deep;
//              warp w looks up and gathers the tile's groups of four entries
//              w, w + 7 (and w + 14), because the TMA issue rate of one warp
//              is far below HBM speed;
//   warp 7     MMA issuer: S^T = K Q^T (M = 64 tokens, N = 64 heads, K = 576)
//              into TMEM, then O^T += V^T P^T (M = 128 latent dims x 4,
//              N = 64 heads, K = 64 tokens) with V read from the same gathered
//              tile (MN-major) and P^T from shared memory; the next tile's QK
//              goes out only after the current tile's PV;
//   warps 8-15 softmax, two warpgroups of 32 heads each: a thread holds 16
//              heads of one token (the M = 64 accumulator fills 16 lanes per
//              quarter; the second half of the lanes reads the next 16
//              columns), exp2 into bf16 P^T rows (one 128-byte row per token,
//              no transpose needed), a lazy rescale of the TMEM accumulator
//              only when a head's running maximum grows by more than 2^8
//              (checked with one predicate-OR barrier per tile), and the
//              epilogue.
// Shared memory: Q 72 KB + 2 x 72 KB tiles + 8 KB P^T.  TMEM: 2 x 64 columns
// for S^T and 4 x 64 columns for O^T.
#include <mutex>

#include "dsa_internal.cuh"
#include "sm100.cuh"
#include "tmap.cuh"

namespace dsa {
using namespace sm100;

namespace mla {
constexpr int kTok = 64;                           // selected entries per tile (MMA M of S^T)
constexpr int kChunks = kRow / 64;                 // 9 column chunks of 64 bf16 (128 bytes)
constexpr int kChunkBytes = kTok * 128;            // one chunk of a tile
constexpr int kStageBytes = kChunks * kChunkBytes; // 72 KB
constexpr int kQChunkBytes = kHeads * 128;
constexpr int kQBytes = kChunks * kQChunkBytes;    // 72 KB
constexpr int kPBytes = kTok * 128;                // P^T: 64 tokens x 64 heads bf16
constexpr int kSmemBytes = kQBytes + 2 * kStageBytes + kPBytes + 1024;
constexpr int kProducers = 7;                      // warps issuing the gathers (TMA issue is per-warp limited)
constexpr int kGroups = kTok / 4;                  // gather4 groups of a tile: group g is taken by warp g % 7
constexpr int kMmaWarp = 7;                        // last warp of warpgroup 1
constexpr int kSoftmaxWarp0 = 8;                   // warpgroups 2 and 3: heads 0-31 and heads 32-63
constexpr int kThreads = 512;
// register split (sums to 61,440 of the 512 x 128 launched): producers / MMA and the two softmax
// warpgroups.  At 80 the one-layer bf16 kernel spills in its producer code; at 88 it does not, and
// prefill's attention takes 2.17 ms instead of 2.19.  The layer-group kernel, spill-free at 80, is
// about 1 % slower at 88, and the packed 8-bit latent's producers keep 80 too.
constexpr uint32_t kRegsTotal = 240;
template <bool kC8, int kNL>
constexpr uint32_t kRegsLow = !kC8 && kNL == 1 ? 88u : 80u;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;                      // S^T of stage b at columns 64 b
constexpr uint32_t kColO = 128;                    // O^T chunk k (dims 128k..) at columns 128 + 64 k
constexpr float kRescaleLog2 = 8.f;
constexpr uint32_t kPolls = 1u << 22;
}  // namespace mla

struct MlaArgs {
  RowMeta m;
  const int32_t* topk_idx;
  const int32_t* row_count;       // optional [rows]: valid entries lead each row (cluster mode uses it)
  int topk, tiles, units, ctas;
  int split;                      // > 1: cluster mode, pieces per row (= cluster size); 1: unit split
  int log2_page, num_pages;
  float scale_log2;               // softmax scale * log2(e)
  __nv_bfloat16* out;
  float* lse;
  float* part_o;                  // [2 * ctas][64][512]
  float* part_ml;                 // [2 * ctas][64][2]
  uint32_t* cta_err;              // [ctas]: each CTA's status bits (zeroed by the CTA itself)
  uint32_t* err;                  // the workspace header: [0] call-wide bits (0 here), [1] number of cta_err words
};

__device__ __forceinline__ int unit_start(int c, int units, int ctas) {
  if ((uint64_t)units * (uint64_t)ctas < (1ull << 32)) return (int)(((uint32_t)c * (uint32_t)units) / (uint32_t)ctas);
  return (int)(((int64_t)c * units) / ctas);
}

__device__ __forceinline__ int cta_of_unit(int u, int units, int ctas) {
  int c = (uint64_t)units * (uint64_t)ctas < (1ull << 32) ? (int)(((uint32_t)u * (uint32_t)ctas) / (uint32_t)units)
                                                           : (int)(((int64_t)u * ctas) / units);
  while (c + 1 < ctas && unit_start(c + 1, units, ctas) <= u) ++c;
  while (c > 0 && unit_start(c, units, ctas) > u) --c;
  return c;
}

// Cluster merge, push side: a softmax thread's latent dims d = 128 k + (this thread's offset in
// `rows`) of the 32 heads h0 .. h0 + 31, read from TMEM (O^T at `src` + 64 k) and stored into the
// shared memory of each head's owner CTA (head h belongs to CTA h / HS), at row h % HS of the
// block `rows` (this piece's block, mapped into the owner's window).  Heads this CTA (cluster rank
// `self`) owns take plain local stores.
template <int HS>
__device__ __forceinline__ void push_piece(uint32_t src, const float* rows, int h0, bool has_valid, int self) {
  constexpr int kOwners = 32 / HS;
  uint32_t ob[kOwners];
#pragma unroll
  for (int i = 0; i < kOwners; ++i) ob[i] = h0 / HS + i == self ? smem_u32(rows) : cluster_map(rows, (uint32_t)(h0 / HS + i));
  tc_fence_after();
#pragma unroll 1
  for (int k = 0; k < 4; ++k) {
    uint32_t o[32];
    tmem_ld32(src + 64 * k, o);
    tmem_wait_ld();
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      const uint32_t dst = ob[jj / HS] + (uint32_t)(((jj % HS) * kLatent + 128 * k) * 4);
      if (h0 / HS + jj / HS == self)
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(dst), "f"(has_valid ? __uint_as_float(o[jj]) : 0.f) : "memory");
      else
        asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dst), "f"(has_valid ? __uint_as_float(o[jj]) : 0.f)
                     : "memory");
    }
  }
}

// fp16 bits of 2^e for -24 <= e <= 15 (subnormal below -14)
__device__ __forceinline__ uint16_t half_pow2_bits(int e) {
  return e >= -14 ? (uint16_t)((e + 15) << 10) : (uint16_t)(1u << (e + 24));
}

// kC8: the latent pool holds packed 8-bit rows [c_KV as 512 e4m3 codes | k_R as 64 bf16] (640 bytes)
// and a scale per slot.  Each producer warp gathers its groups' rows as five 128-byte pieces into the
// slots the first five chunks of those groups would take, waits for the tile's gathers, and expands them in place
// into the tile's usual swizzled 576-wide layout in fp16: c_KV = code * scale, k_R converted.  The
// query row is converted to fp16 in place once it lands, P^T is written in fp16, and both MMAs take
// fp16 operands (kind::f16 with A and B of one type).
// One call may cover the layers of an IndexShare group (one index buffer): its rows are then the
// layers' rows stacked layer-major (q, out, lse and the split-k slots by that combined row), and
// a tile gathers from the latent pool of its own layer, layer = combined row / layer_rows.
// A one-layer call passes a single map (kNL = 1: no layer arithmetic, the smallest parameter block).
template <int kNL>
struct MlaKvMaps {
  CUtensorMap layer[kNL];
};

template <bool kC8, int kNL>
__global__ void __launch_bounds__(mla::kThreads, 1)
    sparse_mla_tc_kernel(const __grid_constant__ MlaKvMaps<kNL> kv, const __grid_constant__ CUtensorMap q_map,
                         const MlaArgs a, const float* __restrict__ latent_scales, int rows_share_pool,
                         int layer_rows) {
  using namespace mla;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + kQBytes;
  uint8_t* sP = sKV + 2 * kStageBytes;

  __shared__ uint64_t kv_full[2], kv_empty[2], s_full[2], s_empty[2];
  __shared__ uint64_t p_full, p_empty, q_full, q_empty, o_full, o_empty, mma_done;
  __shared__ uint64_t cv_full[2], q_conv;   // packed 8-bit latent only: gathers landed, query converted
  __shared__ __align__(16) uint8_t tile_mask4[2][kGroups];   // entry validity, 4 bits per gather4 group
  __shared__ float red[4][kHeads];
  __shared__ float mref[kHeads], alpha[kHeads], lfin[kHeads];
  __shared__ int rescale_tag[2];
  __shared__ uint32_t tmem_base;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const int T = a.tiles;
  uint32_t* const err = a.cta_err + cta;
  const int split = a.split;
  // cluster mode: piece cta % split of row cta / split; otherwise a contiguous range of units
  int u0 = split > 1 ? (cta / split) * T + (cta % split) * T / split : unit_start(cta, a.units, a.ctas);
  int u1 = split > 1 ? (cta / split) * T + (cta % split + 1) * T / split : unit_start(cta + 1, a.units, a.ctas);

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&kv_full[b], kProducers);   // every producer warp arrives (with its own byte count)
      mbar_init(&kv_empty[b], 1);
      mbar_init(&s_full[b], 1);
      mbar_init(&s_empty[b], 8);                 // every softmax warp
    }
    mbar_init(&p_full, 2);                       // both softmax warpgroups
    mbar_init(&p_empty, 1);
    mbar_init(&q_full, 1);
    mbar_init(&q_empty, 1);
    mbar_init(&o_full, 1);
    mbar_init(&o_empty, 8);
    mbar_init(&mma_done, 1);
    if (kC8) {
      for (int b = 0; b < 2; ++b) mbar_init(&cv_full[b], kProducers);   // every producer warp's gathers
      mbar_init(&q_conv, kProducers);                                    // every producer warp
    }
    rescale_tag[0] = rescale_tag[1] = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // rows a tile does not gather keep older finite data (zeros at first): their probability is 0
  for (int i = threadIdx.x; i < 2 * kStageBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(sKV)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&kv.layer[0]);
    prefetch_tmap(&q_map);
  }
  // the index buffer, the queries and the caches are complete past this point (programmatic
  // dependent launch: the prologue above overlaps the previous kernel).  The unit split triggers its
  // merge kernel only at exit (launched while this grid still ran, it made each call about 5 us
  // slower); cluster mode triggers as each CTA enters the cluster merge (4 us off a benchmark step).
  pdl_wait();
  // With row counts (cluster mode only) a row spans only the tiles that hold its first row_count
  // entries, at least one per piece; entries past the count are -1 by contract, so the unit split,
  // which ignores the counts, gives the same result.  The counts are read after the wait; the
  // ranges without them are known before it (computing them only after the wait cost 6 us a call).
  if (split > 1 && a.row_count) {
    const int c = a.row_count[cta / split];
    const int Tr = c < 0 ? split : min(T, max(split, (c + kTok - 1) / kTok));
    u0 = (cta / split) * T + (cta % split) * Tr / split;
    u1 = (cta / split) * T + (cta % split + 1) * Tr / split;
  }
  // this CTA's status bits: cleared after the wait (every earlier kernel of the stream has completed)
  // and before the barrier below, after which a bounded wait may set them.  CTA 0 also writes the
  // workspace header: no call-wide bits, and the number of per-CTA words that dsa_read_status ORs.
  if (threadIdx.x == 0) {
    *err = 0u;
    if (cta == 0) {
      a.err[0] = 0u;
      a.err[1] = (uint32_t)a.ctas;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  // one register split per warpgroup, executed by all of its warps at one instruction: producers and
  // the MMA issuer (warpgroups 0-1) give registers to the two softmax warpgroups
  if (warp < kSoftmaxWarp0) {
  regs_dec<kRegsLow<kC8, kNL>>();
  if (warp < kProducers) {
    // ------------------------------------------------------------------ producers
    // Warp w owns the tile's gather4 groups w, w + 7 (and w + 14): lane l < 4 ng looks up entry
    // l % 4 of its group l / 4 one tile ahead, so the index-buffer and page-table loads stay off
    // the critical path; lane l < 9 ng gathers 128-byte column chunk l % 9 of group l / 9.
    const int ng = (kGroups - warp + kProducers - 1) / kProducers;   // groups of this warp (2 or 3)
    // a row read by one query row only is evicted first (the index buffer, queries and partials stay
    // in L2); rows that a request's other query rows may select again keep their normal priority
    const uint64_t gather_policy = rows_share_pool ? l2_evict_normal() : l2_evict_first();
    int q_loads = 0, cur_row = -1;
    int filled[2] = {0, 0};
    auto lookup = [&](int u) -> int64_t {
      const int rr = u / T, j = u - rr * T, r = kNL > 1 ? rr % layer_rows : rr;   // the row within its layer
      int req, pos;
      row_info(a.m, r, req, pos);
      const int g = warp + kProducers * (lane >> 2);
      const int t = j * kTok + 4 * g + (lane & 3);
      const int e = (lane < 4 * ng && t < a.topk) ? a.topk_idx[(int64_t)r * a.topk + t] : -1;
      if (e < 0 || e > pos) return -1;
      const int64_t slot = token_slot(a.m, req, e, a.log2_page, a.num_pages);
      if (slot < 0) atomicOr(err, kErrBadPage);    // a visible entry whose page is outside the pool: skipped
      return slot;
    };
    constexpr int kPieces = kC8 ? 5 : kChunks;        // 128-byte pieces gathered per row
    // the scale of a looked-up entry (packed 8-bit latent; 0 where the entry is invalid)
    auto scale_of = [&](int64_t slot) -> float { return (kC8 && slot >= 0) ? __ldg(latent_scales + slot) : 0.f; };
    // packed 8-bit latent: expand this warp's groups of tile ip (landed in stage ip & 1) in place
    auto convert = [&](int ip, uint32_t vmask, float scl) -> bool {
      const int bp = ip & 1;
      if (!mbar_wait(&cv_full[bp], (ip >> 1) & 1, err, kErrTmaTimeout, kPolls)) return false;
      uint8_t* stage = sKV + bp * kStageBytes;
      const int rl = lane >> 3, j = lane & 7;
      for (int qg = 0; qg < ng; ++qg) {
        const float sc = __shfl_sync(0xffffffffu, scl, 4 * qg + rl);
        if (((vmask >> (4 * qg)) & 0xFu) == 0u) continue;          // not gathered (uniform in the warp)
        const int t = 4 * (warp + kProducers * qg) + rl;          // this lane's row of the tile
        uint8_t* row = stage + t * 128;
        const int sw = t & 7;                                      // 128-byte swizzle of the row
        uint4 in[5];
#pragma unroll
        for (int pc = 0; pc < 5; ++pc) in[pc] = *reinterpret_cast<const uint4*>(row + pc * kChunkBytes + ((j ^ sw) << 4));
        __syncwarp();                                              // the group's pieces are read before any write
        // sc = m 2^e with m in [1, 2): code * m stays below 896, then the exact power of two
        const uint32_t sb = __float_as_uint(sc);
        const int e = sc > 0.f ? (int)((sb >> 23) & 0xFFu) - 127 : 0;
        const __half2 m2 = __float2half2_rn(sc > 0.f ? __uint_as_float((sb & 0x807FFFFFu) | 0x3F800000u) : 0.f);
        const uint16_t pb = half_pow2_bits(e < -24 ? -24 : (e > 15 ? 15 : e));
        const __half2 p2 = __halves2half2(__ushort_as_half(pb), __ushort_as_half(pb));
#pragma unroll
        for (int pc = 0; pc < 4; ++pc) {
          const uint32_t w4[4] = {in[pc].x, in[pc].y, in[pc].z, in[pc].w};
          uint32_t h[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w4[k >> 1] >> (16 * (k & 1))), __NV_E4M3);
            __half2 v = __hmul2(__hmul2(*reinterpret_cast<const __half2*>(&hr), m2), p2);
            h[k] = *reinterpret_cast<const uint32_t*>(&v);
          }
          // dims 128 pc + 16 j .. + 15: chunk 2 pc + j / 4, units 2 (j % 4) and 2 (j % 4) + 1
          uint8_t* dst = row + (2 * pc + (j >> 2)) * kChunkBytes;
          const int u0 = 2 * (j & 3);
          *reinterpret_cast<uint4*>(dst + ((u0 ^ sw) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
          *reinterpret_cast<uint4*>(dst + (((u0 + 1) ^ sw) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
        {
          const uint32_t w4[4] = {in[4].x, in[4].y, in[4].z, in[4].w};   // k_R dims 8 j .. 8 j + 7, bf16
          uint32_t h[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const __half2 v = __float22half2_rn(__bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[k])));
            h[k] = *reinterpret_cast<const uint32_t*>(&v);
          }
          *reinterpret_cast<uint4*>(row + 8 * kChunkBytes + ((j ^ sw) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
        }
        __syncwarp();
      }
      fence_proxy_async_smem();                                    // generic writes before the MMA's reads
      __syncwarp();
      if (lane == 0) mbar_arrive(&kv_full[bp]);
      return true;
    };
    int64_t nxt = u0 < u1 ? lookup(u0) : -1;
    float nxt_sc = 0.f;
    if constexpr (kC8) nxt_sc = scale_of(nxt);
    uint32_t prev_valid = 0;
    float prev_sc = 0.f;
    bool ok = true;
    for (int u = u0; u < u1; ++u) {
      const int i = u - u0, b = i & 1, n = i >> 1;
      const int r = u / T;
      const int64_t sl = nxt;
      const float cur_sc = nxt_sc;
      // packed 8-bit latent: the previous tile is expanded first (the MMA needs it before it can
      // release the query of a finished row or the stage this tile reuses)
      if constexpr (kC8) {
        if (i > 0 && !(ok = convert(i - 1, prev_valid, prev_sc))) break;
      }
      if (n > 0 && !mbar_wait(&kv_empty[b], (n - 1) & 1, err, kErrMmaTimeout, kPolls)) break;
      bool new_q = false;
      if (r != cur_row) {
        if (q_loads > 0 && !mbar_wait(&q_empty, (q_loads - 1) & 1, err, kErrMmaTimeout, kPolls)) break;
        if (warp == 0 && lane == 0) {
          mbar_arrive_expect_tx(&q_full, kQBytes);
          for (int c = 0; c < kChunks; ++c) tma_load_2d(sQ + c * kQChunkBytes, &q_map, c * 64, r * kHeads, &q_full);
        }
        ++q_loads;
        cur_row = r;
        new_q = true;
      }
      const uint32_t valid = __ballot_sync(0xffffffffu, sl >= 0) & ((1u << (4 * ng)) - 1u);
      // each group with a valid entry is gathered; its invalid entries repeat its first valid row
      const int q = lane / kPieces < ng ? lane / kPieces : 0, c = lane % kPieces;
      const uint32_t gbits = (valid >> (4 * q)) & 0xFu;
      const int first = gbits ? 4 * q + __ffs(gbits) - 1 : 0;
      const int64_t sub = __shfl_sync(0xffffffffu, sl, first);
      int32_t y[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t v = __shfl_sync(0xffffffffu, sl, 4 * q + k);
        y[k] = (int32_t)(v >= 0 ? v : sub);
      }
      uint64_t* land = kC8 ? &cv_full[b] : &kv_full[b];
      if (lane == 0) {
        uint32_t groups = 0;
        for (int qq = 0; qq < ng; ++qq) {
          const uint32_t gb = (valid >> (4 * qq)) & 0xFu;
          tile_mask4[b][warp + kProducers * qq] = (uint8_t)gb;
          groups += gb ? 1u : 0u;
        }
        mbar_arrive_expect_tx(land, groups * (uint32_t)(kPieces * 512));
      }
      __syncwarp();
      ++filled[b];
      if (lane < kPieces * ng && gbits) {
        uint8_t* stage = sKV + b * kStageBytes;
        const int g = warp + kProducers * q;
        tma_gather4_hint(stage + c * kChunkBytes + g * 512, &kv.layer[kNL > 1 ? r / layer_rows : 0], c * 64,
                         y[0], y[1], y[2], y[3], land, gather_policy);
      }
      if constexpr (kC8) {
       if (new_q) {
        // the query row in fp16, in place (same swizzled layout, same element width)
        if (!mbar_wait(&q_full, (q_loads - 1) & 1, err, kErrTmaTimeout, kPolls)) break;
        for (int k = warp * 32 + lane; k < kQBytes / 16; k += kProducers * 32) {
          uint4 v = reinterpret_cast<const uint4*>(sQ)[k];
          uint32_t* w4 = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __half2 h = __float22half2_rn(__bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e])));
            w4[e] = *reinterpret_cast<const uint32_t*>(&h);
          }
          reinterpret_cast<uint4*>(sQ)[k] = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_conv);
       }
        prev_valid = valid;
        prev_sc = cur_sc;
      }
      if (u + 1 < u1) {
        nxt = lookup(u + 1);
        if constexpr (kC8) nxt_sc = scale_of(nxt);
      }
      if constexpr (kC8) {
        if (u + 1 == u1) ok = convert(i, prev_valid, prev_sc);   // the last tile
      }
    }
    // nothing may still be landing in shared memory when the CTA exits
    for (int b = 0; b < 2; ++b)
      if (filled[b] > 0)
        mbar_wait(kC8 ? &cv_full[b] : &kv_full[b], (filled[b] - 1) & 1, err, kErrTmaTimeout, kPolls);
    if (q_loads > 0) mbar_wait(&q_full, (q_loads - 1) & 1, err, kErrTmaTimeout, kPolls);
    (void)ok;
  } else {
    // ------------------------------------------------------------------ MMA issuer (warp 7)
    if (lane == 0) {
      // bf16 operands, or fp16 ones for the packed 8-bit latent (the expanded tile, Q and P^T)
      const uint32_t id_qk = idesc_f16(64, kHeads, !kC8, !kC8, false, false);
      const uint32_t id_pv = idesc_f16(128, kHeads, !kC8, !kC8, true, true);
      // descriptors are built once; per MMA only the start-address field (bytes >> 4) advances
      const uint64_t d_k0 = smem_desc(smem_u32(sKV), 16, 1024, kSwizzle128B);
      const uint64_t d_q = smem_desc(smem_u32(sQ), 16, 1024, kSwizzle128B);
      const uint64_t d_v0 = smem_desc(smem_u32(sKV), kChunkBytes, 1024, kSwizzle128B);
      const uint64_t d_p = smem_desc(smem_u32(sP), kChunkBytes, 1024, kSwizzle128B);
      const uint32_t hi = (uint32_t)(d_k0 >> 32);          // the same for all four descriptors
      const uint32_t k_lo0 = (uint32_t)d_k0, q_lo0 = (uint32_t)d_q, v_lo0 = (uint32_t)d_v0, p_lo0 = (uint32_t)d_p;
      int q_loads = 0, seg = 0, prev_row = -1;
      bool o_init = false, ok = true;
      // PV of tile ip releases a stage and must not wait behind the QK of a later tile: issue
      // whichever of QK(iq) / PV(ip) is ready, PV first.
      const int ntiles = u1 - u0;
      int iq = 0, ip = 0;
      uint32_t idle = 0;
      while (ok && ip < ntiles) {
        bool progressed = false;
        if (ip < iq) {
          const int i = ip, u = u0 + i, b = i & 1, r = u / T, j = u - r * T;
          const bool seg_first = (u == u0) || j == 0;
          const bool seg_last = (u == u1 - 1) || j == T - 1;
          if (mbar_test(&p_full, i & 1) && (!seg_first || seg == 0 || mbar_test(&o_empty, (seg - 1) & 1))) {
            if (seg_first) o_init = false;
            tc_fence_after();
            const volatile uint64_t* tm = reinterpret_cast<const volatile uint64_t*>(tile_mask4[b]);
            if ((tm[0] | tm[1]) != 0) {
              const uint32_t v = opaque_u32(v_lo0 + (uint32_t)((b * kStageBytes) >> 4)), pl = opaque_u32(p_lo0);
              const uint32_t dO = opaque_u32(tmem + kColO);
              if (!o_init) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  mma_ss_lh<false>(dO + 64 * k, v + ((2 * k * kChunkBytes) >> 4), hi, pl, hi, id_pv);
#pragma unroll
                  for (int kk = 1; kk < 4; ++kk)
                    mma_ss_lh<true>(dO + 64 * k, v + ((2 * k * kChunkBytes + kk * 2048) >> 4), hi,
                                    pl + ((kk * 2048) >> 4), hi, id_pv);
                }
              } else {
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll
                  for (int kk = 0; kk < 4; ++kk)
                    mma_ss_lh<true>(dO + 64 * k, v + ((2 * k * kChunkBytes + kk * 2048) >> 4), hi,
                                    pl + ((kk * 2048) >> 4), hi, id_pv);
              }
              o_init = true;
            }
            mma_commit(&kv_empty[b]);
            mma_commit(&p_empty);
            if (seg_last) {
              mma_commit(&o_full);
              ++seg;
            }
            ++ip;
            progressed = true;
          }
        }
        if (iq < ntiles && iq < ip + 1) {
          const int i = iq, u = u0 + i, b = i & 1, n = i >> 1, r = u / T;
          const bool need_q = r != prev_row;
          if (mbar_test(&kv_full[b], n & 1) && (!need_q || mbar_test(kC8 ? &q_conv : &q_full, q_loads & 1)) &&
              (n == 0 || mbar_test(&s_empty[b], (n - 1) & 1))) {
            if (need_q) {
              ++q_loads;
              prev_row = r;
            }
            tc_fence_after();
            const uint32_t kl = opaque_u32(k_lo0 + (uint32_t)((b * kStageBytes) >> 4)), ql = opaque_u32(q_lo0);
            const uint32_t ds = tmem + kColS + 64 * b;
            mma_ss_lh<false>(ds, kl, hi, ql, hi, id_qk);
#pragma unroll
            for (int kk = 1; kk < kChunks * 4; ++kk) {
              const int c = kk >> 2, off = (kk & 3) * 32;
              mma_ss_lh<true>(ds, kl + ((c * kChunkBytes + off) >> 4), hi, ql + ((c * kQChunkBytes + off) >> 4), hi, id_qk);
            }
            mma_commit(&s_full[b]);
            if (u == u1 - 1 || (u + 1) / T != r) mma_commit(&q_empty);
            ++iq;
            progressed = true;
          }
        }
        if (progressed) idle = 0;
        else if (++idle > (kPolls << 2)) {
          atomicOr(err, kErrMmaTimeout);
          ok = false;
        }
      }
      // every MMA issued here has finished before TMEM is released
      mma_commit(&mma_done);
      mbar_wait(&mma_done, 0, err, kErrMmaTimeout, kPolls);
    }
  }
  } else {
    regs_inc<kRegsTotal - kRegsLow<kC8, kNL>>();
    // ------------------------------------------------------------------ softmax + epilogue (warps 8-15)
    // Warpgroup sg (0: warps 8-11, 1: warps 12-15) owns heads 32 sg .. 32 sg + 31: their running
    // maxima, rescales, denominators and outputs.  S^T row (token) tok sits in TMEM lane
    // 32 * quarter + lane % 16; a thread holds 16 of its warpgroup's heads for that token (lanes
    // 0-15 the first 16 columns, lanes 16-31 the next 16).
    const int sg = (warp - kSoftmaxWarp0) >> 2;
    const int bar = 1 + sg;                              // named barrier of this warpgroup
    const int quarter = warp & 3;                       // TMEM lanes this warp may touch
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    const int tok = 16 * quarter + (lane & 15);
    const int h0 = 32 * sg;                             // first head of the warpgroup
    const int hh = h0 + 16 * (lane >> 4);               // first head of this thread
    const int st = threadIdx.x - 32 * (kSoftmaxWarp0 + 4 * sg);   // 0..127 within the warpgroup
    const int first_row = u0 / T;
    float l_acc[16];
    int seg = 0;
    for (int u = u0; u < u1; ++u) {
      const int i = u - u0, b = i & 1, n = i >> 1, r = u / T, j = u - r * T;
      const bool seg_first = (u == u0) || j == 0;
      const bool seg_last = (u == u1 - 1) || j == T - 1;
      if (seg_first) {
#pragma unroll
        for (int h = 0; h < 16; ++h) l_acc[h] = 0.f;
        if (st < 32) mref[h0 + st] = -INFINITY;
      }
      if (!mbar_wait(&kv_full[b], n & 1, err, kErrTmaTimeout, kPolls)) break;
      if (!mbar_wait(&s_full[b], n & 1, err, kErrMmaTimeout, kPolls)) break;
      tc_fence_after();
      uint32_t sv[16];
      tmem_ld16x2_16(tmem + lane_base + kColS + 64 * b + h0, sv);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[b]);
      const bool valid = (tile_mask4[b][tok >> 2] >> (tok & 3)) & 1u;
      float z[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) z[h] = valid ? __uint_as_float(sv[h]) * a.scale_log2 : -INFINITY;
      // The running reference changes only when some head's tile maximum exceeds it by more than
      // 2^kRescaleLog2; one predicate-OR barrier decides whether the exact per-head maxima are needed
      // (always on a segment's first tile, which sets the reference).
      bool need = seg_first;                             // mref was just reset by another thread
#pragma unroll
      for (int h = 0; h < 16; ++h) need |= z[h] > mref[hh + h] + kRescaleLog2;
      const bool resc = named_bar_or(bar, 128, need);
      if (resc) {
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          float mx = z[h];
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          if ((lane & 15) == 0) red[quarter][hh + h] = mx;
        }
        named_bar_sync(bar, 128);
        if (st < 32) {
          const int h = h0 + st;
          const float M = fmaxf(fmaxf(red[0][h], red[1][h]), fmaxf(red[2][h], red[3][h]));
          const float old = mref[h];
          float al = 1.f;
          if (M > -INFINITY && (old == -INFINITY || M > old + kRescaleLog2)) {
            al = old == -INFINITY ? 0.f : exp2f(old - M);
            if (old != -INFINITY) rescale_tag[sg] = i + 1;
            mref[h] = M;
          }
          alpha[h] = al;
        }
        named_bar_sync(bar, 128);
      }
      const bool do_rescale = resc && rescale_tag[sg] == i + 1;
      uint32_t pk[8];
#pragma unroll
      for (int h = 0; h < 16; h += 2) {
        const float m0 = mref[hh + h], m1 = mref[hh + h + 1];
        const float p0 = z[h] == -INFINITY ? 0.f : ex2_approx(z[h] - m0);
        const float p1 = z[h + 1] == -INFINITY ? 0.f : ex2_approx(z[h + 1] - m1);
        uint32_t pb;
        if (kC8) {
          const __half2 v = __floats2half2_rn(p0, p1);
          pb = *reinterpret_cast<const uint32_t*>(&v);
        } else {
          const __nv_bfloat162 v = __floats2bfloat162_rn(p0, p1);
          pb = *reinterpret_cast<const uint32_t*>(&v);
        }
        l_acc[h] = fmaf(l_acc[h], resc ? alpha[hh + h] : 1.f, p0);   // the denominator keeps the fp32 probabilities
        l_acc[h + 1] = fmaf(l_acc[h + 1], resc ? alpha[hh + h + 1] : 1.f, p1);
        pk[h >> 1] = pb;
      }
      // P^T is free once the previous tile's PV has completed (which also settles O^T)
      if (i > 0 && !mbar_wait(&p_empty, (i - 1) & 1, err, kErrMmaTimeout, kPolls)) break;
#pragma unroll
      for (int c = 0; c < 2; ++c)
        *reinterpret_cast<uint4*>(sP + sw128_offset(tok, (hh >> 3) + c)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      if (do_rescale) {
        tc_fence_after();
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {
          uint32_t o[32];
          const uint32_t addr = tmem + lane_base + kColO + 64 * k + h0;
          tmem_ld32(addr, o);
          tmem_wait_ld();
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) o[jj] = __float_as_uint(__uint_as_float(o[jj]) * alpha[h0 + jj]);
          tmem_st32(addr, o);
        }
        tmem_wait_st();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(bar, 128);
      if (st == 0) mbar_arrive(&p_full);

      if (seg_last) {
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          float v = l_acc[h];
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if ((lane & 15) == 0) red[quarter][hh + h] = v;
        }
        named_bar_sync(bar, 128);
        if (st < 32) {
          const float L = (red[0][h0 + st] + red[1][h0 + st]) + (red[2][h0 + st] + red[3][h0 + st]);
          lfin[h0 + st] = L;
          // 1 / l for a whole row's output, in alpha (this tile's rescale factors are no longer read):
          // a division per output element made the epilogue of a whole row about 3 times slower
          alpha[h0 + st] = L > 0.f ? 1.f / L : 0.f;
        }
        named_bar_sync(bar, 128);
        if (!mbar_wait(&o_full, seg & 1, err, kErrMmaTimeout, kPolls)) break;
        tc_fence_after();
        const int seg_start = u0 > r * T ? u0 : r * T;
        const bool whole = seg_start == r * T && j == T - 1;
        const int slot = r == first_row ? 2 * cta : 2 * cta + 1;
        // a piece without valid entries never initialised its accumulator (its l is 0 for every head,
        // and positive for every head otherwise): it contributes zeros, not TMEM contents
        const bool has_valid = lfin[h0] > 0.f;
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {
          const int d = 128 * k + 32 * quarter + lane;
          uint32_t o[32];
          tmem_ld32(tmem + lane_base + kColO + 64 * k + h0, o);
          tmem_wait_ld();
          if (whole) {
            __nv_bfloat16* dst = a.out + (int64_t)r * kHeads * kLatent + d;
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
              dst[(int64_t)(h0 + jj) * kLatent] =
                  __float2bfloat16_rn(has_valid ? __uint_as_float(o[jj]) * alpha[h0 + jj] : 0.f);
          } else if (split > 1) {
            // cluster mode: the piece stays in TMEM, with its m (mref, log2 units) and l (lfin) in
            // shared memory, until the cluster merge below
          } else {
            float* dst = a.part_o + (int64_t)slot * kHeads * kLatent + d;
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) dst[(int64_t)(h0 + jj) * kLatent] = has_valid ? __uint_as_float(o[jj]) : 0.f;
          }
        }
        if (st < 32) {
          const int h = h0 + st;
          const float L = lfin[h];
          if (whole) {
            if (a.lse) a.lse[(int64_t)r * kHeads + h] = L > 0.f ? (mref[h] + log2f(L)) * 0.69314718055994530942f : -INFINITY;
          } else if (split == 1) {
            a.part_ml[((int64_t)slot * kHeads + h) * 2] = L > 0.f ? mref[h] * 0.69314718055994530942f : -INFINITY;
            a.part_ml[((int64_t)slot * kHeads + h) * 2 + 1] = L;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&o_empty);
        ++seg;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (split > 1) {
    // ---- cluster merge.  CTA q of the row's cluster owns heads [q HS, q HS + HS), HS = 64 / split:
    //   out = sum_p w_p O_p,  w_p = 2^{m_p - M} / L,  L = sum_p 2^{m_p - M} l_p,  lse = (M + log2 L) ln 2.
    // Each CTA pushes every head of its piece into the owner's shared memory (remote stores, no
    // round trips): O into [split][HS][512] fp32 in the gather stages, (m, l) into [split][HS][2] in
    // the P^T buffer; then every CTA merges its heads from local shared memory.
    const int r = u0 / T, q = cta % split, HS = kHeads / split, hs0 = q * HS;
    float* buf = reinterpret_cast<float*>(sKV);
    float* mlb = reinterpret_cast<float*>(sP);
    float* wts = mlb + 2 * kHeads;                       // [split][HS]
    // the next call (the next layer's attention) may be launched now: its CTAs take SMs as this
    // grid's CTAs leave, and it reads nothing before its own wait for this grid's completion
    pdl_trigger();
    cluster_sync();                     // every CTA of the cluster is done with its gather stages
    if (warp >= kSoftmaxWarp0) {
      const int sg = (warp - kSoftmaxWarp0) >> 2, quarter = warp & 3, h0 = 32 * sg;
      const int st = threadIdx.x - 32 * (kSoftmaxWarp0 + 4 * sg);
      const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
      const bool has_valid = lfin[h0] > 0.f;   // a piece without valid entries never set its accumulator
      const uint32_t src = tmem + lane_base + kColO + h0;
      const float* my_rows = buf + (q * HS) * kLatent + 32 * quarter + lane;
      if (HS == 32) push_piece<32>(src, my_rows, h0, has_valid, q);
      else if (HS == 16) push_piece<16>(src, my_rows, h0, has_valid, q);
      else push_piece<8>(src, my_rows, h0, has_valid, q);
      if (st < 32) {
        const int h = h0 + st, owner = h / HS;
        const uint32_t dst = cluster_map(mlb + 2 * (q * HS + (h - owner * HS)), owner);
        asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(dst), "f"(mref[h]), "f"(lfin[h]) : "memory");
      }
    }
    cluster_sync();                     // every piece of this CTA's heads is in its shared memory
    if (threadIdx.x < HS) {
      const int h = hs0 + threadIdx.x;
      float M = -INFINITY, L = 0.f;
      for (int p = 0; p < split; ++p) {
        const float m = mlb[2 * (p * HS + threadIdx.x)], l = mlb[2 * (p * HS + threadIdx.x) + 1];
        if (l > 0.f) {
          const float Mn = fmaxf(M, m);
          L = L * exp2f(M - Mn) + l * exp2f(m - Mn);   // M = -inf: L is 0 and so is the product
          M = Mn;
        }
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      for (int p = 0; p < split; ++p) {
        const float m = mlb[2 * (p * HS + threadIdx.x)], l = mlb[2 * (p * HS + threadIdx.x) + 1];
        wts[p * HS + threadIdx.x] = l > 0.f ? exp2f(m - M) * inv : 0.f;
      }
      if (a.lse) a.lse[(int64_t)r * kHeads + h] = L > 0.f ? (M + log2f(L)) * 0.69314718055994530942f : -INFINITY;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < HS * (kLatent / 4); i += kThreads) {
      const int hl = i / (kLatent / 4), d = 4 * (i % (kLatent / 4));
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int p = 0; p < split; ++p) {
        const float w = wts[p * HS + hl];
        const float4 x = *reinterpret_cast<const float4*>(buf + (p * HS + hl) * kLatent + d);
        acc.x = fmaf(w, x.x, acc.x);
        acc.y = fmaf(w, x.y, acc.y);
        acc.z = fmaf(w, x.z, acc.z);
        acc.w = fmaf(w, x.w, acc.w);
      }
      uint2 v;
      __nv_bfloat162* xo = reinterpret_cast<__nv_bfloat162*>(&v);
      xo[0] = __floats2bfloat162_rn(acc.x, acc.y);
      xo[1] = __floats2bfloat162_rn(acc.z, acc.w);
      *reinterpret_cast<uint2*>(a.out + ((int64_t)r * kHeads + hs0 + hl) * kLatent + d) = v;
    }
  }
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// LSE merge of the pieces of rows that were cut between CTAs:
//   out = sum_j e^{m_j - M} O_j / sum_j e^{m_j - M} l_j,  lse = M + ln sum_j e^{m_j - M} l_j.
// One CTA per (CTA boundary b = 1 .. ctas - 1, 16 heads): a boundary inside a row stands for that row,
// once (its first boundary; rows that are not cut are written by the attention kernel), so the grid
// has one CTA per cut row and head group.  Thread (head, 16 consecutive latent dims); the pieces are
// read two at a time with all loads of a pair in flight, and merged online across pairs (the running
// maximum rescales what is already summed).  Launched as a programmatic dependent of the attention
// kernel: the wait below orders every read after that grid's writes.
constexpr int kMergeHeads = 16;
__global__ void __launch_bounds__(512, 2) mla_merge_kernel(MlaArgs a) {
  const int tid = threadIdx.x, T = a.tiles;
  const int h = blockIdx.y * kMergeHeads + (tid >> 5), d0 = (tid & 31) * 16;
  const int ub = unit_start(blockIdx.x + 1, a.units, a.ctas), r = ub / T;
  // no cut here, or not the row's first cut: nothing to do (the wait still orders this grid's end)
  if (ub == r * T || unit_start(blockIdx.x, a.units, a.ctas) > r * T) {
    pdl_wait();
    pdl_trigger();
    return;
  }
  __shared__ int span[3];
  if (tid == 0) {
    // the pieces of row r: CTAs c_first .. c_last.  The first piece sits in its CTA's first-row slot
    // only if that CTA's range starts in row r; every later piece starts its CTA's range.
    const int cf = cta_of_unit(r * T, a.units, a.ctas);
    span[0] = cf;
    span[1] = cta_of_unit(r * T + T - 1, a.units, a.ctas);
    span[2] = unit_start(cf, a.units, a.ctas) / T == r ? 2 * cf : 2 * cf + 1;
  }
  __syncthreads();
  const int c_first = span[0], c_last = span[1], first_slot = span[2];
  pdl_wait();
  pdl_trigger();
  constexpr int G = 2;
  float M = -INFINITY, L = 0.f;
  float acc[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0.f;
  for (int c0 = c_first; c0 <= c_last; c0 += G) {
    float mj[G], lj[G];
    float4 x[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int c = c0 + g;
      mj[g] = -INFINITY;
      lj[g] = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) x[g][q] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c <= c_last) {
        const int slot = c == c_first ? first_slot : 2 * c;
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.part_ml + ((int64_t)slot * kHeads + h) * 2));
        mj[g] = ml.x;
        lj[g] = ml.y;
        const float4* o = reinterpret_cast<const float4*>(a.part_o + ((int64_t)slot * kHeads + h) * kLatent + d0);
#pragma unroll
        for (int q = 0; q < 4; ++q) x[g][q] = __ldcg(o + q);
      }
    }
    float Mn = M;
#pragma unroll
    for (int g = 0; g < G; ++g)
      if (lj[g] > 0.f) Mn = fmaxf(Mn, mj[g]);
    if (Mn == -INFINITY) continue;
    const float sc = M == -INFINITY ? 0.f : expf(M - Mn);
    L *= sc;
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] *= sc;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float wgt = lj[g] > 0.f ? expf(mj[g] - Mn) : 0.f;
      L = fmaf(wgt, lj[g], L);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[4 * q] = fmaf(wgt, x[g][q].x, acc[4 * q]);
        acc[4 * q + 1] = fmaf(wgt, x[g][q].y, acc[4 * q + 1]);
        acc[4 * q + 2] = fmaf(wgt, x[g][q].z, acc[4 * q + 2]);
        acc[4 * q + 3] = fmaf(wgt, x[g][q].w, acc[4 * q + 3]);
      }
    }
    M = Mn;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  uint4 v[2];
  __nv_bfloat162* xo = reinterpret_cast<__nv_bfloat162*>(v);
#pragma unroll
  for (int e = 0; e < 8; ++e) xo[e] = __floats2bfloat162_rn(acc[2 * e] * inv, acc[2 * e + 1] * inv);
  uint4* dst = reinterpret_cast<uint4*>(a.out + ((int64_t)r * kHeads + h) * kLatent + d0);
  dst[0] = v[0];
  dst[1] = v[1];
  if (a.lse && (tid & 31) == 0) a.lse[(int64_t)r * kHeads + h] = L > 0.f ? M + logf(L) : -INFINITY;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {
struct MapKey {
  const void* ptr;
  uint64_t rows;
  bool operator==(const MapKey& o) const { return ptr == o.ptr && rows == o.rows; }
};
struct MapCache {
  std::mutex mu;
  MapKey key[16] = {};
  CUtensorMap map[16];
  int next = 0;
  // 2-D 16-bit tensor [rows, cols] with 2 cols-byte rows, box {64 columns, box_rows}
  bool get(const void* ptr, uint64_t rows, uint32_t box_rows, CUtensorMap* out, uint64_t cols = kRow) {
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < 16; ++i)
      if (key[i] == MapKey{ptr, rows} && key[i].ptr) {
        *out = map[i];
        return true;
      }
    CUtensorMap m;
    if (!encode_2d(&m, ptr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cols, rows, cols * 2, 64, box_rows)) return false;
    key[next] = MapKey{ptr, rows};
    map[next] = m;
    next = (next + 1) % 16;
    *out = m;
    return true;
  }
};
MapCache g_kv_maps, g_kv8_maps, g_q_maps;   // bf16 latent rows, packed 8-bit latent rows (640 bytes), queries
}  // namespace

MlaPlan plan_mla(int num_rows, int topk) {
  MlaPlan p;
  p.tiles = (topk + mla::kTok - 1) / mla::kTok;
  p.units = (int64_t)num_rows * p.tiles > INT32_MAX ? INT32_MAX : num_rows * p.tiles;
  p.ctas = p.units < kMlaCtas ? p.units : kMlaCtas;
  if (p.ctas < 1) p.ctas = 1;
  // few rows: S pieces per row in clusters of S (the largest power of two <= 8 with S R <= 152 and
  // S <= tiles); the workspace below is sized for the unit split either way
  p.split = 1;
  while (p.split < 8 && (int64_t)2 * p.split * num_rows <= kMlaCtas && 2 * p.split <= p.tiles) p.split *= 2;
  p.cta_err_offset = kWorkspaceHeader;
  p.part_offset = p.cta_err_offset + ((size_t)p.ctas * sizeof(uint32_t) + 255) / 256 * 256;
  p.workspace_bytes = p.part_offset + (size_t)2 * p.ctas * kHeads * (kLatent + 2) * sizeof(float);
  return p;
}

cudaError_t launch_sparse_mla(const dsa_cache* layers, int num_layers, const RowMeta& m, int num_rows, const void* q,
                              const int32_t* topk_idx, int topk, float scale, void* out, float* lse,
                              void* workspace, const MlaPlan& plan, cudaStream_t s, const int32_t* row_count) {
  static std::atomic<uint64_t> configured{0};
  cudaError_t set = once_per_device(configured, [] {
    cudaError_t e = cudaFuncSetAttribute(sparse_mla_tc_kernel<false, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         mla::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(sparse_mla_tc_kernel<false, kMlaMaxLayers>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               mla::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(sparse_mla_tc_kernel<true, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               mla::kSmemBytes);
    return e;
  });
  if (set != cudaSuccess) return set;
  if (num_layers < 1 || num_layers > kMlaMaxLayers) return cudaErrorInvalidValue;
  const dsa_cache& c = layers[0];              // the layers share page size, pool size and latent format
  const bool c8 = c.latent_format == DSA_LATENT_E4M3;
  if (c8 && num_layers > 1) return cudaErrorInvalidValue;   // one scale array per call
  const float* ls = c8 ? c.latent_scales : nullptr;
  MlaKvMaps<kMlaMaxLayers> kv_maps;
  CUtensorMap q_map;
  for (int l = 0; l < num_layers; ++l) {
    const dsa_cache& cl = layers[l];
    // a packed 8-bit row is 640 bytes: 320 16-bit columns, gathered as five 64-column pieces
    if (!(c8 ? g_kv8_maps.get(cl.latent, (uint64_t)cl.num_pages * cl.page_size, 1, &kv_maps.layer[l], 320)
             : g_kv_maps.get(cl.latent, (uint64_t)cl.num_pages * cl.page_size, 1, &kv_maps.layer[l])))
      return cudaErrorInvalidValue;
  }
  for (int l = num_layers; l < kMlaMaxLayers; ++l) kv_maps.layer[l] = kv_maps.layer[0];
  // the rows of every layer, stacked layer-major
  const int rows = num_rows * num_layers;
  if (!g_q_maps.get(q, (uint64_t)rows * kHeads, 64, &q_map)) return cudaErrorInvalidValue;
  uint32_t* err = static_cast<uint32_t*>(workspace);
  cudaError_t e = cudaSuccess;
  MlaArgs a;
  a.m = m;
  a.topk_idx = topk_idx;
  a.row_count = row_count;

  a.topk = topk;
  a.tiles = plan.tiles;
  a.units = plan.units;
  a.ctas = plan.split > 1 ? rows * plan.split : plan.ctas;
  a.split = plan.split;
  a.log2_page = ilog2(c.page_size);
  a.num_pages = c.num_pages;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.part_o = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.part_offset);
  a.part_ml = a.part_o + (size_t)2 * plan.ctas * kHeads * kLatent;
  a.cta_err = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + plan.cta_err_offset);
  a.err = err;
  {
    cudaLaunchConfig_t c = {};
    c.gridDim = dim3(a.ctas);
    c.blockDim = dim3(mla::kThreads);
    c.dynamicSmemBytes = mla::kSmemBytes;
    c.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = (unsigned)plan.split;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    c.attrs = at;
    c.numAttrs = plan.split > 1 ? 2 : 1;
    // prefill-like calls (at least 8 query rows per request on average): a request's rows select many of
    // the same cached rows, which keep their normal L2 priority (a 4096-row prefill chunk then reads
    // 1.7 GB from DRAM instead of 8.3 GB); with fewer rows per request (verify) evicting first is faster
    const int share = m.query_start_loc != nullptr && num_rows >= 8 * m.num_requests ? 1 : 0;
    MlaKvMaps<1> one_map;
    one_map.layer[0] = kv_maps.layer[0];
    e = c8               ? cudaLaunchKernelEx(&c, sparse_mla_tc_kernel<true, 1>, one_map, q_map, a, ls, share, num_rows)
        : num_layers > 1 ? cudaLaunchKernelEx(&c, sparse_mla_tc_kernel<false, kMlaMaxLayers>, kv_maps, q_map, a, ls,
                                              share, num_rows)
                         : cudaLaunchKernelEx(&c, sparse_mla_tc_kernel<false, 1>, one_map, q_map, a, ls, share, num_rows);
  }
  count_launches(1);
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (plan.split == 1) {
    // the merge may be scheduled while the attention grid drains (it waits for that grid's writes)
    if (a.ctas > 1) e = launch_pdl(mla_merge_kernel, dim3(a.ctas - 1, kHeads / kMergeHeads), dim3(512), 0, s, a);
    count_launches(1);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace dsa
