// Internal declarations shared by the CUDA translation units of libdsa.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include <atomic>

#include "../../include/dsa.h"

namespace dsa {

constexpr int kIndexHeads = DSA_INDEX_HEADS;   // 32
constexpr int kIndexDim = DSA_INDEX_DIM;       // 128
constexpr int kHeads = DSA_HEADS;              // 64
constexpr int kLatent = DSA_LATENT_DIM;        // 512
constexpr int kRope = DSA_ROPE_DIM;            // 64
constexpr int kRow = DSA_ROW_DIM;              // 576

// Persistent attention grid: one CTA per SM of a GB300 (152 SMs).
constexpr int kMlaCtas = 152;
// Upper bound on the fp32 score block the indexer materialises per launch group.
constexpr size_t kScoreBlockBytes = size_t(256) << 20;
constexpr size_t kWorkspaceHeader = 256;
// Top-k of long rows: positions per chunk CTA (at least), and candidates one chunk may keep.
constexpr int kTopkChunkMin = 32768;
constexpr int kTopkChunkCap = 4096;
constexpr int kTopkMaxChunks = 32;

// ---------------------------------------------------------------------------
// per-device host set-up
// ---------------------------------------------------------------------------
// The runtime applies a kernel's opt-in to more than 48 KB of dynamic shared memory to the current
// device only, so set-up of that kind runs once per device: bit d of `done` records device d.
// Concurrent first calls may both run `setup`, which must therefore be idempotent (setting a kernel
// attribute is).  Devices 64 and above run it on every call.
template <class Setup>
inline cudaError_t once_per_device(std::atomic<uint64_t>& done, Setup setup) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? uint64_t(1) << dev : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = setup();
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// SM count of the current device (persistent grids take one CTA per SM), looked up once per device.
inline int device_sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return kMlaCtas;
  const bool slot = dev >= 0 && dev < 64;
  if (slot) {
    const int n = cached[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = kMlaCtas;
  if (slot) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

// ---------------------------------------------------------------------------
// launch plans: shared by the *_workspace_bytes functions and the launches
// ---------------------------------------------------------------------------
struct IndexerPlan {
  int64_t score_stride;   // floats per row in the score block
  int rows_per_block;     // rows scored and selected per pass
  size_t groups_offset;   // int32 scratch: 4 counts, rows_per_block int4 groups, rows_per_block + 1 tile offsets
  size_t scores_offset;   // fp32 score block [rows_per_block][score_stride]
  int topk_chunk;         // rows longer than this are scanned for top-k candidates by one CTA per chunk
  int topk_chunks;        // chunks of the longest row (0: no row is split)
  size_t cand_offset;     // u64 candidate lists [rows_per_block][topk_chunks][kTopkChunkCap]
  size_t cand_cnt_offset; // u32 candidate counts [rows_per_block][topk_chunks]
  size_t workspace_bytes;
};
IndexerPlan plan_indexer(int num_rows, int max_seq_len, int topk);

struct MlaPlan {
  int tiles;              // 64-entry tiles per row of the index buffer
  int units;              // rows x tiles, split into one contiguous range per CTA
  int ctas;               // persistent CTAs of the unit split (at most one per SM)
  int split;              // > 1: pieces per row, one cluster of `split` CTAs per row (few rows)
  size_t cta_err_offset;  // u32 timeout bits per CTA, after the 256-byte header (status word first)
  size_t part_offset;     // two (64 x 512 + 64 x 2) fp32 partial slots per CTA
  size_t workspace_bytes;
};
MlaPlan plan_mla(int num_rows, int topk);

// Counts every kernel launch the library issues (reported by dsa_kernel_launches).
void count_launches(int n);

// Workspace header (the first kWorkspaceHeader bytes of every workspace, and of the static scratch):
// word 0 holds the call's call-wide status bits, word 1 the number of per-CTA status words that
// follow at byte kWorkspaceHeader (attention calls; 0 for the indexer).  dsa_read_status ORs them.
constexpr int kStatusCtaWords = kWorkspaceHeader / 4;   // index of the first per-CTA word

// Device address of the static scratch array on the current device (looked up on first use).
dsa_status static_scratch_of_current_device(void** out);

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the library is launched as a programmatic
// dependent of the kernel before it in the stream, so that its launch and its prologue overlap that
// kernel's tail.  Each kernel keeps one contract: every CTA calls pdl_wait() (which returns once
// the preceding grid has completed and its writes are visible) before it reads any input memory
// or exits, and calls pdl_trigger() (if at all: without it the next grid starts when this one
// completes) only after its own pdl_wait().  A grid can then start only when its predecessor has
// passed its wait, so every grid before that predecessor has completed; a grid completes only
// after its predecessor has.  (Both are no-ops in a plain launch.)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}
dsa_status report_error(dsa_status st, const char* msg);

// ---------------------------------------------------------------------------
// launchers (defined next to their kernels)
// ---------------------------------------------------------------------------
// one layer's side of an append (device pointers; k_idx NULL for a layer without index keys)
struct AppendLayer {
  uint4* latent;
  int64_t total_slots;
  uint8_t* index_keys;
  float* index_scales;
  float* latent_scales;
  int key_format, latent_format;
  const uint4* c_kv;
  const uint4* k_rope;
  const uint8_t* k_idx;
  int k_idx_format;
  const float* k_idx_scales;
};
constexpr int kMaxAppendLayers = 16;
struct AppendArgs {
  AppendLayer layer[kMaxAppendLayers];
  const int64_t* slot_mapping;
  int num_tokens;
};
AppendLayer append_layer(const dsa_cache& c, const void* c_kv, const void* k_rope, const void* k_idx, int k_idx_format,
                         const float* k_idx_scales);
cudaError_t launch_kv_append(const AppendArgs& a, int num_layers, cudaStream_t s);

struct RowMeta {
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* query_start_loc;   // nullptr: decode (row r = request r)
  int32_t num_requests;
  int32_t block_table_stride;
};

// Scores of rows [row0, row0 + nrows) into scores[(r - row0) * score_stride + s].  group_scratch holds
// 4 + 5 * nrows + 1 ints; err is the device status word; fill_tail writes -inf past each row's last key tile.
// page_log2 >= 0: page mode, one score per unit of 2^min(page_log2, 5) keys: the page itself for pages of
// up to 32 keys, else a part that launch_page_pool combines (pages of at most 128 keys)
cudaError_t launch_indexer_scores(const dsa_cache& c, const RowMeta& m, int row0, int nrows, int max_seq_len,
                                  const void* q_idx, const float* w, float* scores, int64_t score_stride,
                                  bool fill_tail, int32_t* group_scratch, uint32_t* err, cudaStream_t s,
                                  int page_log2 = -1);

struct TopkChunks {
  int chunk = 0, chunks = 0;   // chunks == 0: every row is selected by one CTA
  uint64_t* cand = nullptr;    // [nrows][chunks][kTopkChunkCap] (key << 32 | position)
  uint32_t* cnt = nullptr;     // [nrows][chunks]; 0xFFFFFFFF marks an overflowed chunk
};
// unit_shift > 0: the scores are page scores, a row's visible units are pages 0 .. pos >> unit_shift
cudaError_t launch_topk(const RowMeta& m, int row0, int nrows, const float* scores, int64_t score_stride,
                        int max_seq_len, int topk, int32_t* topk_idx, const TopkChunks& ch, cudaStream_t s,
                        int unit_shift = 0);
cudaError_t launch_page_pool(const RowMeta& m, int row0, int nrows, const float* units, int64_t unit_stride,
                             int page_log2, float* pages, int64_t page_stride, int max_pages, cudaStream_t s);
cudaError_t launch_page_expand(const RowMeta& m, int row0, int nrows, const int32_t* page_idx, int kp, int page_log2,
                               int32_t* token_idx, cudaStream_t s);

// layers[0 .. num_layers) share one index buffer, page size, pool size and latent format; q, out and
// lse hold num_layers * num_rows rows, layer-major; plan is plan_mla(num_layers * num_rows, topk).
// A packed 8-bit latent takes one layer per call.
constexpr int kMlaMaxLayers = 4;
cudaError_t launch_sparse_mla(const dsa_cache* layers, int num_layers, const RowMeta& m, int num_rows, const void* q,
                              const int32_t* topk_idx, int topk, float scale, void* out, float* lse,
                              void* workspace, const MlaPlan& plan, cudaStream_t s,
                              const int32_t* row_count = nullptr);

cudaError_t launch_dcp_candidates(const float* local_scores, int64_t stride, const int32_t* local_idx, int k, int rows,
                                  int rank, int world, float* cand_score, int32_t* cand_pos, cudaStream_t s);
cudaError_t launch_dcp_select(const float* cand_score, const int32_t* cand_pos, int world, int rows, int k, int rank,
                              int32_t* global_idx, int32_t* local_idx, int32_t* local_count, cudaStream_t s);
cudaError_t launch_dcp_merge(const void* outs, const float* lses, int world, int rows, void* out, float* lse,
                             cudaStream_t s);

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
// Request and absolute position of query row r: row i of request b sits at L_b - q_len_b + i.
__device__ __forceinline__ void row_info(const RowMeta& m, int r, int& b, int& pos) {
  if (m.query_start_loc == nullptr) {
    b = r;
    pos = m.seq_lens[r] - 1;
    return;
  }
  int lo = 0, hi = m.num_requests - 1;   // largest b with query_start_loc[b] <= r
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (m.query_start_loc[mid] <= r) lo = mid; else hi = mid - 1;
  }
  b = lo;
  int q_len = m.query_start_loc[b + 1] - m.query_start_loc[b];
  pos = m.seq_lens[b] - q_len + (r - m.query_start_loc[b]);
}

// Physical slot of logical position s of request b, or -1 when the page table or page id is out of range.
__device__ __forceinline__ int64_t token_slot(const RowMeta& m, int b, int s, int log2_page, int num_pages) {
  int lp = s >> log2_page;
  if (s < 0 || lp >= m.block_table_stride) return -1;
  int page = m.block_table[(int64_t)b * m.block_table_stride + lp];
  if (page < 0 || page >= num_pages) return -1;
  return ((int64_t)page << log2_page) + (s & ((1 << log2_page) - 1));
}

__host__ __device__ inline int ilog2(int x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}

}  // namespace dsa
