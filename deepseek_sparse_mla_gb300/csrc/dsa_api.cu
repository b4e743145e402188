// Host side of libdsa: the C ABI entry points of include/dsa.h.
//
// Every entry point validates its arguments on the host, sizes nothing
// dynamically, allocates nothing and never synchronises: it records launches
// on the caller's stream.  Launch plans are pure functions of the shape, so the
// workspace sizes reported to the caller are exactly what the launches use.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "dsa_internal.cuh"

namespace dsa {

static thread_local std::string g_last_error;
static std::atomic<uint64_t> g_launches{0};

void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

static dsa_status fail(dsa_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

static dsa_status ok() { return DSA_OK; }

// Records a message for dsa_last_error() from the library's other translation units.
dsa_status report_error(dsa_status st, const char* msg) { return fail(st, "%s", msg); }

static dsa_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(DSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// dsa_read_status: the OR of a workspace header's call-wide word and its per-CTA words (one warp).
__global__ void __launch_bounds__(32) status_read_kernel(const uint32_t* ws, uint32_t* out) {
  pdl_wait();
  pdl_trigger();
  const uint32_t n = min(__ldcg(ws + 1), (uint32_t)kMlaCtas);
  uint32_t bits = threadIdx.x == 0 ? __ldcg(ws) : 0u;
  for (uint32_t c = threadIdx.x; c < n; c += 32) bits |= __ldcg(ws + kStatusCtaWords + c);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) bits |= __shfl_xor_sync(0xffffffffu, bits, o);
  if (threadIdx.x == 0) *out = bits;
}

static bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

IndexerPlan plan_indexer(int num_rows, int max_seq_len, int topk) {
  IndexerPlan p;
  p.score_stride = ((int64_t)max_seq_len + 255) / 256 * 256;
  int64_t per_row = p.score_stride * (int64_t)sizeof(float);
  int64_t fit = (int64_t)kScoreBlockBytes / per_row;
  if (fit < 1) fit = 1;
  p.rows_per_block = (int)(num_rows < fit ? num_rows : fit);
  if (p.rows_per_block < 1) p.rows_per_block = 1;
  p.groups_offset = kWorkspaceHeader;
  p.scores_offset = p.groups_offset + ((size_t)(4 + 5 * p.rows_per_block + 1) * sizeof(int32_t) + 255) / 256 * 256;
  size_t end = p.scores_offset + (size_t)p.rows_per_block * (size_t)per_row;
  // top-k of rows longer than one chunk: one candidate list per chunk, at most kTopkMaxChunks chunks
  int64_t chunk = (int64_t)16 * topk > kTopkChunkMin ? (int64_t)16 * topk : kTopkChunkMin;
  if ((max_seq_len + chunk - 1) / chunk > kTopkMaxChunks) chunk = ((int64_t)max_seq_len + kTopkMaxChunks - 1) / kTopkMaxChunks;
  chunk = (chunk + 1023) / 1024 * 1024;
  p.topk_chunk = (int)chunk;
  p.topk_chunks = max_seq_len > chunk ? (int)((max_seq_len + chunk - 1) / chunk) : 0;
  p.cand_offset = (end + 255) / 256 * 256;
  p.cand_cnt_offset = p.cand_offset + (size_t)p.rows_per_block * p.topk_chunks * kTopkChunkCap * sizeof(uint64_t);
  p.workspace_bytes = p.cand_cnt_offset + (size_t)p.rows_per_block * p.topk_chunks * sizeof(uint32_t);
  return p;
}

static dsa_status check_cache(const dsa_cache* c, bool need_keys) {
  if (!c) return fail(DSA_ERR_INVALID_ARG, "cache is NULL");
  if (!c->latent) return fail(DSA_ERR_INVALID_ARG, "cache.latent is NULL");
  if (!aligned16(c->latent)) return fail(DSA_ERR_INVALID_ARG, "cache.latent is not 16-byte aligned");
  if (c->num_pages <= 0) return fail(DSA_ERR_INVALID_ARG, "cache.num_pages must be positive (got %d)", c->num_pages);
  if (!pow2(c->page_size) || c->page_size > 1024)
    return fail(DSA_ERR_INVALID_ARG, "cache.page_size must be a power of two in 1..1024 (got %d)", c->page_size);
  if ((int64_t)c->num_pages * c->page_size > (int64_t)INT32_MAX)
    return fail(DSA_ERR_UNSUPPORTED, "cache holds more than 2^31 slots");
  if (c->latent_format != DSA_LATENT_BF16 && c->latent_format != DSA_LATENT_E4M3)
    return fail(DSA_ERR_INVALID_ARG, "cache.latent_format %d is not a dsa_latent_format", c->latent_format);
  if (c->latent_format == DSA_LATENT_E4M3 && !c->latent_scales)
    return fail(DSA_ERR_INVALID_ARG, "an e4m3 latent cache needs cache.latent_scales");
  if (c->latent_format == DSA_LATENT_BF16 && c->latent_scales)
    return fail(DSA_ERR_INVALID_ARG, "a bf16 latent cache takes no cache.latent_scales (layouts are not interchangeable)");
  if (c->latent_scales && (reinterpret_cast<uintptr_t>(c->latent_scales) & 15u))
    return fail(DSA_ERR_INVALID_ARG, "cache.latent_scales is not 16-byte aligned");
  if (c->index_keys) {
    if (c->key_format != DSA_KEY_BF16 && c->key_format != DSA_KEY_FP8_E4M3 && c->key_format != DSA_KEY_INT8)
      return fail(DSA_ERR_INVALID_ARG, "cache.key_format %d is not a dsa_key_format", c->key_format);
    if (!aligned16(c->index_keys)) return fail(DSA_ERR_INVALID_ARG, "cache.index_keys is not 16-byte aligned");
    if (c->key_format == DSA_KEY_FP8_E4M3 && !c->index_scales)
      return fail(DSA_ERR_INVALID_ARG, "e4m3 index keys need cache.index_scales");
    if (c->key_format == DSA_KEY_INT8 && !c->index_scales)
      return fail(DSA_ERR_INVALID_ARG, "int8 index keys need cache.index_scales (binary16)");
    if (c->key_format == DSA_KEY_BF16 && c->index_scales)
      return fail(DSA_ERR_INVALID_ARG, "bf16 index keys take no cache.index_scales (layouts are not interchangeable)");
    if (c->index_scales && (reinterpret_cast<uintptr_t>(c->index_scales) & 15u))
      return fail(DSA_ERR_INVALID_ARG, "cache.index_scales is not 16-byte aligned");
  } else if (need_keys) {
    return fail(DSA_ERR_INVALID_ARG,
                "layer has no indexer keys (cache.index_keys is NULL): a shared layer must reuse the owner's "
                "index buffer instead of scoring");
  }
  return ok();
}

static dsa_status check_batch(const dsa_batch* b, bool need_qsl) {
  if (!b) return fail(DSA_ERR_INVALID_ARG, "batch is NULL");
  if (b->num_requests <= 0) return fail(DSA_ERR_INVALID_ARG, "batch.num_requests must be positive");
  if (b->num_rows < 0) return fail(DSA_ERR_INVALID_ARG, "batch.num_rows is negative");
  if (b->max_seq_len <= 0) return fail(DSA_ERR_INVALID_ARG, "batch.max_seq_len must be positive");
  if (!b->block_table || !b->seq_lens) return fail(DSA_ERR_INVALID_ARG, "batch.block_table / seq_lens is NULL");
  if (b->block_table_stride <= 0) return fail(DSA_ERR_INVALID_ARG, "batch.block_table_stride must be positive");
  if (need_qsl && !b->query_start_loc)
    return fail(DSA_ERR_INVALID_ARG, "batch.query_start_loc is required when requests have several rows");
  if (!b->query_start_loc && b->num_rows != b->num_requests)
    return fail(DSA_ERR_INVALID_ARG, "without query_start_loc every request has exactly one row (num_rows %d != "
                "num_requests %d)", b->num_rows, b->num_requests);
  return ok();
}

static RowMeta row_meta(const dsa_batch* b, bool decode) {
  RowMeta m;
  m.block_table = b->block_table;
  m.seq_lens = b->seq_lens;
  m.query_start_loc = decode ? nullptr : b->query_start_loc;
  m.num_requests = b->num_requests;
  m.block_table_stride = b->block_table_stride;
  return m;
}

static dsa_status sparse_mla_common(const dsa_cache* layer, const dsa_batch* batch, const void* q,
                                    const int32_t* topk_idx, int32_t topk, float scale, void* out, float* lse,
                                    void* workspace, size_t workspace_bytes, void* stream, bool decode,
                                    const int32_t* row_counts = nullptr, int num_layers = 1) {
  if (!layer) return fail(DSA_ERR_INVALID_ARG, "cache is NULL");
  if (num_layers < 1 || num_layers > kMlaMaxLayers)
    return fail(DSA_ERR_UNSUPPORTED, "num_layers %d outside 1..%d", num_layers, kMlaMaxLayers);
  for (int l = 0; l < num_layers; ++l) {
    dsa_status st = check_cache(&layer[l], false);
    if (st != DSA_OK) return num_layers > 1 ? fail(st, "layer %d: %s", l, dsa_last_error()) : st;
    if (layer[l].page_size != layer[0].page_size || layer[l].num_pages != layer[0].num_pages ||
        layer[l].latent_format != layer[0].latent_format)
      return fail(DSA_ERR_INVALID_ARG, "layer %d: page size, page count and latent format must match layer 0's", l);
  }
  dsa_status st = check_batch(batch, !decode);
  if (st != DSA_OK) return st;
  if (!topk_idx)
    return fail(DSA_ERR_INVALID_ARG, "topk_idx is NULL: a shared layer must be given the owner layer's index buffer");
  if (topk < 1 || topk > DSA_MAX_TOPK) return fail(DSA_ERR_INVALID_ARG, "topk must be in 1..%d (got %d)", DSA_MAX_TOPK, topk);
  if (!q || !out) return fail(DSA_ERR_INVALID_ARG, "q / out is NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(DSA_ERR_INVALID_ARG, "q / out is not 16-byte aligned");
  if (!(scale > 0.f) || scale != scale || scale > 1e30f) return fail(DSA_ERR_INVALID_ARG, "scale must be finite and positive");
  if (decode && batch->num_rows != batch->num_requests)
    return fail(DSA_ERR_INVALID_ARG, "decode takes one row per request (num_rows %d, num_requests %d)",
                batch->num_rows, batch->num_requests);
  if (batch->num_rows == 0) return ok();
  if ((int64_t)num_layers * batch->num_rows > INT32_MAX / kHeads)
    return fail(DSA_ERR_UNSUPPORTED, "num_layers * num_rows is too large");
  MlaPlan plan = plan_mla(num_layers * batch->num_rows, topk);
  if (plan.workspace_bytes > 0 && (!workspace || workspace_bytes < plan.workspace_bytes))
    return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu bytes dsa_mla_workspace_bytes requires",
                workspace_bytes, plan.workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(DSA_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  RowMeta m = row_meta(batch, decode);
  if (num_layers > 1 && layer[0].latent_format == DSA_LATENT_E4M3) {
    // a packed 8-bit latent carries one scale array per layer: one call per layer, in order, on the
    // same workspace (the stream orders them)
    const size_t rows = (size_t)batch->num_rows;
    const MlaPlan one = plan_mla(batch->num_rows, topk);
    for (int l = 0; l < num_layers; ++l) {
      cudaError_t e = launch_sparse_mla(&layer[l], 1, m, batch->num_rows,
                                        static_cast<const char*>(q) + l * rows * kHeads * kRow * 2, topk_idx, topk,
                                        scale, static_cast<char*>(out) + l * rows * kHeads * kLatent * 2,
                                        lse ? lse + l * rows * kHeads : nullptr, workspace, one, (cudaStream_t)stream);
      if (e != cudaSuccess) return cuda_status(e, "sparse MLA launch");
    }
    return ok();
  }
  cudaError_t e = launch_sparse_mla(layer, num_layers, m, batch->num_rows, q, topk_idx, topk, scale, out, lse, workspace,
                                    plan, (cudaStream_t)stream, row_counts);
  return cuda_status(e, "sparse MLA launch");
}

}  // namespace dsa

using namespace dsa;

extern "C" {

int32_t dsa_abi_version(void) { return DSA_ABI_VERSION; }

const char* dsa_last_error(void) { return g_last_error.c_str(); }

dsa_status dsa_read_status(const void* workspace, uint32_t* status_out, void* stream) {
  if (!status_out) return fail(DSA_ERR_INVALID_ARG, "status_out is NULL");
  if (reinterpret_cast<uintptr_t>(status_out) & 3u) return fail(DSA_ERR_INVALID_ARG, "status_out is not 4-byte aligned");
  const void* ws = workspace;
  if (!ws) {
    void* scratch = nullptr;
    const dsa_status st = static_scratch_of_current_device(&scratch);
    if (st != DSA_OK) return st;
    ws = scratch;
  } else if (reinterpret_cast<uintptr_t>(ws) & 255u) {
    return fail(DSA_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  }
  cudaError_t e = launch_pdl(status_read_kernel, dim3(1), dim3(32), 0, (cudaStream_t)stream,
                             static_cast<const uint32_t*>(ws), status_out);
  count_launches(1);
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_status(e, "status read launch");
}

dsa_status dsa_check_device_status(uint32_t bits) {
  if (bits == 0) return DSA_OK;
  std::string names;
  const struct { uint32_t bit; const char* name; } known[] = {
      {DSA_DEVICE_TMA_TIMEOUT, "DSA_DEVICE_TMA_TIMEOUT"}, {DSA_DEVICE_MMA_TIMEOUT, "DSA_DEVICE_MMA_TIMEOUT"},
      {DSA_DEVICE_BAD_PAGE, "DSA_DEVICE_BAD_PAGE"}, {DSA_DEVICE_CONFIG, "DSA_DEVICE_CONFIG"}};
  uint32_t rest = bits;
  for (const auto& k : known)
    if (bits & k.bit) {
      names += names.empty() ? "" : " | ";
      names += k.name;
      rest &= ~k.bit;
    }
  if (rest) {
    char buf[32];
    snprintf(buf, sizeof(buf), "%s0x%x", names.empty() ? "" : " | ", rest);
    names += buf;
  }
  return fail(DSA_ERR_DEVICE_CHECK, "device status 0x%x: %s", bits, names.c_str());
}

uint64_t dsa_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

size_t dsa_cache_bytes(int32_t num_pages, int32_t page_size, int32_t key_format, int32_t owner,
                       int32_t latent_format) {
  if (num_pages <= 0 || page_size <= 0) return 0;
  size_t slots = (size_t)num_pages * (size_t)page_size;
  size_t bytes;
  if (latent_format == DSA_LATENT_BF16) bytes = slots * kRow * 2;
  else if (latent_format == DSA_LATENT_E4M3) bytes = slots * (kLatent + kRope * 2 + sizeof(float));
  else return 0;
  if (owner) {
    if (key_format == DSA_KEY_BF16) bytes += slots * kIndexDim * 2;
    else if (key_format == DSA_KEY_FP8_E4M3) bytes += slots * (kIndexDim + sizeof(float));
    else if (key_format == DSA_KEY_INT8) bytes += slots * (kIndexDim + 2);
    else return 0;
  }
  return bytes;
}

size_t dsa_indexer_workspace_bytes(int32_t num_rows, int32_t max_seq_len, int32_t topk) {
  if (num_rows < 0 || max_seq_len <= 0 || topk < 1) return 0;
  return plan_indexer(num_rows > 0 ? num_rows : 1, max_seq_len, topk).workspace_bytes;
}

size_t dsa_mla_workspace_bytes(int32_t num_rows, int32_t topk) {
  if (num_rows < 0 || topk < 1) return 0;
  return plan_mla(num_rows > 0 ? num_rows : 1, topk).workspace_bytes;
}

static dsa_status check_append_layer(const dsa_cache* cache, const void* c_kv, const void* k_rope, const void* k_idx,
                                     int32_t k_idx_format, const float* k_idx_scales) {
  dsa_status st = check_cache(cache, false);
  if (st != DSA_OK) return st;
  if (!c_kv || !k_rope) return fail(DSA_ERR_INVALID_ARG, "c_kv / k_rope is NULL");
  if (!aligned16(c_kv) || !aligned16(k_rope)) return fail(DSA_ERR_INVALID_ARG, "c_kv / k_rope is not 16-byte aligned");
  if (cache->index_keys) {
    if (!k_idx) return fail(DSA_ERR_INVALID_ARG, "this layer owns an indexer cache: k_idx is required");
    if (!aligned16(k_idx)) return fail(DSA_ERR_INVALID_ARG, "k_idx is not 16-byte aligned");
    if (k_idx_format == DSA_KEY_FP8_E4M3) {
      if (cache->key_format != DSA_KEY_FP8_E4M3)
        return fail(DSA_ERR_INVALID_ARG, "e4m3 index keys can only be stored into an e4m3 indexer cache");
      if (!k_idx_scales) return fail(DSA_ERR_INVALID_ARG, "pre-quantised e4m3 keys need k_idx_scales");
      if (reinterpret_cast<uintptr_t>(k_idx_scales) & 3u) return fail(DSA_ERR_INVALID_ARG, "k_idx_scales is not 4-byte aligned");
    } else if (k_idx_format == DSA_KEY_INT8) {
      if (cache->key_format != DSA_KEY_INT8)
        return fail(DSA_ERR_INVALID_ARG, "int8 index keys can only be stored into an int8 indexer cache");
      if (!k_idx_scales) return fail(DSA_ERR_INVALID_ARG, "pre-quantised int8 keys need k_idx_scales (binary16)");
      if (reinterpret_cast<uintptr_t>(k_idx_scales) & 1u) return fail(DSA_ERR_INVALID_ARG, "k_idx_scales is not 2-byte aligned");
    } else if (k_idx_format != DSA_KEY_BF16) {
      return fail(DSA_ERR_INVALID_ARG, "k_idx_format %d is not a dsa_key_format", k_idx_format);
    }
  } else if (k_idx) {
    return fail(DSA_ERR_INVALID_ARG, "k_idx given for a layer without an indexer cache (cache.index_keys is NULL)");
  }
  return ok();
}

dsa_status dsa_kv_append(const dsa_cache* cache, const void* c_kv, const void* k_rope, const void* k_idx,
                         int32_t k_idx_format, const float* k_idx_scales, const int64_t* slot_mapping,
                         int32_t num_tokens, void* stream) {
  return dsa_kv_append_layers(cache, 1, &c_kv, &k_rope, &k_idx, k_idx_format, &k_idx_scales, slot_mapping, num_tokens,
                              stream);
}

dsa_status dsa_kv_append_layers(const dsa_cache* caches, int32_t num_layers, const void* const* c_kv,
                                const void* const* k_rope, const void* const* k_idx, int32_t k_idx_format,
                                const float* const* k_idx_scales, const int64_t* slot_mapping, int32_t num_tokens,
                                void* stream) {
  if (!caches || !c_kv || !k_rope) return fail(DSA_ERR_INVALID_ARG, "caches / c_kv / k_rope is NULL");
  if (num_layers < 1 || num_layers > kMaxAppendLayers)
    return fail(DSA_ERR_UNSUPPORTED, "num_layers %d outside 1..%d", num_layers, kMaxAppendLayers);
  if (num_tokens < 0) return fail(DSA_ERR_INVALID_ARG, "num_tokens is negative");
  for (int l = 0; l < num_layers; ++l) {
    dsa_status st = check_cache(&caches[l], false);
    if (st != DSA_OK) return st;
  }
  if (num_tokens == 0) return ok();                  // a no-op once the caches are valid
  AppendArgs args = {};
  for (int l = 0; l < num_layers; ++l) {
    const void* ki = k_idx ? k_idx[l] : nullptr;
    const float* ks = k_idx_scales ? k_idx_scales[l] : nullptr;
    dsa_status st = check_append_layer(&caches[l], c_kv[l], k_rope[l], ki, k_idx_format, ks);
    if (st != DSA_OK) return num_layers > 1 ? fail(st, "layer %d: %s", l, dsa_last_error()) : st;
    args.layer[l] = append_layer(caches[l], c_kv[l], k_rope[l], caches[l].index_keys ? ki : nullptr, k_idx_format, ks);
  }
  if (!slot_mapping) return fail(DSA_ERR_INVALID_ARG, "slot_mapping is NULL");
  if (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) return fail(DSA_ERR_INVALID_ARG, "slot_mapping is not 8-byte aligned");
  args.slot_mapping = slot_mapping;
  args.num_tokens = num_tokens;
  cudaError_t e = launch_kv_append(args, num_layers, (cudaStream_t)stream);
  return cuda_status(e, "kv append launch");
}

dsa_status dsa_indexer_scores_topk(const dsa_cache* owner, const dsa_batch* batch, const void* q_idx, const float* w,
                                   int32_t topk, int32_t* topk_idx, float* scores_out, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  dsa_status st = check_cache(owner, true);
  if (st != DSA_OK) return st;
  st = check_batch(batch, false);
  if (st != DSA_OK) return st;
  if (topk < 1 || topk > DSA_MAX_TOPK) return fail(DSA_ERR_INVALID_ARG, "topk must be in 1..%d (got %d)", DSA_MAX_TOPK, topk);
  if (!q_idx || !w || !topk_idx) return fail(DSA_ERR_INVALID_ARG, "q_idx / w / topk_idx is NULL");
  if (!aligned16(q_idx)) return fail(DSA_ERR_INVALID_ARG, "q_idx is not 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(w) & 3u) || (reinterpret_cast<uintptr_t>(topk_idx) & 3u) ||
      (reinterpret_cast<uintptr_t>(scores_out) & 3u))
    return fail(DSA_ERR_INVALID_ARG, "w / topk_idx / scores_out is not 4-byte aligned");
  if (batch->num_rows == 0) return ok();
  IndexerPlan plan = plan_indexer(batch->num_rows, batch->max_seq_len, topk);
  if (!workspace || workspace_bytes < plan.workspace_bytes)
    return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu bytes dsa_indexer_workspace_bytes requires",
                workspace_bytes, plan.workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(DSA_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  RowMeta m = row_meta(batch, batch->query_start_loc == nullptr);
  cudaStream_t s = (cudaStream_t)stream;
  char* ws = static_cast<char*>(workspace);
  uint32_t* err = reinterpret_cast<uint32_t*>(ws);
  int32_t* groups = reinterpret_cast<int32_t*>(ws + plan.groups_offset);
  float* block = reinterpret_cast<float*>(ws + plan.scores_offset);
  TopkChunks chunks;
  chunks.chunk = plan.topk_chunk;
  chunks.chunks = plan.topk_chunks;
  chunks.cand = reinterpret_cast<uint64_t*>(ws + plan.cand_offset);
  chunks.cnt = reinterpret_cast<uint32_t*>(ws + plan.cand_cnt_offset);
  // the status word is cleared on the device by the first row block's group-table kernel
  for (int row0 = 0; row0 < batch->num_rows; row0 += plan.rows_per_block) {
    int n = batch->num_rows - row0 < plan.rows_per_block ? batch->num_rows - row0 : plan.rows_per_block;
    float* scores = scores_out ? scores_out + (int64_t)row0 * batch->max_seq_len : block;
    int64_t stride = scores_out ? (int64_t)batch->max_seq_len : plan.score_stride;
    cudaError_t e = launch_indexer_scores(*owner, m, row0, n, batch->max_seq_len, q_idx, w, scores, stride,
                                          scores_out != nullptr, groups, err, s);
    if (e != cudaSuccess) return cuda_status(e, "indexer launch");
    e = launch_topk(m, row0, n, scores, stride, batch->max_seq_len, topk, topk_idx, chunks, s);
    if (e != cudaSuccess) return cuda_status(e, "top-k launch");
  }
  return ok();
}

// Page mode workspace: the indexer plan over units of min(P, 32) keys (its score block holds the
// units' maxima) and, for pages of more than 32 keys, a page-score block after it.
namespace {
struct PagePlan {
  IndexerPlan ix;
  int max_units, max_pages;
  bool pooled;
  int64_t page_stride;
  size_t pages_offset, workspace_bytes;
};
PagePlan plan_pages(int num_rows, int max_seq_len, int page_size, int page_budget) {
  PagePlan p;
  const int unit = page_size < 32 ? page_size : 32;
  p.max_units = (int)(((int64_t)max_seq_len + unit - 1) / unit);
  p.max_pages = (int)(((int64_t)max_seq_len + page_size - 1) / page_size);
  p.pooled = page_size > 32;
  p.ix = plan_indexer(num_rows, p.max_units, page_budget);
  p.page_stride = ((int64_t)p.max_pages + 255) / 256 * 256;
  p.pages_offset = (p.ix.workspace_bytes + 255) / 256 * 256;
  p.workspace_bytes = p.pooled ? p.pages_offset + (size_t)p.ix.rows_per_block * p.page_stride * sizeof(float)
                               : p.ix.workspace_bytes;
  return p;
}
}  // namespace

size_t dsa_indexer_page_workspace_bytes(int32_t num_rows, int32_t max_seq_len, int32_t page_size, int32_t page_budget) {
  if (num_rows < 0 || max_seq_len <= 0 || page_size <= 0 || page_budget < 1) return 0;
  return plan_pages(num_rows > 0 ? num_rows : 1, max_seq_len, page_size, page_budget).workspace_bytes;
}

dsa_status dsa_indexer_page_topk(const dsa_cache* owner, const dsa_batch* batch, const void* q_idx, const float* w,
                                 int32_t page_budget, int32_t* page_idx, int32_t* token_idx, float* page_scores_out,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  dsa_status st = check_cache(owner, true);
  if (st != DSA_OK) return st;
  st = check_batch(batch, false);
  if (st != DSA_OK) return st;
  const int P = owner->page_size;
  if (P > 128)
    return fail(DSA_ERR_UNSUPPORTED, "page-granular selection needs pages of at most 128 keys (got %d)", P);
  if (page_budget < 1 || page_budget > DSA_MAX_TOPK)
    return fail(DSA_ERR_INVALID_ARG, "page_budget must be in 1..%d (got %d)", DSA_MAX_TOPK, page_budget);
  if (token_idx && (int64_t)page_budget * P > DSA_MAX_TOPK)
    return fail(DSA_ERR_INVALID_ARG, "page_budget * page_size = %lld positions exceeds DSA_MAX_TOPK (%d)",
                (long long)page_budget * P, DSA_MAX_TOPK);
  if (!q_idx || !w || !page_idx) return fail(DSA_ERR_INVALID_ARG, "q_idx / w / page_idx is NULL");
  if (!aligned16(q_idx)) return fail(DSA_ERR_INVALID_ARG, "q_idx is not 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(w) & 3u) || (reinterpret_cast<uintptr_t>(page_idx) & 3u) ||
      (reinterpret_cast<uintptr_t>(token_idx) & 3u) || (reinterpret_cast<uintptr_t>(page_scores_out) & 3u))
    return fail(DSA_ERR_INVALID_ARG, "w / page_idx / token_idx / page_scores_out is not 4-byte aligned");
  if (batch->num_rows == 0) return ok();
  const int log2p = ilog2(P);
  const PagePlan pp = plan_pages(batch->num_rows, batch->max_seq_len, P, page_budget);
  const IndexerPlan& plan = pp.ix;
  const int max_pages = pp.max_pages;
  if (!workspace || workspace_bytes < pp.workspace_bytes)
    return fail(DSA_ERR_WORKSPACE,
                "workspace of %zu bytes is smaller than the %zu bytes dsa_indexer_page_workspace_bytes requires",
                workspace_bytes, pp.workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(DSA_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  RowMeta m = row_meta(batch, batch->query_start_loc == nullptr);
  cudaStream_t s = (cudaStream_t)stream;
  char* ws = static_cast<char*>(workspace);
  uint32_t* err = reinterpret_cast<uint32_t*>(ws);
  int32_t* groups = reinterpret_cast<int32_t*>(ws + plan.groups_offset);
  float* block = reinterpret_cast<float*>(ws + plan.scores_offset);
  float* page_block = reinterpret_cast<float*>(ws + pp.pages_offset);
  TopkChunks chunks;
  chunks.chunk = plan.topk_chunk;
  chunks.chunks = plan.topk_chunks;
  chunks.cand = reinterpret_cast<uint64_t*>(ws + plan.cand_offset);
  chunks.cnt = reinterpret_cast<uint32_t*>(ws + plan.cand_cnt_offset);
  for (int row0 = 0; row0 < batch->num_rows; row0 += plan.rows_per_block) {
    int n = batch->num_rows - row0 < plan.rows_per_block ? batch->num_rows - row0 : plan.rows_per_block;
    // pages of up to 32 keys: the indexer writes page scores itself (into page_scores_out if given);
    // larger pages: it writes 32-key unit maxima into the workspace, pooled into page scores next
    float* pages = page_scores_out ? page_scores_out + (int64_t)row0 * max_pages : (pp.pooled ? page_block : block);
    int64_t page_stride = page_scores_out ? (int64_t)max_pages : (pp.pooled ? pp.page_stride : plan.score_stride);
    float* units = pp.pooled ? block : pages;
    int64_t unit_stride = pp.pooled ? plan.score_stride : page_stride;
    cudaError_t e = launch_indexer_scores(*owner, m, row0, n, batch->max_seq_len, q_idx, w, units, unit_stride,
                                          !pp.pooled && page_scores_out != nullptr, groups, err, s, log2p);
    if (e != cudaSuccess) return cuda_status(e, "indexer launch");
    if (pp.pooled) {
      e = launch_page_pool(m, row0, n, units, unit_stride, log2p, pages, page_stride, max_pages, s);
      if (e != cudaSuccess) return cuda_status(e, "page pooling launch");
    }
    e = launch_topk(m, row0, n, pages, page_stride, max_pages, page_budget, page_idx, chunks, s, log2p);
    if (e != cudaSuccess) return cuda_status(e, "page top-k launch");
    if (token_idx) {
      e = launch_page_expand(m, row0, n, page_idx, page_budget, log2p, token_idx, s);
      if (e != cudaSuccess) return cuda_status(e, "page expansion launch");
    }
  }
  return ok();
}

dsa_status dsa_sparse_mla_decode(const dsa_cache* layer, const dsa_batch* batch, const void* q, const int32_t* topk_idx,
                                 int32_t topk, float scale, void* out, float* lse, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  return sparse_mla_common(layer, batch, q, topk_idx, topk, scale, out, lse, workspace, workspace_bytes, stream, true);
}

dsa_status dsa_sparse_mla_decode_layers(const dsa_cache* layers, int32_t num_layers, const dsa_batch* batch,
                                        const void* q, const int32_t* topk_idx, int32_t topk, float scale, void* out,
                                        float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (!layers) return fail(DSA_ERR_INVALID_ARG, "layers is NULL");
  return sparse_mla_common(layers, batch, q, topk_idx, topk, scale, out, lse, workspace, workspace_bytes, stream, true,
                           nullptr, num_layers);
}

dsa_status dsa_sparse_mla_decode_ragged(const dsa_cache* layer, const dsa_batch* batch, const void* q,
                                        const int32_t* topk_idx, int32_t topk, const int32_t* row_counts, float scale,
                                        void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (!row_counts) return fail(DSA_ERR_INVALID_ARG, "row_counts is NULL");
  return sparse_mla_common(layer, batch, q, topk_idx, topk, scale, out, lse, workspace, workspace_bytes, stream, true,
                           row_counts);
}

dsa_status dsa_sparse_mla_prefill(const dsa_cache* layer, const dsa_batch* batch, const void* q, const int32_t* topk_idx,
                                  int32_t topk, float scale, void* out, float* lse, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  return sparse_mla_common(layer, batch, q, topk_idx, topk, scale, out, lse, workspace, workspace_bytes, stream, false);
}


// ---------------------------------------------------------------- decode context parallelism
static dsa_status check_dcp(int32_t world, int32_t rank, int32_t num_rows, int32_t topk) {
  if (world < 1 || world > 8) return fail(DSA_ERR_UNSUPPORTED, "dcp: world %d outside 1..8", world);
  if (rank < 0 || rank >= world) return fail(DSA_ERR_INVALID_ARG, "dcp: rank %d outside 0..%d", rank, world - 1);
  if (num_rows < 0) return fail(DSA_ERR_INVALID_ARG, "dcp: num_rows %d < 0", num_rows);
  if (topk < 1 || topk > DSA_MAX_TOPK) return fail(DSA_ERR_INVALID_ARG, "dcp: topk %d outside 1..%d", topk, DSA_MAX_TOPK);
  if ((int64_t)world * topk > 16384)
    return fail(DSA_ERR_UNSUPPORTED, "dcp: world * topk = %d exceeds 16384", world * topk);
  return ok();
}

dsa_status dsa_dcp_candidates(const float* local_scores, int64_t score_stride, const int32_t* local_idx, int32_t topk,
                              int32_t num_rows, int32_t rank, int32_t world, float* cand_scores, int32_t* cand_pos,
                              void* stream) {
  dsa_status st = check_dcp(world, rank, num_rows, topk);
  if (st != DSA_OK) return st;
  if (num_rows == 0) return ok();
  if (!local_scores || !local_idx || !cand_scores || !cand_pos) return fail(DSA_ERR_INVALID_ARG, "dcp_candidates: NULL pointer");
  if (score_stride < 1) return fail(DSA_ERR_INVALID_ARG, "dcp_candidates: score_stride %lld < 1", (long long)score_stride);
  if ((int64_t)world * score_stride > INT32_MAX)
    return fail(DSA_ERR_UNSUPPORTED, "dcp_candidates: global positions overflow int32");
  cudaError_t e = launch_dcp_candidates(local_scores, score_stride, local_idx, topk, num_rows, rank, world, cand_scores,
                                        cand_pos, static_cast<cudaStream_t>(stream));
  return cuda_status(e, "dcp candidates launch");
}

dsa_status dsa_dcp_select(const float* cand_scores, const int32_t* cand_pos, int32_t world, int32_t num_rows,
                          int32_t topk, int32_t rank, int32_t* global_idx, int32_t* local_idx, int32_t* local_count,
                          void* stream) {
  dsa_status st = check_dcp(world, rank, num_rows, topk);
  if (st != DSA_OK) return st;
  if (num_rows == 0) return ok();
  if (!cand_scores || !cand_pos || !global_idx || !local_idx) return fail(DSA_ERR_INVALID_ARG, "dcp_select: NULL pointer");
  cudaError_t e = launch_dcp_select(cand_scores, cand_pos, world, num_rows, topk, rank, global_idx, local_idx,
                                    local_count, static_cast<cudaStream_t>(stream));
  return cuda_status(e, "dcp select launch");
}

dsa_status dsa_dcp_merge(const void* outs, const float* lses, int32_t world, int32_t num_rows, void* out, float* lse,
                         void* stream) {
  if (world < 1 || world > 8) return fail(DSA_ERR_UNSUPPORTED, "dcp_merge: world %d outside 1..8", world);
  if (num_rows < 0) return fail(DSA_ERR_INVALID_ARG, "dcp_merge: num_rows %d < 0", num_rows);
  if (num_rows == 0) return ok();
  if (!outs || !lses || !out) return fail(DSA_ERR_INVALID_ARG, "dcp_merge: NULL pointer");
  if (!aligned16(outs) || !aligned16(out)) return fail(DSA_ERR_INVALID_ARG, "dcp_merge: outs/out not 16-byte aligned");
  cudaError_t e = launch_dcp_merge(outs, lses, world, num_rows, out, lse, static_cast<cudaStream_t>(stream));
  return cuda_status(e, "dcp merge launch");
}

}  // extern "C"
