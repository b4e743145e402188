/*
 * dsa.h -- C ABI of the GLM-5.2 DeepSeek Sparse Attention (DSA) step on sm_103a.
 *
 * One decoder layer's DSA step over a paged KV cache, in two stages:
 *   1. the lightning indexer scores every visible cached position of every
 *      query row and keeps the top-k positions in an index buffer that
 *      IndexShare layers reuse without rescoring;
 *   2. absorbed sparse MLA attention runs over the selected positions only.
 * The step's own new tokens are first scattered into the caches (append).
 * Beside the step itself: page-granular selection (dsa_indexer_page_topk), a
 * packed 8-bit latent cache (dsa_cache.latent_format), the device steps of
 * decode context parallelism (dsa_dcp_*, dsa_sparse_mla_decode_ragged), and
 * the append of every layer of a step in one launch (dsa_kv_append_layers).
 *
 * Sources: "GLM-5.2 on vLLM Ascend: Request-to-Backend Inference Path",
 * section 8 "The SFA backend, step by step" (write paged cache, select tokens,
 * run sparse attention; the indexer consumes paged indexer keys, sequence
 * lengths and block tables and returns top-k token indices; sparse attention
 * takes the latent query, the separate RoPE query/key, the block table, exact
 * lengths and the indices) and "Failure and Correctness Boundaries";
 * "vLLM Inference Path: GLM-5.2 as an Example", sections "Model Shape",
 * "MLA Projections and KV State", "DSA Indexer" and "Sparse MLA Attention";
 * "Making GLM-5.2 Sparse on TPUs", sections "Separate the indexer from the
 * attention it controls", "Pack requests and reuse prefixes" and "Append new
 * KV without moving the resident cache".
 *
 * Conventions that hold for every entry point:
 *   - Pointers named "device" point to GPU memory owned by the caller; the
 *     library never allocates, frees or retains them.  Structs are read on the
 *     host during the call only.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  No call synchronises the host or allocates memory, so
 *     the calls can be placed in a captured CUDA graph.
 *   - Argument errors are detected on the host before any launch and return a
 *     negative dsa_status; dsa_last_error() then describes the problem.  A
 *     failed launch returns DSA_ERR_CUDA.  Nothing is written on error.
 *   - Device-side metadata (block tables, lengths, slot mappings, indices)
 *     cannot be checked on the host: kernels skip a slot, page id or index
 *     that falls outside its buffer rather than touching memory out of range.
 *   - Kernels never trap.  Every wait on the device is bounded; a wait that
 *     runs out, and a visible position whose page id is out of range, set a
 *     DSA_DEVICE_* bit in the call's workspace instead ("GLM-5.2 on vLLM
 *     Ascend: Request-to-Backend Inference Path", "Failure and Correctness
 *     Boundaries": wrong metadata must surface, not silently change results).
 *     dsa_read_status reads those bits.
 *   - bf16 is IEEE bfloat16; e4m3 is the OCP FP8 E4M3 format.
 *   - All pointers to 16-bit or 8-bit data, and cache.index_scales, must be 16-byte aligned.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Entry points are exported from libdsa.so; everything else in it is hidden. */
#if defined(__GNUC__)
#define DSA_API __attribute__((visibility("default")))
#else
#define DSA_API
#endif

/* Fixed widths of GLM-5.2's DSA layer ("vLLM Inference Path", Model Shape table). */
#define DSA_INDEX_HEADS 32   /* lightning-indexer heads                          */
#define DSA_INDEX_DIM 128    /* indexer head width (query and shared key)        */
#define DSA_HEADS 64         /* MLA attention heads                              */
#define DSA_LATENT_DIM 512   /* c_KV latent width (also the output width)        */
#define DSA_ROPE_DIM 64      /* k_R / q_rope width                               */
#define DSA_ROW_DIM 576      /* one cached latent row: [c_KV(512) | k_R(64)]     */
#define DSA_MAX_TOPK 8192    /* largest supported top-k budget                   */
#define DSA_STATIC_SCRATCH_BYTES (16u << 20)  /* scratch of dsa_indexer_scores_topk_static */

#define DSA_ABI_VERSION 4

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = -1, /* NULL/unaligned pointer, bad size, incompatible layout */
  DSA_ERR_UNSUPPORTED = -2, /* valid request outside what this build implements     */
  DSA_ERR_WORKSPACE = -3,   /* workspace missing or smaller than the *_workspace_bytes figure */
  DSA_ERR_CUDA = -4,        /* a kernel launch failed                                */
  DSA_ERR_DEVICE_CHECK = -5 /* a call's device status held DSA_DEVICE_* bits (dsa_check_device_status) */
} dsa_status;

/* Device status bits of a call (dsa_read_status).  0 means the call ran to completion as specified. */
#define DSA_DEVICE_TMA_TIMEOUT 0x1u /* a bounded wait for a TMA copy into shared memory ran out; the
                                       call's outputs are incomplete                                   */
#define DSA_DEVICE_MMA_TIMEOUT 0x2u /* a bounded wait for tensor-core work or for another warp ran out;
                                       the call's outputs are incomplete                               */
#define DSA_DEVICE_BAD_PAGE 0x4u    /* a visible position's page id in block_table was outside
                                       [0, num_pages), or the table row was shorter than the position
                                       needs: no kernel reads through it; attention skips such entries,
                                       and the indexer's scores at those positions are unspecified      */
#define DSA_DEVICE_CONFIG 0x8u      /* a kernel met a launch shape it cannot hold (the entry points never
                                       launch one)                                                      */

typedef enum {
  DSA_KEY_BF16 = 0,     /* index keys stored as bf16 [.., 128]                        */
  DSA_KEY_FP8_E4M3 = 1, /* index keys stored as e4m3 codes [.., 128] + fp32 scale per token */
  DSA_KEY_INT8 = 2      /* index keys stored as int8 codes [.., 128] + binary16 scale per token
                           ("GLM-5.2 on vLLM Ascend", section 7 and "Quantization and Hardware
                           Branches": INT8 indexer keys with FP16 scales)                    */
} dsa_key_format;

typedef enum {
  DSA_LATENT_BF16 = 0,  /* latent rows [c_KV(512) | k_R(64)] bf16: 1152 bytes per token              */
  DSA_LATENT_E4M3 = 1   /* packed 8-bit latent: [c_KV as 512 e4m3 codes | k_R as 64 bf16] = 640 bytes
                           per token, plus an fp32 scale per token (c_KV = code * scale)            */
} dsa_latent_format;

/*
 * One layer's paged caches (caller-owned device memory).
 *   latent       DSA_LATENT_BF16: [num_pages, page_size, 576] bf16, row = [c_KV(0..511) | k_R(512..575)].
 *                DSA_LATENT_E4M3 (SFA C8, "GLM-5.2 on vLLM Ascend", "Quantization and Hardware
 *                Branches": the main latent KV packed to 8 bits, the RoPE part kept apart):
 *                [num_pages, page_size, 640] bytes, row = [512 e4m3 codes of c_KV | k_R as 64 bf16].
 *   latent_scales [num_pages, page_size] fp32, DSA_LATENT_E4M3 only: c_KV = code * scale, with
 *                scale = amax(c_KV) / 448 per token (1 if amax = 0) as written by dsa_kv_append;
 *                NULL otherwise.
 *   index_keys   [num_pages, page_size, 128] bf16, e4m3 codes or int8 codes; only on a layer
 *                that owns an indexer.  NULL on an IndexShare (shared) layer, which keeps only
 *                its latent pages and reuses the owner's index buffer.
 *   index_scales [num_pages, page_size] per-token scales (dequantised key = code * scale):
 *                fp32 for e4m3 keys; IEEE binary16 for int8 keys (the pointer then addresses
 *                2-byte halves despite its type); NULL for bf16 keys.
 * Token s of request b is stored at slot block_table[b][s / page_size] * page_size
 * + s % page_size ("GLM-5.2 on vLLM Ascend", section 8: the slot mapping scatters new
 * latent KV and indexer keys into their physical cache pages).
 */
typedef struct {
  void* latent;
  void* index_keys;
  float* index_scales;
  int32_t num_pages;
  int32_t page_size;     /* power of two, 1..1024 */
  int32_t key_format;    /* dsa_key_format of index_keys */
  int32_t latent_format; /* dsa_latent_format of latent */
  float* latent_scales;
} dsa_cache;

/*
 * Per-call batch metadata ("GLM-5.2 on vLLM Ascend", section 4 "NPU batch preparation and
 * attention metadata": cumulative query lengths, sequence lengths, block tables; "Making GLM-5.2 Sparse on TPUs", "Pack requests
 * and reuse prefixes": each query row carries its request, absolute position, valid KV length
 * and page-table base).
 *   block_table      device int32 [num_requests, block_table_stride]: physical page ids.
 *   seq_lens         device int32 [num_requests]: L_b, the KV length of request b after this
 *                    step's append.
 *   query_start_loc  device int32 [num_requests + 1]: rows of request b are
 *                    [query_start_loc[b], query_start_loc[b+1]); row i of request b sits at
 *                    position L_b - q_len_b + i and sees positions 0..L_b - q_len_b + i.
 *                    May be NULL in decode calls: then row r is request r's single row.
 *   num_rows         total query rows R (= num_requests in decode).
 *   max_seq_len      host-side upper bound on every seq_lens[b] (sizes the score workspace).
 */
typedef struct {
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  int32_t num_requests;
  int32_t num_rows;
  int32_t max_seq_len;
  int32_t block_table_stride;
} dsa_batch;

/* ABI version (DSA_ABI_VERSION) of the loaded library. */
DSA_API int32_t dsa_abi_version(void);

/* Thread-local description of the last non-OK status returned on this thread ("" if none). */
DSA_API const char* dsa_last_error(void);

/* Number of CUDA kernels this library has launched since it was loaded (all threads). */
DSA_API uint64_t dsa_kernel_launches(void);

/*
 * Device status of the last call that used `workspace`: the OR of the DSA_DEVICE_* bits its kernels
 * set.  workspace is a workspace passed to dsa_indexer_scores_topk, dsa_indexer_page_topk or
 * dsa_sparse_mla_decode / _decode_ragged / _prefill (the bits live in its first bytes, which every
 * such call rewrites), or NULL for the static scratch of dsa_indexer_scores_topk_static on the
 * current device.  ("GLM-5.2 on vLLM Ascend: Request-to-Backend Inference Path", "Failure and
 * Correctness Boundaries".)
 *   status_out  4 bytes of device memory, or of page-locked host memory mapped into the device's
 *               address space (cudaHostAlloc / cudaHostRegister), 4-byte aligned: receives the bits.
 * Enqueues one small kernel on `stream` after the call it reports on (same stream, or an event
 * between streams); *status_out is valid once the stream has passed that point.  Allocates nothing,
 * never synchronises, and may be captured in a graph.  Returns DSA_ERR_INVALID_ARG for a NULL or
 * misaligned status_out or a workspace not 256-byte aligned, DSA_ERR_CUDA if the launch fails.
 */
DSA_API dsa_status dsa_read_status(const void* workspace, uint32_t* status_out, void* stream);

/*
 * DSA_OK when bits == 0; otherwise DSA_ERR_DEVICE_CHECK, with dsa_last_error() naming the bits
 * (for example "device status 0x4: DSA_DEVICE_BAD_PAGE").  A host-side helper: no device access.
 */
DSA_API dsa_status dsa_check_device_status(uint32_t bits);

/*
 * Bytes of one layer's caches: latent pages, plus for an owner layer (owner != 0) the index
 * keys and, for e4m3 / int8 keys, their fp32 / binary16 scales.  Counting the indexer keys matters: leaving
 * them out of admission left memory unbudgeted ("Making GLM-5.2 Sparse on TPUs", "Use
 * independent oracles and test the tests").  Returns 0 for invalid arguments.
 */
DSA_API size_t dsa_cache_bytes(int32_t num_pages, int32_t page_size, int32_t key_format, int32_t owner,
                               int32_t latent_format);

/*
 * Scratch bytes dsa_indexer_scores_topk needs for num_rows rows of up to max_seq_len keys
 * with budget topk.  The figure never depends on the data, so a workspace sized once per
 * shape can be locked and reused ("Serving GLM-5.2-504B on 8x RTX PRO 6000 GPUs",
 * "Reaching 240K context with DCP": a growable workspace locked too small killed the engine).
 */
DSA_API size_t dsa_indexer_workspace_bytes(int32_t num_rows, int32_t max_seq_len, int32_t topk);

/* Scratch bytes dsa_sparse_mla_decode / _prefill need for num_rows rows and budget topk. */
DSA_API size_t dsa_mla_workspace_bytes(int32_t num_rows, int32_t topk);

/*
 * Append this step's tokens to one layer's caches.
 * ("GLM-5.2 on vLLM Ascend", section 8, "Write paged cache"; "Making GLM-5.2 Sparse on TPUs",
 * "Append new KV without moving the resident cache": cost scales with the new rows only and
 * every other slot keeps its contents.)
 *   c_kv          device bf16 [num_tokens, 512]   new latents
 *   k_rope        device bf16 [num_tokens, 64]    new RoPE keys (already rotated)
 *   k_idx         device [num_tokens, 128] new index keys, or NULL.  Required when the cache
 *                 has index_keys, rejected when it has none.  k_idx_format says how it is
 *                 stored: DSA_KEY_BF16 (copied to a bf16 cache, or quantised into an e4m3
 *                 cache: scale = amax / 448 in fp32, or 1 if amax = 0; code =
 *                 round-to-nearest-even, saturating e4m3 of x / scale in IEEE fp32; or into
 *                 an int8 cache: scale = the fp32 quotient amax / 127 rounded to binary16
 *                 (nearest-even, at most 65504, at least 2^-24; 1 if amax = 0), code =
 *                 round-to-nearest-even of x / scale in IEEE fp32 with the stored scale,
 *                 clamped to [-127, 127]), DSA_KEY_FP8_E4M3 (pre-quantised codes, copied with
 *                 k_idx_scales [num_tokens] fp32 into an e4m3 cache) or DSA_KEY_INT8
 *                 (pre-quantised codes, copied with k_idx_scales [num_tokens] binary16 into an
 *                 int8 cache).
 *   slot_mapping  device int64 [num_tokens]: physical slot (page * page_size + offset) of each
 *                 token; a negative slot skips that token, as does one >= num_pages*page_size.
 * Rows are copied bit-exactly.  num_tokens = 0 is a no-op.
 */
DSA_API dsa_status dsa_kv_append(const dsa_cache* cache, const void* c_kv, const void* k_rope, const void* k_idx,
                         int32_t k_idx_format, const float* k_idx_scales, const int64_t* slot_mapping,
                         int32_t num_tokens, void* stream);

/*
 * dsa_kv_append for num_layers layers in one launch: a decoder step appends the same tokens at the
 * same slots in every layer, each layer with its own rows (and, on an indexer-owning layer, keys).
 *   caches        host array [num_layers] of the layers' caches (1 <= num_layers <= 16).
 *   c_kv, k_rope  host arrays [num_layers] of device pointers, as for dsa_kv_append.
 *   k_idx         host array [num_layers] of device pointers, NULL where the layer has no index keys
 *                 (or NULL altogether when none has); k_idx_scales likewise (pre-quantised keys only).
 *   k_idx_format, slot_mapping, num_tokens  as for dsa_kv_append, shared by the layers.
 * Every layer is validated before anything is launched; the result is that of num_layers calls of
 * dsa_kv_append.
 */
DSA_API dsa_status dsa_kv_append_layers(const dsa_cache* caches, int32_t num_layers, const void* const* c_kv,
                                        const void* const* k_rope, const void* const* k_idx, int32_t k_idx_format,
                                        const float* const* k_idx_scales, const int64_t* slot_mapping,
                                        int32_t num_tokens, void* stream);

/*
 * Lightning indexer scores and top-k selection for every query row.
 * ("vLLM Inference Path", "DSA Indexer"; "Making GLM-5.2 Sparse on TPUs", "Separate the indexer
 * from the attention it controls".)
 *   I(r, s) = sum_{h<32} w[r,h] * max(0, sum_{d<128} q_idx[r,h,d] * K[s,d])  for 0 <= s <= pos(r),
 *   K[s] = bf16 key, or e4m3 / int8 code * scale[s].  int8 codes are split exactly on chip into
 *   two e4m3 terms (sm_103a has no integer MMA), so every key format runs on the tensor cores.
 *   topk_idx[r] = the topk positions with the largest I (ties: smaller position first), sorted
 *   ascending; every visible position when pos(r) + 1 <= topk; padded with -1.
 *   owner       cache of the indexer-owning layer (index_keys must be non-NULL).
 *   q_idx       device bf16 [num_rows, 32, 128]
 *   w           device fp32 [num_rows, 32]
 *   topk        1..DSA_MAX_TOPK
 *   topk_idx    device int32 [num_rows, topk] (output: the shared index buffer)
 *   scores_out  optional device fp32 [num_rows, max_seq_len]: I(r, s) for s <= pos(r), -inf
 *               beyond; NULL to skip.
 *   workspace   device scratch of at least dsa_indexer_workspace_bytes(num_rows, max_seq_len,
 *               topk) bytes, 256-byte aligned; dsa_read_status(workspace, ...) gives the call's device
 *               status (DSA_DEVICE_BAD_PAGE for an out-of-range page of a visible key).
 */
DSA_API dsa_status dsa_indexer_scores_topk(const dsa_cache* owner, const dsa_batch* batch, const void* q_idx,
                                   const float* w, int32_t topk, int32_t* topk_idx, float* scores_out,
                                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * Scratch bytes dsa_indexer_page_topk needs for num_rows rows of up to max_seq_len keys, pages of
 * page_size keys and budget page_budget (shape only, like dsa_indexer_workspace_bytes).
 */
DSA_API size_t dsa_indexer_page_workspace_bytes(int32_t num_rows, int32_t max_seq_len, int32_t page_size,
                                                int32_t page_budget);

/*
 * Page-granular selection: the indexer scores pooled into page scores, and a page budget.
 * ("Making GLM-5.2 Sparse on TPUs", "Make the sparsity unit match the memory unit": rank each page
 * by its highest legal token score, masks before the maximum; "Stream indexer scores over live
 * context": masks and page maxima on chip, only page scores reach HBM.)
 *   S(r, p) = max over visible s (0 <= s <= pos(r)) in logical page p of I(r, s), I as in
 *             dsa_indexer_scores_topk; pages 0 .. pos(r) / page_size.
 *   page_idx[r]  = the page_budget pages with the largest S (ties: smaller page), sorted ascending;
 *                  every such page when there are at most page_budget; padded with -1.
 *   token_idx[r] = the visible positions of those pages, ascending, padded with -1 to
 *                  page_budget * page_size: an index buffer for dsa_sparse_mla_decode / _prefill
 *                  with topk = page_budget * page_size.  Optional (NULL to skip).
 *   owner          cache of the indexer-owning layer; page_size <= 128 (DSA_ERR_UNSUPPORTED otherwise).
 *   page_budget    1..DSA_MAX_TOPK; with token_idx, page_budget * page_size <= DSA_MAX_TOPK.
 *   page_idx       device int32 [num_rows, page_budget] (output).
 *   token_idx      device int32 [num_rows, page_budget * page_size] (output) or NULL.
 *   page_scores_out optional device fp32 [num_rows, ceil(max_seq_len / page_size)]: S, -inf beyond
 *                  the row's last page; NULL to skip.
 *   workspace      device scratch of at least dsa_indexer_page_workspace_bytes(...) bytes, 256-byte
 *                  aligned; dsa_read_status(workspace, ...) gives the call's device status.
 * The library has no page counterpart of the static-scratch entry point.
 */
DSA_API dsa_status dsa_indexer_page_topk(const dsa_cache* owner, const dsa_batch* batch, const void* q_idx,
                                         const float* w, int32_t page_budget, int32_t* page_idx, int32_t* token_idx,
                                         float* page_scores_out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * dsa_indexer_scores_topk without a caller workspace.  The pages have no counterpart: this is
 * a convenience of this library for callers that cannot allocate device memory per call (a
 * serving loop whose memory was reserved and locked before it started, or host code without an
 * allocator).  It computes exactly what dsa_indexer_scores_topk computes, with the same
 * arguments apart from the workspace, and allocates nothing.
 *   Scratch: a fixed device array of DSA_STATIC_SCRATCH_BYTES (16 MiB) inside the library, one
 *     per device.  Shapes whose dsa_indexer_workspace_bytes(num_rows, max_seq_len, topk)
 *     exceeds it return DSA_ERR_WORKSPACE before anything is launched (for example, with topk
 *     2048, 32 rows of 90,000 keys or 64 rows of 40,000 keys fit; 64 rows of 131,072 keys do not).
 *   Set-up: the first call on a device, made with that device current, looks the array up
 *     (cudaGetSymbolAddress) and keeps its address for that device's current CUDA context (a new
 *     context, after a device reset say, looks it up again); make that first call before capturing
 *     the stream.  A failed look-up returns DSA_ERR_CUDA.
 *   Zeroing: the call's first kernel clears the array's status header; nothing else in it needs
 *     to start at zero.  dsa_read_status(NULL, ...) reads the last call's device status.
 *   Concurrency: calls whose work overlaps on one device share the array and race; the caller
 *     serialises them (one stream, or an event between streams).
 */
DSA_API dsa_status dsa_indexer_scores_topk_static(const dsa_cache* owner, const dsa_batch* batch, const void* q_idx,
                                          const float* w, int32_t topk, int32_t* topk_idx, float* scores_out,
                                          void* stream);

/*
 * Sparse absorbed MLA over the selected positions, decode form: one query row
 * per request at position seq_lens[b] - 1 (query_start_loc is ignored and may be NULL).
 * ("vLLM Inference Path", "MLA Projections and KV State" and "Sparse MLA Attention";
 * "Making GLM-5.2 Sparse on TPUs", "Separate the indexer ...": absorbed MLA, scale tied to
 * the unabsorbed 192 + 64 width.)
 *   For every row r and head h, over the valid entries s of topk_idx[r] (0 <= s <= pos(r);
 *   -1 padding and out-of-range entries are skipped):
 *     z_s = scale * (q[r,h,0:512] . c_KV[s] + q[r,h,512:576] . k_R[s]),
 *     out[r,h,:] = sum_s softmax(z)_s c_KV[s]   (bf16),   lse[r,h] = ln sum_s exp(z_s)  (fp32).
 *   A row with no valid entry gets out = 0 and lse = -inf.
 *   layer     this layer's cache (only latent, and latent_scales for a packed 8-bit latent, is read;
 *             index_keys may be NULL).  With DSA_LATENT_E4M3, c_KV[s] = code * scale[s]: the kernel
 *             expands each gathered row to fp16 on chip (c_KV and k_R must lie within fp16 range)
 *             and runs the products in fp16 with fp32 accumulation.
 *   q         device bf16 [num_rows, 64, 576]: [q_latent (W^UK absorbed) | q_rope] per head.
 *   topk_idx  device int32 [num_rows, topk]: the owner layer's index buffer.  IndexShare layers
 *             pass the owner's buffer; NULL is rejected ("GLM-5.2 on vLLM Ascend", "Failure and
 *             Correctness Boundaries": a shared layer without the shared buffer is rejected).
 *   scale     softmax scale, normally 1/sqrt(192 + 64) = 1/16.
 *   out       device bf16 [num_rows, 64, 512];  lse: optional device fp32 [num_rows, 64].
 *   workspace device scratch of at least dsa_mla_workspace_bytes(num_rows, topk) bytes, 256-byte
 *             aligned; dsa_read_status(workspace, ...) gives the call's device status
 *             (DSA_DEVICE_BAD_PAGE for a valid entry whose page id is out of range).
 */
DSA_API dsa_status dsa_sparse_mla_decode(const dsa_cache* layer, const dsa_batch* batch, const void* q,
                                 const int32_t* topk_idx, int32_t topk, float scale, void* out, float* lse,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * dsa_sparse_mla_decode for the layers of an IndexShare group in one call: every layer attends with
 * the same index buffer (the owner's), so one launch covers all of them, its units (layer, row,
 * 64-entry tile) spread over every SM.  The result equals num_layers dsa_sparse_mla_decode calls,
 * one per layer, up to the floating-point order of the split-k merge.  ("GLM-5.2 on vLLM Ascend",
 * section 7, "GLM-5.2 shared-indexer construction": shared layers reuse the owner's top-k.)
 *   layers      host array [num_layers] of the layers' caches, 1 <= num_layers <= 4; they must agree in
 *               page_size, num_pages and latent_format (the block table is shared).  A packed 8-bit
 *               latent runs as one launch per layer.
 *   q           device bf16 [num_layers, num_rows, 64, 576]: layer l's queries at [l].
 *   out         device bf16 [num_layers, num_rows, 64, 512];  lse: optional device fp32
 *               [num_layers, num_rows, 64].
 *   workspace   at least dsa_mla_workspace_bytes(num_layers * num_rows, topk) bytes, 256-byte aligned.
 *   Other arguments as for dsa_sparse_mla_decode; DSA_ERR_UNSUPPORTED for num_layers outside 1..4.
 */
DSA_API dsa_status dsa_sparse_mla_decode_layers(const dsa_cache* layers, int32_t num_layers, const dsa_batch* batch,
                                        const void* q, const int32_t* topk_idx, int32_t topk, float scale,
                                        void* out, float* lse, void* workspace, size_t workspace_bytes,
                                        void* stream);

/*
 * dsa_sparse_mla_decode over index buffers whose valid entries lead each row: row r's entries at
 * and past row_counts[r] must be -1 (the caller guarantees it; they are skipped as usual).  The
 * result is dsa_sparse_mla_decode's on the same buffer; the call only spends less time on rows with
 * few entries, since each row's work covers its first row_counts[r] entries rather than all topk.
 * (Used for a rank's share of a DCP selection, which holds about topk / world entries.)
 *   row_counts  device int32 [num_rows], written before the call on the same stream (for example by
 *               dsa_dcp_select); NULL is rejected.  Other arguments as for dsa_sparse_mla_decode.
 */
DSA_API dsa_status dsa_sparse_mla_decode_ragged(const dsa_cache* layer, const dsa_batch* batch, const void* q,
                                        const int32_t* topk_idx, int32_t topk, const int32_t* row_counts,
                                        float scale, void* out, float* lse, void* workspace,
                                        size_t workspace_bytes, void* stream);

/*
 * Same operation for extend/prefill/verify batches: several query rows per request, causal per
 * row (row i of request b sees positions 0..L_b - q_len_b + i; query_start_loc is required).
 * ("Making GLM-5.2 Sparse on TPUs", "Carry sparse reads through prefill" and "Pack requests and
 * reuse prefixes": causality uses P + i, not an offset reset at each chunk.)
 */
DSA_API dsa_status dsa_sparse_mla_prefill(const dsa_cache* layer, const dsa_batch* batch, const void* q,
                                  const int32_t* topk_idx, int32_t topk, float scale, void* out, float* lse,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * Decode context parallelism: the device steps around the two exchanges.
 * ("Serving GLM-5.2-504B on 8x RTX PRO 6000 GPUs", "Reaching 240K context with DCP": the KV is
 * sharded along the sequence across the ranks, each rank scoring only its share of the keys.)
 * Token s of a request lives on rank s mod world at local position s / world; each rank holds
 * its share of every request in its own cache and runs dsa_indexer_scores_topk over it (decode
 * rows only: the local row sees all of its rank's keys).  Then, per rank:
 *   dsa_dcp_candidates  local top-k -> (score, global position) candidates;
 *   all-gather of the candidates (the caller's collective) into [world][num_rows][topk];
 *   dsa_dcp_select      the global top-k (identical on every rank), this rank's share of it as a
 *                       compacted local index buffer, and the share's size per row;
 *   dsa_sparse_mla_decode_ragged over the local cache with that buffer and those sizes (out and
 *                       lse required): each rank's attention covers only its share;
 *   all-gather of out and lse into [world][...];
 *   dsa_dcp_merge       the LSE merge: the single-device attention over the global selection.
 * world is 1..8 and world * topk <= 16384 (DSA_ERR_UNSUPPORTED otherwise); num_rows 0 is a no-op.
 * No workspace; nothing is allocated.  Errors as for the other entry points.
 */

/*
 *   local_scores  device fp32 [num_rows, score_stride]: the rank's indexer scores (scores_out of
 *                 dsa_indexer_scores_topk, whose row stride is the batch's max_seq_len).
 *   local_idx     device int32 [num_rows, topk]: the rank's local top-k (-1 padded).
 *   cand_scores   device fp32 [num_rows, topk] (output): local_scores at local_idx, -inf for -1.
 *   cand_pos      device int32 [num_rows, topk] (output): local_idx * world + rank, -1 for -1.
 */
DSA_API dsa_status dsa_dcp_candidates(const float* local_scores, int64_t score_stride, const int32_t* local_idx,
                                      int32_t topk, int32_t num_rows, int32_t rank, int32_t world,
                                      float* cand_scores, int32_t* cand_pos, void* stream);

/*
 *   cand_scores, cand_pos  device [world, num_rows, topk]: every rank's candidates, rank-major.
 *   global_idx  device int32 [num_rows, topk] (output): the topk candidates with the largest score
 *               (ties: smaller global position), sorted ascending, -1 padded when fewer exist;
 *               equal to dsa_indexer_scores_topk's selection over the unsharded row.
 *   local_idx   device int32 [num_rows, topk] (output): this rank's share of global_idx (positions p
 *               with p mod world == rank) as local positions p / world, ascending, in the first
 *               local_count[r] slots of row r, -1 after them: an index buffer for
 *               dsa_sparse_mla_decode_ragged (or dsa_sparse_mla_decode) over the rank's cache.
 *   local_count optional device int32 [num_rows] (output): the size of this rank's share; NULL to skip.
 */
DSA_API dsa_status dsa_dcp_select(const float* cand_scores, const int32_t* cand_pos, int32_t world,
                                  int32_t num_rows, int32_t topk, int32_t rank, int32_t* global_idx,
                                  int32_t* local_idx, int32_t* local_count, void* stream);

/*
 *   outs   device bf16 [world, num_rows, 64, 512], 16-byte aligned: every rank's out.
 *   lses   device fp32 [world, num_rows, 64]: every rank's lse (-inf: that rank selected nothing).
 *   out    device bf16 [num_rows, 64, 512] (output), 16-byte aligned:
 *          sum_w exp(lse_w - M) out_w / sum_w exp(lse_w - M), M = max_w lse_w; 0 if all are -inf.
 *   lse    optional device fp32 [num_rows, 64] (output): M + ln sum_w exp(lse_w - M), or -inf.
 */
DSA_API dsa_status dsa_dcp_merge(const void* outs, const float* lses, int32_t world, int32_t num_rows, void* out,
                                 float* lse, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
