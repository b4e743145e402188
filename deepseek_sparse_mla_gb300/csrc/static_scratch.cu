// Indexer scores + top-k with library-owned scratch: the one entry point that takes no workspace.
//
// Some callers cannot hand the library a workspace: a serving loop whose device memory was
// reserved and locked before it started, or host code that holds no allocator at all.  For
// them the scratch of dsa_indexer_scores_topk (status word, row-group table, score block) lives
// in a fixed device array of this module, and the call runs the ordinary indexer and top-k
// launches on it.  Nothing is allocated or freed on any call.
//
// Set-up: the first call on a device (with that device current) looks up the array's device
// address with cudaGetSymbolAddress and keeps it, keyed by the device's current CUDA context,
// for later calls; a call under another context (after a device reset re-created the primary
// context, say) looks it up again.  Make that first call before capturing the stream into a graph.
//
// Zeroing: only the status header must start at zero; the call's first kernel clears it on the
// device, as in the workspace entry point.  The group table, the score block and the top-k
// candidate lists are fully written before they are read.  dsa_read_status(NULL, ...) reads the
// header's status bits.
//
// Concurrency: there is one array per device.  Two calls whose work overlaps on the device
// (different streams, or different host threads) share it and race; serialise them.
#include <mutex>

#include <cudaTypedefs.h>

#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_indexer_scratch[DSA_STATIC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

// The calling thread's current CUDA context (the driver entry point is looked up once).
CUcontext current_context() {
  static PFN_cuCtxGetCurrent_v4000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    return cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
                   q == cudaDriverEntryPointSuccess
               ? reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p)
               : nullptr;
  }();
  CUcontext c = nullptr;
  if (fn) fn(&c);
  return c;
}

}  // namespace

// Device address of this device's scratch array, looked up once per device and context.
dsa_status static_scratch_of_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return report_error(DSA_ERR_CUDA, "static scratch: cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return report_error(DSA_ERR_UNSUPPORTED, "static scratch: device ordinal >= 64");
  e = cudaFree(nullptr);                              // make the device's primary context current
  if (e != cudaSuccess) return report_error(DSA_ERR_CUDA, "static scratch: no CUDA context on the current device");
  const CUcontext ctx = current_context();
  std::lock_guard<std::mutex> g(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_indexer_scratch);
    if (e != cudaSuccess || p == nullptr)
      return report_error(DSA_ERR_CUDA, "static scratch: cudaGetSymbolAddress of the scratch array failed");
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return DSA_OK;
}

}  // namespace dsa

extern "C" {

dsa_status dsa_indexer_scores_topk_static(const dsa_cache* owner, const dsa_batch* batch, const void* q_idx,
                                          const float* w, int32_t topk, int32_t* topk_idx, float* scores_out,
                                          void* stream) {
  if (!batch) return dsa::report_error(DSA_ERR_INVALID_ARG, "batch is NULL");
  if (batch->num_rows > 0 && batch->max_seq_len > 0 && topk >= 1 && topk <= DSA_MAX_TOPK) {
    const size_t need = dsa_indexer_workspace_bytes(batch->num_rows, batch->max_seq_len, topk);
    if (need > (size_t)DSA_STATIC_SCRATCH_BYTES)
      return dsa::report_error(DSA_ERR_WORKSPACE,
                               "this shape needs more scratch than the static array holds "
                               "(DSA_STATIC_SCRATCH_BYTES); use dsa_indexer_scores_topk with a caller workspace");
  }
  void* scratch = nullptr;
  dsa_status st = dsa::static_scratch_of_current_device(&scratch);
  if (st != DSA_OK) return st;
  return dsa_indexer_scores_topk(owner, batch, q_idx, w, topk, topk_idx, scores_out, scratch,
                                 (size_t)DSA_STATIC_SCRATCH_BYTES, stream);
}

}  // extern "C"
