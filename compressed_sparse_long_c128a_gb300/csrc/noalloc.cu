// csa_indexer_topk_noalloc: the indexer + top-k entry point for callers that
// cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace: a plugin loaded
// into a host runtime that owns every device byte and exposes no allocator to
// its extensions, or a serving loop that forbids allocation on its hot path
// because an allocation can stall on a device-wide synchronisation or fail
// under memory pressure mid-request.  For them this entry point keeps its
// scratch (the rows' scores and each chunk's top-k candidates) in one
// fixed-size array in device global memory that the library defines itself.
//
// Costs and rules of that choice:
//   * every GPU that loads the library holds kScratchBytes for it until the
//     process exits;
//   * requests whose scratch exceeds kScratchBytes are refused with
//     CSA_ERR_WORKSPACE before anything is enqueued;
//   * all calls share the one array, so calls that can overlap on the GPU (on
//     different streams without ordering between them) race on it; calls on one
//     stream are safe.  Nothing in the array has to start at zero: each call
//     writes every byte it reads before reading it;
//   * the first call on a device looks up the array's device address (host
//     code only holds a stand-in symbol for it) with that device current; make
//     that first call before any stream capture.

#include <mutex>

#include "csa_kernels.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB

// The scratch itself.  In host code this name is only a stand-in symbol; the
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[csa::kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per device.
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSA_ERR_CUDA;
  if (dev < 0 || dev >= csa::kMaxDevices) return CSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return CSA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return CSA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" {

int csa_indexer_topk_noalloc(const void* q_idx, int32_t q_dtype, const float* w, int32_t n_rows, int32_t idx_heads,
                             int32_t idx_dim, const int32_t* seq_id, const int32_t* pos, int32_t ratio,
                             int32_t window, const csa_paged* idx_cache, const csa_block_table* bt, int32_t k,
                             int32_t max_n, int32_t* out_idx, int32_t* err, csa_stream_t stream) {
  using namespace csa;
  const int st = check_indexer_topk(q_idx, q_dtype, w, n_rows, idx_heads, idx_dim, seq_id, pos, ratio, window,
                                    idx_cache, bt, k, max_n, out_idx, err);
  if (st != CSA_OK || n_rows == 0) return st;

  // sized as csa_indexer_topk_workspace_size sizes a workspace (max_n >= 1 so
  // that a request is never sized at zero); the kernels get max_n unchanged
  const int32_t size_n = max_n > 0 ? max_n : 1;
  const size_t score_bytes = align256(sizeof(float) * (size_t)n_rows * size_n);
  const size_t cand_bytes = align256(topk_candidate_bytes(n_rows, max_n, k));
  const size_t deal_bytes = n_rows < kDealMaxCtas ? align256(deal_candidate_bytes(kDealMaxCtas, k)) : 0;
  if (score_bytes + cand_bytes + deal_bytes > kScratchBytes) return CSA_ERR_WORKSPACE;

  void* scratch = nullptr;
  const int sst = scratch_for_current_device(&scratch);
  if (sst != CSA_OK) return sst;

  float* scores = reinterpret_cast<float*>(scratch);
  void* cand = cand_bytes ? reinterpret_cast<uint8_t*>(scratch) + score_bytes : nullptr;
  void* deal = deal_bytes ? reinterpret_cast<uint8_t*>(scratch) + score_bytes + cand_bytes : nullptr;
  return enqueue_indexer_topk(q_idx, q_dtype, w, n_rows, idx_heads, idx_dim, seq_id, pos, ratio, window, idx_cache,
                              bt, k, max_n, out_idx, scores, cand, deal, err, stream);
}

}  // extern "C"
