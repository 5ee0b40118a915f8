// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the encoder is fetched at run time)
#include <cuda_runtime.h>

#include <mutex>

#include "csa_device.cuh"

namespace csa {

// One-time set-up of a launcher, kept per device: function attributes set by
// cudaFuncSetAttribute and device properties belong to the device that is
// current when they are set or read, so each device ordinal has its own slot.
constexpr int kMaxDevices = 64;
struct PerDevice {
  std::mutex mu;
  int64_t value[kMaxDevices] = {};  // launcher-defined; 0 until the first set-up
};

// Runs f(device, slot) under the lock with the current device's slot.
template <typename F>
inline cudaError_t with_device_slot(PerDevice& pd, F f) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(pd.mu);
  return f(dev, pd.value[dev]);
}

// Number of SMs of the current device (looked up once per device).
cudaError_t sm_count(int* n);

// Kernel launches the library has issued (csa_launch_count); counted on the host.
void count_launch();

// Launch with programmatic stream serialization (see pdl_wait in
// csa_device.cuh: every kernel waits for its predecessor before it touches
// memory) and, when cluster_y > 0, clusters of (1, cluster_y, 1) CTAs.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                           int cluster_y, Args... args) {
  count_launch();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_y > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 1;
    attr[n].val.clusterDim.y = (unsigned)cluster_y;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// 2-D bf16 tensor map over `rows` rows of `cols` elements (row stride `stride_bytes`),
// boxes of box_cols x box_rows, 128-byte swizzle; false if it cannot be encoded
// (unaligned base or stride, or no driver entry point).  Defined in api.cu.
bool encode_bf16_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t stride_bytes,
                     uint32_t box_cols, uint32_t box_rows);

// ---- compressor (k_compress.cu)
struct IngestArgs {
  const void* kv;
  const void* gate;
  int32_t in_dtype;
  const int32_t* seq_id;
  const int32_t* pos;
  const float* gamma_swa;
  csa_paged state;
  csa_block_table state_bt;
  csa_paged swa;
  csa_block_table swa_bt;
  int32_t dim;
  float eps;
  RopeTab rope;
  int32_t* err;
};

struct EmitArgs {
  const int32_t* seq_id;
  const int32_t* pos;
  const float* bias;
  const float* gamma_c;
  csa_paged state;
  csa_block_table state_bt;
  csa_paged comp;
  csa_block_table comp_bt;
  int32_t dim, ratio, window;
  float eps;
  RopeTab rope;
  int32_t* err;
};

// query RMSNorm of the call's tokens, run by eight extra warps of the ingest or
// fused kernel (q == nullptr: none)
struct QNormArgs {
  const void* q;
  int32_t q_dtype;
  const float* gamma;
  void* out;
  int32_t out_dtype;
  int32_t heads, dim;
  float eps;
};

cudaError_t launch_ingest(const IngestArgs& a, const QNormArgs& q, int32_t n_tok, cudaStream_t s);
cudaError_t launch_emit(const EmitArgs& a, int32_t n_tok, cudaStream_t s);
// one launch for calls of at most 1024 tokens (D % 8 == 0, D <= 512, 16-byte aligned rows)
bool compress_fused_eligible(const IngestArgs& ia, const EmitArgs& ea, int32_t n_tok);
cudaError_t launch_compress_fused(const IngestArgs& ia, const EmitArgs& ea, const QNormArgs& q, int32_t n_tok,
                                  cudaStream_t s);

// ---- cache store (k_store.cu)
struct StoreArgs {
  const float* rows;
  const int32_t* seq_id;
  const int32_t* row_idx;
  csa_paged cache;
  csa_block_table bt;
  int32_t* err;
};
cudaError_t launch_store(const StoreArgs& a, int32_t n, cudaStream_t s);

// ---- indexer scores + top-k (k_indexer.cu, k_topk.cu)
struct IndexerArgs {
  const void* q_idx;
  int32_t q_dtype;
  const float* w;
  const int32_t* seq_id;
  const int32_t* pos;
  csa_paged cache;
  csa_block_table bt;
  int32_t heads, dim, ratio, window;
  int32_t max_n;    // row stride of the score buffer
  float* scores;    // [n_rows][max_n]
  int32_t* err;
  // tensor-core path, bf16 cache: the cache as [blocks*64][128] rows, 64x64
  // boxes, 128-byte swizzle (set by the launcher)
  CUtensorMap k_map;
  // balanced deal with the selection fused (sel_k > 0): the grid's CTAs share
  // the rows' tiles in proportion to each row's length and each writes the
  // top-sel_k of its range to the candidate lists, which the deal merge turns
  // into the rows' selections; sel_k == 0: one CTA per row and split, every
  // score written to `scores`
  int32_t sel_k;
  int32_t n_rows;
  // two list slots per CTA (2c, 2c + 1: one per row the CTA meets), see DealCandidates
  uint32_t* cand_key;       // [2 grid][2 sel_k] order-preserving keys of the scores
  int32_t* cand_idx;        // [2 grid][2 sel_k] entry indices
  int32_t* cand_cnt;        // [2 grid]
  uint32_t* cand_thr;       // [2 grid] every key of the slot's range at or above it is in its list
  int32_t* cand_row_first;  // [rows] the CTA holding the row's first list
  int32_t* cand_row_ctas;   // [rows] the row's lists
  int32_t* cand_row_seg;    // [rows] the slot of the row's first list within its CTA
};
cudaError_t launch_indexer_scores(const IndexerArgs& a, int32_t n_rows, cudaStream_t s);
// tensor-core scores, 64 heads x 128 dims, bf16 or e2m1 keys (k_indexer_tc.cu)
bool indexer_tc_eligible(const IndexerArgs& a);
// Tiles (128 entries) a CTA of the balanced deal can hold for the fused
// selection, by key format; 0 when the format has no tensor-core path.
int32_t indexer_deal_capacity(int32_t cache_dtype);
// The deal's largest per-CTA tile budget for n_rows rows of at most max_n
// entries on G CTAs (an upper bound of what the device computes), or -1 when
// a deal does not apply (more rows than CTAs).
int32_t indexer_deal_bound(int32_t n_rows, int32_t max_n, int32_t G);
// a.sel_k > 0: balanced deal on G CTAs; else one CTA per row and split
cudaError_t launch_indexer_tc(const IndexerArgs& a, int32_t n_rows, int32_t G, cudaStream_t s);

// Candidate lists of a balanced deal: two list slots per CTA (2c and 2c + 1)
// of 2k (key, index) pairs, a count and a threshold each, and each row's
// first CTA, list count and first slot's segment (written by the indexer's
// CTA 0, so the merge does not compute the deal again): the lists of row r
// are slot 2 first + seg, then slots 2c for the next ctas - 1 CTAs.  A deal
// uses at most kDealMaxCtas CTAs.
constexpr int32_t kDealMaxCtas = 256;
struct DealCandidates {
  uint32_t* key;        // [2 ctas][cap]
  int32_t* idx;         // [2 ctas][cap]
  int32_t* cnt;         // [2 ctas]
  uint32_t* thr;        // [2 ctas]
  int32_t* row_first;   // [kDealMaxRows]
  int32_t* row_ctas;    // [kDealMaxRows]
  int32_t* row_seg;     // [kDealMaxRows]
  int32_t ctas, cap;
};
size_t deal_candidate_bytes(int32_t G, int32_t k);
DealCandidates deal_candidates(void* base, int32_t G, int32_t k);

struct TopkArgs {
  const float* scores;  // [n_rows][max_n]
  const int32_t* pos;
  int32_t ratio, window, max_n, k;
  int32_t* out;  // [n_rows][k]
  int32_t* err;
};
// `cand`: topk_candidate_bytes() of scratch for the two-stage path (nullptr: one CTA per row)
size_t topk_candidate_bytes(int32_t n_rows, int32_t max_n, int32_t k);
cudaError_t launch_topk(const TopkArgs& a, int32_t n_rows, void* cand, cudaStream_t s);
// the rows' selections from the candidate lists of a balanced deal (after the indexer launch)
cudaError_t launch_topk_deal_merge(const TopkArgs& a, int32_t n_rows, const DealCandidates& c, cudaStream_t s);

// Host validation and enqueue of indexer scores + top-k, shared by
// csa_indexer_topk and csa_indexer_topk_noalloc so that both accept and refuse
// the same calls (api.cu).  check_indexer_topk returns CSA_OK for n_rows == 0
// before looking at any pointer; the caller then enqueues nothing.
int check_indexer_topk(const void* q_idx, int32_t q_dtype, const float* w, int32_t n_rows, int32_t idx_heads,
                       int32_t idx_dim, const int32_t* seq_id, const int32_t* pos, int32_t ratio, int32_t window,
                       const csa_paged* idx_cache, const csa_block_table* bt, int32_t k, int32_t max_n,
                       const int32_t* out_idx, const int32_t* err);
// scores: n_rows * max_n floats; cand: topk_candidate_bytes(n_rows, max_n, k)
// bytes or nullptr when 0; deal: deal_candidate_bytes(kDealMaxCtas, k) bytes, or
// nullptr (no balanced deal)
int enqueue_indexer_topk(const void* q_idx, int32_t q_dtype, const float* w, int32_t n_rows, int32_t idx_heads,
                         int32_t idx_dim, const int32_t* seq_id, const int32_t* pos, int32_t ratio, int32_t window,
                         const csa_paged* idx_cache, const csa_block_table* bt, int32_t k, int32_t max_n,
                         int32_t* out_idx, float* scores, void* cand, void* deal, int32_t* err,
                         cudaStream_t stream);

// ---- attention (k_attn.cu)
struct AttnArgs {
  const void* q;
  int32_t q_dtype;
  const int32_t* seq_id;
  const int32_t* pos;
  csa_paged comp;
  csa_block_table comp_bt;
  const int32_t* topk;  // nullptr: dense
  int32_t k;
  csa_paged swa;
  csa_block_table swa_bt;
  void* out;
  int32_t out_dtype;
  float* out_scales;
  int32_t heads, dim, ratio, window, swa_len;
  float scale;
  RopeTab rope;
  int32_t n_splits;
  float* part_o;  // [n_rows][heads][n_splits][dim]
  float* part_ml; // [n_rows][heads][n_splits][2]
  int32_t* err;
  // tensor-core path: bf16 query rows as a [rows*64][512] tensor, 64x64 boxes,
  // 128-byte swizzle (q_tma = 0 when q cannot be described, e.g. unaligned)
  CUtensorMap q_map;
  int32_t q_tma;
};
int32_t attn_splits(int32_t n_rows, int32_t heads, int32_t keys_per_row);
size_t attn_workspace_bytes(int32_t n_rows, int32_t heads, int32_t dim, int32_t n_splits);
cudaError_t launch_attn(const AttnArgs& a, int32_t n_rows, int32_t keys_per_row, cudaStream_t s);
cudaError_t launch_attn_merge(const AttnArgs& a, int32_t n_rows, cudaStream_t s);

// ---- tensor-core attention, D = 512 and H = 64 (k_attn_tc.cu)
bool attn_tc_eligible(const AttnArgs& a);
int32_t attn_tc_splits(int32_t n_rows, int32_t keys_per_row);
cudaError_t launch_attn_tc(const AttnArgs& a, int32_t n_rows, cudaStream_t s);

}  // namespace csa
