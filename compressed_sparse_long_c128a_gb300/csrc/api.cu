// C ABI of libcsa: argument validation and kernel dispatch.  Every hot-path
// entry point validates on the host, enqueues its kernels on the caller's
// stream and returns without synchronising or allocating.

#include <atomic>
#include <cmath>
#include <cstring>

#include "csa_kernels.h"

using namespace csa;

namespace {

constexpr int32_t kVersion = 100;  // 0.1.0

bool dtype_ok(int32_t dt) { return dt >= CSA_F32 && dt <= CSA_E4M3R; }

int check_paged(const csa_paged* c, int32_t dim, int32_t rows_per_block, unsigned allowed_dtypes) {
  if (!c || !c->data || c->num_blocks <= 0) return CSA_ERR_INVALID_ARG;
  if (!dtype_ok(c->dtype)) return CSA_ERR_INVALID_ARG;
  if (!(allowed_dtypes & (1u << c->dtype))) return CSA_ERR_UNSUPPORTED;
  if (c->dim != dim || c->rows_per_block != rows_per_block) return CSA_ERR_INVALID_ARG;
  if ((c->dtype == CSA_E4M3 || c->dtype == CSA_E4M3R || c->dtype == CSA_E2M1) && !c->scales)
    return CSA_ERR_INVALID_ARG;
  if (c->dtype == CSA_E2M1 && dim % 16) return CSA_ERR_INVALID_ARG;
  if (c->dtype == CSA_E4M3R) {
    if (c->tail_bf16 <= 0 || c->tail_bf16 % 16 || c->tail_bf16 > dim || (dim - c->tail_bf16) % 16)
      return CSA_ERR_INVALID_ARG;
  } else if (c->tail_bf16 != 0) {
    return CSA_ERR_INVALID_ARG;
  }
  return CSA_OK;
}

int check_bt(const csa_block_table* bt) {
  if (!bt || !bt->table || bt->num_seqs <= 0 || bt->stride <= 0) return CSA_ERR_INVALID_ARG;
  return CSA_OK;
}

int check_layer(const csa_layer* L) {
  if (!L) return CSA_ERR_INVALID_ARG;
  if (L->ratio <= 0 || L->window <= 0 || L->window > 256 || 256 % L->ratio) return CSA_ERR_INVALID_ARG;
  if (L->dim <= 0 || L->dim % 2 || L->rope_dim < 0 || L->rope_dim % 2 || L->rope_dim > L->dim ||
      L->rope_dim > 2 * kMaxRopePairs)
    return CSA_ERR_INVALID_ARG;
  if (L->heads <= 0 || L->swa <= 0 || L->swa > 256) return CSA_ERR_INVALID_ARG;
  if (!(L->rope_theta > 0.f) || !(L->rms_eps >= 0.f) || !(L->scale > 0.f)) return CSA_ERR_INVALID_ARG;
  return CSA_OK;
}

RopeTab make_rope(int32_t rope_dim, float theta) {
  RopeTab t;
  std::memset(&t, 0, sizeof(t));
  t.rope_dim = rope_dim;
  for (int k = 0; k < rope_dim / 2; ++k) {
    const double f = std::pow((double)theta, -2.0 * k / rope_dim) / (2.0 * 3.14159265358979323846);  // turns / pos
    // f < 1: its 2^64 fixed-point form is an exact product of the double with 2^64, split in halves
    const double hi = std::floor(std::ldexp(f, 32));
    const double lo = std::ldexp(f, 64) - std::ldexp(hi, 32);
    t.turns[k] = ((uint64_t)hi << 32) + (uint64_t)std::llround(lo);
  }
  return t;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA; }

constexpr unsigned kF32 = 1u << CSA_F32, kBF16 = 1u << CSA_BF16, kE4M3 = 1u << CSA_E4M3,
                   kE2M1 = 1u << CSA_E2M1, kE4M3R = 1u << CSA_E4M3R;

size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

// cuTensorMapEncodeTiled, fetched from the driver once.
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiled encode_tiled() {
  static EncodeTiled fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

}  // namespace

namespace {
std::atomic<uint64_t> g_launches{0};
}  // namespace

void csa::count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

cudaError_t csa::sm_count(int* n) {
  static PerDevice sms;
  return with_device_slot(sms, [n](int dev, int64_t& v) {
    if (!v) {
      int c = 0;
      const cudaError_t e = cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      if (c <= 0) return cudaErrorInvalidDevice;
      v = c;
    }
    *n = (int)v;
    return cudaSuccess;
  });
}

bool csa::encode_bf16_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t stride_bytes,
                          uint32_t box_cols, uint32_t box_rows) {
  const EncodeTiled fn = encode_tiled();
  if (!fn || (reinterpret_cast<uintptr_t>(base) & 15) || (stride_bytes & 15) || rows == 0) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {stride_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int csa::check_indexer_topk(const void* q_idx, int32_t q_dtype, const float* w, int32_t n_rows, int32_t idx_heads,
                            int32_t idx_dim, const int32_t* seq_id, const int32_t* pos, int32_t ratio,
                            int32_t window, const csa_paged* idx_cache, const csa_block_table* bt, int32_t k,
                            int32_t max_n, const int32_t* out_idx, const int32_t* err) {
  if (n_rows < 0 || k <= 0 || max_n < 0 || idx_heads <= 0 || idx_dim <= 0) return CSA_ERR_INVALID_ARG;
  if (ratio <= 0 || window <= 0 || 256 % ratio) return CSA_ERR_INVALID_ARG;
  if (n_rows == 0) return CSA_OK;
  if (!q_idx || !w || !seq_id || !pos || !out_idx || !err) return CSA_ERR_INVALID_ARG;
  if (q_dtype != CSA_F32 && q_dtype != CSA_BF16) return CSA_ERR_UNSUPPORTED;
  int st = check_paged(idx_cache, idx_dim, 256 / ratio, kF32 | kBF16 | kE2M1);
  if (st) return st;
  if ((st = check_bt(bt))) return st;
  if ((size_t)idx_heads * idx_dim > 32768 || idx_dim > 256) return CSA_ERR_UNSUPPORTED;
  return CSA_OK;
}

int csa::enqueue_indexer_topk(const void* q_idx, int32_t q_dtype, const float* w, int32_t n_rows, int32_t idx_heads,
                              int32_t idx_dim, const int32_t* seq_id, const int32_t* pos, int32_t ratio,
                              int32_t window, const csa_paged* idx_cache, const csa_block_table* bt, int32_t k,
                              int32_t max_n, int32_t* out_idx, float* scores, void* cand, void* deal,
                              int32_t* err, cudaStream_t stream) {
  IndexerArgs ia{};
  ia.q_idx = q_idx;
  ia.q_dtype = q_dtype;
  ia.w = w;
  ia.seq_id = seq_id;
  ia.pos = pos;
  ia.cache = *idx_cache;
  ia.bt = *bt;
  ia.heads = idx_heads;
  ia.dim = idx_dim;
  ia.ratio = ratio;
  ia.window = window;
  ia.max_n = max_n;
  ia.scores = scores;
  ia.err = err;
  const bool tc = indexer_tc_eligible(ia);
  int n_sm = 0;
  if (sm_count(&n_sm) != cudaSuccess) return CSA_ERR_CUDA;
  const int32_t G = n_sm < kDealMaxCtas ? n_sm : kDealMaxCtas;
  // a balanced deal with the selection fused when the rows' tiles fit the CTAs' key stores
  const int32_t bound = indexer_deal_bound(n_rows, max_n, G);
  if (tc && deal && max_n > 0 && bound >= 0 && bound <= indexer_deal_capacity(idx_cache->dtype)) {
    const DealCandidates dc = deal_candidates(deal, G, k);
    ia.sel_k = k;
    ia.cand_key = dc.key;
    ia.cand_idx = dc.idx;
    ia.cand_cnt = dc.cnt;
    ia.cand_thr = dc.thr;
    ia.cand_row_first = dc.row_first;
    ia.cand_row_ctas = dc.row_ctas;
    ia.cand_row_seg = dc.row_seg;
    if (launch_indexer_tc(ia, n_rows, G, stream) != cudaSuccess) return CSA_ERR_CUDA;
    TopkArgs ta{scores, pos, ratio, window, max_n, k, out_idx, err};
    return cuda_status(launch_topk_deal_merge(ta, n_rows, dc, stream));
  }
  cudaError_t e = tc ? launch_indexer_tc(ia, n_rows, G, stream) : launch_indexer_scores(ia, n_rows, stream);
  if (e != cudaSuccess) return CSA_ERR_CUDA;
  TopkArgs ta{scores, pos, ratio, window, max_n, k, out_idx, err};
  return cuda_status(launch_topk(ta, n_rows, cand, stream));
}

namespace {

// The tensor-core attention's query tensor: n_rows*64 rows of 512 bf16, boxes of
// 64 dims x 64 heads, 128-byte swizzle (the layout of its shared Q operand).
bool encode_q_map(CUtensorMap* m, const void* q, int32_t n_rows) {
  return encode_bf16_map(m, q, 512, (uint64_t)n_rows * 64, 512 * 2, 64, 64);
}

int attn_common(const csa_layer* L, const void* q, int32_t q_dtype, int32_t n_rows, const int32_t* seq_id,
                const int32_t* pos, const csa_paged* comp, const csa_block_table* comp_bt, const int32_t* topk,
                int32_t k, int32_t max_n, const csa_paged* swa, const csa_block_table* swa_bt, void* out,
                int32_t out_dtype, float* out_scales, void* ws, size_t ws_bytes, int32_t* err,
                csa_stream_t stream) {
  int st = check_layer(L);
  if (st) return st;
  if (n_rows < 0 || max_n < 0 || (topk && k <= 0)) return CSA_ERR_INVALID_ARG;
  if (n_rows == 0) return CSA_OK;
  if (!q || !seq_id || !pos || !out || !err) return CSA_ERR_INVALID_ARG;
  if (q_dtype != CSA_F32 && q_dtype != CSA_BF16) return CSA_ERR_UNSUPPORTED;
  if (out_dtype != CSA_F32 && out_dtype != CSA_BF16 && out_dtype != CSA_E4M3) return CSA_ERR_UNSUPPORTED;
  if (out_dtype == CSA_E4M3 && !out_scales) return CSA_ERR_INVALID_ARG;
  if ((st = check_paged(comp, L->dim, 256 / L->ratio, kF32 | kBF16 | kE4M3 | kE4M3R))) return st;
  if ((st = check_paged(swa, L->dim, 256, kF32 | kBF16 | kE4M3 | kE4M3R))) return st;
  if ((st = check_bt(comp_bt)) || (st = check_bt(swa_bt))) return st;
  if (L->dim % 32 || L->dim > 512 || L->heads % 8) return CSA_ERR_UNSUPPORTED;
  const int32_t keys = (topk ? k : max_n) + L->swa;
  AttnArgs a;
  a.q = q;
  a.q_dtype = q_dtype;
  a.seq_id = seq_id;
  a.pos = pos;
  a.comp = *comp;
  a.comp_bt = *comp_bt;
  a.topk = topk;
  a.k = topk ? k : 0;
  a.swa = *swa;
  a.swa_bt = *swa_bt;
  a.out = out;
  a.out_dtype = out_dtype;
  a.out_scales = out_scales;
  a.heads = L->heads;
  a.dim = L->dim;
  a.ratio = L->ratio;
  a.window = L->window;
  a.swa_len = L->swa;
  a.scale = L->scale;
  a.rope = make_rope(L->rope_dim, L->rope_theta);
  const bool tc = attn_tc_eligible(a);
  std::memset(&a.q_map, 0, sizeof(a.q_map));
  a.q_tma = tc && q_dtype == CSA_BF16 && encode_q_map(&a.q_map, q, n_rows);
  a.n_splits = tc ? attn_tc_splits(n_rows, keys) : attn_splits(n_rows, L->heads, keys);
  const size_t need = attn_workspace_bytes(n_rows, L->heads, L->dim, a.n_splits);
  if (need && (!ws || ws_bytes < need)) return CSA_ERR_WORKSPACE;
  a.part_o = reinterpret_cast<float*>(ws);
  a.part_ml = need ? a.part_o + (size_t)n_rows * L->heads * a.n_splits * L->dim : nullptr;
  a.err = err;
  return cuda_status(tc ? launch_attn_tc(a, n_rows, stream) : launch_attn(a, n_rows, keys, stream));
}

}  // namespace

extern "C" {

namespace {

int compress_insert(const csa_layer* L, const void* kv, const void* gate, int32_t in_dtype, int32_t n_tok,
                    const int32_t* seq_id, const int32_t* pos, const float* bias, const float* gamma_c,
                    const float* gamma_swa, const csa_paged* state, const csa_block_table* state_bt,
                    const csa_paged* swa, const csa_block_table* swa_bt, const csa_paged* comp,
                    const csa_block_table* comp_bt, const csa_query_norm* qn, int32_t* err, csa_stream_t stream) {
  int st = check_layer(L);
  if (st) return st;
  if (n_tok < 0) return CSA_ERR_INVALID_ARG;
  if (n_tok == 0) return CSA_OK;
  if (!kv || !gate || !seq_id || !pos || !bias || !gamma_c || !err) return CSA_ERR_INVALID_ARG;
  if (swa && !gamma_swa) return CSA_ERR_INVALID_ARG;
  if (in_dtype != CSA_F32 && in_dtype != CSA_BF16) return CSA_ERR_UNSUPPORTED;
  if (L->dim > 4096) return CSA_ERR_UNSUPPORTED;
  if ((st = check_paged(state, 2 * L->dim, 256, 1u << in_dtype))) return st;
  if (swa && (st = check_paged(swa, L->dim, 256, kF32 | kBF16 | kE4M3 | kE4M3R))) return st;
  if ((st = check_paged(comp, L->dim, 256 / L->ratio, kF32 | kBF16 | kE4M3 | kE4M3R | kE2M1))) return st;
  if ((st = check_bt(state_bt)) || (swa && (st = check_bt(swa_bt))) || (st = check_bt(comp_bt))) return st;
  QNormArgs qa{};
  if (qn) {
    if (!qn->q || !qn->gamma || !qn->q_out) return CSA_ERR_INVALID_ARG;
    if (qn->heads < 1 || qn->heads > 1024) return CSA_ERR_INVALID_ARG;
    if ((qn->q_dtype != CSA_F32 && qn->q_dtype != CSA_BF16) || (qn->out_dtype != CSA_F32 && qn->out_dtype != CSA_BF16))
      return CSA_ERR_UNSUPPORTED;
    const uintptr_t al = reinterpret_cast<uintptr_t>(qn->q) | reinterpret_cast<uintptr_t>(qn->gamma) |
                         reinterpret_cast<uintptr_t>(qn->q_out);
    if (L->dim % 8 || L->dim > 512 || al % 16) return CSA_ERR_UNSUPPORTED;
    qa = QNormArgs{qn->q, qn->q_dtype, qn->gamma, qn->q_out, qn->out_dtype, qn->heads, L->dim, L->rms_eps};
  }
  const RopeTab rt = make_rope(L->rope_dim, L->rope_theta);
  const csa_paged no_swa{};
  const csa_block_table no_swa_bt{};
  IngestArgs ia{kv, gate, in_dtype, seq_id, pos, gamma_swa, *state, *state_bt, swa ? *swa : no_swa,
                swa ? *swa_bt : no_swa_bt, L->dim, L->rms_eps, rt, err};
  EmitArgs ea{seq_id, pos, bias, gamma_c, *state, *state_bt, *comp, *comp_bt, L->dim, L->ratio, L->window,
              L->rms_eps, rt, err};
  if (compress_fused_eligible(ia, ea, n_tok)) return cuda_status(launch_compress_fused(ia, ea, qa, n_tok, stream));
  cudaError_t e = launch_ingest(ia, qa, n_tok, stream);
  if (e != cudaSuccess) return CSA_ERR_CUDA;
  return cuda_status(launch_emit(ea, n_tok, stream));
}

}  // namespace

int csa_compress_insert(const csa_layer* L, const void* kv, const void* gate, int32_t in_dtype, int32_t n_tok,
                        const int32_t* seq_id, const int32_t* pos, const float* bias, const float* gamma_c,
                        const float* gamma_swa, const csa_paged* state, const csa_block_table* state_bt,
                        const csa_paged* swa, const csa_block_table* swa_bt, const csa_paged* comp,
                        const csa_block_table* comp_bt, int32_t* err, csa_stream_t stream) {
  return compress_insert(L, kv, gate, in_dtype, n_tok, seq_id, pos, bias, gamma_c, gamma_swa, state, state_bt, swa,
                         swa_bt, comp, comp_bt, nullptr, err, stream);
}

int csa_compress_insert_qnorm(const csa_layer* L, const void* kv, const void* gate, int32_t in_dtype,
                              int32_t n_tok, const int32_t* seq_id, const int32_t* pos, const float* bias,
                              const float* gamma_c, const float* gamma_swa, const csa_paged* state,
                              const csa_block_table* state_bt, const csa_paged* swa, const csa_block_table* swa_bt,
                              const csa_paged* comp, const csa_block_table* comp_bt, const csa_query_norm* qn,
                              int32_t* err, csa_stream_t stream) {
  if (!qn) return CSA_ERR_INVALID_ARG;
  return compress_insert(L, kv, gate, in_dtype, n_tok, seq_id, pos, bias, gamma_c, gamma_swa, state, state_bt, swa,
                         swa_bt, comp, comp_bt, qn, err, stream);
}

int csa_cache_store(const float* rows, int32_t n, const int32_t* seq_id, const int32_t* row_idx,
                    const csa_paged* cache, const csa_block_table* bt, int32_t* err, csa_stream_t stream) {
  if (n < 0) return CSA_ERR_INVALID_ARG;
  if (n == 0) return CSA_OK;
  if (!rows || !seq_id || !row_idx || !err || !cache) return CSA_ERR_INVALID_ARG;
  int st = check_paged(cache, cache->dim, cache->rows_per_block, kF32 | kBF16 | kE4M3 | kE4M3R | kE2M1);
  if (st) return st;
  if (cache->dim <= 0 || cache->rows_per_block <= 0 || cache->dim % 2) return CSA_ERR_INVALID_ARG;
  if ((st = check_bt(bt))) return st;
  StoreArgs a{rows, seq_id, row_idx, *cache, *bt, err};
  return cuda_status(launch_store(a, n, stream));
}

size_t csa_indexer_topk_workspace_size(int32_t n_rows, int32_t max_n, int32_t k) {
  if (n_rows <= 0 || max_n <= 0 || k <= 0) return 0;
  // the per-row path's scores and chunk candidates, plus (for batches a
  // balanced deal may take) the deal's candidate lists for up to kDealMaxCtas CTAs
  const size_t per_row = align_up(sizeof(float) * (size_t)n_rows * max_n) +
                         align_up(topk_candidate_bytes(n_rows, max_n, k));
  const size_t deal = n_rows < kDealMaxCtas ? align_up(deal_candidate_bytes(kDealMaxCtas, k)) : 0;
  return per_row + deal;
}

int csa_indexer_topk(const void* q_idx, int32_t q_dtype, const float* w, int32_t n_rows, int32_t idx_heads,
                     int32_t idx_dim, const int32_t* seq_id, const int32_t* pos, int32_t ratio, int32_t window,
                     const csa_paged* idx_cache, const csa_block_table* bt, int32_t k, int32_t max_n,
                     int32_t* out_idx, void* ws, size_t ws_bytes, int32_t* err, csa_stream_t stream) {
  const int st = check_indexer_topk(q_idx, q_dtype, w, n_rows, idx_heads, idx_dim, seq_id, pos, ratio, window,
                                    idx_cache, bt, k, max_n, out_idx, err);
  if (st != CSA_OK || n_rows == 0) return st;
  const size_t need = csa_indexer_topk_workspace_size(n_rows, max_n, k);
  if (need && (!ws || ws_bytes < need)) return CSA_ERR_WORKSPACE;
  float* scores = reinterpret_cast<float*>(ws);
  uint8_t* after_scores = reinterpret_cast<uint8_t*>(ws) + align_up(sizeof(float) * (size_t)n_rows * max_n);
  void* cand = topk_candidate_bytes(n_rows, max_n, k) ? after_scores : nullptr;
  void* deal = n_rows < kDealMaxCtas && need
                   ? after_scores + align_up(topk_candidate_bytes(n_rows, max_n, k))
                   : nullptr;
  return enqueue_indexer_topk(q_idx, q_dtype, w, n_rows, idx_heads, idx_dim, seq_id, pos, ratio, window, idx_cache,
                              bt, k, max_n, out_idx, scores, cand, deal, err, stream);
}

size_t csa_sparse_attn_workspace_size(const csa_layer* L, int32_t n_rows, int32_t k_or_max_n) {
  if (!L || n_rows <= 0 || L->heads <= 0 || L->dim <= 0) return 0;
  // the cache dtype decides between the two kernels; size for the larger
  const int32_t keys = k_or_max_n + L->swa;
  const int32_t s = attn_splits(n_rows, L->heads, keys);
  const int32_t s_tc = attn_tc_splits(n_rows, keys);
  const size_t a = attn_workspace_bytes(n_rows, L->heads, L->dim, s);
  const size_t b = attn_workspace_bytes(n_rows, L->heads, L->dim, s_tc);
  return align_up(a > b ? a : b);
}

int csa_sparse_attn_decode(const csa_layer* L, const void* q, int32_t q_dtype, int32_t n_rows,
                           const int32_t* seq_id, const int32_t* pos, const csa_paged* comp,
                           const csa_block_table* comp_bt, const int32_t* topk, int32_t k, int32_t max_n,
                           const csa_paged* swa, const csa_block_table* swa_bt, void* out, int32_t out_dtype,
                           float* out_scales, void* ws, size_t ws_bytes, int32_t* err, csa_stream_t stream) {
  return attn_common(L, q, q_dtype, n_rows, seq_id, pos, comp, comp_bt, topk, k, max_n, swa, swa_bt, out,
                     out_dtype, out_scales, ws, ws_bytes, err, stream);
}

int csa_sparse_attn_prefill(const csa_layer* L, const void* q, int32_t q_dtype, int32_t n_rows,
                            const int32_t* seq_id, const int32_t* pos, const csa_paged* comp,
                            const csa_block_table* comp_bt, const int32_t* topk, int32_t k, int32_t max_n,
                            const csa_paged* swa, const csa_block_table* swa_bt, void* out, int32_t out_dtype,
                            float* out_scales, void* ws, size_t ws_bytes, int32_t* err, csa_stream_t stream) {
  return attn_common(L, q, q_dtype, n_rows, seq_id, pos, comp, comp_bt, topk, k, max_n, swa, swa_bt, out,
                     out_dtype, out_scales, ws, ws_bytes, err, stream);
}

int csa_read_status(int32_t* err, int32_t reset, csa_stream_t stream) {
  if (!err) return CSA_ERR_INVALID_ARG;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, err, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return CSA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return CSA_ERR_CUDA;
  if (reset && v != 0) {
    if (cudaMemsetAsync(err, 0, sizeof(int32_t), stream) != cudaSuccess) return CSA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return CSA_ERR_CUDA;
  }
  return v;
}

const char* csa_status_string(int32_t s) {
  switch (s) {
    case CSA_OK: return "ok";
    case CSA_ERR_INVALID_ARG: return "invalid argument";
    case CSA_ERR_UNSUPPORTED: return "unsupported combination";
    case CSA_ERR_CUDA: return "CUDA error";
    case CSA_ERR_DEVICE_BOUNDS: return "device: unmapped or out-of-range block or index";
    case CSA_ERR_WORKSPACE: return "workspace too small";
    case CSA_ERR_TIMEOUT: return "device: a bounded wait gave up";
    default: return "unknown status";
  }
}

int32_t csa_version(void) { return kVersion; }

uint64_t csa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
