/*
 * csa.h -- compressed sparse attention (c4a / c128a) for GB300 (sm_103a).
 *
 * C ABI of libcsa.so: the decode / chunked-prefill hot path of DeepSeek-V4
 * style compressed sparse attention over caller-owned paged caches.
 *
 * Sources, cited as (page, section):
 *   [Support] "vLLM DeepSeek V4 Support: Efficient Long-context Attention"
 *   [部署]    "vLLM解密：DeepSeek-V4本地部署為何如此困難"
 *   [延迟]    "DeepSeek V4 inference latency optimization"
 *
 * Conventions for every entry point
 *   - All pointers to tensors are DEVICE pointers unless marked (host).  The
 *     caller owns and allocates every buffer: caches, block tables, inputs,
 *     outputs, workspaces and the error word.  The library never allocates,
 *     frees or synchronises inside the four hot-path calls; each enqueues its
 *     kernels on `stream` and returns.
 *   - Host-side validation failures return a negative csa_status and enqueue
 *     nothing.  A failed launch returns CSA_ERR_CUDA.
 *   - Conditions only the device can see (a logical block mapped to -1 or to a
 *     physical block >= num_blocks, an index outside the visible entries) are
 *     recorded in the caller's device error word `err` (first error wins, via
 *     atomicCAS from 0); the offending row or element is skipped, never read
 *     or written out of bounds.  No kernel traps or waits without a bound.
 *     csa_read_status() fetches and optionally clears the word.
 *   - Every call is ordered after all work enqueued before it on `stream`, by
 *     anyone.  Kernels are launched with programmatic dependent launch: a
 *     kernel may start while the previous kernel on the stream is finishing,
 *     but it waits for that kernel to complete before it reads or writes any
 *     memory, so only set-up that touches no memory overlaps.
 *   - Positions are 0-based.  Compressed entry i of a layer with stride
 *     `ratio` and window `window` sums raw tokens [ratio*i, ratio*i+window-1]
 *     and is anchored (rotated) at ratio*i ([延迟] "KV 缓存压缩").  A query at
 *     position p may read entry i iff ratio*i+window-1 < p ([延迟]
 *     "注意力计算剪枝": no entry may contain a future token), i.e. entries
 *     0 .. n-1 with n = p < window ? 0 : (p-window)/ratio + 1.
 */
#ifndef CSA_H
#define CSA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CSA_API __attribute__((visibility("default")))
#else
#define CSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* csa_stream_t; /* the same type as cudaStream_t */

typedef enum {
  CSA_OK = 0,
  CSA_ERR_INVALID_ARG = -1,   /* null pointer, bad size, inconsistent shapes */
  CSA_ERR_UNSUPPORTED = -2,   /* a valid combination the library has no kernel for */
  CSA_ERR_CUDA = -3,          /* a CUDA runtime call or launch failed */
  CSA_ERR_DEVICE_BOUNDS = -4, /* device: unmapped / out-of-range block or index */
  CSA_ERR_WORKSPACE = -5,     /* workspace smaller than the matching *_workspace_size */
  CSA_ERR_TIMEOUT = -6        /* device: a bounded wait inside a kernel gave up */
} csa_status;

typedef enum {
  CSA_F32 = 0,  /* float */
  CSA_BF16 = 1, /* bfloat16 */
  CSA_E4M3 = 2, /* fp8 e4m3 (fn) codes + one fp32 scale per row: value = code * scale */
  CSA_E2M1 = 3, /* fp4 e2m1 codes, two per byte (element 2j in the low nibble), plus one
                   e4m3 scale byte per 16 elements: value = code * scale */
  CSA_E4M3R = 4 /* "partial token-wise fp8" ([部署] §二: decode reads a partial
                   token-wise fp8 cache): per row, the first dim - tail_bf16 elements
                   as e4m3 codes with one fp32 scale per row (amax of those elements
                   / 448), the last tail_bf16 elements (the rotary dims) as bf16 */
} csa_dtype;

/*
 * A paged cache: `num_blocks` physical blocks of `rows_per_block` rows of `dim`
 * elements, rows packed densely:
 *   row r of block b starts at data + (b*rows_per_block + r) * row_bytes,
 *   row_bytes = dim * sizeof(element)  (E2M1: dim/2; E4M3R: dim + tail_bf16,
 *   the codes of elements [0, dim - tail_bf16) then tail_bf16 bf16 values).
 * scales: E4M3, E4M3R: float[num_blocks*rows_per_block], one per row;
 *         E2M1: uint8 e4m3 bytes [num_blocks*rows_per_block][dim/16];
 *         F32 / BF16: unused (may be NULL).
 * tail_bf16: E4M3R only (a multiple of 16, dim - tail_bf16 a multiple of 16);
 *         0 for every other dtype.
 * One logical block covers 256 native positions for every kind of cache
 * ([Support] "KV Cache Memory Management", item 1): a compressed cache has
 * 256/ratio rows per block (64 for c4a, 2 for c128a); a sliding-window cache
 * 256 rows (one per position); a compressor state cache 256 rows of
 * dim = 2*D holding the raw (kv | gate) of one position.
 */
typedef struct {
  void* data;
  void* scales;
  int32_t dtype;
  int32_t num_blocks;
  int32_t rows_per_block;
  int32_t dim;
  int32_t tail_bf16;
} csa_paged;

/* Logical block j of sequence s lives in physical block table[s*stride + j]; -1 = unmapped. */
typedef struct {
  const int32_t* table; /* device, int32 [num_seqs][stride] */
  int32_t num_seqs;
  int32_t stride;
} csa_block_table;

/* One attention layer. */
typedef struct {
  int32_t ratio;    /* compressor stride: 4 (c4a) or 128 (c128a) */
  int32_t window;   /* raw tokens per entry: 8 (c4a) or 128 (c128a) */
  int32_t dim;      /* latent dim D of entries, window rows and query heads */
  int32_t rope_dim; /* rotary dims at the end of D (even, <= D, <= 128) */
  int32_t heads;    /* query heads H */
  int32_t swa;      /* raw sliding-window length (1..256) */
  float rope_theta; /* RoPE base: pair k of the rotary dims turns by pos*theta^(-2k/rope_dim) */
  float rms_eps;    /* RMSNorm epsilon */
  float scale;      /* softmax scale applied to q.k (1/sqrt(D)) */
} csa_layer;

/*
 * csa_compress_insert -- ingest raw tokens: compressor state, sliding-window
 * rows and every compressed entry whose window closes at an ingested token.
 * [部署] §3.2 first fusion (compressor + RMSNorm + RoPE + cache write), third
 * fusion (KV RoPE + K insert for the raw window); [Support] "KV Cache Memory
 * Management" item 2 (compressor state kept as sliding-window KV).
 *
 * For each token j (position pos[j] of sequence seq_id[j]):
 *   state row (logical row pos[j]) := kv[j] | gate[j]            (raw, in_dtype)
 *   swa row   (logical row pos[j]) := RoPE(RMSNorm(kv[j]; gamma_swa), pos[j])  (if swa)
 * then, for each token whose position t satisfies t >= window-1 and
 * (t-window+1) % ratio == 0, entry i = (t-window+1)/ratio becomes
 *   c[d] = sum_{o<window} softmax_o(gate[o,d] + bias[o,d]) * kv[o,d]   (o = offset
 *          in the window, rows read from the state cache, positions ratio*i+o)
 *   comp entry i := RoPE(RMSNorm(c; gamma_c), ratio*i)
 * All state rows of the call are written before any entry is formed, so a
 * window may close on rows ingested earlier in the same call.  The window's
 * earlier rows must already be in the state cache.
 *
 *   kv, gate   [n_tok][D] in_dtype (F32 or BF16)
 *   seq_id,pos [n_tok] int32; (seq, pos) pairs must be distinct within a call
 *   bias       [window][D] float; gamma_c, gamma_swa [D] float
 *   state      dtype == in_dtype, rows_per_block 256, dim 2*D
 *   swa        F32 / BF16 / E4M3 / E4M3R, rows_per_block 256, dim D; or NULL, with
 *              swa_bt and gamma_swa unused (may be NULL): no window rows are
 *              written.  This is the indexer-key compressor ([部署] §3.2 first
 *              fusion: the indexer K cache keeps its own compress + norm + RoPE
 *              + insert), whose keys have no sliding window.
 *   comp       F32 / BF16 / E4M3 / E4M3R / E2M1, rows_per_block 256/ratio, dim D.
 *              E4M3R and E2M1 (D % 16 == 0) quantise as csa_cache_store does.
 *   err        device int32 error word
 */
CSA_API int csa_compress_insert(const csa_layer* layer, const void* kv, const void* gate, int32_t in_dtype,
                        int32_t n_tok, const int32_t* seq_id, const int32_t* pos, const float* bias,
                        const float* gamma_c, const float* gamma_swa, const csa_paged* state,
                        const csa_block_table* state_bt, const csa_paged* swa,
                        const csa_block_table* swa_bt, const csa_paged* comp,
                        const csa_block_table* comp_bt, int32_t* err, csa_stream_t stream);

/*
 * csa_query_norm -- the query half of [部署] §3.2's third fusion (Q norm + KV
 * RoPE + K insert, one kernel with warps statically given to query heads or to
 * the key): per token j and head h,
 *   q_out[j][h] := RMSNorm(q[j][h]; gamma_q)   (over the D dims of the head)
 * RoPE of the query is not applied here: csa_sparse_attn_decode / _prefill
 * rotate it.
 *   q      [n_tok][heads][D] q_dtype (F32 or BF16), 16-byte aligned
 *   gamma  [D] float, 16-byte aligned
 *   q_out  [n_tok][heads][D] out_dtype (F32 or BF16), 16-byte aligned; may equal q
 *          when the dtypes match (each element is read before it is written)
 *   heads  1..1024; eps is the layer's rms_eps.  Requires D % 8 == 0, D <= 512.
 */
typedef struct {
  const void* q;
  int32_t q_dtype;
  int32_t heads;
  const float* gamma;
  void* q_out;
  int32_t out_dtype;
} csa_query_norm;

/*
 * csa_compress_insert_qnorm -- csa_compress_insert with the query RMSNorm of
 * the same tokens fused into its launch ([部署] §3.2 third fusion; [Support]
 * "GPU Compute Saturation", kernel fusions).  The caches are written exactly as
 * csa_compress_insert writes them; qn (required) describes the query rows,
 * one per token.  Extra errors: CSA_ERR_INVALID_ARG when qn, or one of its
 * pointers, is null or heads is outside 1..1024; CSA_ERR_UNSUPPORTED for a
 * dtype other than F32 / BF16, D % 8, D > 512 or a pointer not 16-byte
 * aligned.  With n_tok == 0 the call is a no-op: only qn != NULL is checked.
 */
CSA_API int csa_compress_insert_qnorm(const csa_layer* layer, const void* kv, const void* gate,
                                      int32_t in_dtype, int32_t n_tok, const int32_t* seq_id,
                                      const int32_t* pos, const float* bias, const float* gamma_c,
                                      const float* gamma_swa, const csa_paged* state,
                                      const csa_block_table* state_bt, const csa_paged* swa,
                                      const csa_block_table* swa_bt, const csa_paged* comp,
                                      const csa_block_table* comp_bt, const csa_query_norm* qn,
                                      int32_t* err, csa_stream_t stream);

/*
 * csa_cache_store -- write fp32 rows into a paged cache, quantising to its
 * dtype: logical row row_idx[j] of sequence seq_id[j] := rows[j].  This is the
 * insert of the indexer key cache and the way a caller loads entries it
 * already holds (restored prefix, transferred KV).  [部署] §3.2 first fusion
 * (the indexer K cache keeps its own insert kernel); [Support] "DeepSeek V4
 * Attention Architecture" last paragraph (fp8 attention / fp4 indexer cache).
 * E4M3: scale = amax/448, code = e4m3_rn_satfinite(x * (448/amax)), fp32 math.
 * E2M1: per 16 elements scale = e4m3_rn(amax16/6); code = e2m1_rn_satfinite(x/scale)
 *       (a zero scale gives zero codes).
 * E4M3R: as E4M3 over elements [0, dim - tail_bf16), the rest rounded to bf16.
 *   rows [n][cache->dim] float; seq_id, row_idx [n] int32.
 */
CSA_API int csa_cache_store(const float* rows, int32_t n, const int32_t* seq_id, const int32_t* row_idx,
                    const csa_paged* cache, const csa_block_table* bt, int32_t* err,
                    csa_stream_t stream);

/*
 * csa_indexer_topk -- DSA selection ([部署] §二 item 3; [Support] "DeepSeek
 * Sparse Attention (DSA)").  For each row r at position pos[r] of sequence
 * seq_id[r]: over the n visible entries (see conventions),
 *   s_i = sum_{h<idx_heads} w[r][h] * relu(q_idx[r][h] . key_i)
 * and out_idx[r] receives the min(k, n) indices with the largest s_i, ties to
 * the lower index, in no particular order; the remaining k - min(k, n) slots
 * are -1.
 *   q_idx     [n_rows][idx_heads][idx_dim], q_dtype F32 or BF16
 *   w         [n_rows][idx_heads] float
 *   idx_cache F32 / BF16 / E2M1, rows_per_block 256/ratio, dim idx_dim
 *   out_idx   [n_rows][k] int32
 *   ws        workspace of at least csa_indexer_topk_workspace_size(n_rows, max_n, k)
 *             bytes, max_n >= every row's n.  Contents are scratch: the rows'
 *             scores and, when max_n > 16384, each 16384-entry chunk's top-k
 *             candidates; for batches of fewer than 256 rows, the candidate
 *             lists of the CTAs the rows' tiles are dealt to (two lists of up
 *             to 2k (key, index) pairs a CTA, with a count and a threshold
 *             each, and each row's first list).  Nothing needs to start at zero.
 */
CSA_API int csa_indexer_topk(const void* q_idx, int32_t q_dtype, const float* w, int32_t n_rows,
                     int32_t idx_heads, int32_t idx_dim, const int32_t* seq_id, const int32_t* pos,
                     int32_t ratio, int32_t window, const csa_paged* idx_cache,
                     const csa_block_table* bt, int32_t k, int32_t max_n, int32_t* out_idx,
                     void* ws, size_t ws_bytes, int32_t* err, csa_stream_t stream);
CSA_API size_t csa_indexer_topk_workspace_size(int32_t n_rows, int32_t max_n, int32_t k);

/*
 * csa_sparse_attn_decode -- shared-K=V attention of query rows over their
 * selected compressed entries plus the raw sliding window, one joint softmax,
 * then inverse RoPE ([Support] "DeepSeek V4 Attention Architecture": shared
 * key/value, inverse RoPE, DSA, short sliding window; [部署] §3.2 second
 * fusion: inverse RoPE + fp8 quant).  For row r at p = pos[r]:
 *   keys  = comp entries topk[r][0..k) that are not -1   (topk == NULL: every
 *           visible entry 0..n-1), followed by swa rows max(0,p-swa+1) .. p
 *   q'_h  = RoPE(q[r][h], p);  a_h = softmax_j(scale * q'_h . key_j)
 *   o_h   = RoPE^-1(sum_j a_hj key_j, p)
 * out: BF16 / F32 [n_rows][H][D], or E4M3 codes [n_rows][H][D] with
 * out_scales [n_rows][H] float (scale = amax/448 over the head's D values).
 * A selected index outside the row's visible entries sets CSA_ERR_DEVICE_BOUNDS
 * and is skipped.  Rows are independent; any mix of sequences and positions.
 *   q [n_rows][H][D] q_dtype (F32 or BF16); topk [n_rows][k] int32 or NULL
 *   comp, swa: caches as written by csa_compress_insert
 *   ws: at least csa_sparse_attn_workspace_size(layer, n_rows, k_or_max_n) bytes
 *       (k_or_max_n: k, or the largest n when topk == NULL).  Scratch.
 */
CSA_API int csa_sparse_attn_decode(const csa_layer* layer, const void* q, int32_t q_dtype, int32_t n_rows,
                           const int32_t* seq_id, const int32_t* pos, const csa_paged* comp,
                           const csa_block_table* comp_bt, const int32_t* topk, int32_t k,
                           int32_t max_n, const csa_paged* swa, const csa_block_table* swa_bt,
                           void* out, int32_t out_dtype, float* out_scales, void* ws,
                           size_t ws_bytes, int32_t* err, csa_stream_t stream);

/*
 * csa_sparse_attn_prefill -- the same operation for prefill chunks: many rows
 * per sequence, each with its own causal visibility, top-k and window ([部署]
 * §二: the same attention kernel serves prefill and decode; [Support]
 * "Deployment and Hardware Support": paged prefill reading the paged cache).
 * Arguments and results are those of csa_sparse_attn_decode; rows may mix
 * prefill and decode rows in any order.
 */
CSA_API int csa_sparse_attn_prefill(const csa_layer* layer, const void* q, int32_t q_dtype, int32_t n_rows,
                            const int32_t* seq_id, const int32_t* pos, const csa_paged* comp,
                            const csa_block_table* comp_bt, const int32_t* topk, int32_t k,
                            int32_t max_n, const csa_paged* swa, const csa_block_table* swa_bt,
                            void* out, int32_t out_dtype, float* out_scales, void* ws,
                            size_t ws_bytes, int32_t* err, csa_stream_t stream);
CSA_API size_t csa_sparse_attn_workspace_size(const csa_layer* layer, int32_t n_rows, int32_t k_or_max_n);

/*
 * csa_indexer_topk_noalloc -- csa_indexer_topk for callers that cannot
 * allocate device memory.  The pages have no counterpart: this is a calling
 * convention of this library, not part of the method.
 *
 * Some callers cannot pass a workspace: a plugin inside a host runtime that
 * owns all device memory and gives its extensions no allocator, or a serving
 * loop that may not allocate on its hot path (an allocation can wait for the
 * whole device or fail under memory pressure).  This variant computes exactly
 * what csa_indexer_topk computes, with the same arguments minus the workspace,
 * and keeps its scratch in a fixed 16 MiB array of device memory defined inside
 * the library (held on every GPU that loads the library until the process
 * exits).  It calls no allocator.
 *   - A request whose scratch (csa_indexer_topk_workspace_size(n_rows, max_n,
 *     k)) exceeds 16 MiB returns CSA_ERR_WORKSPACE and enqueues nothing.
 *   - All calls share the one array: calls that can run at the same time on
 *     the GPU (different streams, no ordering between them) race.  Calls on one
 *     stream are safe; no scratch byte needs to start at zero.
 *   - The first call on a device resolves the array's device address with
 *     that device current; make that first call before any stream capture.
 */
CSA_API int csa_indexer_topk_noalloc(const void* q_idx, int32_t q_dtype, const float* w, int32_t n_rows,
                                     int32_t idx_heads, int32_t idx_dim, const int32_t* seq_id,
                                     const int32_t* pos, int32_t ratio, int32_t window,
                                     const csa_paged* idx_cache, const csa_block_table* bt, int32_t k,
                                     int32_t max_n, int32_t* out_idx, int32_t* err, csa_stream_t stream);

/* Copy the device error word to the host (synchronises `stream`); if `reset`, zero it
 * afterwards.  Returns the recorded csa_status (CSA_OK if none) or CSA_ERR_CUDA. */
CSA_API int csa_read_status(int32_t* err, int32_t reset, csa_stream_t stream);

/* Static description of a status code. */
CSA_API const char* csa_status_string(int32_t status);

/* Library version: major*10000 + minor*100 + patch. */
CSA_API int32_t csa_version(void);

/* Kernel launches the library has enqueued in this process so far, over all
 * entry points and devices (a host-side count, also advanced while a stream is
 * being captured into a CUDA graph).  For measurement; not part of the method. */
CSA_API uint64_t csa_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* CSA_H */
