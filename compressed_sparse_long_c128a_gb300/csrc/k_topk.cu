// DSA top-k: the min(k, n) largest indexer scores of each row, equal scores
// going to the lower entry index ("vLLM解密：DeepSeek-V4本地部署為何如此困難"
// §二 item 3: k = 512 on c4a).  The radix select itself is in select.cuh.
//
// Three ways in, by how the indexer left its results:
//   * candidates of a balanced deal (decode batches): the indexer CTAs selected
//     the top-k of their own tile ranges; topk_deal_merge_kernel merges each
//     row's candidate lists (in entry order, so ties still go to the lower index).
//   * a score row of at most 16384 entries (or several chunks of that size):
//     topk_chunk_kernel selects each chunk in shared memory, writing the row's
//     result directly when it is one chunk, else per-chunk candidates that
//     topk_merge_kernel merges.  The global top-k is a subset of the union of
//     the chunks' top-k sets because the order is total.
//   * rows whose candidates would not fit in shared memory: topk_kernel, one
//     CTA streaming the row's scores.

#include "select.cuh"

namespace csa {
namespace {

// ------------------------------------------------------------------ selection streamed from global memory

struct StreamScratch {
  uint32_t hist[4096];
  uint32_t warp_cnt[32];
  uint32_t digit, rem, eq_base, total;
  int out_ctr;
};

// Exact top-min(k, V') of the V' valid keys among positions v in [0, V), read
// through keyf(v, &key) -> valid, by one block of NT threads: three histogram
// passes (12, 12, 8 bits) over the keys in L2, then one pass in position order.
// out(v, slot) receives every selected v at a distinct slot in [0, kk): the keys
// above the k-th key first, then those equal to it, each in position order;
// returns kk.
template <int NT, typename KeyFn, typename Out>
__device__ int stream_select(int V, int k, KeyFn keyf, Out out, StreamScratch& ss) {
  constexpr int kWarps = NT / 32;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    ss.total = 0;
    ss.out_ctr = 0;
    ss.eq_base = 0;
  }
  __syncthreads();
  uint32_t cnt = 0;
  for (int v = threadIdx.x; v < V; v += NT) {
    uint32_t key;
    cnt += keyf(v, key) ? 1u : 0u;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if (lane == 0) atomicAdd(&ss.total, cnt);
  __syncthreads();
  const int total = (int)ss.total;
  const int kk = total < k ? total : k;
  if (kk == total) {  // every valid key is selected: compact in position order
    for (int v0 = 0; v0 < V; v0 += NT) {
      const int v = v0 + threadIdx.x;
      uint32_t key;
      const bool ok = v < V && keyf(v, key);
      const uint32_t bal = __ballot_sync(0xffffffffu, ok);
      if (lane == 0) ss.warp_cnt[wid] = __popc(bal);
      __syncthreads();
      uint32_t off = 0, tot = 0;
      for (int w = 0; w < kWarps; ++w) {
        off += w < wid ? ss.warp_cnt[w] : 0u;
        tot += ss.warp_cnt[w];
      }
      if (ok) out(v, (int)(ss.eq_base + off + __popc(bal & ((1u << lane) - 1u))));
      __syncthreads();
      if (threadIdx.x == 0) ss.eq_base += tot;
      __syncthreads();
    }
    return kk;
  }
  uint32_t prefix = 0, mask = 0, rem = (uint32_t)kk;
  const int shifts[3] = {20, 8, 0};
  const int widths[3] = {12, 12, 8};
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = shifts[pass], nb = 1 << widths[pass];
    for (int b = threadIdx.x; b < nb; b += NT) ss.hist[b] = 0;
    __syncthreads();
    for (int v = threadIdx.x; v < V; v += NT) {
      uint32_t key;
      if (keyf(v, key) && (key & mask) == prefix) atomicAdd(&ss.hist[(key >> sh) & (nb - 1)], 1u);
    }
    __syncthreads();
    if (wid == 0) {
      const int per = nb / 32;
      const int hi = nb - lane * per;  // this lane owns buckets [hi-per, hi), scanned downwards
      uint32_t ls = 0;
      for (int b = hi - 1; b >= hi - per; --b) ls += ss.hist[b];
      uint32_t inc = ls;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      const uint32_t exc = inc - ls;
      if (exc < rem && rem <= inc) {
        uint32_t cum = exc;
        for (int b = hi - 1; b >= hi - per; --b) {
          const uint32_t h = ss.hist[b];
          if (cum + h >= rem) {
            ss.digit = (uint32_t)b;
            ss.rem = rem - cum;
            break;
          }
          cum += h;
        }
      }
    }
    __syncthreads();
    prefix |= ss.digit << sh;
    mask |= (uint32_t)(nb - 1) << sh;
    rem = ss.rem;
    __syncthreads();
  }
  // keys above T go to slots [0, n_gt) and the first `rem` keys equal to T to
  // [n_gt, kk), each group in position order (a deterministic output order)
  const uint32_t T = prefix;
  const uint32_t n_gt = (uint32_t)kk - rem;
  for (int v0 = 0; v0 < V; v0 += NT) {
    const int v = v0 + threadIdx.x;
    uint32_t key = 0;
    const bool ok = v < V && keyf(v, key);
    const bool gt = ok && key > T, eq = ok && key == T;
    const uint32_t bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) ss.warp_cnt[wid] = __popc(bg) | ((uint32_t)__popc(be) << 16);
    __syncthreads();
    uint32_t off_g = 0, off_e = 0, tot_g = 0, tot_e = 0;
    for (int w = 0; w < kWarps; ++w) {
      const uint32_t c = ss.warp_cnt[w];
      off_g += w < wid ? (c & 0xFFFF) : 0u;
      off_e += w < wid ? (c >> 16) : 0u;
      tot_g += c & 0xFFFF;
      tot_e += c >> 16;
    }
    const uint32_t below = (1u << lane) - 1u;
    if (gt) out(v, (int)(ss.out_ctr + off_g + __popc(bg & below)));
    const uint32_t rank = ss.eq_base + off_e + __popc(be & below);
    if (eq && rank < rem) out(v, (int)(n_gt + rank));
    __syncthreads();
    if (threadIdx.x == 0) {
      ss.out_ctr += (int)tot_g;
      ss.eq_base += tot_e;
    }
    __syncthreads();
  }
  return kk;
}

constexpr int kThreads = 1024;

// One CTA per row streaming the row's scores (rows too long for the chunked path).
__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkArgs a) {
  __shared__ StreamScratch ss;
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  int n = n_visible(a.pos[r], a.ratio, a.window);
  if (n > a.max_n) {
    if (threadIdx.x == 0) record_error(a.err, CSA_ERR_DEVICE_BOUNDS);
    n = a.max_n;
  }
  const float* s = a.scores + (int64_t)r * a.max_n;
  int32_t* out = a.out + (int64_t)r * a.k;
  const int kk = stream_select<kThreads>(
      n, a.k,
      [&](int v, uint32_t& key) {
        key = order_key(s[v]);
        return true;
      },
      [&](int v, int slot) { out[slot] = v; }, ss);
  for (int i = kk + threadIdx.x; i < a.k; i += kThreads) out[i] = -1;
}

// ------------------------------------------------------------------ merge of a balanced deal's candidates

constexpr int kDealMergeThreads = 1024;
constexpr int kDealMergeCap = 20480;  // survivors of a row held in shared memory
constexpr int kRankMax = 2048;        // survivors ranked by counting (beyond: radix select)
constexpr size_t kDealMergeSmem = sizeof(uint32_t) * (padded_size(kDealMergeCap) + kDealMergeCap);

// Row r: its CTAs' lists under the deal merged into the row's top-k.  CTA c's
// list holds every key of its range at or above thr_c, and thr_c is at most
// the row's k-th largest key, so the keys at or above max_c thr_c are all in
// the lists and include the row's top-k.  Those survivors are gathered in
// entry order (one warp per list, ballot compaction) and ranked: by counting
// when there are few (rank = keys above + equal keys before, so equal scores
// go to the lower entry index), else by radix select.
__global__ void __launch_bounds__(kDealMergeThreads) topk_deal_merge_kernel(const TopkArgs a,
                                                                            const DealCandidates c, int n_rows) {
  extern __shared__ uint32_t msm[];
  uint32_t* keys = msm;                                                        // padded_size(cap)
  int32_t* idx = reinterpret_cast<int32_t*>(msm + padded_size(kDealMergeCap));  // [cap]
  __shared__ DealShared ds;
  __shared__ int32_t off[kDealMaxRows + 1];  // survivors before each of the row's lists
  __shared__ uint32_t s_thr;
  __shared__ SelectScratch sc;
  __shared__ StreamScratch ss;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_trigger();
  if (warp == 0) deal_compute(a.pos, n_rows, a.ratio, a.window, a.max_n, c.ctas, ds);
  pdl_wait();  // the lists are complete only after the indexer launch
  __syncthreads();
  const int r = blockIdx.x;
  const int first = ds.first[r], ctas = ds.ctas[r];
  const int K = a.k;
  int32_t* out = a.out + (int64_t)r * K;
  if (warp == 0) {
    uint32_t t = 0;
    for (int j = lane; j < ctas; j += 32) t = max(t, c.thr[first + j]);
    for (int o = 16; o > 0; o >>= 1) t = max(t, __shfl_xor_sync(0xffffffffu, t, o));
    if (lane == 0) s_thr = t;
  }
  __syncthreads();
  const uint32_t thr = s_thr;
  // survivors per list
  for (int j = warp; j < ctas; j += kDealMergeThreads / 32) {
    const int n = c.cnt[first + j];
    const uint32_t* lk = c.key + (int64_t)(first + j) * c.cap;
    int cnt = 0;
    for (int i0 = 0; i0 < n; i0 += 32) {
      const int i = i0 + lane;
      cnt += __popc(__ballot_sync(0xffffffffu, i < n && lk[i] >= thr));
    }
    if (lane == 0) off[j + 1] = cnt;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    off[0] = 0;
    for (int j = 0; j < ctas; ++j) off[j + 1] += off[j];
  }
  __syncthreads();
  const int m = off[ctas];
  int kk;
  if (m <= kDealMergeCap) {
    for (int j = warp; j < ctas; j += kDealMergeThreads / 32) {
      const int n = c.cnt[first + j];
      const int64_t base = (int64_t)(first + j) * c.cap;
      int at = off[j];
      for (int i0 = 0; i0 < n; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t key = i < n ? c.key[base + i] : 0u;
        const bool keep = i < n && key >= thr;
        const uint32_t b = __ballot_sync(0xffffffffu, keep);
        if (keep) {
          const int q = at + __popc(b & ((1u << lane) - 1u));
          keys[padded(q)] = key;
          idx[q] = c.idx[base + i];
        }
        at += __popc(b);
      }
    }
    __syncthreads();
    if (m <= kRankMax) {
      for (int i = threadIdx.x; i < m; i += kDealMergeThreads) {
        const uint32_t ki = keys[padded(i)];
        int rank = 0;
        for (int j = 0; j < m; ++j) {
          const uint32_t kj = keys[padded(j)];
          rank += (kj > ki) || (kj == ki && j < i);
        }
        if (rank < K) out[rank] = idx[i];
      }
    } else {
      block_select<kDealMergeThreads>(keys, m, K, sc, [&](int pos, uint32_t rank) { out[rank] = idx[pos]; });
    }
    kk = m < K ? m : K;
  } else {
    kk = stream_select<kDealMergeThreads>(
        ctas * c.cap, K,
        [&](int v, uint32_t& key) {
          const int j = first + v / c.cap, i = v % c.cap;
          if (i >= c.cnt[j]) return false;
          key = c.key[(int64_t)j * c.cap + i];
          return key >= thr;
        },
        [&](int v, int slot) { out[slot] = c.idx[(int64_t)(first + v / c.cap) * c.cap + v % c.cap]; }, ss);
  }
  for (int i = kk + threadIdx.x; i < K; i += kDealMergeThreads) out[i] = -1;
}

constexpr int kChunk = 16384;
constexpr int kChunkThreads = 1024;
constexpr int kMergeThreads = 1024;
constexpr size_t kChunkSmem = sizeof(uint32_t) * padded_size(kChunk);

// One chunk of kChunk scores of a row: its top-k, written as (key, index)
// candidates in index order, or -- when the row is a single chunk -- straight
// to the output (padded with -1).
__global__ void __launch_bounds__(kChunkThreads) topk_chunk_kernel(const TopkArgs a, uint32_t* cand_key,
                                                                    int32_t* cand_idx, int32_t* cand_cnt,
                                                                    int n_chunks) {
  extern __shared__ uint32_t keys[];  // padded_size(kChunk)
  __shared__ SelectScratch sc;
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x, c = blockIdx.y;
  int n = n_visible(a.pos[r], a.ratio, a.window);
  if (n > a.max_n) {
    if (threadIdx.x == 0 && c == 0) record_error(a.err, CSA_ERR_DEVICE_BOUNDS);
    n = a.max_n;
  }
  const int lo = c * kChunk;
  const int len = max(0, min(kChunk, n - lo));
  const bool final_out = n_chunks == 1;
  int32_t* out = a.out + (int64_t)r * a.k;
  if (final_out)
    for (int i = min(len, a.k) + threadIdx.x; i < a.k; i += kChunkThreads) out[i] = -1;
  const int64_t slot = (int64_t)r * n_chunks + c;
  if (len <= 0) {
    if (threadIdx.x == 0 && !final_out) cand_cnt[slot] = 0;
    return;
  }
  const float* s = a.scores + (int64_t)r * a.max_n + lo;
  // all of a thread's loads are issued before any is stored
  constexpr int kLoads = kChunk / kChunkThreads;
  float v[kLoads];
#pragma unroll
  for (int u = 0; u < kLoads; ++u) {
    const int i = threadIdx.x + u * kChunkThreads;
    v[u] = i < len ? s[i] : 0.f;
  }
#pragma unroll
  for (int u = 0; u < kLoads; ++u) {
    const int i = threadIdx.x + u * kChunkThreads;
    if (i < len) keys[padded(i)] = order_key(v[u]);
  }
  __syncthreads();
  if (final_out) {
    block_select<kChunkThreads>(keys, len, a.k, sc, [&](int pos, uint32_t rank) { out[rank] = pos; });
    return;
  }
  uint32_t* ok = cand_key + slot * a.k;
  int32_t* oi = cand_idx + slot * a.k;
  block_select<kChunkThreads>(keys, len, a.k, sc, [&](int pos, uint32_t rank) {
    ok[rank] = keys[padded(pos)];
    oi[rank] = lo + pos;
  });
  if (threadIdx.x == 0) cand_cnt[slot] = min(len, a.k);
}

__global__ void __launch_bounds__(kMergeThreads) topk_merge_kernel(const TopkArgs a, const uint32_t* cand_key,
                                                                    const int32_t* cand_idx,
                                                                    const int32_t* cand_cnt, int n_chunks) {
  extern __shared__ uint32_t msm[];
  const int cap = n_chunks * a.k;
  uint32_t* keys = msm;                                             // padded_size(cap)
  int32_t* idx = reinterpret_cast<int32_t*>(msm + padded_size(cap));  // [cap]
  __shared__ int32_t off[65];
  __shared__ SelectScratch sc;
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  if (threadIdx.x == 0) {
    int32_t t = 0;
    for (int c = 0; c < n_chunks; ++c) {
      off[c] = t;
      t += cand_cnt[(int64_t)r * n_chunks + c];
    }
    off[n_chunks] = t;
  }
  __syncthreads();
  const int total = off[n_chunks];
  for (int c = 0; c < n_chunks; ++c) {
    const int cnt = off[c + 1] - off[c];
    const int64_t slot = (int64_t)r * n_chunks + c;
    for (int j = threadIdx.x; j < cnt; j += kMergeThreads) {
      keys[padded(off[c] + j)] = cand_key[slot * a.k + j];
      idx[off[c] + j] = cand_idx[slot * a.k + j];
    }
  }
  __syncthreads();
  int32_t* out = a.out + (int64_t)r * a.k;
  block_select<kMergeThreads>(keys, total, a.k, sc, [&](int pos, uint32_t rank) { out[rank] = idx[pos]; });
  const int kk = total < a.k ? total : a.k;
  for (int i = kk + threadIdx.x; i < a.k; i += kMergeThreads) out[i] = -1;
}

size_t merge_smem(int32_t n_chunks, int32_t k) {
  const int cap = n_chunks * k;
  return sizeof(uint32_t) * (padded_size(cap) + cap);
}

}  // namespace

int32_t topk_chunks(int32_t max_n) { return (max_n + kChunk - 1) / kChunk; }

// Rows of one chunk need no candidates; more chunks need them and a merge
// whose candidates fit in shared memory.
bool topk_two_stage(int32_t max_n, int32_t k) {
  const int32_t c = topk_chunks(max_n);
  return c >= 2 && c <= 64 && merge_smem(c, k) <= 200 * 1024;
}

size_t topk_candidate_bytes(int32_t n_rows, int32_t max_n, int32_t k) {
  if (!topk_two_stage(max_n, k)) return 0;
  const size_t c = topk_chunks(max_n);
  return (size_t)n_rows * c * ((size_t)k * 8 + 4);
}

cudaError_t launch_topk(const TopkArgs& a, int32_t n_rows, void* cand, cudaStream_t s, Order first) {
  if (n_rows == 0 || a.k == 0) return cudaSuccess;
  static PerDevice chunk_attr;
  cudaError_t e = with_device_slot(chunk_attr, [](int, int64_t& done) {
    if (done) return cudaSuccess;
    const cudaError_t r =
        cudaFuncSetAttribute(topk_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kChunkSmem);
    if (r == cudaSuccess) done = 1;
    return r;
  });
  if (e != cudaSuccess) return e;
  const int32_t nc = topk_chunks(a.max_n);
  if (nc <= 1)
    return launch_k(topk_chunk_kernel, dim3(n_rows, 1), dim3(kChunkThreads), kChunkSmem, s, first, 0, a,
                    (uint32_t*)nullptr, (int32_t*)nullptr, (int32_t*)nullptr, 1);
  if (!topk_two_stage(a.max_n, a.k) || cand == nullptr)
    return launch_k(topk_kernel, dim3(n_rows), dim3(kThreads), 0, s, first, 0, a);
  uint32_t* ck = reinterpret_cast<uint32_t*>(cand);
  int32_t* ci = reinterpret_cast<int32_t*>(ck + (size_t)n_rows * nc * a.k);
  int32_t* cc = ci + (size_t)n_rows * nc * a.k;
  e = launch_k(topk_chunk_kernel, dim3(n_rows, nc), dim3(kChunkThreads), kChunkSmem, s, first, 0, a, ck, ci,
                           cc, nc);
  if (e != cudaSuccess) return e;
  const size_t smem = merge_smem(nc, a.k);
  static PerDevice merge_smem_set;  // the largest dynamic shared memory allowed so far
  e = with_device_slot(merge_smem_set, [smem](int, int64_t& set) {
    if (smem <= 48 * 1024 || (int64_t)smem <= set) return cudaSuccess;
    const cudaError_t r = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem);
    if (r == cudaSuccess) set = (int64_t)smem;
    return r;
  });
  if (e != cudaSuccess) return e;
  return launch_k(topk_merge_kernel, dim3(n_rows), dim3(kMergeThreads), smem, s, kAfterOwnKernel, 0, a,
                  (const uint32_t*)ck,
                  (const int32_t*)ci, (const int32_t*)cc, nc);
}

cudaError_t launch_topk_deal_merge(const TopkArgs& a, int32_t n_rows, const DealCandidates& c, cudaStream_t s) {
  if (n_rows == 0 || a.k == 0) return cudaSuccess;
  static PerDevice attr;
  cudaError_t e = with_device_slot(attr, [](int, int64_t& done) {
    if (done) return cudaSuccess;
    const cudaError_t r = cudaFuncSetAttribute(topk_deal_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)kDealMergeSmem);
    if (r == cudaSuccess) done = 1;
    return r;
  });
  if (e != cudaSuccess) return e;
  return launch_k(topk_deal_merge_kernel, dim3(n_rows), dim3(kDealMergeThreads), kDealMergeSmem, s,
                  kAfterOwnKernel, 0, a, c, (int)n_rows);
}

}  // namespace csa
