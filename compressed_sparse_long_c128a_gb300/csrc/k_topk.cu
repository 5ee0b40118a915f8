// DSA top-k: the min(k, n) largest indexer scores of each row, equal scores
// going to the lower entry index ("vLLM解密：DeepSeek-V4本地部署為何如此困難"
// §二 item 3: k = 512 on c4a).
//
// Exact radix select on an order-preserving 32-bit key of the fp32 score:
// histogram passes over the key's bits (11, 11, 10) fix the k-th largest key T
// and how many entries equal to T are still needed; a last pass in index order
// takes every entry above T and the lowest-indexed entries equal to T.
//
// Scores are cut into chunks of 16384 held in shared memory by a 1024-thread
// CTA.  A row of one chunk is selected and written out directly.  Longer rows
// take two stages: (1) every chunk writes its own top-k as (key, index)
// candidates in index order; (2) one CTA per row selects the top-k of the
// row's candidates, which are in index order chunk after chunk, so ties still
// resolve to the lower entry index.  The global top-k is a subset of the union
// of the chunks' top-k sets because the order is total.  Rows whose candidates
// would not fit in shared memory fall back to one CTA scanning the row.

#include "csa_kernels.h"

namespace csa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkArgs a) {
  __shared__ uint32_t hist[4096];
  __shared__ uint32_t warp_cnt[kWarps];
  __shared__ uint32_t sh_digit, sh_rem, sh_eq_base;
  __shared__ int out_ctr;

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
  const int kk = n < a.k ? n : a.k;
  for (int i = kk + threadIdx.x; i < a.k; i += kThreads) out[i] = -1;
  if (kk == n) {  // every visible entry is selected
    for (int i = threadIdx.x; i < n; i += kThreads) out[i] = i;
    return;
  }

  uint32_t prefix = 0, mask = 0, rem = (uint32_t)kk;
  const int shifts[3] = {20, 8, 0};
  const int widths[3] = {12, 12, 8};
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = shifts[pass];
    const int nb = 1 << widths[pass];
    for (int b = threadIdx.x; b < nb; b += kThreads) hist[b] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const uint32_t key = order_key(s[i]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> sh) & (nb - 1)], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      const int per = nb / 32;
      const int hi = nb - lane * per;  // this lane owns buckets [hi-per, hi), scanned downwards
      uint32_t ls = 0;
      for (int b = hi - 1; b >= hi - per; --b) ls += hist[b];
      uint32_t inc = ls;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
      }
      const uint32_t exc = inc - ls;
      if (exc < rem && rem <= inc) {
        uint32_t cum = exc;
        for (int b = hi - 1; b >= hi - per; --b) {
          const uint32_t h = hist[b];
          if (cum + h >= rem) {
            sh_digit = (uint32_t)b;
            sh_rem = rem - cum;
            break;
          }
          cum += h;
        }
      }
    }
    __syncthreads();
    prefix |= sh_digit << sh;
    mask |= (uint32_t)(nb - 1) << sh;
    rem = sh_rem;
    __syncthreads();
  }

  const uint32_t T = prefix;
  const uint32_t n_gt = (uint32_t)kk - rem;
  if (threadIdx.x == 0) {
    out_ctr = 0;
    sh_eq_base = 0;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int c0 = 0; c0 < n; c0 += kThreads) {
    const int i = c0 + threadIdx.x;
    const uint32_t key = i < n ? order_key(s[i]) : 0u;
    const bool gt = i < n && key > T;
    const bool eq = i < n && key == T;
    if (gt) out[atomicAdd(&out_ctr, 1)] = i;
    const uint32_t bal = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) warp_cnt[wid] = __popc(bal);
    __syncthreads();
    uint32_t off = 0, tot = 0;
    for (int w = 0; w < kWarps; ++w) {
      const uint32_t c = warp_cnt[w];
      off += w < wid ? c : 0u;
      tot += c;
    }
    const uint32_t rank = sh_eq_base + off + __popc(bal & ((1u << lane) - 1u));
    if (eq && rank < rem) out[n_gt + rank] = i;
    __syncthreads();
    if (threadIdx.x == 0) sh_eq_base += tot;
    __syncthreads();
  }
}

// ------------------------------------------------------------------ two-stage select

// Exclusive prefix sum of v over the block; `total` receives the block sum.
template <int NT>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* wsum, uint32_t& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[wid] = x;
  __syncthreads();
  if (wid == 0) {
    uint32_t t = lane < NT / 32 ? wsum[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < NT / 32) wsum[lane] = t;
  }
  __syncthreads();
  const uint32_t base = wid ? wsum[wid - 1] : 0u;
  total = wsum[NT / 32 - 1];
  __syncthreads();
  return base + x - v;
}

// Shared-memory key arrays are padded by one word per 32 (key i at i + i/32), so
// that thread t reading element t*seg + j (a contiguous segment per thread, seg
// = 16) hits 32 distinct banks.
__device__ __forceinline__ int padded(int i) { return i + (i >> 5); }
__host__ __device__ constexpr int padded_size(int n) { return n + (n >> 5) + 1; }

// Histogram of digit (key >> sh) & (nb-1) over the keys matching prefix/mask.
// With `aggregate`, lanes with the same digit are combined before the
// shared-memory atomic (the leading digits of positive scores fall into a
// handful of buckets; later passes see only the keys under the chosen prefix).
template <int NT>
__device__ __forceinline__ void digit_hist(const uint32_t* keys, int n, uint32_t prefix, uint32_t mask, int sh,
                                           int nb, uint32_t* hist, bool aggregate) {
  const int lane = threadIdx.x & 31;
  for (int i0 = 0; i0 < n; i0 += NT) {
    const int i = i0 + threadIdx.x;
    const uint32_t key = i < n ? keys[padded(i)] : 0u;
    const bool in = i < n && (key & mask) == prefix;
    const uint32_t d = in ? (key >> sh) & (uint32_t)(nb - 1) : 0xFFFFFFFFu;
    if (aggregate) {
      const uint32_t peers = __match_any_sync(0xffffffffu, d);
      if (in && lane == __ffs(peers) - 1) atomicAdd(&hist[d], (uint32_t)__popc(peers));
    } else if (in) {
      atomicAdd(&hist[d], 1u);
    }
  }
}

// Top min(k, n) of keys[0..n) (shared memory, padded as above, larger key =
// better, equal keys: lower position first).  Calls emit(position, rank) for
// every selected position, ranks 0.. in increasing position order.  Whole block.
template <int NT, typename Emit>
__device__ void block_select(const uint32_t* keys, int n, int k, Emit emit) {
  __shared__ uint32_t hist[2048];
  __shared__ uint32_t wsum[NT / 32];
  __shared__ uint32_t sh_digit, sh_rem;
  const int kk = n < k ? n : k;
  if (kk == n) {
    for (int i = threadIdx.x; i < n; i += NT) emit(i, (uint32_t)i);
    return;
  }
  uint32_t prefix = 0, mask = 0, rem = (uint32_t)kk;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = shifts[pass], nb = 1 << widths[pass];
    for (int b = threadIdx.x; b < nb; b += NT) hist[b] = 0;
    __syncthreads();
    digit_hist<NT>(keys, n, prefix, mask, sh, nb, hist, pass == 0);
    __syncthreads();
    // the digit d with count(> d) < rem <= count(>= d): thread t owns buckets
    // [nb - (t+1)*bpt, nb - t*bpt), scanned from the top
    const int bpt = (nb + NT - 1) / NT, top = nb - threadIdx.x * bpt;
    uint32_t local = 0;
    for (int j = 0; j < bpt; ++j)
      if (top - 1 - j >= 0) local += hist[top - 1 - j];
    uint32_t tot;
    const uint32_t above = block_excl_scan<NT>(local, wsum, tot);
    if (above < rem && rem <= above + local) {
      uint32_t cum = above;
      for (int j = 0; j < bpt; ++j) {
        const uint32_t h = hist[top - 1 - j];
        if (cum + h >= rem) {
          sh_digit = (uint32_t)(top - 1 - j);
          sh_rem = rem - cum;
          break;
        }
        cum += h;
      }
    }
    __syncthreads();
    prefix |= sh_digit << sh;
    mask |= (uint32_t)(nb - 1) << sh;
    rem = sh_rem;
    __syncthreads();
  }
  // every key above T, and the first `rem` keys equal to T in position order.
  // Thread t owns the contiguous segment [t*seg, t*seg+seg): one scan ranks the
  // equal keys, one more places the selected ones.
  const uint32_t T = prefix;
  const int seg = (n + NT - 1) / NT;
  const int lo = threadIdx.x * seg, hi = min(n, lo + seg);
  uint32_t n_gt = 0, n_eq = 0;
  for (int i = lo; i < hi; ++i) {
    const uint32_t key = keys[padded(i)];
    n_gt += key > T;
    n_eq += key == T;
  }
  uint32_t tot;
  const uint32_t eq0 = block_excl_scan<NT>(n_eq, wsum, tot);
  const uint32_t take_eq = eq0 >= rem ? 0u : min(n_eq, rem - eq0);
  uint32_t rank = block_excl_scan<NT>(n_gt + take_eq, wsum, tot);
  uint32_t eq_seen = 0;
  for (int i = lo; i < hi; ++i) {
    const uint32_t key = keys[padded(i)];
    if (key > T || (key == T && eq_seen++ < take_eq)) emit(i, rank++);
  }
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
    block_select<kChunkThreads>(keys, len, a.k, [&](int pos, uint32_t rank) { out[rank] = pos; });
    return;
  }
  uint32_t* ok = cand_key + slot * a.k;
  int32_t* oi = cand_idx + slot * a.k;
  block_select<kChunkThreads>(keys, len, a.k, [&](int pos, uint32_t rank) {
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
  block_select<kMergeThreads>(keys, total, a.k, [&](int pos, uint32_t rank) { out[rank] = idx[pos]; });
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

}  // namespace csa
