// DSA top-k: the min(k, n) largest indexer scores of each row, equal scores
// going to the lower entry index ("vLLM解密：DeepSeek-V4本地部署為何如此困難"
// §二 item 3: k = 512 on c4a).
//
// Exact radix select on an order-preserving 32-bit key of the fp32 score:
// histogram passes over the key's bits fix the k-th largest key T and how
// many entries equal to T are still needed; a last pass in index order takes
// every entry above T and the lowest-indexed entries equal to T.
//
// Two stages when the candidates fit in shared memory: (1) every chunk of
// 8192 scores of a row selects its own top-k in shared memory and writes
// (key, index) candidates in index order; (2) one CTA per row selects the
// top-k of the row's candidates, which are in index order chunk after chunk,
// so ties still resolve to the lower entry index.  The global top-k is a
// subset of the union of the chunks' top-k sets because the order is total.
// Otherwise one CTA of 1024 threads per row scans the whole row.

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

// Top min(k, n) of keys[0..n) (shared memory, larger key = better, equal keys:
// lower position first).  Calls emit(position, rank) for every selected
// position, ranks 0.. in increasing position order.  Whole block.
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
    for (int i = threadIdx.x; i < n; i += NT) {
      const uint32_t key = keys[i];
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> sh) & (nb - 1)], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x, per = nb / 32, hi = nb - lane * per;
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
  uint32_t eq_base = 0, sel_base = 0;
  for (int c0 = 0; c0 < n; c0 += NT) {
    const int i = c0 + threadIdx.x;
    const uint32_t key = i < n ? keys[i] : 0u;
    const bool gt = i < n && key > T;
    const bool eq = i < n && key == T;
    uint32_t eq_tot, sel_tot;
    const uint32_t eq_rank = eq_base + block_excl_scan<NT>(eq ? 1u : 0u, wsum, eq_tot);
    const bool sel = gt || (eq && eq_rank < rem);
    const uint32_t rank = sel_base + block_excl_scan<NT>(sel ? 1u : 0u, wsum, sel_tot);
    if (sel) emit(i, rank);
    eq_base += eq_tot;
    sel_base += sel_tot;
  }
}

constexpr int kChunk = 8192;
constexpr int kChunkThreads = 512;
constexpr int kMergeThreads = 1024;

__global__ void __launch_bounds__(kChunkThreads) topk_chunk_kernel(const TopkArgs a, uint32_t* cand_key,
                                                                    int32_t* cand_idx, int32_t* cand_cnt,
                                                                    int n_chunks) {
  __shared__ uint32_t keys[kChunk];
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x, c = blockIdx.y;
  int n = n_visible(a.pos[r], a.ratio, a.window);
  if (n > a.max_n) {
    if (threadIdx.x == 0 && c == 0) record_error(a.err, CSA_ERR_DEVICE_BOUNDS);
    n = a.max_n;
  }
  const int lo = c * kChunk;
  const int len = min(kChunk, n - lo);
  const int64_t slot = (int64_t)r * n_chunks + c;
  if (len <= 0) {
    if (threadIdx.x == 0) cand_cnt[slot] = 0;
    return;
  }
  const float* s = a.scores + (int64_t)r * a.max_n + lo;
  for (int i = threadIdx.x; i < len; i += kChunkThreads) keys[i] = order_key(s[i]);
  __syncthreads();
  uint32_t* ok = cand_key + slot * a.k;
  int32_t* oi = cand_idx + slot * a.k;
  block_select<kChunkThreads>(keys, len, a.k, [&](int pos, uint32_t rank) {
    ok[rank] = keys[pos];
    oi[rank] = lo + pos;
  });
  if (threadIdx.x == 0) cand_cnt[slot] = min(len, a.k);
}

__global__ void __launch_bounds__(kMergeThreads) topk_merge_kernel(const TopkArgs a, const uint32_t* cand_key,
                                                                    const int32_t* cand_idx,
                                                                    const int32_t* cand_cnt, int n_chunks) {
  extern __shared__ uint32_t msm[];
  uint32_t* keys = msm;                                            // [n_chunks * k]
  int32_t* idx = reinterpret_cast<int32_t*>(msm + n_chunks * a.k);  // [n_chunks * k]
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
      keys[off[c] + j] = cand_key[slot * a.k + j];
      idx[off[c] + j] = cand_idx[slot * a.k + j];
    }
  }
  __syncthreads();
  int32_t* out = a.out + (int64_t)r * a.k;
  block_select<kMergeThreads>(keys, total, a.k, [&](int pos, uint32_t rank) { out[rank] = idx[pos]; });
  const int kk = total < a.k ? total : a.k;
  for (int i = kk + threadIdx.x; i < a.k; i += kMergeThreads) out[i] = -1;
}

}  // namespace

int32_t topk_chunks(int32_t max_n) { return (max_n + kChunk - 1) / kChunk; }

bool topk_two_stage(int32_t max_n, int32_t k) {
  const int32_t c = topk_chunks(max_n);
  return c >= 1 && c <= 64 && (size_t)c * k * 8 <= 160 * 1024;
}

size_t topk_candidate_bytes(int32_t n_rows, int32_t max_n, int32_t k) {
  if (!topk_two_stage(max_n, k)) return 0;
  const size_t c = topk_chunks(max_n);
  return (size_t)n_rows * c * ((size_t)k * 8 + 4);
}

cudaError_t launch_topk(const TopkArgs& a, int32_t n_rows, void* cand, cudaStream_t s) {
  if (n_rows == 0 || a.k == 0) return cudaSuccess;
  if (!topk_two_stage(a.max_n, a.k) || cand == nullptr) {
    return launch_k(topk_kernel, dim3(n_rows), dim3(kThreads), 0, s, 0, a);
  }
  const int32_t nc = topk_chunks(a.max_n);
  uint32_t* ck = reinterpret_cast<uint32_t*>(cand);
  int32_t* ci = reinterpret_cast<int32_t*>(ck + (size_t)n_rows * nc * a.k);
  int32_t* cc = ci + (size_t)n_rows * nc * a.k;
  cudaError_t e = launch_k(topk_chunk_kernel, dim3(n_rows, nc), dim3(kChunkThreads), 0, s, 0, a, ck, ci, cc, nc);
  if (e != cudaSuccess) return e;
  const size_t smem = (size_t)nc * a.k * 8;
  static size_t smem_set = 0;
  if (smem > 48 * 1024 && smem > smem_set) {
    e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    smem_set = smem;
  }
  return launch_k(topk_merge_kernel, dim3(n_rows), dim3(kMergeThreads), smem, s, 0, a, (const uint32_t*)ck,
                  (const int32_t*)ci, (const int32_t*)cc, nc);
}

}  // namespace csa
