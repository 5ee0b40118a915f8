// DSA top-k: the min(k, n) largest indexer scores of each row, equal scores
// going to the lower entry index ("vLLM解密：DeepSeek-V4本地部署為何如此困難"
// §二 item 3: k = 512 on c4a).
//
// Exact radix select on an order-preserving 32-bit key of the fp32 score:
// three histogram passes over 12 + 12 + 8 bits fix the k-th largest key T and
// how many entries equal to T are still needed; a last pass writes every
// entry above T (any order) and the lowest-indexed entries equal to T, ranked
// by a block-wide scan in index order.  One CTA of 1024 threads per row.

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

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, int32_t n_rows, cudaStream_t s) {
  if (n_rows == 0 || a.k == 0) return cudaSuccess;
  topk_kernel<<<n_rows, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace csa
