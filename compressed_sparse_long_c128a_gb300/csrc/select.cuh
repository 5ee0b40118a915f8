// Block-wide exact top-k selection and the balanced deal of indexer work,
// shared by the indexer (selection fused into its epilogue) and the top-k
// kernels.
//
// Selection is a radix select on an order-preserving 32-bit key of the fp32
// score: histogram passes over the key's bits (11, 11, 10) fix the k-th
// largest key T and how many entries equal to T are still needed; a last pass
// in position order takes every key above T and the lowest-positioned keys
// equal to T, so equal scores go to the lower entry index ("vLLM解密：
// DeepSeek-V4本地部署為何如此困難" §二 item 3: the k largest indexer scores).
#pragma once

#include "csa_kernels.h"

namespace csa {

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Shared-memory key arrays are padded by one word per 32 (key i at i + i/32), so
// that thread t reading element t*seg + j (a contiguous segment per thread)
// hits distinct banks.
__device__ __forceinline__ int padded(int i) { return i + (i >> 5); }
__host__ __device__ constexpr int padded_size(int n) { return n + (n >> 5) + 1; }

// Scratch of one block_select (shared memory, any 4-byte aligned region).
struct SelectScratch {
  uint32_t hist[2048];
  uint32_t wsum[32];
  uint32_t digit, rem;
};

// Exclusive prefix sum of v over the block; `total` receives the block sum.
template <int NT>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* wsum, uint32_t& total) {
  static_assert(NT % 32 == 0 && NT <= 1024, "block of whole warps");
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
// every selected position, ranks 0.. in increasing position order.  Whole
// block of NT threads; `sc` is shared scratch.
template <int NT, typename Emit>
__device__ void block_select(const uint32_t* keys, int n, int k, SelectScratch& sc, Emit emit) {
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
    for (int b = threadIdx.x; b < nb; b += NT) sc.hist[b] = 0;
    __syncthreads();
    digit_hist<NT>(keys, n, prefix, mask, sh, nb, sc.hist, pass == 0);
    __syncthreads();
    // the digit d with count(> d) < rem <= count(>= d): thread t owns buckets
    // [nb - (t+1)*bpt, nb - t*bpt), scanned from the top
    const int bpt = (nb + NT - 1) / NT, top = nb - threadIdx.x * bpt;
    uint32_t local = 0;
    for (int j = 0; j < bpt; ++j)
      if (top - 1 - j >= 0) local += sc.hist[top - 1 - j];
    uint32_t tot;
    const uint32_t above = block_excl_scan<NT>(local, sc.wsum, tot);
    if (above < rem && rem <= above + local) {
      uint32_t cum = above;
      for (int j = 0; j < bpt && top - 1 - j >= 0; ++j) {
        const uint32_t h = sc.hist[top - 1 - j];
        if (cum + h >= rem) {
          sc.digit = (uint32_t)(top - 1 - j);
          sc.rem = rem - cum;
          break;
        }
        cum += h;
      }
    }
    __syncthreads();
    prefix |= sc.digit << sh;
    mask |= (uint32_t)(nb - 1) << sh;
    rem = sc.rem;
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
  const uint32_t eq0 = block_excl_scan<NT>(n_eq, sc.wsum, tot);
  const uint32_t take_eq = eq0 >= rem ? 0u : min(n_eq, rem - eq0);
  uint32_t rank = block_excl_scan<NT>(n_gt + take_eq, sc.wsum, tot);
  uint32_t eq_seen = 0;
  for (int i = lo; i < hi; ++i) {
    const uint32_t key = keys[padded(i)];
    if (key > T || (key == T && eq_seen++ < take_eq)) emit(i, rank++);
  }
}

// ------------------------------------------------------------------ balanced deal

// The indexer's work for a batch of rows dealt to G CTAs in proportion to each
// row's key tiles: row r with t_r tiles (128 entries each) gets
// k_r = ceil(t_r / B) CTAs, B the smallest tile budget with sum_r k_r <= G,
// and its tiles are split into k_r contiguous ranges of equal size (+-1).
// Rows get CTAs in row order.  Every CTA of the indexer and of the merge
// computes the same deal from the rows' positions, so nothing is exchanged.
constexpr int kDealTile = 128;
constexpr int kDealMaxRows = 256;  // rows per deal (8 per lane)

struct DealShared {
  int32_t first[kDealMaxRows];  // first CTA of each row
  int32_t ctas[kDealMaxRows];   // CTAs of each row (0 for a row with no tiles)
  int32_t tiles[kDealMaxRows];
};

// ceil(t / m) for 0 <= t < 2^22 and 1 <= m, from a float reciprocal rm ~ 1/m:
// the estimate is within one of the quotient and is corrected exactly.
__device__ __forceinline__ int32_t ceil_div_small(int32_t t, int32_t m, float rm) {
  int32_t q = __float2int_rn((float)t * rm);
  if (q * m < t) ++q;
  if (q > 0 && (q - 1) * m >= t) --q;
  return q;
}

// Tiles of row r; `ratio` divides 256, so it is a power of two and the
// division is a shift.
__device__ __forceinline__ int32_t deal_row_tiles(const int32_t* pos, int r, int32_t ratio, int32_t window,
                                                  int32_t max_n) {
  const int32_t p = pos[r];
  int32_t n = p < window ? 0 : ((p - window) >> (__ffs(ratio) - 1)) + 1;
  n = n < max_n ? n : max_n;
  return (n + kDealTile - 1) / kDealTile;
}

// One warp (all 32 lanes): fills ds for n_rows <= kDealMaxRows rows dealt to
// G >= n_rows CTAs.  Lane l owns rows [8l, 8l+8).
__device__ __forceinline__ void deal_compute(const int32_t* pos, int n_rows, int32_t ratio, int32_t window,
                                             int32_t max_n, int G, DealShared& ds) {
  const int lane = threadIdx.x & 31;
  int32_t t[8];
  int32_t tmax = 0, tsum = 0;  // at most 256 rows of 2^22 / 128 tiles
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 8 * lane + i;
    t[i] = r < n_rows ? deal_row_tiles(pos, r, ratio, window, max_n) : 0;
    tmax = max(tmax, t[i]);
    tsum += t[i];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
    tsum += __shfl_xor_sync(0xffffffffu, tsum, o);
  }
  // smallest feasible budget in [ceil(T/G), tmax]; tmax is feasible as n_rows <= G
  int32_t lo = (int32_t)((tsum + G - 1) / G), hi = tmax;
  if (lo < 1) lo = 1;
  if (hi < lo) hi = lo;
  while (lo < hi) {
    const int32_t mid = (lo + hi) >> 1;
    const float rm = 1.0f / (float)mid;
    int32_t cnt = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) cnt += ceil_div_small(t[i], mid, rm);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (cnt <= G) hi = mid;
    else lo = mid + 1;
  }
  // CTAs per row and their prefix in row order
  int32_t k[8], mine = 0;
  const float rlo = 1.0f / (float)lo;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    k[i] = ceil_div_small(t[i], lo, rlo);
    mine += k[i];
  }
  int32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int32_t run = incl - mine;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 8 * lane + i;
    if (r < n_rows) {
      ds.first[r] = run;
      ds.ctas[r] = k[i];
      ds.tiles[r] = t[i];
    }
    run += k[i];
  }
}

// The row and tile range of CTA c under the deal (row -1: c has no work).
struct DealSlot {
  int32_t row, t0, nt;
};
__device__ __forceinline__ DealSlot deal_slot(const DealShared& ds, int n_rows, int c) {
  DealSlot s{-1, 0, 0};
  // the last row whose first CTA is <= c (rows with no CTA share their successor's first)
  int lo = 0, hi = n_rows - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ds.first[mid] <= c) lo = mid;
    else hi = mid - 1;
  }
  const int r = lo;
  const int32_t j = c - ds.first[r], k = ds.ctas[r], t = ds.tiles[r];
  if (j < 0 || j >= k) return s;
  s.row = r;
  s.t0 = (int32_t)(((long long)j * t) / k);
  s.nt = (int32_t)(((long long)(j + 1) * t) / k) - s.t0;
  return s;
}

}  // namespace csa
