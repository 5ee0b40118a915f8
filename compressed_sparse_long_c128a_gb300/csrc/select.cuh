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
// hist holds 4096 bucket counts, bucket b at hist_slot(b): thread t < 256
// owns buckets [16t, 16t+16), stored 256 words apart, so that its reads hit
// distinct banks.
struct SelectScratch {
  uint32_t hist[4096];
  uint32_t wsum[32];
  uint32_t digit, rem;
};
__device__ __forceinline__ int hist_slot(uint32_t b) { return (int)((b & 15u) * 256u + (b >> 4)); }

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

// The bucket of the 4096-bucket histogram sc.hist that holds the rem-th
// largest key (buckets counted from the top; 1 <= rem <= the total) into
// sc.digit, and how many keys of that bucket are still needed into sc.rem.
// Threads 0-255 own 16 buckets each; one suffix scan over them finds the
// owner, which walks its own buckets.  Whole block (NT >= 256).
template <int NT>
__device__ __forceinline__ void find_digit(uint32_t rem, SelectScratch& sc) {
  static_assert(NT >= 256, "256 threads own the buckets");
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  uint32_t c[16], s = 0, x = 0;
  if (t < 256) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      c[j] = sc.hist[j * 256 + t];
      s += c[j];
    }
    x = s;  // becomes the sum over this warp's lanes at or above this one
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
      if (lane + o < 32) x += y;
    }
    if (lane == 0) sc.wsum[warp] = x;
  }
  __syncthreads();
  if (t < 256) {
    uint32_t above = x - s;  // keys in the buckets of the threads above this one
    for (int w = warp + 1; w < 8; ++w) above += sc.wsum[w];
    if (above < rem && rem <= above + s) {  // exactly one thread
      uint32_t cum = above;
#pragma unroll
      for (int j = 15; j >= 0; --j) {
        if (cum + c[j] >= rem) {
          sc.digit = (uint32_t)(16 * t + j);
          sc.rem = rem - cum;
          break;
        }
        cum += c[j];
      }
    }
  }
  __syncthreads();
}

// Top min(k, n) of keys[0..n) (shared memory, padded as above, larger key =
// better, equal keys: lower position first).  Calls emit(position, rank) for
// every selected position, ranks 0.. in increasing position order.  Whole
// block of NT >= 256 threads; `sc` is shared scratch.
//
// The k-th largest key T is found by histograms over the keys' own range
// [min, max]: each pass splits the current range into at most 4096 buckets
// (a power-of-two width each) and keeps the bucket holding the rank, so a
// range of b bits takes ceil(b / 12) passes (two when the keys span less than
// 2^24 key values, as the scores of one row usually do).
template <int NT, typename Emit>
__device__ void block_select(const uint32_t* keys, int n, int k, SelectScratch& sc, Emit emit) {
  const int kk = n < k ? n : k;
  if (kk == n) {
    for (int i = threadIdx.x; i < n; i += NT) emit(i, (uint32_t)i);
    return;
  }
  constexpr int kU = 4;  // keys loaded per thread before any is used
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
  for (int i0 = 0; i0 < n; i0 += kU * NT) {
    uint32_t kv[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = i0 + u * NT + threadIdx.x;
      kv[u] = i < n ? keys[padded(i)] : 0u;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (i0 + u * NT + (int)threadIdx.x < n) {
        mn = min(mn, kv[u]);
        mx = max(mx, kv[u]);
      }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    sc.hist[warp] = mn;
    sc.hist[32 + warp] = mx;
  }
  __syncthreads();
  mn = 0xFFFFFFFFu;
  mx = 0u;
  for (int w = 0; w < NT / 32; ++w) {
    mn = min(mn, sc.hist[w]);
    mx = max(mx, sc.hist[32 + w]);
  }
  __syncthreads();
  uint32_t base = mn, rem = (uint32_t)kk;
  uint64_t width = (uint64_t)(mx - mn) + 1;  // the keys still in play lie in [base, base + width)
  while (width > 1) {
    const uint32_t span = (uint32_t)(width - 1);
    const int sh = span < 4096u ? 0 : (32 - __clz(span)) - 12;
    for (int b = threadIdx.x; b < 4096; b += NT) sc.hist[b] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += kU * NT) {
      uint32_t kv[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + u * NT + threadIdx.x;
        kv[u] = i < n ? keys[padded(i)] : 0u;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + u * NT + threadIdx.x;
        const bool in = i < n && kv[u] >= base && (uint64_t)(kv[u] - base) < width;
        const uint32_t d = in ? (kv[u] - base) >> sh : 0xFFFFFFFFu;
        // a warp whose keys share one bucket adds once (keys crowd a few
        // buckets when a few outliers stretch the range)
        const uint32_t d0 = __shfl_sync(0xffffffffu, d, 0);
        if (__all_sync(0xffffffffu, d == d0)) {
          if (lane == 0 && d0 != 0xFFFFFFFFu) atomicAdd(&sc.hist[hist_slot(d0)], 32u);
        } else if (d != 0xFFFFFFFFu) {
          atomicAdd(&sc.hist[hist_slot(d)], 1u);
        }
      }
    }
    __syncthreads();
    find_digit<NT>(rem, sc);
    const uint32_t d = sc.digit;
    rem = sc.rem;
    const uint64_t lo = (uint64_t)d << sh;
    base += (uint32_t)lo;
    width = min(width - lo, (uint64_t)1 << sh);
    __syncthreads();
  }
  // every key above T, and the first `rem` keys equal to T in position order.
  // Thread t owns the contiguous segment [t*seg, t*seg+seg); one scan of the
  // packed counts (above T, equal to T) ranks everything.
  const uint32_t T = base;
  const int seg = (n + NT - 1) / NT;
  const int lo = threadIdx.x * seg, hi = min(n, lo + seg);
  uint32_t n_gt = 0, n_eq = 0;
  for (int i = lo; i < hi; ++i) {
    const uint32_t key = keys[padded(i)];
    n_gt += key > T;
    n_eq += key == T;
  }
  uint32_t tot, gt0, eq0;
  if (n < 65536) {
    const uint32_t packed = block_excl_scan<NT>((n_gt << 16) | n_eq, sc.wsum, tot);
    gt0 = packed >> 16;
    eq0 = packed & 0xFFFFu;
  } else {
    gt0 = block_excl_scan<NT>(n_gt, sc.wsum, tot);
    eq0 = block_excl_scan<NT>(n_eq, sc.wsum, tot);
  }
  // the equal keys before this segment that are taken: min(eq0, rem)
  const uint32_t take_eq = eq0 >= rem ? 0u : min(n_eq, rem - eq0);
  uint32_t rank = gt0 + min(eq0, rem);
  uint32_t eq_seen = 0;
  for (int i = lo; i < hi; ++i) {
    const uint32_t key = keys[padded(i)];
    if (key > T || (key == T && eq_seen++ < take_eq)) emit(i, rank++);
  }
}

// ------------------------------------------------------------------ balanced deal

// The indexer's work for a batch of rows dealt to G CTAs.  Every CTA of the
// indexer computes the same deal from the rows' positions; its CTA 0 hands
// each row's list slots to the merge.  Two forms:
//
//  * even deal: the rows' tiles (128 entries each) are laid end to end and
//    CTA c takes tiles [floor(c T / G), floor((c+1) T / G)) of the T in all,
//    so every CTA streams the same amount.  Used when every non-empty row has
//    at least ceil(T / G) tiles (a CTA then meets at most two rows: the tail
//    of one, the head of the next) and that many tiles fit the CTA.  A CTA
//    keeps one list per row it meets, in list slot 2c (its first row) and
//    2c + 1 (its second).
//  * per-row deal, otherwise: row r with t_r tiles gets k_r = ceil(t_r / B)
//    CTAs, B the smallest budget with sum_r k_r <= G, its tiles split into k_r
//    contiguous ranges of equal size (+-1), one list each in slot 2c.
//
// Either way the lists of row r are, in entry order, slot 2 first_r + seg_r
// and then slot 2c for c = first_r + 1 .. first_r + ctas_r - 1.
constexpr int kDealTile = 128;
constexpr int kDealMaxRows = 256;  // rows per deal (8 per lane)

struct DealShared {
  int32_t first[kDealMaxRows];  // the CTA holding the row's first list
  int32_t ctas[kDealMaxRows];   // CTAs (lists) of each row (0 for a row with no tiles)
  int32_t tiles[kDealMaxRows];
  int32_t seg[kDealMaxRows];    // even deal: 1 if the row is the second one of its first CTA
  int32_t start[kDealMaxRows];  // even deal: the row's first tile in the concatenation
  int32_t even, total;          // the even deal is in use; T
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

// Under the even deal: the first tile of CTA c, and the CTA holding tile g.
// 32-bit unsigned arithmetic is exact: c, G <= kDealMaxCtas + 1, and a deal
// is launched only when T <= G x (the tiles a CTA holds) < 2^16, so every
// product is below 2^32.
__device__ __forceinline__ int32_t even_first_tile(int c, int32_t T, int G) {
  return (int32_t)(((uint32_t)c * (uint32_t)T) / (uint32_t)G);
}
__device__ __forceinline__ int32_t even_cta_of(int32_t g, int32_t T, int G) {
  return (int32_t)((((uint32_t)g + 1u) * (uint32_t)G - 1u) / (uint32_t)T);
}

// One warp (all 32 lanes): fills ds for n_rows <= kDealMaxRows rows dealt to
// G >= n_rows CTAs; `cap` is the most tiles a CTA can take under the even
// deal.  Lane l owns rows [8l, 8l+8).
__device__ __forceinline__ void deal_compute(const int32_t* pos, int n_rows, int32_t ratio, int32_t window,
                                             int32_t max_n, int G, int32_t cap, DealShared& ds) {
  const int lane = threadIdx.x & 31;
  int32_t t[8];
  int32_t tmax = 0, tsum = 0, tmin = 0x7FFFFFFF;  // at most 256 rows of 2^22 / 128 tiles
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 8 * lane + i;
    t[i] = r < n_rows ? deal_row_tiles(pos, r, ratio, window, max_n) : 0;
    tmax = max(tmax, t[i]);
    tsum += t[i];
    if (t[i] > 0) tmin = min(tmin, t[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
    tsum += __shfl_xor_sync(0xffffffffu, tsum, o);
    tmin = min(tmin, __shfl_xor_sync(0xffffffffu, tmin, o));
  }
  const int32_t L = (tsum + G - 1) / G;  // the most tiles of a CTA under the even deal
  if (tsum > 0 && tmin >= L && L <= cap) {
    int32_t mine = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) mine += t[i];
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
        ds.start[r] = run;
        ds.tiles[r] = t[i];
        if (t[i] > 0) {
          const int32_t c1 = even_cta_of(run, tsum, G), c2 = even_cta_of(run + t[i] - 1, tsum, G);
          ds.first[r] = c1;
          ds.ctas[r] = c2 - c1 + 1;
          ds.seg[r] = even_first_tile(c1, tsum, G) == run ? 0 : 1;
        } else {
          ds.first[r] = 0;
          ds.ctas[r] = 0;
          ds.seg[r] = 0;
        }
      }
      run += t[i];
    }
    if (lane == 0) {
      ds.even = 1;
      ds.total = tsum;
    }
    return;
  }
  // smallest feasible budget in [ceil(T/G), tmax]; tmax is feasible as n_rows <= G
  int32_t lo = L, hi = tmax;
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
      ds.seg[r] = 0;
      ds.start[r] = 0;
    }
    run += k[i];
  }
  if (lane == 0) {
    ds.even = 0;
    ds.total = tsum;
  }
}

// The rows and tile ranges of CTA c under the deal: up to two segments
// (row -1: none), each a contiguous tile range [t0, t0 + nt) of one row.
struct DealSlot {
  int32_t row[2], t0[2], nt[2];
};
__device__ __forceinline__ DealSlot deal_slot(const DealShared& ds, int n_rows, int c, int G) {
  DealSlot s{{-1, -1}, {0, 0}, {0, 0}};
  if (ds.even) {
    const int32_t T = ds.total;
    const int32_t g0 = even_first_tile(c, T, G), g1 = even_first_tile(c + 1, T, G);
    if (g1 <= g0) return s;
    // the row holding tile g0: the last row whose first tile is <= g0 (an empty
    // row shares its first tile with the next row, which is the one kept)
    int lo = 0, hi = n_rows - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ds.start[mid] <= g0) lo = mid;
      else hi = mid - 1;
    }
    const int ra = lo;
    const int32_t end_a = ds.start[ra] + ds.tiles[ra];
    s.row[0] = ra;
    s.t0[0] = g0 - ds.start[ra];
    s.nt[0] = min(end_a, g1) - g0;
    if (g1 > end_a) {
      int rb = ra + 1;
      while (rb < n_rows && ds.tiles[rb] == 0) ++rb;
      if (rb < n_rows) {
        s.row[1] = rb;
        s.t0[1] = 0;
        s.nt[1] = g1 - ds.start[rb];
      }
    }
    return s;
  }
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
  s.row[0] = r;
  s.t0[0] = (int32_t)(((uint32_t)j * (uint32_t)t) / (uint32_t)k);
  s.nt[0] = (int32_t)(((uint32_t)(j + 1) * (uint32_t)t) / (uint32_t)k) - s.t0[0];
  return s;
}

}  // namespace csa
