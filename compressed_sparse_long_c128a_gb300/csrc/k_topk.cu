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
#include "tc_ptx.cuh"

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

constexpr int kDealMergeThreads = 256;
constexpr int kMaxMergeCluster = 16;
constexpr int kMergeKeep = 4096;  // survivors a member keeps in shared memory after its first read
constexpr int kMergeKeyWords = (padded_size(kMergeKeep) + 3) & ~3;
constexpr size_t kMergeSmem = sizeof(uint32_t) * (kMergeKeyWords + kMergeKeep);

// Row r: its lists under the deal (one per CTA range of the row, see
// DealCandidates) merged into the row's top-k by one cluster of Cs CTAs.
// List c holds every key of its range at or above thr_c, and thr_c is at most
// the row's k-th largest key, so the keys at or above max_c thr_c
// ("survivors") are all in the lists and include the row's top-k.  Member m of the cluster takes a contiguous run of the row's lists
// (lists are in entry order) and streams its survivors from L2 in every pass:
// a count, three radix-digit histograms (11, 11, 10 bits) summed into rank 0's
// shared memory through the cluster (rank 0 picks each digit and hands it
// back), and a last pass that places every survivor above the k-th key and
// the first equal ones in entry order.
//
// The short way's selection (shared memory to `dst`).
__device__ __forceinline__ void merge_select(const uint32_t* keys, const int32_t* idx, int n, int k, SelectScratch& sc,
                                          int32_t* dst) {
  block_select<kDealMergeThreads>(keys, n, k, sc, [&](int pos, uint32_t rank) { dst[rank] = idx[pos]; });
  for (int i = min(n, k) + threadIdx.x; i < k; i += kDealMergeThreads) dst[i] = -1;
}

//
// A row whose lists hold at most kMergeKeep entries in all, merged by a
// single CTA, takes a shorter way: every list entry is loaded into shared
// memory once (lists in CTA order, each in entry order: the row's entry
// order) and block_select picks the top-k there.  That is exact without the
// survivor filter: each CTA's list holds its range's top-k, which holds every
// entry of the row's top-k that lies in the range.
__global__ void __launch_bounds__(kDealMergeThreads) topk_deal_merge_kernel(const TopkArgs a,
                                                                            const DealCandidates c, int n_rows) {
  constexpr int NT = kDealMergeThreads;
  __shared__ int32_t off[kDealMaxRows + 1];  // start of each of the row's lists in the flattened array
  __shared__ uint32_t hloc[2048];            // this member's histogram of a pass
  __shared__ uint32_t hsum[3][2048];         // rank 0: the cluster's histograms
  __shared__ uint32_t wsum[32];
  __shared__ uint32_t s_thr, s_total, s_digit[3], s_rem[3];
  __shared__ uint32_t s_gt[kMaxMergeCluster], s_eq[kMaxMergeCluster];  // rank 0: members' counts
  __shared__ int32_t s_all;
  // [padded_size(kMergeKeep)] this member's survivors in entry order, when they fit
  // (the short way: every list entry, padded as block_select reads them)
  extern __shared__ uint32_t kept_key[];
  int32_t* kept_idx = reinterpret_cast<int32_t*>(kept_key + kMergeKeyWords);  // [kMergeKeep]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int Cs = gridDim.y, me = (int)tc::cluster_rank();
  // No early launch of the next kernel: the attention behind this one keeps
  // its (large) CTAs waiting on the SMs, which would hold off the CTAs of this
  // launch; it starts as this launch's CTAs exit.
  for (int b = threadIdx.x; b < 3 * 2048; b += NT) (&hsum[0][0])[b] = 0;
  if (threadIdx.x == 0) s_total = 0;
  pdl_wait();  // the lists are complete only after the indexer launch
  tc::cluster_sync();  // rank 0's sums are zero before any member adds
  const int r = blockIdx.x;
  const int first = c.row_first[r], ctas = min(c.row_ctas[r], kDealMaxRows), seg0 = c.row_seg[r];
  // list j of the row lives in slot 2 (first + j), plus seg0 for j = 0
  auto slot = [&](int j) -> int64_t { return 2 * (int64_t)(first + j) + (j == 0 ? seg0 : 0); };
  const int K = a.k;
  int32_t* out = a.out + (int64_t)r * K;
  if (warp == 0) {  // lane l owns lists [8l, 8l+8): counts, thresholds, prefix
    int32_t cnt[8], mine = 0;
    uint32_t t = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int j = 8 * lane + i;
      cnt[i] = j < ctas ? c.cnt[slot(j)] : 0;
      t = j < ctas ? max(t, c.thr[slot(j)]) : t;
      mine += cnt[i];
    }
    for (int o = 16; o > 0; o >>= 1) t = max(t, __shfl_xor_sync(0xffffffffu, t, o));
    int32_t incl = mine;
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int32_t run = incl - mine;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int j = 8 * lane + i;
      if (j <= ctas) off[j] = run;
      run += cnt[i];
    }
    if (lane == 0) s_thr = t;
    if (lane == 31) s_all = incl;
  }
  __syncthreads();
  if (Cs == 1 && s_all <= kMergeKeep) {  // the short way (block-uniform)
    const int all = s_all;
    SelectScratch& sc = *reinterpret_cast<SelectScratch*>(&hsum[0][0]);
    for (int v0 = threadIdx.x; v0 < all; v0 += 8 * NT) {
      uint32_t kb[8];
      int32_t ib[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {  // eight independent loads in flight per thread
        const int v = v0 + u * NT;
        if (v < all) {
          int lo = 0, hi = ctas - 1;  // the list holding flattened entry v
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (off[mid] <= v) lo = mid;
            else hi = mid - 1;
          }
          const int64_t e = slot(lo) * c.cap + (v - off[lo]);
          kb[u] = c.key[e];
          ib[u] = c.idx[e];
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int v = v0 + u * NT;
        if (v < all) {
          kept_key[padded(v)] = kb[u];
          kept_idx[v] = ib[u];
        }
      }
    }
    __syncthreads();
    merge_select(kept_key, kept_idx, all, K, sc, out);
    return;
  }
  const uint32_t thr = s_thr;
  // this member's lists and its thread's contiguous slice of their entries
  const int per = (ctas + Cs - 1) / Cs, jb = min(ctas, me * per), je = min(ctas, jb + per);
  const int vb = off[jb], ve = off[je];
  const int seg = (ve - vb + NT - 1) / NT, v0 = min(ve, vb + (int)threadIdx.x * seg), v1 = min(ve, v0 + seg);
  int j0 = jb;
  while (j0 + 1 < je && off[j0 + 1] <= v0) ++j0;
  // visit(key, idx_pos) over this thread's survivors in entry order, eight loads in flight
  auto visit = [&](auto&& fn) {
    int j = j0;
    for (int v = v0; v < v1; v += 8) {
      int64_t e[8];
      uint32_t kb[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        e[u] = -1;
        if (v + u < v1) {
          while (j + 1 < je && off[j + 1] <= v + u) ++j;
          e[u] = slot(j) * c.cap + (v + u - off[j]);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) kb[u] = e[u] >= 0 ? c.key[e[u]] : 0u;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (e[u] >= 0 && kb[u] >= thr) fn(kb[u], e[u]);
    }
  };
  // survivors: counted, then (when this member's fit) copied to shared memory in
  // entry order so that the later passes read them there
  uint32_t n_mine = 0;
  visit([&](uint32_t, int64_t) { ++n_mine; });
  uint32_t n_member;
  uint32_t at = block_excl_scan<NT>(n_mine, wsum, n_member);
  const bool kept = n_member <= (uint32_t)kMergeKeep;
  if (kept) visit([&](uint32_t key, int64_t e) {
    kept_key[at] = key;
    kept_idx[at] = c.idx[e];
    ++at;
  });
  if (threadIdx.x == 0 && n_member) tc::cluster_red_add(tc::map_shared(&s_total, 0), n_member);
  tc::cluster_sync();
  // the survivors this thread visits in the later passes, in entry order
  const int ks = (int)((n_member + NT - 1) / NT), k0 = min((int)n_member, (int)threadIdx.x * ks),
            k1 = min((int)n_member, k0 + ks);
  auto each = [&](auto&& fn) {
    if (kept) {
      for (int q = k0; q < k1; ++q) fn(kept_key[q], (int64_t)-1 - q);
    } else {
      visit(fn);
    }
  };
  auto index_of = [&](int64_t e) { return e < 0 ? kept_idx[-1 - e] : c.idx[e]; };
  const uint32_t total = tc::cluster_ld(tc::map_shared(&s_total, 0));
  const uint32_t kk = total < (uint32_t)K ? total : (uint32_t)K;
  uint32_t prefix = 0, mask = 0, rem = kk;
  const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3 && kk > 0; ++pass) {
    const int sh = shifts[pass], nb = 1 << widths[pass];
    for (int b = threadIdx.x; b < nb; b += NT) hloc[b] = 0;
    __syncthreads();
    each([&](uint32_t key, int64_t) {
      if ((key & mask) == prefix) atomicAdd(&hloc[(key >> sh) & (uint32_t)(nb - 1)], 1u);
    });
    __syncthreads();
    for (int b = threadIdx.x; b < nb; b += NT)
      if (hloc[b]) tc::cluster_red_add(tc::map_shared(&hsum[pass][b], 0), hloc[b]);
    tc::cluster_sync();
    if (me == 0) {  // the digit d with count(> d) < rem <= count(>= d)
      const int bpt = (nb + NT - 1) / NT, top = nb - threadIdx.x * bpt;
      uint32_t local = 0;
      for (int q = 0; q < bpt; ++q)
        if (top - 1 - q >= 0) local += hsum[pass][top - 1 - q];
      uint32_t tot;
      const uint32_t above = block_excl_scan<NT>(local, wsum, tot);
      if (above < rem && rem <= above + local) {
        uint32_t cum = above;
        for (int q = 0; q < bpt && top - 1 - q >= 0; ++q) {
          const uint32_t h = hsum[pass][top - 1 - q];
          if (cum + h >= rem) {
            s_digit[pass] = (uint32_t)(top - 1 - q);
            s_rem[pass] = rem - cum;
            break;
          }
          cum += h;
        }
      }
    }
    tc::cluster_sync();
    prefix |= tc::cluster_ld(tc::map_shared(&s_digit[pass], 0)) << sh;
    mask |= (uint32_t)(nb - 1) << sh;
    rem = tc::cluster_ld(tc::map_shared(&s_rem[pass], 0));
  }
  // keys above T to slots [0, n_gt), the first `rem` keys equal to T to [n_gt, kk),
  // each group in entry order: member prefixes through rank 0, thread prefixes by scans
  const uint32_t T = prefix;
  uint32_t n_gt = 0, n_eq = 0;
  if (kk > 0) each([&](uint32_t key, int64_t) {
    n_gt += key > T;
    n_eq += key == T;
  });
  uint32_t m_gt, m_eq;
  uint32_t t_gt = block_excl_scan<NT>(n_gt, wsum, m_gt);
  uint32_t t_eq = block_excl_scan<NT>(n_eq, wsum, m_eq);
  if (threadIdx.x == 0) {
    tc::cluster_st(tc::map_shared(&s_gt[me], 0), m_gt);
    tc::cluster_st(tc::map_shared(&s_eq[me], 0), m_eq);
  }
  tc::cluster_sync();
  uint32_t gt_all = 0, gt_before = 0, eq_before = 0;
  for (int q = 0; q < Cs; ++q) {
    const uint32_t g = tc::cluster_ld(tc::map_shared(&s_gt[q], 0));
    const uint32_t e = tc::cluster_ld(tc::map_shared(&s_eq[q], 0));
    gt_all += g;
    gt_before += q < me ? g : 0u;
    eq_before += q < me ? e : 0u;
  }
  t_gt += gt_before;
  t_eq += eq_before;
  if (kk > 0) each([&](uint32_t key, int64_t e) {
    if (key > T) {
      out[t_gt++] = index_of(e);
    } else if (key == T) {
      if (t_eq < rem) out[gt_all + t_eq] = index_of(e);
      ++t_eq;
    }
  });
  if (me == 0)
    for (int i = (int)kk + threadIdx.x; i < K; i += NT) out[i] = -1;
  tc::cluster_sync();  // no member may leave while another still reads rank 0's shared memory
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
  const int r = blockIdx.x;
  int n = n_visible(a.pos[r], a.ratio, a.window);
  if (n > a.max_n) {
    if (threadIdx.x == 0 && blockIdx.y == 0) record_error(a.err, CSA_ERR_DEVICE_BOUNDS);
    n = a.max_n;
  }
  const bool final_out = n_chunks == 1;
  int32_t* out = a.out + (int64_t)r * a.k;
  // CTA (r, y) takes chunks y, y + gridDim.y, ... of row r: a row's chunks past
  // its visible entries cost no CTA of their own
  for (int c = blockIdx.y; c < n_chunks; c += gridDim.y) {
    const int lo = c * kChunk;
    const int len = max(0, min(kChunk, n - lo));
    if (final_out)
      for (int i = min(len, a.k) + threadIdx.x; i < a.k; i += kChunkThreads) out[i] = -1;
    const int64_t slot = (int64_t)r * n_chunks + c;
    if (len <= 0) {
      if (threadIdx.x == 0 && !final_out) cand_cnt[slot] = 0;
      continue;  // block-uniform
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
    } else {
      uint32_t* ok = cand_key + slot * a.k;
      int32_t* oi = cand_idx + slot * a.k;
      block_select<kChunkThreads>(keys, len, a.k, sc, [&](int pos, uint32_t rank) {
        ok[rank] = keys[padded(pos)];
        oi[rank] = lo + pos;
      });
      if (threadIdx.x == 0) cand_cnt[slot] = min(len, a.k);
    }
    __syncthreads();  // the keys are read by the emission before the next chunk overwrites them
  }
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

cudaError_t launch_topk(const TopkArgs& a, int32_t n_rows, void* cand, cudaStream_t s) {
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
    return launch_k(topk_chunk_kernel, dim3(n_rows, 1), dim3(kChunkThreads), kChunkSmem, s, 0, a,
                    (uint32_t*)nullptr, (int32_t*)nullptr, (int32_t*)nullptr, 1);
  if (!topk_two_stage(a.max_n, a.k) || cand == nullptr)
    return launch_k(topk_kernel, dim3(n_rows), dim3(kThreads), 0, s, 0, a);
  uint32_t* ck = reinterpret_cast<uint32_t*>(cand);
  int32_t* ci = reinterpret_cast<int32_t*>(ck + (size_t)n_rows * nc * a.k);
  int32_t* cc = ci + (size_t)n_rows * nc * a.k;
  // up to four CTAs a row, each looping over its chunks
  e = launch_k(topk_chunk_kernel, dim3(n_rows, nc < 4 ? nc : 4), dim3(kChunkThreads), kChunkSmem, s, 0, a, ck, ci,
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
  return launch_k(topk_merge_kernel, dim3(n_rows), dim3(kMergeThreads), smem, s, 0, a,
                  (const uint32_t*)ck,
                  (const int32_t*)ci, (const int32_t*)cc, nc);
}

cudaError_t launch_topk_deal_merge(const TopkArgs& a, int32_t n_rows, const DealCandidates& c, cudaStream_t s) {
  if (n_rows == 0 || a.k == 0) return cudaSuccess;
  static PerDevice attr;
  cudaError_t e = with_device_slot(attr, [](int, int64_t& done) {
    if (done) return cudaSuccess;
    cudaError_t r = cudaFuncSetAttribute(topk_deal_merge_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(topk_deal_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kMergeSmem);
    if (r == cudaSuccess) done = 1;
    return r;
  });
  if (e != cudaSuccess) return e;
  // members per row: a power of two <= 16 keeping at least about four of the
  // deal's lists per member (rows of a few lists merge in one CTA)
  int32_t cs = 1;
  while (cs < kMaxMergeCluster && 4 * cs * n_rows <= c.ctas) cs *= 2;
  return launch_k(topk_deal_merge_kernel, dim3(n_rows, cs), dim3(kDealMergeThreads), kMergeSmem, s, cs, a, c,
                  (int)n_rows);
}

}  // namespace csa
