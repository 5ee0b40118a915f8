// Shared-K=V sparse attention on the sm_103a tensor cores (tcgen05 + TMEM).
//
// Pages: "vLLM DeepSeek V4 Support", "DeepSeek V4 Attention Architecture"
// (one shared key/value vector per entry, inverse RoPE on the output, DSA
// top-k plus a 128-token raw window under one softmax);
// "vLLM解密：DeepSeek-V4本地部署為何如此困難" §3.2 second fusion (inverse
// RoPE fused with the fp8 quantisation of the output).
//
// Shape: D = 512, H = 64 query heads sharing every key (MQA).  One CTA takes
// one query row and a contiguous slice of its key list (selected entries, then
// window rows), in tiles of 64 keys:
//
//   S   [64 heads x 64 keys]    = Q [64 x 512] . K_tile^T [512 x 64]        (M = 64)
//   O^T [512 dims x 64 heads]  += K_tile^T [512 x 64] . P^T [64 x 64]        (4 chunks of 128 dims)
//
// Shared memory holds Q (64 KB, pre-rotated, pre-scaled by scale*log2 e), a
// ring of two 64 KB key tiles and two P buffers.  A key tile is gathered once,
// 128B-swizzled with keys as rows: read K-major it is the B operand of S, read
// MN-major the A operand of O^T (values = keys).  While one tile is in use the
// next is being gathered; the tensor pipe takes S chunks as their rows land
// and O of a tile as soon as its P is written, so the softmax of tile t
// overlaps S_{t+1}.  TMEM: S double-buffered in
// columns 0..127 (M = 64 layout: head h in lane 32*(h/16) + h%16), O^T chunk c
// in 128+64c.
//
// Warp roles (12 warps): warps 0-3 are the softmax (lanes l and l+16 share head 16w+l: the
// row max and the denominator stay in registers) and the epilogue (thread t
// owns TMEM lane t: dim t of an O^T chunk); they also look the tile's row
// addresses up three tiles ahead.  Warps 4-10 gather the rows from the paged
// caches (cp.async for bf16, load + convert for e4m3, whose per-row scale is
// folded into the logits and into P).  Warp 11 allocates TMEM and one lane
// issues the MMAs.  The running per-head max is only raised when a logit
// exceeds it by more than 2^8; raising it rescales O^T in TMEM.
//
// A row's key list may be split over S = 1, 2, 4 or 8 CTAs launched as one
// cluster.  Each CTA stages its unnormalised O (bf16) in its idle ring; after
// a cluster barrier the copy engine hands each peer m the block of the heads
// m merges, with their max and denominator, into m's idle Q area; CTA m then
// merges heads [m*64/S, (m+1)*64/S), normalises, rotates back and stores.

#include "csa_kernels.h"
#include "tc_ptx.cuh"

namespace csa {
namespace {

using namespace tc;

constexpr int kD = 512, kH = 64, kTile = 64, kChunks = 4;
constexpr int kSoftmax = 128, kProducers = 224;
constexpr int kThreads = kSoftmax + kProducers + 32;
constexpr int kMmaWarp = kThreads / 32 - 1;
constexpr int kMergeThreads = 256;  // thread t of the merge takes dims 2t and 2t+1
constexpr uint32_t kQBytes = kH * kD * 2;             // 64 KB
constexpr uint32_t kChunkBytes = kTile * 128 * 2;     // 16 KB: 64 keys x 128 dims
constexpr uint32_t kAtomBytes = kTile * 128;          // 8 KB: 64 keys x 64 dims
constexpr uint32_t kTileBytes = kChunks * kChunkBytes;  // 64 KB
constexpr uint32_t kPBytes = kH * kTile * 2;          // 8 KB: 64 heads x 64 keys
constexpr uint32_t kOffQ = 0, kOffK = kQBytes, kOffP = kOffK + 2 * kTileBytes;
constexpr uint32_t kOffMisc = kOffP + 2 * kPBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 128;  // S double-buffered in 0..127, O^T chunk c at 128 + 64c
constexpr float kRescaleMargin = 8.0f;       // log2 units
constexpr int kRowBufs = 4;                  // tiles whose row addresses are known ahead

struct Misc {
  uint64_t kfull[2][kChunks];  // tile slot, chunk: loaded
  uint64_t kfree[2][kChunks];  // tile slot, chunk: consumed by O^T
  uint64_t o_done[2];          // O^T of the slot's tile complete: P buffer free
  uint64_t s_full[2], p_full[2], rows_ready[kRowBufs], q_raw, q_full, mma_done, recv;
  uint32_t tmem_base;
  int32_t abort;
  alignas(16) float M[kH];  // per-head max (log2 domain) of the slice, for the merge
  alignas(16) float L[kH];  // softmax denominators of the slice
  float red[4][kH];         // merge weights
  float amax[kMergeThreads / 32][32];  // per-warp head maxima of the merged output
  float alpha[kH];          // rescale factor of the last max raise
  alignas(16) float rM[8][32], rL[8][32];  // merged heads' max and denominator of each slice (split rows)
  float rc[kMaxRopePairs], rs[kMaxRopePairs];  // cos / sin of each rotary pair at the row's position
  // by tile mod kRowBufs (released through rows_ready): row addresses for the
  // producers, and each key's validity and e4m3 scale for the softmax
  const uint8_t* rowptr[kRowBufs][kTile];
  alignas(16) float kscale[kRowBufs][kTile];
  alignas(16) int8_t kvalid[kRowBufs][kTile];
};
constexpr uint32_t kSmemBytes = kOffMisc + sizeof(Misc) + 1024;

struct Geo {
  int seq;
  int64_t p, w_lo;
  int32_t n_vis, n_sel, j0, j1, n_tiles;
  __device__ __forceinline__ int keys(int t) const { return min(kTile, j1 - j0 - t * kTile); }
};

__device__ __forceinline__ Geo row_geometry(const AttnArgs& a, int r, int split, int S) {
  Geo g;
  g.seq = a.seq_id[r];
  g.p = a.pos[r];
  g.n_vis = n_visible((int32_t)g.p, a.ratio, a.window);
  g.n_sel = a.topk ? a.k : g.n_vis;
  g.w_lo = g.p - a.swa_len + 1 > 0 ? g.p - a.swa_len + 1 : 0;
  const int32_t n_keys = g.n_sel + (int32_t)(g.p - g.w_lo + 1);
  const int32_t per = (n_keys + S - 1) / S;
  g.j0 = min(n_keys, split * per);
  g.j1 = min(n_keys, g.j0 + per);
  g.n_tiles = (g.j1 - g.j0 + kTile - 1) / kTile;
  return g;
}

// Bounded wait; after the first timeout in the CTA every later wait returns at
// once, so all roles run to the end and TMEM is released.
__device__ __forceinline__ bool wait_or_abort(Misc& ms, uint64_t* bar, uint32_t parity, int32_t* err) {
  if (*reinterpret_cast<volatile int32_t*>(&ms.abort)) return false;
  if (mbar_wait(bar, parity)) return true;
  *reinterpret_cast<volatile int32_t*>(&ms.abort) = 1;
  record_error(err, CSA_ERR_TIMEOUT);
  return false;
}

// ------------------------------------------------------------------ producers

// Row address (and e4m3 scale) of key slot `slot` of tile t, or nullptr if masked.
__device__ __forceinline__ const uint8_t* key_row(const AttnArgs& a, const Geo& g, int t, int slot, bool fp8,
                                                  float& sc) {
  const int32_t j = g.j0 + t * kTile + slot;
  sc = 1.f;
  if (j >= g.j1) return nullptr;
  const csa_paged* c = nullptr;
  int64_t prow = -1;
  if (j < g.n_sel) {
    const int32_t idx = a.topk ? a.topk[(int64_t)blockIdx.x * a.k + j] : j;
    if (idx < 0) return nullptr;
    if (idx >= g.n_vis) {
      record_error(a.err, CSA_ERR_DEVICE_BOUNDS);
      return nullptr;
    }
    c = &a.comp;
    prow = phys_row(a.comp_bt, a.comp, g.seq, idx, a.err);
  } else {
    c = &a.swa;
    prow = phys_row(a.swa_bt, a.swa, g.seq, g.w_lo + (j - g.n_sel), a.err);
  }
  if (prow < 0) return nullptr;
  if (fp8) sc = reinterpret_cast<const float*>(c->scales)[prow];
  return reinterpret_cast<const uint8_t*>(c->data) + prow * row_bytes(*c);
}

// Producers: tile t goes to ring slot t & 1, one 16 KB chunk (128 dims) at a
// time, each chunk as soon as O^T of tile t-2 has released it.  bf16 rows are copied with
// cp.async, each thread's copies arriving on the chunk's barrier as they land
// (the MMA issuer fences them into the async proxy); e4m3 rows are converted
// through registers (E4M3: codes to bf16 exactly, the row scale folded into the
// logits and P; E4M3R: codes times the row scale rounded to bf16, the bf16
// tail copied).  Keys past the slice are not loaded; the rest of the last
// 16-key step of O^T is filled with zeros.
__device__ void producer_role(const AttnArgs& a, const Geo& g, uint8_t* smem, Misc& ms, int pt) {
  const bool fp8 = a.comp.dtype == CSA_E4M3 || a.comp.dtype == CSA_E4M3R;
  const bool tail = a.comp.dtype == CSA_E4M3R;
  const int Dq = tail ? kD - a.comp.tail_bf16 : kD;  // dims [Dq, kD) are bf16 in the row
  const int n = g.n_tiles;
  const uint64_t pol = policy_evict_first();  // every key row is read once per call
  // bf16: thread pt copies 16-byte piece (pt & 15) of keys 6j + (pt >> 4)
  constexpr int kGroups = kProducers / 16, kPerThr = (kTile + kGroups - 1) / kGroups;
  const int kg = pt >> 4, piece = pt & 15;
  for (int t = 0; t < n; ++t) {
    const int slot = t & 1, buf = t % kRowBufs;
    wait_or_abort(ms, &ms.rows_ready[buf], (t / kRowBufs) & 1, a.err);
    const uint32_t prev = ((t - 2) >> 1) & 1;  // use of the slot by tile t-2
    const int lim = min(kTile, (g.keys(t) + 15) & ~15);
    const uint32_t tbase = smem_u32(smem + kOffK) + slot * kTileBytes;
    if (!fp8) {
      const uint8_t* rps[kPerThr];
#pragma unroll
      for (int j = 0; j < kPerThr; ++j) {
        const int k = kGroups * j + kg;
        rps[j] = k < lim ? ms.rowptr[buf][k] : nullptr;
      }
      const uint32_t poff = (piece >> 3) * kAtomBytes;
      for (int c = 0; c < kChunks; ++c) {
        if (t >= 2) wait_or_abort(ms, &ms.kfree[slot][c], prev, a.err);
        const uint32_t cbase = tbase + c * kChunkBytes + poff;
#pragma unroll
        for (int j = 0; j < kPerThr; ++j) {
          const int k = kGroups * j + kg;
          if (k < lim) {
            const uint32_t dst = cbase + (k >> 3) * 1024 + (k & 7) * 128 + (((piece & 7) ^ (k & 7)) << 4);
            cp_async16_hint(dst, rps[j] ? rps[j] + c * 256 + piece * 16 : a.comp.data, rps[j] ? 16u : 0u, pol);
          }
        }
        cp_async_arrive_noinc(&ms.kfull[slot][c]);
      }
    } else {
      // 8 consecutive threads per key row, 16 dims each: 16 code bytes -> 16 bf16
      // (a piece of the bf16 tail: 32 bytes copied).  The loads of all four
      // chunks of the tile are issued first (they wait for no slot), so the
      // tile costs one memory latency, not four; the tail (at most 128 dims)
      // lies in the last chunk.
      constexpr int kIters = (kTile * 8 + kProducers - 1) / kProducers;
      uint4 raw[kChunks][kIters], tl[kIters];
#pragma unroll
      for (int c = 0; c < kChunks; ++c)
#pragma unroll
        for (int it = 0; it < kIters; ++it) {
          const int x = pt + it * kProducers;
          raw[c][it] = make_uint4(0, 0, 0, 0);
          if (c == kChunks - 1) tl[it] = make_uint4(0, 0, 0, 0);
          if (x < lim * 8) {
            const uint8_t* rp = ms.rowptr[buf][x >> 3];
            const int d0 = c * 128 + (x & 7) * 16;
            if (rp && d0 < Dq) {
              raw[c][it] = ldg16_hint(rp + d0, pol);
            } else if (rp && c == kChunks - 1) {
              const uint8_t* tp = rp + Dq + 2 * (d0 - Dq);
              raw[c][it] = ldg16_hint(tp, pol);
              tl[it] = ldg16_hint(tp + 16, pol);
            }
          }
        }
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        if (t >= 2) wait_or_abort(ms, &ms.kfree[slot][c], prev, a.err);
#pragma unroll
        for (int it = 0; it < kIters; ++it) {
          const int x = pt + it * kProducers;
          if (x >= lim * 8) break;
          const uint32_t key = x >> 3, q8 = x & 7;
          const int d0 = c * 128 + q8 * 16;
          uint32_t outw[8];
          if (d0 >= Dq) {
            outw[0] = raw[c][it].x; outw[1] = raw[c][it].y; outw[2] = raw[c][it].z; outw[3] = raw[c][it].w;
            outw[4] = tl[it].x; outw[5] = tl[it].y; outw[6] = tl[it].z; outw[7] = tl[it].w;
          } else {
            const uint32_t w[4] = {raw[c][it].x, raw[c][it].y, raw[c][it].z, raw[c][it].w};
            const float rs = tail ? ms.kscale[buf][key] : 1.f;  // E4M3R: the row scale, applied here
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float2 v = e4m3x2_to_f32x2(w[e >> 1] >> ((e & 1) * 16));
              outw[e] = f32x2_to_bf16x2(v.x * rs, v.y * rs);
            }
          }
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint32_t pc = q8 * 2 + half;  // 16-byte piece of the 256-byte bf16 chunk
            uint8_t* dst = smem + kOffK + slot * kTileBytes + c * kChunkBytes + (pc >> 3) * kAtomBytes +
                           (key >> 3) * 1024 + (key & 7) * 128 + (((pc & 7) ^ (key & 7)) << 4);
            *reinterpret_cast<uint4*>(dst) =
                make_uint4(outw[half * 4], outw[half * 4 + 1], outw[half * 4 + 2], outw[half * 4 + 3]);
          }
        }
        fence_proxy_async();
        mbar_arrive(&ms.kfull[slot][c]);
      }
    }
  }
  cp_async_wait<0>();
}

// ------------------------------------------------------------------ MMA issuer

// One lane issues every MMA.  Work becomes ready in two streams: the S chunks
// of tile t as its rows land (each also needs the S buffer free: O of tile
// t-2 issued, i.e. its softmax done), and O of tile t once its P is written.
// O is issued as soon as it is ready, ahead of the S chunks still waiting for
// rows, because it releases the ring slot the next tile loads into.
__device__ void mma_role(const AttnArgs& a, const Geo& g, uint8_t* smem, Misc& ms, uint32_t tmem) {
  constexpr uint32_t idesc_s = idesc_bf16(64, kTile, 0, 0);   // A = Q (K-major), B = key tile (K-major)
  constexpr uint32_t idesc_o = idesc_bf16(128, kH, 1, 0);     // A = key tile^T (MN-major), B = P (K-major)
  // every operand below is one of these descriptors plus a constant
  const uint64_t d_q = sdesc_sw128(smem_u32(smem + kOffQ), 16, 1024);
  const uint64_t d_ks = sdesc_sw128(smem_u32(smem + kOffK), 16, 1024);
  const uint64_t d_ko = sdesc_sw128(smem_u32(smem + kOffK), kAtomBytes, 1024);
  const uint64_t d_p = sdesc_sw128(smem_u32(smem + kOffP), 16, 1024);
  const int n = g.n_tiles;
  wait_or_abort(ms, &ms.q_full, 0, a.err);
  int st_t = 0, st_c = 0, o_t = 0;  // next S chunk (tile, chunk); next O tile
  int idle = 0;
  while (o_t < n) {
    if (*reinterpret_cast<volatile int32_t*>(&ms.abort)) break;
    if (o_t < st_t && mbar_test(&ms.p_full[o_t & 1], (o_t >> 1) & 1)) {
      const int t = o_t, slot = t & 1;
      tc_fence_after();
      const int ksteps = (g.keys(t) + 15) >> 4;
      const uint32_t toff = (slot * kTileBytes) >> 4, poff = (slot * kPBytes) >> 4;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks)  // 16 keys per step: two 8-key groups of 1 KB
          if (ks < ksteps)
            mma_bf16(tmem + kColO + 64 * c, d_ko + toff + ((c * kChunkBytes + ks * 2048) >> 4),
                     d_p + poff + ((ks * 32) >> 4), idesc_o, (t > 0 || ks > 0) ? 1u : 0u);
        mma_commit(&ms.kfree[slot][c]);  // the chunk can take tile t+2's rows
      }
      mma_commit(&ms.o_done[slot]);
      ++o_t;
      idle = 0;
      continue;
    }
    if (st_t < n && st_t <= o_t + 1 && mbar_test(&ms.kfull[st_t & 1][st_c], (st_t >> 1) & 1)) {
      const int t = st_t, slot = t & 1, c = st_c;
      fence_proxy_async();  // the chunk was written through the generic proxy
      tc_fence_after();
      const uint32_t d_s = tmem + kColS + 64 * slot;
      const uint32_t koff = (slot * kTileBytes + c * kChunkBytes) >> 4;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t k0 = c * 128 + ks * 16;  // first dim of this K step
        mma_bf16(d_s, d_q + (((k0 >> 6) * (kH * 128) + (k0 & 63) * 2) >> 4),
                 d_ks + koff + (((ks >> 2) * kAtomBytes + (ks & 3) * 32) >> 4), idesc_s, (c | ks) != 0);
      }
      if (++st_c == kChunks) {
        mma_commit(&ms.s_full[slot]);
        st_c = 0;
        ++st_t;
      }
      idle = 0;
      continue;
    }
    if (++idle > 4 * kSpinLimit) {
      *reinterpret_cast<volatile int32_t*>(&ms.abort) = 1;
      record_error(a.err, CSA_ERR_TIMEOUT);
      break;
    }
  }
  // nothing may still write TMEM when it is released, even after a timeout
  mma_commit(&ms.mma_done);
  mbar_wait(&ms.mma_done, 0);
}

// ------------------------------------------------------------------ softmax + epilogue

// Rotation of the pair (d, d+1) at the row's position (rotary dims only), the
// logit scale, and bf16 rounding of the pair.
__device__ __forceinline__ uint32_t rot_pack(float q0, float q1, int d, float qs, int R, const Misc& ms) {
  if (d >= kD - R) {
    const float cs = ms.rc[(d - (kD - R)) / 2], sn = ms.rs[(d - (kD - R)) / 2];
    const float t0 = q0 * cs - q1 * sn;
    q1 = q0 * sn + q1 * cs;
    q0 = t0;
  }
  return f32x2_to_bf16x2(q0 * qs, q1 * qs);
}

// Q operand: the row's 64 heads rotated at p, scaled by scale * log2(e),
// rounded to bf16, 128B-swizzled K-major (rows = heads).  bf16 rows arrive
// raw as the CTA's first requests (eight TMA boxes of 64 dims x 64 heads, or
// cp.async when the rows cannot be described by a tensor map), ahead of the
// key lookups, and are then transformed in place; fp32 rows go through
// registers.  The softmax threads then release the MMA issuer through q_full.
__device__ __forceinline__ void fill_q_issue(const AttnArgs& a, uint8_t* smem, Misc& ms, int st) {
  if (a.q_dtype != CSA_BF16) return;
  if (a.q_tma) {
    // eight 64-dim x 64-head boxes land already swizzled
    if (st == 0) {
      mbar_arrive_expect_tx(&ms.q_raw, kQBytes);
      for (int at = 0; at < kD / 64; ++at)
        tma_load_2d(smem + kOffQ + at * (kH * 128), &a.q_map, 64 * at, kH * blockIdx.x, &ms.q_raw);
    }
    return;
  }
  constexpr int kPieces = kH * (kD / 8);  // 16-byte pieces of bf16 (8 dims each)
  const uint16_t* src = reinterpret_cast<const uint16_t*>(a.q) + (int64_t)blockIdx.x * a.heads * kD;
  const uint32_t qbase = smem_u32(smem + kOffQ);
  for (int x = st; x < kPieces; x += kSoftmax) {
    const int h = x >> 6, d0 = (x & 63) * 8;
    cp_async16(qbase + sw128_offset(h, d0, kH), src + h * kD + d0, 16u);
  }
  cp_async_commit();
}

__device__ void fill_q_finish(const AttnArgs& a, uint8_t* smem, Misc& ms, int st) {
  const float qs = a.scale * 1.4426950408889634f;
  const int R = a.rope.rope_dim;
  constexpr int kPieces = kH * (kD / 8);
  if (a.q_dtype == CSA_BF16) {
    if (a.q_tma) {
      if (!mbar_wait(&ms.q_raw, 0)) record_error(a.err, CSA_ERR_TIMEOUT);
    } else {
      cp_async_wait<0>();
    }
    for (int x = st; x < kPieces; x += kSoftmax) {
      const int h = x >> 6, d0 = (x & 63) * 8;
      uint4* p = reinterpret_cast<uint4*>(smem + kOffQ + sw128_offset(h, d0, kH));
      const uint4 v = *p;
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        o[e] = rot_pack(bf16_to_f32((uint16_t)(w[e] & 0xFFFF)), bf16_to_f32((uint16_t)(w[e] >> 16)), d0 + 2 * e, qs,
                        R, ms);
      *p = make_uint4(o[0], o[1], o[2], o[3]);
    }
  } else {
    const int64_t rb = (int64_t)blockIdx.x * a.heads * kD;
    constexpr int kBatch = 8;  // loads in flight per thread
    for (int x0 = st; x0 < kPieces; x0 += kSoftmax * kBatch) {
      float q[kBatch][8];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int x = x0 + u * kSoftmax;
        const int h = x >> 6, d0 = (x & 63) * 8;
        const float4* p4 = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.q) + rb + h * kD + d0);
        const float4 v0 = __ldg(p4), v1 = __ldg(p4 + 1);
        q[u][0] = v0.x; q[u][1] = v0.y; q[u][2] = v0.z; q[u][3] = v0.w;
        q[u][4] = v1.x; q[u][5] = v1.y; q[u][6] = v1.z; q[u][7] = v1.w;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int x = x0 + u * kSoftmax;
        const int h = x >> 6, d0 = (x & 63) * 8;
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] = rot_pack(q[u][2 * e], q[u][2 * e + 1], d0 + 2 * e, qs, R, ms);
        *reinterpret_cast<uint4*>(smem + kOffQ + sw128_offset(h, d0, kH)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  fence_proxy_async();
  mbar_arrive(&ms.q_full);
}

// Softmax threads st < 64 look up key st of tile u: row address for the
// producers, validity and e4m3 scale for the softmax; all 128 release the
// buffer through rows_ready.  (An L2 prefetch of the rows here measured
// slower: each prefetch instruction holds the SM's TMA unit about as long as a
// 1 KB row takes to stream.)
__device__ __forceinline__ void lookup_keys(const AttnArgs& a, const Geo& g, Misc& ms, int u, int st) {
  const int b = u % kRowBufs;
  if (st < kTile) {
    float sc;
    const uint8_t* rp = key_row(a, g, u, st, a.comp.dtype == CSA_E4M3 || a.comp.dtype == CSA_E4M3R, sc);
    ms.rowptr[b][st] = rp;
    ms.kvalid[b][st] = rp != nullptr;
    ms.kscale[b][st] = sc;
  }
  mbar_arrive(&ms.rows_ready[b]);
}

// The 64 head columns of one O^T chunk for this thread's TMEM lane (zeros for
// an empty slice): four loads in flight, one wait.
__device__ __forceinline__ void load_o_chunk(uint32_t taddr, bool any, float* o) {
  if (any) {
#pragma unroll
    for (int i = 0; i < 4; ++i) tmem_ld16(taddr + 16 * i, o + 16 * i);
    tmem_wait_ld();
  } else {
#pragma unroll
    for (int h = 0; h < kH; ++h) o[h] = 0.f;
  }
}

__device__ void softmax_role(const AttnArgs& a, const Geo& g, uint8_t* smem, Misc& ms, uint32_t tmem, int st) {
  fill_q_issue(a, smem, ms, st);
  if (g.n_tiles > 0) lookup_keys(a, g, ms, 0, st);
  fill_q_finish(a, smem, ms, st);
  for (int u = 1; u < min(g.n_tiles, kRowBufs - 1); ++u) lookup_keys(a, g, ms, u, st);
  const int w = st >> 5, l = st & 31;
  // lanes l and l+16 of warp w share head 16w + l (lanes 0-15 hold its TMEM row):
  // lane l takes keys [0, 32) of each tile, lane l+16 keys [32, 64)
  const int hf = l >> 4, h = 16 * w + (l & 15);
  const bool fp8 = a.comp.dtype == CSA_E4M3;  // per-key scales folded into the logits and P
  const uint32_t lane_addr = tmem + ((uint32_t)(w * 32) << 16);
  float m_run = -INFINITY, l_run = 0.f;  // the head's running max; this half's denominator

  for (int t = 0; t < g.n_tiles; ++t) {
    const int slot = t & 1, b = t % kRowBufs;
    const uint32_t use = (t >> 1) & 1;
    wait_or_abort(ms, &ms.s_full[slot], use, a.err);
    tc_fence_after();
    float x[kTile / 2];
    {
      float xt[kTile];
#pragma unroll
      for (int i = 0; i < 4; ++i) tmem_ld16(lane_addr + kColS + 64 * slot + 16 * i, xt + 16 * i);
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < kTile / 2; ++k) {
        const float hi = __shfl_sync(0xffffffffu, xt[kTile / 2 + k], l & 15);
        x[k] = hf ? hi : xt[k];
      }
    }
    wait_or_abort(ms, &ms.rows_ready[b], (t / kRowBufs) & 1, a.err);
    const int k0 = hf * (kTile / 2);
    float mt = -INFINITY;
#pragma unroll
    for (int k4 = 0; k4 < kTile / 8; ++k4) {
      const uint32_t vb = *reinterpret_cast<const uint32_t*>(&ms.kvalid[b][k0 + 4 * k4]);
      float s4[4] = {1.f, 1.f, 1.f, 1.f};
      if (fp8) {
        const float4 sc = *reinterpret_cast<const float4*>(&ms.kscale[b][k0 + 4 * k4]);
        s4[0] = sc.x; s4[1] = sc.y; s4[2] = sc.z; s4[3] = sc.w;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int k = 4 * k4 + e;
        x[k] = ((vb >> (8 * e)) & 0xFF) ? x[k] * s4[e] : -INFINITY;
        mt = fmaxf(mt, x[k]);
      }
    }
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));  // the head's tile max
    if (named_bar_or(1, kSoftmax, mt > m_run + kRescaleMargin)) {
      // raise every head's max to its current maximum; rescale O^T and the denominators
      const float mn = fmaxf(m_run, mt);
      const float al = m_run == -INFINITY ? 0.f : exp2f(m_run - mn);
      if (hf == 0) ms.alpha[h] = al;
      l_run *= al;
      m_run = mn;
      named_bar(1, kSoftmax);
      if (t > 0) {
        // O^T holds exactly the tiles before t once O_{t-1} is complete
        wait_or_abort(ms, &ms.o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, a.err);
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float o[16];
            tmem_ld16(lane_addr + kColO + 64 * c + 16 * i, o);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] *= ms.alpha[16 * i + j];
            tmem_st16(lane_addr + kColO + 64 * c + 16 * i, o);
          }
        }
        tmem_wait_st();
      }
    }
    // probabilities of this head for this half of the tile's keys: 64 bytes of
    // the head's P row, 8 keys per 16-byte piece; P carries each key's dequant scale
    uint32_t pw[kTile / 4];
    float ls[4] = {0.f, 0.f, 0.f, 0.f};
    if (m_run == -INFINITY) {
#pragma unroll
      for (int k = 0; k < kTile / 4; ++k) pw[k] = 0u;
    } else {
#pragma unroll
      for (int k = 0; k < kTile / 2; k += 2) {
        float p0 = fast_exp2(x[k] - m_run), p1 = fast_exp2(x[k + 1] - m_run);  // exp2(-inf) = 0
        ls[(k >> 1) & 3] += p0 + p1;
        if (fp8) {
          p0 *= ms.kscale[b][k0 + k];
          p1 *= ms.kscale[b][k0 + k + 1];
        }
        pw[k / 2] = f32x2_to_bf16x2(p0, p1);
      }
    }
    l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
    // the P buffer is free once O_{t-2} has consumed it
    if (t >= 2) wait_or_abort(ms, &ms.o_done[slot], ((t - 2) >> 1) & 1, a.err);
    uint8_t* prow = smem + kOffP + slot * kPBytes + (h >> 3) * 1024 + (h & 7) * 128;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<uint4*>(prow + (((4 * hf + c) ^ (h & 7)) << 4)) =
          make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
    fence_proxy_async();
    tc_fence_before();
    mbar_arrive(&ms.p_full[slot]);
    // tile t-1 is done with its address buffer: look ahead
    if (t + kRowBufs - 1 < g.n_tiles) lookup_keys(a, g, ms, t + kRowBufs - 1, st);
  }
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 16);  // both halves of the head's keys

  // ---- epilogue
  if (g.n_tiles > 0) wait_or_abort(ms, &ms.o_done[(g.n_tiles - 1) & 1], ((g.n_tiles - 1) >> 1) & 1, a.err);
  tc_fence_after();
  if (hf == 0) {
    ms.M[h] = m_run;
    ms.L[h] = l_run;  // sum over the slice's keys of 2^(x - M[h])
  }
  named_bar(1, kSoftmax);
  const int S = gridDim.y;
  const uint32_t my_lane = lane_addr;
  if (S == 1) {
    // stage the row's unnormalised O^T as [64 heads][512 dims] fp32 in the idle key ring
    float* stage = reinterpret_cast<float*>(smem + kOffK);
    for (int c = 0; c < kChunks; ++c) {
      float o[kH];
      load_o_chunk(my_lane + kColO + 64 * c, g.n_tiles > 0, o);
#pragma unroll
      for (int hh = 0; hh < kH; ++hh) stage[hh * kD + 128 * c + st] = o[hh];
    }
    return;
  }
  // split row: stage the slice's unnormalised O in bf16 in the idle ring, grouped
  // by the CTA that merges each head: [merger][512 dims][heads of the merger]
  const int per = kH / S, lper = __ffs(per) - 1;  // per is a power of two
  uint8_t* stage = smem + kOffK;
  for (int c = 0; c < kChunks; ++c) {
    float o[kH];
    load_o_chunk(my_lane + kColO + 64 * c, g.n_tiles > 0, o);
    const int d = 128 * c + st;
#pragma unroll
    for (int q = 0; q < kH / 8; ++q) {
      const int m = (8 * q) >> lper, hh = (8 * q) & (per - 1);
      uint32_t wv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) wv[e] = f32x2_to_bf16x2(o[8 * q + 2 * e], o[8 * q + 2 * e + 1]);
      *reinterpret_cast<uint4*>(stage + (((size_t)m * kD + d) * per + hh) * 2) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
  }
  fence_proxy_async();  // the copy engine reads the staging
}

// Inverse rotation at p and store of head h of row r; lane holds dims [16 lane, 16 lane + 16).
__device__ void store_head16(const AttnArgs& a, const Misc& ms, int r, int h, float* v, int lane) {
  const int R = a.rope.rope_dim;
#pragma unroll
  for (int e = 0; e < 16; e += 2) {
    const int d = 16 * lane + e;
    if (d >= kD - R) {
      const float cs = ms.rc[(d - (kD - R)) / 2], sn = ms.rs[(d - (kD - R)) / 2];
      const float x0 = v[e], x1 = v[e + 1];
      v[e] = x0 * cs + x1 * sn;
      v[e + 1] = -x0 * sn + x1 * cs;
    }
  }
  const int64_t ob = ((int64_t)r * a.heads + h) * kD + 16 * lane;
  if (a.out_dtype == CSA_E4M3) {
    float am = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) am = fmaxf(am, fabsf(v[e]));
    am = warp_max(am);
    const float inv = am > 0.f ? 448.0f / am : 0.0f;
    uint32_t wv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      wv[q] = (uint32_t)f32x2_to_e4m3x2(v[4 * q] * inv, v[4 * q + 1] * inv) |
              ((uint32_t)f32x2_to_e4m3x2(v[4 * q + 2] * inv, v[4 * q + 3] * inv) << 16);
    *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(a.out) + ob) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    if (lane == 0) a.out_scales[(int64_t)r * a.heads + h] = am / 448.0f;
  } else if (a.out_dtype == CSA_BF16) {
    uint32_t wv[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) wv[q] = f32x2_to_bf16x2(v[2 * q], v[2 * q + 1]);
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.out) + ob);
    dst[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    dst[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
  } else {
    float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + ob);
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  }
}

// Unsplit row: all 8 warps normalise the staged O (8 heads a warp) and store.
__device__ void finish_local(const AttnArgs& a, uint8_t* smem, const Misc& ms) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* stage = reinterpret_cast<const float*>(smem + kOffK);
  for (int h = warp; h < kH; h += kThreads / 32) {
    const float4* src = reinterpret_cast<const float4*>(stage + h * kD + 16 * lane);
    float v[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 x = src[q];
      v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
    }
    const float inv = ms.L[h] > 0.f ? 1.0f / ms.L[h] : 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] *= inv;
    store_head16(a, ms, blockIdx.x, h, v, lane);
  }
}

// Split row, after the cluster barrier: every CTA hands each peer m the staged
// block of m's heads, with their max and denominator, through the copy engine
// (into m's idle Q^T area and rM/rL); CTA m then merges heads
// [m*64/S, (m+1)*64/S) over the S slices, thread t taking dims 2t and 2t+1,
// rotates back, quantises and stores.
template <int S>
__device__ void merge_split(const AttnArgs& a, uint8_t* smem, Misc& ms) {
  constexpr int kPer = kH / S;
  constexpr uint32_t kBlk = kD * kPer * 2;  // bf16 block of one merger
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int me = blockIdx.y;
  const size_t row = blockIdx.x;
  const uint8_t* stage = smem + kOffK;
  if (t == 0) {
#pragma unroll 1
    for (int m = 0; m < S; ++m) {
      if (m == me) continue;
      const uint32_t bar = map_shared(&ms.recv, m);
      bulk_copy_to_peer(map_shared(smem + kOffQ + me * kBlk, m), stage + m * kBlk, kBlk, bar);
      bulk_copy_to_peer(map_shared(&ms.rM[me][0], m), &ms.M[m * kPer], kPer * 4, bar);
      bulk_copy_to_peer(map_shared(&ms.rL[me][0], m), &ms.L[m * kPer], kPer * 4, bar);
    }
    bulk_commit();
  }
  if (t < kPer) {
    ms.rM[me][t] = ms.M[me * kPer + t];
    ms.rL[me][t] = ms.L[me * kPer + t];
  }
  if (!mbar_wait(&ms.recv, 0)) record_error(a.err, CSA_ERR_TIMEOUT);
  named_bar(3, kMergeThreads);
  if (t < kPer) {  // weights 2^(M_s - max) / sum_s 2^(M_s - max) L_s into ms.red[2][s * kPer + t]
    float mg = -INFINITY;
#pragma unroll
    for (int sl = 0; sl < S; ++sl) mg = fmaxf(mg, ms.rM[sl][t]);
    float lg = 0.f, f[S];
#pragma unroll
    for (int sl = 0; sl < S; ++sl) {
      const float mv = ms.rM[sl][t];
      f[sl] = mv == -INFINITY ? 0.f : exp2f(mv - mg);
      lg += f[sl] * ms.rL[sl][t];
    }
    const float inv = lg > 0.f ? 1.0f / lg : 0.f;
#pragma unroll
    for (int sl = 0; sl < S; ++sl) ms.red[2][sl * kPer + t] = f[sl] * inv;
  }
  named_bar(3, kMergeThreads);
  float v[2][kPer];
#pragma unroll
  for (int hh = 0; hh < kPer; ++hh) v[0][hh] = v[1][hh] = 0.f;
#pragma unroll
  for (int sl = 0; sl < S; ++sl) {
    const uint8_t* blk = sl == me ? stage + me * kBlk : smem + kOffQ + sl * kBlk;
    // dims 2t and 2t+1: 2 * kPer consecutive bf16
    const uint4* src = reinterpret_cast<const uint4*>(blk + (size_t)2 * t * kPer * 2);
#pragma unroll
    for (int q = 0; q < kPer / 4; ++q) {
      const uint4 u = src[q];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int k = 8 * q + e, dd = k / kPer, hh = k % kPer;
        const float x = bf16_to_f32((uint16_t)(w[e >> 1] >> ((e & 1) * 16)));
        v[dd][hh] = fmaf(ms.red[2][sl * kPer + hh], x, v[dd][hh]);
      }
    }
  }
  // inverse rotation of the pair (2t, 2t+1)
  const int R = a.rope.rope_dim, d = 2 * t;
  if (d >= kD - R) {
    const float cs = ms.rc[(d - (kD - R)) / 2], sn = ms.rs[(d - (kD - R)) / 2];
#pragma unroll
    for (int hh = 0; hh < kPer; ++hh) {
      const float x0 = v[0][hh], x1 = v[1][hh];
      v[0][hh] = x0 * cs + x1 * sn;
      v[1][hh] = -x0 * sn + x1 * cs;
    }
  }
  const int h0 = me * kPer;
  const int64_t ob = (int64_t)row * a.heads * kD + d;
  if (a.out_dtype == CSA_E4M3) {
    // per-head amax over the 512 dims, from the warps' maxima
#pragma unroll
    for (int hh = 0; hh < kPer; ++hh) {
      const float am = warp_max(fmaxf(fabsf(v[0][hh]), fabsf(v[1][hh])));
      if (lane == 0) ms.amax[warp][hh] = am;
    }
    named_bar(3, kMergeThreads);
#pragma unroll
    for (int hh = 0; hh < kPer; ++hh) {
      float am = 0.f;
#pragma unroll
      for (int w = 0; w < kMergeThreads / 32; ++w) am = fmaxf(am, ms.amax[w][hh]);
      const float inv = am > 0.f ? 448.0f / am : 0.0f;
      *reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(a.out) + ob + (int64_t)(h0 + hh) * kD) =
          f32x2_to_e4m3x2(v[0][hh] * inv, v[1][hh] * inv);
      if (t == 0) a.out_scales[(int64_t)row * a.heads + h0 + hh] = am / 448.0f;
    }
  } else if (a.out_dtype == CSA_BF16) {
#pragma unroll
    for (int hh = 0; hh < kPer; ++hh)
      *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(a.out) + ob + (int64_t)(h0 + hh) * kD) =
          f32x2_to_bf16x2(v[0][hh], v[1][hh]);
  } else {
#pragma unroll
    for (int hh = 0; hh < kPer; ++hh)
      *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.out) + ob + (int64_t)(h0 + hh) * kD) =
          make_float2(v[0][hh], v[1][hh]);
  }
  if (t == 0) bulk_wait_read();  // the staging stays valid until the engine has read it
}

__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc& ms = *reinterpret_cast<Misc*>(smem + kOffMisc);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int r = blockIdx.x;
  pdl_trigger();

  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      for (int c = 0; c < kChunks; ++c) {
        mbar_init(&ms.kfull[b][c], kProducers);
        mbar_init(&ms.kfree[b][c], 1);
      }
      mbar_init(&ms.o_done[b], 1);
      mbar_init(&ms.s_full[b], 1);
      mbar_init(&ms.p_full[b], kSoftmax);
    }
    for (int b = 0; b < kRowBufs; ++b) mbar_init(&ms.rows_ready[b], kSoftmax);
    mbar_init(&ms.q_raw, 1);
    mbar_init(&ms.q_full, kSoftmax);
    mbar_init(&ms.mma_done, 1);
    mbar_init(&ms.recv, 1);
    mbar_init_fence();
    ms.abort = 0;
  }
  if (warp == kMmaWarp) tmem_alloc(&ms.tmem_base, kTmemCols);
  pdl_wait();  // before any access to memory: the previous kernel on the stream may still be running
  const Geo g = row_geometry(a, r, blockIdx.y, gridDim.y);
  if (tid < kH) ms.M[tid] = -INFINITY;
  if (tid < a.rope.rope_dim / 2) rope_cs(a.rope, tid, g.p, ms.rc[tid], ms.rs[tid]);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;

  if (warp < 4) {
    softmax_role(a, g, smem, ms, tmem, tid);
  } else if (warp < kMmaWarp) {
    producer_role(a, g, smem, ms, tid - kSoftmax);
  } else if ((tid & 31) == 0) {
    mma_role(a, g, smem, ms, tmem);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (gridDim.y == 1) {
    finish_local(a, smem, ms);
    return;
  }
  // every slice is staged and every CTA's tensor pipe is idle (its Q^T area is
  // free) before anyone copies; each receive barrier expects its S-1 blocks
  if (tid == 0) {
    const uint32_t per = kH / gridDim.y;
    mbar_arrive_expect_tx(&ms.recv, (gridDim.y - 1) * (kD * per * 2 + 2 * per * 4));
  }
  cluster_sync();
  if (tid >= kMergeThreads) return;
  switch (gridDim.y) {
    case 2: merge_split<2>(a, smem, ms); break;
    case 4: merge_split<4>(a, smem, ms); break;
    default: merge_split<8>(a, smem, ms); break;
  }
}

}  // namespace

bool attn_tc_eligible(const AttnArgs& a) {
  const uintptr_t al = reinterpret_cast<uintptr_t>(a.comp.data) | reinterpret_cast<uintptr_t>(a.swa.data);
  return a.dim == kD && a.heads == kH && a.comp.dtype == a.swa.dtype && a.comp.tail_bf16 == a.swa.tail_bf16 &&
         (a.comp.dtype == CSA_BF16 || a.comp.dtype == CSA_E4M3 || a.comp.dtype == CSA_E4M3R) &&
         a.comp.tail_bf16 <= kD / kChunks && a.rope.rope_dim <= 128 && al % 16 == 0;
}

int32_t attn_tc_splits(int32_t n_rows, int32_t keys_per_row) {
  // a power of two <= 8 (one cluster per row), about one CTA per SM in all, and
  // at least 256 keys per CTA
  const int32_t tiles = (keys_per_row + 127) / 128;
  int32_t s = 1;
  while (s < 8 && 2 * s * n_rows <= 148 && 2 * s <= tiles) s *= 2;
  return s;
}

cudaError_t launch_attn_tc(const AttnArgs& a, int32_t n_rows, cudaStream_t s) {
  static PerDevice attrs;
  cudaError_t e = with_device_slot(attrs, [](int, int64_t& done) {
    if (done) return cudaSuccess;
    cudaError_t r = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (r == cudaSuccess) r = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
    if (r == cudaSuccess) done = 1;
    return r;
  });
  if (e != cudaSuccess) return e;
  return launch_k(attn_tc_kernel, dim3(n_rows, a.n_splits), dim3(kThreads), kSmemBytes, s, a.n_splits,
                  a);
}

}  // namespace csa
