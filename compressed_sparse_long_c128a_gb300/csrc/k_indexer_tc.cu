// DSA indexer scores on the sm_103a tensor cores: s_i = sum_h w_h relu(q_h . k_i)
// ("vLLM解密：DeepSeek-V4本地部署為何如此困難" §二 item 3; "vLLM DeepSeek V4
// Support", "DeepSeek Sparse Attention (DSA)"; fp4 indexer cache: "DeepSeek V4
// Attention Architecture", last paragraph).
//
// Shape: 64 indexer heads x 128 dims.  One CTA takes one query row and a
// contiguous range of 128-entry tiles.  Entries are the M dimension:
//   S^T [128 entries x 64 heads] = K_idx [128 x 128] . Q_idx^T [128 x 64]
// so thread t of the epilogue warps owns TMEM lane t = entry t, reads its 64
// head dots and forms one score.  TMEM holds two S^T buffers so the epilogue
// of tile i overlaps the MMA of tile i+1.
//
// Keys reach shared memory as 128B-swizzled K-major bf16 tiles.  A tile is two
// 64-entry paged blocks; a bf16 block is 16 KB contiguous, so a bf16 tile
// arrives as four TMA boxes (64 dims x 64 entries) issued by one thread.  An
// e2m1 block is 4 KB of codes plus 512 B of e4m3 scales, each contiguous: one
// thread issues four bulk copies per tile into a six-deep raw ring, and six
// warps turn the codes into bf16 (exact: a 2-bit e2m1 significand times a
// 4-bit e4m3 one fits bf16's 8 bits).
//
// Two ways to cut the work:
//   * balanced deal (decode batches, IndexerArgs::sel_k > 0): the grid is one
//     wave of G CTAs, and every CTA derives from the rows' positions the same
//     deal of each row's tiles in proportion to its length (select.cuh), so
//     short and long rows finish together.  The CTA keeps its scores in shared
//     memory and, after its last tile, selects their top-k itself; the deal
//     merge then combines each row's candidate lists.  No score reaches HBM.
//   * one CTA per row and split (sel_k == 0, prefill-sized batches): every
//     score goes to the caller's scratch for the top-k kernels.
//
// Warps 0-3: epilogue; then the producers (bf16: warps 4-10, one TMA thread;
// e2m1: warps 4-14, warp 4 issues the bulk copies and ten warps convert); the
// last warp: TMEM allocation + MMA issue.  After the last tile every warp runs
// the selection.

#include "select.cuh"
#include "tc_ptx.cuh"

namespace csa {
namespace {

using namespace tc;

constexpr int kHI = 64, kDI = 128, kTile = kDealTile;
constexpr int kEpi = 128;
constexpr uint32_t kQBytes = kHI * kDI * 2;        // 16 KB: 2 K-atoms of 64 rows x 128 B
constexpr uint32_t kStageBytes = kTile * kDI * 2;  // 32 KB: 2 K-atoms of 128 rows x 128 B
constexpr uint32_t kAtomBytes = kTile * 128;       // 16 KB
constexpr int kRowsPerBlock = 64;                  // entries per 256-position block (c4a)
constexpr uint32_t kBlockCodes = kRowsPerBlock * kDI / 2;    // 4 KB of e2m1 codes per block
constexpr uint32_t kBlockScales = kRowsPerBlock * kDI / 16;  // 512 B of e4m3 scales per block
constexpr uint32_t kRawCodes = 2 * kBlockCodes;
constexpr uint32_t kRawBytes = kRawCodes + 2 * kBlockScales;  // 9 KB per tile
constexpr int kTblMax = 1024;  // block-table entries a CTA caches (= 512 tiles)

// Shared-memory plan per key format.
template <bool kFp4, int kR = 1>
struct Plan {
  // warps 0-3 epilogue; then the producers (bf16: one TMA thread in warp 4;
  // e2m1: warp 4 issues the bulk copies, the other ten convert); the last warp
  // allocates TMEM and issues the MMAs
  static constexpr int kProd = kFp4 ? 352 : 224;
  static constexpr int kThreads = kEpi + kProd + 32;
  static constexpr int kMmaWarp = (kEpi + kProd) / 32;
  static constexpr int kConvThreads = kProd - 32;
  static constexpr int kStages = kFp4 ? 3 : 4;       // bf16 tiles the MMA reads
  static constexpr int kRaw = kFp4 ? 6 : 0;          // raw e2m1 tiles in flight
  // kR query rows share every key tile (prefill: four rows of one sequence as
  // N = 256 of the MMA); the fused selection is for single rows only
  static constexpr int kCapTiles = kR > 1 ? 0 : (kFp4 ? 64 : 104);  // tiles whose keys the fused selection holds
  static constexpr uint32_t kTmemCols = 2 * 64 * kR;  // two S^T buffers of 64 kR columns
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffStage = kR * kQBytes;
  static constexpr uint32_t kOffRaw = kOffStage + kStages * kStageBytes;
  static constexpr uint32_t kOffKeys = kOffRaw + kRaw * kRawBytes;
  static constexpr uint32_t kKeyBytes = ((uint32_t)padded_size(kCapTiles * kTile) * 4 + 1023) & ~1023u;
  static constexpr uint32_t kOffMisc = kOffKeys + kKeyBytes;
};

struct Misc {
  uint64_t full[4], empty[4], raw_full[6], raw_empty[6], tfull[2], tempty[2], mma_done, qswap;
  uint32_t tmem_base;
  int32_t abort;
  int32_t row[2], t0[2], nt[2];  // the CTA's segments (row -1: none)
  int32_t nr, rr[4], rn[4];      // multi-row CTA: its rows and their visible entries
  alignas(16) float w[4][kHI];
  int32_t tbl[kTblMax];     // physical blocks of the CTA's tiles (-1: unmapped / out of range)
  uint32_t hist0[2][2048];  // fused selection: counts of each segment's keys' top 11 bits, built during the loop
};

// Scratch of the selection after the loop, in the drained stage ring.
struct PickScratch {
  uint32_t hist1[2048];
  uint32_t wsum[32];
  uint32_t digit, rem, above;
};

template <bool kFp4, int kR = 1>
constexpr uint32_t smem_bytes() {
  return Plan<kFp4, kR>::kOffMisc + sizeof(Misc) + 1024;
}
static_assert(sizeof(DealShared) <= kStageBytes, "the deal is built in the idle stage ring");
static_assert(sizeof(SelectScratch) + sizeof(PickScratch) <= kStageBytes,
              "the selection scratch reuses the drained stage ring");
static_assert(smem_bytes<false>() <= 227 * 1024 && smem_bytes<true>() <= 227 * 1024 &&
                  smem_bytes<false, 4>() <= 227 * 1024, "shared memory");

__device__ __forceinline__ bool wait_or_abort(Misc& ms, uint64_t* bar, uint32_t parity, int32_t* err) {
  if (*reinterpret_cast<volatile int32_t*>(&ms.abort)) return false;
  if (mbar_wait(bar, parity)) return true;
  *reinterpret_cast<volatile int32_t*>(&ms.abort) = 1;
  record_error(err, CSA_ERR_TIMEOUT);
  return false;
}

// The CTA's tiles: segment 0, then segment 1 (under the even deal, the head
// of the next row).  Local tile i < nt[0] is tile t0[0] + i of row[0]; the
// rest are tiles 0.. of row[1].
struct Range {
  int nseg, nt_all;
  int nr, rr[4];
  int32_t rn[4];  // multi-row CTA: rows sharing the tiles (one sequence) and their visible entries
  int row[2], seq[2];
  int32_t n[2], t0[2], nt[2];  // visible entries of the row, first tile, tile count
  __device__ __forceinline__ int seg_of(int i) const { return i >= nt[0] ? 1 : 0; }
  __device__ __forceinline__ int32_t tile_of(int i) const { return i >= nt[0] ? t0[1] + i - nt[0] : t0[0] + i; }
};

// High and low bytes of the bf16 bits of the e2m1 magnitudes 0, 0.5, 1, 1.5, 2,
// 3, 4, 6, as byte-permute tables indexed by the 3-bit magnitude code.
constexpr uint32_t kMagHi03 = 0x3F3F3F00u, kMagHi47 = 0x40404040u;
constexpr uint32_t kMagLo03 = 0xC0800000u, kMagLo47 = 0xC0804000u;

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Eight e2m1 codes (nibble j of w is value j) times one scale (bf16, in both
// halves of scale2) -> four bf16x2 words, word e holding values 2e and 2e+1.
// The magnitudes come from byte-permute lookups, the signs from a permute of
// the codes' sign bits.  The multiply is exact: a 2-bit e2m1 significand times
// a 4-bit e4m3 one fits bf16's 8 bits, and the products stay in bf16's normal
// range (2^-10 .. 2688).
__device__ __forceinline__ void e2m1x8_bf16x2(uint32_t w, uint32_t scale2, uint32_t o[4]) {
  const uint32_t mag = w & 0x77777777u;
  const uint32_t sl = (w << 4) & 0x80808080u;  // sign of value 2e at bit 7 of byte e
  const uint32_t sh = w & 0x80808080u;         // sign of value 2e+1 at bit 7 of byte e
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t sel = mag >> (16 * h);  // values 4h..4h+3 (the permute reads 4 nibbles)
    const uint32_t hi = __byte_perm(kMagHi03, kMagHi47, sel) | __byte_perm(sl, sh, h ? 0x7362u : 0x5140u);
    const uint32_t lo = __byte_perm(kMagLo03, kMagLo47, sel);
    o[2 * h] = bf16x2_mul(__byte_perm(lo, hi, 0x5140u), scale2);
    o[2 * h + 1] = bf16x2_mul(__byte_perm(lo, hi, 0x7362u), scale2);
  }
}

// e4m3 scale -> its bf16 bits in both halves (exact: 4 significant bits)
__device__ __forceinline__ uint32_t e4m3_bf16x2(uint8_t v) {
  const uint32_t b = __float_as_uint(e4m3_to_f32(v)) >> 16;
  return b | (b << 16);
}

// Physical block of tile-half h (0, 1) of tile i of the range, or -1 when
// unmapped or past the visible entries (then nothing is loaded).
__device__ __forceinline__ int32_t tile_block(const Misc& ms, const Range& g, int i, int h) {
  const int32_t e = g.tile_of(i) * kTile + h * kRowsPerBlock;
  const int32_t j = 2 * i + h;  // the cached table follows the CTA's tiles
  return (e < g.n[g.seg_of(i)] && j < kTblMax) ? ms.tbl[j] : -1;
}

// bf16: one thread issues each tile as up to four TMA boxes (two blocks x two
// 64-dim atoms).
template <bool kFp4, int kR>
__device__ void producer_bf16(const IndexerArgs& a, const Range& g, uint8_t* smem, Misc& ms) {
  using P = Plan<kFp4, kR>;
  const uint64_t pol = policy_evict_first();
  for (int i = 0; i < g.nt_all; ++i) {
    const int s = i % P::kStages;
    if (i >= P::kStages) wait_or_abort(ms, &ms.empty[s], ((i / P::kStages) - 1) & 1, a.err);
    int32_t pb[2];
    uint32_t bytes = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      pb[h] = tile_block(ms, g, i, h);
      if (pb[h] >= 0) bytes += kRowsPerBlock * kDI * 2;
    }
    mbar_arrive_expect_tx(&ms.full[s], bytes);
    uint8_t* sb = smem + P::kOffStage + s * kStageBytes;
#pragma unroll
    for (int h = 0; h < 2; ++h)
      if (pb[h] >= 0)
#pragma unroll
        for (int at = 0; at < kDI / 64; ++at)
          tma_load_2d_hint(sb + at * kAtomBytes + h * (kRowsPerBlock * 128), &a.k_map, 64 * at,
                           pb[h] * kRowsPerBlock, &ms.full[s], pol);
  }
}

// e2m1, issuing thread: each tile's codes and scales as four bulk copies into
// the raw ring (layout per tile: [128 entries][64 code bytes] then
// [128 entries][8 scale bytes]).
template <bool kFp4, int kR>
__device__ void producer_raw(const IndexerArgs& a, const Range& g, uint8_t* smem, Misc& ms) {
  using P = Plan<kFp4, kR>;
  const uint8_t* codes = reinterpret_cast<const uint8_t*>(a.cache.data);
  const uint8_t* scales = reinterpret_cast<const uint8_t*>(a.cache.scales);
  const uint64_t pol = policy_evict_first();
  for (int i = 0; i < g.nt_all; ++i) {
    const int rs = i % P::kRaw;
    if (i >= P::kRaw) wait_or_abort(ms, &ms.raw_empty[rs], ((i / P::kRaw) - 1) & 1, a.err);
    int32_t pb[2];
    uint32_t bytes = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      pb[h] = tile_block(ms, g, i, h);
      if (pb[h] >= 0) bytes += kBlockCodes + kBlockScales;
    }
    mbar_arrive_expect_tx(&ms.raw_full[rs], bytes);
    uint8_t* rb = smem + P::kOffRaw + rs * kRawBytes;
#pragma unroll
    for (int h = 0; h < 2; ++h)
      if (pb[h] >= 0) {
        bulk_load_hint(rb + h * kBlockCodes, codes + (int64_t)pb[h] * kBlockCodes, kBlockCodes, &ms.raw_full[rs],
                       pol);
        bulk_load_hint(rb + kRawCodes + h * kBlockScales, scales + (int64_t)pb[h] * kBlockScales, kBlockScales,
                       &ms.raw_full[rs], pol);
      }
  }
}

// e2m1, converting warps: raw tile -> bf16 tile of the stage ring.  A code of
// an unloaded block is stale; its entry's score is not used.
template <bool kFp4, int kR>
__device__ void converter(const IndexerArgs& a, const Range& g, uint8_t* smem, Misc& ms, int ct) {
  using P = Plan<kFp4, kR>;
  for (int i = 0; i < g.nt_all; ++i) {
    const int rs = i % P::kRaw, s = i % P::kStages;
    wait_or_abort(ms, &ms.raw_full[rs], (i / P::kRaw) & 1, a.err);
    if (i >= P::kStages) wait_or_abort(ms, &ms.empty[s], ((i / P::kStages) - 1) & 1, a.err);
    const uint8_t* rb = smem + P::kOffRaw + rs * kRawBytes;
    uint8_t* sb = smem + P::kOffStage + s * kStageBytes;
    // 16 bytes of codes = 32 values = 64 bytes of bf16 = 4 swizzled pieces
    for (int x = ct; x < kTile * 4; x += P::kConvThreads) {
      const uint32_t key = x >> 2, q = x & 3;
      const uint4 c4 = *reinterpret_cast<const uint4*>(rb + key * 64 + q * 16);
      const uint8_t* sc = rb + kRawCodes + key * 8 + q * 2;
      const uint32_t s0 = e4m3_bf16x2(sc[0]), s1 = e4m3_bf16x2(sc[1]);
      const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
      for (int half = 0; half < 4; ++half) {  // 8 values -> one 16-byte piece
        uint32_t o[4];
        e2m1x8_bf16x2(cw[half], half < 2 ? s0 : s1, o);
        const uint32_t piece = q * 4 + half;  // 0..15 over the 128 dims
        *reinterpret_cast<uint4*>(sb + (piece >> 3) * kAtomBytes + (key >> 3) * 1024 + (key & 7) * 128 +
                                  (((piece & 7) ^ (key & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    fence_proxy_async();
    mbar_arrive(&ms.full[s]);
    mbar_arrive(&ms.raw_empty[rs]);
  }
}

// Q_idx^T of `row` into the Q area, by threads [t0, t0 + nthr) of the CTA:
// bf16, 128B-swizzled K-major, rows = heads (at N rows n_off.. of an operand
// of n_all rows); 8 dims per 16-byte piece, each thread's loads (kB at a
// time) issued before its stores.
template <int kB>
__device__ __forceinline__ void load_q(const IndexerArgs& a, int row, uint8_t* q_smem, int t, int nthr,
                                       int n_off = 0, uint32_t n_all = kHI) {
  constexpr int kPieces = kHI * kDI / 8;
  for (int x0 = t; x0 < kPieces; x0 += kB * nthr) {
    uint32_t w[kB][4];
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int x = x0 + u * nthr;
      if (x >= kPieces) break;
      const int64_t qb = (int64_t)row * kHI * kDI + 8 * x;
      if (a.q_dtype == CSA_BF16) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q_idx) + qb));
        w[u][0] = v.x; w[u][1] = v.y; w[u][2] = v.z; w[u][3] = v.w;
      } else {
        const float4* src = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.q_idx) + qb);
        const float4 v0 = __ldg(src), v1 = __ldg(src + 1);
        w[u][0] = f32x2_to_bf16x2(v0.x, v0.y);
        w[u][1] = f32x2_to_bf16x2(v0.z, v0.w);
        w[u][2] = f32x2_to_bf16x2(v1.x, v1.y);
        w[u][3] = f32x2_to_bf16x2(v1.z, v1.w);
      }
    }
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int x = x0 + u * nthr;
      if (x >= kPieces) break;
      const int h = x / (kDI / 8), d0 = 8 * (x % (kDI / 8));
      *reinterpret_cast<uint4*>(q_smem + sw128_offset(n_off + h, d0, n_all)) =
          make_uint4(w[u][0], w[u][1], w[u][2], w[u][3]);
    }
  }
}

// The MMA warp: lane 0 issues every MMA.  At the start of a second segment the
// whole warp waits for the first segment's MMAs to finish reading Q and loads
// the second row's Q_idx in its place (the producers keep streaming tiles
// meanwhile).
template <bool kFp4, int kR>
__device__ void mma_role(const IndexerArgs& a, const Range& g, uint8_t* smem, Misc& ms, uint32_t tmem, int lane) {
  using P = Plan<kFp4, kR>;
  constexpr uint32_t idesc = idesc_bf16(128, kHI * kR, 0, 0);
  const uint32_t stage0 = smem_u32(smem + P::kOffStage), qbase = smem_u32(smem + P::kOffQ);
  for (int i = 0; i < g.nt_all; ++i) {
    const int s = i % P::kStages, b = i & 1;
    if (kR == 1 && g.nseg == 2 && i == g.nt[0]) {
      if (lane == 0) mma_commit(&ms.qswap);
      __syncwarp();
      wait_or_abort(ms, &ms.qswap, 0, a.err);
      load_q<kFp4 ? 4 : 8>(a, g.row[1], smem + P::kOffQ, lane, 32);  // L2-warm: prefetched at the start
      fence_proxy_async();
      __syncwarp();
    }
    wait_or_abort(ms, &ms.full[s], (i / P::kStages) & 1, a.err);
    if (i >= 2) wait_or_abort(ms, &ms.tempty[b], ((i >> 1) - 1) & 1, a.err);
    tc_fence_after();
    if (lane == 0) {
#pragma unroll
      for (int ks = 0; ks < kDI / 16; ++ks) {
        const uint64_t ad =
            sdesc_sw128(stage0 + s * kStageBytes + (ks >> 2) * kAtomBytes + (ks & 3) * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(qbase + (ks >> 2) * (kR * kHI * 128) + (ks & 3) * 32, 16, 1024);
        mma_bf16(tmem + kR * kHI * b, ad, bd, idesc, ks > 0);
      }
      mma_commit(&ms.empty[s]);
      mma_commit(&ms.tfull[b]);
    }
    __syncwarp();
  }
  // nothing may still write TMEM when it is released, even after a timeout
  if (lane == 0) {
    mma_commit(&ms.mma_done);
    if (!mbar_wait(&ms.mma_done, 0)) record_error(a.err, CSA_ERR_TIMEOUT);
  }
  __syncwarp();
}

// Scores of the range: to shared memory as order keys (fused selection) or to
// the caller's score scratch.  An entry of an unmapped block scores -inf.
template <bool kFp4, int kR>
__device__ void epilogue_role(const IndexerArgs& a, const Range& g, uint8_t* smem, Misc& ms, uint32_t tmem,
                              int et, int j0 = 0, int j1 = 0) {
  using P = Plan<kFp4, kR>;
  const uint32_t lane_addr = tmem + ((uint32_t)((et >> 5) * 32) << 16);
  float w[kHI];
#pragma unroll
  for (int h = 0; h < kHI; ++h) w[h] = ms.w[0][h];
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + P::kOffKeys);
  float* out = a.scores + (int64_t)g.row[0] * a.max_n;
  if constexpr (kR > 1) {
    // every row of the CTA reads the same tile: row j's 64 head dots are TMEM
    // columns 64 kR b + 64 j of this thread's lane.  This thread takes rows
    // [j0, j1) of entry et; four partial sums keep the dependent chain short.
    j1 = min(j1, g.nr);
    for (int i = 0; i < g.nt_all; ++i) {
      const int b = i & 1;
      wait_or_abort(ms, &ms.tfull[b], (i >> 1) & 1, a.err);
      tc_fence_after();
      const int32_t e = g.tile_of(i) * kTile + et, jt = 2 * i + et / kRowsPerBlock;
      const bool mapped = jt < kTblMax && ms.tbl[jt] >= 0;
      for (int j = j0; j < j1; ++j) {
        float v[kHI];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld16(lane_addr + kR * kHI * b + kHI * j + 16 * q, v + 16 * q);
        tmem_wait_ld();
        const float4* w4 = reinterpret_cast<const float4*>(ms.w[j]);
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int q = 0; q < kHI / 4; ++q) {
          const float4 ww = w4[q];
          s4[0] = fmaf(ww.x, fmaxf(v[4 * q], 0.f), s4[0]);
          s4[1] = fmaf(ww.y, fmaxf(v[4 * q + 1], 0.f), s4[1]);
          s4[2] = fmaf(ww.z, fmaxf(v[4 * q + 2], 0.f), s4[2]);
          s4[3] = fmaf(ww.w, fmaxf(v[4 * q + 3], 0.f), s4[3]);
        }
        const float s = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        if (e < g.rn[j]) a.scores[(int64_t)g.rr[j] * a.max_n + e] = mapped ? s : -INFINITY;
      }
      tc_fence_before();
      mbar_arrive(&ms.tempty[b]);
    }
    return;
  }
  int seg = 0;
  for (int i = 0; i < g.nt_all; ++i) {
    const int b = i & 1;
    if (g.nseg == 2 && i == g.nt[0]) {  // the second row's weights
      seg = 1;
#pragma unroll
      for (int h = 0; h < kHI; ++h) w[h] = ms.w[1][h];
    }
    wait_or_abort(ms, &ms.tfull[b], (i >> 1) & 1, a.err);
    tc_fence_after();
    float s = 0.f;
    if constexpr (kFp4) {
      // the row's 64 head dots in two halves of 32 columns (registers for 512 threads)
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float v[kHI / 2];
        tmem_ld16(lane_addr + 64 * b + 32 * half, v);
        tmem_ld16(lane_addr + 64 * b + 32 * half + 16, v + 16);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < kHI / 2; ++h) s = fmaf(w[32 * half + h], fmaxf(v[h], 0.f), s);
      }
    } else {
      float v[kHI];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld16(lane_addr + 64 * b + 16 * q, v + 16 * q);
      tmem_wait_ld();
#pragma unroll
      for (int h = 0; h < kHI; ++h) s = fmaf(w[h], fmaxf(v[h], 0.f), s);
    }
    tc_fence_before();
    mbar_arrive(&ms.tempty[b]);
    const int32_t e = g.tile_of(i) * kTile + et, j = 2 * i + et / kRowsPerBlock;
    if (e < g.n[seg]) {
      const float sc = (j < kTblMax && ms.tbl[j] >= 0) ? s : -INFINITY;
      if (a.sel_k > 0) {
        const uint32_t key = order_key(sc);
        keys[padded(i * kTile + et)] = key;
        atomicAdd(&ms.hist0[seg][key >> 21], 1u);
      } else {
        out[e] = sc;
      }
    }
  }
}

template <bool kFp4, int kR>
__global__ void __launch_bounds__(Plan<kFp4, kR>::kThreads, 1) indexer_tc_kernel(const __grid_constant__ IndexerArgs a) {
  using P = Plan<kFp4, kR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc& ms = *reinterpret_cast<Misc*>(smem + P::kOffMisc);
  const int tid = threadIdx.x, warp = tid >> 5;
  pdl_trigger();
  pdl_wait();  // before any access to memory: the previous kernel on the stream may still be running

  // the CTA's rows and tile ranges
  if (a.sel_k > 0) {
    DealShared& ds = *reinterpret_cast<DealShared*>(smem + P::kOffStage);
    if (warp == 0) deal_compute(a.pos, a.n_rows, a.ratio, a.window, a.max_n, gridDim.x, P::kCapTiles, ds);
    __syncthreads();
    if (blockIdx.x == 0)  // each row's list slots, for the merge
      for (int r = tid; r < a.n_rows; r += P::kThreads) {
        a.cand_row_first[r] = ds.first[r];
        a.cand_row_ctas[r] = ds.ctas[r];
        a.cand_row_seg[r] = ds.seg[r];
      }
    if (tid == 0) {
      const DealSlot sl = deal_slot(ds, a.n_rows, blockIdx.x, gridDim.x);
      for (int q = 0; q < 2; ++q) {
        ms.row[q] = sl.row[q];
        ms.t0[q] = sl.t0[q];
        ms.nt[q] = sl.nt[q];
      }
    }
  } else if (tid == 0) {
    // one row per blockIdx.x, its tiles split in equal parts over gridDim.y.
    // With kR rows a CTA, blockIdx.x = 4q leads rows 4q..4q+3: it takes every
    // one of them in the sequence of row 4q (they then share every key tile);
    // the others exit, unless their own sequence differs, when they take
    // their row alone.
    const int r = blockIdx.x;
    int nr = 1;
    ms.rr[0] = r;
    if constexpr (kR > 1) {
      const int lead = r & ~(kR - 1);
      const int lead_seq = a.seq_id[lead];
      if (r != lead && a.seq_id[r] == lead_seq) {
        nr = 0;
      } else if (r == lead) {
        nr = 0;
        for (int j = 0; j < kR && lead + j < a.n_rows; ++j)
          if (a.seq_id[lead + j] == lead_seq) ms.rr[nr++] = lead + j;
      }
    }
    int32_t tiles = 0;
    for (int j = 0; j < nr; ++j) tiles = max(tiles, deal_row_tiles(a.pos, ms.rr[j], a.ratio, a.window, a.max_n));
    const int32_t per = (tiles + gridDim.y - 1) / gridDim.y;
    ms.nr = nr;
    ms.row[0] = nr ? ms.rr[0] : -1;
    ms.t0[0] = min(tiles, (int32_t)blockIdx.y * per);
    ms.nt[0] = min(tiles, ms.t0[0] + per) - ms.t0[0];
    ms.row[1] = -1;
    ms.t0[1] = ms.nt[1] = 0;
  }
  __syncthreads();
  Range g;
  g.nseg = ms.row[0] < 0 ? 0 : (ms.row[1] < 0 ? 1 : 2);
  if (g.nseg == 0) return;  // a CTA the deal left without work
  for (int q = 0; q < 2; ++q) {
    g.row[q] = ms.row[q];
    g.t0[q] = ms.t0[q];
    g.nt[q] = q < g.nseg ? ms.nt[q] : 0;
  }
  if (a.sel_k > 0 && g.nt[0] + g.nt[1] > P::kCapTiles) {
    // the launcher's bound and the deal rule this out; never overrun the key store
    if (tid == 0) record_error(a.err, CSA_ERR_DEVICE_BOUNDS);
    g.nt[0] = min(g.nt[0], P::kCapTiles);
    g.nt[1] = min(g.nt[1], P::kCapTiles - g.nt[0]);
    if (g.nt[1] == 0) g.nseg = 1;
  }
  g.nt_all = g.nt[0] + g.nt[1];
  for (int q = 0; q < g.nseg; ++q) {
    g.seq[q] = a.seq_id[g.row[q]];
    g.n[q] = n_visible(a.pos[g.row[q]], a.ratio, a.window);
    if (g.n[q] > a.max_n) {
      if (tid == 0 && (a.sel_k > 0 ? g.t0[q] == 0 : blockIdx.y == 0)) record_error(a.err, CSA_ERR_DEVICE_BOUNDS);
      g.n[q] = a.max_n;
    }
  }
  if (g.nseg == 1) {
    g.seq[1] = -1;
    g.n[1] = 0;
  }
  g.nr = 0;
  if constexpr (kR > 1) {
    // the CTA's rows (one sequence): each row's visible entries; the tiles
    // cover the longest (g.n[0] is its count)
    g.nr = ms.nr;
    g.n[0] = 0;
    for (int j = 0; j < g.nr; ++j) {
      g.rr[j] = ms.rr[j];
      g.rn[j] = n_visible(a.pos[g.rr[j]], a.ratio, a.window);
      if (g.rn[j] > a.max_n) {
        if (tid == 0 && blockIdx.y == 0) record_error(a.err, CSA_ERR_DEVICE_BOUNDS);
        g.rn[j] = a.max_n;
      }
      g.n[0] = max(g.n[0], g.rn[j]);
    }
  }

  if (tid == 0) {
    for (int s = 0; s < 4; ++s) {
      mbar_init(&ms.full[s], kFp4 ? P::kConvThreads : 1);
      mbar_init(&ms.empty[s], 1);
    }
    for (int s = 0; s < 6; ++s) {
      mbar_init(&ms.raw_full[s], 1);
      mbar_init(&ms.raw_empty[s], P::kConvThreads);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ms.tfull[b], 1);
      mbar_init(&ms.tempty[b], kR > 1 ? 2 * kEpi : kEpi);
    }
    mbar_init(&ms.mma_done, 1);
    mbar_init(&ms.qswap, 1);
    mbar_init_fence();
    ms.abort = 0;
  }
  if constexpr (kR > 1) {
    if (tid < g.nr * kHI) ms.w[tid / kHI][tid % kHI] = a.w[(int64_t)g.rr[tid / kHI] * kHI + tid % kHI];
  } else {
    if (tid < g.nseg * kHI) ms.w[tid / kHI][tid % kHI] = a.w[(int64_t)g.row[tid / kHI] * kHI + tid % kHI];
  }
  for (int b = tid; b < 2 * 2048; b += P::kThreads) (&ms.hist0[0][0])[b] = 0;
  {
    // block-table entries of the CTA's tiles, two blocks a tile
    const int32_t nblk = min(kTblMax, g.nt_all * (kTile / kRowsPerBlock));
    for (int j = tid; j < nblk; j += P::kThreads) {
      const int i = j / (kTile / kRowsPerBlock), q = g.seg_of(i);
      const int32_t lb = g.tile_of(i) * (kTile / kRowsPerBlock) + j % (kTile / kRowsPerBlock);
      int32_t pb = -1;
      if (g.seq[q] >= 0 && g.seq[q] < a.bt.num_seqs && lb < a.bt.stride) {
        pb = a.bt.table[(int64_t)g.seq[q] * a.bt.stride + lb];
        if (pb >= a.cache.num_blocks) pb = -1;
      }
      if (pb < 0 && lb * kRowsPerBlock < g.n[q]) record_error(a.err, CSA_ERR_DEVICE_BOUNDS);
      ms.tbl[j] = pb;
    }
  }
  if (warp == P::kMmaWarp) tmem_alloc(&ms.tmem_base, P::kTmemCols);
  if constexpr (kR > 1) {
    for (int j = 0; j < g.nr; ++j) load_q<4>(a, g.rr[j], smem + P::kOffQ, tid, P::kThreads, kHI * j, kR * kHI);
  } else {
    load_q<4>(a, g.row[0], smem + P::kOffQ, tid, P::kThreads);
    // the second row's Q_idx (swapped in by the MMA warp mid-loop) into L2 now
    if (g.nseg == 2 && tid < kHI * kDI * 2 / 128) {
      const char* q1 = reinterpret_cast<const char*>(a.q_idx) +
                       (int64_t)g.row[1] * kHI * kDI * (a.q_dtype == CSA_BF16 ? 2 : 4);
      for (int o = tid * 128; o < kHI * kDI * (a.q_dtype == CSA_BF16 ? 2 : 4); o += kHI * kDI * 2)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(q1 + o));
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;

  if (warp < 4) {
    epilogue_role<kFp4, kR>(a, g, smem, ms, tmem, tid, 0, kR / 2);
  } else if (kR > 1 && warp >= 5 && warp < 9) {
    // multi-row: warps 5-8 (idle producers of the bf16 plan) take the other
    // half of the rows; warp w reads TMEM lanes 32 (w mod 4) ..
    epilogue_role<kFp4, kR>(a, g, smem, ms, tmem, 32 * (warp & 3) + (tid & 31), kR / 2, kR);
  } else if (warp < P::kMmaWarp) {
    if constexpr (!kFp4) {
      if (tid == kEpi) producer_bf16<kFp4, kR>(a, g, smem, ms);
    } else {
      if (warp == kEpi / 32) {
        if (tid == kEpi) producer_raw<kFp4, kR>(a, g, smem, ms);
      } else {
        converter<kFp4, kR>(a, g, smem, ms, tid - kEpi - 32);
      }
    }
  } else {
    mma_role<kFp4, kR>(a, g, smem, ms, tmem, tid & 31);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == P::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, P::kTmemCols);
  }
  if (kR > 1 || a.sel_k <= 0) return;

  // fused selection, once per segment.  The list a segment hands to the merge
  // is every key of its range at or above T22, the k-th largest key with its
  // low 10 bits cleared (a superset of the range's top-k, in entry order), with
  // T22 itself: the merge keeps only keys at or above the largest T22 of the
  // row's lists, which is at most the row's own k-th key.  Radix digits: the
  // top 11 bits were counted during the loop; one more pass fixes the next 11.
  PickScratch& pk = *reinterpret_cast<PickScratch*>(smem + P::kOffStage);
  SelectScratch& sc = *reinterpret_cast<SelectScratch*>(smem + P::kOffStage + sizeof(PickScratch));
  const int cap = 2 * a.sel_k;  // list capacity per slot
  for (int q = 0; q < g.nseg; ++q) {
    const int i0 = q ? g.nt[0] : 0;  // the segment's first local tile; its keys start at i0 * kTile
    const int32_t e0 = g.t0[q] * kTile;
    const int n_local = max(0, min(g.n[q], (g.t0[q] + g.nt[q]) * kTile) - e0);
    const uint32_t* keys = reinterpret_cast<const uint32_t*>(smem + P::kOffKeys) + padded(i0 * kTile);
    const uint32_t* hist0 = ms.hist0[q];
    const int64_t slot = 2 * (int64_t)blockIdx.x + q;
    uint32_t* ck = a.cand_key + slot * cap;
    int32_t* ci = a.cand_idx + slot * cap;
    uint32_t T = 0;  // every key qualifies when the range has at most k of them
    if (n_local > a.sel_k) {
      for (int b = tid; b < 2048; b += P::kThreads) pk.hist1[b] = 0;
      uint32_t rem = (uint32_t)a.sel_k, d0 = 0, d1 = 0;
      for (int pass = 0; pass < 2; ++pass) {
        const uint32_t* hist = pass == 0 ? hist0 : pk.hist1;
        if (pass == 1) {
          for (int i = tid; i < n_local; i += P::kThreads) {
            const uint32_t key = keys[padded(i)];
            if ((key >> 21) == d0) atomicAdd(&pk.hist1[(key >> 10) & 2047u], 1u);
          }
          __syncthreads();
        }
        // the digit d with count(> d) < rem <= count(>= d), buckets scanned from the top
        constexpr int kBpt = (2048 + P::kThreads - 1) / P::kThreads;
        const int top = 2048 - tid * kBpt;
        uint32_t local = 0;
        for (int jj = 0; jj < kBpt; ++jj)
          if (top - 1 - jj >= 0) local += hist[top - 1 - jj];
        uint32_t tot;
        const uint32_t above = block_excl_scan<P::kThreads>(local, pk.wsum, tot);
        if (above < rem && rem <= above + local) {
          uint32_t cum = above;
          for (int jj = 0; jj < kBpt && top - 1 - jj >= 0; ++jj) {
            const uint32_t h = hist[top - 1 - jj];
            if (cum + h >= rem) {
              pk.digit = (uint32_t)(top - 1 - jj);
              pk.rem = rem - cum;
              break;
            }
            cum += h;
          }
        }
        __syncthreads();
        if (pass == 0) d0 = pk.digit;
        else d1 = pk.digit;
        rem = pk.rem;
        __syncthreads();
      }
      T = (d0 << 21) | (d1 << 10);
    }
    // keys at or above T, in entry order: one count per thread segment, one scan
    const int seg = (n_local + P::kThreads - 1) / P::kThreads;
    const int lo = tid * seg, hi = min(n_local, lo + seg);
    uint32_t mine = 0;
    for (int i = lo; i < hi; ++i) mine += keys[padded(i)] >= T;
    uint32_t total;
    uint32_t at = block_excl_scan<P::kThreads>(mine, pk.wsum, total);
    if ((int)total <= cap) {
      for (int i = lo; i < hi; ++i) {
        const uint32_t key = keys[padded(i)];
        if (key >= T) {
          ck[at] = key;
          ci[at] = e0 + i;
          ++at;
        }
      }
      if (tid == 0) {
        a.cand_cnt[slot] = (int32_t)total;
        a.cand_thr[slot] = T;
      }
    } else {
      // many keys tie within T's 22-bit bucket: the exact top-k instead, with its
      // k-th key as the threshold (still a lower bound of the row's k-th key)
      if (tid == 0) pk.digit = 0xFFFFFFFFu;  // reused as the block minimum of the selected keys
      __syncthreads();
      uint32_t kth = 0xFFFFFFFFu;
      block_select<P::kThreads>(keys, n_local, a.sel_k, sc, [&](int pos, uint32_t rank) {
        const uint32_t key = keys[padded(pos)];
        ck[rank] = key;
        ci[rank] = e0 + pos;
        kth = min(kth, key);
      });
      for (int o = 16; o > 0; o >>= 1) kth = min(kth, __shfl_xor_sync(0xffffffffu, kth, o));
      if ((tid & 31) == 0) atomicMin(&pk.digit, kth);
      __syncthreads();
      if (tid == 0) {
        a.cand_cnt[slot] = a.sel_k;
        a.cand_thr[slot] = pk.digit;
      }
    }
    __syncthreads();  // the scratch is reused by the next segment
  }
}

}  // namespace

int32_t indexer_deal_capacity(int32_t cache_dtype) {
  if (cache_dtype == CSA_BF16) return Plan<false>::kCapTiles;
  if (cache_dtype == CSA_E2M1) return Plan<true>::kCapTiles;
  return 0;
}

int32_t indexer_deal_bound(int32_t n_rows, int32_t max_n, int32_t G) {
  if (n_rows <= 0 || n_rows >= G || n_rows > kDealMaxRows) return -1;
  // the device picks the smallest feasible budget; ceil(T / (G - n_rows)) is
  // always feasible (sum_r ceil(t_r / B) <= T / B + n_rows) and T <= n_rows * tiles(max_n)
  const int64_t tiles = (max_n + kTile - 1) / kTile;
  const int64_t T = (int64_t)n_rows * tiles;
  const int64_t B = (T + (G - n_rows) - 1) / (G - n_rows);
  return (int32_t)(B < tiles ? B : tiles);
}

// Two list slots per CTA (even deal: one per row the CTA meets).
size_t deal_candidate_bytes(int32_t G, int32_t k) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  return 2 * up((size_t)2 * G * 2 * k * 4) + 2 * up((size_t)2 * G * 4) + 3 * up((size_t)kDealMaxRows * 4);
}

DealCandidates deal_candidates(void* base, int32_t G, int32_t k) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  uint8_t* p = reinterpret_cast<uint8_t*>(base);
  const size_t lists = up((size_t)2 * G * 2 * k * 4), words = up((size_t)2 * G * 4),
               rows = up((size_t)kDealMaxRows * 4);
  DealCandidates c;
  c.key = reinterpret_cast<uint32_t*>(p);
  c.idx = reinterpret_cast<int32_t*>(p + lists);
  c.cnt = reinterpret_cast<int32_t*>(p + 2 * lists);
  c.thr = reinterpret_cast<uint32_t*>(p + 2 * lists + words);
  c.row_first = reinterpret_cast<int32_t*>(p + 2 * lists + 2 * words);
  c.row_ctas = reinterpret_cast<int32_t*>(p + 2 * lists + 2 * words + rows);
  c.row_seg = reinterpret_cast<int32_t*>(p + 2 * lists + 2 * words + 2 * rows);
  c.ctas = G;
  c.cap = 2 * k;
  return c;
}

bool indexer_tc_eligible(const IndexerArgs& a) {
  const uintptr_t d = reinterpret_cast<uintptr_t>(a.cache.data), s = reinterpret_cast<uintptr_t>(a.cache.scales);
  return a.heads == kHI && a.dim == kDI && a.cache.rows_per_block == kRowsPerBlock &&
         ((a.cache.dtype == CSA_BF16 && d % 16 == 0) || (a.cache.dtype == CSA_E2M1 && d % 16 == 0 && s % 16 == 0));
}

template <bool kFp4, int kR>
static cudaError_t launch_indexer_tc_t(const IndexerArgs& args, int32_t n_rows, int32_t G, cudaStream_t s) {
  using P = Plan<kFp4, kR>;
  static PerDevice attrs;
  cudaError_t e = with_device_slot(attrs, [](int, int64_t& done) {
    if (done) return cudaSuccess;
    const cudaError_t r = cudaFuncSetAttribute(indexer_tc_kernel<kFp4, kR>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes<kFp4, kR>());
    if (r == cudaSuccess) done = 1;
    return r;
  });
  if (e != cudaSuccess) return e;
  IndexerArgs a = args;
  a.n_rows = n_rows;
  if (!kFp4 && !encode_bf16_map(&a.k_map, a.cache.data, kDI, (uint64_t)a.cache.num_blocks * kRowsPerBlock, kDI * 2,
                                64, kRowsPerBlock))
    return cudaErrorInvalidValue;
  if (a.sel_k > 0)
    return launch_k(indexer_tc_kernel<kFp4, kR>, dim3(G), dim3(P::kThreads), smem_bytes<kFp4, kR>(), s, 0, a);
  const int32_t tiles = (a.max_n + kTile - 1) / kTile;
  // one CTA per SM: as many splits per row as fit in a single wave
  int32_t splits = n_rows > 0 ? G / n_rows : 1;
  if (splits > tiles) splits = tiles;
  // every CTA's range must fit the cached block-table slice (kTblMax blocks)
  const int32_t tiles_per_cta_max = kTblMax * kRowsPerBlock / kTile;
  const int32_t min_splits = (tiles + tiles_per_cta_max - 1) / tiles_per_cta_max;
  if (splits < min_splits) splits = min_splits;
  if (splits < 1) splits = 1;
  return launch_k(indexer_tc_kernel<kFp4, kR>, dim3(n_rows, splits), dim3(P::kThreads), smem_bytes<kFp4, kR>(), s,
                  0, a);
}

cudaError_t launch_indexer_tc(const IndexerArgs& a, int32_t n_rows, int32_t G, cudaStream_t s) {
  if (a.cache.dtype == CSA_E2M1) return launch_indexer_tc_t<true, 1>(a, n_rows, G, s);
  // score-scratch batches of many rows (prefill chunks): four rows of a
  // sequence share every key tile
  if (a.sel_k <= 0 && n_rows >= 2 * G) return launch_indexer_tc_t<false, 4>(a, n_rows, G, s);
  return launch_indexer_tc_t<false, 1>(a, n_rows, G, s);
}

}  // namespace csa
