// DSA indexer scores on the sm_103a tensor cores: s_i = sum_h w_h relu(q_h . k_i)
// ("vLLM解密：DeepSeek-V4本地部署為何如此困難" §二 item 3; "vLLM DeepSeek V4
// Support", "DeepSeek Sparse Attention (DSA)"; fp4 indexer cache: "DeepSeek V4
// Attention Architecture", last paragraph).
//
// Shape: 64 indexer heads x 128 dims.  One CTA takes one query row and a
// contiguous range of 128-entry tiles.  Entries are the M dimension:
//   S^T [128 entries x 64 heads] = K_idx [128 x 128] . Q_idx^T [128 x 64]
// so thread t of the epilogue warps owns TMEM lane t = entry t, reads its 64
// head dots, and writes one score.  Keys go into a 4-stage ring of
// 128B-swizzled K-major tiles.  A tile is two 64-entry paged blocks, 16 KB
// each and contiguous in a bf16 cache, so bf16 tiles arrive as four TMA boxes
// (64 dims x 64 entries); e2m1 rows (64 code bytes + 8 e4m3 scale bytes) come
// by cp.async into a raw ring and are dequantised to bf16 (exact: a 2-bit
// e2m1 significand times a 4-bit e4m3 one fits bf16).
// TMEM holds two S^T buffers so the epilogue of tile i overlaps the MMA of i+1.
//
// Warps 0-3: epilogue; warps 4-10: producers; warp 11: TMEM allocation + MMA issue.

#include "csa_kernels.h"
#include "tc_ptx.cuh"

namespace csa {
namespace {

using namespace tc;

constexpr int kHI = 64, kDI = 128, kTile = 128, kStages = 4;
constexpr int kEpi = 128, kProd = 224;
constexpr int kThreads = kEpi + kProd + 32;
constexpr int kMmaWarp = (kEpi + kProd) / 32;
constexpr uint32_t kQBytes = kHI * kDI * 2;         // 16 KB: 2 K-atoms of 64 rows x 128 B
constexpr uint32_t kStageBytes = kTile * kDI * 2;   // 32 KB: 2 K-atoms of 128 rows x 128 B
constexpr uint32_t kAtomBytes = kTile * 128;        // 16 KB
constexpr uint32_t kRawCodes = kTile * kDI / 2;     // 8 KB of e2m1 codes per tile
constexpr uint32_t kRawScales = kTile * kDI / 16;   // 1 KB of e4m3 scales per tile
constexpr uint32_t kRawBytes = kRawCodes + kRawScales;
constexpr uint32_t kOffQ = 0, kOffStage = kQBytes, kOffRaw = kOffStage + kStages * kStageBytes;
constexpr uint32_t kOffMisc = kOffRaw + kStages * kRawBytes;
constexpr uint32_t kTmemCols = 128;
constexpr int kRowsPerBlock = 64;  // entries per 256-position block (c4a)
constexpr int kTblMax = 1024;      // block-table entries a CTA caches (= 512 tiles)

struct Misc {
  uint64_t full[kStages], empty[kStages], tfull[2], tempty[2];
  uint32_t tmem_base;
  int32_t abort;
  float w[kHI];
  int32_t tbl[kTblMax];  // physical blocks of the CTA's entry range (-1: unmapped / out of range)
};
constexpr uint32_t kSmemBytes = kOffMisc + sizeof(Misc) + 1024;

__device__ __forceinline__ bool wait_or_abort(Misc& ms, uint64_t* bar, uint32_t parity, int32_t* err) {
  if (*reinterpret_cast<volatile int32_t*>(&ms.abort)) return false;
  if (mbar_wait(bar, parity)) return true;
  *reinterpret_cast<volatile int32_t*>(&ms.abort) = 1;
  record_error(err, CSA_ERR_TIMEOUT);
  return false;
}

struct Range {
  int seq;
  int32_t n, t0, nt;  // visible entries, first tile, tile count
};

__device__ __forceinline__ Range row_range(const IndexerArgs& a, int r) {
  Range g;
  g.seq = a.seq_id[r];
  g.n = n_visible(a.pos[r], a.ratio, a.window);
  if (g.n > a.max_n) {
    record_error(a.err, CSA_ERR_DEVICE_BOUNDS);
    g.n = a.max_n;
  }
  const int32_t tiles = (g.n + kTile - 1) / kTile;
  const int32_t per = (tiles + gridDim.y - 1) / gridDim.y;
  g.t0 = min(tiles, (int32_t)blockIdx.y * per);
  g.nt = min(tiles, g.t0 + per) - g.t0;
  return g;
}

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

// Physical row of entry e of this CTA's range, from the cached block table; -1 if unmapped.
__device__ __forceinline__ int64_t entry_row(const Misc& ms, int32_t blk0, int32_t e) {
  const int32_t j = (e / kRowsPerBlock) - blk0;
  if (j < 0 || j >= kTblMax) return -1;  // the launcher keeps every CTA's range inside the cache
  const int32_t pb = ms.tbl[j];
  return pb < 0 ? -1 : (int64_t)pb * kRowsPerBlock + (e % kRowsPerBlock);
}

// bf16 with a tensor map: one thread issues each tile as up to four TMA boxes
// (two blocks x two 64-dim atoms); a block that is unmapped or past the visible
// entries is not loaded (its scores are not used).
__device__ void producer_tma(const IndexerArgs& a, const Range& g, uint8_t* smem, Misc& ms) {
  const int32_t blk0 = g.t0 * kTile / kRowsPerBlock;
  for (int i = 0; i < g.nt; ++i) {
    const int s = i % kStages;
    if (i >= kStages) wait_or_abort(ms, &ms.empty[s], ((i / kStages) - 1) & 1, a.err);
    const int32_t e0 = (g.t0 + i) * kTile;
    int32_t pb[2];
    uint32_t bytes = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int32_t e = e0 + h * kRowsPerBlock, j = e / kRowsPerBlock - blk0;
      pb[h] = (e < g.n && j >= 0 && j < kTblMax) ? ms.tbl[j] : -1;
      if (pb[h] >= 0) bytes += kRowsPerBlock * kDI * 2;
    }
    mbar_arrive_expect_tx(&ms.full[s], bytes);
    uint8_t* sb = smem + kOffStage + s * kStageBytes;
#pragma unroll
    for (int h = 0; h < 2; ++h)
      if (pb[h] >= 0)
#pragma unroll
        for (int at = 0; at < kDI / 64; ++at)
          tma_load_2d(sb + at * kAtomBytes + h * (kRowsPerBlock * 128), &a.k_map, 64 * at, pb[h] * kRowsPerBlock,
                      &ms.full[s]);
  }
}

// Each thread derives its own rows' addresses from the cached table, so issuing
// a tile needs no barrier; e2m1 tiles need one before the conversion reads
// bytes other threads copied.
__device__ void producer_role(const IndexerArgs& a, const Range& g, uint8_t* smem, Misc& ms, int pt) {
  const bool fp4 = a.cache.dtype == CSA_E2M1;
  const uint32_t stage0 = smem_u32(smem + kOffStage), raw0 = smem_u32(smem + kOffRaw);
  const int32_t blk0 = g.t0 * kTile / kRowsPerBlock;
  const uint8_t* base = reinterpret_cast<const uint8_t*>(a.cache.data);
  const uint8_t* sbase = reinterpret_cast<const uint8_t*>(a.cache.scales);
  for (int i = 0; i < g.nt + 2; ++i) {
    if (i < g.nt) {
      const int s = i % kStages;
      if (i >= kStages) wait_or_abort(ms, &ms.empty[s], ((i / kStages) - 1) & 1, a.err);
      const int32_t e0 = (g.t0 + i) * kTile;
      if (!fp4) {
        // 16 consecutive threads per 256-byte row
        const uint32_t sb = stage0 + s * kStageBytes;
        for (int x = pt; x < kTile * 16; x += kProd) {
          const uint32_t key = x >> 4, piece = x & 15;
          const int32_t e = e0 + (int32_t)key;
          const int64_t pr = e < g.n ? entry_row(ms, blk0, e) : -1;
          const uint32_t dst = sb + (piece >> 3) * kAtomBytes + (key >> 3) * 1024 + (key & 7) * 128 +
                               (((piece & 7) ^ (key & 7)) << 4);
          cp_async16(dst, pr >= 0 ? base + pr * (kDI * 2) + piece * 16 : base, pr >= 0 ? 16u : 0u);
        }
      } else {
        // raw ring: [128 rows][64 code bytes] then [128 rows][8 scale bytes]
        const uint32_t rb = raw0 + s * kRawBytes;
        for (int x = pt; x < kTile * 4; x += kProd) {
          const uint32_t key = x >> 2, piece = x & 3;
          const int32_t e = e0 + (int32_t)key;
          const int64_t pr = e < g.n ? entry_row(ms, blk0, e) : -1;
          cp_async16(rb + key * 64 + piece * 16, pr >= 0 ? base + pr * (kDI / 2) + piece * 16 : base,
                     pr >= 0 ? 16u : 0u);
        }
        // two entries' 8 scale bytes per 16-byte piece; entries 2x, 2x+1 share a block
        for (int x = pt; x < kTile / 2; x += kProd) {
          const int32_t e = e0 + 2 * x;
          const int64_t pr = e < g.n ? entry_row(ms, blk0, e) : -1;
          const bool both = e + 1 < g.n;
          if (pr >= 0 && both) {
            cp_async16(rb + kRawCodes + x * 16, sbase + pr * (kDI / 16), 16u);
          } else {
            const uint2 v0 = pr >= 0 ? *reinterpret_cast<const uint2*>(sbase + pr * (kDI / 16)) : make_uint2(0, 0);
            *reinterpret_cast<uint4*>(smem + kOffRaw + s * kRawBytes + kRawCodes + x * 16) =
                make_uint4(v0.x, v0.y, 0u, 0u);
          }
        }
      }
    }
    cp_async_commit();
    if (i >= 2) {
      // the tile issued two groups ago has landed
      cp_async_wait<2>();
      const int ii = i - 2, s = ii % kStages;
      if (fp4) {
        named_bar(2, kProd);  // every producer's copies of tile ii are visible
        const uint8_t* rb = smem + kOffRaw + s * kRawBytes;
        uint8_t* sb = smem + kOffStage + s * kStageBytes;
        // 16 bytes of codes = 32 values = 64 bytes of bf16 = 4 swizzled pieces
        for (int x = pt; x < kTile * 4; x += kProd) {
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
        named_bar(2, kProd);  // the raw stage may be refilled only after everyone converted
      }
      fence_proxy_async();
      mbar_arrive(&ms.full[s]);
    }
  }
  cp_async_wait<0>();
}

__device__ void mma_role(const IndexerArgs& a, const Range& g, uint8_t* smem, Misc& ms, uint32_t tmem) {
  constexpr uint32_t idesc = idesc_bf16(128, kHI, 0, 0);
  const uint32_t stage0 = smem_u32(smem + kOffStage), qbase = smem_u32(smem + kOffQ);
  for (int i = 0; i < g.nt; ++i) {
    const int s = i % kStages, b = i & 1;
    wait_or_abort(ms, &ms.full[s], (i / kStages) & 1, a.err);
    if (i >= 2) wait_or_abort(ms, &ms.tempty[b], ((i >> 1) - 1) & 1, a.err);
    tc_fence_after();
#pragma unroll
    for (int ks = 0; ks < kDI / 16; ++ks) {
      const uint64_t ad = sdesc_sw128(stage0 + s * kStageBytes + (ks >> 2) * kAtomBytes + (ks & 3) * 32, 16, 1024);
      const uint64_t bd = sdesc_sw128(qbase + (ks >> 2) * (kHI * 128) + (ks & 3) * 32, 16, 1024);
      mma_bf16(tmem + 64 * b, ad, bd, idesc, ks > 0);
    }
    mma_commit(&ms.empty[s]);
    mma_commit(&ms.tfull[b]);
  }
}

__device__ void epilogue_role(const IndexerArgs& a, const Range& g, Misc& ms, uint32_t tmem, int et) {
  const uint32_t lane_addr = tmem + ((uint32_t)((et >> 5) * 32) << 16);
  float w[kHI];
#pragma unroll
  for (int h = 0; h < kHI; ++h) w[h] = ms.w[h];
  float* out = a.scores + (int64_t)blockIdx.x * a.max_n;
  const int32_t blk0 = g.t0 * kTile / kRowsPerBlock;
  for (int i = 0; i < g.nt; ++i) {
    const int b = i & 1;
    wait_or_abort(ms, &ms.tfull[b], (i >> 1) & 1, a.err);
    tc_fence_after();
    float v[kHI];
#pragma unroll
    for (int q = 0; q < 4; ++q) tmem_ld16(lane_addr + 64 * b + 16 * q, v + 16 * q);
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive(&ms.tempty[b]);
    float s = 0.f;
#pragma unroll
    for (int h = 0; h < kHI; ++h) s = fmaf(w[h], fmaxf(v[h], 0.f), s);
    const int32_t e = (g.t0 + i) * kTile + et, j = e / kRowsPerBlock - blk0;
    // an unmapped block (reported when the table was cached) scores 0
    if (e < g.n) out[e] = (j >= 0 && j < kTblMax && ms.tbl[j] >= 0) ? s : 0.f;
  }
}

__global__ void __launch_bounds__(kThreads, 1) indexer_tc_kernel(const __grid_constant__ IndexerArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc& ms = *reinterpret_cast<Misc*>(smem + kOffMisc);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int r = blockIdx.x;
  const Range g = row_range(a, r);

  if (tid == 0) {
    const bool tma = a.k_tma && a.cache.dtype == CSA_BF16;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ms.full[s], tma ? 1 : kProd);
      mbar_init(&ms.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ms.tfull[b], 1);
      mbar_init(&ms.tempty[b], kEpi);
    }
    mbar_init_fence();
    ms.abort = 0;
  }
  if (tid < kHI) ms.w[tid] = a.w[(int64_t)r * kHI + tid];
  {
    // block-table slice of the CTA's entry range
    const int32_t blk0 = g.t0 * kTile / kRowsPerBlock;
    const int32_t nblk = min(kTblMax, (g.nt * kTile + kRowsPerBlock - 1) / kRowsPerBlock);
    for (int j = tid; j < nblk; j += kThreads) {
      const int32_t lb = blk0 + j;
      int32_t pb = -1;
      if (g.seq >= 0 && g.seq < a.bt.num_seqs && lb < a.bt.stride) {
        pb = a.bt.table[(int64_t)g.seq * a.bt.stride + lb];
        if (pb >= a.cache.num_blocks) pb = -1;
      }
      if (pb < 0 && lb * kRowsPerBlock < g.n) record_error(a.err, CSA_ERR_DEVICE_BOUNDS);
      ms.tbl[j] = pb;
    }
  }
  if (warp == kMmaWarp) tmem_alloc(&ms.tmem_base, kTmemCols);
  // Q_idx^T: bf16, 128B-swizzled K-major, rows = heads; 8 dims per 16-byte
  // piece, every thread's loads issued before its stores
  {
    constexpr int kPieces = kHI * kDI / 8;
    constexpr int kPer = (kPieces + kThreads - 1) / kThreads;
    uint32_t w[kPer][4];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int x = min(tid + u * kThreads, kPieces - 1);  // clamped; stored below only when in range
      const int64_t qb = (int64_t)r * kHI * kDI + 8 * x;
      if (a.q_dtype == CSA_BF16) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q_idx) + qb));
        w[u][0] = v.x; w[u][1] = v.y; w[u][2] = v.z; w[u][3] = v.w;
      } else {
        const float4* src = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.q_idx) + qb);
        const float4 v0 = __ldg(src), v1 = __ldg(src + 1);
        w[u][0] = (uint32_t)f32_to_bf16(v0.x) | ((uint32_t)f32_to_bf16(v0.y) << 16);
        w[u][1] = (uint32_t)f32_to_bf16(v0.z) | ((uint32_t)f32_to_bf16(v0.w) << 16);
        w[u][2] = (uint32_t)f32_to_bf16(v1.x) | ((uint32_t)f32_to_bf16(v1.y) << 16);
        w[u][3] = (uint32_t)f32_to_bf16(v1.z) | ((uint32_t)f32_to_bf16(v1.w) << 16);
      }
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int x = tid + u * kThreads;
      if (x >= kPieces) break;
      const int h = x / (kDI / 8), d0 = 8 * (x % (kDI / 8));
      *reinterpret_cast<uint4*>(smem + kOffQ + sw128_offset(h, d0, kHI)) = make_uint4(w[u][0], w[u][1], w[u][2], w[u][3]);
    }
  }
  fence_proxy_async();
  pdl_trigger();
  pdl_wait();  // caches and the score scratch may be in use by the previous launch until here
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;

  if (warp < 4) {
    epilogue_role(a, g, ms, tmem, tid);
  } else if (warp < kMmaWarp) {
    if (!(a.k_tma && a.cache.dtype == CSA_BF16)) producer_role(a, g, smem, ms, tid - kEpi);
    else if (tid == kEpi) producer_tma(a, g, smem, ms);
  } else if ((tid & 31) == 0) {
    mma_role(a, g, smem, ms, tmem);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool indexer_tc_eligible(const IndexerArgs& a) {
  return a.heads == kHI && a.dim == kDI && a.cache.rows_per_block == kRowsPerBlock &&
         (a.cache.dtype == CSA_BF16 || a.cache.dtype == CSA_E2M1);
}

cudaError_t launch_indexer_tc(const IndexerArgs& args, int32_t n_rows, cudaStream_t s) {
  static PerDevice attrs;
  cudaError_t e = with_device_slot(attrs, [](int, int64_t& done) {
    if (done) return cudaSuccess;
    const cudaError_t r =
        cudaFuncSetAttribute(indexer_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (r == cudaSuccess) done = 1;
    return r;
  });
  if (e != cudaSuccess) return e;
  int n_sm = 0;
  if ((e = sm_count(&n_sm)) != cudaSuccess) return e;
  IndexerArgs a = args;
  a.k_tma = a.cache.dtype == CSA_BF16 &&
            encode_bf16_map(&a.k_map, a.cache.data, kDI, (uint64_t)a.cache.num_blocks * kRowsPerBlock, kDI * 2,
                            64, kRowsPerBlock);
  const int32_t tiles = (a.max_n + kTile - 1) / kTile;
  // one CTA per SM: as many splits per row as fit in a single wave
  int32_t splits = n_rows > 0 ? n_sm / n_rows : 1;
  if (splits > tiles) splits = tiles;
  // every CTA's range must fit the cached block-table slice (kTblMax blocks)
  const int32_t tiles_per_cta_max = kTblMax * kRowsPerBlock / kTile;
  const int32_t min_splits = (tiles + tiles_per_cta_max - 1) / tiles_per_cta_max;
  if (splits < min_splits) splits = min_splits;
  if (splits < 1) splits = 1;
  return launch_k(indexer_tc_kernel, dim3(n_rows, splits), dim3(kThreads), kSmemBytes, s, kStreamOrder, 0, a);
}

}  // namespace csa
