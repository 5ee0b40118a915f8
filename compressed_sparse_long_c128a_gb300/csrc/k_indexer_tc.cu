// DSA indexer scores on the sm_103a tensor cores: s_i = sum_h w_h relu(q_h . k_i)
// ("vLLM解密：DeepSeek-V4本地部署為何如此困難" §二 item 3; "vLLM DeepSeek V4
// Support", "DeepSeek Sparse Attention (DSA)"; fp4 indexer cache: "DeepSeek V4
// Attention Architecture", last paragraph).
//
// Shape: 64 indexer heads x 128 dims.  One CTA takes one query row and a
// contiguous range of 128-entry tiles.  Entries are the M dimension:
//   S^T [128 entries x 64 heads] = K_idx [128 x 128] . Q_idx^T [128 x 64]
// so thread t of the epilogue warps owns TMEM lane t = entry t, reads its 64
// head dots, and writes one score.  Keys are gathered into a 4-stage ring of
// 128B-swizzled K-major tiles: bf16 rows by cp.async; e2m1 rows (64 code bytes
// + 8 e4m3 scale bytes) by cp.async into a raw ring, then dequantised to bf16
// (exact: a 2-bit e2m1 significand times a 4-bit e4m3 one fits bf16).
// TMEM holds two S^T buffers so the epilogue of tile i overlaps the MMA of i+1.
//
// Warps 0-3: epilogue; warps 4-6: producers; warp 7: TMEM allocation + MMA issue.

#include "csa_kernels.h"
#include "tc_ptx.cuh"

namespace csa {
namespace {

using namespace tc;

constexpr int kHI = 64, kDI = 128, kTile = 128, kStages = 4;
constexpr int kEpi = 128, kProd = 96;
constexpr int kThreads = kEpi + kProd + 32;
constexpr uint32_t kQBytes = kHI * kDI * 2;         // 16 KB: 2 K-atoms of 64 rows x 128 B
constexpr uint32_t kStageBytes = kTile * kDI * 2;   // 32 KB: 2 K-atoms of 128 rows x 128 B
constexpr uint32_t kAtomBytes = kTile * 128;        // 16 KB
constexpr uint32_t kRawCodes = kTile * kDI / 2;     // 8 KB of e2m1 codes per tile
constexpr uint32_t kRawScales = kTile * kDI / 16;   // 1 KB of e4m3 scales per tile
constexpr uint32_t kRawBytes = kRawCodes + kRawScales;
constexpr uint32_t kOffQ = 0, kOffStage = kQBytes, kOffRaw = kOffStage + kStages * kStageBytes;
constexpr uint32_t kOffMisc = kOffRaw + kStages * kRawBytes;
constexpr uint32_t kTmemCols = 128;

struct Misc {
  uint64_t full[kStages], empty[kStages], tfull[2], tempty[2];
  uint32_t tmem_base;
  int32_t abort;
  float w[kHI];
  const uint8_t* rowptr[kTile];   // codes (or bf16 row) of each entry of the tile being issued
  const uint8_t* sclptr[kTile];   // e2m1 scale bytes of each entry
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

// e2m1 code -> bf16 bits of code * scale (exact)
__device__ __forceinline__ uint32_t e2m1_bf16(uint32_t code, float scale) {
  return f32_to_bf16(e2m1_to_f32(code) * scale);
}

__device__ void producer_role(const IndexerArgs& a, const Range& g, uint8_t* smem, Misc& ms, int pt) {
  const bool fp4 = a.cache.dtype == CSA_E2M1;
  const uint32_t stage0 = smem_u32(smem + kOffStage), raw0 = smem_u32(smem + kOffRaw);
  for (int i = 0; i < g.nt + 2; ++i) {
    if (i < g.nt) {
      const int s = i % kStages;
      if (i >= kStages) wait_or_abort(ms, &ms.empty[s], ((i / kStages) - 1) & 1, a.err);
      const int32_t e0 = (g.t0 + i) * kTile;
      for (int slot = pt; slot < kTile; slot += kProd) {
        const int32_t e = e0 + slot;
        const uint8_t* rp = nullptr;
        const uint8_t* sp = nullptr;
        if (e < g.n) {
          const int64_t prow = phys_row(a.bt, a.cache, g.seq, e, a.err);
          if (prow >= 0) {
            rp = reinterpret_cast<const uint8_t*>(a.cache.data) + prow * (fp4 ? kDI / 2 : kDI * 2);
            if (fp4) sp = reinterpret_cast<const uint8_t*>(a.cache.scales) + prow * (kDI / 16);
          }
        }
        ms.rowptr[slot] = rp;
        ms.sclptr[slot] = sp;
      }
      named_bar(2, kProd);
      if (!fp4) {
        // 16 consecutive threads per 256-byte row
        const uint32_t sb = stage0 + s * kStageBytes;
        for (int x = pt; x < kTile * 16; x += kProd) {
          const uint32_t key = x >> 4, piece = x & 15;
          const uint8_t* rp = ms.rowptr[key];
          const uint32_t dst = sb + (piece >> 3) * kAtomBytes + (key >> 3) * 1024 + (key & 7) * 128 +
                               (((piece & 7) ^ (key & 7)) << 4);
          cp_async16(dst, rp ? rp + piece * 16 : a.cache.data, rp ? 16u : 0u);
        }
      } else {
        // raw ring: [128 rows][64 code bytes] then [128 rows][8 scale bytes]
        const uint32_t rb = raw0 + s * kRawBytes;
        for (int x = pt; x < kTile * 4; x += kProd) {
          const uint32_t key = x >> 2, piece = x & 3;
          const uint8_t* rp = ms.rowptr[key];
          cp_async16(rb + key * 64 + piece * 16, rp ? rp + piece * 16 : a.cache.data, rp ? 16u : 0u);
        }
        for (int x = pt; x < kTile / 2; x += kProd) {  // two rows' 8 scale bytes per 16-byte piece
          const uint8_t* s0 = ms.sclptr[2 * x];
          const uint8_t* s1 = ms.sclptr[2 * x + 1];
          if (s0 && s1 && s1 == s0 + 8) {
            cp_async16(rb + kRawCodes + x * 16, s0, 16u);
          } else {
            uint2 v0 = s0 ? *reinterpret_cast<const uint2*>(s0) : make_uint2(0, 0);
            uint2 v1 = s1 ? *reinterpret_cast<const uint2*>(s1) : make_uint2(0, 0);
            *reinterpret_cast<uint4*>(smem + kOffRaw + s * kRawBytes + kRawCodes + x * 16) =
                make_uint4(v0.x, v0.y, v1.x, v1.y);
          }
        }
      }
      named_bar(2, kProd);  // rowptr / sclptr are rewritten for the next tile
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
          const float s0 = e4m3_to_f32(sc[0]), s1 = e4m3_to_f32(sc[1]);
          const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
          for (int half = 0; half < 4; ++half) {  // 8 values -> one 16-byte piece
            const float scl = half < 2 ? s0 : s1;
            const uint32_t word = cw[half];
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t lo = (word >> (8 * e)) & 0xF, hi = (word >> (8 * e + 4)) & 0xF;
              o[e] = e2m1_bf16(lo, scl) | (e2m1_bf16(hi, scl) << 16);
            }
            const uint32_t piece = q * 4 + half;  // 0..15 over the 128 dims
            *reinterpret_cast<uint4*>(sb + (piece >> 3) * kAtomBytes + (key >> 3) * 1024 + (key & 7) * 128 +
                                      (((piece & 7) ^ (key & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
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
    const int32_t e = (g.t0 + i) * kTile + et;
    if (e < g.n) out[e] = s;
  }
}

__global__ void __launch_bounds__(kThreads, 1) indexer_tc_kernel(const IndexerArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc& ms = *reinterpret_cast<Misc*>(smem + kOffMisc);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int r = blockIdx.x;
  const Range g = row_range(a, r);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ms.full[s], kProd);
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
  if (warp == 7) tmem_alloc(&ms.tmem_base, kTmemCols);
  // Q_idx^T: bf16, 128B-swizzled K-major, rows = heads
  for (int x = tid; x < kHI * kDI / 2; x += kThreads) {
    const int h = x / (kDI / 2), d = 2 * (x % (kDI / 2));
    const int64_t qb = ((int64_t)r * kHI + h) * kDI + d;
    const uint32_t v = (uint32_t)f32_to_bf16(load_elem(a.q_idx, a.q_dtype, qb)) |
                       ((uint32_t)f32_to_bf16(load_elem(a.q_idx, a.q_dtype, qb + 1)) << 16);
    *reinterpret_cast<uint32_t*>(smem + kOffQ + sw128_offset(h, d, kHI)) = v;
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;

  if (warp < 4) {
    epilogue_role(a, g, ms, tmem, tid);
  } else if (warp < 7) {
    producer_role(a, g, smem, ms, tid - kEpi);
  } else if ((tid & 31) == 0) {
    mma_role(a, g, smem, ms, tmem);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 7) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool indexer_tc_eligible(const IndexerArgs& a) {
  return a.heads == kHI && a.dim == kDI && (a.cache.dtype == CSA_BF16 || a.cache.dtype == CSA_E2M1);
}

cudaError_t launch_indexer_tc(const IndexerArgs& a, int32_t n_rows, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(indexer_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int32_t tiles = (a.max_n + kTile - 1) / kTile;
  int32_t splits = n_rows > 0 ? (148 + n_rows - 1) / n_rows : 1;
  if (splits > tiles) splits = tiles;
  if (splits < 1) splits = 1;
  indexer_tc_kernel<<<dim3(n_rows, splits), kThreads, kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace csa
